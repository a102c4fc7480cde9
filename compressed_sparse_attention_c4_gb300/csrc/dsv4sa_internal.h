// dsv4sa_internal.h -- launchers and per-file error-word readers shared by the
// C-ABI front end (api.cu) and the kernel files.  Not installed; not part of
// the public interface.
#pragma once

#include <cstdint>
#include <cuda_runtime_api.h>

#include "../../include/dsv4sa.h"

namespace dsv4sa {

int launch_indexer_logits(const dsv4sa_pool_desc* kpool, const int32_t* page_table, int32_t pt_stride,
                          const int32_t* q_seq, const int32_t* n_vis, const uint8_t* q_fp8, const float* q_scale,
                          const float* w, int32_t T, int32_t Hi, int32_t n_max, float* logits,
                          int64_t logits_stride, cudaStream_t stream);
int launch_indexer_logits_fp4(const dsv4sa_pool_desc* kpool, const int32_t* page_table, int32_t pt_stride,
                              const int32_t* q_seq, const int32_t* n_vis, const uint8_t* q_fp4,
                              const uint8_t* q_e8m0, const float* w, int32_t T, int32_t Hi, int32_t n_max,
                              float* logits, int64_t logits_stride, cudaStream_t stream);

// top-k: chunk length and chunk count used for a given (n_max, k); 0 chunks = unsupported.
void topk_plan(int32_t n_max, int32_t k, int32_t* chunk_len, int32_t* n_chunks);
// Optional: the KV pool (default layout) whose rows of the selected entries are
// prefetched into L2 as they are selected (query t's page table row q_seq[t]).
struct TopkPrefetch {
  const dsv4sa_pool_desc* pool;
  const int32_t* page_table;
  int32_t pt_stride;
  const int32_t* q_seq;
};
int launch_topk(const float* logits, int64_t logits_stride, const int32_t* n_vis, int32_t T, int32_t n_max,
                int32_t k, int32_t* idx, int32_t idx_stride, void* ws, size_t ws_bytes, cudaStream_t stream,
                const TopkPrefetch* prefetch);

int launch_copy(void* dst, const void* src, int64_t bytes, cudaStream_t stream);
int launch_copy_background(void* dst, const void* src, int64_t bytes, cudaStream_t stream);
int launch_window_indices(const int32_t* pos, int32_t T, int32_t window, int32_t ring, int32_t* idx_w,
                          int32_t idx_stride, cudaStream_t stream);
int launch_compress_indices(const int32_t* n_vis, int32_t T, int32_t kc, int32_t* idx, int32_t idx_stride,
                            cudaStream_t stream);

// attention: number of 128-row chunks of a query, and splits for a mode.
int32_t attn_chunks(int32_t kc, int32_t kw);
int32_t attn_splits(int32_t mode, int32_t kc, int32_t kw);
int launch_sparse_attn(int32_t mode, const dsv4sa_attn_args* a, cudaStream_t stream);
int launch_topk_sparse_attn(const dsv4sa_attn_args* a, const float* logits, int64_t logits_stride,
                            const int32_t* n_vis, int32_t n_max, int32_t k, void* topk_ws, size_t topk_ws_bytes,
                            cudaStream_t stream);
int attn_plan(int32_t mode, int32_t T, int32_t H, int32_t kc, int32_t kw, int32_t* nsplit, int32_t* rows_per_split,
              int32_t* launches);

// Raise a kernel's dynamic shared-memory limit once per (device, kernel slot),
// so repeated calls (and calls under stream capture) make no attribute call.
bool smem_attr_once(int device, int slot, const void* kernel, int bytes);

uint32_t read_error_word_indexer(cudaStream_t stream, bool clear);
uint32_t read_error_word_topk(cudaStream_t stream, bool clear);
uint32_t read_error_word_attn(cudaStream_t stream, bool clear);
uint32_t read_error_word_attn_decode(cudaStream_t stream, bool clear);
uint32_t read_error_word_writer(cudaStream_t stream, bool clear);
uint32_t read_error_word_compress(cudaStream_t stream, bool clear);
int launch_selftest_wait_timeout(int32_t* result, cudaStream_t stream);
int launch_compress_windows(const void* kv, const void* score, int64_t tok_stride, int64_t n_tok,
                            const int32_t* first_tok,
                            const int32_t* prev_tok, const int32_t* position, int32_t n, int32_t ratio,
                            int32_t overlap, const float* ape, const float* norm_w, float eps, const float* rope_cs,
                            int32_t rope_rows, void* out, cudaStream_t stream);
int launch_compress_online(const void* kv, const void* score, int64_t tok_stride, const int32_t* state_idx,
                           float* state, int32_t* state_count, int32_t slots, const int32_t* position, int32_t T,
                           const float* ape, const float* norm_w, float eps, const float* rope_cs, int32_t rope_rows,
                           void* out, int32_t* done, cudaStream_t stream);
int launch_cache_write(const dsv4sa_pool_desc* pool, const int32_t* page_table, int32_t pt_stride,
                       const int32_t* row_seq, const int32_t* row_entry, const void* rows, int32_t n,
                       bool rotate, cudaStream_t stream);

}  // namespace dsv4sa
