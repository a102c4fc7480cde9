// api.cpp -- the extern "C" entry points of libdsv4sa.so: host-side validation
// of every argument, then the launchers in the kernel files.  Nothing here
// allocates device memory or synchronises, except dsv4sa_check_errors.
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda_runtime_api.h>

#include "../../include/dsv4sa.h"
#include "dsv4sa_internal.h"

namespace {

constexpr int64_t kKvPageBytes = 64 * 448 + 64 * 128 + 64 * 32;   // 38912
constexpr int64_t kIdxPageBytes = 64 * 128 + 64 * 8;              // 8704
constexpr int64_t kIdxFp4PageBytes = 64 * 64 + 64 * 4;            // 4352

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// The kernels address pages with the default layout; a descriptor must match it.
bool pool_ok(const dsv4sa_pool_desc* d, int32_t kind) {
  if (!d || !d->base || d->kind != kind || d->num_pages < 1) return false;
  if (!aligned(d->base, 1024)) return false;
  dsv4sa_pool_desc ref;
  if (dsv4sa_pool_desc_init(&ref, kind, d->base, d->num_pages) != DSV4SA_OK) return false;
  return d->page_size == ref.page_size && d->nope_dim == ref.nope_dim && d->rope_dim == ref.rope_dim &&
         d->scale_group == ref.scale_group && d->n_scales == ref.n_scales && d->page_stride == ref.page_stride &&
         d->nope_off == ref.nope_off && d->rope_off == ref.rope_off && d->scale_off == ref.scale_off &&
         d->nope_row == ref.nope_row && d->rope_row == ref.rope_row && d->scale_row == ref.scale_row;
}

}  // namespace

namespace dsv4sa {

bool smem_attr_once(int device, int slot, const void* kernel, int bytes) {
  constexpr int kDevices = 64, kSlots = 16;
  static std::atomic<int> done[kDevices][kSlots];
  static std::mutex mu;
  if (device < 0 || device >= kDevices || slot < 0 || slot >= kSlots) return false;
  if (done[device][slot].load(std::memory_order_acquire) >= bytes) return true;
  std::lock_guard<std::mutex> lock(mu);
  if (done[device][slot].load(std::memory_order_relaxed) >= bytes) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
  done[device][slot].store(bytes, std::memory_order_release);
  return true;
}

}  // namespace dsv4sa

extern "C" {

DSV4SA_API int dsv4sa_version(void) { return 100; }

DSV4SA_API const char* dsv4sa_status_string(int s) {
  switch (s) {
    case DSV4SA_OK: return "ok";
    case DSV4SA_ERR_INVALID_ARG: return "invalid argument";
    case DSV4SA_ERR_UNSUPPORTED: return "unsupported size";
    case DSV4SA_ERR_WORKSPACE: return "workspace missing or too small";
    case DSV4SA_ERR_CUDA: return "CUDA runtime error";
    case DSV4SA_ERR_INDEX_OOB: return "index or page id out of range (device)";
    case DSV4SA_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

DSV4SA_API size_t dsv4sa_pool_bytes(int32_t kind, int64_t num_pages) {
  if (num_pages < 0) return 0;
  if (kind == DSV4SA_POOL_KV) return static_cast<size_t>(num_pages) * kKvPageBytes;
  if (kind == DSV4SA_POOL_IDXK) return static_cast<size_t>(num_pages) * kIdxPageBytes;
  if (kind == DSV4SA_POOL_IDXK_FP4) return static_cast<size_t>(num_pages) * kIdxFp4PageBytes;
  return 0;
}

DSV4SA_API int dsv4sa_pool_desc_init(dsv4sa_pool_desc* d, int32_t kind, void* base, int64_t num_pages) {
  if (!d || num_pages < 1 || !aligned(base, 1024)) return DSV4SA_ERR_INVALID_ARG;
  std::memset(d, 0, sizeof(*d));
  d->kind = kind;
  d->page_size = DSV4SA_PAGE_SIZE;
  d->scale_group = DSV4SA_SCALE_GROUP;
  d->num_pages = num_pages;
  d->base = base;
  if (kind == DSV4SA_POOL_KV) {
    d->nope_dim = DSV4SA_NOPE_DIM;
    d->rope_dim = DSV4SA_ROPE_DIM;
    d->n_scales = DSV4SA_NOPE_DIM / DSV4SA_SCALE_GROUP;
    d->page_stride = kKvPageBytes;
    d->nope_off = 0;
    d->rope_off = 64 * 448;
    d->scale_off = 64 * 448 + 64 * 128;
    d->nope_row = 448;
    d->rope_row = 128;
    d->scale_row = 32;
  } else if (kind == DSV4SA_POOL_IDXK) {
    d->nope_dim = DSV4SA_IDX_DIM;
    d->rope_dim = 0;
    d->n_scales = DSV4SA_IDX_DIM / DSV4SA_SCALE_GROUP;
    d->page_stride = kIdxPageBytes;
    d->nope_off = 0;
    d->rope_off = 0;
    d->scale_off = 64 * 128;
    d->nope_row = 128;
    d->rope_row = 0;
    d->scale_row = 8;
  } else if (kind == DSV4SA_POOL_IDXK_FP4) {
    d->nope_dim = DSV4SA_IDX_DIM;
    d->rope_dim = 0;
    d->scale_group = 32;
    d->n_scales = DSV4SA_IDX_DIM / 32;
    d->page_stride = kIdxFp4PageBytes;
    d->nope_off = 0;
    d->rope_off = 0;
    d->scale_off = 64 * 64;
    d->nope_row = 64;
    d->rope_row = 0;
    d->scale_row = 4;
  } else {
    return DSV4SA_ERR_INVALID_ARG;
  }
  return DSV4SA_OK;
}

DSV4SA_API int dsv4sa_indexer_logits(const dsv4sa_pool_desc* kpool, const int32_t* page_table, int32_t pt_stride,
                                     const int32_t* q_seq, const int32_t* n_vis, const uint8_t* q_fp8,
                                     const float* q_scale, const float* w, int32_t T, int32_t Hi, int32_t n_max,
                                     float* logits, int64_t logits_stride, cudaStream_t stream) {
  if (T < 0 || n_max < 0 || pt_stride < 0 || logits_stride < 0) return DSV4SA_ERR_INVALID_ARG;
  if (Hi < 1 || Hi > DSV4SA_MAX_IDX_HEADS) return DSV4SA_ERR_UNSUPPORTED;
  if (T == 0 || n_max == 0) return DSV4SA_OK;
  if (!pool_ok(kpool, DSV4SA_POOL_IDXK)) return DSV4SA_ERR_INVALID_ARG;
  if (!page_table || !q_seq || !n_vis || !q_fp8 || !q_scale || !w || !logits) return DSV4SA_ERR_INVALID_ARG;
  if (!aligned(q_fp8, 16) || !aligned(q_scale, 8) || !aligned(logits, 4)) return DSV4SA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(n_max) > static_cast<int64_t>(pt_stride) * DSV4SA_PAGE_SIZE) return DSV4SA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(n_max) > logits_stride) return DSV4SA_ERR_INVALID_ARG;
  return dsv4sa::launch_indexer_logits(kpool, page_table, pt_stride, q_seq, n_vis, q_fp8, q_scale, w, T, Hi, n_max,
                                       logits, logits_stride, stream);
}

DSV4SA_API int dsv4sa_indexer_logits_fp4(const dsv4sa_pool_desc* kpool, const int32_t* page_table,
                                         int32_t pt_stride, const int32_t* q_seq, const int32_t* n_vis,
                                         const uint8_t* q_fp4, const uint8_t* q_e8m0, const float* w, int32_t T,
                                         int32_t Hi, int32_t n_max, float* logits, int64_t logits_stride,
                                         cudaStream_t stream) {
  if (T < 0 || n_max < 0 || pt_stride < 0 || logits_stride < 0) return DSV4SA_ERR_INVALID_ARG;
  if (Hi < 1 || Hi > DSV4SA_MAX_IDX_HEADS_FP4) return DSV4SA_ERR_UNSUPPORTED;
  if (T == 0 || n_max == 0) return DSV4SA_OK;
  if (!pool_ok(kpool, DSV4SA_POOL_IDXK_FP4)) return DSV4SA_ERR_INVALID_ARG;
  if (!page_table || !q_seq || !n_vis || !q_fp4 || !q_e8m0 || !w || !logits) return DSV4SA_ERR_INVALID_ARG;
  if (!aligned(q_fp4, 16) || !aligned(q_e8m0, 4) || !aligned(logits, 4)) return DSV4SA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(n_max) > static_cast<int64_t>(pt_stride) * DSV4SA_PAGE_SIZE) return DSV4SA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(n_max) > logits_stride) return DSV4SA_ERR_INVALID_ARG;
  return dsv4sa::launch_indexer_logits_fp4(kpool, page_table, pt_stride, q_seq, n_vis, q_fp4, q_e8m0, w, T, Hi,
                                           n_max, logits, logits_stride, stream);
}

DSV4SA_API size_t dsv4sa_topk_workspace_size(int32_t T, int32_t n_max, int32_t k) {
  int32_t chunk, nch;
  dsv4sa::topk_plan(n_max, k, &chunk, &nch);
  if (nch <= 1 || T <= 0) return 0;
  return static_cast<size_t>(T) * nch * k * 8;
}

DSV4SA_API int dsv4sa_topk(const float* logits, int64_t logits_stride, const int32_t* n_vis, int32_t T,
                           int32_t n_max, int32_t k, int32_t* idx, int32_t idx_stride, void* ws, size_t ws_bytes,
                           cudaStream_t stream) {
  if (T < 0 || n_max < 0 || logits_stride < 0) return DSV4SA_ERR_INVALID_ARG;
  if (k < 1 || k > DSV4SA_MAX_TOPK) return DSV4SA_ERR_UNSUPPORTED;
  if (idx_stride < k) return DSV4SA_ERR_INVALID_ARG;
  if (T == 0) return DSV4SA_OK;
  if (!n_vis || !idx || (n_max > 0 && !logits)) return DSV4SA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(n_max) > logits_stride && n_max > 0) return DSV4SA_ERR_INVALID_ARG;
  int32_t chunk, nch;
  dsv4sa::topk_plan(n_max, k, &chunk, &nch);
  if (nch == 0) return DSV4SA_ERR_UNSUPPORTED;
  if (nch > 1 && (!ws || ws_bytes < dsv4sa_topk_workspace_size(T, n_max, k) || !aligned(ws, 16)))
    return DSV4SA_ERR_WORKSPACE;
  return dsv4sa::launch_topk(logits, logits_stride, n_vis, T, n_max, k, idx, idx_stride, ws, ws_bytes, stream,
                             nullptr);
}

DSV4SA_API int dsv4sa_topk_prefetch(const float* logits, int64_t logits_stride, const int32_t* n_vis, int32_t T,
                                    int32_t n_max, int32_t k, int32_t* idx, int32_t idx_stride, void* ws,
                                    size_t ws_bytes, const dsv4sa_pool_desc* kv_pool, const int32_t* kv_page_table,
                                    int32_t kv_pt_stride, const int32_t* q_seq, cudaStream_t stream) {
  if (T < 0 || n_max < 0 || logits_stride < 0) return DSV4SA_ERR_INVALID_ARG;
  if (k < 1 || k > DSV4SA_MAX_TOPK) return DSV4SA_ERR_UNSUPPORTED;
  if (idx_stride < k) return DSV4SA_ERR_INVALID_ARG;
  if (T == 0) return DSV4SA_OK;
  if (!n_vis || !idx || (n_max > 0 && !logits)) return DSV4SA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(n_max) > logits_stride && n_max > 0) return DSV4SA_ERR_INVALID_ARG;
  if (!pool_ok(kv_pool, DSV4SA_POOL_KV) || !kv_page_table || kv_pt_stride < 1 || !q_seq) return DSV4SA_ERR_INVALID_ARG;
  int32_t chunk, nch;
  dsv4sa::topk_plan(n_max, k, &chunk, &nch);
  if (nch == 0) return DSV4SA_ERR_UNSUPPORTED;
  if (nch > 1 && (!ws || ws_bytes < dsv4sa_topk_workspace_size(T, n_max, k) || !aligned(ws, 16)))
    return DSV4SA_ERR_WORKSPACE;
  const dsv4sa::TopkPrefetch pf{kv_pool, kv_page_table, kv_pt_stride, q_seq};
  return dsv4sa::launch_topk(logits, logits_stride, n_vis, T, n_max, k, idx, idx_stride, ws, ws_bytes, stream, &pf);
}

DSV4SA_API int dsv4sa_window_indices(const int32_t* pos, int32_t T, int32_t window, int32_t ring, int32_t* idx_w,
                                     int32_t idx_stride, cudaStream_t stream) {
  if (T < 0 || window < 0 || ring < 0 || idx_stride < window) return DSV4SA_ERR_INVALID_ARG;
  if (T == 0 || window == 0) return DSV4SA_OK;
  if (!pos || !idx_w) return DSV4SA_ERR_INVALID_ARG;
  return dsv4sa::launch_window_indices(pos, T, window, ring, idx_w, idx_stride, stream);
}

DSV4SA_API int dsv4sa_compress_indices(const int32_t* n_vis, int32_t T, int32_t kc, int32_t* idx,
                                       int32_t idx_stride, cudaStream_t stream) {
  if (T < 0 || kc < 0 || idx_stride < kc) return DSV4SA_ERR_INVALID_ARG;
  if (T == 0 || kc == 0) return DSV4SA_OK;
  if (!n_vis || !idx) return DSV4SA_ERR_INVALID_ARG;
  return dsv4sa::launch_compress_indices(n_vis, T, kc, idx, idx_stride, stream);
}

DSV4SA_API size_t dsv4sa_attn_workspace_size(int32_t mode, int32_t T, int32_t H, int32_t kc, int32_t kw) {
  if (T <= 0 || H <= 0 || kc < 0 || kw < 0) return 0;
  const int32_t ns = dsv4sa::attn_splits(mode, kc, kw);
  if (ns <= 1) return 0;
  return static_cast<size_t>(T) * ns * H * (512 + 2) * sizeof(float);
}

DSV4SA_API int dsv4sa_attn_plan(int32_t mode, int32_t T, int32_t H, int32_t kc, int32_t kw, int32_t* nsplit,
                                int32_t* rows_per_split, int32_t* launches) {
  if (T < 0 || H < 1 || H > DSV4SA_MAX_HEADS || kc < 0 || kw < 0) return DSV4SA_ERR_INVALID_ARG;
  if (mode != DSV4SA_ATTN_DECODE && mode != DSV4SA_ATTN_PREFILL) return DSV4SA_ERR_INVALID_ARG;
  return dsv4sa::attn_plan(mode, T, H, kc, kw, nsplit, rows_per_split, launches);
}

static int attn_validate(int32_t mode, const dsv4sa_attn_args* a) {
  if (!a) return DSV4SA_ERR_INVALID_ARG;
  if (a->T < 0 || a->kc < 0 || a->kw < 0) return DSV4SA_ERR_INVALID_ARG;
  if (a->H < 1 || a->H > DSV4SA_MAX_HEADS) return DSV4SA_ERR_UNSUPPORTED;
  if (a->kc > DSV4SA_MAX_TOPK || a->kw > 1024) return DSV4SA_ERR_UNSUPPORTED;
  if (a->T == 0) return DSV4SA_OK;
  if (!a->q || !a->attn_sink || !a->q_seq || !a->out) return DSV4SA_ERR_INVALID_ARG;
  if (!aligned(a->q, 16) || !aligned(a->out, 16)) return DSV4SA_ERR_INVALID_ARG;
  if (a->kc > 0) {
    if (!pool_ok(a->comp, DSV4SA_POOL_KV) || !a->comp_pt || !a->idx_c) return DSV4SA_ERR_INVALID_ARG;
    if (a->idx_c_stride < a->kc || a->comp_pt_stride < 1) return DSV4SA_ERR_INVALID_ARG;
  }
  if (a->kw > 0) {
    if (!pool_ok(a->win, DSV4SA_POOL_KV) || !a->win_pt || (!a->idx_w && !a->win_pos)) return DSV4SA_ERR_INVALID_ARG;
    if ((a->idx_w && a->idx_w_stride < a->kw) || a->win_pt_stride < 1 || a->win_ring < 0) return DSV4SA_ERR_INVALID_ARG;
  }
  if (a->rope_cs && (!a->rope_pos || a->rope_rows < 1 || !aligned(a->rope_cs, 16))) return DSV4SA_ERR_INVALID_ARG;
  const size_t need = dsv4sa_attn_workspace_size(mode, a->T, a->H, a->kc, a->kw);
  if (need > 0 && (!a->ws || a->ws_bytes < need || !aligned(a->ws, 16))) return DSV4SA_ERR_WORKSPACE;
  return DSV4SA_OK;
}

static int attn_common(int32_t mode, const dsv4sa_attn_args* a, cudaStream_t stream) {
  const int rc = attn_validate(mode, a);
  if (rc != DSV4SA_OK || a->T == 0) return rc;
  return dsv4sa::launch_sparse_attn(mode, a, stream);
}

DSV4SA_API int dsv4sa_sparse_attn_decode(const dsv4sa_attn_args* a, cudaStream_t stream) {
  return attn_common(DSV4SA_ATTN_DECODE, a, stream);
}

DSV4SA_API int dsv4sa_sparse_attn_prefill(const dsv4sa_attn_args* a, cudaStream_t stream) {
  return attn_common(DSV4SA_ATTN_PREFILL, a, stream);
}

DSV4SA_API int dsv4sa_topk_sparse_attn_decode(const dsv4sa_attn_args* a, const float* logits, int64_t logits_stride,
                                              const int32_t* n_vis, int32_t n_max, int32_t k, void* topk_ws,
                                              size_t topk_ws_bytes, cudaStream_t stream) {
  const int rc = attn_validate(DSV4SA_ATTN_DECODE, a);
  if (rc != DSV4SA_OK || a->T == 0) return rc;
  if (n_max < 0 || logits_stride < 0) return DSV4SA_ERR_INVALID_ARG;
  if (k < 1 || k > DSV4SA_MAX_TOPK) return DSV4SA_ERR_UNSUPPORTED;
  if (k != a->kc || a->idx_c_stride < k) return DSV4SA_ERR_INVALID_ARG;
  if (!n_vis || (n_max > 0 && !logits)) return DSV4SA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(n_max) > logits_stride && n_max > 0) return DSV4SA_ERR_INVALID_ARG;
  int32_t chunk, nch;
  dsv4sa::topk_plan(n_max, k, &chunk, &nch);
  if (nch == 0) return DSV4SA_ERR_UNSUPPORTED;
  if (nch > 1 && (!topk_ws || topk_ws_bytes < dsv4sa_topk_workspace_size(a->T, n_max, k) || !aligned(topk_ws, 16)))
    return DSV4SA_ERR_WORKSPACE;
  return dsv4sa::launch_topk_sparse_attn(a, logits, logits_stride, n_vis, n_max, k, topk_ws, topk_ws_bytes, stream);
}

DSV4SA_API int dsv4sa_cache_write(const dsv4sa_pool_desc* pool, const int32_t* page_table, int32_t pt_stride,
                                  const int32_t* row_seq, const int32_t* row_entry, const void* rows, int32_t n,
                                  cudaStream_t stream) {
  if (n < 0 || pt_stride < 1) return DSV4SA_ERR_INVALID_ARG;
  if (!pool_ok(pool, DSV4SA_POOL_KV) && !pool_ok(pool, DSV4SA_POOL_IDXK) && !pool_ok(pool, DSV4SA_POOL_IDXK_FP4))
    return DSV4SA_ERR_INVALID_ARG;
  if (n == 0) return DSV4SA_OK;
  if (!page_table || !row_seq || !row_entry || !rows || !aligned(rows, 16)) return DSV4SA_ERR_INVALID_ARG;
  return dsv4sa::launch_cache_write(pool, page_table, pt_stride, row_seq, row_entry, rows, n, false, stream);
}

DSV4SA_API int dsv4sa_cache_write_rotated(const dsv4sa_pool_desc* pool, const int32_t* page_table,
                                          int32_t pt_stride, const int32_t* row_seq, const int32_t* row_entry,
                                          const void* rows, int32_t n, cudaStream_t stream) {
  if (n < 0 || pt_stride < 1 || !pool_ok(pool, DSV4SA_POOL_IDXK_FP4)) return DSV4SA_ERR_INVALID_ARG;
  if (n == 0) return DSV4SA_OK;
  if (!page_table || !row_seq || !row_entry || !rows || !aligned(rows, 16)) return DSV4SA_ERR_INVALID_ARG;
  return dsv4sa::launch_cache_write(pool, page_table, pt_stride, row_seq, row_entry, rows, n, true, stream);
}

DSV4SA_API int dsv4sa_compress_windows(const void* kv, const void* score, int64_t tok_stride, int64_t n_tok,
                                       const int32_t* first_tok, const int32_t* prev_tok, const int32_t* position,
                                       int32_t n, int32_t ratio, int32_t overlap, const float* ape,
                                       const float* norm_w, float eps, const float* rope_cs, int32_t rope_rows,
                                       void* out, cudaStream_t stream) {
  if (n < 0 || n_tok < 0 || rope_rows < 1 || !(eps >= 0.f)) return DSV4SA_ERR_INVALID_ARG;
  if (overlap != 0 && overlap != 1) return DSV4SA_ERR_INVALID_ARG;
  if (overlap ? ratio != 4 : (ratio < 1 || ratio > 1024)) return DSV4SA_ERR_UNSUPPORTED;
  const int64_t width = overlap ? 1024 : 512;
  if (tok_stride < width || tok_stride % 8 != 0) return DSV4SA_ERR_INVALID_ARG;
  if (n == 0) return DSV4SA_OK;
  if (!kv || !score || !first_tok || (overlap && !prev_tok) || !position || !ape || !norm_w || !rope_cs || !out)
    return DSV4SA_ERR_INVALID_ARG;
  if (!aligned(kv, 16) || !aligned(score, 16) || !aligned(ape, 16) || !aligned(norm_w, 16) || !aligned(rope_cs, 16) ||
      !aligned(out, 16))
    return DSV4SA_ERR_INVALID_ARG;
  return dsv4sa::launch_compress_windows(kv, score, tok_stride, n_tok, first_tok, prev_tok, position, n, ratio,
                                         overlap, ape, norm_w, eps, rope_cs, rope_rows, out, stream);
}

DSV4SA_API int dsv4sa_compress_online_c128(const void* kv, const void* score, int64_t tok_stride, int32_t T,
                                           const int32_t* state_idx, float* state, int32_t* state_count,
                                           int32_t slots, const int32_t* position, const float* ape,
                                           const float* norm_w, float eps, const float* rope_cs, int32_t rope_rows,
                                           void* out, int32_t* done, cudaStream_t stream) {
  if (T < 0 || slots < 1 || rope_rows < 1 || !(eps >= 0.f)) return DSV4SA_ERR_INVALID_ARG;
  if (tok_stride < 512 || tok_stride % 8 != 0) return DSV4SA_ERR_INVALID_ARG;
  if (T == 0) return DSV4SA_OK;
  if (!kv || !score || !state_idx || !state || !state_count || !position || !ape || !norm_w || !rope_cs || !out ||
      !done)
    return DSV4SA_ERR_INVALID_ARG;
  if (!aligned(kv, 16) || !aligned(score, 16) || !aligned(state, 16) || !aligned(ape, 16) || !aligned(norm_w, 16) ||
      !aligned(rope_cs, 16) || !aligned(out, 16))
    return DSV4SA_ERR_INVALID_ARG;
  return dsv4sa::launch_compress_online(kv, score, tok_stride, state_idx, state, state_count, slots, position, T,
                                        ape, norm_w, eps, rope_cs, rope_rows, out, done, stream);
}

DSV4SA_API int dsv4sa_copy_async(void* dst, const void* src, size_t bytes, cudaStream_t stream) {
  if (bytes == 0) return DSV4SA_OK;
  if (!dst || !src || bytes % 16 != 0 || !aligned(dst, 16) || !aligned(src, 16)) return DSV4SA_ERR_INVALID_ARG;
  return dsv4sa::launch_copy(dst, src, static_cast<int64_t>(bytes), stream);
}

DSV4SA_API int dsv4sa_copy_async_background(void* dst, const void* src, size_t bytes, cudaStream_t stream) {
  if (bytes == 0) return DSV4SA_OK;
  if (!dst || !src || bytes % 16 != 0 || !aligned(dst, 16) || !aligned(src, 16)) return DSV4SA_ERR_INVALID_ARG;
  return dsv4sa::launch_copy_background(dst, src, static_cast<int64_t>(bytes), stream);
}

DSV4SA_API int dsv4sa_selftest_wait_timeout(int32_t* result, cudaStream_t stream) {
  if (!result || !aligned(result, 4)) return DSV4SA_ERR_INVALID_ARG;
  return dsv4sa::launch_selftest_wait_timeout(result, stream);
}

DSV4SA_API int dsv4sa_check_errors(cudaStream_t stream, uint32_t* bits_out) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return DSV4SA_ERR_CUDA;
  const uint32_t bits = dsv4sa::read_error_word_indexer(stream, true) | dsv4sa::read_error_word_topk(stream, true) |
                        dsv4sa::read_error_word_attn(stream, true) | dsv4sa::read_error_word_attn_decode(stream, true) |
                        dsv4sa::read_error_word_writer(stream, true) |
                        dsv4sa::read_error_word_compress(stream, true);
  if (cudaGetLastError() != cudaSuccess) return DSV4SA_ERR_CUDA;
  if (bits_out) *bits_out = bits;
  if (bits & 2u) return DSV4SA_ERR_DEVICE_TIMEOUT;
  if (bits & 1u) return DSV4SA_ERR_INDEX_OOB;
  return DSV4SA_OK;
}

}  // extern "C"
