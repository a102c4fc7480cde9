// step.cpp -- one decode serving step as a CUDA graph owned by the library.
//
// The step is the path's calls in their serving order: the packed inputs from
// pinned host memory (the indexer's part, then the attention's part on a second
// stream that runs beside the indexer), indexer logits, top-k, decode
// attention ("DeepSeek-V4 全面解读" §2.10 steps 6-9 and §2.11 step 7; "DeepSeek-V4
// in SGLang" 算法2: paged MQA logits, top-512, sparse attention).  It is run
// once eagerly, so per-device set-up (kernel attributes, driver entry points)
// happens outside the capture, then captured from the launch stream; the
// programmatic-dependent launches of the kernels become graph edges.
#include <cstdint>
#include <new>

#include <cuda_runtime_api.h>

#include "../../include/dsv4sa.h"

struct dsv4sa_step {
  dsv4sa_step_desc desc;
  dsv4sa_attn_args attn;      // a copy: the desc's pointer may not outlive create
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr;
  cudaEvent_t join = nullptr;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
};

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The step's calls on `stream` (and the second stream).
int run_body(dsv4sa_step* st, cudaStream_t stream) {
  const dsv4sa_step_desc& d = st->desc;
  int rc = dsv4sa_copy_async(d.dev_in, d.host_in, d.in_split, stream);
  if (rc != DSV4SA_OK) return rc;
  if (cudaEventRecord(st->fork, stream) != cudaSuccess) return DSV4SA_ERR_CUDA;
  if (cudaStreamWaitEvent(st->side, st->fork, 0) != cudaSuccess) return DSV4SA_ERR_CUDA;
  rc = dsv4sa_copy_async_background(static_cast<uint8_t*>(d.dev_in) + d.in_split,
                                    static_cast<const uint8_t*>(d.host_in) + d.in_split, d.in_bytes - d.in_split,
                                    st->side);
  if (rc != DSV4SA_OK) return rc;
  if (cudaEventRecord(st->join, st->side) != cudaSuccess) return DSV4SA_ERR_CUDA;
  rc = dsv4sa_indexer_logits(d.kpool, d.page_table, d.pt_stride, d.q_seq, d.n_vis, d.q_fp8, d.q_scale, d.w, d.T,
                             d.Hi, d.n_max, d.logits, d.logits_stride, stream);
  if (rc != DSV4SA_OK) return rc;
  // the top-k prefetches the attention's rows: its page table and q_seq come with the second copy
  if (cudaStreamWaitEvent(stream, st->join, 0) != cudaSuccess) return DSV4SA_ERR_CUDA;
  const dsv4sa_attn_args& a = st->attn;
  rc = a.kc > 0 && a.comp
           ? dsv4sa_topk_prefetch(d.logits, d.logits_stride, d.n_vis, d.T, d.n_max, d.k, d.idx, d.idx_stride,
                                  d.topk_ws, d.topk_ws_bytes, a.comp, a.comp_pt, a.comp_pt_stride, a.q_seq, stream)
           : dsv4sa_topk(d.logits, d.logits_stride, d.n_vis, d.T, d.n_max, d.k, d.idx, d.idx_stride, d.topk_ws,
                         d.topk_ws_bytes, stream);
  if (rc != DSV4SA_OK) return rc;
  return dsv4sa_sparse_attn_decode(&st->attn, stream);
}

void release(dsv4sa_step* st) {
  if (st->exec) cudaGraphExecDestroy(st->exec);
  if (st->graph) cudaGraphDestroy(st->graph);
  if (st->join) cudaEventDestroy(st->join);
  if (st->fork) cudaEventDestroy(st->fork);
  if (st->side) cudaStreamDestroy(st->side);
  delete st;
}

}  // namespace

extern "C" {

DSV4SA_API int dsv4sa_step_create(dsv4sa_step** out, const dsv4sa_step_desc* desc, cudaStream_t stream) {
  if (!out || !desc || !desc->attn || !desc->host_in || !desc->dev_in) return DSV4SA_ERR_INVALID_ARG;
  if (desc->in_bytes == 0 || desc->in_bytes % 16 != 0 || desc->in_split % 16 != 0 ||
      desc->in_split > desc->in_bytes || !aligned16(desc->host_in) || !aligned16(desc->dev_in))
    return DSV4SA_ERR_INVALID_ARG;
  if (!stream) return DSV4SA_ERR_INVALID_ARG;   // the legacy default stream cannot be captured
  dsv4sa_step* st = new (std::nothrow) dsv4sa_step;
  if (!st) return DSV4SA_ERR_CUDA;
  st->desc = *desc;
  st->attn = *desc->attn;
  st->attn.idx_c = desc->idx;
  st->attn.idx_c_stride = desc->idx_stride;
  st->desc.attn = &st->attn;
  if (cudaStreamCreateWithFlags(&st->side, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&st->fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&st->join, cudaEventDisableTiming) != cudaSuccess) {
    release(st);
    return DSV4SA_ERR_CUDA;
  }
  int rc = run_body(st, stream);   // eager: set-up outside the capture, arguments validated
  if (rc == DSV4SA_OK && cudaStreamSynchronize(stream) != cudaSuccess) rc = DSV4SA_ERR_CUDA;
  if (rc != DSV4SA_OK) {
    release(st);
    return rc;
  }
  if (cudaStreamBeginCapture(stream, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    release(st);
    return DSV4SA_ERR_CUDA;
  }
  rc = run_body(st, stream);
  cudaGraph_t g = nullptr;
  const cudaError_t ce = cudaStreamEndCapture(stream, &g);   // always ends the capture
  st->graph = g;
  if (rc == DSV4SA_OK && (ce != cudaSuccess || !g)) rc = DSV4SA_ERR_CUDA;
  if (rc == DSV4SA_OK && cudaGraphInstantiate(&st->exec, g, 0) != cudaSuccess) rc = DSV4SA_ERR_CUDA;
  if (rc != DSV4SA_OK) {
    release(st);
    return rc;
  }
  *out = st;
  return DSV4SA_OK;
}

DSV4SA_API int dsv4sa_step_launch(dsv4sa_step* step, cudaStream_t stream) {
  if (!step || !step->exec) return DSV4SA_ERR_INVALID_ARG;
  return cudaGraphLaunch(step->exec, stream) == cudaSuccess ? DSV4SA_OK : DSV4SA_ERR_CUDA;
}

DSV4SA_API int dsv4sa_step_destroy(dsv4sa_step* step) {
  if (!step) return DSV4SA_ERR_INVALID_ARG;
  release(step);
  return DSV4SA_OK;
}

}  // extern "C"
