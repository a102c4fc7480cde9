// index.cu -- index assembly for sparse attention ("DeepSeek-V4 全面解读" §2.8:
// get_window_topk_idxs, get_compress_topk_idxs; §2.11 step 4: the window and
// compressed index lists are both handed to one sparse_attn call).
#include "common.cuh"
#include "dsv4sa_internal.h"

namespace dsv4sa {
namespace {

// idx_w[t, j] = p = pos[t] - window + 1 + j (current token included), -1 if p < 0;
// p % ring when ring > 0 (slot of a circular window cache).
__global__ void window_indices_kernel(const int32_t* __restrict__ pos, int32_t T, int32_t window, int32_t ring,
                                      int32_t* __restrict__ idx, int32_t stride) {
  griddep_launch();
  griddep_wait();
  const int64_t total = static_cast<int64_t>(T) * window;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = i / window;
    const int32_t j = static_cast<int32_t>(i - t * window);
    const int64_t p = static_cast<int64_t>(__ldg(pos + t)) - window + 1 + j;
    idx[t * stride + j] = p < 0 ? -1 : static_cast<int32_t>(ring > 0 ? p % ring : p);
  }
}

// idx[t, j] = j for j < min(n_vis[t], kc), else -1.
__global__ void compress_indices_kernel(const int32_t* __restrict__ n_vis, int32_t T, int32_t kc,
                                        int32_t* __restrict__ idx, int32_t stride) {
  griddep_launch();
  griddep_wait();
  const int64_t total = static_cast<int64_t>(T) * kc;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = i / kc;
    const int32_t j = static_cast<int32_t>(i - t * kc);
    idx[t * stride + j] = j < __ldg(n_vis + t) ? j : -1;
  }
}

int grid_for(int64_t total) {
  const int64_t blocks = (total + 255) / 256;
  return static_cast<int>(blocks < 4096 ? (blocks < 1 ? 1 : blocks) : 4096);
}

// Copy of a buffer the device can address (device memory, or pinned host
// memory mapped into the address space) by the SMs: 16-byte loads, four per
// thread in flight before their stores, grid-stride.  For step-sized inputs it
// starts sooner than a copy-engine transfer.  It does not trigger its
// dependents early: a following kernel that reads the destination before its
// own dependency wait (the attention's early window) starts only after the copy.
__global__ void __launch_bounds__(256) copy_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src,
                                                   int64_t n16) {
  griddep_wait();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (i + u * stride < n16) v[u] = src[i + u * stride];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (i + u * stride < n16) dst[i + u * stride] = v[u];
  }
}

// The same copy with one warp per SM and at most 32 registers a thread
// (__maxnreg__(32)): it fits beside a kernel that leaves one warp's
// worth of registers free on every SM (the indexer: 384 threads x 168), so the
// two run at the same time instead of one waiting for the other's SMs.
__global__ void __maxnreg__(32) copy_narrow_kernel(uint4* __restrict__ dst,
                                                   const uint4* __restrict__ src, int64_t n16) {
  griddep_wait();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (i + u * stride < n16) v[u] = src[i + u * stride];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (i + u * stride < n16) dst[i + u * stride] = v[u];
  }
}

}  // namespace

int launch_copy_background(void* dst, const void* src, int64_t bytes, cudaStream_t stream) {
  const int64_t n16 = bytes / 16;
  if (n16 == 0) return DSV4SA_OK;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSV4SA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return DSV4SA_ERR_CUDA;
  const int64_t want = (n16 + 4 * 32 - 1) / (4 * 32);
  const int64_t grid = want < static_cast<int64_t>(sms) ? want : static_cast<int64_t>(sms);
  return launch_pdl(copy_narrow_kernel, dim3(static_cast<unsigned>(grid)), dim3(32), 0, stream,
                    static_cast<uint4*>(dst), static_cast<const uint4*>(src), n16) == cudaSuccess
             ? DSV4SA_OK
             : DSV4SA_ERR_CUDA;
}

int launch_copy(void* dst, const void* src, int64_t bytes, cudaStream_t stream) {
  const int64_t n16 = bytes / 16;
  if (n16 == 0) return DSV4SA_OK;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSV4SA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return DSV4SA_ERR_CUDA;
  const int64_t want = (n16 + 4 * 256 - 1) / (4 * 256);
  const int64_t grid = want < static_cast<int64_t>(sms) * 4 ? want : static_cast<int64_t>(sms) * 4;
  return launch_pdl(copy_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, stream, static_cast<uint4*>(dst),
                    static_cast<const uint4*>(src), n16) == cudaSuccess
             ? DSV4SA_OK
             : DSV4SA_ERR_CUDA;
}

int launch_window_indices(const int32_t* pos, int32_t T, int32_t window, int32_t ring, int32_t* idx_w,
                          int32_t idx_stride, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(T) * window;
  if (total == 0) return DSV4SA_OK;
  return launch_pdl(window_indices_kernel, dim3(grid_for(total)), dim3(256), 0, stream, pos, T, window, ring, idx_w,
                    idx_stride) == cudaSuccess
             ? DSV4SA_OK
             : DSV4SA_ERR_CUDA;
}

int launch_compress_indices(const int32_t* n_vis, int32_t T, int32_t kc, int32_t* idx, int32_t idx_stride,
                            cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(T) * kc;
  if (total == 0) return DSV4SA_OK;
  return launch_pdl(compress_indices_kernel, dim3(grid_for(total)), dim3(256), 0, stream, n_vis, T, kc, idx,
                    idx_stride) == cudaSuccess
             ? DSV4SA_OK
             : DSV4SA_ERR_CUDA;
}

}  // namespace dsv4sa
