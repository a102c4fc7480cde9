// topk.cu -- exact per-query top-k over the indexer logits.
//
// idx[t, :] = the k entries s < n_vis[t] with the largest logit, ascending,
// -1 padded; all visible entries when n_vis[t] <= k ("DeepSeek-V4 全面解读"
// §2.10 Indexer step 9; "DeepSeek-V4 in SGLang" 概念3 / 算法2: top-512, no
// top-k below 512 compressed entries).  Among equal scores the lower entry
// index wins; -0.0 equals +0.0 and NaN ranks below every number.  A row whose
// n_vis is negative is not routed through top-k and is left untouched.
//
// Scores are mapped to order-preserving 32-bit keys, so the selection is exact
// integer work.  A block-wide radix select (11 + 11 + 10 bits, shared-memory
// histograms) finds the k-th largest key and how many of its ties to take; an
// order-preserving compaction (warp ballots + one block scan per round) then
// emits the selected entries in ascending order.
//
// Long rows are cut into chunks: stage 1 (one CTA per chunk) keeps each
// chunk's exact top-k as (key, index) candidates in the workspace -- every
// member of the row's top-k is in its chunk's top-k under the same order --
// and stage 2 (one CTA per row) selects the final k among the candidates,
// which are already in ascending index order.  Rows that fit in one chunk are
// finished by stage 1 alone.
#include "common.cuh"
#include "dsv4sa_internal.h"

namespace dsv4sa {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMinChunk = 4096;
constexpr int kMaxChunk = 16384;
constexpr int kMaxCand = 32768;

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t b = __float_as_uint(f);
  if ((b & 0x7FFFFFFFu) > 0x7F800000u) return 0u;  // NaN: lowest
  if ((b & 0x7FFFFFFFu) == 0u) b = 0u;             // -0 == +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Block-wide exclusive scan of one int per thread; returns the block total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_buf, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_buf[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kWarps ? warp_buf[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kWarps) warp_buf[lane] = w;  // inclusive warp prefix
  }
  __syncthreads();
  total = warp_buf[kWarps - 1];
  const int before = warp == 0 ? 0 : warp_buf[warp - 1];
  __syncthreads();
  return before + x - v;
}

struct SelectScratch {
  uint32_t hist[2048];
  int warp_buf[kWarps];
  int found_bin;
  int found_above;
};

// Radix select over keys[0, n): the k-th largest key and the number of its
// ties (lowest indices first) that belong to the top k.  Requires n > k >= 1.
__device__ void radix_select(const uint32_t* keys, int n, int k, SelectScratch& sc, uint32_t& kth, int& need) {
  const int tid = threadIdx.x;
  uint32_t prefix = 0, pmask = 0;
  int rem = k;
  const int shifts[3] = {21, 10, 0};
  const int widths[3] = {11, 11, 10};
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = shifts[pass];
    const int nbins = 1 << widths[pass];
    const uint32_t dmask = static_cast<uint32_t>(nbins - 1);
    for (int b = tid; b < nbins; b += kThreads) sc.hist[b] = 0u;
    __syncthreads();
    for (int i = tid; i < n; i += kThreads) {
      const uint32_t key = keys[i];
      if ((key & pmask) == prefix) atomicAdd(&sc.hist[(key >> shift) & dmask], 1u);
    }
    __syncthreads();
    // thread tid owns bins [nbins - (tid + 1) * per, nbins - tid * per), highest first
    const int per = nbins / kThreads;
    int cnt[4];
    int local = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      cnt[q] = 0;
      if (q < per) {
        cnt[q] = static_cast<int>(sc.hist[nbins - 1 - (tid * per + q)]);
        local += cnt[q];
      }
    }
    int total;
    const int above = block_exclusive_scan(local, sc.warp_buf, total);
    if (above < rem && above + local >= rem) {
      int acc = above;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (q < per) {
          if (acc + cnt[q] >= rem) {
            sc.found_bin = nbins - 1 - (tid * per + q);
            sc.found_above = acc;
            break;
          }
          acc += cnt[q];
        }
      }
    }
    __syncthreads();
    const int bin = sc.found_bin;
    rem -= sc.found_above;
    prefix |= static_cast<uint32_t>(bin) << shift;
    pmask |= dmask << shift;
    __syncthreads();
  }
  kth = prefix;
  need = rem;
}

// Emit, in ascending position, every i in [0, n) with keys[i] > kth plus the
// first `need` positions with keys[i] == kth.  emit(pos, i) is called once per
// selected element with its output rank.
template <class Emit>
__device__ void ordered_compact(const uint32_t* keys, int n, uint32_t kth, int need, SelectScratch& sc, Emit emit) {
  const int tid = threadIdx.x;
  int gt_base = 0, eq_base = 0;
  for (int r0 = 0; r0 < n; r0 += kThreads) {
    const int i = r0 + tid;
    const uint32_t key = i < n ? keys[i] : 0u;
    const bool gt = i < n && key > kth;
    const bool eq = i < n && key == kth;
    // packed (gt count, eq count << 16) prefix over the round
    const int packed = (gt ? 1 : 0) | (eq ? (1 << 16) : 0);
    int total;
    const int before = block_exclusive_scan(packed, sc.warp_buf, total);
    const int gt_before = gt_base + (before & 0xFFFF);
    const int eq_before = eq_base + (before >> 16);
    if (gt || (eq && eq_before < need)) emit(gt_before + min(eq_before, need), i);
    gt_base += total & 0xFFFF;
    eq_base += total >> 16;
  }
}

struct TopkParams {
  const float* logits;
  const int32_t* n_vis;
  int32_t* idx;
  uint32_t* cand_key;   // [T][nchunks][k]
  int32_t* cand_idx;    // [T][nchunks][k]
  int64_t logits_stride;
  int32_t idx_stride;
  int32_t T;
  int32_t n_max;
  int32_t k;
  int32_t chunk;
  int32_t nchunks;      // chunks of a row of length n_max
};

// Visible entries of row t clamped to n_max; -1 marks a row to leave untouched.
__device__ __forceinline__ int clamp_n(const TopkParams& p, int t) {
  const int n = __ldg(p.n_vis + t);
  return n < 0 ? -1 : (n > p.n_max ? p.n_max : n);
}

__global__ void __launch_bounds__(kThreads) topk_chunk_kernel(const TopkParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  SelectScratch& sc = *reinterpret_cast<SelectScratch*>(smem);
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem + sizeof(SelectScratch));
  const int t = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
  const int n = clamp_n(p, t);
  if (n < 0) return;
  int32_t* out = p.idx + static_cast<int64_t>(t) * p.idx_stride;
  if (n <= p.k) {
    if (c == 0)
      for (int j = tid; j < p.k; j += kThreads) out[j] = j < n ? j : -1;
    return;
  }
  const int nch = (n + p.chunk - 1) / p.chunk;
  if (c >= nch) return;
  const int lo = c * p.chunk;
  const int m = min(n, lo + p.chunk) - lo;
  const float* row = p.logits + static_cast<int64_t>(t) * p.logits_stride + lo;
  for (int i = tid; i < m; i += kThreads) keys[i] = order_key(__ldg(row + i));
  __syncthreads();
  const int64_t cbase = (static_cast<int64_t>(t) * p.nchunks + c) * p.k;
  if (nch > 1 && m <= p.k) {
    for (int i = tid; i < m; i += kThreads) {
      p.cand_key[cbase + i] = keys[i];
      p.cand_idx[cbase + i] = lo + i;
    }
    return;
  }
  uint32_t kth;
  int need;
  radix_select(keys, m, p.k, sc, kth, need);
  if (nch == 1) {
    ordered_compact(keys, m, kth, need, sc, [&](int pos, int i) { out[pos] = lo + i; });
  } else {
    ordered_compact(keys, m, kth, need, sc, [&](int pos, int i) {
      p.cand_key[cbase + pos] = keys[i];
      p.cand_idx[cbase + pos] = lo + i;
    });
  }
}

__global__ void __launch_bounds__(kThreads) topk_merge_kernel(const TopkParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  SelectScratch& sc = *reinterpret_cast<SelectScratch*>(smem);
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem + sizeof(SelectScratch));
  const int t = blockIdx.x, tid = threadIdx.x;
  const int n = clamp_n(p, t);
  if (n <= p.k) return;  // includes rows left untouched (n < 0)
  const int nch = (n + p.chunk - 1) / p.chunk;
  if (nch <= 1) return;
  // gather candidates in chunk order (ascending entry index)
  int m = 0;
  for (int c = 0; c < nch; ++c) {
    const int len = min(n, (c + 1) * p.chunk) - c * p.chunk;
    const int cnt = min(len, p.k);
    const uint32_t* src = p.cand_key + (static_cast<int64_t>(t) * p.nchunks + c) * p.k;
    for (int i = tid; i < cnt; i += kThreads) keys[m + i] = src[i];
    m += cnt;
  }
  __syncthreads();
  uint32_t kth;
  int need;
  radix_select(keys, m, p.k, sc, kth, need);
  int32_t* out = p.idx + static_cast<int64_t>(t) * p.idx_stride;
  // candidate position i -> (chunk, offset); chunk offsets are multiples of k except the tail
  ordered_compact(keys, m, kth, need, sc, [&](int pos, int i) {
    int c = 0, off = i;
    for (;; ++c) {
      const int len = min(n, (c + 1) * p.chunk) - c * p.chunk;
      const int cnt = min(len, p.k);
      if (off < cnt) break;
      off -= cnt;
    }
    out[pos] = p.cand_idx[(static_cast<int64_t>(t) * p.nchunks + c) * p.k + off];
  });
}

}  // namespace

void topk_plan(int32_t n_max, int32_t k, int32_t* chunk_len, int32_t* n_chunks) {
  *chunk_len = 0;
  *n_chunks = 0;
  if (k < 1 || k > DSV4SA_MAX_TOPK || n_max < 0) return;
  const int64_t cand_chunks = kMaxCand / k;            // chunks the merge can hold
  int64_t chunk = kMinChunk;
  if (static_cast<int64_t>(n_max) > chunk * cand_chunks)
    chunk = (static_cast<int64_t>(n_max) + cand_chunks - 1) / cand_chunks;
  chunk = (chunk + 511) / 512 * 512;
  if (chunk < k + 1) chunk = (k + 512) / 512 * 512;
  if (chunk > kMaxChunk) return;
  const int64_t nch = n_max <= 0 ? 1 : (n_max + chunk - 1) / chunk;
  if (nch * k > kMaxCand && nch > 1) return;
  *chunk_len = static_cast<int32_t>(chunk);
  *n_chunks = static_cast<int32_t>(nch < 1 ? 1 : nch);
}

int launch_topk(const float* logits, int64_t logits_stride, const int32_t* n_vis, int32_t T, int32_t n_max,
                int32_t k, int32_t* idx, int32_t idx_stride, void* ws, size_t ws_bytes, cudaStream_t stream) {
  int32_t chunk, nch;
  topk_plan(n_max, k, &chunk, &nch);
  if (nch == 0) return DSV4SA_ERR_UNSUPPORTED;
  TopkParams p{};
  p.logits = logits;
  p.n_vis = n_vis;
  p.idx = idx;
  p.logits_stride = logits_stride;
  p.idx_stride = idx_stride;
  p.T = T;
  p.n_max = n_max;
  p.k = k;
  p.chunk = chunk;
  p.nchunks = nch;
  if (nch > 1) {
    const size_t need = static_cast<size_t>(T) * nch * k * 8;
    if (!ws || ws_bytes < need) return DSV4SA_ERR_WORKSPACE;
    p.cand_key = static_cast<uint32_t*>(ws);
    p.cand_idx = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + static_cast<size_t>(T) * nch * k * 4);
  }
  if (T == 0) return DSV4SA_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSV4SA_ERR_CUDA;
  const int smem1 = static_cast<int>(sizeof(SelectScratch)) + chunk * 4;
  if (!smem_attr_once(dev, 8, reinterpret_cast<const void*>(topk_chunk_kernel), smem1)) return DSV4SA_ERR_CUDA;
  topk_chunk_kernel<<<dim3(nch, T), kThreads, smem1, stream>>>(p);
  if (cudaGetLastError() != cudaSuccess) return DSV4SA_ERR_CUDA;
  if (nch > 1) {
    const int smem2 = static_cast<int>(sizeof(SelectScratch)) + nch * k * 4;
    if (!smem_attr_once(dev, 9, reinterpret_cast<const void*>(topk_merge_kernel), smem2)) return DSV4SA_ERR_CUDA;
    topk_merge_kernel<<<T, kThreads, smem2, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return DSV4SA_ERR_CUDA;
  }
  return DSV4SA_OK;
}

uint32_t read_error_word_topk(cudaStream_t stream, bool clear) {
  uint32_t v = 0;
  cudaMemcpyFromSymbolAsync(&v, g_err_word, sizeof(v), 0, cudaMemcpyDeviceToHost, stream);
  cudaStreamSynchronize(stream);
  if (clear && v) {
    const uint32_t z = 0;
    cudaMemcpyToSymbolAsync(g_err_word, &z, sizeof(z), 0, cudaMemcpyHostToDevice, stream);
    cudaStreamSynchronize(stream);
  }
  return v;
}

}  // namespace dsv4sa
