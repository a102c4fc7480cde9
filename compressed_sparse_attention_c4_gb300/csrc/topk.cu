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
// integer work.  One 256-thread CTA selects from up to 4096 keys held in
// registers; thread t owns positions t, t + NT, t + 2 NT, ... (NT threads) so
// every load is coalesced:
//   1. a block min/max of the keys fixes the bits all keys share, so the first
//      radix digit starts at the highest bit that varies (indexer logits sit
//      in a narrow range, where the top bits of the key are nearly constant);
//   2. radix passes of 11 bits: a 2048-bin shared-memory histogram (the
//      adaptive first digit spreads the keys, so the atomics rarely collide),
//      then a block scan from the top bin finds the digit of the k-th largest key;
//   3. the output rank of every selected entry is the number of selected
//      entries at lower positions: warp ballots count them per (round, warp),
//      one block scan over those (round, warp) counts gives the offsets,
//      so entries come out in ascending order with the lowest-index ties first.
// Longer rows are cut into chunks: stage 1 keeps each chunk's exact top-k as
// (key, index) candidates -- every member of the row's top-k is in its chunk's
// top-k under the same order -- and stage 2 selects the final k among the
// candidates, which are already in ascending index order.
#include <mutex>

#include "common.cuh"
#include "dsv4sa_internal.h"

namespace dsv4sa {
namespace {

constexpr int kChunkThreads = 256;             // stage 1: one CTA per chunk of <= 4096 keys
constexpr int kPer = 16;                       // keys per thread
constexpr int kChunk = kChunkThreads * kPer;   // 4096
constexpr int kMergeThreads = 1024;            // stage 2: one CTA per row
constexpr int kMaxCand = 32768;                // candidates the merge holds (32 per thread)
constexpr int kMaxWarps = 32;

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t b = __float_as_uint(f);
  if ((b & 0x7FFFFFFFu) > 0x7F800000u) return 0u;  // NaN: lowest
  if ((b & 0x7FFFFFFFu) == 0u) b = 0u;             // -0 == +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

struct Scratch {
  uint32_t hist[2048];
  int warp_buf[kMaxWarps];
  uint32_t red_min[kMaxWarps];
  uint32_t red_max[kMaxWarps];
  int found_bin;
  int found_above;
};

// Exclusive block scan of one int per thread (NT threads); returns the total.
template <int NT>
__device__ __forceinline__ int block_scan(int v, int* warp_buf, int& total) {
  constexpr int kWarps = NT / 32;
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
    if (lane < kWarps) warp_buf[lane] = w;
  }
  __syncthreads();
  total = warp_buf[kWarps - 1];
  const int before = warp == 0 ? 0 : warp_buf[warp - 1];
  __syncthreads();
  return before + x - v;
}

// Select among the valid keys of all threads (key[i] valid when valid_mask bit i
// is set; at least k + 1 valid keys overall, k >= 1).  Returns the k-th largest
// key and how many of its ties (lowest positions first) belong to the top k.
template <int NT, int P>
__device__ void radix_select(const uint32_t (&key)[P], uint32_t valid_mask, int k, Scratch& sc, uint32_t& kth,
                             int& need) {
  constexpr int kWarps = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // 1. min / max of the valid keys
  uint32_t mn = 0xFFFFFFFFu, mx = 0u;
#pragma unroll
  for (int i = 0; i < P; ++i) {
    if (valid_mask >> i & 1u) {
      mn = min(mn, key[i]);
      mx = max(mx, key[i]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  if (lane == 0) {
    sc.red_min[warp] = mn;
    sc.red_max[warp] = mx;
  }
  __syncthreads();
  mn = lane < kWarps ? sc.red_min[lane] : 0xFFFFFFFFu;
  mx = lane < kWarps ? sc.red_max[lane] : 0u;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  const uint32_t diff = mn ^ mx;
  if (diff == 0u) {  // every valid key equal
    kth = mx;
    need = k;
    return;
  }
  int hi = 31 - __clz(diff);                 // highest varying bit
  uint32_t pmask = hi == 31 ? 0u : (0xFFFFFFFFu << (hi + 1));
  uint32_t prefix = mx & pmask;
  int rem = k;
  // 2. radix passes over bits [lo, hi]
  while (hi >= 0) {
    const int lo = hi - 10 > 0 ? hi - 10 : 0;
    const uint32_t dmask = (2u << (hi - lo)) - 1u;
    for (int b = tid; b < 2048; b += NT) sc.hist[b] = 0u;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < P; ++i) {
      if ((valid_mask >> i & 1u) && (key[i] & pmask) == prefix) atomicAdd(&sc.hist[(key[i] >> lo) & dmask], 1u);
    }
    __syncthreads();
    // thread tid owns bins [2048 - (tid + 1) B, 2048 - tid B), highest first
    constexpr int B = 2048 / NT;
    int cb[B];
    int local = 0;
#pragma unroll
    for (int q = 0; q < B; ++q) {
      cb[q] = static_cast<int>(sc.hist[2047 - tid * B - q]);
      local += cb[q];
    }
    int total;
    const int above = block_scan<NT>(local, sc.warp_buf, total);
    if (above < rem && above + local >= rem) {
      int acc = above;
#pragma unroll
      for (int q = 0; q < B; ++q) {
        if (acc < rem && acc + cb[q] >= rem) {
          sc.found_bin = 2047 - tid * B - q;
          sc.found_above = acc;
        }
        acc += cb[q];
      }
    }
    __syncthreads();
    rem -= sc.found_above;
    prefix |= static_cast<uint32_t>(sc.found_bin) << lo;
    pmask |= dmask << lo;
    hi = lo - 1;
    __syncthreads();
  }
  kth = prefix;
  need = rem;
}

// Output ranks.  Thread t holds the keys of positions q * blockDim + t
// (round q); an entry is selected if key > kth, or key == kth and fewer than
// `need` equal keys sit at lower positions.  emit(rank, q) is called once per
// selected entry, rank = number of selected entries at lower positions.
template <int NT, int P, class Emit>
__device__ void ordered_emit(const uint32_t (&key)[P], uint32_t valid_mask, uint32_t kth, int need, Scratch& sc,
                             uint32_t* cnt /* [P][NT / 32] */, Emit emit) {
  constexpr int kWarps = NT / 32;
  static_assert(P * kWarps <= NT, "one scan entry per thread");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int q = 0; q < P; ++q) {
    const bool ok = valid_mask >> q & 1u;
    const uint32_t bg = __ballot_sync(0xffffffffu, ok && key[q] > kth);
    const uint32_t be = __ballot_sync(0xffffffffu, ok && key[q] == kth);
    if (lane == 0) cnt[q * kWarps + warp] = __popc(bg) | (__popc(be) << 16);
  }
  __syncthreads();
  // exclusive scan of the packed (greater, equal) counts in (round, warp) order;
  // both totals stay below 2^16
  int total;
  const int mine = tid < P * kWarps ? static_cast<int>(cnt[tid]) : 0;
  const int before = block_scan<NT>(mine, sc.warp_buf, total);
  if (tid < P * kWarps) cnt[tid] = static_cast<uint32_t>(before);
  __syncthreads();
  const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
  for (int q = 0; q < P; ++q) {
    const bool ok = valid_mask >> q & 1u;
    const bool gt = ok && key[q] > kth, eq = ok && key[q] == kth;
    const uint32_t bg = __ballot_sync(0xffffffffu, gt);
    const uint32_t be = __ballot_sync(0xffffffffu, eq);
    const uint32_t off = cnt[q * kWarps + warp];
    const int gt_before = static_cast<int>(off & 0xFFFFu) + __popc(bg & lt);
    const int eq_before = static_cast<int>(off >> 16) + __popc(be & lt);
    if (gt) emit(gt_before + min(eq_before, need), q);
    else if (eq && eq_before < need) emit(gt_before + eq_before, q);
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
  int32_t chunk;        // 4096
  int32_t nchunks;      // chunks of a row of length n_max
};

// Visible entries of row t clamped to n_max; -1 marks a row to leave untouched.
__device__ __forceinline__ int clamp_n(const TopkParams& p, int t) {
  const int n = __ldg(p.n_vis + t);
  return n < 0 ? -1 : (n > p.n_max ? p.n_max : n);
}

__global__ void __launch_bounds__(kChunkThreads) topk_chunk_kernel(const TopkParams p) {
  constexpr int NT = kChunkThreads;
  __shared__ Scratch sc;
  __shared__ uint32_t cnt[kPer * (NT / 32)];
  griddep_launch();
  griddep_wait();
  const int t = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
  const int n = clamp_n(p, t);
  if (n < 0) return;
  int32_t* out = p.idx + static_cast<int64_t>(t) * p.idx_stride;
  if (n <= p.k) {
    if (c == 0)
      for (int j = tid; j < p.k; j += NT) out[j] = j < n ? j : -1;
    return;
  }
  const int nch = (n + kChunk - 1) / kChunk;
  if (c >= nch) return;
  const int lo = c * kChunk;
  const int m = min(n, lo + kChunk) - lo;
  const int64_t cbase = (static_cast<int64_t>(t) * p.nchunks + c) * p.k;
  const float* row = p.logits + static_cast<int64_t>(t) * p.logits_stride + lo;
  // unconditional loads from clamped (always valid) addresses, so all of them
  // are in flight together; positions past the chunk are masked afterwards
  float v[kPer];
#pragma unroll
  for (int q = 0; q < kPer; ++q) v[q] = __ldg(row + min(q * NT + tid, m - 1));
  uint32_t key[kPer];
  uint32_t vmask = 0;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const bool in = q * NT + tid < m;
    key[q] = in ? order_key(v[q]) : 0u;
    vmask |= (in ? 1u : 0u) << q;
  }
  if (nch > 1 && m <= p.k) {  // a short tail chunk: every entry is a candidate
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      if (vmask >> q & 1u) {
        const int pos = q * NT + tid;
        p.cand_key[cbase + pos] = key[q];
        p.cand_idx[cbase + pos] = lo + pos;
      }
    }
    return;
  }
  uint32_t kth;
  int need;
  radix_select<NT>(key, vmask, p.k, sc, kth, need);
  if (nch == 1) {
    ordered_emit<NT>(key, vmask, kth, need, sc, cnt, [&](int r, int q) { out[r] = lo + q * NT + tid; });
  } else {
    ordered_emit<NT>(key, vmask, kth, need, sc, cnt, [&](int r, int q) {
      p.cand_key[cbase + r] = key[q];
      p.cand_idx[cbase + r] = lo + q * NT + tid;
    });
  }
}

// Stage 2: the row's candidates (each chunk's top-k, in chunk order) -> top-k.
template <int NT, int P>
__global__ void __launch_bounds__(NT) topk_merge_kernel(const TopkParams p) {
  __shared__ Scratch sc;
  __shared__ int chunk_start[65];
  __shared__ uint32_t cnt[P * (NT / 32)];
  griddep_launch();
  griddep_wait();
  const int t = blockIdx.x, tid = threadIdx.x;
  const int n = clamp_n(p, t);
  if (n <= p.k) return;  // includes rows left untouched (n < 0)
  const int nch = (n + kChunk - 1) / kChunk;
  if (nch <= 1) return;
  if (tid == 0) {
    int acc = 0;
    for (int c = 0; c < nch; ++c) {
      chunk_start[c] = acc;
      acc += min(min(n, (c + 1) * kChunk) - c * kChunk, p.k);
    }
    chunk_start[nch] = acc;
  }
  __syncthreads();
  const int m = chunk_start[nch];
  // candidate position -> chunk c (ascending entry order) and offset within it
  auto cand = [&](int pos, int& c, int& off) {
    c = 0;
    while (chunk_start[c + 1] <= pos) ++c;
    off = pos - chunk_start[c];
  };
  uint32_t key[P];
  uint32_t vmask = 0;
#pragma unroll
  for (int q = 0; q < P; ++q) {
    int c, off;
    cand(min(q * NT + tid, m - 1), c, off);   // clamped: every load valid and in flight together
    key[q] = __ldg(p.cand_key + (static_cast<int64_t>(t) * p.nchunks + c) * p.k + off);
  }
#pragma unroll
  for (int q = 0; q < P; ++q) {
    const bool in = q * NT + tid < m;
    if (!in) key[q] = 0u;
    vmask |= (in ? 1u : 0u) << q;
  }
  uint32_t kth;
  int need;
  radix_select<NT>(key, vmask, p.k, sc, kth, need);
  int32_t* out = p.idx + static_cast<int64_t>(t) * p.idx_stride;
  ordered_emit<NT>(key, vmask, kth, need, sc, cnt, [&](int r, int q) {
    int c, off;
    cand(q * NT + tid, c, off);
    out[r] = p.cand_idx[(static_cast<int64_t>(t) * p.nchunks + c) * p.k + off];
  });
}

}  // namespace

void topk_plan(int32_t n_max, int32_t k, int32_t* chunk_len, int32_t* n_chunks) {
  *chunk_len = 0;
  *n_chunks = 0;
  if (k < 1 || k > DSV4SA_MAX_TOPK || n_max < 0) return;
  const int64_t nch = n_max <= kChunk ? 1 : (static_cast<int64_t>(n_max) + kChunk - 1) / kChunk;
  if (nch > 1 && (nch * k > kMaxCand || nch > 64)) return;
  *chunk_len = kChunk;
  *n_chunks = static_cast<int32_t>(nch);
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
  if (launch_pdl(topk_chunk_kernel, dim3(nch, T), dim3(kChunkThreads), 0, stream, p) != cudaSuccess)
    return DSV4SA_ERR_CUDA;
  if (nch > 1) {
    const cudaError_t e = (nch * k <= 2048)
                              ? launch_pdl(topk_merge_kernel<256, 8>, dim3(T), dim3(256), 0, stream, p)
                              : launch_pdl(topk_merge_kernel<kMergeThreads, kMaxCand / kMergeThreads>, dim3(T),
                                           dim3(kMergeThreads), 0, stream, p);
    if (e != cudaSuccess) return DSV4SA_ERR_CUDA;
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

// ---------------------------------------------------------------- scratch-free variant
//
// dsv4sa_topk_noalloc: the same selection as dsv4sa_topk, but the candidate
// scratch of the chunked stage lives in a file-scope device array instead of a
// caller workspace, for callers that cannot allocate device memory at call time
// (see dsv4sa.h).  Every GPU that loads the library holds this array until the
// process exits.

namespace dsv4sa {
namespace {

static __device__ __align__(256) uint8_t g_topk_scratch[DSV4SA_TOPK_NOALLOC_SCRATCH_BYTES];

// Device address of g_topk_scratch on the current device.  In host code the
// symbol's name is only a host-side stand-in, so the address is asked of the
// runtime once per device, with that device current, and cached.
void* noalloc_scratch(int dev) {
  constexpr int kMaxDevices = 64;
  static void* addr[kMaxDevices] = {};
  static std::mutex mu;
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_topk_scratch) != cudaSuccess) return nullptr;
    addr[dev] = ptr;
  }
  return addr[dev];
}

}  // namespace
}  // namespace dsv4sa

extern "C" DSV4SA_API int dsv4sa_topk_noalloc(const float* logits, int64_t logits_stride, const int32_t* n_vis,
                                              int32_t T, int32_t n_max, int32_t k, int32_t* idx, int32_t idx_stride,
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
  const size_t need = nch > 1 ? static_cast<size_t>(T) * nch * k * 8 : 0;
  if (need > DSV4SA_TOPK_NOALLOC_SCRATCH_BYTES) return DSV4SA_ERR_UNSUPPORTED;  // beyond the fixed scratch
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSV4SA_ERR_CUDA;
  void* scratch = dsv4sa::noalloc_scratch(dev);
  if (!scratch) return DSV4SA_ERR_CUDA;
  return dsv4sa::launch_topk(logits, logits_stride, n_vis, T, n_max, k, idx, idx_stride, scratch,
                             DSV4SA_TOPK_NOALLOC_SCRATCH_BYTES, stream);
}
