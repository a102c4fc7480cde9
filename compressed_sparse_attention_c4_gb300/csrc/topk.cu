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
// integer work.  One 1024-thread CTA selects from up to 16384 keys held in
// registers; thread t owns the 16 consecutive positions 16 t .. 16 t + 15
// (four 16-byte loads):
//   1. a lower bound of the k-th largest key: every thread's largest key is a
//      distinct entry, so the k-th largest of the thread maxima -- located by
//      one 12-bit radix pass over those maxima, one key per thread -- bounds
//      it from below;
//   2. the keys at or above the bound (a few percent of a row) are compacted
//      into shared memory in position order;
//   3. on the compacted keys, two per thread: the min/max of the keys fixes the
//      bits they share, a 12-bit radix pass finds the digit of the k-th
//      largest key and the few keys sharing it are ranked directly (more
//      passes only when many share it); each thread counts its selected keys
//      and one block scan gives the output offsets, so entries come out in
//      ascending order with the lowest-index ties first.
// With fewer threads holding keys than k, or too many keys above the bound,
// step 3 runs on all the keys instead.
// Longer rows are cut into chunks of 16384: stage 1 keeps each chunk's exact
// top-k as (key, index) candidates -- every member of the row's top-k is in its
// chunk's top-k under the same order -- and stage 2 selects the final k among
// the candidates, which sit contiguously in ascending index order.
#include <mutex>

#include "common.cuh"
#include "dsv4sa_internal.h"

namespace dsv4sa {
namespace {

constexpr int kThreads = 1024;               // one CTA per row or chunk
constexpr int kWarps = kThreads / 32;
constexpr int kPer = 16;                     // keys per thread, stage 1
constexpr int kChunk = kThreads * kPer;      // 16384
constexpr int kMergePer = 32;                // candidates per thread, stage 2
constexpr int kMaxCand = kThreads * kMergePer;   // 32768
constexpr int kBins = 4096;                  // 12-bit radix digit
constexpr int kRankCap = 256;                // keys ranked directly after a pass
constexpr int kCandCap = 2 * kThreads;       // contenders compacted into shared memory

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t b = __float_as_uint(f);
  if ((b & 0x7FFFFFFFu) > 0x7F800000u) return 0u;  // NaN: lowest
  if ((b & 0x7FFFFFFFu) == 0u) b = 0u;             // -0 == +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

struct Scratch {
  uint32_t hist[kBins];
  uint32_t cand[kRankCap];
  uint32_t scan[kWarps];
  uint32_t red_min[kWarps];
  uint32_t red_max[kWarps];
  uint32_t red_low[kWarps];
  uint32_t red_groups[kWarps];
  int found_bin;
  int found_above;
  int found_count;
  int n_cand;
  uint32_t kth;
  int need;
  uint32_t ckey[kCandCap];    // contenders' keys, in position order
  uint16_t cpos[kCandCap];    // their positions within the CTA's keys
};

// Exclusive scan of one uint32 per thread over the block; returns the total.
__device__ __forceinline__ uint32_t block_scan(uint32_t v, uint32_t* buf, uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) buf[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = buf[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    buf[lane] = w;
  }
  __syncthreads();
  total = buf[kWarps - 1];
  const uint32_t before = warp == 0 ? 0u : buf[warp - 1];
  __syncthreads();
  return before + x - v;
}

// One radix pass over digit bits [lo, hi] of the valid keys whose bits above hi
// equal `prefix` (under pmask).  Finds the digit value holding the rem-th
// largest such key; on return sc.found_bin / found_above / found_count hold
// that digit, the number of keys with a larger digit, and the keys sharing it.
template <int P>
__device__ void radix_pass(const uint32_t (&key)[P], uint32_t valid_mask, uint32_t pmask, uint32_t prefix, int hi,
                           int lo, int rem, Scratch& sc) {
  const int tid = threadIdx.x;
  const uint32_t dmask = (2u << (hi - lo)) - 1u;
  for (int b = tid; b < kBins; b += kThreads) sc.hist[b] = 0u;
  __syncthreads();
#pragma unroll
  for (int i = 0; i < P; ++i) {
    if ((valid_mask >> i & 1u) && (key[i] & pmask) == prefix) atomicAdd(&sc.hist[(key[i] >> lo) & dmask], 1u);
  }
  __syncthreads();
  // thread tid owns bins [kBins - (tid + 1) B, kBins - tid B), highest first
  constexpr int B = kBins / kThreads;
  uint32_t cb[B];
  uint32_t local = 0;
#pragma unroll
  for (int q = 0; q < B; ++q) {
    cb[q] = sc.hist[kBins - 1 - tid * B - q];
    local += cb[q];
  }
  uint32_t total;
  const int above = static_cast<int>(block_scan(local, sc.scan, total));
  if (above < rem && above + static_cast<int>(local) >= rem) {
    int acc = above;
#pragma unroll
    for (int q = 0; q < B; ++q) {
      if (acc < rem && acc + static_cast<int>(cb[q]) >= rem) {
        sc.found_bin = kBins - 1 - tid * B - q;
        sc.found_above = acc;
        sc.found_count = static_cast<int>(cb[q]);
      }
      acc += static_cast<int>(cb[q]);
    }
  }
  if (tid == 0) sc.n_cand = 0;
  __syncthreads();
}

// Select among the valid keys of all threads (key[i] valid when valid_mask bit i
// is set; at least k valid keys overall, k >= 1).  Returns the k-th largest key
// and how many of its ties (lowest positions first) belong to the top k.
template <int P>
__device__ void radix_select(const uint32_t (&key)[P], uint32_t valid_mask, int k, Scratch& sc, uint32_t& kth,
                             int& need) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t mn = 0xFFFFFFFFu, mx = 0u;
#pragma unroll
  for (int i = 0; i < P; ++i) {
    if (valid_mask >> i & 1u) {
      mn = min(mn, key[i]);
      mx = max(mx, key[i]);
    }
  }
  const bool holds = valid_mask != 0u;
  {
    const uint32_t wmn = __reduce_min_sync(0xffffffffu, mn);
    const uint32_t wmx = __reduce_max_sync(0xffffffffu, mx);
    const uint32_t wlow = __reduce_min_sync(0xffffffffu, holds ? mx : 0xFFFFFFFFu);
    const uint32_t wgroups = __reduce_add_sync(0xffffffffu, holds ? 1u : 0u);
    if (lane == 0) {
      sc.red_min[warp] = wmn;
      sc.red_max[warp] = wmx;
      sc.red_low[warp] = wlow;
      sc.red_groups[warp] = wgroups;
    }
  }
  __syncthreads();
  mn = __reduce_min_sync(0xffffffffu, sc.red_min[lane]);
  mx = __reduce_max_sync(0xffffffffu, sc.red_max[lane]);
  const uint32_t low = __reduce_min_sync(0xffffffffu, sc.red_low[lane]);
  const int groups = static_cast<int>(__reduce_add_sync(0xffffffffu, sc.red_groups[lane]));
  if (groups >= k && low > mn) {  // keys below the bound cannot be selected
    mn = low;
#pragma unroll
    for (int i = 0; i < P; ++i)
      if (key[i] < low) valid_mask &= ~(1u << i);
  }
  const uint32_t diff = mn ^ mx;
  if (diff == 0u) {  // every remaining key equal
    kth = mx;
    need = k;
    return;
  }
  int hi = 31 - __clz(diff);  // highest varying bit
  uint32_t pmask = hi == 31 ? 0u : (0xFFFFFFFFu << (hi + 1));
  uint32_t prefix = mx & pmask;
  int rem = k;
  while (hi >= 0) {
    const int lo = hi - 11 > 0 ? hi - 11 : 0;
    radix_pass<P>(key, valid_mask, pmask, prefix, hi, lo, rem, sc);
    rem -= sc.found_above;
    prefix |= static_cast<uint32_t>(sc.found_bin) << lo;
    pmask |= ((2u << (hi - lo)) - 1u) << lo;
    hi = lo - 1;
    const int count = sc.found_count;
    if (hi >= 0 && count <= kRankCap) {
      // gather the keys of the found digit and rank them directly
#pragma unroll
      for (int i = 0; i < P; ++i) {
        if ((valid_mask >> i & 1u) && (key[i] & pmask) == prefix) sc.cand[atomicAdd(&sc.n_cand, 1)] = key[i];
      }
      __syncthreads();
      if (tid < count) {
        const uint32_t mine = sc.cand[tid];
        int gt = 0, eq = 0;
        for (int j = 0; j < count; ++j) {
          const uint32_t o = sc.cand[j];
          gt += o > mine ? 1 : 0;
          eq += o == mine ? 1 : 0;
        }
        if (gt < rem && gt + eq >= rem) {  // every tie of the k-th key writes the same values
          sc.kth = mine;
          sc.need = rem - gt;
        }
      }
      __syncthreads();
      kth = sc.kth;
      need = sc.need;
      return;
    }
    __syncthreads();
  }
  kth = prefix;
  need = rem;
}

// Output ranks.  Thread t holds positions t P .. t P + P - 1; an entry is
// selected if key > kth, or key == kth and fewer than `need` equal keys sit at
// lower positions.  emit(rank, i) is called once per selected entry, rank =
// number of selected entries at lower positions.
template <int P, class Emit>
__device__ void ordered_emit(const uint32_t (&key)[P], uint32_t valid_mask, uint32_t kth, int need, Scratch& sc,
                             Emit emit) {
  uint32_t ng = 0, ne = 0;
#pragma unroll
  for (int i = 0; i < P; ++i) {
    const bool ok = valid_mask >> i & 1u;
    ng += (ok && key[i] > kth) ? 1u : 0u;
    ne += (ok && key[i] == kth) ? 1u : 0u;
  }
  // packed (greater, equal) counts: both totals stay at or below 2^15
  uint32_t total;
  const uint32_t before = block_scan(ng | (ne << 16), sc.scan, total);
  int g = static_cast<int>(before & 0xFFFFu), e = static_cast<int>(before >> 16);
#pragma unroll
  for (int i = 0; i < P; ++i) {
    const bool ok = valid_mask >> i & 1u;
    if (ok && key[i] > kth) {
      emit(g + min(e, need), i);
      ++g;
    } else if (ok && key[i] == kth) {
      if (e < need) emit(g + e, i);
      ++e;
    }
  }
}

// Selection and ordered output in one: emit(rank, key, pos) once per selected
// key, pos = tid * P + i its position among the CTA's keys.
//   1. a lower bound of the k-th largest key: when k or more threads hold keys,
//      one 12-bit radix pass over the thread maxima finds the digit of the k-th
//      largest maximum; its lower edge bounds the k-th largest key from below
//      (k distinct maxima are at least that large);
//   2. the keys at or above the bound (a few percent of the row) are compacted
//      into shared memory in position order;
//   3. the selection and the ordered emit run on the compacted keys, two per
//      thread.  When there is no bound or too many keys pass it, the same two
//      steps run on all the keys.
template <int P, class Emit>
__device__ void select_emit(const uint32_t (&key)[P], uint32_t valid_mask, int k, Scratch& sc, Emit emit) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t tmax = 0u;
#pragma unroll
  for (int i = 0; i < P; ++i)
    if (valid_mask >> i & 1u) tmax = max(tmax, key[i]);
  const bool holds = valid_mask != 0u;
  {
    const uint32_t wmin = __reduce_min_sync(0xffffffffu, holds ? tmax : 0xFFFFFFFFu);
    const uint32_t wmax = __reduce_max_sync(0xffffffffu, tmax);
    const uint32_t wcnt = __reduce_add_sync(0xffffffffu, holds ? 1u : 0u);
    if (lane == 0) {
      sc.red_min[warp] = wmin;
      sc.red_max[warp] = wmax;
      sc.red_groups[warp] = wcnt;
    }
  }
  __syncthreads();
  const uint32_t lo_t = __reduce_min_sync(0xffffffffu, sc.red_min[lane]);
  const uint32_t hi_t = __reduce_max_sync(0xffffffffu, sc.red_max[lane]);
  const int nhold = static_cast<int>(__reduce_add_sync(0xffffffffu, sc.red_groups[lane]));
  bool bounded = false;
  uint32_t bound = 0u;
  if (nhold >= k) {
    bounded = true;
    if (lo_t == hi_t) {
      bound = hi_t;
    } else {
      const int hb = 31 - __clz(lo_t ^ hi_t), lb = hb - 11 > 0 ? hb - 11 : 0;
      const uint32_t pmask = hb == 31 ? 0u : (0xFFFFFFFFu << (hb + 1));
      const uint32_t tk[1] = {tmax};
      radix_pass<1>(tk, holds ? 1u : 0u, pmask, hi_t & pmask, hb, lb, k, sc);
      bound = (hi_t & pmask) | (static_cast<uint32_t>(sc.found_bin) << lb);
    }
  }
  uint32_t mine = 0u;
#pragma unroll
  for (int i = 0; i < P; ++i) mine += ((valid_mask >> i & 1u) && key[i] >= bound) ? 1u : 0u;
  uint32_t total;
  uint32_t off = block_scan(mine, sc.scan, total);
  if (!bounded || total > static_cast<uint32_t>(kCandCap)) {
    uint32_t kth;
    int need;
    radix_select<P>(key, valid_mask, k, sc, kth, need);
    ordered_emit<P>(key, valid_mask, kth, need, sc, [&](int r, int i) { emit(r, key[i], tid * P + i); });
    return;
  }
#pragma unroll
  for (int i = 0; i < P; ++i) {
    if ((valid_mask >> i & 1u) && key[i] >= bound) {
      sc.ckey[off] = key[i];
      sc.cpos[off] = static_cast<uint16_t>(tid * P + i);
      ++off;
    }
  }
  __syncthreads();
  uint32_t ck[2];
  uint32_t cmask = 0u;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const uint32_t c = 2u * tid + j;
    ck[j] = c < total ? sc.ckey[c] : 0u;
    cmask |= (c < total ? 1u : 0u) << j;
  }
  uint32_t kth;
  int need;
  radix_select<2>(ck, cmask, k, sc, kth, need);
  ordered_emit<2>(ck, cmask, kth, need, sc, [&](int r, int j) { emit(r, ck[j], sc.cpos[2 * tid + j]); });
}

struct TopkParams {
  const float* logits;
  const int32_t* n_vis;
  int32_t* idx;
  uint32_t* cand_key;   // [T][nchunks * k]: chunk c's candidates at c * k
  int32_t* cand_idx;    // [T][nchunks * k]
  int64_t logits_stride;
  int32_t idx_stride;
  int32_t T;
  int32_t n_max;
  int32_t k;
  int32_t nchunks;      // chunks of a row of length n_max
  int32_t vec_logits;   // rows start 16-byte aligned and span a multiple of 4 floats
  int32_t vec_cand;     // candidate rows likewise
};

// Visible entries of row t clamped to n_max; -1 marks a row to leave untouched.
__device__ __forceinline__ int clamp_n(const TopkParams& p, int t) {
  const int n = __ldg(p.n_vis + t);
  return n < 0 ? -1 : (n > p.n_max ? p.n_max : n);
}

// Loads positions tid P .. tid P + P - 1 of a row of m >= 1 values.  All loads
// are unconditional, from clamped addresses inside the row's allocation, so
// they are in flight together; positions >= m are masked afterwards.
template <int P, class T, class Conv>
__device__ __forceinline__ void load_row(const T* row, int m, bool vec, uint32_t (&key)[P], uint32_t& vmask,
                                         Conv conv) {
  static_assert(sizeof(T) == 4 && P % 4 == 0, "4-byte elements, whole vectors");
  const int base = threadIdx.x * P;
  if (vec) {
    const uint4* r4 = reinterpret_cast<const uint4*>(row);
    const int last = (m - 1) >> 2;
    uint4 x[P / 4];
#pragma unroll
    for (int j = 0; j < P / 4; ++j) x[j] = __ldg(r4 + min(base / 4 + j, last));
#pragma unroll
    for (int j = 0; j < P / 4; ++j) {
      key[4 * j] = conv(reinterpret_cast<const T&>(x[j].x));
      key[4 * j + 1] = conv(reinterpret_cast<const T&>(x[j].y));
      key[4 * j + 2] = conv(reinterpret_cast<const T&>(x[j].z));
      key[4 * j + 3] = conv(reinterpret_cast<const T&>(x[j].w));
    }
  } else {
    T v[P];
#pragma unroll
    for (int i = 0; i < P; ++i) v[i] = __ldg(row + min(base + i, m - 1));
#pragma unroll
    for (int i = 0; i < P; ++i) key[i] = conv(v[i]);
  }
  vmask = 0;
#pragma unroll
  for (int i = 0; i < P; ++i) {
    const bool in = base + i < m;
    if (!in) key[i] = 0u;
    vmask |= (in ? 1u : 0u) << i;
  }
}

// Stage 1 (and the whole selection for rows of up to one chunk).
__global__ void __launch_bounds__(kThreads, 1) topk_chunk_kernel(const TopkParams p) {
  __shared__ Scratch sc;
  griddep_launch();
  griddep_wait();
  const int t = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
  const int n = clamp_n(p, t);
  if (n < 0) return;
  int32_t* out = p.idx + static_cast<int64_t>(t) * p.idx_stride;
  if (n <= p.k) {
    if (c == 0)
      for (int j = tid; j < p.k; j += kThreads) out[j] = j < n ? j : -1;
    return;
  }
  const int nch = (n + kChunk - 1) / kChunk;
  if (c >= nch) return;
  const int lo = c * kChunk;
  const int m = min(n, lo + kChunk) - lo;
  const int64_t cbase = (static_cast<int64_t>(t) * p.nchunks + c) * p.k;
  const float* row = p.logits + static_cast<int64_t>(t) * p.logits_stride + lo;
  uint32_t key[kPer];
  uint32_t vmask;
  load_row<kPer>(row, m, p.vec_logits != 0, key, vmask, [](float f) { return order_key(f); });
  const int first = lo + tid * kPer;   // entry index of this thread's first position
  if (nch > 1 && m <= p.k) {  // a short tail chunk: every entry is a candidate
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      if (vmask >> i & 1u) {
        p.cand_key[cbase + tid * kPer + i] = key[i];
        p.cand_idx[cbase + tid * kPer + i] = first + i;
      }
    }
    return;
  }
  if (nch == 1) {
    select_emit<kPer>(key, vmask, p.k, sc, [&](int r, uint32_t, int pos) { out[r] = lo + pos; });
  } else {
    select_emit<kPer>(key, vmask, p.k, sc, [&](int r, uint32_t kv, int pos) {
      p.cand_key[cbase + r] = kv;
      p.cand_idx[cbase + r] = lo + pos;
    });
  }
}

// Stage 2: the row's candidates (each chunk's top-k, contiguous in chunk
// order) -> top-k.
__global__ void __launch_bounds__(kThreads, 1) topk_merge_kernel(const TopkParams p) {
  __shared__ Scratch sc;
  griddep_launch();
  griddep_wait();
  const int t = blockIdx.x;
  const int n = clamp_n(p, t);
  if (n <= p.k) return;  // includes rows left untouched (n < 0)
  const int nch = (n + kChunk - 1) / kChunk;
  if (nch <= 1) return;
  const int m = (nch - 1) * p.k + min(n - (nch - 1) * kChunk, p.k);
  const int64_t rbase = static_cast<int64_t>(t) * p.nchunks * p.k;
  uint32_t key[kMergePer];
  uint32_t vmask;
  load_row<kMergePer>(p.cand_key + rbase, m, p.vec_cand != 0, key, vmask, [](uint32_t x) { return x; });
  int32_t* out = p.idx + static_cast<int64_t>(t) * p.idx_stride;
  const int32_t* ci = p.cand_idx + rbase;
  select_emit<kMergePer>(key, vmask, p.k, sc, [&](int r, uint32_t, int pos) { out[r] = __ldg(ci + pos); });
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
  p.nchunks = nch;
  p.vec_logits = (reinterpret_cast<uintptr_t>(logits) % 16 == 0 && logits_stride % 4 == 0) ? 1 : 0;
  if (nch > 1) {
    const size_t need = static_cast<size_t>(T) * nch * k * 8;
    if (!ws || ws_bytes < need) return DSV4SA_ERR_WORKSPACE;
    p.cand_key = static_cast<uint32_t*>(ws);
    p.cand_idx = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + static_cast<size_t>(T) * nch * k * 4);
    p.vec_cand = (reinterpret_cast<uintptr_t>(ws) % 16 == 0 && (static_cast<int64_t>(nch) * k) % 4 == 0) ? 1 : 0;
  }
  if (T == 0) return DSV4SA_OK;
  if (launch_pdl(topk_chunk_kernel, dim3(nch, T), dim3(kThreads), 0, stream, p) != cudaSuccess)
    return DSV4SA_ERR_CUDA;
  if (nch > 1 && launch_pdl(topk_merge_kernel, dim3(T), dim3(kThreads), 0, stream, p) != cudaSuccess)
    return DSV4SA_ERR_CUDA;
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
