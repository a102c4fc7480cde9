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
// integer work.  One 1024-thread CTA selects from up to 16384 keys: one bulk
// copy brings the chunk into shared memory and thread t takes the 16
// consecutive positions 16 t .. 16 t + 15;
//   1. a lower bound of the k-th largest key: every thread's largest key is a
//      distinct entry; each warp sorts its 32 thread maxima in registers and
//      offers its ceil(k / 32)-th largest, and the smallest offer bounds the
//      k-th largest key from below (no pass over the whole block);
//   2. the keys at or above the bound (a few percent of a row) are compacted
//      into shared memory in position order;
//   3. on the compacted keys, four per thread: the min/max of the keys fixes
//      the bits they share, an 11-bit radix pass finds the digit of the k-th
//      largest key and the few keys sharing it are ranked directly (more
//      passes only when many share it); each thread counts its selected keys
//      and one block scan gives the output offsets, so entries come out in
//      ascending order with the lowest-index ties first.
// With too few warps holding keys, or too many keys above the bound, step 3
// runs on all the keys instead.
// Longer rows are cut into chunks of 16384: stage 1 keeps each chunk's exact
// top-k as (key, index) candidates -- every member of the row's top-k is in its
// chunk's top-k under the same order -- and stage 2 selects the final k among
// the candidates, which sit contiguously in ascending index order.
// Optionally, each selected entry's row of the KV pool the attention will
// gather from is prefetched into L2 as the index is written.
#include <mutex>

#include "common.cuh"
#include "dsv4sa_internal.h"

namespace dsv4sa {
namespace {

constexpr int kThreads = 1024;               // one CTA per row or chunk
constexpr int kWarps = kThreads / 32;
constexpr int kPer = 16;                     // values per thread, stage 1
constexpr int kChunk = kThreads * kPer;      // 16384
constexpr int kMergePer = 32;                // candidates per thread, stage 2
constexpr int kMaxCand = kThreads * kMergePer;   // 32768
constexpr int kBins = 2048;                  // 11-bit radix digit
constexpr int kRankCap = 256;                // keys ranked directly after a pass
constexpr int kCandCap = 4096;               // contenders compacted into shared memory
constexpr int kSelThreads = 512;             // threads that select among the contenders
constexpr int kCandPer = kCandCap / kSelThreads;
constexpr int kPtCache = 1024;               // page-table entries staged for the row prefetches

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t b = __float_as_uint(f);
  if ((b & 0x7FFFFFFFu) > 0x7F800000u) return 0u;  // NaN: lowest
  if ((b & 0x7FFFFFFFu) == 0u) b = 0u;             // -0 == +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// The float a (non-NaN) order key stands for: x >= key_float(kk) exactly when
// order_key(x) >= kk, for every non-NaN x.
__device__ __forceinline__ float key_float(uint32_t kk) {
  return __uint_as_float((kk & 0x80000000u) ? (kk ^ 0x80000000u) : ~kk);
}

struct Scratch {
  uint32_t keys[kChunk];      // fallback: every key of the chunk in position order
  uint32_t hist[kBins];
  uint32_t ckey[kCandCap];    // contenders' keys, in position order
  uint16_t cpos[kCandCap];    // their positions within the CTA's keys
  uint32_t cand[kRankCap];
  uint32_t selkey[DSV4SA_MAX_TOPK];   // selected contenders' keys and positions, by output rank
  uint16_t sel[DSV4SA_MAX_TOPK];
  uint32_t scan[kWarps];
  unsigned long long scan64[kWarps];
  uint32_t red_min[kWarps];
  uint32_t red_max[kWarps];
  uint32_t red_low[kWarps];
  uint32_t red_groups[kWarps];
  uint32_t wbound[kWarps];    // per warp: a key value, and how many distinct keys are at or above it
  uint32_t wcount[kWarps];
  int32_t pt[kPtCache];       // the query's page-table row of the prefetch pool, when it fits
  int found_bin;
  int found_above;
  int found_count;
  int n_cand;
  uint32_t kth;
  int need;
};
constexpr int kScratchBytes = static_cast<int>(sizeof(Scratch));

// Barrier over the first NT threads of the CTA (all of them: __syncthreads).
template <int NT>
__device__ __forceinline__ void group_sync() {
  if constexpr (NT == kThreads) {
    __syncthreads();
  } else {
    named_barrier_sync(1, NT);
  }
}

// Exclusive scan of one value per thread over the first NT threads; returns
// the total.  T is uint32_t or unsigned long long (packed fields that never carry).
template <int NT, class T>
__device__ __forceinline__ T group_scan(T v, T* buf, T& total) {
  constexpr int W = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  T x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) buf[warp] = x;
  group_sync<NT>();
  const T w = lane < W ? buf[lane] : T(0);
  T wx = w;
#pragma unroll
  for (int o = 1; o < W; o <<= 1) {
    const T y = __shfl_up_sync(0xffffffffu, wx, o);
    if (lane >= o) wx += y;
  }
  total = __shfl_sync(0xffffffffu, wx, W - 1);
  const T before = __shfl_sync(0xffffffffu, wx - w, warp);   // exclusive prefix of this warp
  group_sync<NT>();
  return before + x - v;
}

// One radix pass over digit bits [lo, hi] (at most 11 bits) of the valid keys
// whose bits above hi equal `prefix` (under pmask).  Finds the digit value
// holding the rem-th largest such key; on return sc.found_bin / found_above /
// found_count hold that digit, the number of keys with a larger digit, and the
// keys sharing it.
template <int NT, int P>
__device__ void radix_pass(const uint32_t (&key)[P], uint32_t valid_mask, uint32_t pmask, uint32_t prefix, int hi,
                           int lo, int rem, Scratch& sc) {
  constexpr int B = kBins / NT;   // bins owned by a thread in the scan
  const int tid = threadIdx.x;
  const uint32_t dmask = (2u << (hi - lo)) - 1u;
#pragma unroll
  for (int q = 0; q < B; ++q) sc.hist[tid * B + q] = 0u;
  group_sync<NT>();
#pragma unroll
  for (int i = 0; i < P; ++i) {
    if ((valid_mask >> i & 1u) && (key[i] & pmask) == prefix) atomicAdd(&sc.hist[(key[i] >> lo) & dmask], 1u);
  }
  group_sync<NT>();
  // thread tid owns bins [kBins - (tid + 1) B, kBins - tid B), highest first
  uint32_t cb[B];
  uint32_t local = 0;
#pragma unroll
  for (int q = 0; q < B; ++q) {
    cb[q] = sc.hist[kBins - 1 - tid * B - q];
    local += cb[q];
  }
  uint32_t total;
  const int above = static_cast<int>(group_scan<NT>(local, sc.scan, total));
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
  group_sync<NT>();
}

// Select among the valid keys of the first NT threads (key[i] valid when
// valid_mask bit i is set; at least k valid keys overall, k >= 1).  Returns the
// k-th largest key and how many of its ties (lowest positions first) belong to
// the top k.
template <int NT, int P>
__device__ void radix_select(const uint32_t (&key)[P], uint32_t valid_mask, int k, Scratch& sc, uint32_t& kth,
                             int& need) {
  constexpr int W = NT / 32;
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
  group_sync<NT>();
  mn = __reduce_min_sync(0xffffffffu, lane < W ? sc.red_min[lane] : 0xFFFFFFFFu);
  mx = __reduce_max_sync(0xffffffffu, lane < W ? sc.red_max[lane] : 0u);
  const uint32_t low = __reduce_min_sync(0xffffffffu, lane < W ? sc.red_low[lane] : 0xFFFFFFFFu);
  const int groups = static_cast<int>(__reduce_add_sync(0xffffffffu, lane < W ? sc.red_groups[lane] : 0u));
  if (groups >= k && low > mn) {  // keys below the smallest thread maximum cannot be selected
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
#pragma unroll 1
  while (hi >= 0) {
    const int lo = hi - 10 > 0 ? hi - 10 : 0;
    radix_pass<NT, P>(key, valid_mask, pmask, prefix, hi, lo, rem, sc);
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
      group_sync<NT>();
      for (int c = tid; c < count; c += NT) {
        const uint32_t mine = sc.cand[c];
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
      group_sync<NT>();
      kth = sc.kth;
      need = sc.need;
      return;
    }
    group_sync<NT>();
  }
  kth = prefix;
  need = rem;
}

// Output ranks.  Thread t (of the first NT) holds positions t P .. t P + P - 1;
// an entry is selected if key > kth, or key == kth and fewer than `need` equal
// keys sit at lower positions.  emit(rank, i) is called once per selected
// entry, rank = number of selected entries at lower positions.
template <int NT, int P, class Emit>
__device__ void ordered_emit(const uint32_t (&key)[P], uint32_t valid_mask, uint32_t kth, int need, Scratch& sc,
                             Emit emit) {
  uint32_t ng = 0, ne = 0;
#pragma unroll
  for (int i = 0; i < P; ++i) {
    const bool ok = valid_mask >> i & 1u;
    ng += (ok && key[i] > kth) ? 1u : 0u;
    ne += (ok && key[i] == kth) ? 1u : 0u;
  }
  // packed (greater, equal) counts: both totals stay below 2^16
  uint32_t total;
  const uint32_t before = group_scan<NT>(ng | (ne << 16), sc.scan, total);
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

// A lower bound of the k-th largest key, with no pass over the block: every
// thread's largest key is a distinct entry; each warp sorts its 32 thread maxima
// (bitonic, in registers) and offers its r-th largest, r = ceil(k / 32) (or its
// smallest, when fewer threads hold keys), together with how many of its
// maxima are at least that large.  The smallest offer is a bound whenever the
// counts add up to k.  Returns false (no bound) otherwise.
__device__ __forceinline__ bool warp_sort_bound(uint32_t tmax, bool holds, int k, Scratch& sc, uint32_t& bound) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t v = holds ? tmax : 0u;
#pragma unroll
  for (int kk = 2; kk <= 32; kk <<= 1) {
#pragma unroll
    for (int j = kk >> 1; j > 0; j >>= 1) {
      const uint32_t o = __shfl_xor_sync(0xffffffffu, v, j);
      const bool lower = (lane & j) == 0, desc = (lane & kk) == 0;
      v = (lower == desc) ? max(v, o) : min(v, o);   // descending overall
    }
  }
  const int holders = __popc(__ballot_sync(0xffffffffu, holds));
  const int r = min((k + 31) / 32, holders);          // lanes 0 .. holders-1 hold the real maxima
  const uint32_t offer = __shfl_sync(0xffffffffu, v, max(r - 1, 0));
  if (lane == 0) {
    sc.wbound[warp] = offer;
    sc.wcount[warp] = static_cast<uint32_t>(r);
  }
  __syncthreads();
  const uint32_t c = sc.wcount[lane];
  const uint32_t b = c > 0 ? sc.wbound[lane] : 0xFFFFFFFFu;
  const uint32_t count = __reduce_add_sync(0xffffffffu, c);
  bound = __reduce_min_sync(0xffffffffu, b);
  return count >= static_cast<uint32_t>(k);
}

// The selection among the C <= kCandCap contenders in sc.ckey / sc.cpos
// (position order), by the first kSelThreads threads (the caller's other
// threads have left).  The radix select sees the contenders strided over the
// threads (c = tid + kSelThreads j), so every thread holds a few; the ranks
// are then taken over contiguous runs (c = kCandPer tid + j, position order)
// and the selected keys and positions land in sc.selkey / sc.sel[rank].
__device__ void select_contenders(int C, int k, Scratch& sc) {
  const int tid = threadIdx.x;
  uint32_t kth;
  int need;
  {
    uint32_t ck[kCandPer];
    uint32_t cmask = 0u;
#pragma unroll
    for (int j = 0; j < kCandPer; ++j) {
      const int c = tid + kSelThreads * j;
      ck[j] = c < C ? sc.ckey[c] : 0u;
      cmask |= (c < C ? 1u : 0u) << j;
    }
    radix_select<kSelThreads, kCandPer>(ck, cmask, k, sc, kth, need);
  }
  uint32_t ck[kCandPer];
  uint32_t cmask = 0u;
#pragma unroll
  for (int j = 0; j < kCandPer; ++j) {
    const int c = kCandPer * tid + j;
    ck[j] = c < C ? sc.ckey[c] : 0u;
    cmask |= (c < C ? 1u : 0u) << j;
  }
  ordered_emit<kSelThreads, kCandPer>(ck, cmask, kth, need, sc, [&](int r, int j) {
    sc.selkey[r] = ck[j];
    sc.sel[r] = sc.cpos[kCandPer * tid + j];
  });
  group_sync<kSelThreads>();
}

// Full selection over keys held as contiguous positions (thread t: t P .. t P
// + P - 1), all 1024 threads; the result lands in sc.selkey / sc.sel[rank].
template <int P>
__device__ void select_all_keys(const uint32_t (&key)[P], uint32_t valid_mask, int k, Scratch& sc) {
  const int tid = threadIdx.x;
  uint32_t kth;
  int need;
  radix_select<kThreads, P>(key, valid_mask, k, sc, kth, need);
  ordered_emit<kThreads, P>(key, valid_mask, kth, need, sc, [&](int r, int i) {
    sc.selkey[r] = key[i];
    sc.sel[r] = static_cast<uint16_t>(tid * P + i);
  });
  __syncthreads();
}

// The full selection over a chunk's m keys staged in position order in
// sc.keys (the rare case without a usable bound), kept out of line so the
// common path stays short.
__device__ __noinline__ void select_all_staged(int m, int k, Scratch& sc) {
  __syncthreads();
  uint32_t key[kPer];
  uint32_t vmask = 0u;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    key[i] = sc.keys[threadIdx.x * kPer + i];
    vmask |= (static_cast<int>(threadIdx.x) * kPer + i < m ? 1u : 0u) << i;
  }
  select_all_keys<kPer>(key, vmask, k, sc);
}

// Selection over keys held as contiguous positions (thread t: t P .. t P + P - 1),
// all 1024 threads.  The contenders (keys at or above a warp-sorted bound) go
// to select_contenders; with no bound or too many contenders the whole
// selection runs on all the keys.  The result is in sc.selkey / sc.sel[rank];
// returns how many of the first threads remain (the others have nothing left
// to do and return 0).
template <int P>
__device__ int select_keys(const uint32_t (&key)[P], uint32_t valid_mask, int k, Scratch& sc) {
  const int tid = threadIdx.x;
  uint32_t tmax = 0u;
#pragma unroll
  for (int i = 0; i < P; ++i)
    if (valid_mask >> i & 1u) tmax = max(tmax, key[i]);
  uint32_t bound = 0u;
  const bool bounded = warp_sort_bound(tmax, valid_mask != 0u, k, sc, bound);
  uint32_t mine = 0u;
#pragma unroll
  for (int i = 0; i < P; ++i) mine += ((valid_mask >> i & 1u) && key[i] >= bound) ? 1u : 0u;
  uint32_t total;
  uint32_t off = group_scan<kThreads>(mine, sc.scan, total);
  if (!bounded || total > static_cast<uint32_t>(kCandCap)) {
    select_all_keys<P>(key, valid_mask, k, sc);
    return kThreads;
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
  if (tid >= kSelThreads) return 0;
  select_contenders(static_cast<int>(total), k, sc);
  return kSelThreads;
}

// Selection over a chunk's m <= 16384 scores as loaded: thread t holds the four
// 16-byte groups j = 0..3 at float positions 4 (1024 j + t) .. + 3, positions
// >= m already NaN.  The bound, the count and the compaction compare the floats
// themselves (NaN never passes, -0 equals +0); only the contenders become
// order keys.  Result and return value as select_keys.
__device__ int select_scores(const float (&x)[kPer], int m, int k, Scratch& sc) {
  const int tid = threadIdx.x;
  float tm = x[0];
#pragma unroll
  for (int i = 1; i < kPer; ++i) tm = fmaxf(tm, x[i]);   // NaN ignored unless all are NaN
  const bool holds = !isnan(tm);
  uint32_t bound = 0u;
  const bool bounded = warp_sort_bound(holds ? order_key(tm) : 0u, holds, k, sc, bound);
  const float bf = key_float(bound);
  unsigned long long cnt = 0ull;   // contenders of group j in bits 16 j .. 16 j + 15
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t c = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) c += x[4 * j + i] >= bf ? 1u : 0u;
    cnt |= static_cast<unsigned long long>(c) << (16 * j);
  }
  unsigned long long tot64;
  const unsigned long long before = group_scan<kThreads>(cnt, sc.scan64, tot64);
  int C = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) C += static_cast<int>((tot64 >> (16 * j)) & 0xFFFFu);
  if (!bounded || C > kCandCap) {   // rare: every key through the full selection, out of line
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) sc.keys[4 * (1024 * j + tid) + i] = order_key(x[4 * j + i]);
    select_all_staged(m, k, sc);
    return kThreads;
  }
  int off = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    int o = off + static_cast<int>((before >> (16 * j)) & 0xFFFFu);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (x[4 * j + i] >= bf) {
        sc.ckey[o] = order_key(x[4 * j + i]);
        sc.cpos[o] = static_cast<uint16_t>(4 * (1024 * j + tid) + i);
        ++o;
      }
    }
    off += static_cast<int>((tot64 >> (16 * j)) & 0xFFFFu);
  }
  __syncthreads();
  if (tid >= kSelThreads) return 0;
  select_contenders(C, k, sc);
  return kSelThreads;
}

struct TopkParams {
  const float* logits;
  const int32_t* n_vis;
  int32_t* idx;
  uint32_t* cand_key;   // [T][nchunks * k]: chunk c's candidates at c * k
  int32_t* cand_idx;    // [T][nchunks * k]
  // optional: the KV pool the selected entries will be gathered from, whose
  // rows are prefetched into L2 as they are selected
  const uint8_t* pf_base;
  const int32_t* pf_pt;
  const int32_t* pf_seq;
  int64_t pf_page_stride;
  int64_t pf_num_pages;
  int32_t pf_pt_stride;
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

// Stage the query's page-table row of the prefetch pool in shared memory (when
// it fits), so the prefetches at the end need no global load.
__device__ __forceinline__ void stage_prefetch_pt(const TopkParams& p, int t, Scratch& sc) {
  if (p.pf_base == nullptr || p.pf_pt_stride > kPtCache) return;
  const int32_t* row = p.pf_pt + static_cast<int64_t>(__ldg(p.pf_seq + t)) * p.pf_pt_stride;
  for (int e = threadIdx.x; e < p.pf_pt_stride; e += kThreads) sc.pt[e] = __ldg(row + e);
}

// Prefetch into L2 the row of compressed entry e of query t in the optional KV
// pool (default page layout: the slot's codes, rope values and scales).  The
// staged page-table row must be visible (a barrier after stage_prefetch_pt).
__device__ __forceinline__ void prefetch_row(const TopkParams& p, int t, int e, const Scratch& sc) {
  if (p.pf_base == nullptr || e < 0 || e >= p.pf_pt_stride * 64) return;
  const int32_t page = p.pf_pt_stride <= kPtCache
                           ? sc.pt[e >> 6]
                           : __ldg(p.pf_pt + static_cast<int64_t>(__ldg(p.pf_seq + t)) * p.pf_pt_stride + (e >> 6));
  if (page < 0 || page >= p.pf_num_pages) return;   // the attention flags it; nothing to fetch
  const uint8_t* base = p.pf_base + static_cast<int64_t>(page) * p.pf_page_stride;
  const int slot = e & 63;
  // one prefetch per 128-byte line: the 448 code bytes (4 or 5 lines), the rope
  // values (one line) and the scales (one line)
  const uint8_t* nope = base + slot * 448;
  const uint8_t* last = nope + 447;
  for (const uint8_t* a = nope; a <= last; a += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
  if ((reinterpret_cast<uintptr_t>(nope) & 127u) > (reinterpret_cast<uintptr_t>(last) & 127u))
    asm volatile("prefetch.global.L2 [%0];" ::"l"(last));
  asm volatile("prefetch.global.L2 [%0];" ::"l"(base + 28672 + slot * 128));
  asm volatile("prefetch.global.L2 [%0];" ::"l"(base + 36864 + slot * 32));
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

// Scores of a chunk of m >= 1 values for select_emit_scores: four coalesced
// 16-byte loads per thread (group j: float positions 4 (1024 j + t) .. + 3),
// from clamped addresses, all in flight together; positions >= m become NaN.
__device__ __forceinline__ void load_scores(const float* row, int m, bool vec, float (&x)[kPer]) {
  const int tid = threadIdx.x;
  if (vec) {
    const float4* r4 = reinterpret_cast<const float4*>(row);
    const int last = (m - 1) >> 2;
    float4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = __ldg(r4 + min(1024 * j + tid, last));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[4 * j] = v[j].x;
      x[4 * j + 1] = v[j].y;
      x[4 * j + 2] = v[j].z;
      x[4 * j + 3] = v[j].w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) x[4 * j + i] = __ldg(row + min(4 * (1024 * j + tid) + i, m - 1));
  }
  if (4 * (1024 * 3 + tid) + 3 >= m) {   // only threads that reach past the chunk
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (4 * (1024 * j + tid) + i >= m) x[4 * j + i] = __uint_as_float(0x7FC00000u);
  }
}

// Stage 1 (and the whole selection for rows of up to one chunk).
__global__ void __launch_bounds__(kThreads, 1) topk_chunk_kernel(const TopkParams p) {
  extern __shared__ __align__(128) uint8_t topk_smem[];
  Scratch& sc = *reinterpret_cast<Scratch*>(topk_smem);
  griddep_launch();
  // the row's small inputs into L2 while the previous kernel finishes (a
  // prefetch is only a hint: later writes by that kernel are still seen)
  if (threadIdx.x == 0) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p.n_vis + blockIdx.y));
    if (p.pf_base) asm volatile("prefetch.global.L2 [%0];" ::"l"(p.pf_seq + blockIdx.y));
  }
  griddep_wait();
  const int t = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
  const int n = clamp_n(p, t);
  if (n < 0) return;
  int32_t* out = p.idx + static_cast<int64_t>(t) * p.idx_stride;
  if (n <= p.k) {
    if (c == 0) {
      stage_prefetch_pt(p, t, sc);
      __syncthreads();
      for (int j = tid; j < p.k; j += kThreads) {
        out[j] = j < n ? j : -1;
        if (j < n) prefetch_row(p, t, j, sc);
      }
    }
    return;
  }
  const int nch = (n + kChunk - 1) / kChunk;
  if (c >= nch) return;
  const int lo = c * kChunk;
  const int m = min(n, lo + kChunk) - lo;
  const int64_t cbase = (static_cast<int64_t>(t) * p.nchunks + c) * p.k;
  const float* row = p.logits + static_cast<int64_t>(t) * p.logits_stride + lo;
  if (nch > 1 && m <= p.k) {  // a short tail chunk: every entry is a candidate
    for (int i = tid; i < m; i += kThreads) {
      p.cand_key[cbase + i] = order_key(__ldg(row + i));
      p.cand_idx[cbase + i] = lo + i;
    }
    return;
  }
  if (nch == 1) stage_prefetch_pt(p, t, sc);   // made visible by the barriers of the selection
  float x[kPer];
  load_scores(row, m, p.vec_logits != 0, x);
  const int act = select_scores(x, m, p.k, sc);
  // thread r of the active ones writes output rank r (and prefetches its row)
  for (int r = tid; act > 0 && r < p.k; r += act) {
    const int pos = lo + static_cast<int>(sc.sel[r]);
    if (nch == 1) {
      out[r] = pos;
      prefetch_row(p, t, pos, sc);
    } else {
      p.cand_key[cbase + r] = sc.selkey[r];
      p.cand_idx[cbase + r] = pos;
    }
  }
}

// Stage 2: the row's candidates (each chunk's top-k, contiguous in chunk
// order) -> top-k.
__global__ void __launch_bounds__(kThreads, 1) topk_merge_kernel(const TopkParams p) {
  extern __shared__ __align__(128) uint8_t topk_smem[];
  Scratch& sc = *reinterpret_cast<Scratch*>(topk_smem);
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
  stage_prefetch_pt(p, t, sc);   // made visible by the barriers of the selection
  load_row<kMergePer>(p.cand_key + rbase, m, p.vec_cand != 0, key, vmask, [](uint32_t x) { return x; });
  int32_t* out = p.idx + static_cast<int64_t>(t) * p.idx_stride;
  const int32_t* ci = p.cand_idx + rbase;
  const int act = select_keys<kMergePer>(key, vmask, p.k, sc);
  for (int r = threadIdx.x; act > 0 && r < p.k; r += act) {
    const int e = __ldg(ci + sc.sel[r]);
    out[r] = e;
    prefetch_row(p, t, e, sc);
  }
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
                int32_t k, int32_t* idx, int32_t idx_stride, void* ws, size_t ws_bytes, cudaStream_t stream,
                const TopkPrefetch* prefetch) {
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
  if (prefetch && prefetch->pool) {
    p.pf_base = static_cast<const uint8_t*>(prefetch->pool->base);
    p.pf_page_stride = prefetch->pool->page_stride;
    p.pf_num_pages = prefetch->pool->num_pages;
    p.pf_pt = prefetch->page_table;
    p.pf_pt_stride = prefetch->pt_stride;
    p.pf_seq = prefetch->q_seq;
  }
  if (nch > 1) {
    const size_t need = static_cast<size_t>(T) * nch * k * 8;
    if (!ws || ws_bytes < need) return DSV4SA_ERR_WORKSPACE;
    p.cand_key = static_cast<uint32_t*>(ws);
    p.cand_idx = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + static_cast<size_t>(T) * nch * k * 4);
    p.vec_cand = (reinterpret_cast<uintptr_t>(ws) % 16 == 0 && (static_cast<int64_t>(nch) * k) % 4 == 0) ? 1 : 0;
  }
  if (T == 0) return DSV4SA_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSV4SA_ERR_CUDA;
  if (!smem_attr_once(dev, 13, reinterpret_cast<const void*>(topk_chunk_kernel), kScratchBytes) ||
      !smem_attr_once(dev, 14, reinterpret_cast<const void*>(topk_merge_kernel), kScratchBytes))
    return DSV4SA_ERR_CUDA;
  if (launch_pdl(topk_chunk_kernel, dim3(nch, T), dim3(kThreads), kScratchBytes, stream, p) != cudaSuccess)
    return DSV4SA_ERR_CUDA;
  if (nch > 1 && launch_pdl(topk_merge_kernel, dim3(T), dim3(kThreads), kScratchBytes, stream, p) != cudaSuccess)
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
                             DSV4SA_TOPK_NOALLOC_SCRATCH_BYTES, stream, nullptr);
}
