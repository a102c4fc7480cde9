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
// integer work.  One 1024-thread CTA selects from up to 16384 scores, held in
// registers, 16 per thread, as loaded (coalesced 16-byte groups):
//   1. a lower bound of the k-th largest key: every thread's largest score is a
//      distinct entry; each warp sorts its 32 thread maxima in registers and
//      offers its ceil(k / 32)-th largest, and the smallest offer bounds the
//      k-th largest key from below; the largest maximum is the row's maximum;
//   2. the scores at or above the bound (the contenders, a few percent of a
//      row) are compacted into shared memory in position order, and while
//      they are written an 11-bit radix histogram of the bits below the
//      highest one that differs between the bound and the maximum is built;
//   3. the histogram gives the digit holding the k-th largest key; the few
//      contenders sharing it are ranked directly (more passes over the
//      contenders only when many share it);
//   4. each thread takes a contiguous run of contenders, counts those above
//      the k-th key and equal to it, and one block scan gives the output ranks,
//      so entries come out in ascending position order with the lowest-index
//      ties first.
// The bound needs k distinct thread maxima; a row spread over fewer threads
// takes every entry as a contender (so do rows with heavy ties).  After an
// idle stretch every new stretch of instructions is fetched from memory, which
// costs more than the arithmetic, so the code is kept short: one copy of each
// step, loops over the contenders rather than unrolled variants.
// Longer rows are cut into chunks of 16384: stage 1 keeps each chunk's exact
// top-k as (key, index) candidates -- every member of the row's top-k is in its
// chunk's top-k under the same order -- and stage 2 selects the final k among
// the candidates (up to 32 consecutive ones per thread), which sit
// contiguously in ascending index order.
// Optionally, each selected entry's row of the KV pool the attention will
// gather from is prefetched into L2 as the index is written.
#include <mutex>

#include "common.cuh"
#include "dsv4sa_internal.h"

namespace dsv4sa {
namespace {

constexpr int kThreads = 1024;               // one CTA per row or chunk
constexpr int kWarps = kThreads / 32;
constexpr int kPer = 16;                     // scores per thread, stage 1
constexpr int kChunk = kThreads * kPer;      // 16384
constexpr int kMergePer = 32;                // candidates per thread, stage 2
constexpr int kMaxCand = kThreads * kMergePer;   // 32768
constexpr int kBins = 2048;                  // 11-bit radix digit
constexpr int kRankCap = 64;                 // keys ranked directly after a pass
constexpr int kPtCache = kThreads;           // page-table entries staged for the row prefetches (one per thread)

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t b = __float_as_uint(f);
  if ((b & 0x7FFFFFFFu) > 0x7F800000u) return 0u;  // NaN: lowest
  if ((b & 0x7FFFFFFFu) == 0u) b = 0u;             // -0 == +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// The float a nonzero order key stands for: for every non-NaN x,
// x >= key_float(kk) exactly when order_key(x) >= kk.
__device__ __forceinline__ float key_float(uint32_t kk) {
  return __uint_as_float((kk & 0x80000000u) ? (kk ^ 0x80000000u) : ~kk);
}

struct Scratch {
  uint32_t hist[kBins];
  uint32_t cand[kRankCap];
  unsigned long long scan64[kWarps];
  uint32_t scan[kWarps];
  uint32_t wbound[kWarps];    // per warp: its offer, how many maxima are at or above it,
  uint32_t wcount[kWarps];    // and its largest maximum
  uint32_t wmax[kWarps];
  int32_t pt[kPtCache];       // the query's page-table row of the prefetch pool, when it fits
  uint16_t selq[DSV4SA_MAX_TOPK];   // the selected contenders, by output rank
  int found_bin;
  int found_above;
  int found_count;
  int n_cand;
  uint32_t kth;
  int need;
};
// The contenders follow the scratch: their keys, then their positions (uint16).
constexpr int kScratchBytes = (static_cast<int>(sizeof(Scratch)) + 15) / 16 * 16;
constexpr int kChunkSmem = kScratchBytes + kChunk * 6;
constexpr int kMergeSmem = kScratchBytes + kMaxCand * 6;

// Exclusive scan of one value per thread over the CTA; returns the total.
// Packed fields (that never carry) scan together.  One barrier: every warp
// scans the warp totals itself; a caller puts a barrier between two scans on
// the same buffer (each call site here is followed by one before the next).
template <class T>
__device__ __forceinline__ T block_scan(T v, T* buf, T& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  T x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) buf[warp] = x;
  __syncthreads();
  const T w = buf[lane];
  T wx = w;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T y = __shfl_up_sync(0xffffffffu, wx, o);
    if (lane >= o) wx += y;
  }
  total = __shfl_sync(0xffffffffu, wx, 31);
  const T before = __shfl_sync(0xffffffffu, wx - w, warp);   // exclusive prefix of this warp
  return before + x - v;
}

// Step 1: each warp sorts its threads' largest keys (tmax, when the thread
// holds any) and offers its ceil(k / 32)-th largest; also the warp's largest
// key.  Returns, for the whole CTA, the bound on the k-th largest key (0, the
// smallest key there is, when fewer than k distinct maxima exist: every entry
// then contends) and the largest key.
__device__ __forceinline__ void block_bound(uint32_t tmax, bool holds, int k, Scratch& sc, uint32_t& lo_key,
                                            uint32_t& mx) {
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
    sc.wbound[warp] = r > 0 ? offer : 0xFFFFFFFFu;
    sc.wcount[warp] = static_cast<uint32_t>(r);
    sc.wmax[warp] = holders > 0 ? v : 0u;
  }
  __syncthreads();
  const uint32_t count = __reduce_add_sync(0xffffffffu, sc.wcount[lane]);
  mx = __reduce_max_sync(0xffffffffu, sc.wmax[lane]);
  const uint32_t b = __reduce_min_sync(0xffffffffu, sc.wbound[lane]);
  lo_key = count >= static_cast<uint32_t>(k) ? b : 0u;
}

// Digit geometry of the first radix pass over keys in [lo_key, mx]: bits
// [lo, hi] with the bits above hi common to the whole range.
struct Digits {
  int hi;
  int lo;
  uint32_t pmask;
  uint32_t prefix;
  uint32_t dmask;
  __device__ __forceinline__ void first(uint32_t lo_key, uint32_t mx) {
    hi = 31 - __clz(lo_key ^ mx);
    lo = hi - 10 > 0 ? hi - 10 : 0;
    pmask = hi == 31 ? 0u : (0xFFFFFFFFu << (hi + 1));
    prefix = mx & pmask;
    dmask = (2u << (hi - lo)) - 1u;
  }
};

// Steps 3 and 4 over the C contenders ck (position order, keys >= lo_key, at
// least k of them, the largest mx), whose first-pass histogram (Digits::first)
// is in sc.hist unless lo_key == mx.  sc.selq[rank] = the contender selected at
// that output rank, visible to the CTA on return.  sc.hist is left zero.
__device__ void select_contenders(const uint32_t* ck, int C, int k, uint32_t lo_key, uint32_t mx, Scratch& sc) {
  const int tid = threadIdx.x;
  uint32_t kth = mx;
  int need = k;
  if (lo_key != mx) {
    Digits d;
    d.first(lo_key, mx);
    int rem = k;
    bool built = true;   // the first pass's histogram came with the compaction
#pragma unroll 1
    while (true) {
      if (!built) {
        for (int c = tid; c < C; c += kThreads) {
          const uint32_t key = ck[c];
          if ((key & d.pmask) == d.prefix) atomicAdd(&sc.hist[(key >> d.lo) & d.dmask], 1u);
        }
        __syncthreads();
      }
      built = false;
      // thread t owns bins 2047 - 2 t and 2046 - 2 t (highest first), and clears them
      const uint32_t c0 = sc.hist[kBins - 1 - 2 * tid], c1 = sc.hist[kBins - 2 - 2 * tid];
      sc.hist[kBins - 1 - 2 * tid] = 0u;
      sc.hist[kBins - 2 - 2 * tid] = 0u;
      uint32_t total;
      const int above = static_cast<int>(block_scan<uint32_t>(c0 + c1, sc.scan, total));
      if (above < rem && above + static_cast<int>(c0 + c1) >= rem) {
        const bool first = above + static_cast<int>(c0) >= rem;
        sc.found_bin = first ? kBins - 1 - 2 * tid : kBins - 2 - 2 * tid;
        sc.found_above = first ? above : above + static_cast<int>(c0);
        sc.found_count = static_cast<int>(first ? c0 : c1);
      }
      if (tid == 0) sc.n_cand = 0;
      __syncthreads();
      rem -= sc.found_above;
      d.prefix |= static_cast<uint32_t>(sc.found_bin) << d.lo;
      d.pmask |= d.dmask << d.lo;
      const int cnt = sc.found_count;
      if (d.lo == 0) {   // every bit decided: the k-th key itself
        kth = d.prefix;
        need = rem;
        break;
      }
      if (cnt <= kRankCap) {
        // the contenders of the found digit, ranked directly
        for (int c = tid; c < C; c += kThreads) {
          const uint32_t key = ck[c];
          if ((key & d.pmask) == d.prefix) sc.cand[atomicAdd(&sc.n_cand, 1)] = key;
        }
        __syncthreads();
        if (tid < cnt) {
          const uint32_t mine = sc.cand[tid];
          int gt = 0, eq = 0;
          for (int j = 0; j < cnt; ++j) {
            const uint32_t o = sc.cand[j];
            gt += o > mine ? 1 : 0;
            eq += o == mine ? 1 : 0;
          }
          if (gt < rem && gt + eq >= rem) {   // every tie of the k-th key writes the same values
            sc.kth = mine;
            sc.need = rem - gt;
          }
        }
        __syncthreads();
        kth = sc.kth;
        need = sc.need;
        break;
      }
      d.hi = d.lo - 1;
      d.lo = d.hi - 10 > 0 ? d.hi - 10 : 0;
      d.dmask = (2u << (d.hi - d.lo)) - 1u;
    }
  }
  // ---- output ranks: thread t takes contenders [R t, R t + R)
  const int R = (C + kThreads - 1) / kThreads;
  const int c0 = min(C, R * tid), c1 = min(C, c0 + R);
  uint32_t ng = 0, ne = 0;
  for (int c = c0; c < c1; ++c) {
    const uint32_t key = ck[c];
    ng += key > kth ? 1u : 0u;
    ne += key == kth ? 1u : 0u;
  }
  uint32_t total;
  const uint32_t before = block_scan<uint32_t>(ng | (ne << 16), sc.scan, total);   // both totals < 2^16
  int g = static_cast<int>(before & 0xFFFFu), e = static_cast<int>(before >> 16);
  for (int c = c0; c < c1; ++c) {
    const uint32_t key = ck[c];
    if (key > kth) {
      sc.selq[g + min(e, need)] = static_cast<uint16_t>(c);
      ++g;
    } else if (key == kth) {
      if (e < need) sc.selq[g + e] = static_cast<uint16_t>(c);
      ++e;
    }
  }
  __syncthreads();
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
  int32_t warm;         // 1: the grid has one more row of CTAs, the first (see topk_chunk_kernel)
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

// Stage 1 (and the whole selection for rows of up to one chunk).  Thread t
// holds the chunk's 16-byte groups t, t + 1024, t + 2048, t + 3072 (group j:
// positions 4 (1024 j + t) .. + 3).
__global__ void __launch_bounds__(kThreads, 1) topk_chunk_kernel(const TopkParams p) {
  extern __shared__ __align__(128) uint8_t topk_smem[];
  Scratch& sc = *reinterpret_cast<Scratch*>(topk_smem);
  uint32_t* ck = reinterpret_cast<uint32_t*>(topk_smem + kScratchBytes);
  uint16_t* cp = reinterpret_cast<uint16_t*>(topk_smem + kScratchBytes + kChunk * 4);
  griddep_launch();
  // With p.warm, CTA (0, 0) selects from a synthetic row and writes nothing.
  // It is scheduled first and needs nothing from the previous kernel, so when
  // that kernel leaves an SM free it runs while the scores are still being
  // computed, and brings the selection's instructions into L2: after an idle
  // stretch they would otherwise be fetched from memory, one stretch at a
  // time, by every CTA -- which costs the selection more than its arithmetic.
  const bool dry = p.warm && blockIdx.y == 0;
  if (p.warm && blockIdx.y == 0 && blockIdx.x != 0) return;
  const int t = blockIdx.y - p.warm, c = dry ? 0 : blockIdx.x, tid = threadIdx.x;
  // the row's small inputs into L2 while the previous kernel finishes (a
  // prefetch is only a hint: later writes by that kernel are still seen)
  if (threadIdx.x == 0 && !dry) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p.n_vis + t));
    if (p.pf_base) asm volatile("prefetch.global.L2 [%0];" ::"l"(p.pf_seq + t));
  }
  sc.hist[2 * threadIdx.x] = 0u;
  sc.hist[2 * threadIdx.x + 1] = 0u;
  if (!dry) griddep_wait();
  const int lo = c * kChunk;
  // the warm-up CTA reads (and then ignores) up to the first 64 KB of the KV
  // pool, which nothing writes during the step, so the load code is warm as well
  const float* row = dry ? reinterpret_cast<const float*>(p.pf_base)
                         : p.logits + static_cast<int64_t>(t) * p.logits_stride + lo;
  // The chunk's scores go out together with the row's length: every position
  // below n_max lies inside the row, so the loads (four coalesced 16-byte
  // loads per thread, clamped addresses) need not wait for n.
  const int mcap = dry ? static_cast<int>(min(static_cast<int64_t>(kChunk), p.pf_num_pages * p.pf_page_stride / 4))
                       : min(p.n_max, lo + kChunk) - lo;
  float x[kPer];
  {
    float4 v[4];
    if (mcap > 0 && (dry || p.vec_logits)) {
      const float4* r4 = reinterpret_cast<const float4*>(row);
      const int last = (mcap - 1) >> 2;
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = __ldg(r4 + min(kThreads * j + tid, last));
    } else if (mcap > 0) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int q = 4 * (kThreads * j + tid);
        v[j] = make_float4(__ldg(row + min(q, mcap - 1)), __ldg(row + min(q + 1, mcap - 1)),
                           __ldg(row + min(q + 2, mcap - 1)), __ldg(row + min(q + 3, mcap - 1)));
      }
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[4 * j] = v[j].x;
      x[4 * j + 1] = v[j].y;
      x[4 * j + 2] = v[j].z;
      x[4 * j + 3] = v[j].w;
    }
    if (dry) {   // distinct-enough synthetic scores: the common path of the selection
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        asm volatile("" ::"f"(v[j].x), "f"(v[j].y), "f"(v[j].z), "f"(v[j].w));   // the loads stay in this path
        const uint32_t h = static_cast<uint32_t>(4 * (kThreads * j + tid)) * 2654435761u;
        x[4 * j] = static_cast<float>((h >> 8) & 0xFFFFFu);
        x[4 * j + 1] = static_cast<float>(((h * 3u) >> 8) & 0xFFFFFu);
        x[4 * j + 2] = static_cast<float>(((h * 5u) >> 8) & 0xFFFFFu);
        x[4 * j + 3] = static_cast<float>(((h * 7u) >> 8) & 0xFFFFFu);
      }
    }
  }
  const int seq = (!dry && p.pf_base) ? __ldg(p.pf_seq + t) : 0;   // for the row prefetches at the end
  const int n = dry ? kChunk : clamp_n(p, t);
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
  const int m = min(n, lo + kChunk) - lo;
  const int64_t cbase = (static_cast<int64_t>(t) * p.nchunks + c) * p.k;
  if (nch > 1 && m <= p.k) {  // a short tail chunk: every entry is a candidate
    for (int i = tid; i < m; i += kThreads) {
      p.cand_key[cbase + i] = order_key(__ldg(row + i));
      p.cand_idx[cbase + i] = lo + i;
    }
    return;
  }
  // the page-table row of the prefetch pool: loaded while the selection runs,
  // staged in shared memory after it
  const bool pt_stage = !dry && nch == 1 && p.pf_base != nullptr && p.pf_pt_stride <= kPtCache;
  int32_t ptv = 0;
  uint32_t valid = 0u;   // bit 4 j + i: position 4 (1024 j + tid) + i < m
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int left = m - 4 * (kThreads * j + tid);
    valid |= (left >= 4 ? 0xFu : (left > 0 ? (1u << left) - 1u : 0u)) << (4 * j);
  }
  // ---- 1. bound (NaN scores are the lowest keys, 0)
  float tm = -INFINITY;
  bool num = false;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const bool v = (valid >> i & 1u) && !isnan(x[i]);
    tm = v ? fmaxf(tm, x[i]) : tm;
    num = num || v;
  }
  const bool holds = valid != 0u;
  uint32_t lo_key, mx;
  block_bound(num ? order_key(tm) : 0u, holds, p.k, sc, lo_key, mx);
  if (pt_stage && tid < p.pf_pt_stride) ptv = __ldg(p.pf_pt + static_cast<int64_t>(seq) * p.pf_pt_stride + tid);
  // ---- 2. contenders: count per group, packed scan (group j in bits 16 j ..), compaction + histogram
  const float bf = key_float(lo_key);
  const bool all = lo_key == 0u;   // NaN scores contend too
  uint32_t cm = 0u;
#pragma unroll
  for (int i = 0; i < kPer; ++i) cm |= ((valid >> i & 1u) && (all || x[i] >= bf) ? 1u : 0u) << i;
  unsigned long long cnt = 0ull;
#pragma unroll
  for (int j = 0; j < 4; ++j) cnt |= static_cast<unsigned long long>(__popc(cm >> (4 * j) & 0xFu)) << (16 * j);
  unsigned long long tot64;
  const unsigned long long before = block_scan<unsigned long long>(cnt, sc.scan64, tot64);
  Digits d;
  const bool hist = lo_key != mx;
  if (hist) d.first(lo_key, mx);
  int C = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    int o = C + static_cast<int>((before >> (16 * j)) & 0xFFFFu);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (cm >> (4 * j + i) & 1u) {
        const uint32_t key = order_key(x[4 * j + i]);
        ck[o] = key;
        cp[o] = static_cast<uint16_t>(4 * (kThreads * j + tid) + i);
        if (hist) atomicAdd(&sc.hist[(key >> d.lo) & d.dmask], 1u);
        ++o;
      }
    }
    C += static_cast<int>((tot64 >> (16 * j)) & 0xFFFFu);
  }
  __syncthreads();
  // ---- 3, 4
  select_contenders(ck, C, p.k, lo_key, mx, sc);
  if (dry && p.pf_pt_stride > kPtCache) return;   // its prefetches would read a page table
  if (pt_stage) {
    if (tid < p.pf_pt_stride) sc.pt[tid] = ptv;
    __syncthreads();
  }
  for (int r = tid; r < p.k; r += kThreads) {
    const int q = sc.selq[r];
    const int e = lo + cp[q];
    if (nch == 1) {
      if (!dry) out[r] = e;
      prefetch_row(p, t, e, sc);   // warm-up: page ids from unstaged shared memory, range-checked hints only
    } else {
      p.cand_key[cbase + r] = ck[q];
      p.cand_idx[cbase + r] = e;
    }
  }
}

// Stage 2: the row's candidates (each chunk's top-k, contiguous in chunk
// order) -> top-k.  The m candidates are spread evenly over the block: thread t
// holds the `per` consecutive candidates from per * t (per = ceil(m / 1024)
// rounded up to a multiple of 4, at most 32), so the lower bound of step 1 has
// a thread maximum from as many threads as possible.
__global__ void __launch_bounds__(kThreads, 1) topk_merge_kernel(const TopkParams p) {
  extern __shared__ __align__(128) uint8_t topk_smem[];
  Scratch& sc = *reinterpret_cast<Scratch*>(topk_smem);
  uint32_t* ck = reinterpret_cast<uint32_t*>(topk_smem + kScratchBytes);
  uint16_t* cp = reinterpret_cast<uint16_t*>(topk_smem + kScratchBytes + kMaxCand * 4);
  griddep_launch();
  sc.hist[2 * threadIdx.x] = 0u;
  sc.hist[2 * threadIdx.x + 1] = 0u;
  griddep_wait();
  const int t = blockIdx.x, tid = threadIdx.x;
  const int n = clamp_n(p, t);
  if (n <= p.k) return;  // includes rows left untouched (n < 0)
  const int nch = (n + kChunk - 1) / kChunk;
  if (nch <= 1) return;
  const int m = (nch - 1) * p.k + min(n - (nch - 1) * kChunk, p.k);
  const int64_t rbase = static_cast<int64_t>(t) * p.nchunks * p.k;
  const uint32_t* ckg = p.cand_key + rbase;
  const int per = min(kMergePer, (((m + kThreads - 1) / kThreads) + 3) & ~3);
  const int base = per * tid;
  uint32_t key[kMergePer];
  if (p.vec_cand) {
    const uint4* c4 = reinterpret_cast<const uint4*>(ckg);
    const int last = (m - 1) >> 2;
#pragma unroll
    for (int j = 0; j < kMergePer / 4; ++j) {
      const uint4 v = 4 * j < per ? __ldg(c4 + min(base / 4 + j, last)) : make_uint4(0u, 0u, 0u, 0u);
      key[4 * j] = v.x;
      key[4 * j + 1] = v.y;
      key[4 * j + 2] = v.z;
      key[4 * j + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < kMergePer; ++i) key[i] = i < per ? __ldg(ckg + min(base + i, m - 1)) : 0u;
  }
  // the page-table row of the prefetch pool: loaded while the selection runs,
  // staged in shared memory after it
  const bool pt_stage = p.pf_base != nullptr && p.pf_pt_stride <= kPtCache;
  const int seq = pt_stage ? __ldg(p.pf_seq + t) : 0;
  int32_t ptv = 0;
  const int cnt = max(0, min(per, m - base));   // this thread's candidates
  const uint32_t valid = cnt >= 32 ? 0xFFFFFFFFu : (1u << cnt) - 1u;
  uint32_t tmax = 0u;
#pragma unroll
  for (int i = 0; i < kMergePer; ++i)
    if (valid >> i & 1u) tmax = max(tmax, key[i]);
  uint32_t lo_key, mx;
  block_bound(tmax, valid != 0u, p.k, sc, lo_key, mx);
  if (pt_stage && tid < p.pf_pt_stride) ptv = __ldg(p.pf_pt + static_cast<int64_t>(seq) * p.pf_pt_stride + tid);
  uint32_t cm = 0u;
#pragma unroll
  for (int i = 0; i < kMergePer; ++i) cm |= ((valid >> i & 1u) && key[i] >= lo_key ? 1u : 0u) << i;
  uint32_t C;
  int o = static_cast<int>(block_scan<uint32_t>(static_cast<uint32_t>(__popc(cm)), sc.scan, C));
  Digits d;
  const bool hist = lo_key != mx;
  if (hist) d.first(lo_key, mx);
#pragma unroll
  for (int i = 0; i < kMergePer; ++i) {
    if (cm >> i & 1u) {
      ck[o] = key[i];
      cp[o] = static_cast<uint16_t>(base + i);
      if (hist) atomicAdd(&sc.hist[(key[i] >> d.lo) & d.dmask], 1u);
      ++o;
    }
  }
  __syncthreads();
  int32_t* out = p.idx + static_cast<int64_t>(t) * p.idx_stride;
  const int32_t* ci = p.cand_idx + rbase;
  select_contenders(ck, static_cast<int>(C), p.k, lo_key, mx, sc);
  if (pt_stage) {
    if (tid < p.pf_pt_stride) sc.pt[tid] = ptv;
    __syncthreads();
  }
  for (int r = tid; r < p.k; r += kThreads) {
    const int e = __ldg(ci + cp[sc.selq[r]]);
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
  if (!smem_attr_once(dev, 13, reinterpret_cast<const void*>(topk_chunk_kernel), kChunkSmem) ||
      !smem_attr_once(dev, 14, reinterpret_cast<const void*>(topk_merge_kernel), kMergeSmem))
    return DSV4SA_ERR_CUDA;
  p.warm = (prefetch && prefetch->pool) ? 1 : 0;   // the serving form: the warm-up CTA (see the kernel)
  if (launch_pdl(topk_chunk_kernel, dim3(nch, T + p.warm), dim3(kThreads), kChunkSmem, stream, p) != cudaSuccess)
    return DSV4SA_ERR_CUDA;
  if (nch > 1 && launch_pdl(topk_merge_kernel, dim3(T), dim3(kThreads), kMergeSmem, stream, p) != cudaSuccess)
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
