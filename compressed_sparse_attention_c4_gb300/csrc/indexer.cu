// indexer.cu -- C4 indexer logits on the sm_103a tensor cores.
//
// Computes, for every query t and visible compressed entry s < n_vis[t],
//   I[t, s] = sum_h w[t, h] * ReLU( sum_d qhat[t, h, d] * khat[s, d] )
// ("DeepSeek-V4 全面解读" §2.10 Indexer steps 6-8; "DeepSeek-V4 in SGLang"
// 算法2 Paged MQA Logits: the cheap FP8 scoring pass over a paged cache).
//
// Design (one GPU, persistent CTAs, warp specialised; 20 warps):
//   * The unit of work is a tile of 128 consecutive entries of one query (two
//     64-slot pages).  All (query, tile) pairs form one flat list that is cut
//     into equal contiguous ranges, one per CTA, so ragged n_vis balances.
//   * Every role handles a tile in a fixed, short sequence of steps, and the
//     roles that are slowest per tile are split over several warps that take
//     tiles in turn: a single thread cannot issue a tile's copies or MMAs, or
//     a warp finish its epilogue, in the time HBM (decode) or L2 (prefill,
//     where all queries read the same keys) delivers the next tile.
//   * warps 16 and 17 (producers, alternate tiles): lanes 0-3 wait for a free
//     stage of an 8-stage ring and issue the tile's four copies side by side --
//     the two key pages (3-D TMA box per page, 128-byte swizzle) and their fp32
//     scales (1-D bulk copies into a 16-slot scale ring).  Lane u holds the
//     page ids of the producer's tile 32r + u of round r and loads those of
//     round r + 1 while round r is issued, so no copy waits on a global load.
//   * warps 18 and 19 (MMA issuers, alternate tiles): one thread each issues
//     tcgen05.mma kind::f8f6f4, M = 128 entries, N = Hi (padded to 16), K = 32
//     per instruction, two instructions per 64-dim scale block into two TMEM
//     accumulators (the block scales of q and k differ per block, so the
//     blocks cannot share an accumulator), one commit per tile.  Accumulators
//     rotate over 4 TMEM stages (2 when Hi > 64).  Warp 18 also loads the q
//     blocks: query k + 1's (one TMA box of Hi rows, into the other of two q
//     buffers) when query k starts.
//   * warps 0-15 (four epilogue groups of 128 threads, tile i to group i % 4;
//     two groups, i % 2, when Hi > 64 and only 2 accumulator stages fit):
//     each thread owns one TMEM lane = one entry; once the tile's MMAs are
//     complete the group frees its key stage, then applies the per-entry key
//     scales, the per-head q scales, ReLU, the head weights and the sum over
//     heads with packed fp32x2 arithmetic, and writes one logit.
#include "common.cuh"
#include "dsv4sa_internal.h"

namespace dsv4sa {
namespace {

constexpr int kStages = 8;
constexpr int kTileRows = 128;
constexpr int kKeyPage = 64 * 128;      // bytes of FP8 keys per page
constexpr int kScalePage = 64 * 8;      // bytes of fp32 scales per page (2 per slot)
constexpr int kStageBytes = 2 * kKeyPage;   // 16384: the keys of a tile's two pages
// The tiles' key scales live in a ring of their own, 16 tiles deep, so a key
// stage is free again as soon as the tile's MMAs are complete.  Slot i % 16 is
// next written by the copy of tile i + 16, which waits for key stage i % 8 to
// be released by the epilogue of tile i + 8; that tile belongs to the same
// epilogue group as tile i (the groups take tiles i % 4, or i % 2 when Hi > 64,
// in order), so the group has read tile i's scales by then.
constexpr int kScaleSlots = 16;
constexpr int kScaleSlotBytes = 2 * kScalePage;
constexpr int kMaxHiP = 128;
// FP8 kernel: 20 warps (5 per SM sub-partition, which leaves 96 registers a
// thread).  Warps 0-15 are four epilogue groups of four (group g = warp / 4
// takes the tiles i % 4 == g; warp % 4 is its TMEM lane quarter), 16 and 17
// the producers (alternate tiles), 18 and 19 the MMA issuers (alternate
// tiles; warp 18 also loads the queries' q blocks).
// Tile i uses accumulator stage i % 4 (i % 2 when Hi > 64); the epilogue
// group of tile i must also own tile i - 4 (i - 2), the previous user of that
// stage, so its parity waits on the stage's barriers never run two phases
// ahead: the number of groups in use equals the number of stages (groups 2
// and 3 stay idle when Hi > 64).
constexpr int kEpiGroups = 4;
constexpr int kProdWarp = 16;
constexpr int kMmaWarp = 18;
constexpr int kWarps8 = 20;
constexpr int kThreads8 = kWarps8 * 32;
// FP4 kernel: 12 warps (roles below).
constexpr int kThreads = 384;
constexpr int kWarps = kThreads / 32;

struct IndexerParams {
  const int32_t* page_table;
  const int32_t* q_seq;
  const int32_t* n_vis;
  const uint8_t* q_fp8;     // FP8 kernel: e4m3 codes [T][Hi][128]; FP4 kernel: e2m1 codes [T][Hi][64]
  const float* q_scale;     // FP8 kernel: [T][Hi][2]
  const uint8_t* q_e8m0;    // FP4 kernel: [T][Hi][4]
  const float* w;
  const uint8_t* scale_base;   // pool base + scale block offset
  float* logits;
  int64_t page_stride;
  int64_t num_pages;
  int64_t logits_stride;
  int32_t pt_stride;
  int32_t T;
  int32_t Hi;
  int32_t HiP;
  int32_t n_max;
};

struct SmemLayout {
  static constexpr int kStageOff = 0;
  static constexpr int kScaleOff = kStages * kStageBytes;             // kScaleSlots x 2 pages of scales
  static constexpr int kQOff = kScaleOff + kScaleSlots * kScaleSlotBytes;   // 2 q buffers
  static constexpr int kConstOff = kQOff + 2 * kMaxHiP * 128;         // per WG: q scales, weights
  static constexpr int kConstBytes = kMaxHiP / 2 * 16 + kMaxHiP / 2 * 8 + kMaxHiP / 2 * 16 + 16;
  static constexpr int kBarOff = kConstOff + kEpiGroups * kConstBytes;
  static constexpr int kNumBars = 2 * kStages + 12;
  static constexpr int kTmemOff = kBarOff + kNumBars * 8;
  static constexpr int kScanOff = kTmemOff + 16;                      // ints
  static constexpr int kBytes = kScanOff + (kWarps8 + 8) * 4;
};
constexpr int kSmemBytes = SmemLayout::kBytes + 1024;  // + alignment slack

__device__ __forceinline__ int clamp_n(const IndexerParams& p, int n) {
  return n < 0 ? 0 : (n > p.n_max ? p.n_max : n);
}
__device__ __forceinline__ int tiles_of(const IndexerParams& p, int t) {
  return (clamp_n(p, __ldg(p.n_vis + t)) + kTileRows - 1) / kTileRows;
}

// Position in the flat (query, tile) list.
struct Cursor {
  int t;
  int j;
  int nt;   // tiles of query t
  int ord;  // queries with tiles passed since the start of the walk
  __device__ __forceinline__ void advance(const IndexerParams& p) {
    ++j;
    if (j >= nt) {
      while (j >= nt && t < p.T) {
        ++t;
        j = 0;
        nt = (t < p.T) ? tiles_of(p, t) : 0;
      }
      ++ord;
    }
  }
  // m steps at once (queries without tiles are skipped as by advance)
  __device__ __forceinline__ void advance_by(const IndexerParams& p, int m) {
    j += m;
    while (j >= nt && t < p.T) {
      j -= nt;
      ++t;
      nt = (t < p.T) ? tiles_of(p, t) : 0;
      if (nt > 0) ++ord;
    }
  }
};

// bar.red.or over the n threads of named barrier id: whether any passed true
// (also a barrier for them).
__device__ __forceinline__ bool group_any_ix(bool v, uint32_t id, uint32_t n) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(v ? 1u : 0u), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// Exclusive scan over the block (NT threads); returns the total.
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

// Work range of this CTA: tiles [start, start + count) of the flat (query,
// tile) list cut evenly over the grid, and the cursor at `start`, found by a
// block-wide scan of the queries' tile counts.  All threads call it; it ends
// with a barrier (preceded by a tensor-core fence, so TMEM allocation results
// are visible after it).
template <int NT>
__device__ void work_range(const IndexerParams& p, int* scan, int& count, Cursor& c0) {
  constexpr int kThreads = NT;
  int* res = scan + NT / 32;
  if (threadIdx.x == 0) {
    res[0] = p.T;
    res[1] = 0;
  }
  long long start, end;
  if (p.T <= kThreads) {
    // one pass: every query's tile count, its exclusive prefix and the total
    const int t = threadIdx.x;
    if (t < p.T) asm volatile("prefetch.global.L1 [%0];" ::"l"(p.q_seq + t));   // read right after
    const int nt = t < p.T ? tiles_of(p, t) : 0;
    int tot;
    const int before = block_scan<NT>(nt, scan, tot);
    start = static_cast<long long>(tot) * blockIdx.x / gridDim.x;
    end = static_cast<long long>(tot) * (blockIdx.x + 1) / gridDim.x;
    if (nt > 0 && start >= before && start < before + nt) {
      res[0] = t;
      res[1] = static_cast<int>(start - before);
    }
  } else {
    long long total = 0;
    for (int base = 0; base < p.T; base += kThreads) {
      const int t = base + threadIdx.x;
      int tot;
      block_scan<NT>(t < p.T ? tiles_of(p, t) : 0, scan, tot);
      total += tot;
    }
    start = total * blockIdx.x / gridDim.x;
    end = total * (blockIdx.x + 1) / gridDim.x;
    long long acc = 0;
    for (int base = 0; base < p.T; base += kThreads) {
      const int t = base + threadIdx.x;
      const int nt = t < p.T ? tiles_of(p, t) : 0;
      int tot;
      const int before = block_scan<NT>(nt, scan, tot);
      if (nt > 0 && start >= acc + before && start < acc + before + nt) {
        res[0] = t;
        res[1] = static_cast<int>(start - acc - before);
      }
      acc += tot;
    }
  }
  count = static_cast<int>(end - start);
  tc_fence_before();
  __syncthreads();
  c0.t = res[0];
  c0.j = res[1];
  c0.nt = (c0.t < p.T) ? tiles_of(p, c0.t) : 0;
  c0.ord = 0;
}

__global__ void __launch_bounds__(kThreads8, 1)
    indexer_logits_kernel(const __grid_constant__ CUtensorMap key_map, const __grid_constant__ CUtensorMap q_map,
                          const IndexerParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SmemLayout::kBarOff);
  uint64_t* full = bars;                    // [kStages] TMA -> MMA
  uint64_t* empty = bars + kStages;         // [kStages] epilogue (the tile's MMAs are complete) -> TMA
  uint64_t* acc_full = bars + 2 * kStages;  // [4] MMA -> epilogue
  uint64_t* acc_empty = acc_full + 4;       // [4] epilogue -> MMA
  uint64_t* q_full = acc_full + 8;          // [2] q block TMA -> MMA
  uint64_t* q_empty = acc_full + 10;        // [2] both MMA warps -> q block TMA
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + SmemLayout::kTmemOff);
  int* scan = reinterpret_cast<int*>(smem + SmemLayout::kScanOff);   // [kWarps8] scan scratch, then results

  const int warp = static_cast<int>(warp_id());
  const int lane = static_cast<int>(lane_id());
  const int HiP = p.HiP;
  const int lg_acc = (HiP <= 64) ? 2 : 1;             // log2 of the TMEM accumulator stages (2 x HiP columns each)
  const int nacc = 1 << lg_acc;
  const uint32_t tmem_cols = (nacc * 2 * HiP <= 256) ? 256u : 512u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);   // one thread of the tile's epilogue group
    }
    for (int a = 0; a < 4; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 4);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&q_full[a], 1);
      mbar_init(&q_empty[a], 2);   // each MMA warp commits once per query
    }
    fence_mbar_init();
    prefetch_tensormap(&key_map);
    prefetch_tensormap(&q_map);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_holder, tmem_cols);
    tmem_relinquish();
  }
  // The q buffers start as zeros: a q block fills rows [0, Hi), so the rows of
  // padded heads (Hi to HiP) stay zero.
  for (int u = threadIdx.x; u < 2 * kMaxHiP * 128 / 16; u += kThreads8)
    reinterpret_cast<uint4*>(smem + SmemLayout::kQOff)[u] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();   // before the tensor core reads them (the barrier in work_range orders it)
  griddep_launch();
  // The small inputs into L2 while the previous kernel finishes: the lengths and
  // sequence ids every CTA scans first, and this CTA's share of the queries'
  // FP8 q, scales and weights (a prefetch is only a hint: later writes by that
  // kernel are still seen).  Every address lies inside its buffer.
  {
    const int tid = threadIdx.x;
    for (int t = tid * 32; t < p.T; t += kThreads8 * 32) {
      asm volatile("prefetch.global.L2 [%0];" ::"l"(p.n_vis + t));
      asm volatile("prefetch.global.L2 [%0];" ::"l"(p.q_seq + t));
    }
    const int64_t th = static_cast<int64_t>(p.T) * p.Hi;
    const int64_t q_lines = (th * 128 + 127) / 128, s_lines = (th * 8 + 127) / 128, w_lines = (th * 4 + 127) / 128;
    const int64_t step = static_cast<int64_t>(gridDim.x) * kThreads8;
    for (int64_t l = blockIdx.x + static_cast<int64_t>(gridDim.x) * tid; l < q_lines + s_lines + w_lines; l += step) {
      const uint8_t* a = l < q_lines ? p.q_fp8 + l * 128
                         : l < q_lines + s_lines ? reinterpret_cast<const uint8_t*>(p.q_scale) + (l - q_lines) * 128
                                                 : reinterpret_cast<const uint8_t*>(p.w) + (l - q_lines - s_lines) * 128;
      asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
    }
  }
  griddep_wait();  // inputs may come from the previous kernel of the stream

  int count;
  Cursor c0;
  work_range<kThreads8>(p, scan, count, c0);   // ends with a barrier
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (count > 0) {
    if (warp == kProdWarp || warp == kProdWarp + 1) {
      // ================= producers: key pages + scales, alternate tiles =================
      const int pw = warp - kProdWarp;
      const int mine = count > pw ? (count - pw + 1) / 2 : 0;   // tiles pw, pw + 2, ...
      Cursor cl = c0;                                            // this lane's next own tile
      cl.advance_by(p, pw + 2 * lane);
      // page ids of own tile k (k % 32 == lane); the cursor then moves to own tile k + 32
      auto fetch = [&](int k, int& pid0, int& pid1, int& second) {
        pid0 = pid1 = second = 0;
        if (k < mine) {
          const int n = clamp_n(p, __ldg(p.n_vis + cl.t));
          const int32_t* row = p.page_table + static_cast<int64_t>(__ldg(p.q_seq + cl.t)) * p.pt_stride;
          pid0 = __ldg(row + min(2 * cl.j, p.pt_stride - 1));
          pid1 = __ldg(row + min(2 * cl.j + 1, p.pt_stride - 1));
          second = (cl.j * kTileRows + 64) < n ? 1 : 0;
          cl.advance_by(p, 64);
        }
      };
      int c_pid0, c_pid1, c_sec, n_pid0, n_pid1, n_sec;
      fetch(lane, c_pid0, c_pid1, c_sec);
      fetch(32 + lane, n_pid0, n_pid1, n_sec);
      const uint64_t pol = l2_evict_first_policy();
      int issued = 0;
      bool ok = true;
      for (int r = 0; 32 * r < mine && ok; ++r) {
        if (r > 0) {
          c_pid0 = n_pid0;
          c_pid1 = n_pid1;
          c_sec = n_sec;
          fetch(32 * (r + 1) + lane, n_pid0, n_pid1, n_sec);
        }
        const int kn = min(32, mine - 32 * r);
        for (int u = 0; u < kn; ++u) {
          const int pid0 = __shfl_sync(0xffffffffu, c_pid0, u);
          const int pid1 = __shfl_sync(0xffffffffu, c_pid1, u);
          const bool second = __shfl_sync(0xffffffffu, c_sec, u) != 0;
          const int i = pw + 2 * (32 * r + u);
          const int s = i & (kStages - 1);
          // lanes 0-3 wait for the stage and issue the tile's four copies side
          // by side: lanes 0, 1 the key pages (TMA), lanes 2, 3 their scales
          int okl = 1;
          if (lane < 4) okl = mbar_wait(&empty[s], ((i / kStages) & 1) ^ 1) ? 1 : 0;
          ok = __all_sync(0xffffffffu, okl) != 0;
          if (!ok) break;
          if (lane < 4) {
            const int pg = lane & 1;
            const bool want = pg == 0 || second;
            int pid = pg ? pid1 : pid0;
            if (pid < 0 || pid >= p.num_pages) {
              if (want && lane < 2) raise_error(kErrIndex);
              pid = 0;
            }
            if (lane == 0)
              mbar_arrive_expect_tx(&full[s], second ? 2 * (kKeyPage + kScalePage) : (kKeyPage + kScalePage));
            __syncwarp(0xFu);   // the expected bytes are posted before any copy lands
            if (want) {
              // the keys are read once per step: evicted first, so the logits
              // this kernel writes stay in L2 for the top-k
              if (lane < 2) {
                tma_load_3d_hint(smem + SmemLayout::kStageOff + s * kStageBytes + pg * kKeyPage, &key_map, &full[s], 0,
                                 0, pid, pol);
              } else {
                bulk_load_hint(smem + SmemLayout::kScaleOff + (i % kScaleSlots) * kScaleSlotBytes + pg * kScalePage,
                               p.scale_base + pid * p.page_stride, kScalePage, &full[s], pol);
              }
            }
          }
          ++issued;
        }
      }
      // drain: wait (bounded) for the copies this warp issued before leaving
      if (lane == 0)
        for (int k = (issued > kStages / 2 ? issued - kStages / 2 : 0); k < issued; ++k) {
          const int i = pw + 2 * k;
          mbar_wait(&full[i % kStages], (i / kStages) & 1);
        }
      __syncwarp();
    } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
      // ================= MMA issuers, alternate tiles =================
      // Each walks its own tiles only.  The q buffers alternate per query of
      // the CTA's range (ordinal k in buffer k % 2); a warp commits once for
      // every query of the range as it passes it, so buffer k % 2 is refilled
      // (with query k + 2) only after both warps' MMAs on query k are done.
      // Before committing query k a warp waits until query k - 2's commits
      // are complete, so every phase of a buffer's barrier collects exactly the
      // two commits of one query.  Warp 18 also loads the q blocks (one TMA
      // box of Hi rows), at most two queries ahead of its tiles.
      const int mw = warp - kMmaWarp;
      if (lane == 0) {
        const uint32_t idesc = make_idesc(kFmtE4M3, kFmtE4M3, 0, 0, 128, HiP);
        const uint64_t a_desc0 = smem_desc_sw128(smem_u32(smem + SmemLayout::kStageOff), 16, 1024);
        const uint64_t b_desc0 = smem_desc_sw128(smem_u32(smem + SmemLayout::kQOff), 16, 1024);
        const uint32_t q_bytes = static_cast<uint32_t>(p.Hi) * 128u;
        Cursor ce = c0;
        ce.advance_by(p, count - 1);
        const int n_q = ce.ord + 1;   // queries with tiles in the range
        auto prior_done = [&](int k) {   // the commits of query k - 2 (same buffer) are complete
          return mbar_wait(&q_empty[k & 1], ((k >> 1) & 1) ^ 1);
        };
        int q_loaded = 0, q_t = c0.t;
        auto load_q = [&]() -> bool {
          const int k = q_loaded;
          if (k > 0) {
            ++q_t;
            while (q_t + 1 < p.T && tiles_of(p, q_t) == 0) ++q_t;
          }
          if (!prior_done(k)) return false;
          mbar_arrive_expect_tx(&q_full[k & 1], q_bytes);
          tma_load_3d(smem + SmemLayout::kQOff + (k & 1) * (kMaxHiP * 128), &q_map, &q_full[k & 1], 0, 0, q_t);
          ++q_loaded;
          return true;
        };
        int committed = 0, waited = -1, last = -1;
        auto commit_to = [&](int k) -> bool {   // commit every query before ordinal k
          for (; committed < k; ++committed) {
            if (!prior_done(committed)) return false;
            mma_commit(&q_empty[committed & 1]);
          }
          return true;
        };
        Cursor c = c0;
        if (mw < count) c.advance_by(p, mw);
        bool ok = true;
        for (int i = mw; i < count; i += 2) {
          ok = commit_to(c.ord);
          if (mw == 0)
            while (ok && q_loaded < min(c.ord + 2, n_q)) ok = load_q();
          if (ok && waited != c.ord) {
            ok = mbar_wait(&q_full[c.ord & 1], (c.ord >> 1) & 1);
            waited = c.ord;
          }
          const int s = i & (kStages - 1);
          const int a = i & (nacc - 1);
          ok = ok && mbar_wait(&full[s], (i / kStages) & 1) && mbar_wait(&acc_empty[a], ((i >> lg_acc) & 1) ^ 1);
          if (!ok) break;
          tc_fence_after();
          // descriptor start addresses advance in 16-byte units: stage s, q
          // buffer of this query, 32-byte steps along K
          const uint64_t ad = a_desc0 + static_cast<uint64_t>(s * (kStageBytes >> 4));
          const uint64_t bd = b_desc0 + static_cast<uint64_t>((c.ord & 1) * ((kMaxHiP * 128) >> 4));
          const uint32_t d0 = tmem_base + static_cast<uint32_t>(a * 2 * HiP);
#pragma unroll
          for (int blk = 0; blk < 2; ++blk) {
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
              const uint64_t koff = static_cast<uint64_t>((blk * 2 + kk) * 2);
              mma_f8f6f4(d0 + blk * HiP, ad + koff, bd + koff, idesc, kk);
            }
          }
          mma_commit(&acc_full[a]);
          last = i;
          if (i + 2 < count) c.advance_by(p, 2);
        }
        if (ok) commit_to(n_q);
        // make sure no MMA is still writing TMEM when the CTA deallocates it
        if (last >= 0) mbar_wait(&acc_full[last & (nacc - 1)], (last >> lg_acc) & 1);
      }
      __syncwarp();
    } else {
      // ================= epilogue groups =================
      const int e = warp >> 2;               // group: tiles with i % ngroups == e
      const int ngroups = nacc;              // one group per accumulator stage
      const int g = warp & 3;                // TMEM lane quarter of this warp
      const int row = g * 32 + lane;         // entry within the tile
      const int tid_wg = row;                // thread within the group
      uint8_t* cbase = smem + SmemLayout::kConstOff + e * SmemLayout::kConstBytes;
      float4* cq = reinterpret_cast<float4*>(cbase);                          // {q0[h], q0[h+1], q1[h], q1[h+1]}
      float2* cw = reinterpret_cast<float2*>(cbase + kMaxHiP / 2 * 16);       // {w[h], w[h+1]}
      // {r[h], r[h+1], c[h], c[h+1]}: r = q1 / q0, c = w * q0 (the ratio form below)
      float4* cr = reinterpret_cast<float4*>(cbase + kMaxHiP / 2 * 24);
      bool ratio_q = false;   // every head of the query has q0 > 0 and a finite ratio
      Cursor c = c0;
      if (e < count) c.advance_by(p, e);
      int cur_t = -1, n = 0;
      bool dead = false;
      for (int i = e; e < ngroups && i < count; i += ngroups) {
        if (c.t != cur_t) {
          named_barrier_sync(1 + e, 128);
          for (int hp = tid_wg; hp < kMaxHiP / 2; hp += 128) {   // pairs past Hi stay zero
            float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
            float2 ww = make_float2(0.f, 0.f);
            const int64_t qh = static_cast<int64_t>(c.t) * p.Hi + 2 * hp;
            if (2 * hp < p.Hi) {
              q.x = __ldg(p.q_scale + 2 * qh);
              q.z = __ldg(p.q_scale + 2 * qh + 1);
              ww.x = __ldg(p.w + qh);
            }
            if (2 * hp + 1 < p.Hi) {
              q.y = __ldg(p.q_scale + 2 * qh + 2);
              q.w = __ldg(p.q_scale + 2 * qh + 3);
              ww.y = __ldg(p.w + qh + 1);
            }
            cq[hp] = q;
            cw[hp] = ww;
          }
          bool bad = false;
          for (int hp = tid_wg; hp < kMaxHiP / 2; hp += 128) {
            const float4 q = cq[hp];
            const float2 ww = cw[hp];
            // padded heads (q = 0, w = 0) take r = 0, c = 0: they add nothing either way
            const float r0 = q.x > 0.f ? q.z / q.x : 0.f, r1 = q.y > 0.f ? q.w / q.y : 0.f;
            const bool live0 = 2 * hp < p.Hi, live1 = 2 * hp + 1 < p.Hi;
            bad |= live0 && !(q.x > 0.f && isfinite(r0) && isfinite(ww.x * q.x));
            bad |= live1 && !(q.y > 0.f && isfinite(r1) && isfinite(ww.y * q.y));
            cr[hp] = make_float4(r0, r1, ww.x * q.x, ww.y * q.y);
          }
          ratio_q = !group_any_ix(bad, 1 + e, 128);   // also the barrier that publishes cq, cw, cr
          cur_t = c.t;
          n = clamp_n(p, __ldg(p.n_vis + c.t));
        }
        const int a = i & (nacc - 1);
        if (!dead) {
          const int okw = (lane == 0) ? (mbar_wait(&acc_full[a], (i >> lg_acc) & 1) ? 1 : 0) : 0;
          dead = __shfl_sync(0xffffffffu, okw, 0) == 0;
        }
        // a warp whose wait gave up (the error is raised) does no more work but
        // keeps walking its tiles, so the group's barriers stay matched
        if (dead) {
          if (i + ngroups < count) c.advance_by(p, ngroups);
          continue;
        }
        tc_fence_after();
        // the tile's MMAs are complete, so its key stage is free again
        if (lane == 0 && g == 0) mbar_arrive(&empty[i & (kStages - 1)]);
        const float2 sk = *reinterpret_cast<const float2*>(smem + SmemLayout::kScaleOff +
                                                           (i % kScaleSlots) * kScaleSlotBytes +
                                                           (row >> 6) * kScalePage + (row & 63) * 8);
        const float2 sk0 = make_float2(sk.x, sk.x), sk1 = make_float2(sk.y, sk.y);
        // Ratio form (k scale sk0 > 0, q scale q0 > 0): sk0 q0 D0 + sk1 q1 D1 =
        // sk0 q0 (D0 + alpha r D1) with alpha = sk1 / sk0, r = q1 / q0, so
        // w ReLU(.) = sk0 c ReLU(D0 + alpha r D1) with c = w q0: three packed
        // FMA-pipe operations per head pair instead of five.
        const float alpha = sk.y / sk.x;
        const bool ratio = ratio_q && sk.x > 0.f && isfinite(alpha);
        const float2 al = make_float2(alpha, alpha);
        float2 acc = make_float2(0.f, 0.f);
        const uint32_t tb = tmem_base + (static_cast<uint32_t>(g * 32) << 16) + static_cast<uint32_t>(a * 2 * HiP);
        for (int hc = 0; hc < HiP; hc += 16) {   // HiP is a multiple of 16
          float d0[16], d1[16];
          tmem_ld16(tb + hc, d0);
          tmem_ld16(tb + HiP + hc, d1);
          tmem_ld_wait();
          if (ratio) {
#pragma unroll
            for (int u = 0; u < 16; u += 2) {
              const float4 rc = cr[(hc + u) >> 1];
              const float2 gr = mul2(al, make_float2(rc.x, rc.y));
              float2 v = fma2(make_float2(d1[u], d1[u + 1]), gr, make_float2(d0[u], d0[u + 1]));
              v.x = fmaxf(v.x, 0.f);
              v.y = fmaxf(v.y, 0.f);
              acc = fma2(v, make_float2(rc.z, rc.w), acc);
            }
          } else {
#pragma unroll
            for (int u = 0; u < 16; u += 2) {
              const float4 q = cq[(hc + u) >> 1];
              const float2 ww = cw[(hc + u) >> 1];
              // v = sk0 * (q0 * D0) + sk1 * (q1 * D1) for heads (h, h+1)
              const float2 a0 = mul2(make_float2(d0[u], d0[u + 1]), make_float2(q.x, q.y));
              const float2 a1 = mul2(make_float2(d1[u], d1[u + 1]), make_float2(q.z, q.w));
              float2 v = fma2(a0, sk0, mul2(a1, sk1));
              v.x = fmaxf(v.x, 0.f);
              v.y = fmaxf(v.y, 0.f);
              acc = fma2(v, ww, acc);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[a]);
        const int sidx = c.j * kTileRows + row;
        if (sidx < n)
          p.logits[static_cast<int64_t>(c.t) * p.logits_stride + sidx] = ratio ? sk.x * (acc.x + acc.y) : acc.x + acc.y;
        if (i + ngroups < count) c.advance_by(p, ngroups);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, tmem_cols);
  }
}

// ---------------------------------------------------------------- FP4 keys and query
//
// The same logits over an IDXK_FP4 pool with an FP4 query ("DeepSeek-V4 全面解读"
// §2.10 Indexer step 3, FP4 quant-sim of q and k, and §3.5 fp4_quant_kernel;
// "tilelang量化内核拆解DeepSeek-V4.1-Flash-NVFP4的fp4_gemm与sparse_attn实现"
// §model.py 如何驱动: E2M1 values with one E8M0 scale per 32):
//   I[t, s] = sum_h w[t, h] * ReLU( sum_b 2^(eq[t,h,b] - 127) 2^(ek[s,b] - 127) D[t,h,s,b] ),
//   D[t,h,s,b] = sum_{d in block b} e2m1(q[t,h,d]) * e2m1(k[s,d])      (b = d / 32)
// Every E2M1 value is exactly an E4M3 value, so the block products run on the
// FP8 tensor-core instruction.  Each page (4352 B: codes, then E8M0 bytes)
// lands with one bulk copy; a conversion pass turns a tile's codes into E4M3
// rows in the MMA's 128-byte swizzled layout; each 32-value block has its own
// accumulator (one K = 32 instruction per block), so D stays exact and the
// power-of-two scales are applied in the epilogue.
// Warps 0 and 11 copy pages (alternate tiles; page ids read ahead as in the FP8
// kernel); warp 1 issues the MMAs; warps 2-5 and 6-9 are two groups of 128
// threads that take alternate tiles: each converts its tile (and stages the
// query's E4M3 rows and scale factors when the query changes), then runs the
// epilogue of the same tile once the MMA is done; thread = TMEM lane = tile row.
// Hi <= 64 (the accumulators of both groups fill the 512 TMEM columns).

constexpr int kF4MmaWarp = 1;                 // FP4 kernel roles: warps 0 and 11 copy, 1 issues MMAs
constexpr int kF4ProducerB = 11;
constexpr int kF4Page = 4352;                 // bytes of one IDXK_FP4 page: 64 x 64 codes + 64 x 4 E8M0
constexpr int kF4RawStages = 8;
constexpr int kF4RawStage = 2 * kF4Page;      // 8704
constexpr int kF4MaxHi = 64;

struct F4Layout {
  static constexpr int kA = 0;                               // 2 x [128 rows][128 B] E4M3, swizzled
  static constexpr int kQ = kA + 2 * 16384;                  // 2 x [64 rows][128 B] E4M3, swizzled
  static constexpr int kRaw = kQ + 2 * kF4MaxHi * 128;       // raw pages ring
  static constexpr int kFac = kRaw + kF4RawStages * kF4RawStage;   // 2 x [64][4] fp32 q scale factors
  static constexpr int kW = kFac + 2 * kF4MaxHi * 16;        // 2 x [64] fp32 head weights
  static constexpr int kBar = kW + 2 * kF4MaxHi * 4;
  static constexpr int kNumBars = 2 * kF4RawStages + 4;
  static constexpr int kTmem = kBar + kNumBars * 8;
  static constexpr int kScan = kTmem + 16;
  static constexpr int kBytes = kScan + (kWarps + 8) * 4;
};
constexpr int kF4SmemBytes = F4Layout::kBytes + 1024;

// 2^(e - 127) for an E8M0 byte (0xFF: NaN), exactly.
__device__ __forceinline__ float e8m0_value(uint32_t e) {
  return e == 0xFFu ? __uint_as_float(0x7FC00000u) : (e == 0u ? __uint_as_float(0x00400000u) : __uint_as_float(e << 23));
}

// Four E2M1 codes (nibbles 0..3 of x, low nibble first) -> four E4M3 bytes of
// the same values: the magnitude through a byte permutation of the table
// {0, 0.5, 1, 1.5, 2, 3, 4, 6}, the sign bit moved to bit 7 of its byte.
__device__ __forceinline__ uint32_t e2m1x4_to_e4m3(uint32_t x) {
  const uint32_t mag = __byte_perm(0x3C383000u, 0x4C484440u, x & 0x7777u);
  const uint32_t spread = (x & 0xFu) | ((x & 0xF0u) << 4) | ((x & 0xF00u) << 8) | ((x & 0xF000u) << 12);
  return mag | ((spread & 0x08080808u) << 4);
}

// 16 packed E2M1 codes (8 bytes) -> 16 E4M3 bytes.
__device__ __forceinline__ uint4 e2m1x16_to_e4m3(uint32_t w0, uint32_t w1) {
  return make_uint4(e2m1x4_to_e4m3(w0 & 0xFFFFu), e2m1x4_to_e4m3(w0 >> 16), e2m1x4_to_e4m3(w1 & 0xFFFFu),
                    e2m1x4_to_e4m3(w1 >> 16));
}

__global__ void __launch_bounds__(kThreads, 1) indexer_logits_fp4_kernel(const IndexerParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + F4Layout::kBar);
  uint64_t* raw_full = bars;                          // [stages] page copies landed
  uint64_t* raw_empty = bars + kF4RawStages;          // [stages] a group has converted the stage
  uint64_t* a_full = bars + 2 * kF4RawStages;         // [2] group e's A rows (and q) are ready
  uint64_t* acc_full = a_full + 2;                    // [2] group e's accumulators are written
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + F4Layout::kTmem);
  int* scan = reinterpret_cast<int*>(smem + F4Layout::kScan);

  const int warp = static_cast<int>(warp_id());
  const int lane = static_cast<int>(lane_id());
  const int HiP = p.HiP;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kF4RawStages; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], 4);
    }
    for (int e = 0; e < 2; ++e) {
      mbar_init(&a_full[e], 4);
      mbar_init(&acc_full[e], 1);
    }
    fence_mbar_init();
  }
  if (warp == kF4MmaWarp) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  griddep_launch();
  if (threadIdx.x < 32)   // the lengths and sequence ids every CTA scans first
    for (int t = threadIdx.x * 32; t < p.T; t += 32 * 32) {
      asm volatile("prefetch.global.L2 [%0];" ::"l"(p.n_vis + t));
      asm volatile("prefetch.global.L2 [%0];" ::"l"(p.q_seq + t));
    }
  griddep_wait();  // inputs may come from the previous kernel of the stream

  int count;
  Cursor c0;
  work_range<kThreads>(p, scan, count, c0);   // ends with a barrier
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (count > 0) {
    if (warp == 0 || warp == kF4ProducerB) {
      // ================= producers: one bulk copy per page, alternate tiles =================
      const int pw = warp == 0 ? 0 : 1;
      const int mine = count > pw ? (count - pw + 1) / 2 : 0;
      Cursor cl = c0;
      cl.advance_by(p, pw + 2 * lane);
      auto fetch = [&](int k, int& pid0, int& pid1, int& second) {
        pid0 = pid1 = second = 0;
        if (k < mine) {
          const int n = clamp_n(p, __ldg(p.n_vis + cl.t));
          const int32_t* row = p.page_table + static_cast<int64_t>(__ldg(p.q_seq + cl.t)) * p.pt_stride;
          pid0 = __ldg(row + min(2 * cl.j, p.pt_stride - 1));
          pid1 = __ldg(row + min(2 * cl.j + 1, p.pt_stride - 1));
          second = (cl.j * kTileRows + 64) < n ? 1 : 0;
          cl.advance_by(p, 64);
        }
      };
      int c_pid0, c_pid1, c_sec, n_pid0, n_pid1, n_sec;
      fetch(lane, c_pid0, c_pid1, c_sec);
      fetch(32 + lane, n_pid0, n_pid1, n_sec);
      const uint64_t pol = l2_evict_first_policy();
      int issued = 0;
      bool ok = true;
      for (int r = 0; 32 * r < mine && ok; ++r) {
        if (r > 0) {
          c_pid0 = n_pid0;
          c_pid1 = n_pid1;
          c_sec = n_sec;
          fetch(32 * (r + 1) + lane, n_pid0, n_pid1, n_sec);
        }
        const int kn = min(32, mine - 32 * r);
        for (int u = 0; u < kn; ++u) {
          int pid0 = __shfl_sync(0xffffffffu, c_pid0, u);
          int pid1 = __shfl_sync(0xffffffffu, c_pid1, u);
          const bool second = __shfl_sync(0xffffffffu, c_sec, u) != 0;
          int okl = 1;
          if (lane == 0) {
            const int i = pw + 2 * (32 * r + u);
            const int s = i % kF4RawStages;
            okl = mbar_wait(&raw_empty[s], ((i / kF4RawStages) & 1) ^ 1) ? 1 : 0;
            if (okl) {
              if (pid0 < 0 || pid0 >= p.num_pages) { raise_error(kErrIndex); pid0 = 0; }
              if (pid1 < 0 || pid1 >= p.num_pages) { if (second) raise_error(kErrIndex); pid1 = 0; }
              uint8_t* st = smem + F4Layout::kRaw + s * kF4RawStage;
              mbar_arrive_expect_tx(&raw_full[s], second ? 2 * kF4Page : kF4Page);
              bulk_load_hint(st, p.scale_base + pid0 * p.page_stride, kF4Page, &raw_full[s], pol);
              if (second) bulk_load_hint(st + kF4Page, p.scale_base + pid1 * p.page_stride, kF4Page, &raw_full[s], pol);
              ++issued;
            }
          }
          ok = __shfl_sync(0xffffffffu, okl, 0) != 0;
          if (!ok) break;
        }
      }
      // drain: wait (bounded) for the copies this warp issued before leaving
      if (lane == 0)
        for (int k = (issued > kF4RawStages / 2 ? issued - kF4RawStages / 2 : 0); k < issued; ++k) {
          const int i = pw + 2 * k;
          mbar_wait(&raw_full[i % kF4RawStages], (i / kF4RawStages) & 1);
        }
      __syncwarp();
    } else if (warp == kF4MmaWarp) {
      // ================= MMA issuer: four K = 32 blocks, four accumulators =================
      if (lane == 0) {
        const uint32_t idesc = make_idesc(kFmtE4M3, kFmtE4M3, 0, 0, 128, HiP);
        int done = 0;
        for (int i = 0; i < count; ++i) {
          const int e = i & 1;
          if (!mbar_wait(&a_full[e], (i >> 1) & 1)) break;
          tc_fence_after();
          const uint32_t a_base = smem_u32(smem + F4Layout::kA + e * 16384);
          const uint32_t b_base = smem_u32(smem + F4Layout::kQ + e * (kF4MaxHi * 128));
          const uint32_t d0 = tmem_base + static_cast<uint32_t>(e * 4 * HiP);
#pragma unroll
          for (int blk = 0; blk < 4; ++blk)
            mma_f8f6f4(d0 + blk * HiP, smem_desc_sw128(a_base + blk * 32, 16, 1024),
                       smem_desc_sw128(b_base + blk * 32, 16, 1024), idesc, 0);
          mma_commit(&acc_full[e]);
          done = i + 1;
        }
        // no MMA may still write TMEM when the CTA deallocates it
        if (done > 0) mbar_wait(&acc_full[(done - 1) & 1], ((done - 1) >> 1) & 1);
      }
      __syncwarp();
    } else if (warp >= 2 && warp <= 9) {
      // ================= two groups: convert, then epilogue, alternate tiles =================
      const int e = (warp - 2) >> 2;
      const int g = warp & 3;                // TMEM lane quarter of this warp
      const int row = g * 32 + lane;         // tile row = TMEM lane
      const int tid_g = (warp - 2 - 4 * e) * 32 + lane;
      uint8_t* abuf = smem + F4Layout::kA + e * 16384;
      uint8_t* qbuf = smem + F4Layout::kQ + e * (kF4MaxHi * 128);
      float4* fac = reinterpret_cast<float4*>(smem + F4Layout::kFac + e * (kF4MaxHi * 16));
      float* wv = reinterpret_cast<float*>(smem + F4Layout::kW + e * (kF4MaxHi * 4));
      Cursor c = c0;
      if (e == 1 && count > 1) c.advance(p);
      int cur_t = -1, n = 0;
      for (int i = e; i < count; i += 2) {
        if (c.t != cur_t) {
          // the query's E4M3 rows (two threads per head), scale factors and
          // weights, once every thread of the group is past its last epilogue
          named_barrier_sync(1 + e, 128);
          const int h = tid_g >> 1, half = tid_g & 1;
          if (h < HiP) {
            const int64_t qh = static_cast<int64_t>(c.t) * p.Hi + h;
            uint4 v0 = make_uint4(0u, 0u, 0u, 0u), v1 = v0;
            if (h < p.Hi) {
              const uint4* src = reinterpret_cast<const uint4*>(p.q_fp8 + qh * 64 + half * 32);
              v0 = __ldg(src);
              v1 = __ldg(src + 1);
            }
            *reinterpret_cast<uint4*>(qbuf + sw128_offset(h, 4 * half)) = e2m1x16_to_e4m3(v0.x, v0.y);
            *reinterpret_cast<uint4*>(qbuf + sw128_offset(h, 4 * half + 1)) = e2m1x16_to_e4m3(v0.z, v0.w);
            *reinterpret_cast<uint4*>(qbuf + sw128_offset(h, 4 * half + 2)) = e2m1x16_to_e4m3(v1.x, v1.y);
            *reinterpret_cast<uint4*>(qbuf + sw128_offset(h, 4 * half + 3)) = e2m1x16_to_e4m3(v1.z, v1.w);
            if (half == 0) {
              // padded heads: factors and weight 0, so they add nothing
              const uint32_t ew = h < p.Hi ? __ldg(reinterpret_cast<const uint32_t*>(p.q_e8m0) + qh) : 0u;
              fac[h] = h < p.Hi ? make_float4(e8m0_value(ew & 0xFFu), e8m0_value((ew >> 8) & 0xFFu),
                                              e8m0_value((ew >> 16) & 0xFFu), e8m0_value(ew >> 24))
                                : make_float4(0.f, 0.f, 0.f, 0.f);
              wv[h] = h < p.Hi ? __ldg(p.w + qh) : 0.f;
            }
          }
          named_barrier_sync(1 + e, 128);   // fac / wv are read by every thread of the group
          cur_t = c.t;
          n = clamp_n(p, __ldg(p.n_vis + c.t));
        }
        const int s = i % kF4RawStages;
        if (!mbar_wait(&raw_full[s], (i / kF4RawStages) & 1)) break;
        // ---- convert this row: 64 bytes of codes -> 128 E4M3 bytes, swizzled
        const uint8_t* src = smem + F4Layout::kRaw + s * kF4RawStage + (row >> 6) * kF4Page;
        const uint4* cw = reinterpret_cast<const uint4*>(src + (row & 63) * 64);
        const uint32_t ek = *reinterpret_cast<const uint32_t*>(src + 4096 + (row & 63) * 4);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint4 v = cw[u];
          *reinterpret_cast<uint4*>(abuf + sw128_offset(row, 2 * u)) = e2m1x16_to_e4m3(v.x, v.y);
          *reinterpret_cast<uint4*>(abuf + sw128_offset(row, 2 * u + 1)) = e2m1x16_to_e4m3(v.z, v.w);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&raw_empty[s]);
        fence_proxy_async_smem();   // A and q rows are read by the tensor core
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[e]);
        const float k0 = e8m0_value(ek & 0xFFu), k1 = e8m0_value((ek >> 8) & 0xFFu);
        const float k2 = e8m0_value((ek >> 16) & 0xFFu), k3 = e8m0_value(ek >> 24);
        if (!mbar_wait(&acc_full[e], (i >> 1) & 1)) break;
        tc_fence_after();
        // ---- epilogue: per head, the four block sums with their scales, ReLU, weight
        const uint32_t tb = tmem_base + (static_cast<uint32_t>(g * 32) << 16) + static_cast<uint32_t>(e * 4 * HiP);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};   // four partial head sums: independent FMA chains
        for (int h0 = 0; h0 < HiP; h0 += 16) {
          float d0[16], d1[16], d2[16], d3[16];
          tmem_ld16(tb + h0, d0);
          tmem_ld16(tb + HiP + h0, d1);
          tmem_ld16(tb + 2 * HiP + h0, d2);
          tmem_ld16(tb + 3 * HiP + h0, d3);
          tmem_ld_wait();
#pragma unroll
          for (int x = 0; x < 16; ++x) {
            const float4 f = fac[h0 + x];
            // each D times a power of two is exact; three roundings in the sum
            float v = d0[x] * (f.x * k0);
            v = fmaf(d1[x], f.y * k1, v);
            v = fmaf(d2[x], f.z * k2, v);
            v = fmaf(d3[x], f.w * k3, v);
            acc[x & 3] = fmaf(wv[h0 + x], fmaxf(v, 0.f), acc[x & 3]);
          }
        }
        tc_fence_before();
        const int sidx = c.j * kTileRows + row;
        if (sidx < n)
          p.logits[static_cast<int64_t>(c.t) * p.logits_stride + sidx] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
        c.advance(p);
        if (i + 1 < count) c.advance(p);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kF4MmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(ptr);
  }();
  return fn;
}

}  // namespace

int launch_indexer_logits(const dsv4sa_pool_desc* kpool, const int32_t* page_table, int32_t pt_stride,
                          const int32_t* q_seq, const int32_t* n_vis, const uint8_t* q_fp8, const float* q_scale,
                          const float* w, int32_t T, int32_t Hi, int32_t n_max, float* logits,
                          int64_t logits_stride, cudaStream_t stream) {
  EncodeTiledFn encode = get_encode_fn();
  if (!encode) return DSV4SA_ERR_CUDA;
  CUtensorMap key_map;
  const cuuint64_t gdim[3] = {128, 64, static_cast<cuuint64_t>(kpool->num_pages)};
  const cuuint64_t gstride[2] = {128, static_cast<cuuint64_t>(kpool->page_stride)};
  const cuuint32_t box[3] = {128, 64, 1};
  const cuuint32_t estride[3] = {1, 1, 1};
  void* gbase = static_cast<uint8_t*>(kpool->base) + kpool->nope_off;
  if (encode(&key_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, gbase, gdim, gstride, box, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return DSV4SA_ERR_INVALID_ARG;

  IndexerParams p;
  p.page_table = page_table;
  p.q_seq = q_seq;
  p.n_vis = n_vis;
  p.q_fp8 = q_fp8;
  p.q_scale = q_scale;
  p.w = w;
  p.scale_base = static_cast<const uint8_t*>(kpool->base) + kpool->scale_off;
  p.logits = logits;
  p.page_stride = kpool->page_stride;
  p.num_pages = kpool->num_pages;
  p.logits_stride = logits_stride;
  p.pt_stride = pt_stride;
  p.T = T;
  p.Hi = Hi;
  p.HiP = (Hi + 15) / 16 * 16;
  p.n_max = n_max;

  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSV4SA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return DSV4SA_ERR_CUDA;
  if (!smem_attr_once(dev, 0, reinterpret_cast<const void*>(indexer_logits_kernel), kSmemBytes))
    return DSV4SA_ERR_CUDA;
  const long long max_tiles = static_cast<long long>(T) * ((n_max + kTileRows - 1) / kTileRows);
  if (max_tiles == 0) return DSV4SA_OK;
  // q blocks: [T][Hi][128] bytes, one box of Hi rows per query, 128-byte swizzled
  CUtensorMap q_map;
  const cuuint64_t qdim[3] = {128, static_cast<cuuint64_t>(Hi), static_cast<cuuint64_t>(T)};
  const cuuint64_t qstride[2] = {128, static_cast<cuuint64_t>(Hi) * 128};
  const cuuint32_t qbox[3] = {128, static_cast<cuuint32_t>(Hi), 1};
  if (encode(&q_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(q_fp8), qdim, qstride, qbox, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return DSV4SA_ERR_INVALID_ARG;
  // one SM is left free, so the next kernel's first CTA starts at once (a
  // programmatic dependent: it may run while the logits are being computed)
  const int cap = sms > 1 ? sms - 1 : 1;
  const int grid = static_cast<int>(max_tiles < cap ? max_tiles : cap);
  const cudaError_t err =
      launch_pdl(indexer_logits_kernel, dim3(grid), dim3(kThreads8), kSmemBytes, stream, key_map, q_map, p);
  return err == cudaSuccess ? DSV4SA_OK : DSV4SA_ERR_CUDA;
}

int launch_indexer_logits_fp4(const dsv4sa_pool_desc* kpool, const int32_t* page_table, int32_t pt_stride,
                              const int32_t* q_seq, const int32_t* n_vis, const uint8_t* q_fp4,
                              const uint8_t* q_e8m0, const float* w, int32_t T, int32_t Hi, int32_t n_max,
                              float* logits, int64_t logits_stride, cudaStream_t stream) {
  IndexerParams p{};
  p.page_table = page_table;
  p.q_seq = q_seq;
  p.n_vis = n_vis;
  p.q_fp8 = q_fp4;
  p.q_e8m0 = q_e8m0;
  p.w = w;
  p.scale_base = static_cast<const uint8_t*>(kpool->base);   // the page base: codes, then E8M0 bytes
  p.logits = logits;
  p.page_stride = kpool->page_stride;
  p.num_pages = kpool->num_pages;
  p.logits_stride = logits_stride;
  p.pt_stride = pt_stride;
  p.T = T;
  p.Hi = Hi;
  p.HiP = (Hi + 15) / 16 * 16;
  p.n_max = n_max;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSV4SA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return DSV4SA_ERR_CUDA;
  if (!smem_attr_once(dev, 15, reinterpret_cast<const void*>(indexer_logits_fp4_kernel), kF4SmemBytes))
    return DSV4SA_ERR_CUDA;
  const long long max_tiles = static_cast<long long>(T) * ((n_max + kTileRows - 1) / kTileRows);
  if (max_tiles == 0) return DSV4SA_OK;
  const int cap = sms > 1 ? sms - 1 : 1;   // as the FP8 kernel
  const int grid = static_cast<int>(max_tiles < cap ? max_tiles : cap);
  const cudaError_t err = launch_pdl(indexer_logits_fp4_kernel, dim3(grid), dim3(kThreads), kF4SmemBytes, stream, p);
  return err == cudaSuccess ? DSV4SA_OK : DSV4SA_ERR_CUDA;
}

uint32_t read_error_word_indexer(cudaStream_t stream, bool clear) {
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
