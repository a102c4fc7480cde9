// attn.cu -- sparse attention with attention sink over gathered FP8/BF16 KV rows.
//
// For query t, head h and the multiset J of valid indices of
// idx_c[t] (compressed pool) ++ idx_w[t] (raw-token window pool):
//   o[t, h] = sum_j e^{a_j} kv_j / (sum_j e^{a_j} + e^{sink_h}),  a_j = scale * q[t, h] . kv_j
// ("DeepSeek-V4 全面解读" §3.7 sparse_attn_kernel: gather by int32 index, -1 is
// an invalid slot scored -inf, FlashAttention-style online softmax, sink added
// to the denominator after the loop; "tilelang量化内核拆解…" sparse_attn 实现拆解:
// running max starts at -1e30 so an all-invalid row gives zeros; heads padded
// to 16; "DeepSeek-V4 in SGLang" MQALayer: one kv tensor is both K and V.)
//
// Design.  A CTA owns one query, a group of up to 64 heads (padded to 16, 32 or
// 64) and one or more chunks of 128 gathered rows.  Warps 8-15 (gather) and
// warps 0-7 (compute) work on consecutive chunks at the same time, handing the
// single KV tile over through mbarriers:
//   1. gather: locate each row (index -> page id), fetch its 448 FP8 codes,
//      7 fp32 scales and 64 BF16 rope values in 32-byte pieces (consecutive
//      lanes read consecutive pieces of a row) -- all loads in flight before
//      the tile is free -- then dequantise the nope part
//      to BF16 (hardware e4m3x2 -> f16x2 converts, fp32 scale) into a
//      128 x 512 BF16 tile in the 128-byte-swizzled layout the tensor core
//      reads; invalid rows become zero rows.
//   2. S^T = KV . Q^T on tcgen05 (kind::f16, M = 128 rows, N = heads, K = 512):
//      TMEM lane r holds the scores of row r for every head.
//   3. online softmax in the exp2 domain: per-head max and sum across the 128
//      rows with a transposing warp reduction plus a 4-way cross-warp step;
//      P is written to shared memory in BF16; the output accumulator is
//      rescaled in TMEM when the running max moves.
//   4. O^T += V^T . P^T on tcgen05 (M = 128 dims per block, 4 blocks, N = heads,
//      K = 128 rows); the KV tile is read MN-major, so the same shared tile
//      serves as K (K-major) and V (MN-major).
// Decode splits the rows of a query across CTAs and merges the partial
// (O, max, sum) triples by log-sum-exp, adding the sink once: 2, 4 or 8 splits
// run as a thread-block cluster in the decode kernel (attn_decode.cu); this
// kernel takes the other split counts, whose partials merge in a second
// kernel.  Prefill runs all chunks of a query in one CTA and writes the
// normalised BF16 output directly.
#include "attn_common.cuh"

namespace dsv4sa {
namespace {

using namespace attn;

constexpr int kComputeThreads = 256;     // warps 0-7: MMA issue, softmax, epilogue
constexpr int kGatherThreads = 256;      // warps 8-15: row gather + dequantisation
constexpr int kThreads = kComputeThreads + kGatherThreads;
template <int HN>
struct Smem {
  static constexpr int kKv = 0;
  static constexpr int kQ = kKvBytes;                 // 8 column blocks x HN rows x 128 B
  static constexpr int kP = kQ + 8 * HN * 128;        // 2 row blocks x HN rows x 128 B
  static constexpr int kRowp = kP + 2 * HN * 128;     // uint64 [2][128]
  static constexpr int kFlags = kRowp + 2 * kRows * 8;  // int [2] chunk valid, then uint32 [2][4] row-valid bits
  static constexpr int kRowScale = kFlags + 48;       // float [128][8]: the scale slots of the chunk's rows
  static constexpr int kRedMax = kRowScale + kRows * 32;  // float [4][HN]
  static constexpr int kRedSum = kRedMax + 4 * HN * 4;
  static constexpr int kMRun = kRedSum + 4 * HN * 4;  // float [HN] each
  static constexpr int kLRun = kMRun + HN * 4;
  static constexpr int kAlpha = kLRun + HN * 4;
  static constexpr int kFac = kAlpha + HN * 4;
  static constexpr int kBar = kFac + HN * 4;          // 4 mbarriers
  static constexpr int kTmem = kBar + 32;
  static constexpr int kBytes = kTmem + 16;
};

// bar.red.or over the threads of named barrier `id` (n threads): every
// participant learns whether any of them passed true.  Also a barrier.
__device__ __forceinline__ bool group_any(bool v, uint32_t id, uint32_t n) {
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

// One thread of a group polls the mbarrier (bounded); the whole group learns
// the outcome, so every member takes the same path afterwards.
__device__ __forceinline__ bool group_wait(uint64_t* bar, uint32_t parity, uint32_t id, uint32_t n, bool leader) {
  const bool bad = leader ? !mbar_wait(bar, parity) : false;
  return !group_any(bad, id, n);
}

constexpr uint32_t kBarCompute = 1;   // named barrier of warps 0-7
constexpr uint32_t kBarGather = 2;    // named barrier of warps 8-15

template <int HN>
__global__ void __launch_bounds__(kThreads, 1) sparse_attn_kernel(const AttnParams p) {
  using S = Smem<HN>;
  extern __shared__ uint8_t smem_raw[];
  // 128-byte swizzled operand tiles need 1024-byte aligned bases
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* kv = smem + S::kKv;
  uint8_t* qs = smem + S::kQ;
  uint8_t* ps = smem + S::kP;
  uint64_t* rowp = reinterpret_cast<uint64_t*>(smem + S::kRowp);   // [2][kRows]
  int* chunk_valid = reinterpret_cast<int*>(smem + S::kFlags);      // [2]
  uint32_t* rvmask = reinterpret_cast<uint32_t*>(smem + S::kFlags + 16);   // [2][4]: row r valid = bit r
  uint4* row_scale = reinterpret_cast<uint4*>(smem + S::kRowScale);  // [kRows][2]
  float* red_max = reinterpret_cast<float*>(smem + S::kRedMax);
  float* red_sum = reinterpret_cast<float*>(smem + S::kRedSum);
  float* m_run = reinterpret_cast<float*>(smem + S::kMRun);
  float* l_run = reinterpret_cast<float*>(smem + S::kLRun);
  float* alpha = reinterpret_cast<float*>(smem + S::kAlpha);
  float* fac = reinterpret_cast<float*>(smem + S::kFac);
  uint64_t* bar_s = reinterpret_cast<uint64_t*>(smem + S::kBar);   // S MMA done
  uint64_t* bar_o = bar_s + 1;                                       // PV MMA done
  uint64_t* bar_full = bar_s + 2;                                    // gather -> compute: chunk in the tile
  uint64_t* bar_free = bar_s + 3;                                    // compute -> gather: chunk's rows read
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + S::kTmem);

  constexpr int HW = HN / 2;  // heads handled per warp in the softmax
  constexpr uint32_t kTmemCols = HN == 64 ? 512u : (HN == 32 ? 256u : 128u);
  constexpr uint32_t kColS = 0, kColO = HN;   // S^T: HN columns; O^T: 4 blocks x HN columns

  const int split = blockIdx.x;
  const int t = blockIdx.y;
  const int h0 = blockIdx.z * HN;
  const int tid = threadIdx.x;
  const uint32_t warp = warp_id(), lane = lane_id();

  if (tid == 0) {
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    mbar_init(bar_full, kGatherThreads / 32);
    mbar_init(bar_free, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_holder, kTmemCols);
    tmem_relinquish();
  }
  griddep_launch();
  // Without early_window every input may come from the previous kernel of the
  // stream.  With it the caller guarantees that only idx_c does, so the window
  // rows (and q) are processed while that kernel still runs; the gather warps
  // wait before the first compressed chunk, everybody before the epilogue.
  if (!p.early_window) griddep_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  // Rows of this CTA: its share of the window list, then its share of the
  // compressed list; a chunk holds rows of one list (window chunks first).
  const int ws0 = min(p.kw, split * p.kw_split), ws1 = min(p.kw, ws0 + p.kw_split);
  const int cs0 = min(p.kc, split * p.kc_split), cs1 = min(p.kc, cs0 + p.kc_split);
  const int nwch = (ws1 - ws0 + kRows - 1) / kRows;
  const int nch = nwch + (cs1 - cs0 + kRows - 1) / kRows;
  // chunk c: window (or compressed) rows [c0, c0 + c_rows) of that list
  auto chunk_at = [&](int c, int& c0, int& c_rows, bool& window) {
    window = c < nwch;
    c0 = window ? ws0 + c * kRows : cs0 + (c - nwch) * kRows;
    c_rows = min(kRows, (window ? ws1 : cs1) - c0);
  };
  bool ok = true;
  bool pv_issued = false;   // compute: O holds a partial sum

  if (tid >= kComputeThreads) {
    // =========================== gather warps ===========================
    // Per chunk: locate the rows (index -> page), load them (all loads in
    // flight together), wait until the tensor core no longer reads the tile,
    // dequantise into it, hand it over.  The loads of chunk c + 1 overlap the
    // compute warps' work on chunk c.
    const int gt = tid - kComputeThreads;
    const int seq = __ldg(p.q_seq + t);
    const int32_t* cpt = p.comp_pt + static_cast<int64_t>(seq) * p.comp_pt_stride;
    const int32_t* wpt = p.win_pt + static_cast<int64_t>(seq) * p.win_pt_stride;
    const int32_t wpos = p.idx_w ? 0 : __ldg(p.win_pos + t);   // window from the position
    // warm L2 with the query's compressed page-table row (a step input): the
    // compressed chunks then locate their rows without a DRAM round trip
    if (p.kc > 0)
      for (int e = gt * 32; e < p.comp_pt_stride; e += kGatherThreads * 32)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(cpt + e));
    uint32_t ph_o = 0;
    bool pv_out = false;      // a PV reading the tile was handed over and not yet waited for
    bool tile_init = false;   // every row of the tile holds finite values
    for (int c = 0; c < nch; ++c) {
      int c0, c_rows;
      bool window;
      chunk_at(c, c0, c_rows, window);
      if (p.early_window && c == nwch) griddep_wait();   // idx_c comes from the previous kernel
      uint64_t* rp_buf = rowp + (c & 1) * kRows;
      // ---- 1. row addresses.  Index and page-id loads are unconditional, from
      // clamped (always valid) addresses, then masked.
      bool valid = false;
      if (gt < kRows) {
        const int gi = c0 + gt;   // index into this chunk's list
        const bool in_c = !window && gt < c_rows;
        const bool in_w = window && gt < c_rows;
        int32_t ec = -1, ew = -1;
        if (!window) {
          ec = __ldg(p.idx_c + static_cast<int64_t>(t) * p.idx_c_stride + min(gi, p.kc - 1));
        } else if (p.idx_w) {
          ew = __ldg(p.idx_w + static_cast<int64_t>(t) * p.idx_w_stride + min(gi, p.kw - 1));
        } else {
          const int64_t pw = static_cast<int64_t>(wpos) - p.kw + 1 + gi;
          ew = pw < 0 ? -1 : static_cast<int32_t>(p.win_ring > 0 ? pw % p.win_ring : pw);
        }
        const int32_t e = in_c ? ec : (in_w ? ew : -1);
        const int32_t lim = in_c ? p.comp_pt_stride * 64 : p.win_pt_stride * 64;
        const int32_t* ptr = in_c ? cpt : wpt;
        const int32_t page = __ldg(ptr + (min(max(e, 0), lim - 1) >> 6));
        const int64_t np = in_c ? p.comp_num_pages : p.win_num_pages;
        uint64_t rp = 0;
        if (e >= 0) {
          if (e >= lim || page < 0 || page >= np) {
            raise_error(kErrIndex);
          } else {
            const uint8_t* base = in_c ? p.comp_base : p.win_base;
            const int64_t stride = in_c ? p.comp_page_stride : p.win_page_stride;
            rp = reinterpret_cast<uint64_t>(base + static_cast<int64_t>(page) * stride) | static_cast<uint64_t>(e & 63);
          }
        }
        rp_buf[gt] = rp;
        valid = rp != 0;
        const uint32_t bits = __ballot_sync(0xffffffffu, valid);   // warps 8-11: rows 32 w .. 32 w + 31
        if (lane == 0) rvmask[(c & 1) * 4 + (gt >> 5)] = bits;
      }
      const bool any = group_any(valid, kBarGather, kGatherThreads);   // also publishes rp_buf in the group
      if (gt == 0) chunk_valid[c & 1] = any ? 1 : 0;
      if (any && ok) {
        // ---- 2. gather + dequantise into the swizzled BF16 tile.  A task is a
        // 32-byte piece of one row: 32 FP8 codes (nope pieces 0-13, dims
        // 32 j .. 32 j + 31, with the scale of their 64-dim group) or 16 BF16
        // rope values (pieces 14-17).  Task k -> row r = 4 a + (k & 3) and piece
        // j, with a = (k >> 2) / 18, j = (k >> 2) % 18: one warp instruction
        // reads 8 consecutive pieces of 4 rows (a few 128-byte lines), and its
        // shared-memory stores hit 4 rows whose swizzle phases differ.
        constexpr int kPieces = 18;
        constexpr int kTasks = kRows * kPieces;
        constexpr int kIters = kTasks / kGatherThreads;
        static_assert(kTasks % kGatherThreads == 0, "whole iterations");
        uint4 raw[kIters][2];
        // the 8 scale slots of each row (7 used), one thread per row
        if (gt < kRows) {
          const uint64_t rp = gt < c_rows && rp_buf[gt] ? rp_buf[gt] : reinterpret_cast<uint64_t>(p.any_page);
          const uint4* src = reinterpret_cast<const uint4*>(
              reinterpret_cast<const uint8_t*>(rp & ~uint64_t(63)) + kPageScaleOff + (rp & 63) * 32);
          row_scale[2 * gt] = __ldg(src);
          row_scale[2 * gt + 1] = __ldg(src + 1);
        }
#pragma unroll
        for (int it = 0; it < kIters; ++it) {
          const int k = it * kGatherThreads + gt;
          const int jk = k >> 2, r = 4 * (jk / kPieces) + (k & 3), j = jk % kPieces;
          if (r < c_rows) {   // rows past the chunk are never loaded
            // invalid rows read slot 0 of a valid page and are zeroed afterwards:
            // the loads are unconditional, so all of them are in flight together
            const uint64_t rp = rp_buf[r] ? rp_buf[r] : reinterpret_cast<uint64_t>(p.any_page);
            const uint8_t* page = reinterpret_cast<const uint8_t*>(rp & ~uint64_t(63));
            const int slot = static_cast<int>(rp & 63);
            const uint4* src = j < 14 ? reinterpret_cast<const uint4*>(page + slot * 448 + j * 32)
                                      : reinterpret_cast<const uint4*>(page + kPageRopeOff + slot * 128 + (j - 14) * 32);
            raw[it][0] = __ldg(src);
            raw[it][1] = __ldg(src + 1);
          }
        }
        // ---- 3. the previous chunk's PV still reads the tile: wait for it
        if (pv_out) {
          ok = group_wait(bar_o, ph_o, kBarGather, kGatherThreads, gt == 0);
          ph_o ^= 1u;
          pv_out = false;
        }
        named_barrier_sync(kBarGather, kGatherThreads);   // row_scale visible in the group
        if (ok) {
          const float* scale_of = reinterpret_cast<const float*>(row_scale);
#pragma unroll
          for (int it = 0; it < kIters; ++it) {
            const int k = it * kGatherThreads + gt;
            const int jk = k >> 2, r = 4 * (jk / kPieces) + (k & 3), j = jk % kPieces;
            if (r >= c_rows && tile_init) continue;   // rows past the chunk keep finite stale values
            float scl = scale_of[r * 8 + (j < 14 ? j >> 1 : 0)];
            if (r >= c_rows || rp_buf[r] == 0) {
              scl = 0.f;
              raw[it][0] = raw[it][1] = make_uint4(0u, 0u, 0u, 0u);
            }
            if (j < 14) {
              uint8_t* blk = kv + (j >> 1) * kKvBlock;
              const uint32_t u0 = static_cast<uint32_t>((j & 1) * 4);
#pragma unroll
              for (int x = 0; x < 2; ++x) {
                uint4 lo, hi;
                dequant16(raw[it][x], scl, lo, hi);
                *reinterpret_cast<uint4*>(blk + sw128_offset(r, u0 + 2 * x)) = lo;
                *reinterpret_cast<uint4*>(blk + sw128_offset(r, u0 + 2 * x + 1)) = hi;
              }
            } else {
              const uint32_t u0 = static_cast<uint32_t>((j - 14) * 2);
              *reinterpret_cast<uint4*>(kv + 7 * kKvBlock + sw128_offset(r, u0)) = raw[it][0];
              *reinterpret_cast<uint4*>(kv + 7 * kKvBlock + sw128_offset(r, u0 + 1)) = raw[it][1];
            }
          }
          fence_proxy_async_smem();   // the tile is read by the tensor core
          tile_init = true;
          pv_out = true;              // the compute warps run a PV over this tile
        }
      }
      // ---- 4. hand over once the compute warps are done with chunk c - 1
      if (c > 0) ok = group_wait(bar_free, (c - 1) & 1, kBarGather, kGatherThreads, gt == 0) && ok;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_full);
    }
  } else {
    // =========================== compute warps ===========================
    // Q block of this head group -> swizzled K-major tile (8 column blocks of 64 dims)
    {
      constexpr int kQIters = HN * 64 / kComputeThreads;
      const uint4* qsrc = reinterpret_cast<const uint4*>(p.q);
      uint4 qv[kQIters];
#pragma unroll
      for (int i = 0; i < kQIters; ++i) {   // clamped head: unconditional loads, all in flight
        const int u = i * kComputeThreads + tid, h = min(h0 + (u >> 6), p.H - 1);
        qv[i] = __ldg(qsrc + (static_cast<int64_t>(t) * p.H + h) * 64 + (u & 63));
      }
#pragma unroll
      for (int i = 0; i < kQIters; ++i)
        if (h0 + ((i * kComputeThreads + tid) >> 6) >= p.H) qv[i] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int i = 0; i < kQIters; ++i) {
        const int u = i * kComputeThreads + tid, h = u >> 6, v = u & 63;
        *reinterpret_cast<uint4*>(qs + (v >> 3) * (HN * 128) + sw128_offset(h, v & 7)) = qv[i];
      }
    }
    fence_proxy_async_smem();
    if (tid < HN) {
      m_run[tid] = -1e30f;
      l_run[tid] = 0.f;
    }
    named_barrier_sync(kBarCompute, kComputeThreads);

    const uint32_t idesc_s = make_idesc(kFmtBF16, kFmtBF16, 0, 0, 128, HN);
    const uint32_t idesc_o = make_idesc(kFmtBF16, kFmtBF16, 1, 0, 128, HN);
    uint32_t ph_s = 0, ph_o = 0;
    bool pv_pending = false;  // a PV MMA was issued and not waited for
    for (int c = 0; c < nch; ++c) {
      ok = group_wait(bar_full, c & 1, kBarCompute, kComputeThreads, tid == 0);
      if (!ok) break;
      if (chunk_valid[c & 1] == 0) {   // nothing to attend in this chunk
        named_barrier_sync(kBarCompute, kComputeThreads);
        if (tid == 0) mbar_arrive(bar_free);
        continue;
      }
      // ---- S^T = KV . Q^T  (M = 128 rows, N = HN heads, K = 512)
      if (tid == 0) {
        tc_fence_after();
        const uint32_t kv_a = smem_u32(kv), q_a = smem_u32(qs);
#pragma unroll
        for (int kk = 0; kk < 32; ++kk) {
          const uint32_t koff = static_cast<uint32_t>((kk & 3) * 32);
          mma_f16(tmem + kColS, smem_desc_sw128(kv_a + (kk >> 2) * kKvBlock + koff, 16, 1024),
                  smem_desc_sw128(q_a + (kk >> 2) * (HN * 128) + koff, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar_s);
      }
      ok = group_wait(bar_s, ph_s, kBarCompute, kComputeThreads, tid == 0);
      ph_s ^= 1u;
      if (!ok) break;
      tc_fence_after();

      // ---- online softmax (exp2 domain): thread (lane group g, head half hh)
      // holds row r = 32 g + lane for HN / 2 heads; per-head max and sum over
      // the rows by a transposing warp reduction plus a 4-way cross-warp step
      const uint32_t g = warp & 3u, hh = warp >> 2;
      const int r = static_cast<int>(g * 32 + lane);
      const bool rvalid = ((rvmask[(c & 1) * 4 + g] >> lane) & 1u) != 0u;
      float sv[HW];
      tmem_load_cols<HW>(tmem + ((g * 32u) << 16) + kColS + hh * HW, sv);
#pragma unroll
      for (int i = 0; i < HW; ++i) sv[i] = rvalid ? sv[i] * p.scale_log2 : -INFINITY;
      {
        float tmp[HW];
#pragma unroll
        for (int i = 0; i < HW; ++i) tmp[i] = sv[i];
        const float m = TransposeReduce<HW>::run(tmp, lane, 16u, OpMax());
        constexpr int kRep = 32 / HW;  // lanes holding the same head
        if ((lane & (kRep - 1)) == 0) red_max[g * HN + hh * HW + lane / kRep] = m;
      }
      // the previous PV reads P and writes O: it must be complete before both
      // are touched (the gather warps already waited for it, so this is quick)
      if (pv_pending) {
        ok = group_wait(bar_o, ph_o, kBarCompute, kComputeThreads, tid == 0);
        ph_o ^= 1u;
        pv_pending = false;
        if (!ok) break;
        tc_fence_after();
      } else {
        named_barrier_sync(kBarCompute, kComputeThreads);
      }
      if (tid < HN) {
        const float mc = fmaxf(fmaxf(red_max[tid], red_max[HN + tid]), fmaxf(red_max[2 * HN + tid], red_max[3 * HN + tid]));
        const float mo = m_run[tid];
        const float mn = fmaxf(mo, mc);
        alpha[tid] = exp2f(mo - mn);
        m_run[tid] = mn;
      }
      named_barrier_sync(kBarCompute, kComputeThreads);
      if (tid == 0) mbar_arrive(bar_free);   // the rows of this chunk are no longer needed
      {
        uint8_t* prow = ps + (r >> 6) * (HN * 128);
        const uint32_t unit = static_cast<uint32_t>((r & 63) >> 3);
        const int byte_in_unit = (r & 7) * 2;
#pragma unroll
        for (int i = 0; i < HW; ++i) {
          const int h = static_cast<int>(hh) * HW + i;
          const float pv = exp2f(sv[i] - m_run[h]);
          sv[i] = pv;
          *reinterpret_cast<__nv_bfloat16*>(prow + sw128_offset(h, unit) + byte_in_unit) = __float2bfloat16_rn(pv);
        }
        const float l = TransposeReduce<HW>::run(sv, lane, 16u, OpAdd());
        constexpr int kRep = 32 / HW;
        if ((lane & (kRep - 1)) == 0) red_sum[g * HN + hh * HW + lane / kRep] = l;
      }
      fence_proxy_async_smem();
      // rescale the running output when the max moved (the previous PV is complete)
      if (pv_issued) {
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const uint32_t mb = hh * 2 + b;
          const uint32_t ta = tmem + ((g * 32u) << 16) + kColO + mb * HN;
          constexpr int kC = HN < 32 ? HN : 32;   // columns per batch
#pragma unroll
          for (int j0 = 0; j0 < HN; j0 += kC) {
            float v[kC];
            tmem_load_cols<kC>(ta + j0, v);
#pragma unroll
            for (int x = 0; x < kC; ++x) v[x] *= alpha[j0 + x];
#pragma unroll
            for (int j = 0; j < kC; j += 16) tmem_st16(ta + j0 + j, v + j);
          }
        }
        tmem_st_wait();
      }
      tc_fence_before();
      named_barrier_sync(kBarCompute, kComputeThreads);
      if (tid < HN) {
        l_run[tid] = l_run[tid] * alpha[tid] + (red_sum[tid] + red_sum[HN + tid]) +
                     (red_sum[2 * HN + tid] + red_sum[3 * HN + tid]);
      }

      // ---- O^T += V^T . P^T  (M = 128 dims x 4 blocks, N = HN, K = 128 rows)
      if (tid == 0) {
        tc_fence_after();
        const uint32_t kv_a = smem_u32(kv), p_a = smem_u32(ps);
#pragma unroll
        for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            mma_f16(tmem + kColO + mb * HN, smem_desc_sw128(kv_a + (2 * mb) * kKvBlock + kk * 2048, kKvBlock, 1024),
                    smem_desc_sw128(p_a + (kk >> 2) * (HN * 128) + (kk & 3) * 32, 16, 1024), idesc_o,
                    (pv_issued || kk > 0) ? 1u : 0u);
          }
        }
        mma_commit(bar_o);
      }
      pv_issued = true;
      pv_pending = true;
    }
    if (ok && pv_pending) {
      ok = group_wait(bar_o, ph_o, kBarCompute, kComputeThreads, tid == 0);
      ph_o ^= 1u;
      tc_fence_after();
    }
  }

  // =========================== epilogue ===========================
  if (p.early_window) griddep_wait();   // outputs are written after the previous kernels completed
  // one outcome for the whole CTA, so every thread takes the same branches
  // below; the fences order the completed MMAs (observed by the compute warps)
  // before TMEM reads by any warp
  tc_fence_before();
  ok = __syncthreads_and(ok ? 1 : 0) != 0;
  tc_fence_after();
  const uint32_t g = warp & 3u;
  const uint32_t hh = (warp >> 2) & 1u;   // compute warps: block pair of the output
  const bool compute = tid < kComputeThreads;
  if (ok) {
    const bool finalize = p.merge == kMergeNone;
    if (tid < HN && h0 + tid < p.H) {
      const int h = h0 + tid;
      if (finalize) {
        const float sink2 = __ldg(p.sink + h) * kLog2e;
        const float M = fmaxf(m_run[tid], sink2);
        const float L = l_run[tid] * exp2f(m_run[tid] - M) + (sink2 > -INFINITY ? exp2f(sink2 - M) : 0.f);
        fac[tid] = L > 0.f ? exp2f(m_run[tid] - M) / L : 0.f;   // an empty denominator gives a zero output
        if (p.lse) p.lse[static_cast<int64_t>(t) * p.H + h] = L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
      } else {
        float* mlw = p.ws_ml + ((static_cast<int64_t>(t) * p.nsplit + split) * p.H + h) * 2;
        mlw[0] = m_run[tid];
        mlw[1] = l_run[tid];
      }
    }
    __syncthreads();
    if (finalize) {
      // normalised BF16 output staged as [head][512] in the (now idle) KV tile,
      // then written with 16-byte coalesced stores
      uint16_t* stage = reinterpret_cast<uint16_t*>(kv);
      const float4* rrow = rope_row(p, t);
      if (compute) {
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const uint32_t mb = hh * 2 + b;
          const int d = static_cast<int>(mb * 128 + g * 32 + lane);
          const uint32_t ta = tmem + ((g * 32u) << 16) + kColO + mb * HN;
          constexpr int kC = HN < 32 ? HN : 32;   // columns per batch
#pragma unroll
          for (int j0 = 0; j0 < HN; j0 += kC) {
            float v[kC];
            if (pv_issued) {
              tmem_load_cols<kC>(ta + j0, v);
            } else {
#pragma unroll
              for (int x = 0; x < kC; ++x) v[x] = 0.f;
            }
#pragma unroll
            for (int x = 0; x < kC; ++x) v[x] *= fac[j0 + x];
            if (rrow != nullptr && d >= 512 - 64) {   // warp-uniform: mb == 3, g >= 2
              // inverse rotary embedding: dims (d, d ^ 1) form one pair, held by lanes (l, l ^ 1)
              const float2 cs = __ldg(reinterpret_cast<const float2*>(rrow) + ((d - (512 - 64)) >> 1));
#pragma unroll
              for (int x = 0; x < kC; ++x) {
                const float other = __shfl_xor_sync(0xffffffffu, v[x], 1);
                v[x] = (lane & 1) ? fmaf(v[x], cs.x, -(other * cs.y)) : fmaf(v[x], cs.x, other * cs.y);
              }
            }
#pragma unroll
            for (int x = 0; x < kC; ++x) {
              const __nv_bfloat16 o = __float2bfloat16_rn(v[x]);
              stage[(j0 + x) * 512 + d] = *reinterpret_cast<const uint16_t*>(&o);
            }
          }
        }
      }
      __syncthreads();
      const int hreal = min(HN, p.H - h0);
      const uint4* src = reinterpret_cast<const uint4*>(stage);
      uint4* dst = reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(t) * p.H + h0) * 512);
      for (int u = tid; u < hreal * 64; u += kThreads) dst[u] = src[u];
    } else {
      // fp32 partial O, stored [t][split][dim][head].  Staged through shared
      // memory (the idle KV and Q tiles, rows padded to HN + 4 floats so the
      // 16-byte stores of 8 consecutive dims hit distinct banks), then written
      // with coalesced 16-byte stores: with one head group per query the
      // CTA's partial is one contiguous block.
      constexpr int kLd = HN + 4;
      float* stage = reinterpret_cast<float*>(kv);
      if (compute) {
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const uint32_t mb = hh * 2 + b;
          const int d = static_cast<int>(mb * 128 + g * 32 + lane);
          const uint32_t ta = tmem + ((g * 32u) << 16) + kColO + mb * HN;
          constexpr int kC = HN < 32 ? HN : 32;   // columns per batch
#pragma unroll
          for (int j0 = 0; j0 < HN; j0 += kC) {
            float v[kC];
            if (pv_issued) {
              tmem_load_cols<kC>(ta + j0, v);
            } else {
#pragma unroll
              for (int x = 0; x < kC; ++x) v[x] = 0.f;
            }
#pragma unroll
            for (int x = 0; x < kC; x += 4)
              *reinterpret_cast<float4*>(stage + d * kLd + j0 + x) = make_float4(v[x], v[x + 1], v[x + 2], v[x + 3]);
          }
        }
      }
      __syncthreads();
      float* wo = p.ws_o + (static_cast<int64_t>(t) * p.nsplit + split) * 512 * p.H + h0;
      const int hreal = min(HN, p.H - h0);
      if ((p.H & 3) == 0 && (hreal & 3) == 0) {
        const int q4 = hreal >> 2;
        for (int e = tid; e < 512 * q4; e += kThreads) {
          const int d = e / q4, c = e - d * q4;
          *reinterpret_cast<float4*>(wo + static_cast<int64_t>(d) * p.H + 4 * c) =
              *reinterpret_cast<const float4*>(stage + d * kLd + 4 * c);
        }
      } else {
        for (int e = tid; e < 512 * hreal; e += kThreads) {
          const int d = e / hreal, h = e - d * hreal;
          wo[static_cast<int64_t>(d) * p.H + h] = stage[d * kLd + h];
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Merge the split partials of one query over a 16-dim slab: log-sum-exp over
// the splits, the sink added once, BF16 output written after a transpose in
// shared memory.  Each thread owns 4 (dim, head) elements and issues all of
// their split loads before using any.
constexpr int kMergeThreads = 256;
constexpr int kMergeDims = 16;
constexpr int kMergeMaxSplits = 24;

__global__ void __launch_bounds__(kMergeThreads) attn_merge_kernel(const AttnParams p) {
  __shared__ float fac[kMergeMaxSplits][128];   // exp2(m_s - M) / L per split and head
  __shared__ float tile[kMergeDims][129];       // [dim][head] of this slab
  griddep_launch();
  griddep_wait();
  const int t = blockIdx.x, slab = blockIdx.y, tid = threadIdx.x;
  const int H = p.H, ns = p.nsplit;
  for (int h = tid; h < H; h += kMergeThreads) {
    const float sink2 = __ldg(p.sink + h) * kLog2e;
    float ms[kMergeMaxSplits], ls[kMergeMaxSplits];
    float M = sink2;
#pragma unroll
    for (int s = 0; s < kMergeMaxSplits; ++s) {
      if (s < ns) {
        const float2 ml = *reinterpret_cast<const float2*>(p.ws_ml + ((static_cast<int64_t>(t) * ns + s) * H + h) * 2);
        ms[s] = ml.x;
        ls[s] = ml.y;
        if (ml.y > 0.f) M = fmaxf(M, ml.x);
      }
    }
    float L = sink2 > -INFINITY ? exp2f(sink2 - M) : 0.f;   // a sink of -inf adds nothing
#pragma unroll
    for (int s = 0; s < kMergeMaxSplits; ++s) {
      if (s < ns) {
        const float f = ls[s] > 0.f ? exp2f(ms[s] - M) : 0.f;
        fac[s][h] = f;
        L += ls[s] * f;
      }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;   // an empty denominator gives a zero output
    for (int s = 0; s < ns; ++s) fac[s][h] *= inv;
    if (p.lse && slab == 0)
      p.lse[static_cast<int64_t>(t) * H + h] = L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
  }
  __syncthreads();
  // every split's partial is finite (zero where nothing was attended): no guards
  const int n_el = kMergeDims * H;
  const float* base = p.ws_o + (static_cast<int64_t>(t) * ns * 512 + slab * kMergeDims) * H;
  for (int e0 = 0; e0 < n_el; e0 += 4 * kMergeThreads) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int s = 0; s < ns; ++s) {
      float v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)   // clamped index: unconditional loads, all in flight
        v[i] = __ldg(base + static_cast<int64_t>(s) * 512 * H + min(e0 + tid + i * kMergeThreads, n_el - 1));
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int e = e0 + tid + i * kMergeThreads;
        if (e < n_el) acc[i] = fmaf(fac[s][e % H], v[i], acc[i]);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = e0 + tid + i * kMergeThreads;
      if (e < n_el) tile[e / H][e % H] = acc[i];
    }
  }
  __syncthreads();
  const float4* rrow = rope_row(p, t);
  for (int u = tid; u < H * 2; u += kMergeThreads) {
    const int h = u >> 1, c = (u & 1) * 8;
    float o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = tile[c + i][h];
    const int d0 = slab * kMergeDims + c;
    if (rrow != nullptr && d0 >= 512 - 64) {   // inverse rotary embedding of the last 64 dims
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float4 cs = __ldg(rrow + ((d0 - (512 - 64)) >> 2) + i);
        const float2 a = rotate_back(o[4 * i], o[4 * i + 1], cs.x, cs.y);
        const float2 b = rotate_back(o[4 * i + 2], o[4 * i + 3], cs.z, cs.w);
        o[4 * i] = a.x;
        o[4 * i + 1] = a.y;
        o[4 * i + 2] = b.x;
        o[4 * i + 3] = b.y;
      }
    }
    uint4 v;
    v.x = pack_bf16x2(o[0], o[1]);
    v.y = pack_bf16x2(o[2], o[3]);
    v.z = pack_bf16x2(o[4], o[5]);
    v.w = pack_bf16x2(o[6], o[7]);
    *reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(t) * H + h) * 512 + slab * kMergeDims + c) = v;
  }
}

template <int HN>
int launch_hn(const AttnParams& p, int groups, cudaStream_t stream) {
  static_assert(512 * (HN + 4) * 4 <= Smem<HN>::kP, "partial staging must fit in the KV and Q tiles");
  constexpr int bytes = Smem<HN>::kBytes + 1024;  // + alignment slack
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSV4SA_ERR_CUDA;
  if (!smem_attr_once(dev, HN / 16, reinterpret_cast<const void*>(sparse_attn_kernel<HN>), bytes))
    return DSV4SA_ERR_CUDA;
  if (launch_pdl(sparse_attn_kernel<HN>, dim3(p.nsplit, p.T, groups), dim3(kThreads), bytes, stream, p) !=
      cudaSuccess)
    return DSV4SA_ERR_CUDA;
  if (p.merge == kMergeWorkspace &&
      launch_pdl(attn_merge_kernel, dim3(p.T, 512 / kMergeDims), dim3(kMergeThreads), 0, stream, p) != cudaSuccess)
    return DSV4SA_ERR_CUDA;
  return DSV4SA_OK;
}

}  // namespace

int32_t attn_chunks(int32_t kc, int32_t kw) { return (kc + kw + kRows - 1) / kRows; }

// Upper bound of the splits a mode may use (sizes the workspace).
int32_t attn_splits(int32_t mode, int32_t kc, int32_t kw) {
  const int32_t n = attn_chunks(kc, kw);
  if (n <= 1 || mode != DSV4SA_ATTN_DECODE) return 1;
  return n > kMaxClusterSplits ? n : kMaxClusterSplits;
}

struct SplitPlan {
  int32_t nsplit;
  int32_t merge;
};

// How the rows of a query are split over CTAs.  Prefill: all rows in one CTA.
// Decode: up to sms / (queries x head groups) splits so the grid is one wave;
// each split takes an equal share of the window and of the compressed list.
// A power-of-two number (2, 4 or 8) of splits of at most 4 chunks each runs as
// a cluster that merges behind one cluster barrier, otherwise splits of at
// least one 128-row chunk merge in a second kernel.
static int32_t rows_of_split(int32_t kc, int32_t kw, int32_t n) {
  return (kc + n - 1) / n + (kw + n - 1) / n;
}

static SplitPlan plan_splits(int32_t mode, int32_t kc, int32_t kw, int32_t ctas_per_split, int32_t sms, int hn) {
  const SplitPlan none{1, kMergeNone};
  const int32_t rows = kc + kw;
  if (mode != DSV4SA_ATTN_DECODE || rows <= kRows) return none;
  int32_t max_splits = sms / (ctas_per_split > 0 ? ctas_per_split : 1);
  if (max_splits < 2) return none;
  const int32_t max_cluster = attn::decode_max_cluster(hn);
  int32_t cs = 1;
  while (cs * 2 <= max_splits && cs * 2 <= max_cluster) cs *= 2;
  if (cs >= 2 && rows_of_split(kc, kw, cs) <= 4 * kRows) return SplitPlan{cs, kMergeCluster};
  int32_t n = max_splits;
  const int32_t chunks = (rows + kRows - 1) / kRows;
  if (n > chunks) n = chunks;
  if (n <= 1) return none;
  return SplitPlan{n, kMergeWorkspace};
}

int attn_plan(int32_t mode, int32_t T, int32_t H, int32_t kc, int32_t kw, int32_t* nsplit, int32_t* rows_per_split,
              int32_t* launches) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSV4SA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return DSV4SA_ERR_CUDA;
  const int hn = H <= 16 ? 16 : (H <= 32 ? 32 : 64);
  const int groups = (H + hn - 1) / hn;
  const SplitPlan sp = plan_splits(mode, kc, kw, T * groups, sms, hn);
  if (nsplit) *nsplit = sp.nsplit;
  if (rows_per_split) *rows_per_split = rows_of_split(kc, kw, sp.nsplit);
  if (launches) *launches = T == 0 ? 0 : (sp.merge == kMergeWorkspace ? 2 : 1);
  return DSV4SA_OK;
}

// The launch parameters and plan of an attention call.
static int fill_params(int32_t mode, const dsv4sa_attn_args* a, AttnParams& p, int& hn, int& groups) {
  p.q = static_cast<const uint16_t*>(a->q);
  p.sink = a->attn_sink;
  p.q_seq = a->q_seq;
  p.kc = a->kc;
  p.kw = a->kw;
  if (a->kc > 0) {
    p.comp_base = static_cast<const uint8_t*>(a->comp->base);
    p.comp_page_stride = a->comp->page_stride;
    p.comp_num_pages = a->comp->num_pages;
    p.comp_pt = a->comp_pt;
    p.comp_pt_stride = a->comp_pt_stride;
    p.idx_c = a->idx_c;
    p.idx_c_stride = a->idx_c_stride;
  }
  if (a->kw > 0) {
    p.win_base = static_cast<const uint8_t*>(a->win->base);
    p.win_page_stride = a->win->page_stride;
    p.win_num_pages = a->win->num_pages;
    p.win_pt = a->win_pt;
    p.win_pt_stride = a->win_pt_stride;
    p.idx_w = a->idx_w;
    p.idx_w_stride = a->idx_w_stride;
    p.win_pos = a->win_pos;
    p.win_ring = a->win_ring;
  }
  if (a->rope_cs) {
    p.rope_cs = reinterpret_cast<const float4*>(a->rope_cs);
    p.rope_pos = a->rope_pos;
    p.rope_rows = a->rope_rows;
  }
  // rows of a missing list are never addressed; keep the pointers non-null
  if (!p.comp_pt) { p.comp_pt = a->q_seq; }
  if (!p.win_pt) { p.win_pt = a->q_seq; }
  p.any_page = a->kc > 0 ? p.comp_base : p.win_base;
  p.out = static_cast<uint16_t*>(a->out);
  p.lse = a->lse;
  p.T = a->T;
  p.H = a->H;
  p.scale_log2 = a->softmax_scale * kLog2e;
  hn = a->H <= 16 ? 16 : (a->H <= 32 ? 32 : 64);
  groups = (a->H + hn - 1) / hn;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSV4SA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return DSV4SA_ERR_CUDA;
  const SplitPlan sp = plan_splits(mode, a->kc, a->kw, a->T * groups, sms, hn);
  p.nsplit = sp.nsplit;
  p.merge = sp.merge;
  p.kc_split = (a->kc + sp.nsplit - 1) / sp.nsplit;
  p.kw_split = (a->kw + sp.nsplit - 1) / sp.nsplit;
  p.early_window = (a->flags & DSV4SA_ATTN_EARLY_WINDOW) ? 1 : 0;
  if (p.merge != kMergeNone) {
    const size_t o_bytes = static_cast<size_t>(a->T) * p.nsplit * a->H * 512 * sizeof(float);
    p.ws_o = static_cast<float*>(a->ws);
    p.ws_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(a->ws) + o_bytes);
  }
  return DSV4SA_OK;
}

int launch_sparse_attn(int32_t mode, const dsv4sa_attn_args* a, cudaStream_t stream) {
  AttnParams p{};
  int hn = 0, groups = 0;
  const int rc = fill_params(mode, a, p, hn, groups);
  if (rc != DSV4SA_OK || a->T == 0) return rc;
  if (mode == DSV4SA_ATTN_DECODE && p.merge == kMergeCluster) return attn::launch_decode_cluster(p, hn, groups, stream);
  switch (hn) {
    case 16: return launch_hn<16>(p, groups, stream);
    case 32: return launch_hn<32>(p, groups, stream);
    default: return launch_hn<64>(p, groups, stream);
  }
}

// Top-k then decode attention.  When the decode runs as clusters and each row
// has at most 16384 entries, one kernel does both (the CTAs of a query's cluster select its list, then gather it);
// otherwise the top-k kernel (prefetching the selected rows into L2) and the
// attention run one after the other.
int launch_topk_sparse_attn(const dsv4sa_attn_args* a, const float* logits, int64_t logits_stride,
                            const int32_t* n_vis, int32_t n_max, int32_t k, void* topk_ws, size_t topk_ws_bytes,
                            cudaStream_t stream) {
  AttnParams p{};
  int hn = 0, groups = 0;
  const int rc = fill_params(DSV4SA_ATTN_DECODE, a, p, hn, groups);
  if (rc != DSV4SA_OK || a->T == 0) return rc;
  const bool fuse = p.merge == kMergeCluster && k <= a->kc && n_max <= attn::kFusedMaxRow &&
                    p.kc_split <= attn::kFusedMaxSplitRows && reinterpret_cast<uintptr_t>(logits) % 16 == 0 &&
                    logits_stride % 4 == 0;
  if (fuse) {
    p.fused = 1;
    p.topk_k = k;
    p.n_max = n_max;
    p.logits = logits;
    p.logits_stride = logits_stride;
    p.n_vis = n_vis;
    p.idx_c_out = const_cast<int32_t*>(a->idx_c);
    return attn::launch_decode_cluster(p, hn, groups, stream);
  }
  const TopkPrefetch pf{a->comp, a->comp_pt, a->comp_pt_stride, a->q_seq};
  const int rt = launch_topk(logits, logits_stride, n_vis, a->T, n_max, k, const_cast<int32_t*>(a->idx_c),
                             a->idx_c_stride, topk_ws, topk_ws_bytes, stream, a->kc > 0 ? &pf : nullptr);
  if (rt != DSV4SA_OK) return rt;
  return launch_sparse_attn(DSV4SA_ATTN_DECODE, a, stream);
}

uint32_t read_error_word_attn(cudaStream_t stream, bool clear) {
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
