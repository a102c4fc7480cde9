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
// 64) and one or more chunks of 128 gathered rows.  Per chunk:
//   1. gather: 256 threads fetch each valid row's 448 FP8 codes, 7 fp32 scales
//      and 64 BF16 rope values with 16-byte read-only loads, dequantise the
//      nope part to BF16 (hardware e4m3x2 -> f16x2 converts, fp32 scale) and
//      write a 128 x 512 BF16 tile in the 128-byte-swizzled layout the tensor
//      core reads; invalid rows become zero rows.
//   2. S^T = KV . Q^T on tcgen05 (kind::f16, M = 128 rows, N = heads, K = 512):
//      TMEM lane r holds the scores of row r for every head.
//   3. online softmax in the exp2 domain: per-head max and sum across the 128
//      rows with a transposing warp reduction plus a 4-way cross-warp step;
//      P is written to shared memory in BF16; the output accumulator is
//      rescaled in TMEM when the running max moves.
//   4. O^T += V^T . P^T on tcgen05 (M = 128 dims per block, 4 blocks, N = heads,
//      K = 128 rows); the KV tile is read MN-major, so the same shared tile
//      serves as K (K-major) and V (MN-major).
// Decode splits the rows of a query across CTAs (one chunk each) and merges the
// partial (O, max, sum) triples by log-sum-exp in a second kernel, adding the
// sink once; prefill runs all chunks of a query in one CTA and writes the
// normalised BF16 output directly.
#include <cmath>

#include "common.cuh"
#include "dsv4sa_internal.h"

namespace dsv4sa {
namespace {

constexpr int kRows = 128;               // gathered rows per chunk = MMA M
constexpr int kThreads = 256;
constexpr int kKvBlock = kRows * 128;    // bytes of one 64-dim column block of the tile
constexpr int kKvBytes = 8 * kKvBlock;   // 128 x 512 BF16
constexpr int kPageRopeOff = 28672;      // default KV page layout (see dsv4sa.h)
constexpr int kPageScaleOff = 36864;
constexpr float kLog2e = 1.4426950408889634f;

struct AttnParams {
  const uint16_t* q;
  const float* sink;
  const int32_t* q_seq;
  const uint8_t* any_page;   // a valid page address used for masked-off loads
  const uint8_t* comp_base;
  const int32_t* comp_pt;
  const int32_t* idx_c;
  const uint8_t* win_base;
  const int32_t* win_pt;
  const int32_t* idx_w;
  uint16_t* out;
  float* lse;
  float* ws_o;
  float* ws_ml;
  int64_t comp_page_stride;
  int64_t comp_num_pages;
  int64_t win_page_stride;
  int64_t win_num_pages;
  int32_t comp_pt_stride;
  int32_t idx_c_stride;
  int32_t kc;
  int32_t win_pt_stride;
  int32_t idx_w_stride;
  int32_t kw;
  int32_t T;
  int32_t H;
  int32_t rows_per_split;   // gathered rows handled by one CTA (in chunks of 128)
  int32_t nsplit;
  int32_t merge;            // kMergeNone / kMergeWorkspace / kMergeCluster
  float scale_log2;
};

// How the splits of one query are combined.
constexpr int kMergeNone = 0;        // one CTA per query: normalise in the epilogue
constexpr int kMergeWorkspace = 1;   // fp32 partials in the workspace, merged by attn_merge_kernel
constexpr int kMergeCluster = 2;     // the splits form a thread-block cluster and merge through DSMEM
constexpr int kMaxClusterSplits = 8;

template <int HN>
struct Smem {
  static constexpr int kKv = 0;
  static constexpr int kQ = kKvBytes;                 // 8 column blocks x HN rows x 128 B
  static constexpr int kP = kQ + 8 * HN * 128;        // 2 row blocks x HN rows x 128 B
  static constexpr int kRowp = kP + 2 * HN * 128;     // uint64 [128]
  static constexpr int kRedMax = kRowp + kRows * 8;   // float [4][HN]
  static constexpr int kRedSum = kRedMax + 4 * HN * 4;
  static constexpr int kMRun = kRedSum + 4 * HN * 4;  // float [HN] each
  static constexpr int kLRun = kMRun + HN * 4;
  static constexpr int kAlpha = kLRun + HN * 4;
  static constexpr int kFac = kAlpha + HN * 4;
  static constexpr int kMl = kFac + HN * 4;           // float2 [HN]: (max, sum) shared with the cluster
  static constexpr int kBar = kMl + HN * 8;           // 2 mbarriers
  static constexpr int kTmem = kBar + 16;
  static constexpr int kBytes = kTmem + 16;
};

// One thread polls, the whole block learns the outcome.
__device__ __forceinline__ bool block_wait(uint64_t* bar, uint32_t parity) {
  int bad = 0;
  if (threadIdx.x == 0) bad = mbar_wait(bar, parity) ? 0 : 1;
  return __syncthreads_or(bad) == 0;
}

// Transposing warp reduction: each lane starts with L values (one per head);
// after the call lane l holds the reduction over all 32 lanes of head
// l >> log2(32 / L).  Uses L - 1 + log2(32 / L) shuffles instead of 5 L.
template <int L>
struct TransposeReduce {
  template <class Op>
  __device__ __forceinline__ static float run(float* v, uint32_t lane, uint32_t s, Op op) {
    const bool upper = (lane & s) != 0;
#pragma unroll
    for (int i = 0; i < L / 2; ++i) {
      const float send = upper ? v[i] : v[i + L / 2];
      const float keep = upper ? v[i + L / 2] : v[i];
      v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, s));
    }
    return TransposeReduce<L / 2>::run(v, lane, s >> 1, op);
  }
};
template <>
struct TransposeReduce<1> {
  template <class Op>
  __device__ __forceinline__ static float run(float* v, uint32_t, uint32_t s, Op op) {
    float x = v[0];
    for (; s > 0; s >>= 1) x = op(x, __shfl_xor_sync(0xffffffffu, x, s));
    return x;
  }
};
struct OpMax {
  __device__ __forceinline__ float operator()(float a, float b) const { return fmaxf(a, b); }
};
struct OpAdd {
  __device__ __forceinline__ float operator()(float a, float b) const { return a + b; }
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// 16 E4M3 codes times one fp32 scale -> 16 BF16 values (two 16-byte units).
__device__ __forceinline__ void dequant16(const uint4 codes, float scale, uint4& lo, uint4& hi) {
  const uint32_t w[4] = {codes.x, codes.y, codes.z, codes.w};
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2_raw h01 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[i] & 0xFFFFu), __NV_E4M3);
    const __half2_raw h23 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[i] >> 16), __NV_E4M3);
    const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
    const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
    o[2 * i] = pack_bf16x2(f01.x * scale, f01.y * scale);
    o[2 * i + 1] = pack_bf16x2(f23.x * scale, f23.y * scale);
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

template <int HN>
__global__ void __launch_bounds__(kThreads, 1) sparse_attn_kernel(const AttnParams p) {
  using S = Smem<HN>;
  extern __shared__ uint8_t smem_raw[];
  // 128-byte swizzled operand tiles need 1024-byte aligned bases
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* kv = smem + S::kKv;
  uint8_t* qs = smem + S::kQ;
  uint8_t* ps = smem + S::kP;
  uint64_t* rowp = reinterpret_cast<uint64_t*>(smem + S::kRowp);
  float* red_max = reinterpret_cast<float*>(smem + S::kRedMax);
  float* red_sum = reinterpret_cast<float*>(smem + S::kRedSum);
  float* m_run = reinterpret_cast<float*>(smem + S::kMRun);
  float* l_run = reinterpret_cast<float*>(smem + S::kLRun);
  float* alpha = reinterpret_cast<float*>(smem + S::kAlpha);
  float* fac = reinterpret_cast<float*>(smem + S::kFac);
  uint64_t* bar_s = reinterpret_cast<uint64_t*>(smem + S::kBar);
  uint64_t* bar_o = bar_s + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + S::kTmem);

  constexpr int HW = HN / 2;  // heads handled per warp in the softmax
  constexpr uint32_t kTmemCols = HN == 64 ? 512u : (HN == 32 ? 256u : 128u);
  constexpr uint32_t kColS = 0, kColO = HN;

  const int split = blockIdx.x;
  const int t = blockIdx.y;
  const int h0 = blockIdx.z * HN;
  const int tid = threadIdx.x;
  const uint32_t warp = warp_id(), lane = lane_id();
  const uint32_t g = warp & 3u;           // TMEM lane group
  const uint32_t hh = warp >> 2;          // head half (softmax) / block pair (epilogue)

  if (tid == 0) {
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_holder, kTmemCols);
    tmem_relinquish();
  }
  griddep_launch();
  griddep_wait();  // q, indices and the pools may come from the previous kernel of the stream
  if (tid < HN) {
    m_run[tid] = -1e30f;
    l_run[tid] = 0.f;
  }
  // Q block of this head group -> swizzled K-major tile (8 column blocks of 64 dims)
  {
    // every load is issued before the first store: one memory latency for the block
    constexpr int kQIters = HN * 64 / kThreads;
    const uint4* qsrc = reinterpret_cast<const uint4*>(p.q);
    uint4 qv[kQIters];
#pragma unroll
    for (int i = 0; i < kQIters; ++i) {   // clamped head: unconditional loads, all in flight
      const int u = i * kThreads + tid, h = min(h0 + (u >> 6), p.H - 1);
      qv[i] = __ldg(qsrc + (static_cast<int64_t>(t) * p.H + h) * 64 + (u & 63));
    }
#pragma unroll
    for (int i = 0; i < kQIters; ++i)
      if (h0 + ((i * kThreads + tid) >> 6) >= p.H) qv[i] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int i = 0; i < kQIters; ++i) {
      const int u = i * kThreads + tid, h = u >> 6, v = u & 63;
      *reinterpret_cast<uint4*>(qs + (v >> 3) * (HN * 128) + sw128_offset(h, v & 7)) = qv[i];
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  const int seq = __ldg(p.q_seq + t);
  const int32_t* cpt = p.comp_pt + static_cast<int64_t>(seq) * p.comp_pt_stride;
  const int32_t* wpt = p.win_pt + static_cast<int64_t>(seq) * p.win_pt_stride;
  const uint32_t idesc_s = make_idesc(kFmtBF16, kFmtBF16, 0, 0, 128, HN);
  const uint32_t idesc_o = make_idesc(kFmtBF16, kFmtBF16, 1, 0, 128, HN);
  uint32_t ph_s = 0, ph_o = 0;
  bool pv_issued = false;   // O holds a partial sum
  bool pv_pending = false;  // a PV MMA was issued and not waited for
  bool ok = true;

  const int r_begin = split * p.rows_per_split;
  const int r_end = min(p.kc + p.kw, r_begin + p.rows_per_split);
  for (int c0 = r_begin; c0 < r_end; c0 += kRows) {
    const int c_rows = min(kRows, r_end - c0);   // rows of this chunk
    // ---- 1. row addresses of this chunk (rowp is not read by any MMA in flight)
    int valid = 0;
    if (tid < kRows) {
      // index and page-id loads are issued unconditionally from clamped (always
      // valid) addresses, then masked: two dependent memory latencies per chunk
      const int gi = c0 + tid;
      const bool in_c = tid < c_rows && gi < p.kc;
      const bool in_w = tid < c_rows && !in_c && gi < p.kc + p.kw;
      const int32_t ec = p.kc > 0 ? __ldg(p.idx_c + static_cast<int64_t>(t) * p.idx_c_stride + min(gi, p.kc - 1)) : -1;
      const int32_t ew = p.kw > 0 ? __ldg(p.idx_w + static_cast<int64_t>(t) * p.idx_w_stride +
                                          min(max(gi - p.kc, 0), p.kw - 1))
                                  : -1;
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
      rowp[tid] = rp;
      valid = rp != 0;
    }
    if (__syncthreads_count(valid) == 0) continue;  // nothing to attend in this chunk
    // the previous chunk's PV reads the KV tile and P and writes O: wait for it
    if (pv_pending) {
      ok = block_wait(bar_o, ph_o);
      ph_o ^= 1u;
      pv_pending = false;
      if (!ok) break;
      tc_fence_after();
    }

    // ---- 2. gather + dequantise into the swizzled BF16 tile.  A task is one
    // 64-dim group of one row: 64 FP8 codes + their scale (nope groups 0-6) or
    // 32 BF16 rope values (half of group 7).  Consecutive lanes take
    // consecutive groups of a row, so a warp reads contiguous row segments.
    {
      // task k -> row r = 8 * (k / 72) + k % 8, group g = (k / 8) % 9: the 8 lanes
      // of a store phase hold 8 consecutive rows, whose 128-byte swizzle phases
      // differ, so the shared-memory stores are conflict-free
      constexpr int kTasks = kRows * 9;                       // 7 nope groups + 2 rope halves
      constexpr int kIters = (kTasks + kThreads - 1) / kThreads;
      uint4 raw[kIters][4];
      float scl[kIters];
      bool valid_task[kIters];
#pragma unroll
      for (int it = 0; it < kIters; ++it) {
        const int k = it * kThreads + tid;
        const int r = (k / 72) * 8 + (k & 7), g = (k >> 3) % 9;
        // invalid rows read slot 0 of the pool's first page (always valid) and
        // are zeroed afterwards: the loads are unconditional, so all are in flight
        const uint64_t rp0 = k < kTasks ? rowp[r] : 0;
        const uint64_t rp = rp0 ? rp0 : reinterpret_cast<uint64_t>(p.any_page);
        const uint8_t* page = reinterpret_cast<const uint8_t*>(rp & ~uint64_t(63));
        const int slot = static_cast<int>(rp & 63);
        const int gg = g < 7 ? g : 0;
        const uint4* src = g < 7 ? reinterpret_cast<const uint4*>(page + slot * 448 + g * 64)
                                 : reinterpret_cast<const uint4*>(page + kPageRopeOff + slot * 128 + (g - 7) * 64);
#pragma unroll
        for (int x = 0; x < 4; ++x) raw[it][x] = __ldg(src + x);
        scl[it] = __ldg(reinterpret_cast<const float*>(page + kPageScaleOff + slot * 32) + gg);
        valid_task[it] = rp0 != 0;
      }
#pragma unroll
      for (int it = 0; it < kIters; ++it) {
        if (!valid_task[it]) {
          scl[it] = 0.f;
#pragma unroll
          for (int x = 0; x < 4; ++x) raw[it][x] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
#pragma unroll
      for (int it = 0; it < kIters; ++it) {
        const int k = it * kThreads + tid;
        if (k >= kTasks) continue;
        const int r = (k / 72) * 8 + (k & 7), g = (k >> 3) % 9;
        if (g < 7) {
          uint8_t* blk = kv + g * kKvBlock;
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            uint4 lo, hi;
            dequant16(raw[it][x], scl[it], lo, hi);
            *reinterpret_cast<uint4*>(blk + sw128_offset(r, 2 * x)) = lo;
            *reinterpret_cast<uint4*>(blk + sw128_offset(r, 2 * x + 1)) = hi;
          }
        } else {
#pragma unroll
          for (int x = 0; x < 4; ++x)
            *reinterpret_cast<uint4*>(kv + 7 * kKvBlock + sw128_offset(r, (g - 7) * 4 + x)) = raw[it][x];
        }
      }
    }
    fence_proxy_async_smem();
    __syncthreads();

    // ---- 3. S^T = KV . Q^T  (M = 128 rows, N = HN heads, K = 512)
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
    ok = block_wait(bar_s, ph_s);
    ph_s ^= 1u;
    if (!ok) break;
    tc_fence_after();

    // ---- 4. online softmax (exp2 domain)
    const int r = static_cast<int>(g * 32 + lane);
    const bool rvalid = rowp[r] != 0;
    float sv[HW];
    {
      const uint32_t ta = tmem + ((g * 32u) << 16) + kColS + hh * HW;
#pragma unroll
      for (int j = 0; j < HW; j += 16) tmem_ld16(ta + j, sv + j);
      tmem_ld_wait();
    }
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
    __syncthreads();
    if (tid < HN) {
      const float mc = fmaxf(fmaxf(red_max[tid], red_max[HN + tid]), fmaxf(red_max[2 * HN + tid], red_max[3 * HN + tid]));
      const float mo = m_run[tid];
      const float mn = fmaxf(mo, mc);
      alpha[tid] = exp2f(mo - mn);
      m_run[tid] = mn;
    }
    __syncthreads();
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
    // rescale the running output when the max moved (previous PV has completed)
    if (pv_issued) {
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const uint32_t mb = hh * 2 + b;
        const uint32_t ta = tmem + ((g * 32u) << 16) + kColO + mb * HN;
#pragma unroll
        for (int j = 0; j < HN; j += 16) {
          float v[16];
          tmem_ld16(ta + j, v);
          tmem_ld_wait();
#pragma unroll
          for (int x = 0; x < 16; ++x) v[x] *= alpha[j + x];
          tmem_st16(ta + j, v);
        }
      }
      tmem_st_wait();
    }
    tc_fence_before();
    __syncthreads();
    if (tid < HN) {
      l_run[tid] = l_run[tid] * alpha[tid] + (red_sum[tid] + red_sum[HN + tid]) +
                   (red_sum[2 * HN + tid] + red_sum[3 * HN + tid]);
    }

    // ---- 5. O^T += V^T . P^T  (M = 128 dims x 4 blocks, N = HN, K = 128 rows)
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

  // ---- epilogue
  if (ok && pv_pending) {
    ok = block_wait(bar_o, ph_o);
    ph_o ^= 1u;
    tc_fence_after();
  }
  __syncthreads();
  if (p.merge == kMergeCluster) {
    // The CTAs of a cluster hold the splits of one query.  Every CTA passes
    // every cluster barrier, whatever happened before, so none waits forever.
    //  1. each CTA publishes its per-head (max, sum); every CTA combines them
    //     with the sink into the same global max M and denominator L;
    //  2. each CTA writes its O scaled by exp2(m - M) / L as fp32 [head][512]
    //     into its own (idle) KV tile;
    //  3. CTA r sums the slices of dims it owns over all CTAs' tiles (DSMEM
    //     reads, fixed order) and writes them as BF16.
    float2* ml = reinterpret_cast<float2*>(smem + S::kMl);
    const bool have_o = ok && pv_issued;
    const uint32_t crank = cluster_ctarank();
    const int csize = p.nsplit;
    if (tid < HN) ml[tid] = make_float2(m_run[tid], have_o ? l_run[tid] : 0.f);
    cluster_sync();
    if (tid < HN) {
      const int h = h0 + tid;
      const float sink2 = h < p.H ? __ldg(p.sink + h) * kLog2e : 0.f;
      float M = sink2;
      for (int c = 0; c < csize; ++c) {
        const float2 v = ld_cluster_f2(cluster_map(ml + tid, static_cast<uint32_t>(c)));
        if (v.y > 0.f) M = fmaxf(M, v.x);
      }
      float L = exp2f(sink2 - M);
      for (int c = 0; c < csize; ++c) {
        const float2 v = ld_cluster_f2(cluster_map(ml + tid, static_cast<uint32_t>(c)));
        if (v.y > 0.f) L += v.y * exp2f(v.x - M);
      }
      const float2 mine = ml[tid];
      fac[tid] = mine.y > 0.f ? exp2f(mine.x - M) / L : 0.f;
      if (crank == 0 && p.lse && h < p.H) p.lse[static_cast<int64_t>(t) * p.H + h] = (M + log2f(L)) * 0.6931471805599453f;
    }
    __syncthreads();
    float* stage = reinterpret_cast<float*>(kv);   // [HN][512]
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const uint32_t mb = hh * 2 + b;
      const int d = static_cast<int>(mb * 128 + g * 32 + lane);
      const uint32_t ta = tmem + ((g * 32u) << 16) + kColO + mb * HN;
#pragma unroll
      for (int j = 0; j < HN; j += 16) {
        float v[16];
        if (have_o) {
          tmem_ld16(ta + j, v);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int x = 0; x < 16; ++x) v[x] = 0.f;
        }
#pragma unroll
        for (int x = 0; x < 16; ++x) stage[(j + x) * 512 + d] = v[x] * fac[j + x];
      }
    }
    cluster_sync();
    {
      // dims in groups of 4; CTA crank owns groups [q0, q1)
      const int q0 = static_cast<int>(crank) * 128 / csize, q1 = (static_cast<int>(crank) + 1) * 128 / csize;
      const int nq = q1 - q0;
      const int hreal = min(HN, p.H - h0);
      uint32_t peer[kMaxClusterSplits];
#pragma unroll
      for (int c = 0; c < kMaxClusterSplits; ++c) peer[c] = c < csize ? cluster_map(stage, static_cast<uint32_t>(c)) : 0u;
      for (int e = tid; e < hreal * nq; e += kThreads) {
        const int h = e / nq, q = q0 + (e - h * nq);
        const uint32_t off = static_cast<uint32_t>((h * 512 + 4 * q) * 4);
        float4 acc = ld_cluster_f4(peer[0] + off);
#pragma unroll
        for (int c = 1; c < kMaxClusterSplits; ++c) {
          if (c < csize) {
            const float4 v = ld_cluster_f4(peer[c] + off);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
          }
        }
        uint2 o;
        o.x = pack_bf16x2(acc.x, acc.y);
        o.y = pack_bf16x2(acc.z, acc.w);
        *reinterpret_cast<uint2*>(p.out + (static_cast<int64_t>(t) * p.H + h0 + h) * 512 + 4 * q) = o;
      }
    }
    cluster_sync();   // no CTA leaves while a peer may still read its tile
  } else if (ok) {
    const bool finalize = p.nsplit == 1;
    if (tid < HN && h0 + tid < p.H) {
      const int h = h0 + tid;
      if (finalize) {
        const float sink2 = __ldg(p.sink + h) * kLog2e;
        const float M = fmaxf(m_run[tid], sink2);
        const float L = l_run[tid] * exp2f(m_run[tid] - M) + exp2f(sink2 - M);
        fac[tid] = exp2f(m_run[tid] - M) / L;
        if (p.lse) p.lse[static_cast<int64_t>(t) * p.H + h] = (M + log2f(L)) * 0.6931471805599453f;
      } else {
        float* ml = p.ws_ml + ((static_cast<int64_t>(t) * p.nsplit + split) * p.H + h) * 2;
        ml[0] = m_run[tid];
        ml[1] = l_run[tid];
      }
    }
    __syncthreads();
    if (finalize) {
      // normalised BF16 output staged as [head][512] in the (now idle) KV tile,
      // then written with 16-byte coalesced stores
      uint16_t* stage = reinterpret_cast<uint16_t*>(kv);
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const uint32_t mb = hh * 2 + b;
        const int d = static_cast<int>(mb * 128 + g * 32 + lane);
        const uint32_t ta = tmem + ((g * 32u) << 16) + kColO + mb * HN;
#pragma unroll
        for (int j = 0; j < HN; j += 16) {
          float v[16];
          if (pv_issued) {
            tmem_ld16(ta + j, v);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int x = 0; x < 16; ++x) v[x] = 0.f;
          }
#pragma unroll
          for (int x = 0; x < 16; ++x) {
            const __nv_bfloat16 o = __float2bfloat16_rn(v[x] * fac[j + x]);
            stage[(j + x) * 512 + d] = *reinterpret_cast<const uint16_t*>(&o);
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
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const uint32_t mb = hh * 2 + b;
        const int d = static_cast<int>(mb * 128 + g * 32 + lane);
        const uint32_t ta = tmem + ((g * 32u) << 16) + kColO + mb * HN;
#pragma unroll
        for (int j = 0; j < HN; j += 16) {
          float v[16];
          if (pv_issued) {
            tmem_ld16(ta + j, v);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int x = 0; x < 16; ++x) v[x] = 0.f;
          }
#pragma unroll
          for (int x = 0; x < 16; x += 4)
            *reinterpret_cast<float4*>(stage + d * kLd + j + x) = make_float4(v[x], v[x + 1], v[x + 2], v[x + 3]);
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
    float L = exp2f(sink2 - M);
#pragma unroll
    for (int s = 0; s < kMergeMaxSplits; ++s) {
      if (s < ns) {
        const float f = ls[s] > 0.f ? exp2f(ms[s] - M) : 0.f;
        fac[s][h] = f;
        L += ls[s] * f;
      }
    }
    const float inv = 1.f / L;
    for (int s = 0; s < ns; ++s) fac[s][h] *= inv;
    if (p.lse && slab == 0) p.lse[static_cast<int64_t>(t) * H + h] = (M + log2f(L)) * 0.6931471805599453f;
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
  for (int u = tid; u < H * 2; u += kMergeThreads) {
    const int h = u >> 1, c = (u & 1) * 8;
    uint4 v;
    v.x = pack_bf16x2(tile[c][h], tile[c + 1][h]);
    v.y = pack_bf16x2(tile[c + 2][h], tile[c + 3][h]);
    v.z = pack_bf16x2(tile[c + 4][h], tile[c + 5][h]);
    v.w = pack_bf16x2(tile[c + 6][h], tile[c + 7][h]);
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
  if (p.merge == kMergeCluster) {
    return launch_cluster_pdl(sparse_attn_kernel<HN>, dim3(p.nsplit, p.T, groups), dim3(kThreads), bytes, p.nsplit,
                              stream, p) == cudaSuccess
               ? DSV4SA_OK
               : DSV4SA_ERR_CUDA;
  }
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
  if (n == 0) return 1;
  return mode == DSV4SA_ATTN_DECODE ? n : 1;
}

// Rows per CTA.  Prefill: all rows of a query in one CTA.  Decode: split the
// rows so that (queries x head groups x splits) fills the GPU in one wave,
// with at least one full 128-row chunk per CTA.
static int32_t rows_per_split(int32_t mode, int32_t rows, int32_t ctas_per_split, int32_t sms) {
  if (mode != DSV4SA_ATTN_DECODE || rows <= kRows) return rows > 0 ? rows : 1;
  int32_t max_splits = sms / (ctas_per_split > 0 ? ctas_per_split : 1);
  if (max_splits < 1) max_splits = 1;
  int32_t rps = (rows + max_splits - 1) / max_splits;
  if (rps < kRows) rps = kRows;
  return rps;
}

int launch_sparse_attn(int32_t mode, const dsv4sa_attn_args* a, cudaStream_t stream) {
  AttnParams p{};
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
  const int hn = a->H <= 16 ? 16 : (a->H <= 32 ? 32 : 64);
  const int groups = (a->H + hn - 1) / hn;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSV4SA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return DSV4SA_ERR_CUDA;
  const int32_t rows = a->kc + a->kw;
  p.rows_per_split = rows_per_split(mode, rows, a->T * groups, sms);
  p.nsplit = rows > 0 ? (rows + p.rows_per_split - 1) / p.rows_per_split : 1;
  p.merge = p.nsplit == 1 ? kMergeNone : (p.nsplit <= kMaxClusterSplits ? kMergeCluster : kMergeWorkspace);
  if (p.merge == kMergeWorkspace) {
    const size_t o_bytes = static_cast<size_t>(a->T) * p.nsplit * a->H * 512 * sizeof(float);
    p.ws_o = static_cast<float*>(a->ws);
    p.ws_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(a->ws) + o_bytes);
  }
  if (a->T == 0) return DSV4SA_OK;
  switch (hn) {
    case 16: return launch_hn<16>(p, groups, stream);
    case 32: return launch_hn<32>(p, groups, stream);
    default: return launch_hn<64>(p, groups, stream);
  }
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
