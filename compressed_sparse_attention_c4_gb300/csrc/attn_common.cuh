// attn_common.cuh -- pieces shared by the two sparse-attention kernel files:
// the launch parameters, the default KV page layout offsets, the inverse-RoPE
// helpers, the transposing warp reduction, TMEM column loads and the FP8 -> BF16
// dequantisation of 16 codes.  ("DeepSeek-V4 全面解读" §3.7 sparse_attn_kernel;
// "DeepSeek-V4 in SGLang" MQALayer: one kv tensor is both K and V.)
#pragma once

#include <cmath>

#include "common.cuh"
#include "dsv4sa_internal.h"

namespace dsv4sa {
namespace attn {

constexpr int kRows = 128;               // gathered rows per chunk = MMA M
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
  const int32_t* win_pos;   // window indices from positions when idx_w is null
  const float4* rope_cs;    // (cos, sin) pairs [rope_rows][32] as float4 [rope_rows][16], or null
  const int32_t* rope_pos;
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
  int32_t win_ring;
  int32_t T;
  int32_t H;
  int32_t kc_split;         // compressed rows per CTA (the split's share of kc)
  int32_t kw_split;         // window rows per CTA (the split's share of kw)
  int32_t nsplit;
  int32_t early_window;     // the window rows' inputs may be read before griddep_wait
  int32_t merge;            // kMergeNone / kMergeWorkspace / kMergeCluster
  int32_t rope_rows;
  float scale_log2;
  // Decode with the top-k inside (attn_decode.cu): query t's compressed list is
  // selected by the CTAs of its cluster from logits[t][0 .. n_vis[t]) (the
  // topk_k largest, ascending, -1 padded to kc) and written to idx_c_out; a row
  // with n_vis[t] < 0 keeps the list it has in idx_c.
  int32_t fused;
  int32_t topk_k;           // entries selected per row (<= kc; list slots past k are -1)
  int32_t n_max;
  const float* logits;
  const int32_t* n_vis;
  int32_t* idx_c_out;
  int64_t logits_stride;
};

// How the splits of one query are combined.
constexpr int kMergeNone = 0;        // one CTA per query: normalise in the epilogue
constexpr int kMergeWorkspace = 1;   // fp32 partials in the workspace, merged by attn_merge_kernel
constexpr int kMergeCluster = 2;     // the splits form a thread-block cluster and merge through the L2 workspace
constexpr int kMaxClusterSplits = 8;

// Inverse rotary embedding of the output: the rotation table row of query t
// (16 float4 = 32 (cos, sin) pairs), or null when there is no rotation or the
// position is out of range (flagged).
__device__ __forceinline__ const float4* rope_row(const AttnParams& p, int t) {
  if (p.rope_cs == nullptr) return nullptr;
  const int r = __ldg(p.rope_pos + t);
  if (r < 0 || r >= p.rope_rows) {
    if (threadIdx.x == 0) raise_error(kErrIndex);
    return nullptr;
  }
  return p.rope_cs + static_cast<int64_t>(r) * 16;
}

// (x + i y) times the conjugate of (c + i s)
__device__ __forceinline__ float2 rotate_back(float x, float y, float c, float s) {
  return make_float2(fmaf(x, c, y * s), fmaf(y, c, -(x * s)));
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

// N consecutive TMEM columns of this thread's lane (N a multiple of 8), all
// loads issued before the one wait.
template <int N>
__device__ __forceinline__ void tmem_load_cols(uint32_t ta, float* v) {
  static_assert(N % 4 == 0, "whole 4-column loads");
#pragma unroll
  for (int j = 0; j + 32 <= N; j += 32) tmem_ld32(ta + j, v + j);
  constexpr int j16 = N / 32 * 32;
  if (N - j16 >= 16) tmem_ld16(ta + j16, v + j16);
  constexpr int j8 = j16 + (N - j16) / 16 * 16;
  if (N - j8 >= 8) tmem_ld8(ta + j8, v + j8);
  constexpr int j4 = j8 + (N - j8) / 8 * 8;
  if (N - j4 >= 4) tmem_ld4(ta + j4, v + j4);
  tmem_ld_wait();
}

// 16 E4M3 codes times one fp32 scale -> 16 BF16 values (two 16-byte units).
__device__ __forceinline__ void dequant16(const uint4 codes, float scale, uint4& lo, uint4& hi) {
  const uint32_t w[4] = {codes.x, codes.y, codes.z, codes.w};
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2_raw h01 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[i] & 0xFFFFu), __NV_E4M3);
    const __half2_raw h23 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[i] >> 16), __NV_E4M3);
    const float2 s2 = make_float2(scale, scale);
    const float2 f01 = mul2(__half22float2(*reinterpret_cast<const __half2*>(&h01)), s2);
    const float2 f23 = mul2(__half22float2(*reinterpret_cast<const __half2*>(&h23)), s2);
    o[2 * i] = pack_bf16x2(f01.x, f01.y);
    o[2 * i + 1] = pack_bf16x2(f23.x, f23.y);
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// Decode attention whose splits form a thread-block cluster (attn_decode.cu):
// p.nsplit = cluster size (2, 4 or 8), hn = heads per CTA (16, 32 or 64).
int launch_decode_cluster(const AttnParams& p, int hn, int groups, cudaStream_t stream);
// The largest cluster that kernel supports for hn heads per CTA (its merge slots fit in shared memory).
int decode_max_cluster(int hn);
// The longest row the decode kernel selects from itself (fused top-k), and the
// most compressed rows a CTA may take in that mode.
constexpr int kFusedMaxRow = 16384;
constexpr int kFusedMaxSplitRows = 256;

}  // namespace attn
}  // namespace dsv4sa
