// writer.cu -- the KV-cache writer: new BF16 rows quantised into a paged pool.
//
// For each new row (an entry s of the sequence whose page-table row is
// row_seq[r]): every 64-value block of the quantised part gets
// amax = max(max |x|, 1e-4), scale = amax * fp32(1/448) and E4M3 codes
// RNE(clamp(x / scale, -448, 448)), all in fp32 ("DeepSeek-V4 全面解读" §3.4
// act_quant_kernel); the codes and the fp32 scale go to slot s % 64 of page
// page_table[row_seq[r]][s / 64] ("DeepSeek-V4 in SGLang" 概念5
// DeepSeekV4TokenToKVPool).  KV pool: 448 nope values quantised (7 blocks),
// 64 rope values stored as BF16 unchanged.  Indexer-key pool: 128 values
// quantised (2 blocks).
//
// FP4 indexer-key pool ("DeepSeek-V4 全面解读" §3.5 fp4_quant_kernel and §3.3
// fast_round_scale; "tilelang量化内核拆解…" 32-group E8M0 scales): every
// 32-value block gets e = ceil(log2(fp32(max(amax, 6 * 2^-126) * fp32(1/6)))),
// read off the fp32 exponent and mantissa fields, and E2M1 codes
// RNE(clamp(x * 2^-e, -6, 6)) -- x * 2^-e is x / 2^e exactly -- packed two per
// byte, value 2j in the low nibble; the scale is stored as the E8M0 byte e + 127.
//
// Each lane owns 16 consecutive values of a row (one 32-byte load), so a
// 64-value block is four neighbouring lanes (a 32-value FP4 block two) and a
// KV row (512 values) is one warp, an indexer key (128 values) a quarter warp.  The block's absmax is a
// max over the bit patterns of |x| (order-preserving for non-negative floats)
// across those four lanes; the 16 codes of a lane are one 16-byte store, so a
// block's 64 codes leave as one contiguous 64-byte piece.
#include "common.cuh"
#include "dsv4sa_internal.h"

namespace dsv4sa {
namespace {

constexpr int kThreads = 256;
constexpr float kFp8MaxInv = 1.0f / 448.0f;   // fp8_max_inv, rounded to fp32
constexpr float kAmaxFloor = 1e-4f;
constexpr float kFp4MaxInv = 1.0f / 6.0f;                     // fp4_max_inv, rounded to fp32
constexpr float kFp4AmaxFloor = 6.0f * 1.1754943508222875e-38f;   // 6 * 2^-126 (exact)

struct WriterParams {
  const int32_t* page_table;
  const int32_t* row_seq;
  const int32_t* row_entry;
  const uint4* rows;        // bf16 [n][row_len], 16-byte aligned
  uint8_t* base;
  int64_t page_stride;
  int64_t num_pages;
  int64_t nope_off;
  int64_t rope_off;
  int64_t scale_off;
  int32_t nope_row;
  int32_t rope_row;
  int32_t scale_row;
  int32_t pt_stride;
  int32_t n;
};

// A resident grid walks the rows grid-stride; a lane's next row (entry,
// sequence and its 32 bytes of values) is loaded while the current one is
// looked up, converted and stored, so the row loads stay in flight.
template <int kLanesPerRow, int kQuantBlocks>
__global__ void __launch_bounds__(kThreads) cache_write_kernel(const WriterParams p) {
  constexpr int kRowsPerWarp = 32 / kLanesPerRow;
  constexpr int kRowLen = kLanesPerRow * 16;
  griddep_launch();
  griddep_wait();   // the rows may come from the previous kernel of the stream
  const int lane = static_cast<int>(threadIdx.x & 31u);
  const int sub = lane / kLanesPerRow;           // row of the warp's group
  const int c = lane % kLanesPerRow;             // 16-value chunk of the row
  const bool rope = c >= kQuantBlocks * 4;       // KV rows: values 448..511
  const int64_t stride = static_cast<int64_t>(gridDim.x) * (kThreads / 32) * kRowsPerWarp;
  int64_t r = ((static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5) * kRowsPerWarp + sub;
  if (r - sub >= p.n) return;                    // warp-uniform
  // clamped rows: every lane loads, so the shuffles below see the full warp
  auto load = [&](int64_t row, int& s, int& seq, uint4& v0, uint4& v1) {
    const int64_t rc = row < p.n ? row : p.n - 1;
    s = __ldg(p.row_entry + rc);
    seq = __ldg(p.row_seq + rc);
    const uint4* src = p.rows + rc * (kRowLen / 8) + c * 2;
    v0 = __ldg(src);
    v1 = __ldg(src + 1);
  };
  int s, seq;
  uint4 v0, v1;
  load(r, s, seq, v0, v1);
  for (; r - sub < p.n; r += stride) {
    bool live = r < p.n;
    const bool ok = s >= 0 && (s >> 6) < p.pt_stride && seq >= 0;
    const int page = __ldg(p.page_table + static_cast<int64_t>(ok ? seq : 0) * p.pt_stride + (ok ? s >> 6 : 0));
    int s_next, seq_next;
    uint4 v0_next, v1_next;
    load(r + stride, s_next, seq_next, v0_next, v1_next);
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    uint32_t mag = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) mag = max(mag, max((w[j] << 16) & 0x7FFFFFFFu, w[j] & 0x7FFF0000u));
    mag = max(mag, __shfl_xor_sync(0xffffffffu, mag, 1));
    mag = max(mag, __shfl_xor_sync(0xffffffffu, mag, 2));
    if (live && (!ok || page < 0 || page >= p.num_pages)) {
      if (c == 0) raise_error(kErrIndex);
      live = false;
    }
    if (live) {
      const int slot = s & 63;
      uint8_t* pg = p.base + static_cast<int64_t>(page) * p.page_stride;
      if (rope) {                                 // stored as they are
        uint4* dst = reinterpret_cast<uint4*>(pg + p.rope_off + static_cast<int64_t>(slot) * p.rope_row) +
                     (c - kQuantBlocks * 4) * 2;
        dst[0] = v0;
        dst[1] = v1;
      } else {
        const float scale = __fmul_rn(fmaxf(__uint_as_float(mag), kAmaxFloor), kFp8MaxInv);
        uint32_t codes[4];
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
          uint32_t pair = 0;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float x0 = __uint_as_float(w[j + h] << 16), x1 = __uint_as_float(w[j + h] & 0xFFFF0000u);
            const float y0 = fminf(fmaxf(__fdiv_rn(x0, scale), -448.f), 448.f);
            const float y1 = fminf(fmaxf(__fdiv_rn(x1, scale), -448.f), 448.f);
            pair |= static_cast<uint32_t>(static_cast<uint16_t>(
                        __nv_cvt_float2_to_fp8x2(make_float2(y0, y1), __NV_SATFINITE, __NV_E4M3)))
                    << (16 * h);
          }
          codes[j / 2] = pair;
        }
        *reinterpret_cast<uint4*>(pg + p.nope_off + static_cast<int64_t>(slot) * p.nope_row + c * 16) =
            make_uint4(codes[0], codes[1], codes[2], codes[3]);
        if ((c & 3) == 0)
          reinterpret_cast<float*>(pg + p.scale_off + static_cast<int64_t>(slot) * p.scale_row)[c >> 2] = scale;
      }
    }
    s = s_next;
    seq = seq_next;
    v0 = v0_next;
    v1 = v1_next;
  }
}

// E2M1 code of an fp32 value in [-6, 6]: the nearest of 0, 0.5, 1, 1.5, 2, 3,
// 4, 6 with ties to the code whose mantissa bit is clear (0.25 -> 0, 0.75 -> 1,
// 1.25 -> 1, 1.75 -> 2, 2.5 -> 2, 3.5 -> 4, 5 -> 4), counted as the thresholds
// the magnitude passes; bit 3 is the sign (-0 -> 8).
__device__ __forceinline__ uint32_t e2m1_code(float y) {
  const float a = fabsf(y);
  const uint32_t m = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) + (a >= 3.5f) + (a > 5.0f);
  return m | ((__float_as_uint(y) >> 28) & 8u);
}

// fp32 nearest to 128^-0.5, the scale of the order-128 Hadamard rotation.
constexpr float kRot128 = 0x1.6a09e6p-4f;

// fp32 -> BF16 bits, round to nearest, ties to even (finite values).
__device__ __forceinline__ uint32_t bf16_bits_rne(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
}

// The order-128 Hadamard rotation of a key held 16 values a lane across the 8
// lanes of a quarter warp ("DeepSeek-V4 全面解读" §2.9, the compressor's rotate
// path): fp32 butterflies (a + b, a - b) of strides 1, 2, 4, 8 inside the lane,
// then 16, 32, 64 across lanes c ^ 1, c ^ 2, c ^ 4 (the lane holding the lower
// index keeps a + b), then the fp32 scale 128^-0.5 and one rounding to BF16.
// w holds the lane's 16 BF16 values, two per word, and receives the result.
__device__ __forceinline__ void hadamard128_bf16(uint32_t (&w)[8], int c) {
  float v[16];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    v[2 * j] = __uint_as_float(w[j] << 16);
    v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
  }
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if ((i & h) == 0) {
        const float a = v[i], b = v[i + h];
        v[i] = __fadd_rn(a, b);
        v[i + h] = __fsub_rn(a, b);
      }
    }
  }
#pragma unroll
  for (int m = 1; m < 8; m <<= 1) {
    const bool upper = (c & m) != 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, v[i], m);
      v[i] = upper ? __fsub_rn(o, v[i]) : __fadd_rn(v[i], o);
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j)
    w[j] = bf16_bits_rne(__fmul_rn(v[2 * j], kRot128)) | (bf16_bits_rne(__fmul_rn(v[2 * j + 1], kRot128)) << 16);
}

// Indexer keys into an IDXK_FP4 pool: a quarter warp per key, 16 values a
// lane, a 32-value block per lane pair; a lane's 16 codes leave as one 8-byte
// store, a key's four exponent bytes as one 4-byte store by its first lane.
// kRotate: each key is first rotated (hadamard128_bf16) and the rotated BF16
// values are quantised.
template <bool kRotate>
__global__ void __launch_bounds__(kThreads) fp4_key_write_kernel(const WriterParams p) {
  griddep_launch();
  griddep_wait();   // the rows may come from the previous kernel of the stream
  const int lane = static_cast<int>(threadIdx.x & 31u);
  const int sub = lane >> 3, c = lane & 7;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * (kThreads / 32) * 4;
  for (int64_t r0 = ((static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5) * 4; r0 < p.n;
       r0 += stride) {   // warp-uniform: every lane takes part in the shuffles
    const int64_t r = r0 + sub;
    bool live = r < p.n;
    const int64_t rc = live ? r : p.n - 1;
    const int s = __ldg(p.row_entry + rc), seq = __ldg(p.row_seq + rc);
    const uint4* src = p.rows + rc * 16 + c * 2;
    const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
    uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    if constexpr (kRotate) hadamard128_bf16(w, c);
    uint32_t mag = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) mag = max(mag, max((w[j] << 16) & 0x7FFFFFFFu, w[j] & 0x7FFF0000u));
    mag = max(mag, __shfl_xor_sync(0xffffffffu, mag, 1));   // the block's lane pair
    const float t = __fmul_rn(fmaxf(__uint_as_float(mag), kFp4AmaxFloor), kFp4MaxInv);
    const uint32_t tb = __float_as_uint(t);                 // normal: t >= 2^-126
    const int e = static_cast<int>((tb >> 23) & 0xFFu) - 127 + ((tb & 0x7FFFFFu) != 0u ? 1 : 0);
    const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);   // 2^-e, e in [-126, 126]
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float x0 = __uint_as_float(w[j] << 16), x1 = __uint_as_float(w[j] & 0xFFFF0000u);
      const uint32_t byte = e2m1_code(fminf(fmaxf(__fmul_rn(x0, inv), -6.f), 6.f)) |
                            (e2m1_code(fminf(fmaxf(__fmul_rn(x1, inv), -6.f), 6.f)) << 4);
      if (j < 4) lo |= byte << (8 * j);
      else hi |= byte << (8 * (j - 4));
    }
    // the four exponent bytes of the key, from lanes 0, 2, 4, 6 of its quarter warp
    const uint32_t eb = static_cast<uint32_t>(e + 127);
    const int q0 = lane & ~7;
    const uint32_t e8 = __shfl_sync(0xffffffffu, eb, q0) | (__shfl_sync(0xffffffffu, eb, q0 + 2) << 8) |
                        (__shfl_sync(0xffffffffu, eb, q0 + 4) << 16) | (__shfl_sync(0xffffffffu, eb, q0 + 6) << 24);
    const bool ok = s >= 0 && (s >> 6) < p.pt_stride && seq >= 0;
    const int page = __ldg(p.page_table + static_cast<int64_t>(ok ? seq : 0) * p.pt_stride + (ok ? s >> 6 : 0));
    if (live && (!ok || page < 0 || page >= p.num_pages)) {
      if (c == 0) raise_error(kErrIndex);
      live = false;
    }
    if (live) {
      const int slot = s & 63;
      uint8_t* pg = p.base + static_cast<int64_t>(page) * p.page_stride;
      *reinterpret_cast<uint2*>(pg + p.nope_off + static_cast<int64_t>(slot) * p.nope_row + c * 8) =
          make_uint2(lo, hi);
      if (c == 0) *reinterpret_cast<uint32_t*>(pg + p.scale_off + static_cast<int64_t>(slot) * p.scale_row) = e8;
    }
  }
}

template <int kLanesPerRow, int kQuantBlocks>
cudaError_t launch_writer(const WriterParams& p, cudaStream_t stream) {
  static int resident = 0;                       // CTAs per SM, queried once
  if (resident == 0 &&
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, cache_write_kernel<kLanesPerRow, kQuantBlocks>,
                                                    kThreads, 0) != cudaSuccess)
    return cudaErrorUnknown;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorUnknown;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return cudaErrorUnknown;
  const int64_t rows_per_block = static_cast<int64_t>(kThreads / 32) * (32 / kLanesPerRow);
  const int64_t want = (p.n + rows_per_block - 1) / rows_per_block;
  const int64_t full = static_cast<int64_t>(sms) * (resident > 0 ? resident : 1);
  const int64_t blocks = want < full ? want : full;
  return launch_pdl(cache_write_kernel<kLanesPerRow, kQuantBlocks>, dim3(static_cast<unsigned>(blocks)),
                    dim3(kThreads), 0, stream, p);
}

}  // namespace

int launch_cache_write(const dsv4sa_pool_desc* pool, const int32_t* page_table, int32_t pt_stride,
                       const int32_t* row_seq, const int32_t* row_entry, const void* rows, int32_t n,
                       bool rotate, cudaStream_t stream) {
  WriterParams p{};
  const bool kv = pool->kind == DSV4SA_POOL_KV;
  p.page_table = page_table;
  p.row_seq = row_seq;
  p.row_entry = row_entry;
  p.rows = static_cast<const uint4*>(rows);
  p.base = static_cast<uint8_t*>(pool->base);
  p.page_stride = pool->page_stride;
  p.num_pages = pool->num_pages;
  p.nope_off = pool->nope_off;
  p.rope_off = pool->rope_off;
  p.scale_off = pool->scale_off;
  p.nope_row = pool->nope_row;
  p.rope_row = pool->rope_row;
  p.scale_row = pool->scale_row;
  p.pt_stride = pt_stride;
  p.n = n;
  if (n == 0) return DSV4SA_OK;
  if (pool->kind == DSV4SA_POOL_IDXK_FP4) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DSV4SA_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return DSV4SA_ERR_CUDA;
    const int64_t rows_per_block = (kThreads / 32) * 4;
    const int64_t want = (static_cast<int64_t>(n) + rows_per_block - 1) / rows_per_block;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    const int64_t blocks = want < cap ? want : cap;
    const cudaError_t e =
        rotate ? launch_pdl(fp4_key_write_kernel<true>, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0,
                            stream, p)
               : launch_pdl(fp4_key_write_kernel<false>, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0,
                            stream, p);
    return e == cudaSuccess ? DSV4SA_OK : DSV4SA_ERR_CUDA;
  }
  if (rotate) return DSV4SA_ERR_UNSUPPORTED;   // rotation is the FP4 key path only
  const cudaError_t e = kv ? launch_writer<32, 7>(p, stream) : launch_writer<8, 2>(p, stream);
  return e == cudaSuccess ? DSV4SA_OK : DSV4SA_ERR_CUDA;
}

uint32_t read_error_word_writer(cudaStream_t stream, bool clear) {
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
