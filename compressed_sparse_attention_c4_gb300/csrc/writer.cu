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
// One warp per (row, 64-value block): each lane holds two values, the block's
// absmax is a warp max over the bit patterns of |x| (order-preserving for
// non-negative floats), the pair is converted with one fp32x2 -> e4m3x2
// instruction and stored as two bytes, so a block's 64 codes are one coalesced
// 64-byte store.
#include "common.cuh"
#include "dsv4sa_internal.h"

namespace dsv4sa {
namespace {

constexpr int kThreads = 256;
constexpr float kFp8MaxInv = 1.0f / 448.0f;   // fp8_max_inv, rounded to fp32
constexpr float kAmaxFloor = 1e-4f;

struct WriterParams {
  const int32_t* page_table;
  const int32_t* row_seq;
  const int32_t* row_entry;
  const uint16_t* rows;     // bf16 [n][row_len]
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
  int32_t row_len;          // 512 (KV) or 128 (keys)
  int32_t quant_blocks;     // 7 or 2
  int32_t tasks_per_row;    // quant_blocks + (1 for the rope copy of a KV row)
};

__global__ void __launch_bounds__(kThreads) cache_write_kernel(const WriterParams p) {
  griddep_launch();
  griddep_wait();   // the rows may come from the previous kernel of the stream
  const int lane = static_cast<int>(threadIdx.x & 31u);
  const int64_t task = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  if (task >= static_cast<int64_t>(p.n) * p.tasks_per_row) return;
  const int r = static_cast<int>(task / p.tasks_per_row);
  const int b = static_cast<int>(task - static_cast<int64_t>(r) * p.tasks_per_row);
  const int32_t s = __ldg(p.row_entry + r);
  const int32_t seq = __ldg(p.row_seq + r);
  if (s < 0 || (s >> 6) >= p.pt_stride || seq < 0) {
    if (lane == 0) raise_error(kErrIndex);
    return;
  }
  const int32_t page = __ldg(p.page_table + static_cast<int64_t>(seq) * p.pt_stride + (s >> 6));
  if (page < 0 || page >= p.num_pages) {
    if (lane == 0) raise_error(kErrIndex);
    return;
  }
  const int slot = s & 63;
  uint8_t* pg = p.base + static_cast<int64_t>(page) * p.page_stride;
  const uint16_t* src = p.rows + static_cast<int64_t>(r) * p.row_len;
  if (b == p.quant_blocks) {   // rope: 64 BF16 values copied as they are
    const uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(src + 448) + lane);
    reinterpret_cast<uint32_t*>(pg + p.rope_off + static_cast<int64_t>(slot) * p.rope_row)[lane] = v;
    return;
  }
  const uint32_t pair = __ldg(reinterpret_cast<const uint32_t*>(src + b * 64) + lane);
  const float x0 = __uint_as_float(pair << 16), x1 = __uint_as_float(pair & 0xFFFF0000u);
  const uint32_t mag = max(__float_as_uint(x0) & 0x7FFFFFFFu, __float_as_uint(x1) & 0x7FFFFFFFu);
  const float amax = fmaxf(__uint_as_float(__reduce_max_sync(0xffffffffu, mag)), kAmaxFloor);
  const float scale = __fmul_rn(amax, kFp8MaxInv);
  const float y0 = fminf(fmaxf(__fdiv_rn(x0, scale), -448.f), 448.f);
  const float y1 = fminf(fmaxf(__fdiv_rn(x1, scale), -448.f), 448.f);
  const __nv_fp8x2_storage_t codes = __nv_cvt_float2_to_fp8x2(make_float2(y0, y1), __NV_SATFINITE, __NV_E4M3);
  reinterpret_cast<uint16_t*>(pg + p.nope_off + static_cast<int64_t>(slot) * p.nope_row + b * 64)[lane] =
      static_cast<uint16_t>(codes);
  if (lane == 0)
    reinterpret_cast<float*>(pg + p.scale_off + static_cast<int64_t>(slot) * p.scale_row)[b] = scale;
}

}  // namespace

int launch_cache_write(const dsv4sa_pool_desc* pool, const int32_t* page_table, int32_t pt_stride,
                       const int32_t* row_seq, const int32_t* row_entry, const void* rows, int32_t n,
                       cudaStream_t stream) {
  WriterParams p{};
  const bool kv = pool->kind == DSV4SA_POOL_KV;
  p.page_table = page_table;
  p.row_seq = row_seq;
  p.row_entry = row_entry;
  p.rows = static_cast<const uint16_t*>(rows);
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
  p.row_len = kv ? 512 : 128;
  p.quant_blocks = kv ? 7 : 2;
  p.tasks_per_row = kv ? 8 : 2;
  if (n == 0) return DSV4SA_OK;
  const int64_t warps = static_cast<int64_t>(n) * p.tasks_per_row;
  const int64_t blocks = (warps * 32 + kThreads - 1) / kThreads;
  if (blocks > 0x7FFFFFFF) return DSV4SA_ERR_UNSUPPORTED;
  return launch_pdl(cache_write_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0, stream, p) ==
                 cudaSuccess
             ? DSV4SA_OK
             : DSV4SA_ERR_CUDA;
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
