// compress.cu -- the KV compressor: windows of raw-token projections pooled
// into one compressed entry ("DeepSeek-V4 全面解读" §2.9 Compressor; "DeepSeek-V4
// in SGLang" 概念2 C4 / C128, 算法3 online C128).
//
// For one window: per feature f (512), the slot scores (score + ape of the
// token's place in its window) are softmax-normalised over the window's slots
// and weight the slot kv values; the pooled row is RMS-normalised (§2.5) with
// weight norm_w and its last 64 dims rotated forward by the (cos, sin) table
// row of the entry's position (§2.6), then rounded to BF16.  With the overlap
// transform (ratio 4) a window has 2r slots: the previous window's tokens,
// their first 512 features, then its own tokens, their last 512 features.
//
// Layout: one CTA of 128 threads per entry (or per token for the online form);
// thread i owns features 4i .. 4i + 3, so every slot row is one coalesced
// 1 KB read (8 bytes a thread) and the two rotary pairs of a thread's four
// features never leave the thread.  The softmax is a running max / sum over
// the slots in fp32, the RMS a block reduction.
#include "common.cuh"
#include "dsv4sa_internal.h"

namespace dsv4sa {
namespace {

constexpr int kThreads = 128;
constexpr int kDim = 512;
constexpr int kRopeFirst = kDim - 64;
constexpr int kBatch = 8;      // window slots whose loads are in flight together

struct CompressParams {
  const uint16_t* kv;        // bf16 rows, tok_stride elements apart
  const uint16_t* score;
  const int32_t* first_tok;  // windows: first token row of the window
  const int32_t* prev_tok;   // windows: first token row of the previous window, or -1
  const int32_t* position;   // table row of the entry
  const float* ape;          // [ratio][coff * 512]
  const float* norm_w;       // [512]
  const float4* rope_cs;     // [rope_rows][16] float4 = 32 (cos, sin) pairs
  uint16_t* out;             // bf16 [n][512]
  int64_t tok_stride;
  int64_t n_tok;             // windows: token rows in kv / score
  int32_t n;
  int32_t ratio;
  int32_t overlap;
  int32_t rope_rows;
  float eps;
  // online C128
  const int32_t* state_idx;
  float* state;              // [slots][3][512]: running max, sum, weighted kv
  int32_t* state_count;
  int32_t* done;
  int32_t slots;
};

__device__ __forceinline__ uint32_t to_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ void load4(const uint16_t* row, int f, float* v) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(row + f));
  v[0] = __uint_as_float(u.x << 16);
  v[1] = __uint_as_float(u.x & 0xFFFF0000u);
  v[2] = __uint_as_float(u.y << 16);
  v[3] = __uint_as_float(u.y & 0xFFFF0000u);
}

// Running softmax-weighted sum: fold one slot (score s, value x) into (m, l, a).
__device__ __forceinline__ void fold(float s, float x, float& m, float& l, float& a) {
  if (s == -INFINITY) return;
  const float mn = fmaxf(m, s);
  const float c = expf(m - mn);   // m = -inf at the start: c = 0
  const float e = expf(s - mn);
  l = fmaf(l, c, e);
  a = fmaf(a, c, e * x);
  m = mn;
}

// RMS-normalise, rotate (features 448..511) and store one entry; c[4] are the
// pooled values of this thread's features.  Every thread of the CTA calls it.
__device__ void finish_entry(const CompressParams& p, float* c, int pos, uint16_t* dst, float* red) {
  const int tid = threadIdx.x, f = 4 * tid;
  float ss = c[0] * c[0] + c[1] * c[1] + c[2] * c[2] + c[3] * c[3];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((tid & 31) == 0) red[tid >> 5] = ss;
  __syncthreads();
  const float tot = (red[0] + red[1]) + (red[2] + red[3]);
  __syncthreads();   // red is reused by the next entry of this CTA
  const float inv = rsqrtf(tot / kDim + p.eps);
  const float4 w = __ldg(reinterpret_cast<const float4*>(p.norm_w) + tid);
  c[0] *= inv * w.x;
  c[1] *= inv * w.y;
  c[2] *= inv * w.z;
  c[3] *= inv * w.w;
  if (f >= kRopeFirst) {
    if (pos >= 0 && pos < p.rope_rows) {
      const float4 cs = __ldg(p.rope_cs + static_cast<int64_t>(pos) * 16 + ((f - kRopeFirst) >> 2));
      // (x + i y)(cos + i sin), pairs (f, f + 1) and (f + 2, f + 3)
      const float x0 = c[0], y0 = c[1], x1 = c[2], y1 = c[3];
      c[0] = fmaf(x0, cs.x, -(y0 * cs.y));
      c[1] = fmaf(y0, cs.x, x0 * cs.y);
      c[2] = fmaf(x1, cs.z, -(y1 * cs.w));
      c[3] = fmaf(y1, cs.z, x1 * cs.w);
    } else if (f == kRopeFirst) {
      raise_error(kErrIndex);
    }
  }
  uint2 o;
  o.x = to_bf16x2(c[0], c[1]);
  o.y = to_bf16x2(c[2], c[3]);
  *reinterpret_cast<uint2*>(dst + f) = o;
}

__global__ void __launch_bounds__(kThreads) compress_windows_kernel(const CompressParams p) {
  __shared__ float red[kThreads / 32];
  griddep_launch();
  griddep_wait();
  const int tid = threadIdx.x, f = 4 * tid;
  const int r = p.ratio;
  const int coff = p.overlap ? 2 : 1;
  for (int e = blockIdx.x; e < p.n; e += gridDim.x) {
    const int cur = __ldg(p.first_tok + e);
    const int prev = p.overlap ? __ldg(p.prev_tok + e) : -1;
    const int pos = __ldg(p.position + e);
    if (cur < 0 || cur + r > p.n_tok || (prev >= 0 && prev + r > p.n_tok)) {   // CTA-uniform
      if (tid == 0) raise_error(kErrIndex);
      *reinterpret_cast<uint2*>(p.out + static_cast<int64_t>(e) * kDim + f) = make_uint2(0u, 0u);
      continue;
    }
    float m[4], l[4], a[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      m[i] = -INFINITY;
      l[i] = 0.f;
      a[i] = 0.f;
    }
    // slot k < nprev: token prev + k, features [0, 512) (the previous window's
    // overlapping half); else token cur + k - nprev, the last 512 features.
    // Loads of kBatch slots are issued before any of them is folded.
    const int nprev = prev >= 0 ? r : 0;
    const int nslots = nprev + r;
    const int half = (coff - 1) * kDim;
    for (int k0 = 0; k0 < nslots; k0 += kBatch) {
      float kv[kBatch][4], sc[kBatch][4];
      float4 ap[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int k = min(k0 + u, nslots - 1);   // clamped: unconditional loads
        const bool own = k >= nprev;
        const int64_t row = own ? cur + (k - nprev) : prev + k;
        const int j = own ? k - nprev : k;
        const int off = own ? half : 0;
        load4(p.kv + row * p.tok_stride + off, f, kv[u]);
        load4(p.score + row * p.tok_stride + off, f, sc[u]);
        ap[u] = __ldg(reinterpret_cast<const float4*>(p.ape + static_cast<int64_t>(j) * coff * kDim + off) + tid);
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        if (k0 + u >= nslots) break;
        fold(sc[u][0] + ap[u].x, kv[u][0], m[0], l[0], a[0]);
        fold(sc[u][1] + ap[u].y, kv[u][1], m[1], l[1], a[1]);
        fold(sc[u][2] + ap[u].z, kv[u][2], m[2], l[2], a[2]);
        fold(sc[u][3] + ap[u].w, kv[u][3], m[3], l[3], a[3]);
      }
    }
    float c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = l[i] > 0.f ? a[i] / l[i] : 0.f;
    finish_entry(p, c, pos, p.out + static_cast<int64_t>(e) * kDim, red);
  }
}

__global__ void __launch_bounds__(kThreads) compress_online_kernel(const CompressParams p) {
  __shared__ float red[kThreads / 32];
  griddep_launch();
  griddep_wait();
  const int tid = threadIdx.x, f = 4 * tid;
  for (int t = blockIdx.x; t < p.n; t += gridDim.x) {
    const int s = __ldg(p.state_idx + t);
    if (s < 0 || s >= p.slots) {   // CTA-uniform
      if (tid == 0) {
        raise_error(kErrIndex);
        p.done[t] = 0;
      }
      continue;
    }
    const int cnt = p.state_count[s];
    __syncthreads();                // every thread has read the count before it changes
    if (cnt < 0 || cnt >= 128) {    // a corrupt state: flagged, left alone
      if (tid == 0) {
        raise_error(kErrIndex);
        p.done[t] = 0;
      }
      continue;
    }
    float* st = p.state + static_cast<int64_t>(s) * 3 * kDim;
    float4 m = *reinterpret_cast<float4*>(st + f);
    float4 l = *reinterpret_cast<float4*>(st + kDim + f);
    float4 a = *reinterpret_cast<float4*>(st + 2 * kDim + f);
    float kv[4], sc[4];
    load4(p.kv + static_cast<int64_t>(t) * p.tok_stride, f, kv);
    load4(p.score + static_cast<int64_t>(t) * p.tok_stride, f, sc);
    const float4 ap = __ldg(reinterpret_cast<const float4*>(p.ape + static_cast<int64_t>(cnt) * kDim) + tid);
    fold(sc[0] + ap.x, kv[0], m.x, l.x, a.x);
    fold(sc[1] + ap.y, kv[1], m.y, l.y, a.y);
    fold(sc[2] + ap.z, kv[2], m.z, l.z, a.z);
    fold(sc[3] + ap.w, kv[3], m.w, l.w, a.w);
    if (cnt + 1 < 128) {
      *reinterpret_cast<float4*>(st + f) = m;
      *reinterpret_cast<float4*>(st + kDim + f) = l;
      *reinterpret_cast<float4*>(st + 2 * kDim + f) = a;
      if (tid == 0) {
        p.state_count[s] = cnt + 1;
        p.done[t] = 0;
      }
    } else {
      float c[4] = {l.x > 0.f ? a.x / l.x : 0.f, l.y > 0.f ? a.y / l.y : 0.f, l.z > 0.f ? a.z / l.z : 0.f,
                    l.w > 0.f ? a.w / l.w : 0.f};
      finish_entry(p, c, __ldg(p.position + t), p.out + static_cast<int64_t>(t) * kDim, red);
      *reinterpret_cast<float4*>(st + f) = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      *reinterpret_cast<float4*>(st + kDim + f) = make_float4(0.f, 0.f, 0.f, 0.f);
      *reinterpret_cast<float4*>(st + 2 * kDim + f) = make_float4(0.f, 0.f, 0.f, 0.f);
      if (tid == 0) {
        p.state_count[s] = 0;
        p.done[t] = 1;
      }
    }
  }
}

int grid_for(int n) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  const int full = sms * 16;   // 16 CTAs of 128 threads per SM
  return n < full ? n : full;
}

}  // namespace

int launch_compress_windows(const void* kv, const void* score, int64_t tok_stride, int64_t n_tok,
                            const int32_t* first_tok,
                            const int32_t* prev_tok, const int32_t* position, int32_t n, int32_t ratio,
                            int32_t overlap, const float* ape, const float* norm_w, float eps, const float* rope_cs,
                            int32_t rope_rows, void* out, cudaStream_t stream) {
  CompressParams p{};
  p.kv = static_cast<const uint16_t*>(kv);
  p.score = static_cast<const uint16_t*>(score);
  p.first_tok = first_tok;
  p.prev_tok = prev_tok;
  p.position = position;
  p.ape = ape;
  p.norm_w = norm_w;
  p.rope_cs = reinterpret_cast<const float4*>(rope_cs);
  p.out = static_cast<uint16_t*>(out);
  p.tok_stride = tok_stride;
  p.n_tok = n_tok;
  p.n = n;
  p.ratio = ratio;
  p.overlap = overlap;
  p.rope_rows = rope_rows;
  p.eps = eps;
  if (n == 0) return DSV4SA_OK;
  const int grid = grid_for(n);
  if (grid < 1) return DSV4SA_ERR_CUDA;
  return launch_pdl(compress_windows_kernel, dim3(grid), dim3(kThreads), 0, stream, p) == cudaSuccess
             ? DSV4SA_OK
             : DSV4SA_ERR_CUDA;
}

int launch_compress_online(const void* kv, const void* score, int64_t tok_stride, const int32_t* state_idx,
                           float* state, int32_t* state_count, int32_t slots, const int32_t* position, int32_t T,
                           const float* ape, const float* norm_w, float eps, const float* rope_cs, int32_t rope_rows,
                           void* out, int32_t* done, cudaStream_t stream) {
  CompressParams p{};
  p.kv = static_cast<const uint16_t*>(kv);
  p.score = static_cast<const uint16_t*>(score);
  p.position = position;
  p.ape = ape;
  p.norm_w = norm_w;
  p.rope_cs = reinterpret_cast<const float4*>(rope_cs);
  p.out = static_cast<uint16_t*>(out);
  p.tok_stride = tok_stride;
  p.n = T;
  p.ratio = 128;
  p.rope_rows = rope_rows;
  p.eps = eps;
  p.state_idx = state_idx;
  p.state = state;
  p.state_count = state_count;
  p.done = done;
  p.slots = slots;
  if (T == 0) return DSV4SA_OK;
  const int grid = grid_for(T);
  if (grid < 1) return DSV4SA_ERR_CUDA;
  return launch_pdl(compress_online_kernel, dim3(grid), dim3(kThreads), 0, stream, p) == cudaSuccess
             ? DSV4SA_OK
             : DSV4SA_ERR_CUDA;
}

namespace {
// Failure-path self-test: one thread waits, bounded, on an mbarrier nothing
// arrives on.  The wait gives up after the library's wait limit, raises the
// timeout bit and returns; result[0] = 1 if the wait had completed, else 0.
__global__ void wait_timeout_kernel(int32_t* result) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) result[0] = mbar_wait(&bar, 0) ? 1 : 0;
}
}  // namespace

int launch_selftest_wait_timeout(int32_t* result, cudaStream_t stream) {
  wait_timeout_kernel<<<1, 32, 0, stream>>>(result);
  return cudaGetLastError() == cudaSuccess ? DSV4SA_OK : DSV4SA_ERR_CUDA;
}

uint32_t read_error_word_compress(cudaStream_t stream, bool clear) {
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
