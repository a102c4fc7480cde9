/*
 * dsv4sa.h -- C ABI of the GB300 (sm_103a) library for DeepSeek-V4-style
 * compressed sparse attention: C4 indexer logits -> per-query top-k ->
 * sparse attention with an attention sink over a paged FP8/BF16 KV cache.
 *
 * Sources, cited by page title and section:
 *   [V4]   "DeepSeek-V4 全面解读：架构设计与 inference/encoding 源码深度解析"
 *          (wangjunjian.com): §2.5 RMSNorm, §2.6 RoPE, §2.8 KV Cache 索引辅助函数,
 *          §2.9 Compressor, §2.10 Indexer, §2.11 Attention, §3.2 数据类型别名,
 *          §3.4 act_quant_kernel, §3.7 sparse_attn_kernel.
 *   [SGL]  "DeepSeek-V4 in SGLang 深度理解分析": 概念2 分层压缩 (C4/C128),
 *          概念3 C4 Indexer, 概念5 DeepSeekV4TokenToKVPool, 算法2 Paged MQA
 *          Logits + TopK, 算法3 online C128, MQALayer.forward (k=kv, v=kv,
 *          attn_sink, inverse RoPE of the output).
 *   [NVFP4] "tilelang量化内核拆解DeepSeek-V4.1-Flash-NVFP4的fp4_gemm与sparse_attn实现":
 *          section "sparse_attn 实现拆解" (running max starts at -1e30; heads
 *          padded to 16).
 *
 * Conventions shared by every entry point
 *   - Every pointer argument named as a device buffer is a CUDA device pointer
 *     owned by the caller.  The library never allocates, frees or synchronises
 *     inside the compute entry points; scratch memory comes from a caller
 *     workspace whose size the matching *_workspace_size function returns.
 *   - Calls enqueue kernels on the given stream and return immediately with a
 *     dsv4sa_status.  Host-side validation failures return
 *     DSV4SA_ERR_INVALID_ARG / DSV4SA_ERR_UNSUPPORTED before anything is
 *     enqueued; a failed launch returns DSV4SA_ERR_CUDA.
 *   - Kernels never trap.  Conditions they detect on the device (an index or a
 *     page id out of range, a wait that ran out of time) set bits of a
 *     device error word; dsv4sa_check_errors() reads and clears it.
 *   - Results are deterministic: identical inputs give identical bits.
 *   - Everything here targets one GPU; the library holds no global state other
 *     than the device error words.
 */
#ifndef DSV4SA_H_
#define DSV4SA_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define DSV4SA_API __attribute__((visibility("default")))
#else
#define DSV4SA_API
#endif

/* Fixed geometry of the cache format ([SGL] 概念5 NopeFp8RopeBf16Pack; [V4] §2.2
 * ModelArgs head_dim 512, rope_head_dim 64, window_size 128). */
#define DSV4SA_PAGE_SIZE   64   /* slots (compressed entries or raw tokens) per page */
#define DSV4SA_HEAD_DIM    512  /* = nope 448 (FP8 E4M3) + rope 64 (BF16)          */
#define DSV4SA_NOPE_DIM    448
#define DSV4SA_ROPE_DIM    64
#define DSV4SA_SCALE_GROUP 64   /* one fp32 scale per 64 FP8 elements               */
#define DSV4SA_IDX_DIM     128  /* indexer head dim                                 */
#define DSV4SA_MAX_HEADS   128  /* query heads per call                             */
#define DSV4SA_MAX_IDX_HEADS 128
#define DSV4SA_MAX_IDX_HEADS_FP4 64
#define DSV4SA_MAX_TOPK    2048

typedef enum {
  DSV4SA_OK = 0,
  DSV4SA_ERR_INVALID_ARG = 1,    /* null pointer, bad size, stride or alignment   */
  DSV4SA_ERR_UNSUPPORTED = 2,    /* a size outside what the kernels implement     */
  DSV4SA_ERR_WORKSPACE = 3,      /* workspace missing or smaller than required    */
  DSV4SA_ERR_CUDA = 4,           /* a CUDA runtime call or launch failed          */
  DSV4SA_ERR_INDEX_OOB = 5,      /* device: an index or page id was out of range  */
  DSV4SA_ERR_DEVICE_TIMEOUT = 6  /* device: a bounded wait ran out of time        */
} dsv4sa_status;

typedef enum {
  DSV4SA_POOL_KV = 0,       /* attention KV rows: 448 e4m3 + 7 fp32 scales + 64 bf16   */
  DSV4SA_POOL_IDXK = 1,     /* indexer keys: 128 e4m3 + 2 fp32 scales                  */
  DSV4SA_POOL_IDXK_FP4 = 2  /* indexer keys, FP4 variant: 128 e2m1 + 4 e8m0 scales     */
} dsv4sa_pool_kind;

/*
 * Paged-pool layout descriptor ([SGL] 概念5 DeepSeekV4TokenToKVPool: a paged pool
 * holding the single-head KV, nope part FP8 with a per-block scale, rope part
 * BF16).  A pool is `num_pages` pages of `page_stride` bytes at `base`; each
 * page is three structure-of-arrays blocks, every row 16-byte aligned:
 *
 *   KV page   (38912 B): nope  [64][448] e4m3   at  0
 *                        rope  [64][64]  bf16   at  28672   (128 B per slot)
 *                        scale [64][8]   fp32   at  36864   (7 used, 32 B per slot)
 *   IDXK page ( 8704 B): key   [64][128] e4m3   at  0
 *                        scale [64][2]   fp32   at  8192
 *   IDXK_FP4 page (4352 B): key [64][64] bytes  at  0      (128 e2m1 codes, two per
 *                        byte, value 2j in the low nibble of byte j)
 *                        scale [64][4]   e8m0   at  4096   (one per 32 values)
 *
 * ([V4] §3.5 fp4_quant_kernel: FP4 E2M1 in blocks of 32 with a power-of-two
 * scale; [NVFP4] 32-group E8M0 scales for the indexer's q and k.)  Value of
 * element d of an IDXK_FP4 slot = e2m1(code[d]) * 2^(e8m0[d / 32] - 127).
 * The indexer (dsv4sa_indexer_logits) reads IDXK pools; IDXK_FP4 pools are
 * written by dsv4sa_cache_write and dsv4sa_cache_write_rotated and read by
 * dsv4sa_indexer_logits_fp4.
 *
 * Entry s of a sequence lives at slot s % 64 of page page_table[seq][s / 64].
 * Value of nope element d of a slot = e4m3(code[d]) * scale[d / 64].
 * `base` is a device pointer owned by the caller, 1024-byte aligned.
 */
typedef struct {
  int32_t kind;          /* dsv4sa_pool_kind                                       */
  int32_t page_size;     /* 64                                                     */
  int32_t nope_dim;      /* FP8 elements per slot: 448 (KV) | 128 (IDXK)           */
  int32_t rope_dim;      /* BF16 elements per slot: 64 (KV) | 0 (IDXK)             */
  int32_t scale_group;   /* 64 (32 for IDXK_FP4)                                   */
  int32_t n_scales;      /* scales used per slot: 7 (KV) | 2 (IDXK) | 4 (IDXK_FP4) */
  int64_t num_pages;
  int64_t page_stride;   /* bytes between pages                                    */
  int64_t nope_off;      /* byte offset of the FP8 block inside a page             */
  int64_t rope_off;      /* byte offset of the BF16 block (KV only)                */
  int64_t scale_off;     /* byte offset of the fp32 scale block                    */
  int32_t nope_row;      /* bytes per slot in the code block  (448 | 128 | 64)     */
  int32_t rope_row;      /* bytes per slot in the BF16 block  (128 | 0)            */
  int32_t scale_row;     /* bytes per slot in the scale block (32 | 8 | 4)         */
  int32_t reserved;
  void*   base;          /* device pointer, caller-owned                           */
} dsv4sa_pool_desc;

/* Bytes needed for a pool of `num_pages` pages of the given kind (0 on a bad kind). */
DSV4SA_API size_t dsv4sa_pool_bytes(int32_t kind, int64_t num_pages);

/* Fill `d` with the default layout above for `base` (host-only; no device access).
 * Returns DSV4SA_ERR_INVALID_ARG for a null `d`, a bad kind, num_pages < 1 or a
 * base that is not 1024-byte aligned. */
DSV4SA_API int dsv4sa_pool_desc_init(dsv4sa_pool_desc* d, int32_t kind, void* base,
                                     int64_t num_pages);

/*
 * Stage 1 -- C4 indexer logits ([V4] §2.10 steps 6-8; [SGL] 算法2 paged MQA logits).
 *
 *   logits[t, s] = sum_h w[t, h] * ReLU( sum_d qhat[t, h, d] * khat[s, d] ),   s < n_vis[t]
 *
 * where qhat = e4m3(q_fp8) * q_scale[.., d / 64] and khat is the key pool entry s
 * of sequence q_seq[t] dequantised the same way.  The FP8 x FP8 products run on
 * the tensor cores with fp32 accumulation, one accumulator per 64-dim scale
 * block; scales, ReLU and the weighted head sum are applied in fp32.
 *
 *   kpool        IDXK pool descriptor (host struct; its base is a device pointer)
 *   page_table   device int32 [rows][pt_stride]: page ids of each sequence
 *   q_seq        device int32 [T]: row of page_table used by query t
 *   n_vis        device int32 [T]: visible entries of query t; clamped to [0, n_max]
 *   q_fp8        device uint8 [T][Hi][128] e4m3 codes, 16-byte aligned
 *   q_scale      device fp32  [T][Hi][2]
 *   w            device fp32  [T][Hi]   final per-head weights
 *   T, Hi        queries and indexer heads (1 <= Hi <= 128; padded to 16 inside)
 *   n_max        upper bound of n_vis; requires n_max <= pt_stride * 64 and
 *                n_max <= logits_stride
 *   logits       device fp32 [T][logits_stride]; entries s >= n_vis[t] are not written
 * Page ids must lie in [0, num_pages); an id outside sets DSV4SA_ERR_INDEX_OOB on
 * the device and the affected logits are unspecified.
 * The launch uses one persistent CTA per SM but one, so that the first CTA of
 * the next kernel on the stream (a programmatic dependent) can start at once;
 * the key pages are read with an L2 evict-first policy.
 */
DSV4SA_API int dsv4sa_indexer_logits(const dsv4sa_pool_desc* kpool, const int32_t* page_table,
                                     int32_t pt_stride, const int32_t* q_seq,
                                     const int32_t* n_vis, const uint8_t* q_fp8,
                                     const float* q_scale, const float* w, int32_t T,
                                     int32_t Hi, int32_t n_max, float* logits,
                                     int64_t logits_stride, cudaStream_t stream);

/*
 * Stage 1, FP4 variant -- the same logits with FP4 keys and an FP4 query
 * ([V4] §2.10 Indexer step 3, FP4 quant-sim of q and k, and §3.5
 * fp4_quant_kernel; [NVFP4] §model.py 如何驱动: E2M1 values, one E8M0 scale
 * per 32):
 *
 *   logits[t, s] = sum_h w[t, h] * ReLU( sum_d qhat[t, h, d] * khat[s, d] ),   s < n_vis[t]
 *
 * with qhat[t, h, d] = e2m1(code) * 2^(q_e8m0[t, h, d / 32] - 127) and khat the
 * IDXK_FP4 pool entry s of sequence q_seq[t] dequantised the same way.  The
 * E2M1 x E2M1 products of each 32-value block are summed exactly on the
 * tensor cores (fp32 accumulation, one accumulator per block); the two
 * power-of-two scales, ReLU and the weighted head sum are applied in fp32.
 *
 *   kpool        IDXK_FP4 pool descriptor (host struct; base is a device pointer)
 *   page_table, pt_stride, q_seq, n_vis, w, T, n_max, logits, logits_stride:
 *                as dsv4sa_indexer_logits
 *   q_fp4        device uint8 [T][Hi][64]: 128 E2M1 codes per head, two per
 *                byte, value 2j in the low nibble of byte j; 16-byte aligned
 *   q_e8m0       device uint8 [T][Hi][4]: one E8M0 byte per 32 values; 4-byte aligned
 *   Hi           1 <= Hi <= DSV4SA_MAX_IDX_HEADS_FP4 (padded to 16 inside)
 * Errors: as dsv4sa_indexer_logits; a pool of another kind is INVALID_ARG,
 * Hi > 64 is UNSUPPORTED.
 */
DSV4SA_API int dsv4sa_indexer_logits_fp4(const dsv4sa_pool_desc* kpool, const int32_t* page_table,
                                         int32_t pt_stride, const int32_t* q_seq, const int32_t* n_vis,
                                         const uint8_t* q_fp4, const uint8_t* q_e8m0, const float* w, int32_t T,
                                         int32_t Hi, int32_t n_max, float* logits, int64_t logits_stride,
                                         cudaStream_t stream);

/*
 * Stage 2 -- per-query top-k ([V4] §2.10 step 9; [SGL] 概念3 top-512, 算法2).
 *
 * idx[t, :] = the k entries s < n_vis[t] with the largest logits[t, s], in
 * ascending entry order, padded with -1.  Among equal scores the lower entry
 * index is taken.  When n_vis[t] <= k every visible entry is taken ([SGL] 算法2:
 * below 512 compressed entries no top-k is needed).  -0.0 equals +0.0; NaN
 * ranks below every number.  Exact: integer compares of order-preserving keys.
 *
 *   logits   device fp32 [T][logits_stride]
 *   n_vis    device int32 [T], clamped to n_max; a row with n_vis[t] < 0 is
 *            left untouched (a row that takes another index list, e.g. C128)
 *   k        1..2048; n_max <= min(64, 32768 / k) * 16384 when n_max > 16384
 *   idx      device int32 [T][idx_stride], idx_stride >= k
 *   ws       device workspace of at least dsv4sa_topk_workspace_size(T, n_max, k) bytes
 *            (may be null when that size is 0)
 */
DSV4SA_API size_t dsv4sa_topk_workspace_size(int32_t T, int32_t n_max, int32_t k);
DSV4SA_API int dsv4sa_topk(const float* logits, int64_t logits_stride, const int32_t* n_vis,
                           int32_t T, int32_t n_max, int32_t k, int32_t* idx,
                           int32_t idx_stride, void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * dsv4sa_topk plus an L2 prefetch of what the attention will gather next: the
 * same selection, bit for bit, and as each selected entry's index is written
 * its row of kv_pool (the compressed KV pool the decode attention reads, in the
 * default layout) is prefetched into L2, so the attention's gather of those
 * rows finds them there or in flight.  No value changes; only timing.
 *
 *   kv_pool        the compressed KV pool (DSV4SA_POOL_KV descriptor)
 *   kv_page_table  device int32 [.][kv_pt_stride]; query t reads row q_seq[t]
 *   q_seq          device int32 [T]
 * Entries outside the page table or on a page id out of range are not
 * prefetched (the attention flags them).  Other arguments and errors as
 * dsv4sa_topk; a bad descriptor returns DSV4SA_ERR_INVALID_ARG.
 * The launch carries one extra CTA that runs the selection once on a
 * synthetic row, without waiting for the previous kernel of the stream and
 * without writing anything (it reads up to the first 64 KB of kv_pool, and
 * prefetches range-checked lines of it): scheduled first, on an SM the
 * preceding indexer leaves free, it brings the selection's instructions into
 * L2 before the row CTAs run.
 */
DSV4SA_API int dsv4sa_topk_prefetch(const float* logits, int64_t logits_stride, const int32_t* n_vis,
                                    int32_t T, int32_t n_max, int32_t k, int32_t* idx, int32_t idx_stride,
                                    void* ws, size_t ws_bytes, const dsv4sa_pool_desc* kv_pool,
                                    const int32_t* kv_page_table, int32_t kv_pt_stride, const int32_t* q_seq,
                                    cudaStream_t stream);

/*
 * Scratch-free top-k.  The pages have no counterpart: this entry point exists
 * for callers that cannot allocate device memory when they call the library --
 * a serving engine that reserves all device memory in its own pool at start-up
 * and forbids allocations afterwards, a runtime that must never take the
 * implicit synchronisation of cudaMalloc/cudaFree on its hot path, or an
 * embedded caller without access to an allocator.  It computes exactly what
 * dsv4sa_topk computes, bit for bit, and takes no workspace argument: the
 * candidate scratch of long rows lives in a file-scope device array of
 * DSV4SA_TOPK_NOALLOC_SCRATCH_BYTES (8 MiB) that every GPU which loads the
 * library holds until the process exits.  The function allocates nothing
 * (no cudaMalloc, cudaFree or allocating library routine).
 *
 *   - Size limit: T * chunks * k * 8 bytes must fit the scratch, where chunks =
 *     ceil(n_max / 16384) when n_max > 16384 (rows of up to 16384 entries,
 *     64K tokens of C4 context, need no scratch).  Larger requests return
 *     DSV4SA_ERR_UNSUPPORTED before anything is enqueued; e.g. k = 512 allows
 *     T * chunks <= 2048 (128 queries at 1M tokens of context).
 *   - Set-up: the first call on a device looks up the scratch's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make that
 *     first call before any stream capture.
 *   - Sharing: every call uses the same scratch, which keeps the last call's
 *     contents (nothing in it needs to start at zero).  Calls that overlap on
 *     the GPU -- on different streams, or from different threads -- race on it;
 *     the caller must order them.
 * Other arguments and errors as dsv4sa_topk.
 */
#define DSV4SA_TOPK_NOALLOC_SCRATCH_BYTES (8u << 20)
DSV4SA_API int dsv4sa_topk_noalloc(const float* logits, int64_t logits_stride, const int32_t* n_vis,
                                   int32_t T, int32_t n_max, int32_t k, int32_t* idx,
                                   int32_t idx_stride, cudaStream_t stream);

/*
 * Index assembly ([V4] §2.8 get_window_topk_idxs / get_compress_topk_idxs).
 *
 * dsv4sa_window_indices: idx_w[t, j] for j < window is the raw position
 *   p = pos[t] - window + 1 + j (the current token included), -1 when p < 0;
 *   with ring > 0 the stored value is p % ring (slot of a circular window cache,
 *   as in decode), else p itself.
 * dsv4sa_compress_indices: idx[t, j] = j for j < min(n_vis[t], kc), else -1
 *   (all visible compressed entries, used when a layer has no indexer, e.g. C128).
 */
DSV4SA_API int dsv4sa_window_indices(const int32_t* pos, int32_t T, int32_t window,
                                     int32_t ring, int32_t* idx_w, int32_t idx_stride,
                                     cudaStream_t stream);
DSV4SA_API int dsv4sa_compress_indices(const int32_t* n_vis, int32_t T, int32_t kc,
                                       int32_t* idx, int32_t idx_stride, cudaStream_t stream);

/*
 * Stage 3 -- sparse attention with attention sink ([V4] §3.7 sparse_attn_kernel,
 * §2.11 step 7; [NVFP4] sparse_attn 实现拆解; [SGL] MQALayer k=kv, v=kv).
 *
 * For query t and head h, over the multiset J of valid indices in
 * idx_c[t, :kc] (entries of the compressed pool) ++ idx_w[t, :kw] (entries of
 * the window pool), index -1 being an invalid slot:
 *
 *   a_j  = softmax_scale * q[t, h, :] . kv_j          (kv_j: dequantised row, 512 dims)
 *   o    = sum_j e^{a_j} kv_j / ( sum_j e^{a_j} + e^{attn_sink[h]} )
 *
 * evaluated as an online softmax whose running max starts at -1e30, so a row
 * with no valid index yields exactly 0.  The single kv row serves as K and V.
 * QK^T and PV run on the tensor cores in BF16 with fp32 accumulation (the FP8
 * nope part is dequantised to BF16 on the gather); P is rounded to BF16 for
 * PV; the output is rounded to BF16 (round to nearest even).
 */
typedef struct {
  const void*  q;              /* device bf16 [T][H][512], 16-byte aligned                 */
  int32_t      T;              /* query tokens                                             */
  int32_t      H;              /* query heads, 1..128 (padded to a multiple of 16 inside)  */
  float        softmax_scale;  /* e.g. 1/sqrt(512)                                         */
  int32_t      flags;          /* DSV4SA_ATTN_* flags below, 0 by default                   */
  const float* attn_sink;      /* device fp32 [H]                                          */
  const int32_t* q_seq;        /* device int32 [T]: page-table row of query t              */
  const dsv4sa_pool_desc* comp;/* KV pool of compressed entries (may be null when kc == 0) */
  const int32_t* comp_pt;      /* device int32 [rows][comp_pt_stride]                      */
  int32_t      comp_pt_stride;
  int32_t      kc;             /* compressed indices per query, 0..2048                    */
  const int32_t* idx_c;        /* device int32 [T][idx_c_stride]; entries < comp_pt_stride*64 */
  int32_t      idx_c_stride;
  int32_t      kw;             /* window indices per query, 0..1024                        */
  const dsv4sa_pool_desc* win; /* KV pool of raw window tokens (may be null when kw == 0)  */
  const int32_t* win_pt;       /* device int32 [rows][win_pt_stride]                       */
  int32_t      win_pt_stride;
  int32_t      idx_w_stride;
  const int32_t* idx_w;        /* device int32 [T][idx_w_stride]; entries < win_pt_stride*64 */
  void*        out;            /* bf16 [T][H][512]; device memory, or host memory the device
                                  can address (e.g. pinned): the kernel writes it directly */
  float*       lse;            /* optional fp32 [T][H]: ln(sum e^a + e^sink), as `out`     */
  void*        ws;             /* device workspace (decode only; see workspace_size)       */
  size_t       ws_bytes;
  /* Window indices computed in the kernel instead of read from idx_w: when
   * idx_w is null and win_pos is not, window index j of query t is
   * p = win_pos[t] - kw + 1 + j, or -1 when p < 0, taken mod win_ring when
   * win_ring > 0 -- exactly what dsv4sa_window_indices writes (the pages'
   * get_window_topk_idxs), without the extra launch and round trip. */
  const int32_t* win_pos;      /* device int32 [T] (optional)                               */
  int32_t      win_ring;
  int32_t      reserved1;
  /* Inverse rotary embedding of the output ([V4] §2.11 step 8 with §2.6
   * apply_rotary_emb inverse=True; [SGL] MQALayer step 7), fused into the
   * output write: when rope_cs is not null, the last 64 dims of o[t, h] are
   * taken as 32 complex pairs (o[448 + 2i], o[449 + 2i]) and multiplied by the
   * conjugate of rope_cs[rope_pos[t]][i] = (cos, sin) before the output is
   * rounded to BF16 (one rounding, of the rotated fp32 value).  The table is the
   * caller's precomputed freqs_cis (any frequencies, YaRN or not).  A position
   * outside [0, rope_rows) sets DSV4SA_ERR_INDEX_OOB on the device and that
   * query's output is written unrotated.  Null rope_cs: no rotation. */
  const float*   rope_cs;      /* device fp32 [rope_rows][32][2], 16-byte aligned (optional) */
  const int32_t* rope_pos;     /* device int32 [T]: table row of query t                   */
  int32_t        rope_rows;
  int32_t        reserved2;
} dsv4sa_attn_args;

/* flags: the caller guarantees that, of this call's inputs, only idx_c may be
 * written by the kernels that precede it on the stream (q, attn_sink, q_seq,
 * the window positions or idx_w, the pools and page tables are not).  The
 * kernel then processes the window rows while the preceding kernel (e.g. the
 * top-k that produces idx_c) still runs, and waits for it before the
 * compressed rows.  Results are identical with and without the flag. */
#define DSV4SA_ATTN_EARLY_WINDOW 1

/* Modes of the attention entry points. */
#define DSV4SA_ATTN_DECODE  0   /* few queries: the gathered rows of each query are split
                                   over several CTAs and merged by log-sum-exp          */
#define DSV4SA_ATTN_PREFILL 1   /* many queries: one CTA runs the whole online softmax   */

/* Workspace bytes the given mode needs for these arguments (0 for prefill).
 * An upper bound over devices: a decode call may use less of it. */
DSV4SA_API size_t dsv4sa_attn_workspace_size(int32_t mode, int32_t T, int32_t H, int32_t kc,
                                             int32_t kw);

/* How a call with these arguments splits its work on the current device
 * (host only; reads the device's SM count).  Outputs, each optional:
 *   nsplit          CTAs per (query, 64-head group) over which the rows are split
 *   rows_per_split  gathered rows per CTA
 *   launches        kernel launches the call enqueues (1, or 2 when the
 *                   splits are merged by a second kernel)
 * Returns DSV4SA_OK, DSV4SA_ERR_INVALID_ARG or DSV4SA_ERR_CUDA. */
DSV4SA_API int dsv4sa_attn_plan(int32_t mode, int32_t T, int32_t H, int32_t kc, int32_t kw, int32_t* nsplit,
                                int32_t* rows_per_split, int32_t* launches);

/* Entries of an index list that are >= 64 * (page-table stride), or page ids
 * outside [0, num_pages), are treated as invalid and set DSV4SA_ERR_INDEX_OOB on
 * the device.  Both entry points compute the same function; they differ only in
 * how the work is split across CTAs. */
DSV4SA_API int dsv4sa_sparse_attn_decode(const dsv4sa_attn_args* args, cudaStream_t stream);
DSV4SA_API int dsv4sa_sparse_attn_prefill(const dsv4sa_attn_args* args, cudaStream_t stream);

/*
 * Top-k and decode attention in one call: exactly what dsv4sa_topk (writing
 * its selection into attn->idx_c) followed by dsv4sa_sparse_attn_decode
 * computes, bit for bit ([V4] §2.10 step 9 then §3.7; [SGL] 算法2).
 * attn->idx_c is in/out: a row with n_vis[t] >= 0 is written with the query's
 * k = attn->kc largest-scoring entries (ascending, -1 padded, all of them when
 * n_vis[t] <= k); a row with n_vis[t] < 0 keeps the list it holds (a C128 row,
 * say) and is attended over as given.
 * When the decode attention runs as thread-block clusters and rows have at
 * most 16384 entries, one kernel does both: the CTAs of a query's cluster
 * select its list from the logits together and gather their rows at once, so
 * no SM idles between a selection and the attention that waits for it.
 * Otherwise the two run as separate kernels (the top-k then prefetches the
 * selected rows into L2).
 *   logits, logits_stride, n_vis, n_max   as dsv4sa_topk (logits 16-byte
 *            aligned with logits_stride % 4 == 0 for the one-kernel form)
 *   k        must equal attn->kc
 *   topk_ws  dsv4sa_topk's workspace, needed only when rows are longer than
 *            16384 entries (dsv4sa_topk_workspace_size), else may be null
 * attn->flags & DSV4SA_ATTN_EARLY_WINDOW: only the logits (and idx_c rows with
 * n_vis < 0) may come from the previous kernel of the stream.
 * Errors: as the two calls it stands for; k != attn->kc is DSV4SA_ERR_INVALID_ARG.
 */
DSV4SA_API int dsv4sa_topk_sparse_attn_decode(const dsv4sa_attn_args* attn, const float* logits,
                                              int64_t logits_stride, const int32_t* n_vis, int32_t n_max,
                                              int32_t k, void* topk_ws, size_t topk_ws_bytes, cudaStream_t stream);

/*
 * KV-cache writer: quantise n new BF16 rows into a paged pool ("DeepSeek-V4
 * 全面解读" §3.4 act_quant_kernel; "DeepSeek-V4 in SGLang" 概念5
 * DeepSeekV4TokenToKVPool).  Row r is entry row_entry[r] of the sequence whose
 * page-table row is row_seq[r]; it goes to slot entry % 64 of page
 * page_table[row_seq[r]][entry / 64].  Every 64-value block that is quantised
 * gets, in fp32: amax = max(max |x|, 1e-4), scale = amax * fp32(1/448),
 * codes = E4M3 round-to-nearest-even of clamp(x / scale, -448, 448).
 *
 *   pool        DSV4SA_POOL_KV: rows are bf16 [n][512]; the 448 nope values
 *               are quantised (7 scales), the 64 rope values stored unchanged.
 *               DSV4SA_POOL_IDXK: rows are bf16 [n][128] (2 scales).
 *               DSV4SA_POOL_IDXK_FP4: rows are bf16 [n][128]; every 32-value
 *               block gets, in fp32 ([V4] §3.5 fp4_quant_kernel, §3.3
 *               fast_round_scale): e = ceil(log2(max(amax, 6 * 2^-126) *
 *               fp32(1/6))), codes = E2M1 round-to-nearest-even of
 *               clamp(x / 2^e, -6, 6), the scale stored as the E8M0 byte e + 127.
 *   page_table  device int32 [rows][pt_stride]
 *   row_seq, row_entry  device int32 [n]
 *   rows        device bf16, 16-byte aligned
 * A row whose entry or page id is out of range is skipped and sets
 * DSV4SA_ERR_INDEX_OOB on the device (dsv4sa_check_errors).  Rows writing the
 * same slot in one call race (the caller gives distinct slots).
 */
DSV4SA_API int dsv4sa_cache_write(const dsv4sa_pool_desc* pool, const int32_t* page_table, int32_t pt_stride,
                                  const int32_t* row_seq, const int32_t* row_entry, const void* rows, int32_t n,
                                  cudaStream_t stream);

/*
 * The compressor's rotate path into an FP4 key pool ("DeepSeek-V4 全面解读"
 * §2.9: indexer keys rotated by a Hadamard transform, then FP4-quantised).
 * Each BF16 row x[128] becomes y = H_128 x * 128^-0.5 (H_128 the Sylvester
 * Hadamard matrix, H[i][j] = (-1)^popcount(i & j)), computed as fp32
 * butterflies (a + b, a - b) of strides 1, 2, 4, ..., 64, a multiply by the
 * fp32 value of 128^-0.5 and one rounding to BF16 (nearest, ties to even);
 * y is then quantised exactly as dsv4sa_cache_write does for
 * DSV4SA_POOL_IDXK_FP4.  Since H_128 * 128^-0.5 is orthogonal, logits of a
 * query rotated the same way equal those of the unrotated pair up to rounding.
 *
 *   pool        a DSV4SA_POOL_IDXK_FP4 pool (any other kind: INVALID_ARG)
 *   other arguments and errors as dsv4sa_cache_write; rows whose rotation
 *   leaves the fp32 range are not supported.
 */
DSV4SA_API int dsv4sa_cache_write_rotated(const dsv4sa_pool_desc* pool, const int32_t* page_table,
                                          int32_t pt_stride, const int32_t* row_seq, const int32_t* row_entry,
                                          const void* rows, int32_t n, cudaStream_t stream);

/*
 * KV compressor ([V4] §2.9 Compressor; [SGL] 概念2 C4 / C128, 算法3 online C128):
 * windows of raw-token projections pooled into compressed entries, BF16
 * [n][512] out (quantise them into a pool with dsv4sa_cache_write).  Inputs are
 * the outputs of the model's wkv / wgate projections, BF16 rows of
 * coff * 512 values (coff = 2 with the overlap transform, else 1), token rows
 * tok_stride elements apart.  For entry e with window tokens first_tok[e] ..
 * first_tok[e] + ratio - 1, per feature f: the slot scores score + ape[j]
 * (j = the token's place in its window) are softmax-normalised over the slots
 * and weight the slot kv; with overlap the slots are the previous window's
 * tokens (prev_tok[e] .., their features [0, 512)) then the window's own
 * (features [512, 1024)); prev_tok[e] = -1: no previous window (first window).
 * The pooled row x is RMS-normalised, x / sqrt(mean(x^2) + eps) * norm_w, its
 * last 64 dims rotated forward by the (cos, sin) row position[e] of rope_cs,
 * and rounded to BF16.  Windows reaching past n_tok token rows, or positions
 * outside [0, rope_rows), set DSV4SA_ERR_INDEX_OOB on the device (the entry is
 * written as zeros, or unrotated).
 *
 *   kv, score   device bf16 [n_tok][tok_stride], 16-byte aligned, tok_stride a
 *               multiple of 8 and >= coff * 512
 *   ape         device fp32 [ratio][coff * 512];  norm_w  device fp32 [512]
 *   rope_cs     device fp32 [rope_rows][32][2];   all 16-byte aligned
 *   ratio       4 with overlap = 1, or any 1..1024 with overlap = 0 (C128: 128)
 */
DSV4SA_API int dsv4sa_compress_windows(const void* kv, const void* score, int64_t tok_stride, int64_t n_tok,
                                       const int32_t* first_tok, const int32_t* prev_tok, const int32_t* position,
                                       int32_t n, int32_t ratio, int32_t overlap, const float* ape,
                                       const float* norm_w, float eps, const float* rope_cs, int32_t rope_rows,
                                       void* out, cudaStream_t stream);

/*
 * Online C128 compression ([SGL] 算法3: O(1) state per sequence): token t of
 * this call (kv, score rows [512], BF16) joins the open window of state slot
 * state_idx[t]; state holds fp32 [slots][3][512] (running max, sum and
 * weighted kv per feature) and state_count [slots] the tokens folded so far.
 * The token's score gets ape[state_count] added.  When the count reaches 128
 * the entry (normalised and rotated by row position[t], as above) is written
 * to out[t], done[t] = 1 and the slot is reset (max -inf, sum and kv 0, count
 * 0); otherwise done[t] = 0.  A fresh slot is max -inf, sum 0, kv 0, count 0.
 * Each slot appears at most once per call.  An out-of-range slot or count sets
 * DSV4SA_ERR_INDEX_OOB and the token is skipped.
 */
DSV4SA_API int dsv4sa_compress_online_c128(const void* kv, const void* score, int64_t tok_stride, int32_t T,
                                           const int32_t* state_idx, float* state, int32_t* state_count,
                                           int32_t slots, const int32_t* position, const float* ape,
                                           const float* norm_w, float eps, const float* rope_cs, int32_t rope_rows,
                                           void* out, int32_t* done, cudaStream_t stream);

/* Copy `bytes` (a multiple of 16) from src to dst with the SMs (a kernel of
 * 16-byte loads and stores on `stream`); either side may be device memory or
 * pinned host memory the device can address.  For the few hundred kilobytes to
 * megabytes of a serving step's inputs it starts sooner than a copy-engine
 * transfer.  Both pointers 16-byte aligned; the ranges must not overlap. */
DSV4SA_API int dsv4sa_copy_async(void* dst, const void* src, size_t bytes, cudaStream_t stream);

/* The same copy, same arguments and errors, by one warp per SM with at most 32
 * registers a thread: it runs beside a kernel that occupies the SMs' shared
 * memory and all but one warp's worth of registers (dsv4sa_indexer_logits), for
 * a copy issued on another stream while that kernel runs. */
DSV4SA_API int dsv4sa_copy_async_background(void* dst, const void* src, size_t bytes, cudaStream_t stream);

/* Failure-path self-test: one thread of one CTA waits on an mbarrier that
 * nothing arrives on, with the library's bounded wait (the same code every
 * kernel's waits use).  After the wait limit (2 s) it gives up, sets
 * DSV4SA_ERR_DEVICE_TIMEOUT on the device and returns, leaving the context
 * usable; result (device int32) receives 0 (1 would mean the wait completed).
 * Read the status with dsv4sa_check_errors. */
DSV4SA_API int dsv4sa_selftest_wait_timeout(int32_t* result, cudaStream_t stream);

/* Synchronise `stream`, then read and clear the device error words of the
 * current device.  Returns DSV4SA_OK, DSV4SA_ERR_INDEX_OOB,
 * DSV4SA_ERR_DEVICE_TIMEOUT or DSV4SA_ERR_CUDA; `bits_out` (optional) receives
 * the raw bits (1 = index/page out of range, 2 = wait timeout). */
DSV4SA_API int dsv4sa_check_errors(cudaStream_t stream, uint32_t* bits_out);

/*
 * One decode serving step as a CUDA graph owned by the library: the step's
 * packed inputs copied from pinned host memory (bytes [0, in_split) by
 * dsv4sa_copy_async before the indexer, the rest by
 * dsv4sa_copy_async_background on a second stream beside the indexer), then
 * dsv4sa_indexer_logits, dsv4sa_topk and dsv4sa_sparse_attn_decode with the
 * arguments below, the attention waiting for the second copy.  The argument
 * pointers are the device buffers the kernels read and write: the input
 * views inside dev_in, the pools, logits, idx, workspaces; attn->out and
 * attn->lse may be pinned host memory, so one launch moves the inputs in and
 * the results out.  The buffers must stay valid while the step exists; the
 * caller refills host_in between launches and synchronises the launch stream
 * before reading the results.
 */
typedef struct {
  const void* host_in;        /* pinned host, in_bytes, 16-byte aligned                   */
  void* dev_in;               /* device, in_bytes, 16-byte aligned                        */
  size_t in_bytes;            /* multiple of 16                                           */
  size_t in_split;            /* multiple of 16, <= in_bytes: the indexer's and top-k's part */
  /* dsv4sa_indexer_logits */
  const dsv4sa_pool_desc* kpool;
  const int32_t* page_table;
  int32_t pt_stride;
  int32_t T;
  const int32_t* q_seq;
  const int32_t* n_vis;
  const uint8_t* q_fp8;
  const float* q_scale;
  const float* w;
  int32_t Hi;
  int32_t n_max;
  float* logits;
  int64_t logits_stride;
  /* dsv4sa_topk */
  int32_t k;
  int32_t idx_stride;
  int32_t* idx;
  void* topk_ws;
  size_t topk_ws_bytes;
  /* dsv4sa_sparse_attn_decode (attn->idx_c is the top-k's idx) */
  const dsv4sa_attn_args* attn;
} dsv4sa_step_desc;

typedef struct dsv4sa_step dsv4sa_step;   /* opaque */

/* Build the step: one eager run on `stream` (so per-device set-up happens
 * outside the capture; it synchronises the stream), then a capture of the same
 * calls into a graph.  Errors of any call are returned as they are; *out is
 * set only on DSV4SA_OK. */
DSV4SA_API int dsv4sa_step_create(dsv4sa_step** out, const dsv4sa_step_desc* desc, cudaStream_t stream);
/* Launch the step's graph on `stream` (asynchronous). */
DSV4SA_API int dsv4sa_step_launch(dsv4sa_step* step, cudaStream_t stream);
/* Free the graph, its second stream and events (after its launches finished). */
DSV4SA_API int dsv4sa_step_destroy(dsv4sa_step* step);

/* Static text for a status code. */
DSV4SA_API const char* dsv4sa_status_string(int status);

/* Library version as 10000*major + 100*minor + patch. */
DSV4SA_API int dsv4sa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* DSV4SA_H_ */
