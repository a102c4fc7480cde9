// attn_decode.cu -- decode sparse attention: the gathered rows of one query split
// over the CTAs of a thread-block cluster.
//
// Computes, for query t and head h over the multiset J of valid indices of
// idx_c[t] ++ (window of raw tokens),
//   o[t, h] = sum_j e^{a_j} kv_j / (sum_j e^{a_j} + e^{sink_h}),  a_j = scale * q[t, h] . kv_j
// ("DeepSeek-V4 全面解读" §3.7 sparse_attn_kernel; "tilelang量化内核拆解…"
// sparse_attn 实现拆解: running max starts at -1e30, an all-invalid row gives
// zeros; "DeepSeek-V4 in SGLang" MQALayer: one kv tensor is both K and V).
//
// Design.  CS CTAs (2, 4 or 8) form a cluster per (query, group of up to 64
// heads); CTA r owns 1/CS of the window list and 1/CS of the compressed list.
// Every warp of a CTA takes part in every phase, one phase after the other:
//   1. gather: thread (row r = tid / 4, quarter q = tid % 4) loads its row's
//      FP8 codes in the 16-byte pieces q, q + 4, ..., q + 24 (piece j of a
//      quarter holds 16 dims of scale group j), rope pieces q and q + 4 and the
//      row's 7 scales, all in flight together; then it dequantises into the
//      128 x 512 BF16 tile (128-byte swizzle, K-major for S, read MN-major for
//      PV).  Rows that are invalid or past the chunk are written as zeros.
//   2. S^T = KV . Q^T on tcgen05 (kind::f16, M = 128 rows, N = heads), issued by
//      one thread, completion on an mbarrier.
//   3. softmax in the exp2 domain: warp (lane quarter g, head slice s) holds the
//      scores of rows 32 g .. 32 g + 31 for a quarter of the heads; per-head max
//      and sum by a transposing warp reduction and a 4-way step through shared
//      memory; P written in BF16; O rescaled in TMEM when the max moves.
//   4. O^T += V^T . P^T (M = 128 dims x 4 blocks, N = heads, K = rows).
// The window rows only need the query's position, so with the early-window
// flag they are processed while the top-k that precedes this kernel still
// runs; the query's page-table row is staged in shared memory at the same time,
// so after the top-k a compressed row is located with one global load (its
// index) and one shared-memory load (its page).
// Merge, with no trip through global memory: once its last PV is done a CTA
// arrives on a cluster barrier (its tiles may now be written by the others),
// stages, for each other CTA of the cluster, its per-head (max, sum) and its
// unscaled O (BF16) over that CTA's 1/CS slice of dims, waits on the barrier, and
// sends each staged slot with one bulk copy into the owner's shared memory,
// completing on the owner's mbarrier.  The owner forms the global max and the
// denominator (the sink added once) from the CS (max, sum) pairs, scales and
// sums its own partial (still in TMEM) and the received ones, and writes its
// slice as BF16.  A second split barrier keeps every CTA alive until the copies
// out of its shared memory have landed.
#include "attn_common.cuh"

namespace dsv4sa {
namespace {

using namespace attn;

constexpr int kThreadsD = 512;
constexpr int kPtCache = 1024;     // page-table entries of the query's sequence kept in shared memory
constexpr float kRescaleSlack = 8.f;   // log2 units the running max may trail a chunk's max by before O is rescaled

template <int HN>
struct DSmem {
  static constexpr int kKv = 0;                          // BF16 tile; in the merge: receive slots + staging
  static constexpr int kQ = kKvBytes;                    // 8 column blocks x HN rows x 128 B
  static constexpr int kP = kQ + 8 * HN * 128;           // 2 row blocks x HN rows x 128 B
  static constexpr int kTiles = kP + 2 * HN * 128;       // end of the tiles (the merge may use all of them)
  static constexpr int kPt = kTiles;                     // int32 [kPtCache]
  static constexpr int kRowIdx = kPt + kPtCache * 4;    // int32 [kFusedMaxSplitRows]: fused mode, this CTA's compressed rows
  static constexpr int kRowValid = kRowIdx + kFusedMaxSplitRows * 4;   // uint8 [2][128]
  static constexpr int kRedMax = kRowValid + 256;        // float [4][HN]
  static constexpr int kRedSum = kRedMax + 4 * HN * 4;   // float [4][HN]; merge: factors [8][HN] over both
  static constexpr int kMUsed = kRedSum + 4 * HN * 4;    // float [HN] each
  static constexpr int kLRun = kMUsed + HN * 4;
  static constexpr int kAlpha = kLRun + HN * 4;
  static constexpr int kSink = kAlpha + HN * 4;          // float [HN]: the heads' sinks x log2(e)
  static constexpr int kMl = kSink + HN * 4;             // float2 [kMaxClusterSplits][HN]: every split's (m, l)
  static constexpr int kBar = kMl + kMaxClusterSplits * HN * 8;   // 4 mbarriers
  static constexpr int kTmem = kBar + 32;
  static constexpr int kBytes = kTmem + 16;
};

// Bytes of one merge slot: the sender's per-head (max, sum) in fp32, then its
// unscaled partial O over the receiver's slice of dims, [dim][head] BF16 with
// rows of hn + 8 values (the 16-byte pad spreads a warp's vector accesses over
// every bank).  (Moving these slots between SMs is bandwidth-bound, so BF16
// halves the merge; its rounding, 2^-9 of a partial, is the size of the
// output's own.)
__host__ __device__ constexpr int merge_row(int hn) { return hn + 8; }
__host__ __device__ constexpr int merge_slot_bytes(int hn, int cs) { return hn * 8 + (512 / cs) * merge_row(hn) * 2; }

// The largest cluster whose receive slots and staging fit in the tiles.
template <int HN>
constexpr int max_cluster() {
  return 2 * 7 * merge_slot_bytes(HN, 8) <= DSmem<HN>::kTiles ? 8 : (2 * 3 * merge_slot_bytes(HN, 4) <= DSmem<HN>::kTiles ? 4 : 2);
}

// The loads of one row piece set: thread (row, quarter) holds the 16-byte code
// pieces quarter + 4 j (j = 0..6: 16 dims of scale group j), rope pieces
// quarter and quarter + 4, and the row's 8 scale slots.
struct RowLoads {
  uint4 nope[7];
  uint4 rope[2];
  uint4 scl[2];
};

// One thread issues S^T = KV . Q^T: 32 MMAs of K = 16 over the 512 dims.
template <int HN>
__device__ __forceinline__ void issue_s(uint32_t d_tmem, const uint8_t* kv, const uint8_t* qs) {
  const uint32_t idesc = make_idesc(kFmtBF16, kFmtBF16, 0, 0, 128, HN);
  const uint64_t a0 = smem_desc_sw128(smem_u32(kv), 16, 1024), b0 = smem_desc_sw128(smem_u32(qs), 16, 1024);
#pragma unroll
  for (int kk = 0; kk < 32; ++kk) {   // descriptor + (byte offset >> 4) addresses the next 16 dims
    const uint32_t ao = ((kk >> 2) * kKvBlock + (kk & 3) * 32) >> 4, bo = ((kk >> 2) * (HN * 128) + (kk & 3) * 32) >> 4;
    mma_f16(d_tmem, a0 + ao, b0 + bo, idesc, kk > 0 ? 1u : 0u);
  }
}

// One thread issues O^T (+)= V^T . P^T: 4 blocks of 128 dims x 8 MMAs of 16 rows.
template <int HN>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, const uint8_t* kv, const uint8_t* ps, bool accumulate) {
  const uint32_t idesc = make_idesc(kFmtBF16, kFmtBF16, 1, 0, 128, HN);
  const uint64_t a0 = smem_desc_sw128(smem_u32(kv), kKvBlock, 1024), b0 = smem_desc_sw128(smem_u32(ps), 16, 1024);
#pragma unroll
  for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t ao = (2 * mb * kKvBlock + kk * 2048) >> 4, bo = ((kk >> 2) * (HN * 128) + (kk & 3) * 32) >> 4;
      mma_f16(d_tmem + mb * HN, a0 + ao, b0 + bo, idesc, (accumulate || kk > 0) ? 1u : 0u);
    }
  }
}

// ---------------------------------------------------------------- fused top-k
// The selection of dsv4sa_topk ("DeepSeek-V4 全面解读" §2.10 step 9; "DeepSeek-V4
// in SGLang" 算法2: the k largest index scores of a query, ascending, lower
// index first among equal scores, -0 == +0, NaN below every number), taken by
// the CS CTAs of the query's cluster together, in the KV tile of each CTA
// (idle until the query's rows are gathered):
//   1. each CTA loads its 1/CS share of the row (coalesced 16-byte loads);
//      every thread's largest score is a distinct entry, so each warp sorts its
//      32 thread maxima and offers its r-th largest (r = ceil(k / (16 CS)))
//      with how many maxima are at least that large; the offers go to every
//      CTA and the smallest one bounds the k-th largest score from below;
//   2. each CTA counts its scores at or above the bound and tells every CTA;
//   3. each CTA packs its contenders (order key, position) into its segment of
//      the array (padded to a multiple of 8) and copies the segment into every
//      other CTA with 16-byte stores -- the array is in position order and
//      identical everywhere;
//   4. every CTA finds the k-th largest key among the contenders (radix passes
//      of 11 bits on the shared-memory array, the few keys of the found digit
//      ranked directly) and takes the output ranks of the contenders in
//      position order; CTA r keeps ranks [r kc_split, (r + 1) kc_split) as its
//      compressed rows and writes them to idx_c_out.
// When the offers do not add up to k (a short row) every valid score is a
// contender (at most 16384).  The padding has key 0 (a NaN's key, the lowest):
// with at least k real contenders it never displaces one, and the ranking
// skips it.
struct FusedScratch {                       // at the start of the (idle) KV tile
  uint2 offers[kMaxClusterSplits * 16];     // per CTA and warp: (key, count)
  uint32_t counts[kMaxClusterSplits];       // contenders per CTA
  uint32_t hist[2048];
  uint32_t scan[16];
  unsigned long long scan64[16];
  uint32_t red[2][16];
  uint32_t cand[256];
  int found_bin, found_above, found_count, n_cand;
  uint32_t kth;
  int need;
};
constexpr int kFusedCand = 16384 + 8 * kMaxClusterSplits;  // contenders, with each CTA's padding
constexpr int kFusedKeyOff = 16384;                         // uint32 [kFusedCand] contender keys
constexpr int kFusedPosOff = kFusedKeyOff + kFusedCand * 4;  // uint16 [kFusedCand] contender positions
static_assert(sizeof(FusedScratch) <= kFusedKeyOff, "fused scratch header");
static_assert(kFusedPosOff + kFusedCand * 2 <= kKvBytes, "fused scratch fits the KV tile");

__device__ __forceinline__ uint32_t order_key_f(float f) {
  uint32_t b = __float_as_uint(f);
  if ((b & 0x7FFFFFFFu) > 0x7F800000u) return 0u;  // NaN: lowest
  if ((b & 0x7FFFFFFFu) == 0u) b = 0u;             // -0 == +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
// The float a (non-NaN) order key stands for: x >= key_float_f(k) iff order_key_f(x) >= k.
__device__ __forceinline__ float key_float_f(uint32_t kk) {
  return __uint_as_float((kk & 0x80000000u) ? (kk ^ 0x80000000u) : ~kk);
}

// Exclusive scan over the CTA's 512 threads; returns the total.
template <class T>
__device__ __forceinline__ T cta_scan(T v, T* buf, T& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  T x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) buf[warp] = x;
  __syncthreads();
  const T w = lane < 16 ? buf[lane] : T(0);
  T wx = w;
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) {
    const T y = __shfl_up_sync(0xffffffffu, wx, o);
    if (lane >= o) wx += y;
  }
  total = __shfl_sync(0xffffffffu, wx, 15);
  const T before = __shfl_sync(0xffffffffu, wx - w, warp);
  __syncthreads();
  return before + x - v;
}

// The k-th largest of the keys ckey[0..C) (at least k of them real; padding,
// position 0xFFFF, has key 0) and how many of its ties, lowest positions first,
// belong to the top k.  The key range starts from the smallest real key.
__device__ void select_kth(const uint32_t* ckey, const uint16_t* cpos, int C, int k, FusedScratch& s, uint32_t& kth,
                           int& need) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t mn = 0xFFFFFFFFu, mx = 0u;
#pragma unroll 1
  for (int c = tid; c < C; c += kThreadsD) {
    if (cpos[c] == 0xFFFFu) continue;
    mn = min(mn, ckey[c]);
    mx = max(mx, ckey[c]);
  }
  mn = __reduce_min_sync(0xffffffffu, mn);
  mx = __reduce_max_sync(0xffffffffu, mx);
  if (lane == 0) {
    s.red[0][warp] = mn;
    s.red[1][warp] = mx;
  }
  __syncthreads();
  mn = __reduce_min_sync(0xffffffffu, lane < 16 ? s.red[0][lane] : 0xFFFFFFFFu);
  mx = __reduce_max_sync(0xffffffffu, lane < 16 ? s.red[1][lane] : 0u);
  if (mn == mx) {   // every key equal
    kth = mx;
    need = k;
    return;
  }
  int hi = 31 - __clz(mn ^ mx);
  uint32_t pmask = hi == 31 ? 0u : (0xFFFFFFFFu << (hi + 1));
  uint32_t prefix = mx & pmask;
  int rem = k;
#pragma unroll 1
  while (hi >= 0) {
    const int lo = hi - 10 > 0 ? hi - 10 : 0;
    const uint32_t dmask = (2u << (hi - lo)) - 1u;
#pragma unroll
    for (int q = 0; q < 4; ++q) s.hist[tid * 4 + q] = 0u;
    __syncthreads();
#pragma unroll 1
    for (int c = tid; c < C; c += kThreadsD) {
      const uint32_t key = ckey[c];
      if ((key & pmask) == prefix) atomicAdd(&s.hist[(key >> lo) & dmask], 1u);
    }
    __syncthreads();
    uint32_t cb[4], local = 0;   // bins [2048 - 4 (tid + 1), 2048 - 4 tid), highest first
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      cb[q] = s.hist[2047 - tid * 4 - q];
      local += cb[q];
    }
    uint32_t tot;
    const int above = static_cast<int>(cta_scan<uint32_t>(local, s.scan, tot));
    if (above < rem && above + static_cast<int>(local) >= rem) {
      int acc = above;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (acc < rem && acc + static_cast<int>(cb[q]) >= rem) {
          s.found_bin = 2047 - tid * 4 - q;
          s.found_above = acc;
          s.found_count = static_cast<int>(cb[q]);
        }
        acc += static_cast<int>(cb[q]);
      }
    }
    if (tid == 0) s.n_cand = 0;
    __syncthreads();
    rem -= s.found_above;
    prefix |= static_cast<uint32_t>(s.found_bin) << lo;
    pmask |= dmask << lo;
    hi = lo - 1;
    const int count = s.found_count;
    if (hi >= 0 && count <= 256) {   // rank the keys of the found digit directly
#pragma unroll 1
      for (int c = tid; c < C; c += kThreadsD) {
        const uint32_t key = ckey[c];
        if ((key & pmask) == prefix) s.cand[atomicAdd(&s.n_cand, 1)] = key;
      }
      __syncthreads();
#pragma unroll 1
      for (int i = tid; i < count; i += kThreadsD) {
        const uint32_t mine = s.cand[i];
        int gt = 0, eq = 0;
#pragma unroll 4
        for (int j = 0; j < count; ++j) {
          gt += s.cand[j] > mine ? 1 : 0;
          eq += s.cand[j] == mine ? 1 : 0;
        }
        if (gt < rem && gt + eq >= rem) {   // every tie of the k-th key writes the same values
          s.kth = mine;
          s.need = rem - gt;
        }
      }
      __syncthreads();
      kth = s.kth;
      need = s.need;
      return;
    }
    __syncthreads();
  }
  kth = prefix;
  need = rem;
}

// The fused selection for query t (every thread of every CTA of the cluster
// calls it; n_t = clamp(n_vis[t], <= n_max) is the same in all of them).
// Writes rowidx[0 .. kc_split) with this CTA's share of the kc list slots
// (the k selected entries in order, then -1) and that share of idx_c_out[t].
__device__ void fused_topk(const AttnParams& p, int t, int n_t, int crank, int CS, uint8_t* kv, int32_t* rowidx) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = p.topk_k, share0 = crank * p.kc_split;
  int32_t* out = p.idx_c_out + static_cast<int64_t>(t) * p.idx_c_stride;
  // slots past the selection (every slot at or past min(n_t, k)) hold -1; with
  // no selection needed (n_t <= k) the slots below n_t hold 0 .. n_t - 1
  for (int r = tid; r < p.kc_split; r += kThreadsD) {
    const int g = share0 + r;
    if (g >= p.kc) continue;
    if (g >= k || n_t <= k) {
      const int32_t e = g < n_t && g < k ? g : -1;
      rowidx[r] = e;
      out[g] = e;
    }
  }
  if (n_t <= k) {
    __syncthreads();
    return;
  }
  FusedScratch& s = *reinterpret_cast<FusedScratch*>(kv);
  uint32_t* ckey = reinterpret_cast<uint32_t*>(kv + kFusedKeyOff);
  uint16_t* cpos = reinterpret_cast<uint16_t*>(kv + kFusedPosOff);
  // ---- 1. this CTA's share: float positions [crank len, (crank + 1) len), four groups
  // of 2048 at most; thread tid holds float4 q = crank len / 4 + tid + 512 j of group j
  const int len = (p.n_max + CS * 2048 - 1) / (CS * 2048) * 2048;
  const int ngroups = len / 2048;   // <= 4 (rows of at most 16384 entries over >= 2 CTAs)
  const float* row = p.logits + static_cast<int64_t>(t) * p.logits_stride;
  float x[16];
  uint32_t vmask = 0u;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int q = crank * len / 4 + tid + 512 * j;
    const bool in_grp = j < ngroups;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (in_grp && 4 * q < n_t) {
      if (4 * q + 3 < n_t) {
        v = __ldcg(reinterpret_cast<const float4*>(row) + q);
      } else {   // the row's last partial group of four
        v.x = __ldcg(row + 4 * q);
        if (4 * q + 1 < n_t) v.y = __ldcg(row + 4 * q + 1);
        if (4 * q + 2 < n_t) v.z = __ldcg(row + 4 * q + 2);
      }
    }
    x[4 * j] = v.x;
    x[4 * j + 1] = v.y;
    x[4 * j + 2] = v.z;
    x[4 * j + 3] = v.w;
#pragma unroll
    for (int i = 0; i < 4; ++i) vmask |= ((in_grp && 4 * q + i < n_t) ? 1u : 0u) << (4 * j + i);
  }
  // thread maximum over its valid non-NaN scores
  float tm = __uint_as_float(0x7FC00000u);
#pragma unroll
  for (int i = 0; i < 16; ++i)
    if (vmask >> i & 1u) tm = fmaxf(tm, x[i]);
  const bool holds = !isnan(tm);
  uint32_t v = holds ? order_key_f(tm) : 0u;
#pragma unroll
  for (int kk = 2; kk <= 32; kk <<= 1) {
#pragma unroll
    for (int j = kk >> 1; j > 0; j >>= 1) {
      const uint32_t o = __shfl_xor_sync(0xffffffffu, v, j);
      const bool lower = (lane & j) == 0, desc = (lane & kk) == 0;
      v = (lower == desc) ? max(v, o) : min(v, o);   // descending overall
    }
  }
  {
    const int holders = __popc(__ballot_sync(0xffffffffu, holds));
    const int r = min((k + 16 * CS - 1) / (16 * CS), holders);
    const uint32_t offer = __shfl_sync(0xffffffffu, v, max(r - 1, 0));
    if (lane < CS)
      st_cluster_v2u32(cluster_map(smem_u32(&s.offers[crank * 16 + warp]), static_cast<uint32_t>(lane)), offer,
                       static_cast<uint32_t>(r));
  }
  cluster_sync();   // every warp's offer is in every CTA
  uint32_t bound, total_offered;
  {
    uint32_t b = 0xFFFFFFFFu, cnt = 0u;
    for (int i = lane; i < 16 * CS; i += 32) {
      const uint2 o = s.offers[i];
      cnt += o.y;
      if (o.y > 0) b = min(b, o.x);
    }
    bound = __reduce_min_sync(0xffffffffu, b);
    total_offered = __reduce_add_sync(0xffffffffu, cnt);
  }
  const bool bounded = total_offered >= static_cast<uint32_t>(k);
  const float bf = key_float_f(bound);
  // ---- 2. contenders of each group: valid scores at or above the bound (every valid
  // score, NaN included, when there is no bound)
  unsigned long long cnt64 = 0ull;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t c = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) c += ((vmask >> (4 * j + i) & 1u) && (!bounded || x[4 * j + i] >= bf)) ? 1u : 0u;
    cnt64 |= static_cast<unsigned long long>(c) << (16 * j);
  }
  unsigned long long tot64;
  const unsigned long long before = cta_scan<unsigned long long>(cnt64, s.scan64, tot64);
  int mine_total = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) mine_total += static_cast<int>((tot64 >> (16 * j)) & 0xFFFFu);
  if (tid < CS)
    st_cluster_u32(cluster_map(smem_u32(&s.counts[crank]), static_cast<uint32_t>(tid)), static_cast<uint32_t>(mine_total));
  cluster_sync();   // every CTA's count is in every CTA
  int C = 0;
  // ---- 3. contenders into every CTA, in position order: each CTA packs its own
  // into its segment of its own array (padded to a multiple of 8 with key 0
  // and position 0xFFFF, which the ranking skips), then copies the segment into
  // the other CTAs with 16-byte stores
  int pbase = 0, ptot = 0, mine_pad = 0;
  for (int c = 0; c < CS; ++c) {
    const int pc = (static_cast<int>(s.counts[c]) + 7) & ~7;
    pbase += c < crank ? pc : 0;
    ptot += pc;
    if (c == crank) mine_pad = pc;
  }
  {
    int off = pbase;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int o = off + static_cast<int>((before >> (16 * j)) & 0xFFFFu);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if ((vmask >> (4 * j + i) & 1u) && (!bounded || x[4 * j + i] >= bf)) {
          ckey[o] = order_key_f(x[4 * j + i]);
          cpos[o] = static_cast<uint16_t>(4 * (crank * len / 4 + tid + 512 * j) + i);
          ++o;
        }
      }
      off += static_cast<int>((tot64 >> (16 * j)) & 0xFFFFu);
    }
    for (int o = pbase + mine_total + tid; o < pbase + mine_pad; o += kThreadsD) {
      ckey[o] = 0u;
      cpos[o] = 0xFFFFu;
    }
  }
  __syncthreads();
  {
    // units: key chunks of 4 (16 bytes), then position chunks of 8, for each other CTA
    const int ku = mine_pad / 4, pu = mine_pad / 8, per_dst = ku + pu;
#pragma unroll 1
    for (int u = tid; u < (CS - 1) * per_dst; u += kThreadsD) {
      const int dd = u / per_dst, w = u - dd * per_dst;
      const uint32_t d = static_cast<uint32_t>(dd < crank ? dd : dd + 1);
      if (w < ku) {
        st_cluster_v4u32(cluster_map(smem_u32(ckey + pbase + 4 * w), d), reinterpret_cast<const uint4*>(ckey + pbase)[w]);
      } else {
        const int v = w - ku;
        st_cluster_v4u32(cluster_map(smem_u32(cpos + pbase + 8 * v), d), reinterpret_cast<const uint4*>(cpos + pbase)[v]);
      }
    }
  }
  C = ptot;
  cluster_sync();   // the contender array is complete in every CTA
  // ---- 4. the k-th largest key, then output ranks over contiguous runs (position order)
  uint32_t kth;
  int need;
  select_kth(ckey, cpos, C, k, s, kth, need);
  const int run = (C + kThreadsD - 1) / kThreadsD;
  const int c0 = min(C, tid * run), c1 = min(C, c0 + run);
  uint32_t ng = 0, ne = 0;
  for (int c = c0; c < c1; ++c) {
    const bool real = cpos[c] != 0xFFFFu;   // padding is never selected
    ng += real && ckey[c] > kth ? 1u : 0u;
    ne += real && ckey[c] == kth ? 1u : 0u;
  }
  uint32_t tot;
  const uint32_t pre = cta_scan<uint32_t>(ng | (ne << 16), s.scan, tot);   // totals < 2^16
  int g = static_cast<int>(pre & 0xFFFFu), e = static_cast<int>(pre >> 16);
  for (int c = c0; c < c1; ++c) {
    int rank = -1;
    if (cpos[c] == 0xFFFFu) {
    } else if (ckey[c] > kth) {
      rank = g + min(e, need);
      ++g;
    } else if (ckey[c] == kth) {
      if (e < need) rank = g + e;
      ++e;
    }
    if (rank >= share0 && rank < share0 + p.kc_split) {   // rank < k <= kc
      const int32_t pos = static_cast<int32_t>(cpos[c]);
      rowidx[rank - share0] = pos;
      out[rank] = pos;
    }
  }
  __syncthreads();
}

template <int HN>
__global__ void __launch_bounds__(kThreadsD, 1) sparse_attn_decode_kernel(const AttnParams p) {
  using S = DSmem<HN>;
  extern __shared__ uint8_t smem_raw[];
  // 128-byte swizzled operand tiles need 1024-byte aligned bases
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* kv = smem + S::kKv;
  uint8_t* qs = smem + S::kQ;
  uint8_t* ps = smem + S::kP;
  int32_t* ptc = reinterpret_cast<int32_t*>(smem + S::kPt);
  uint8_t* rowvalid = smem + S::kRowValid;
  int32_t* rowidx = reinterpret_cast<int32_t*>(smem + S::kRowIdx);
  float* red_max = reinterpret_cast<float*>(smem + S::kRedMax);
  float* red_sum = reinterpret_cast<float*>(smem + S::kRedSum);
  float* m_used = reinterpret_cast<float*>(smem + S::kMUsed);
  float* l_run = reinterpret_cast<float*>(smem + S::kLRun);
  float* alpha = reinterpret_cast<float*>(smem + S::kAlpha);
  float* sink2s = reinterpret_cast<float*>(smem + S::kSink);
  uint64_t* bar_s = reinterpret_cast<uint64_t*>(smem + S::kBar);   // S MMA done
  uint64_t* bar_o = bar_s + 1;                                       // PV MMA done
  uint64_t* bar_recv = bar_s + 2;                                    // merge: the other splits' slots landed
  uint64_t* bar_ml = bar_s + 3;                                      // merge: the other splits' (m, l) landed
  float2* mlr = reinterpret_cast<float2*>(smem + S::kMl);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + S::kTmem);

  constexpr int HQ = HN / 4;   // heads per warp in the softmax and the output pass
  constexpr uint32_t kTmemCols = HN == 64 ? 512u : (HN == 32 ? 256u : 128u);
  constexpr uint32_t kColS = 0, kColO = HN;   // S^T: HN columns; O^T: 4 blocks x HN columns

  const int crank = static_cast<int>(cluster_ctarank());
  const int CS = p.nsplit;
  const int slice = 512 / CS;                       // dims of the output this CTA reduces
  const int slot_bytes = merge_slot_bytes(HN, CS);
  const int t = blockIdx.y;
  const int h0 = blockIdx.z * HN;
  const int hreal = min(HN, p.H - h0);
  const int tid = threadIdx.x;
  const uint32_t warp = warp_id(), lane = lane_id();

  if (tid == 0) {
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    mbar_init(bar_recv, 1);
    mbar_init(bar_ml, (CS - 1) * HN);   // one remote arrival per head from every other split
    fence_mbar_init();
    // the CS - 1 slots the other CTAs of the cluster will copy in
    mbar_arrive_expect_tx(bar_recv, static_cast<uint32_t>((CS - 1) * slot_bytes));
  }
  if (warp == 0) {
    tmem_alloc(tmem_holder, kTmemCols);
    tmem_relinquish();
  }
  cluster_arrive();   // this CTA's barriers are initialised (waited for before the loop)
  griddep_launch();
  if (p.fused && tid == 0) asm volatile("prefetch.global.L2 [%0];" ::"l"(p.n_vis + blockIdx.y));
  // Without early_window every input may come from the previous kernel of the
  // stream; with it the caller guarantees that only idx_c (or, fused, the
  // logits) does.
  bool waited = false;
  if (!p.early_window) {
    griddep_wait();
    waited = true;
  }

  const int seq = __ldg(p.q_seq + t);
  const int32_t* cpt = p.comp_pt + static_cast<int64_t>(seq) * p.comp_pt_stride;
  const int32_t* wpt = p.win_pt + static_cast<int64_t>(seq) * p.win_pt_stride;
  const bool pt_cached = p.kc > 0 && p.comp_pt_stride <= kPtCache;
  {
    // Q block of this head group -> swizzled K-major tile; padded heads are zero
    constexpr int kQIters = HN * 64 / kThreadsD;
    const uint4* qsrc = reinterpret_cast<const uint4*>(p.q);
    uint4 qv[kQIters];
#pragma unroll
    for (int i = 0; i < kQIters; ++i) {
      const int u = i * kThreadsD + tid, h = h0 + (u >> 6);
      qv[i] = h < p.H ? __ldg(qsrc + (static_cast<int64_t>(t) * p.H + h) * 64 + (u & 63)) : make_uint4(0u, 0u, 0u, 0u);
    }
    // the query's compressed page-table row (a step input, not produced by the previous kernel)
    if (pt_cached)
      for (int e = tid; e < p.comp_pt_stride; e += kThreadsD) ptc[e] = __ldg(cpt + e);
#pragma unroll
    for (int i = 0; i < kQIters; ++i) {
      const int u = i * kThreadsD + tid, h = u >> 6, v = u & 63;
      *reinterpret_cast<uint4*>(qs + (v >> 3) * (HN * 128) + sw128_offset(h, v & 7)) = qv[i];
    }
  }
  fence_proxy_async_smem();
  if (tid < HN) {
    m_used[tid] = -1e30f;
    l_run[tid] = 0.f;
    // the sinks now, not in the merge: after an idle stretch they are a cold load
    sink2s[tid] = tid < hreal ? __ldg(p.sink + h0 + tid) * kLog2e : -INFINITY;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  // rows of this CTA: its share of the window list, then of the compressed list
  const int ws0 = min(p.kw, crank * p.kw_split), ws1 = min(p.kw, ws0 + p.kw_split);
  const int cs0 = min(p.kc, crank * p.kc_split), cs1 = min(p.kc, cs0 + p.kc_split);
  const int nwch = (ws1 - ws0 + kRows - 1) / kRows;
  const int nch = nwch + (cs1 - cs0 + kRows - 1) / kRows;
  const int32_t wpos = p.idx_w ? 0 : __ldg(p.win_pos + t);

  const int row = tid >> 2, quarter = tid & 3;
  int n_t = -1;   // fused mode: the query's visible entries (-1: its list is in idx_c)
  const uint32_t g = warp & 3u;        // TMEM lane quarter of this warp
  const uint32_t hs = warp >> 2;       // softmax / output: head slice; staging: O block
  bool ok = true;
  bool pv_issued = false;              // O holds a partial sum
  bool pv_pending = false;             // a PV was issued and not yet waited for
  uint32_t ph_s = 0, ph_o = 0;

  // Locate this thread's row of chunk c and issue its loads; returns whether
  // any row of the chunk is valid (a CTA-wide vote that also publishes rowvalid).
  auto fetch = [&](int c, RowLoads& ld) -> bool {
    const bool window = c < nwch;
    const int c0 = window ? ws0 + c * kRows : cs0 + (c - nwch) * kRows;
    const int c_rows = min(kRows, (window ? ws1 : cs1) - c0);
    if (!window && !waited) {   // idx_c comes from the previous kernel
      griddep_wait();
      waited = true;
    }
    const uint8_t* page = nullptr;
    int slot = 0;
    if (row < c_rows) {
      const int gi = c0 + row;
      int32_t e;
      if (!window) {
        e = (p.fused && n_t >= 0) ? rowidx[gi - cs0] : __ldg(p.idx_c + static_cast<int64_t>(t) * p.idx_c_stride + gi);
      } else if (p.idx_w) {
        e = __ldg(p.idx_w + static_cast<int64_t>(t) * p.idx_w_stride + gi);
      } else {
        const int64_t pw = static_cast<int64_t>(wpos) - p.kw + 1 + gi;
        e = pw < 0 ? -1 : static_cast<int32_t>(p.win_ring > 0 ? pw % p.win_ring : pw);
      }
      if (e >= 0) {
        const int32_t lim = (window ? p.win_pt_stride : p.comp_pt_stride) * 64;
        if (e < lim) {
          const int32_t pg = window ? __ldg(wpt + (e >> 6)) : (pt_cached ? ptc[e >> 6] : __ldg(cpt + (e >> 6)));
          const int64_t np = window ? p.win_num_pages : p.comp_num_pages;
          if (pg >= 0 && pg < np) {
            page = (window ? p.win_base : p.comp_base) +
                   static_cast<int64_t>(pg) * (window ? p.win_page_stride : p.comp_page_stride);
            slot = e & 63;
          } else if (quarter == 0) {
            raise_error(kErrIndex);
          }
        } else if (quarter == 0) {
          raise_error(kErrIndex);
        }
      }
    }
    const bool valid = page != nullptr;
    if (valid) {
      const uint4* np4 = reinterpret_cast<const uint4*>(page + slot * 448) + quarter;
      const uint4* rp4 = reinterpret_cast<const uint4*>(page + kPageRopeOff + slot * 128) + quarter;
      const uint4* sp4 = reinterpret_cast<const uint4*>(page + kPageScaleOff + slot * 32);
#pragma unroll
      for (int j = 0; j < 7; ++j) ld.nope[j] = __ldg(np4 + 4 * j);
      ld.rope[0] = __ldg(rp4);
      ld.rope[1] = __ldg(rp4 + 4);
      ld.scl[0] = __ldg(sp4);
      ld.scl[1] = __ldg(sp4 + 1);
    } else {
#pragma unroll
      for (int j = 0; j < 7; ++j) ld.nope[j] = make_uint4(0u, 0u, 0u, 0u);
      ld.rope[0] = ld.rope[1] = ld.scl[0] = ld.scl[1] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (quarter == 0) rowvalid[(c & 1) * 128 + row] = valid ? 1 : 0;
    return __syncthreads_or(valid ? 1 : 0) != 0;
  };

  RowLoads ld;
  bool any = false;
  bool topk_done = !p.fused;
  cluster_wait();   // every CTA's barriers are initialised: remote arrivals may start
  // Each split sends its (m, l) per head to the others as soon as its last
  // chunk's softmax is done (before its PV), so the merge factors are ready
  // when the partial outputs arrive.
  bool ml_sent = false;
  auto send_ml = [&](float m, float l) {   // threads tid < HN
#pragma unroll 1
    for (int o = 0; o < CS; ++o) {
      if (o == crank) continue;
      st_cluster_v2f32(cluster_map(smem_u32(mlr + crank * HN + tid), static_cast<uint32_t>(o)), m, l);
      mbar_arrive_remote(cluster_map(smem_u32(bar_ml), static_cast<uint32_t>(o)));
    }
  };
  if (p.fused) cluster_arrive();   // with the wait before the selection: every CTA runs before any remote store
  // Chunk c's loads are issued in iteration c - 1, right after chunk c - 1 is in
  // the tile, so they are in flight while chunk c - 1's S, softmax and PV run.
  // Fused mode: the selection runs before the first compressed chunk is fetched
  // (while the window rows' loads are in flight when there are any).
#pragma unroll 1
  for (int c = -1; c < nch; ++c) {
    if (!topk_done && (c == 0 || c + 1 == nwch)) {
      if (!waited) {
        griddep_wait();
        waited = true;
      }
      const int nv = __ldg(p.n_vis + t);
      n_t = nv < 0 ? -1 : min(nv, p.n_max);
      cluster_wait();
      if (n_t >= 0) fused_topk(p, t, n_t, crank, CS, kv, rowidx);
      topk_done = true;
    }
    if (c >= 0) {
      // ---- the previous PV reads the tile and P: wait for it before overwriting
      if (pv_pending) {
        ok = mbar_wait(bar_o, ph_o) && ok;
        ph_o ^= 1u;
        pv_pending = false;
        tc_fence_after();
      }
      if (any) {   // uniform across the CTA
        // ---- dequantise into the tile (invalid rows and rows past the chunk become zeros)
        const float sc[7] = {__uint_as_float(ld.scl[0].x), __uint_as_float(ld.scl[0].y), __uint_as_float(ld.scl[0].z),
                             __uint_as_float(ld.scl[0].w), __uint_as_float(ld.scl[1].x), __uint_as_float(ld.scl[1].y),
                             __uint_as_float(ld.scl[1].z)};
        const uint32_t u0 = static_cast<uint32_t>(2 * quarter);
#pragma unroll
        for (int j = 0; j < 7; ++j) {
          uint4 lo, hi;
          dequant16(ld.nope[j], sc[j], lo, hi);
          uint8_t* blk = kv + j * kKvBlock;
          *reinterpret_cast<uint4*>(blk + sw128_offset(row, u0)) = lo;
          *reinterpret_cast<uint4*>(blk + sw128_offset(row, u0 + 1)) = hi;
        }
        *reinterpret_cast<uint4*>(kv + 7 * kKvBlock + sw128_offset(row, quarter)) = ld.rope[0];
        *reinterpret_cast<uint4*>(kv + 7 * kKvBlock + sw128_offset(row, quarter + 4)) = ld.rope[1];
        fence_proxy_async_smem();   // the tile is read by the tensor core
      }
      __syncthreads();
    }
    const bool cur = c >= 0 && any;
    // The first compressed chunk's loads wait for the previous kernel (its
    // indices): with a window chunk in hand they go out after its PV instead.
    const bool defer = cur && !waited && c + 1 == nwch && c + 1 < nch;
    // ---- S^T = KV . Q^T, issued before the next chunk's loads (whose
    // addresses may wait on index loads)
    if (cur && tid == 0) {
      tc_fence_after();
      issue_s<HN>(tmem + kColS, kv, qs);
      mma_commit(bar_s);
    }
    if (!defer) any = c + 1 < nch ? fetch(c + 1, ld) : false;   // the next chunk's loads go out now
    if (!cur) continue;
    ok = mbar_wait(bar_s, ph_s) && ok;
    ph_s ^= 1u;
    tc_fence_after();
    // ---- online softmax: row r = 32 g + lane, heads hs * HQ .. hs * HQ + HQ - 1
    const int r = static_cast<int>(g * 32 + lane);
    const bool rv = rowvalid[(c & 1) * 128 + r] != 0;
    float sv[HQ];
    tmem_load_cols<HQ>(tmem + ((g * 32u) << 16) + kColS + hs * HQ, sv);
#pragma unroll
    for (int i = 0; i < HQ; ++i) sv[i] = rv ? sv[i] * p.scale_log2 : -INFINITY;
    constexpr int kRep = 32 / HQ;   // lanes holding the same head after the transposing reduction
    {
      float tmp[HQ];
#pragma unroll
      for (int i = 0; i < HQ; ++i) tmp[i] = sv[i];
      const float m = TransposeReduce<HQ>::run(tmp, lane, 16u, OpMax());
      if ((lane & (kRep - 1)) == 0) red_max[g * HN + hs * HQ + lane / kRep] = m;
    }
    __syncthreads();
    // The max a head's probabilities are taken against: the running one,
    // unless this chunk's max exceeds it by more than the slack (then the
    // chunk's max, and O is rescaled).  Every thread derives the same value.
    auto max_used = [&](int h) {
      const float mc = fmaxf(fmaxf(red_max[h], red_max[HN + h]), fmaxf(red_max[2 * HN + h], red_max[3 * HN + h]));
      const float mu = m_used[h];
      return mc > mu + kRescaleSlack ? mc : mu;
    };
    {
      uint8_t* prow = ps + (r >> 6) * (HN * 128);
      const uint32_t unit = static_cast<uint32_t>((r & 63) >> 3);
      const int byte_in_unit = (r & 7) * 2;
#pragma unroll
      for (int i = 0; i < HQ; ++i) {
        const int h = static_cast<int>(hs) * HQ + i;
        const float pv = ex2_approx(sv[i] - max_used(h));
        sv[i] = pv;
        *reinterpret_cast<__nv_bfloat16*>(prow + sw128_offset(h, unit) + byte_in_unit) = __float2bfloat16_rn(pv);
      }
      const float l = TransposeReduce<HQ>::run(sv, lane, 16u, OpAdd());
      if ((lane & (kRep - 1)) == 0) red_sum[g * HN + hs * HQ + lane / kRep] = l;
    }
    bool resc = false;
    float mnew = 0.f;
    if (tid < HN) {
      mnew = max_used(tid);
      const float a = ex2_approx(m_used[tid] - mnew);
      alpha[tid] = a;
      resc = pv_issued && a != 1.f;
    }
    fence_proxy_async_smem();   // P is read by the tensor core
    tc_fence_before();          // this chunk's S reads are ordered before the next S MMA
    const bool rescale = __syncthreads_or(resc ? 1 : 0) != 0;
    if (tid < HN) {
      m_used[tid] = mnew;
      const float lr = l_run[tid] * alpha[tid] + (red_sum[tid] + red_sum[HN + tid]) + (red_sum[2 * HN + tid] + red_sum[3 * HN + tid]);
      l_run[tid] = lr;
    }
    if (rescale) {
      // warp (g, block hs) owns dims 128 hs + 32 g .. + 31 of every head
      const uint32_t ta = tmem + ((g * 32u) << 16) + kColO + hs * HN;
#pragma unroll 1
      for (int j0 = 0; j0 < HN; j0 += 16) {
        float v[16];
        tmem_load_cols<16>(ta + j0, v);
#pragma unroll
        for (int x = 0; x < 16; ++x) v[x] *= alpha[j0 + x];
        tmem_st16(ta + j0, v);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncthreads();
    }
    // ---- O^T += V^T . P^T
    if (tid == 0) {
      tc_fence_after();
      issue_pv<HN>(tmem + kColO, kv, ps, pv_issued);
      mma_commit(bar_o);
    }
    pv_issued = true;
    pv_pending = true;
    if (c + 1 == nch) {   // the last chunk: (m, l) are final, sent while its PV runs
      if (tid < HN) send_ml(m_used[tid], l_run[tid]);
      ml_sent = true;
    }
    if (defer) any = fetch(c + 1, ld);
  }
  // the last chunk had no valid row (or there was none): (m, l) are final now
  if (!ml_sent && tid < HN) send_ml(m_used[tid], pv_issued ? l_run[tid] : 0.f);

  if (!waited) griddep_wait();   // outputs (lse below) are written after the previous kernels completed
  // factors, while the last PV runs: global max and denominator per head, the sink added once
  float* facs = red_max;               // [CS][HN] over the red_max / red_sum arrays (idle now)
  if (tid < HN) {
    ok = mbar_wait(bar_ml, 0) && ok;   // the other splits' (m, l)
    auto src_ml = [&](int c) -> float2 {
      return c == crank ? make_float2(m_used[tid], pv_issued ? l_run[tid] : 0.f) : mlr[c * HN + tid];
    };
    float M = -INFINITY, L = 0.f;
    if (tid < hreal) {
      const float sink2 = sink2s[tid];
      M = sink2;
      for (int c = 0; c < CS; ++c) {
        const float2 ml = src_ml(c);
        if (ml.y > 0.f) M = fmaxf(M, ml.x);
      }
      L = sink2 > -INFINITY ? exp2f(sink2 - M) : 0.f;   // a sink of -inf adds nothing
      for (int c = 0; c < CS; ++c) {
        const float2 ml = src_ml(c);
        if (ml.y > 0.f) L += ml.y * exp2f(ml.x - M);
      }
      if (crank == 0 && p.lse)
        p.lse[static_cast<int64_t>(t) * p.H + h0 + tid] = L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;   // an empty denominator gives zeros
    for (int c = 0; c < CS; ++c) {
      const float2 ml = src_ml(c);
      facs[c * HN + tid] = ml.y > 0.f ? exp2f(ml.x - M) * inv : 0.f;
    }
  }
  if (pv_pending) {
    ok = mbar_wait(bar_o, ph_o) && ok;
    tc_fence_after();
  }
  tc_fence_before();
  ok = __syncthreads_and(ok ? 1 : 0) != 0;
  tc_fence_after();
  const bool have_o = ok && pv_issued;

  // =========================== cluster merge ===========================
  // Receive slots of the other CS - 1 splits at [0, R), this CTA's outgoing
  // slots staged at [R, 2 R), R = (CS - 1) slot_bytes, both inside the idle tiles.
  cluster_arrive();   // this CTA's tiles are idle: the other CTAs may copy into them
  const int R = (CS - 1) * slot_bytes;
  uint8_t* stage = smem + R;
  auto dst_index = [&](int o) { return o < crank ? o : o - 1; };   // slot order in the staging area
  {
    // warp (g, block hs) holds dims d = 128 hs + 32 g + lane of every head
    const int d = static_cast<int>(hs * 128 + g * 32 + lane);
    const int owner = d / slice;   // warp-uniform: a slice is at least 64 aligned dims
    if (owner != crank) {
      uint4* so = reinterpret_cast<uint4*>(stage + dst_index(owner) * slot_bytes + HN * 8 + (d - owner * slice) * merge_row(HN) * 2);
      const uint32_t ta = tmem + ((g * 32u) << 16) + kColO + hs * HN;
#pragma unroll 1
      for (int j0 = 0; j0 < HN; j0 += 16) {
        float v[16];
        if (have_o) {
          tmem_load_cols<16>(ta + j0, v);
        } else {
#pragma unroll
          for (int x = 0; x < 16; ++x) v[x] = 0.f;
        }
#pragma unroll
        for (int x = 0; x < 16; x += 8)
          so[(j0 + x) / 8] = make_uint4(pack_bf16x2(v[x], v[x + 1]), pack_bf16x2(v[x + 2], v[x + 3]),
                                        pack_bf16x2(v[x + 4], v[x + 5]), pack_bf16x2(v[x + 6], v[x + 7]));
      }
    }
  }
  fence_proxy_async_smem();   // the staged slots are read by the bulk-copy engine
  __syncthreads();            // also publishes the factors
  cluster_wait();             // every CTA's tiles are idle
  if (tid == 0) {
    for (int o = 0; o < CS; ++o) {
      if (o == crank) continue;
      const int at = crank < o ? crank : crank - 1;   // this CTA's slot in o's receive area
      bulk_copy_to_cluster(cluster_map(smem_u32(smem + at * slot_bytes), static_cast<uint32_t>(o)),
                           stage + dst_index(o) * slot_bytes, static_cast<uint32_t>(slot_bytes),
                           cluster_map(smem_u32(bar_recv), static_cast<uint32_t>(o)));
    }
  }
  ok = mbar_wait(bar_recv, 0) && ok;   // the other splits' slots have landed here
  cluster_arrive();                    // ... so their copies out of the senders are complete
  // output: this CTA's dims [crank slice, (crank + 1) slice): its own partial
  // from TMEM plus the received ones, scaled by their factors; inverse rotary
  // embedding of the last 64 dims; BF16 staged as [head][slice] in the idle Q
  // tile, then written with 16-byte stores (a head's slice is contiguous)
  {
    const float4* rrow = rope_row(p, t);
    __nv_bfloat16* ostage = reinterpret_cast<__nv_bfloat16*>(qs);
    const int nblk = slice >= 128 ? slice / 128 : 1;
#pragma unroll 1
    for (int b = 0; b < nblk; ++b) {
      const int blk = (crank * slice) / 128 + b;
      const int d = blk * 128 + static_cast<int>(g * 32 + lane);
      if (d / slice != crank) continue;   // warp-uniform (a half block when slice is 64)
      const int dl = d - crank * slice;
      float acc[HQ];
      if (have_o) {
        tmem_load_cols<HQ>(tmem + ((g * 32u) << 16) + kColO + blk * HN + hs * HQ, acc);
#pragma unroll
        for (int i = 0; i < HQ; ++i) acc[i] *= facs[crank * HN + hs * HQ + i];
      } else {
#pragma unroll
        for (int i = 0; i < HQ; ++i) acc[i] = 0.f;
      }
#pragma unroll 1
      for (int c = 0; c < CS; ++c) {
        if (c == crank) continue;
        // this dim's HQ heads of source c: HQ consecutive BF16 values of row dl
        const uint4* so = reinterpret_cast<const uint4*>(smem + (c < crank ? c : c - 1) * slot_bytes + HN * 8 +
                                                         (dl * merge_row(HN) + static_cast<int>(hs) * HQ) * 2);
#pragma unroll
        for (int i0 = 0; i0 < HQ; i0 += 8) {
          float pv[8];
          if (HQ - i0 >= 8) {
            const uint4 u = so[i0 / 8];
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[x]));
              pv[2 * x] = f.x;
              pv[2 * x + 1] = f.y;
            }
          } else {   // HQ = 4: half a vector
            const uint2 u = *reinterpret_cast<const uint2*>(so);
            const uint32_t w[2] = {u.x, u.y};
#pragma unroll
            for (int x = 0; x < 2; ++x) {
              const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[x]));
              pv[2 * x] = f.x;
              pv[2 * x + 1] = f.y;
            }
          }
#pragma unroll
          for (int x = 0; x < 8 && i0 + x < HQ; ++x) {
            const int h = static_cast<int>(hs) * HQ + i0 + x;
            acc[i0 + x] = fmaf(facs[c * HN + h], pv[x], acc[i0 + x]);
          }
        }
      }
      if (rrow != nullptr && d >= 512 - 64) {   // warp-uniform: dims (d, d ^ 1) form one pair, lanes (l, l ^ 1)
        const float2 cs = __ldg(reinterpret_cast<const float2*>(rrow) + ((d - (512 - 64)) >> 1));
#pragma unroll
        for (int i = 0; i < HQ; ++i) {
          const float other = __shfl_xor_sync(0xffffffffu, acc[i], 1);
          acc[i] = (lane & 1) ? fmaf(acc[i], cs.x, -(other * cs.y)) : fmaf(acc[i], cs.x, other * cs.y);
        }
      }
#pragma unroll
      for (int i = 0; i < HQ; ++i) ostage[(static_cast<int>(hs) * HQ + i) * slice + dl] = __float2bfloat16_rn(acc[i]);
    }
    __syncthreads();
    const int units = slice / 8;   // 16-byte units of a head's slice
    const uint4* src = reinterpret_cast<const uint4*>(ostage);
#pragma unroll 1
    for (int u = tid; u < hreal * units; u += kThreadsD) {
      const int h = u / units, v = u - h * units;
      *reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(t) * p.H + h0 + h) * 512 + crank * slice + 8 * v) = src[u];
    }
  }
  tc_fence_before();
  cluster_wait();   // every CTA has received its slots: no copy reads this CTA's staging any more
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int HN>
int launch_hn_decode(const AttnParams& p, int groups, cudaStream_t stream) {
  constexpr int bytes = DSmem<HN>::kBytes + 1024;   // + alignment slack
  static_assert(bytes <= 227 * 1024, "shared memory of one CTA");
  if (p.nsplit < 2 || p.nsplit > max_cluster<HN>() || 2 * (p.nsplit - 1) * merge_slot_bytes(HN, p.nsplit) > DSmem<HN>::kTiles)
    return DSV4SA_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSV4SA_ERR_CUDA;
  if (!smem_attr_once(dev, 8 + HN / 16, reinterpret_cast<const void*>(sparse_attn_decode_kernel<HN>), bytes))
    return DSV4SA_ERR_CUDA;
  return launch_cluster_pdl(sparse_attn_decode_kernel<HN>, dim3(p.nsplit, p.T, groups), dim3(kThreadsD), bytes,
                            p.nsplit, stream, p) == cudaSuccess
             ? DSV4SA_OK
             : DSV4SA_ERR_CUDA;
}

}  // namespace

namespace attn {

int decode_max_cluster(int hn) {
  return hn <= 16 ? max_cluster<16>() : (hn <= 32 ? max_cluster<32>() : max_cluster<64>());
}

int launch_decode_cluster(const AttnParams& p, int hn, int groups, cudaStream_t stream) {
  switch (hn) {
    case 16: return launch_hn_decode<16>(p, groups, stream);
    case 32: return launch_hn_decode<32>(p, groups, stream);
    default: return launch_hn_decode<64>(p, groups, stream);
  }
}

}  // namespace attn

uint32_t read_error_word_attn_decode(cudaStream_t stream, bool clear) {
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
