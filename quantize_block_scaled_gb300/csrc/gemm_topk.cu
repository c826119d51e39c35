// NVFP4 block-scaled GEMM with a fused scoring epilogue and per-row top-k,
// for sm_103a (tcgen05 tensor cores, tensor memory, TMA, thread-block
// clusters with distributed shared memory).
//
// What it computes (nvfp4-megamoe-kernel pages: commit db07d17 "dequant
// formula is lut[w] * weight_scale * weight_scale_2"; commit 107d62d "the MMA
// output is (A * SFA) @ (B * SFB), missing gsa*gsb ... sqrt(softplus(logit *
// gsa * gsb))"; CORRECTNESS_BACKLOG.md section 5 "sqrt(softplus(X @ W_gate))
// + e_bias, top-k selection"):
//   logit[m,n] = gsa * gsb * sum_k e2m1(A[m,k]) sfa[m,k/16] e2m1(B[n,k]) sfb[n,k/16]
//   score      = logit                              (identity epilogue)
//              = sqrt(softplus(logit)) + bias[n]    (router epilogue)
//   output     = the k best scores of each row, descending, ties by lower n.
// FP32 logits never go to global memory (unless a debug buffer is given).
//
// Work split.  One thread-block cluster per 128-row tile of A.  Its C =
// n_split x k_split CTAs each multiply the tile by one slice of B's columns
// (BN = 128 or 256 of them) over one slice of K, so a decode-sized problem
// (a few rows, a 1 MB weight) spreads its weight read over up to 16 SMs and
// a prefill-sized one gives every SM a tile.
//
// Per CTA, 6 warps during the main loop:
//   warp 0     producer: TMA loads of the A and B code tiles (128-byte rows,
//              128-byte swizzle) and of the scale bytes into a ring of
//              stages of K = 512.
//   warp 1     MMA issuer (one thread): eight 128 x BN x 64 kind::mxf4nvf4
//              block-scaled MMAs per stage into one TMEM accumulator, one
//              commit per stage.
//   warps 2-5  write each stage's E4M3 scale words (staged with its tiles by
//              TMA, or loaded from global memory when the scale rows are not
//              16-byte aligned) into tensor memory with tcgen05.st, each warp
//              the lanes of its own sub-partition.
//
// Then one of two epilogues.
//  Direct (no K split, k <= 32): the thread that owns TMEM lane r owns row
//    r.  It walks its columns 32 at a time: scores the whole chunk
//    branch-free (independent columns give the exponential, log and square
//    root instruction-level parallelism), then compares each score with the
//    current k-th best and inserts into a sorted register list.  With an N
//    split, each CTA pushes its per-row lists to the row's owner in the
//    cluster (remote shared-memory stores), which merges them.
//  Reduce (K split, or k > 32): each CTA pushes its FP32 partial sums to the
//    owner of each row, laid out [K slice][column][row]; the owner's warps
//    then take one row each, sum the K slices in a fixed order, score, and
//    select: a 5-level butterfly of sorted 8-lists for k <= 8, k rounds of
//    a warp arg-max for k <= 32, and a radix select + bitonic sort on keys in
//    shared memory otherwise (the indexer's top-512).
//
// The pages' WIP fused router kernel (TMA warp, MMA warp, four epilogue warps
// with per-thread heaps) is prior art; the split, the scale-factor path and
// the selection schemes here are this library's own.
//
// Every wait on an mbarrier is bounded: after ~1 s of SM clock it records
// NVFP4_DEVICE_TIMEOUT in the workspace, tells the CTA's other warps to stop,
// lets the copies already issued land, frees tensor memory and returns.

#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "nvfp4.h"
#include "ptx.cuh"

namespace nvfp4 {
namespace {

using namespace ptx;

constexpr int BM = 128;              // MMA M: rows of A per tile
constexpr int BKB = 128;             // bytes of a K sub-tile per row = 256 FP4 elements (one TMA box, one swizzle atom)
constexpr int kSub = 2;              // K sub-tiles per pipeline stage: K = 512 per stage
constexpr int kMmaPerStage = 4 * kSub;  // MMAs of K = 64 per stage
constexpr int kThreads = 192;        // 6 warps
constexpr int kWarps = 6;
constexpr int kMaxStages = 4;
constexpr int kMaxCluster = 16;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfTmemBase = 256;  // scale factors live after the (<= 256-column) accumulator
constexpr uint32_t kCtrlBytes = 256;
// control block: 3 barriers per stage and 4 more, then the TMEM address and
// the abort flag at byte 224
constexpr uint32_t kCtrlSlot = 224;
static_assert((3 * kMaxStages + 4) * 8 <= kCtrlSlot, "barriers precede the TMEM slot");
constexpr long long kWaitLimit = 2000000000LL;  // SM cycles (~1 s)
constexpr int kSmallCols = 16;       // reduce path, small rows: <= 16 columns per lane (N <= 512)

// One stage: A and B code tiles of kSub sub-tiles each (sub-tile u of A at
// u * BM * BKB, a 128-byte-swizzled box), then (scales by TMA) the stage's
// scale bytes, SFA rows then SFB rows, 16 kSub bytes each.  Tensor memory
// per stage: the SFA words of the kMmaPerStage MMAs (4 columns each), then
// the SFB words (4 columns per MMA and 128-row atom).
template <int BN>
struct Layout {
  static constexpr int kAtomsB = BN / 128;
  static constexpr uint32_t kSubA = BM * BKB;
  static constexpr uint32_t kSubB = BN * BKB;
  static constexpr uint32_t kA = kSub * kSubA;
  static constexpr uint32_t kB = kSub * kSubB;
  static constexpr uint32_t offB = kA;
  static constexpr uint32_t kSfRow = 16 * kSub;
  static constexpr uint32_t offSf = kA + kB;
  static constexpr uint32_t kSf = (BM + BN) * kSfRow;
  static constexpr uint32_t kStage = offSf + kSf;  // 72 KB (BN 128) / 108 KB (BN 256)
  static constexpr uint32_t kSfbCol = 4 * kMmaPerStage;
  static constexpr uint32_t kSfTmemPerStage = kSfbCol + 4 * kMmaPerStage * kAtomsB;
  // stages whose scale columns fit in TMEM after the accumulator
  static constexpr int kStagesMax = static_cast<int>((kTmemCols - kSfTmemBase) / kSfTmemPerStage) < kMaxStages
                                        ? static_cast<int>((kTmemCols - kSfTmemBase) / kSfTmemPerStage)
                                        : kMaxStages;
  static_assert(kStage % 1024 == 0, "stages must keep 1 KB alignment for the 128-byte swizzle");
};

struct Params {
  const uint8_t* sfa;
  const uint8_t* sfb;
  const float* gsa;
  const float* gsb;
  const float* bias;
  int32_t* topk_idx;
  float* topk_score;
  float* topk_weight;
  float* logits;
  uint32_t* status;
  int M, N, K;
  int k;
  int epilogue;
  int num_k_tiles;
  int n_split, k_split;
  int stages;
  int sf_tma;             // scales by TMA with the stage's tiles (rows and base 16-byte aligned, K % 256 == 0);
                          // else the scale warps load them from global memory
  uint32_t region_bytes;  // pipeline ring, reused after the main loop (1 KB multiple)
  int direct;             // direct epilogue (k_split == 1, k <= 32)
  int ro;                 // rows of a tile owned by each CTA of the cluster
  int bulk;               // reduce path: rows arrive by bulk copy in a receive area beside the ring
  uint32_t recv_bytes;    // reduce path, bulk: bytes of that receive area (at the start of rowmem)
  uint32_t bias_off;      // reduce path: offset in rowmem of the staged biases (N floats)
  int rpc;                // rows per cluster tile (<= BM; smaller spreads few long rows over more clusters)
  int heads;              // indexer head reduction: A rows per token (32, 64 or 128), 0 = off
  const float* head_w;    // [tokens, heads] head weights (head reduction)
  int large;              // reduce path: rows through shared-memory keys (k > 32 or N > 512)
  int cand_cap;           // large path: power of two >= k
  uint32_t row_bytes;     // large path: bytes of one warp's key buffer (16-byte multiple)
  int vec_out;            // outputs 16-byte aligned (k == 8 rows take vector stores)
};

// Instruction descriptor of kind::mxf4nvf4: E2M1 A and B (format 1), E4M3
// scales (bit 23 = 0), both operands K-major, N >> 3 at bit 17, M >> 4 at
// bit 24, scale-factor ids 0, dense K = 64.
__host__ __device__ constexpr uint32_t make_idesc(int m, int n) {
  return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile uint32_t* abort) {
  bool ok = true;
  if (lane_id() == 0) ok = mbar_wait_bounded(bar, parity, abort, kWaitLimit);
  return __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
}

__device__ __forceinline__ void record_timeout(uint32_t* status, volatile uint32_t* abort) {
  *abort = 1u;
  atomicOr(status, NVFP4_DEVICE_TIMEOUT);
}

// Order-preserving map of a float to an unsigned key (larger float, larger key).
__device__ __forceinline__ uint32_t float_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
// (score key, column) packed so that a larger value is a better entry:
// higher score first, then lower column.  0 is below every real entry.
__device__ __forceinline__ uint64_t entry(float s, int n) {
  return (static_cast<uint64_t>(float_key(s)) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(n));
}
__device__ __forceinline__ int entry_col(uint64_t e) {
  return static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(e));
}
__device__ __forceinline__ float entry_score(uint64_t e) {
  return key_float(static_cast<uint32_t>(e >> 32));
}

// sqrt(softplus(z)) with softplus(z) = max(z, 0) + log1p(exp(-|z|)).  For
// u = exp(-|z|) < 2^-5 log1p(u) is taken from the first three terms of its
// Mercator series u - u^2/2 + u^3/3 (truncation below u^4/4, relative 8e-6);
// otherwise from the fast log of 1 + u.  The square root is the hardware
// approximation (no branch to a slow path, so columns interleave).  Relative
// error ~1e-5, far inside the 1e-3 the scores are held to.
__device__ __forceinline__ float router_weight(float z) {
  const float u = __expf(-fabsf(z));
  const float l = (u < 0.03125f) ? u * (1.0f - u * (0.5f - u * 0.333333343f)) : __logf(1.0f + u);
  float r;
  asm("sqrt.approx.f32 %0, %1;" : "=f"(r) : "f"(fmaxf(z, 0.0f) + l));
  return r;
}


// Sorted (descending) insertion into a KMAX-entry register list; equal
// scores keep the earlier entry ahead.
template <int KMAX>
__device__ __forceinline__ void list_insert(float (&tv)[KMAX], int (&ti)[KMAX], float (&tw)[KMAX],
                                            float s, int n, float w) {
#pragma unroll
  for (int i = KMAX - 1; i > 0; --i) {
    if (s > tv[i - 1]) {
      tv[i] = tv[i - 1];
      ti[i] = ti[i - 1];
      tw[i] = tw[i - 1];
    } else if (s > tv[i]) {
      tv[i] = s;
      ti[i] = n;
      tw[i] = w;
    }
  }
  if (s > tv[0]) {
    tv[0] = s;
    ti[0] = n;
    tw[0] = w;
  }
}

// The k-th best score of a sorted list: the minimum over its first k slots
// (a predicated reduction; selecting slot k-1 directly would make the
// compiler index the array and move it to local memory).
template <int KMAX>
__device__ __forceinline__ float list_kth(const float (&tv)[KMAX], int k) {
  float t = __int_as_float(0x7F800000);
#pragma unroll
  for (int i = 0; i < KMAX; ++i) t = fminf(t, i < k ? tv[i] : __int_as_float(0x7F800000));
  return t;
}

template <int KMAX>
__device__ __forceinline__ void list_init(float (&tv)[KMAX], int (&ti)[KMAX], float (&tw)[KMAX]) {
#pragma unroll
  for (int i = 0; i < KMAX; ++i) {
    tv[i] = -__int_as_float(0x7F800000);
    ti[i] = -1;
    tw[i] = 0.0f;
  }
}

template <int KMAX>
__device__ __forceinline__ void list_store(const Params& p, int64_t grow, const float (&tv)[KMAX],
                                           const int (&ti)[KMAX], const float (&tw)[KMAX]) {
  const int64_t o = grow * p.k;
  // normalised router weights: over the sum of the selected ones, in slot order
  float sum = 0.0f;
  if (p.epilogue == NVFP4_EPILOGUE_SQRT_SOFTPLUS_BIAS_NORM) {
#pragma unroll
    for (int i = 0; i < KMAX; ++i)
      if (i < p.k && ti[i] >= 0) sum += tw[i];
  }
  float wv[KMAX];
#pragma unroll
  for (int i = 0; i < KMAX; ++i) wv[i] = tw[i];
  if (p.epilogue == NVFP4_EPILOGUE_SQRT_SOFTPLUS_BIAS_NORM && sum > 0.0f) {
#pragma unroll
    for (int i = 0; i < KMAX; ++i)
      if (ti[i] >= 0) wv[i] = tw[i] / sum;
  }
  if (KMAX == 8 && p.k == 8 && p.vec_out) {
    // a row's eight outputs of each kind are 32 contiguous bytes: two
    // 16-byte stores each instead of eight scalar ones
    int4* ip = reinterpret_cast<int4*>(p.topk_idx + o);
    float4* sp = reinterpret_cast<float4*>(p.topk_score + o);
    ip[0] = make_int4(ti[0], ti[1], ti[2], ti[3]);
    ip[1] = make_int4(ti[4], ti[5], ti[6], ti[7]);
    sp[0] = make_float4(tv[0], tv[1], tv[2], tv[3]);
    sp[1] = make_float4(tv[4], tv[5], tv[6], tv[7]);
    if (p.topk_weight) {
      float4* wp = reinterpret_cast<float4*>(p.topk_weight + o);
      wp[0] = make_float4(wv[0], wv[1], wv[2], wv[3]);
      wp[1] = make_float4(wv[4], wv[5], wv[6], wv[7]);
    }
    return;
  }
#pragma unroll
  for (int i = 0; i < KMAX; ++i) {
    if (i < p.k) {  // empty slots hold -1 / -inf / 0 already
      p.topk_idx[o + i] = ti[i];
      p.topk_score[o + i] = tv[i];
      if (p.topk_weight) p.topk_weight[o + i] = wv[i];
    }
  }
}

// Normalised router weights for rows whose weights are already in global
// memory (k <= 32, one warp, after a block barrier).
__device__ __forceinline__ void normalize_row_weights(const Params& p, int64_t grow) {
  const uint32_t lane = lane_id();
  const int64_t o = grow * p.k + lane;
  const bool has = static_cast<int>(lane) < p.k && p.topk_idx[o] >= 0;
  const float w = has ? p.topk_weight[o] : 0.0f;
  float sum = w;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, off);
  if (has && sum > 0.0f) p.topk_weight[o] = w / sum;
}

// ---------------------------------------------------------------- reduce-path rows

struct RowCtx {
  float* recv;        // partial sums of this CTA's rows: [k_split][ro][rs] (row-major)
  const float* bias;  // router epilogue: all N biases, staged in shared memory
  int ro;             // rows owned per CTA
  int rs;             // floats per received row (n_split * BN; column n at offset n)
  int k_split;
  float gab;
};

// Logit of owned row rr, column n: the K slices' partial sums in slice order.
__device__ __forceinline__ float row_logit(const RowCtx& c, int rr, int n) {
  float acc = 0.0f;
  for (int ks = 0; ks < c.k_split; ++ks) acc += c.recv[(ks * c.ro + rr) * c.rs + n];
  return acc * c.gab;
}

// Sum of v[j] over the 32 lanes of the warp, column j ending in lane j
// (recursive halving: each step keeps one half of the columns and adds the
// partner lane's copy of it).
__device__ __forceinline__ float warp_reduce_scatter32(float (&v)[32]) {
  const uint32_t lane = lane_id();
#pragma unroll
  for (int half = 16; half >= 1; half >>= 1) {
    const bool upper = (lane & static_cast<uint32_t>(half)) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, half);
    }
  }
  return v[0];
}

// Floats of the staged token rows ahead of the per-quarter partial sums
// (head reduction: at most 4 tokens of BN + 4 floats in a 128-row tile).
__host__ __device__ constexpr int vrow_cap_floats(int bn) { return 4 * (bn + 4); }

// Sorting networks on keys where a larger key is a better entry.
template <typename T>
__device__ __forceinline__ void ce_desc(T& a, T& b) {
  const T hi = a > b ? a : b;
  const T lo = a > b ? b : a;
  a = hi;
  b = lo;
}

// Sort 8 keys descending (Batcher's odd-even merge sort network, 19 comparators).
template <typename T>
__device__ __forceinline__ void sort8_desc(T (&v)[8]) {
  ce_desc(v[0], v[1]); ce_desc(v[2], v[3]); ce_desc(v[4], v[5]); ce_desc(v[6], v[7]);
  ce_desc(v[0], v[2]); ce_desc(v[1], v[3]); ce_desc(v[4], v[6]); ce_desc(v[5], v[7]);
  ce_desc(v[1], v[2]); ce_desc(v[5], v[6]);
  ce_desc(v[0], v[4]); ce_desc(v[1], v[5]); ce_desc(v[2], v[6]); ce_desc(v[3], v[7]);
  ce_desc(v[2], v[4]); ce_desc(v[3], v[5]);
  ce_desc(v[1], v[2]); ce_desc(v[3], v[4]); ce_desc(v[5], v[6]);
}

// r := the 8 best of two descending lists r and g, descending.  The
// elementwise max of r against g reversed is bitonic and holds them; three
// half-cleaner levels sort it.
template <typename T>
__device__ __forceinline__ void merge_top8(T (&r)[8], const T (&g)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) r[i] = r[i] > g[7 - i] ? r[i] : g[7 - i];
  ce_desc(r[0], r[4]); ce_desc(r[1], r[5]); ce_desc(r[2], r[6]); ce_desc(r[3], r[7]);
  ce_desc(r[0], r[2]); ce_desc(r[1], r[3]); ce_desc(r[4], r[6]); ce_desc(r[5], r[7]);
  ce_desc(r[0], r[1]); ce_desc(r[2], r[3]); ce_desc(r[4], r[5]); ce_desc(r[6], r[7]);
}

// The 8 best 32-bit keys of the whole warp, in every lane: each lane sorts
// its 8, then 5 butterfly levels each keep the best 8 of two sorted lists.
__device__ __forceinline__ void warp_top8_u32(uint32_t (&v)[8]) {
  sort8_desc(v);
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = __shfl_xor_sync(0xFFFFFFFFu, v[i], o);
    merge_top8(v, w);
  }
}

// Entries (64-bit keys) that carry a float payload through the networks.
__device__ __forceinline__ void ce_pay(uint64_t& a, float& wa, uint64_t& b, float& wb) {
  const bool swap = b > a;
  const uint64_t hi = swap ? b : a, lo = swap ? a : b;
  const float whi = swap ? wb : wa, wlo = swap ? wa : wb;
  a = hi;
  b = lo;
  wa = whi;
  wb = wlo;
}
__device__ __forceinline__ void sort8_pay(uint64_t (&v)[8], float (&w)[8]) {
  ce_pay(v[0], w[0], v[1], w[1]); ce_pay(v[2], w[2], v[3], w[3]);
  ce_pay(v[4], w[4], v[5], w[5]); ce_pay(v[6], w[6], v[7], w[7]);
  ce_pay(v[0], w[0], v[2], w[2]); ce_pay(v[1], w[1], v[3], w[3]);
  ce_pay(v[4], w[4], v[6], w[6]); ce_pay(v[5], w[5], v[7], w[7]);
  ce_pay(v[1], w[1], v[2], w[2]); ce_pay(v[5], w[5], v[6], w[6]);
  ce_pay(v[0], w[0], v[4], w[4]); ce_pay(v[1], w[1], v[5], w[5]);
  ce_pay(v[2], w[2], v[6], w[6]); ce_pay(v[3], w[3], v[7], w[7]);
  ce_pay(v[2], w[2], v[4], w[4]); ce_pay(v[3], w[3], v[5], w[5]);
  ce_pay(v[1], w[1], v[2], w[2]); ce_pay(v[3], w[3], v[4], w[4]); ce_pay(v[5], w[5], v[6], w[6]);
}
__device__ __forceinline__ void merge_top8_pay(uint64_t (&r)[8], float (&rw)[8], const uint64_t (&g)[8],
                                               const float (&gw)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const bool take = g[7 - i] > r[i];
    r[i] = take ? g[7 - i] : r[i];
    rw[i] = take ? gw[7 - i] : rw[i];
  }
  ce_pay(r[0], rw[0], r[4], rw[4]); ce_pay(r[1], rw[1], r[5], rw[5]);
  ce_pay(r[2], rw[2], r[6], rw[6]); ce_pay(r[3], rw[3], r[7], rw[7]);
  ce_pay(r[0], rw[0], r[2], rw[2]); ce_pay(r[1], rw[1], r[3], rw[3]);
  ce_pay(r[4], rw[4], r[6], rw[6]); ce_pay(r[5], rw[5], r[7], rw[7]);
  ce_pay(r[0], rw[0], r[1], rw[1]); ce_pay(r[2], rw[2], r[3], rw[3]);
  ce_pay(r[4], rw[4], r[5], rw[5]); ce_pay(r[6], rw[6], r[7], rw[7]);
}

// Reduce path with k <= 32 and N <= 512, where the K split is at least 2.
// Step 1, every thread of the CTA: sum the K slices of each (owned row,
// 4-column group) in slice order, apply the epilogue, and leave the score in
// slice 0 and the unbiased weight in slice 1 of the receive area (each cell
// is read and rewritten by the one thread that owns it).  Step 2, one warp
// per row: columns lane + 32 i, top-k selection, outputs.
__device__ void rows_small(const Params& p, const RowCtx& c, int owned, int64_t grow0) {
  const uint32_t lane = lane_id();
  const int warp = static_cast<int>(threadIdx.x >> 5);
  const bool router = p.epilogue != NVFP4_EPILOGUE_IDENTITY;
  const int slice = c.ro * c.rs;  // floats per K slice
  const int groups = (p.N + 3) >> 2;
  for (int it = static_cast<int>(threadIdx.x); it < owned * groups; it += kThreads) {
    const int rr = it / groups;
    const int n0 = 4 * (it - rr * groups);
    float* cell = c.recv + rr * c.rs + n0;
    float4 a = *reinterpret_cast<const float4*>(cell);
#pragma unroll 8
    for (int ks = 1; ks < c.k_split; ++ks) {
      const float4 v = *reinterpret_cast<const float4*>(cell + ks * slice);
      a.x += v.x;
      a.y += v.y;
      a.z += v.z;
      a.w += v.w;
    }
    float sv[4], wv[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + j;
      const float z = (j == 0 ? a.x : j == 1 ? a.y : j == 2 ? a.z : a.w) * c.gab;
      wv[j] = router ? router_weight(z) : z;
      sv[j] = n < p.N ? (router ? wv[j] + c.bias[n] : z) : -__int_as_float(0x7F800000);
      if (p.logits != nullptr && n < p.N) p.logits[(grow0 + rr) * p.N + n] = z;
    }
    *reinterpret_cast<float4*>(cell) = make_float4(sv[0], sv[1], sv[2], sv[3]);
    *reinterpret_cast<float4*>(cell + slice) = make_float4(wv[0], wv[1], wv[2], wv[3]);
  }
  __syncthreads();
  const int want = p.k < p.N ? p.k : p.N;
  for (int rr = warp; rr < owned; rr += kWarps) {
    const float* S = c.recv + rr * c.rs;
    const float* W = S + slice;
    const int64_t grow = grow0 + rr;
    uint64_t mine = 0ull;  // this lane's output slot: (score key, column) entry
    float mine_w = 0.0f;
    if (p.k <= 8) {
      // Selection on 32-bit keys: the score key's top 23 bits and 511 - column.
      // Exact ties still go to the lower column; scores closer than 2^-14
      // relative may trade places at the boundary (a near-tie).
      uint32_t e[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int n = static_cast<int>(lane) + 32 * i;
        e[i] = n < p.N ? ((float_key(S[n]) & 0xFFFFFE00u) | (511u - static_cast<uint32_t>(n))) : 0u;
      }
      if (p.N > 256) {  // warp-uniform: columns lane + 256 + 32 i too; keep the lane's best 8
        uint32_t f[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int n = static_cast<int>(lane) + 256 + 32 * i;
          f[i] = n < p.N ? ((float_key(S[n]) & 0xFFFFFE00u) | (511u - static_cast<uint32_t>(n))) : 0u;
        }
        sort8_desc(e);
        sort8_desc(f);
        merge_top8(e, f);
      }
      warp_top8_u32(e);  // every lane now holds the same 8 picks
      // pick lane & 7 through a select tree on its bits (a chain of equality
      // selects is turned into an indexed local-memory load by the compiler)
      const bool b0 = lane & 1u, b1 = lane & 2u, b2 = lane & 4u;
      const uint32_t x0 = b0 ? e[1] : e[0], x1 = b0 ? e[3] : e[2];
      const uint32_t x2 = b0 ? e[5] : e[4], x3 = b0 ? e[7] : e[6];
      const uint32_t key = b2 ? (b1 ? x3 : x2) : (b1 ? x1 : x0);
      // Exact score and weight of pick lane (lanes 0..7), then an exact
      // bitonic sort of those eight entries across the lanes.
      const int n = 511 - static_cast<int>(key & 0x1FFu);
      const bool has = lane < 8 && key != 0u;
      mine = has ? entry(S[n], n) : 0ull;
      mine_w = has ? W[n] : 0.0f;
#pragma unroll
      for (int size = 2; size <= 8; size <<= 1) {
#pragma unroll
        for (int j = size >> 1; j > 0; j >>= 1) {
          const uint64_t other = __shfl_xor_sync(0xFFFFFFFFu, mine, j);
          const float other_w = __shfl_xor_sync(0xFFFFFFFFu, mine_w, j);
          // descending overall: the lower lane of a pair keeps the larger entry
          // in blocks sorted descending ((lane & size) == 0), the smaller otherwise
          const bool lower = (lane & j) == 0;
          const bool desc = (lane & size) == 0 || size == 8;
          const bool take = desc == lower ? other > mine : other < mine;
          if (take) {
            mine = other;
            mine_w = other_w;
          }
        }
      }
    } else {
      uint64_t e[kSmallCols];
#pragma unroll
      for (int i = 0; i < kSmallCols; ++i) {
        const int n = static_cast<int>(lane) + 32 * i;
        e[i] = n < p.N ? entry(S[n], n) : 0ull;
      }
      for (int t = 0; t < want; ++t) {  // k rounds of a warp arg-max
        uint64_t best = e[0];
#pragma unroll
        for (int i = 1; i < kSmallCols; ++i) best = e[i] > best ? e[i] : best;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const uint64_t other = __shfl_xor_sync(0xFFFFFFFFu, best, o);
          best = other > best ? other : best;
        }
#pragma unroll
        for (int i = 0; i < kSmallCols; ++i) e[i] = e[i] == best ? 0ull : e[i];
        if (static_cast<int>(lane) == t) {
          mine = best;
          mine_w = W[entry_col(best)];
        }
      }
    }
    if (p.epilogue == NVFP4_EPILOGUE_SQRT_SOFTPLUS_BIAS_NORM) {  // warp-uniform
      float sum = static_cast<int>(lane) < want ? mine_w : 0.0f;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, off);
      if (sum > 0.0f) mine_w = mine_w / sum;
    }
    if (static_cast<int>(lane) < p.k) {
      const int64_t o = grow * p.k + lane;
      if (static_cast<int>(lane) < want) {
        p.topk_idx[o] = entry_col(mine);
        p.topk_score[o] = entry_score(mine);
        if (p.topk_weight) p.topk_weight[o] = mine_w;
      } else {
        p.topk_idx[o] = -1;
        p.topk_score[o] = -__int_as_float(0x7F800000);
        if (p.topk_weight) p.topk_weight[o] = 0.0f;
      }
    }
  }
}

// Warp inclusive prefix sum.
__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v) {
  const uint32_t lane = lane_id();
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, v, o);
    if (lane >= static_cast<uint32_t>(o)) v += t;
  }
  return v;
}

// Sort 32 * P entries descending across the warp, entry e = lane * P + j in
// v[j] (bitonic network: strides below P inside a lane, the rest by shuffles).
template <int P>
__device__ __forceinline__ void warp_bitonic_desc(uint64_t (&v)[P]) {
  const uint32_t lane = lane_id();
  constexpr int kN = 32 * P;
#pragma unroll
  for (int size = 2; size <= kN; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride < P) {
#pragma unroll
        for (int j = 0; j < P; ++j) {
          if ((j & stride) == 0) {
            const int e = static_cast<int>(lane) * P + j;
            const bool desc = (e & size) == 0;
            const uint64_t x = v[j], y = v[j | stride];
            const bool swap = desc ? (y > x) : (x > y);
            v[j] = swap ? y : x;
            v[j | stride] = swap ? x : y;
          }
        }
      } else {
        const int lx = stride / P;
#pragma unroll
        for (int j = 0; j < P; ++j) {
          const int e = static_cast<int>(lane) * P + j;
          const uint64_t other = __shfl_xor_sync(0xFFFFFFFFu, v[j], lx);
          const bool lower = (e & stride) == 0;
          const bool desc = (e & size) == 0;
          const bool keep_max = desc == lower;
          v[j] = keep_max ? (other > v[j] ? other : v[j]) : (other < v[j] ? other : v[j]);
        }
      }
    }
  }
}

__device__ __forceinline__ void store_entry(const Params& p, const RowCtx& c, int rr, int64_t o, uint64_t e) {
  const int n = entry_col(e);
  const float sc = entry_score(e);
  p.topk_idx[o] = n;
  p.topk_score[o] = sc;
  if (p.topk_weight)
    p.topk_weight[o] = p.epilogue != NVFP4_EPILOGUE_IDENTITY ? router_weight(row_logit(c, rr, n)) : sc;
}

__device__ __forceinline__ void store_empty(const Params& p, int64_t o) {
  p.topk_idx[o] = -1;
  p.topk_score[o] = -__int_as_float(0x7F800000);
  if (p.topk_weight) p.topk_weight[o] = 0.0f;
}

// Shared-memory slot of entry e of a run of 32 * P candidates that one warp
// reads and writes as e = lane * P + j: each lane's P entries are
// XOR-rotated by the lane so a warp's accesses spread over the banks.
template <int P>
__device__ __forceinline__ int run_slot(int e) {
  const int local = e & (32 * P - 1);
  return (e & ~(32 * P - 1)) | (local ^ ((local / P) & (P - 1)));
}

// Sort the run cand[base .. base + 32P) descending in place through registers.
template <int P>
__device__ void sort_run(uint64_t* cand, int base) {
  const uint32_t lane = lane_id();
  uint64_t v[P];
#pragma unroll
  for (int j = 0; j < P; ++j) v[j] = cand[run_slot<P>(base + static_cast<int>(lane) * P + j)];
  warp_bitonic_desc<P>(v);
#pragma unroll
  for (int j = 0; j < P; ++j) cand[run_slot<P>(base + static_cast<int>(lane) * P + j)] = v[j];
}

// Entries of the sorted run cand[base .. base + len) that are greater than x.
template <int P>
__device__ __forceinline__ int count_above(const uint64_t* cand, int base, int len, uint64_t x) {
  int lo = 0, hi = len;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (cand[run_slot<P>(base + mid)] > x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// Block-wide exclusive prefix sum of one value per thread; `tot` gets the
// block total.  `red` holds kWarps words; two block barriers.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* red, uint32_t* tot) {
  const uint32_t lane = lane_id();
  const int warp = static_cast<int>(threadIdx.x >> 5);
  const uint32_t incl = warp_incl_scan(v);
  if (lane == 31) red[warp] = incl;
  __syncthreads();
  uint32_t before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const uint32_t t = red[w];
    before += w < warp ? t : 0u;
    all += t;
  }
  __syncthreads();  // red is reused by the next call
  *tot = all;
  return before + incl - v;
}

// Sort the W = cap / (32P) runs, then place every candidate by its rank
// (its index in its run plus the entries of the other runs above it;
// entries are distinct) and write the outputs.
template <int P>
__device__ void sort_runs_and_store(const Params& p, const RowCtx& c, int rr, int64_t grow, uint64_t* cand) {
  const int warp = static_cast<int>(threadIdx.x >> 5);
  constexpr int kLen = 32 * P;
  const int runs = p.cand_cap / kLen;  // <= 4
  if (warp < runs) sort_run<P>(cand, warp * kLen);
  __syncthreads();
  for (int e = static_cast<int>(threadIdx.x); e < p.cand_cap; e += kThreads) {
    const uint64_t x = cand[run_slot<P>(e)];
    if (x == 0ull) continue;  // padding
    const int w = e / kLen;
    int rank = e - w * kLen;
    for (int o = 0; o < runs; ++o)
      if (o != w) rank += count_above<P>(cand, o * kLen, kLen, x);
    if (rank < p.k) store_entry(p, c, rr, grow * p.k + rank, x);
  }
}

// General rows (k > 32 or N > 512), every thread of the CTA on one row at a
// time: keys of all N scores in shared memory; the want-th largest key T by
// a search over 2-bit digits (per digit, the counts of keys >= each of three
// thresholds); the keys above T and the lowest-column keys equal to T in
// column order (two block scans); runs of up to 256 candidates sorted by
// up to four warps in registers, merged by rank; outputs.
__device__ void rows_large(const Params& p, const RowCtx& c, int owned, int64_t grow0, uint32_t* keys,
                           uint64_t* cand, uint32_t* red) {
  const uint32_t lane = lane_id();
  const int warp = static_cast<int>(threadIdx.x >> 5);
  const int tid = static_cast<int>(threadIdx.x);
  const int n_all = p.N;
  const int n4 = (n_all + 3) >> 2;  // key quads (keys past N are 0, below every real key)
  const bool router = p.epilogue != NVFP4_EPILOGUE_IDENTITY;
  const uint4* keys4 = reinterpret_cast<const uint4*>(keys);
  const uint32_t want = static_cast<uint32_t>(p.k < n_all ? p.k : n_all);
  const int qp = (n4 + kThreads - 1) / kThreads;  // quads per thread, in column order
  const int q_lo = min(n4, tid * qp), q_hi = min(n4, q_lo + qp);
  for (int rr = 0; rr < owned; ++rr) {
    const int64_t grow = grow0 + rr;
    const float* rowp = c.recv + rr * c.rs;
    for (int q = tid; q < n4; q += kThreads) {
      float4 acc = *reinterpret_cast<const float4*>(rowp + 4 * q);
      for (int ks = 1; ks < c.k_split; ++ks) {
        const float4 t = *reinterpret_cast<const float4*>(rowp + ks * c.ro * c.rs + 4 * q);
        acc.x += t.x;
        acc.y += t.y;
        acc.z += t.z;
        acc.w += t.w;
      }
      uint32_t kq[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int n = 4 * q + j;
        const float z = (j == 0 ? acc.x : j == 1 ? acc.y : j == 2 ? acc.z : acc.w) * c.gab;
        if (p.logits != nullptr && n < n_all) p.logits[grow * n_all + n] = z;
        kq[j] = n < n_all ? float_key(router ? router_weight(z) + c.bias[n] : z) : 0u;
      }
      reinterpret_cast<uint4*>(keys)[q] = make_uint4(kq[0], kq[1], kq[2], kq[3]);
    }
    __syncthreads();
    // T: per 2-bit digit from the top, the largest d with at least `want`
    // keys >= T | d << b (thresholds >= 1, so the zero keys never count).
    uint32_t T = 0;
#pragma unroll 1
    for (int b = 30; b >= 0; b -= 2) {
      const uint32_t t1 = T | (1u << b), t2 = T | (2u << b), t3 = T | (3u << b);
      uint32_t c1 = 0, c2 = 0, c3 = 0;
      for (int q = tid; q < n4; q += kThreads) {
        const uint4 k4 = keys4[q];
        const uint32_t kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          c1 += kk[j] >= t1;
          c2 += kk[j] >= t2;
          c3 += kk[j] >= t3;
        }
      }
      c1 = __reduce_add_sync(0xFFFFFFFFu, c1);
      c2 = __reduce_add_sync(0xFFFFFFFFu, c2);
      c3 = __reduce_add_sync(0xFFFFFFFFu, c3);
      uint32_t* slot = red + ((b >> 1) & 1) * (4 * kWarps);  // alternate buffers: one barrier per digit
      if (lane == 0) {
        slot[warp] = c1;
        slot[kWarps + warp] = c2;
        slot[2 * kWarps + warp] = c3;
      }
      __syncthreads();
      uint32_t s1 = 0, s2 = 0, s3 = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        s1 += slot[w];
        s2 += slot[kWarps + w];
        s3 += slot[2 * kWarps + w];
      }
      T = s3 >= want ? t3 : s2 >= want ? t2 : s1 >= want ? t1 : T;
    }
    uint32_t* scan = red + 8 * kWarps;
    // keys above T and equal to T among this thread's quads (column order)
    uint32_t gt_cnt = 0, eq_cnt = 0;
    for (int q = q_lo; q < q_hi; ++q) {
      const uint4 k4 = keys4[q];
      const uint32_t kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        gt_cnt += kk[j] > T;
        eq_cnt += kk[j] == T && kk[j] != 0u;
      }
    }
    uint32_t gt_total = 0, eq_total = 0;
    block_excl_scan(gt_cnt, scan, &gt_total);
    uint32_t eq_rank = block_excl_scan(eq_cnt, scan, &eq_total);
    const uint32_t need_eq = want - gt_total;
    uint32_t take_cnt = 0;
    for (int q = q_lo; q < q_hi; ++q) {
      const uint4 k4 = keys4[q];
      const uint32_t kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const bool eq = kk[j] == T && kk[j] != 0u;
        take_cnt += kk[j] > T || (eq && eq_rank < need_eq);
        eq_rank += eq;
      }
    }
    eq_rank -= eq_cnt;
    uint32_t out = 0;
    uint32_t pos = block_excl_scan(take_cnt, scan, &out);
    const int P = p.cand_cap <= 128 ? 1 : p.cand_cap / 128;  // 4 runs of 32P (2 runs for 64)
    for (int q = q_lo; q < q_hi; ++q) {
      const uint4 k4 = keys4[q];
      const uint32_t kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const bool eq = kk[j] == T && kk[j] != 0u;
        if (kk[j] > T || (eq && eq_rank < need_eq)) {
          const int n = 4 * q + j;
          const int e = static_cast<int>(pos++);
          const int slot_e = P == 1 ? e : P == 2 ? run_slot<2>(e) : P == 4 ? run_slot<4>(e) : run_slot<8>(e);
          cand[slot_e] = (static_cast<uint64_t>(kk[j]) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(n));
        }
        eq_rank += eq;
      }
    }
    for (int e = static_cast<int>(out) + tid; e < p.cand_cap; e += kThreads) {
      const int slot_e = P == 1 ? e : P == 2 ? run_slot<2>(e) : P == 4 ? run_slot<4>(e) : run_slot<8>(e);
      cand[slot_e] = 0ull;
    }
    for (int t = static_cast<int>(out) + tid; t < p.k; t += kThreads)  // slots past N
      store_empty(p, grow * p.k + t);
    __syncthreads();
    switch (P) {
      case 1: sort_runs_and_store<1>(p, c, rr, grow, cand); break;
      case 2: sort_runs_and_store<2>(p, c, rr, grow, cand); break;
      case 4: sort_runs_and_store<4>(p, c, rr, grow, cand); break;
      default: sort_runs_and_store<8>(p, c, rr, grow, cand); break;
    }
    __syncthreads();  // keys and candidates are rewritten for the next row
    if (p.epilogue == NVFP4_EPILOGUE_SQRT_SOFTPLUS_BIAS_NORM && p.topk_weight && warp == 0)
      normalize_row_weights(p, grow);  // k <= 32 (the outputs are visible after the barrier)
  }
}

// ---------------------------------------------------------------- the kernel

template <int BN, int KMAX>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_topk_kernel(const __grid_constant__ CUtensorMap tma_a,
                     const __grid_constant__ CUtensorMap tma_b,
                     const __grid_constant__ CUtensorMap tma_sfa, const __grid_constant__ CUtensorMap tma_sfb,
                     const __grid_constant__ Params p) {
  using L = Layout<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const int warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();
  const int S = p.stages;
  uint8_t* ctrl = smem + p.region_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(ctrl);
  auto full_bar = [&](int s) { return smem_addr(&bars[s]); };
  auto empty_bar = [&](int s) { return smem_addr(&bars[kMaxStages + s]); };
  auto sfready_bar = [&](int s) { return smem_addr(&bars[2 * kMaxStages + s]); };
  const uint32_t tfull_bar = smem_addr(&bars[3 * kMaxStages]);
  const uint32_t drain_bar = smem_addr(&bars[3 * kMaxStages + 1]);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + kCtrlSlot);
  volatile uint32_t* abort = reinterpret_cast<volatile uint32_t*>(ctrl + kCtrlSlot + 4);
  uint8_t* rowmem = ctrl + kCtrlBytes;

  const int csize = p.n_split * p.k_split;
  const int rank = static_cast<int>(cluster_ctarank());
  const int mt = blockIdx.x / csize;
  const int n_idx = rank % p.n_split;
  const int k_idx = rank / p.n_split;
  const int m0 = mt * p.rpc;
  const int n0 = n_idx * BN;
  const int vr = min(p.rpc, p.M - m0);  // valid rows of this tile
  // rows as the epilogue owns them: A rows, or tokens under head reduction
  const int vrow = p.heads ? vr / p.heads : vr;
  const int64_t out0 = p.heads ? m0 / p.heads : m0;  // output row of the tile's first owned row
  const int kt0 = k_idx * p.num_k_tiles / p.k_split;
  const int nk = (k_idx + 1) * p.num_k_tiles / p.k_split - kt0;
  const int ncols = min(BN, p.N - n0);
  const int mma_n = min(BN, (ncols + 15) & ~15);
  constexpr int kUnits = 1 + L::kAtomsB;  // scale atoms per stage: SFA + SFB's

  // The next kernel on the stream may set up while this one runs (it waits
  // for our completion before touching memory); the tensor maps are kernel
  // parameters, so their descriptors can be fetched before the previous
  // kernel has finished.
  pdl_launch_dependents();
  if (threadIdx.x == 32) {
    prefetch_tensormap(&tma_a);
    prefetch_tensormap(&tma_b);
    if (p.sf_tma) {
      prefetch_tensormap(&tma_sfa);
      prefetch_tensormap(&tma_sfb);
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(sfready_bar(s), 4);  // one arrival per scale warp
    }
    mbar_init(tfull_bar, 1);
    mbar_init(drain_bar, 1);
    mbar_init(smem_addr(&bars[3 * kMaxStages + 2]), 1);  // rows received by bulk copy
    *abort = 0u;
    fence_mbar_init();
    if (p.bulk) {
      // Bytes this CTA will receive: each K slice's partials of its own rows,
      // every column slice padded to 4 floats.
      const int owned = max(0, min(p.ro, vrow - rank * p.ro));
      uint32_t per_row = 0;
      for (int ni = 0; ni < p.n_split; ++ni) per_row += ((min(BN, p.N - ni * BN) + 3) & ~3) * 4;
      mbar_arrive_expect_tx(smem_addr(&bars[3 * kMaxStages + 2]),
                            per_row * static_cast<uint32_t>(owned * p.k_split));
    }
  }
  pdl_wait();  // the previous kernel's outputs (our A operand, scales, ...) are complete
  // Tensor memory is taken only once the previous kernel has finished, so a
  // CTA that starts early never holds it while waiting; one CTA per SM (the
  // host pads shared memory above half of the SM's) means the allocation
  // never waits for another CTA of this grid.
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    // The first stages need no empty-slot wait: start their loads now,
    // ahead of the block barrier.
    const int pre = min(S, nk);
    for (int i = 0; i < pre; ++i) {
      const uint32_t st = sbase + i * L::kStage;
      mbar_arrive_expect_tx(full_bar(i), p.sf_tma ? L::kStage : L::offSf);
#pragma unroll
      for (int u = 0; u < kSub; ++u) {
        tma_load_2d(st + u * L::kSubA, &tma_a, full_bar(i), ((kt0 + i) * kSub + u) * BKB, m0);
        tma_load_2d(st + L::offB + u * L::kSubB, &tma_b, full_bar(i), ((kt0 + i) * kSub + u) * BKB, n0);
      }
      if (p.sf_tma) {
        tma_load_2d(st + L::offSf, &tma_sfa, full_bar(i), (kt0 + i) * L::kSfRow, m0);
        tma_load_2d(st + L::offSf + BM * L::kSfRow, &tma_sfb, full_bar(i), (kt0 + i) * L::kSfRow, n0);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  // Peers' receive barriers must exist before a copy targets them: arrive
  // here, wait just before the first copy (the main loop runs in between).
  if (p.bulk) cluster_arrive();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool acc_ready = false;  // epilogue warps: the accumulator is complete

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const int pre = min(S, nk);  // stages already loaded during set-up
    int last = pre - 1;
    for (int i = pre; i < nk; ++i) {
      const int s = i % S;
      const uint32_t ph = (i / S) & 1;
      if (!warp_wait(empty_bar(s), ph ^ 1u, abort)) {
        if (lane == 0) record_timeout(p.status, abort);
        break;
      }
      const uint32_t st = sbase + s * L::kStage;
      const int kt = kt0 + i;
      if (lane == 0) {
        mbar_arrive_expect_tx(full_bar(s), p.sf_tma ? L::kStage : L::offSf);
#pragma unroll
        for (int u = 0; u < kSub; ++u) {
          tma_load_2d(st + u * L::kSubA, &tma_a, full_bar(s), (kt * kSub + u) * BKB, m0);
          tma_load_2d(st + L::offB + u * L::kSubB, &tma_b, full_bar(s), (kt * kSub + u) * BKB, n0);
        }
        if (p.sf_tma) {
          tma_load_2d(st + L::offSf, &tma_sfa, full_bar(s), kt * L::kSfRow, m0);
          tma_load_2d(st + L::offSf + BM * L::kSfRow, &tma_sfb, full_bar(s), kt * L::kSfRow, n0);
        }
      }
      last = i;
    }
    if (lane == 0) {  // let every copy issued here land before the CTA can exit
      uint32_t never = 0;
      for (int s = 0; s < S; ++s) {
        const int i_s = last - (((last - s) % S) + S) % S;
        if (last >= 0 && i_s >= 0 &&
            !mbar_wait_bounded(full_bar(s), (i_s / S) & 1, &never, kWaitLimit))
          record_timeout(p.status, abort);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc = make_idesc(BM, mma_n);
    bool ok = true;
    for (int i = 0; i < nk; ++i) {
      const int s = i % S;
      const uint32_t ph = (i / S) & 1;
      // (with the scales in the stage, the scale warps arrive on sfready(s)
      // only after full(s) has completed, which then covers A and B too)
      if ((!p.sf_tma && !warp_wait(full_bar(s), ph, abort)) || !warp_wait(sfready_bar(s), ph, abort)) {
        if (lane == 0) record_timeout(p.status, abort);
        ok = false;
        break;
      }
      if (lane == 0) {
        tc_fence_after();
        const uint32_t st = sbase + s * L::kStage;
        const uint32_t sf_col = tmem + kSfTmemBase + s * L::kSfTmemPerStage;
        // MMAs that lie wholly past K (a short last stage) are skipped
        const int nmma = min(kMmaPerStage, (p.K - (kt0 + i) * kMmaPerStage * 64 + 63) / 64);
#pragma unroll
        for (int kk = 0; kk < kMmaPerStage; ++kk) {
          if (kk < nmma)
            tc_mma_nvf4(tmem, smem_desc(st + (kk / 4) * L::kSubA + (kk % 4) * 32, 16, 1024, 2),
                        smem_desc(st + L::offB + (kk / 4) * L::kSubB + (kk % 4) * 32, 16, 1024, 2), idesc,
                        sf_col + kk * 4, sf_col + L::kSfbCol + kk * 4 * L::kAtomsB, (i | kk) != 0 ? 1u : 0u);
        }
        tc_commit(empty_bar(s));  // frees the stage once these MMAs have read it
      }
      __syncwarp();
    }
    if (lane == 0) {
      if (ok) tc_commit(tfull_bar);
      uint32_t never = 0;
      tc_commit(drain_bar);
      if (!mbar_wait_bounded(drain_bar, 0, &never, kWaitLimit)) record_timeout(p.status, abort);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ scale factors
    // The block-scaled MMA reads the scales of MMA step kk (K = 64) of a
    // 128-row atom from 4 TMEM columns: lane l (in every 32-lane
    // sub-partition alike) holds, in column 4 kk + c, the scale word kk of
    // row 32 c + l.  Each of the four warps writes the words of its lanes
    // into its own sub-partition with tcgen05.st, so the tensor pipe carries
    // no scales.  The words come with the stage's tiles (TMA), or, when the
    // scale rows are not 16-byte aligned, straight from global memory.
    const uint32_t lane_sel = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int64_t sf_ld = p.K / 16;  // scale bytes per row
    const int kwords = p.K / 64;     // scale words per row
    for (int i = 0; i < nk; ++i) {
      const int s = i % S;
      const uint32_t ph = (i / S) & 1;
      // SFA: column 4 kk + c; SFB atom a - 1: column kSfbCol + 4 (kk kAtomsB + a - 1) + c
      uint32_t ra[4 * kMmaPerStage], rb[4 * kMmaPerStage * L::kAtomsB];
      if (p.sf_tma) {
        // the stage has landed; then the MMAs that read this slot's TMEM
        // columns in the previous round have completed (full(s) of this
        // round follows empty(s))
        if (!warp_wait(full_bar(s), ph, abort)) {
          if (lane == 0) record_timeout(p.status, abort);
          break;
        }
        const uint32_t sst = sbase + s * L::kStage + L::offSf;
#pragma unroll
        for (int a = 0; a < kUnits; ++a)
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int h = 0; h < kSub; ++h) {
              uint32_t w[4];
              ld_shared_v4(sst + ((a == 0 ? 0 : BM + (a - 1) * 128) + c * 32 + static_cast<int>(lane)) * L::kSfRow +
                               h * 16, w);
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int kk = h * 4 + j;
                if (a == 0) ra[kk * 4 + c] = w[j];
                else rb[(kk * L::kAtomsB + (a - 1)) * 4 + c] = w[j];
              }
            }
      } else {
        const int kw0 = (kt0 + i) * kMmaPerStage;  // first scale word of the stage
#pragma unroll
        for (int a = 0; a < kUnits; ++a)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int r = (a == 0 ? m0 : n0 + (a - 1) * 128) + 32 * c + static_cast<int>(lane);
            const bool row_ok = r < (a == 0 ? p.M : p.N);
            const uint32_t* rowp = reinterpret_cast<const uint32_t*>(
                (a == 0 ? p.sfa : p.sfb) + (row_ok ? static_cast<int64_t>(r) * sf_ld : 0));
#pragma unroll
            for (int kk = 0; kk < kMmaPerStage; ++kk) {
              const uint32_t w = (row_ok && kw0 + kk < kwords) ? __ldg(rowp + kw0 + kk) : 0u;
              if (a == 0) ra[kk * 4 + c] = w;
              else rb[(kk * L::kAtomsB + (a - 1)) * 4 + c] = w;
            }
          }
        // the MMAs that read this slot's TMEM columns S stages ago have completed
        if (i >= S && !warp_wait(empty_bar(s), ph ^ 1u, abort)) {
          if (lane == 0) record_timeout(p.status, abort);
          break;
        }
      }
      tc_fence_after();
      const uint32_t sf_col = tmem + lane_sel + kSfTmemBase + s * L::kSfTmemPerStage;
      static_assert(4 * kMmaPerStage == 32, "one 32-column store per 128-row atom");
      tmem_st_32x32b_x32(sf_col, ra);
      tmem_st_32x32b_x32(sf_col + L::kSfbCol, *reinterpret_cast<uint32_t(*)[32]>(rb));
      if constexpr (L::kAtomsB == 2)
        tmem_st_32x32b_x32(sf_col + L::kSfbCol + 32, *reinterpret_cast<uint32_t(*)[32]>(rb + 32));
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sfready_bar(s));
    }
    __syncwarp();
    if (p.epilogue != NVFP4_EPILOGUE_IDENTITY) {
      // The epilogue reads every bias of its columns (the row phase of the
      // reduce path: all N; the direct path: this CTA's): stage them while
      // the MMAs run.
      float* bias_s = reinterpret_cast<float*>(rowmem + p.bias_off);
      if (p.direct) {
        for (int c = (warp - 2) * 32 + static_cast<int>(lane); c < ncols; c += 128) bias_s[c] = __ldg(p.bias + n0 + c);
        asm volatile("bar.sync 1, 128;" ::: "memory");  // the four scale warps read all of them
      } else {
        for (int n = (warp - 2) * 32 + static_cast<int>(lane); n < p.N; n += 128) bias_s[n] = __ldg(p.bias + n);
      }
    }
    if (warp_wait(tfull_bar, 0, abort)) {
      acc_ready = true;
      tc_fence_after();
    } else if (lane == 0) {
      record_timeout(p.status, abort);
    }
  }

  const float gab = __ldg(p.gsa) * __ldg(p.gsb);
  const int quarter = warp & 3;  // epilogue warps read TMEM lanes 32*quarter .. +31
  const int row = quarter * 32 + static_cast<int>(lane);
  // Direct path with an N split: the per-row lists go to their owners' stage
  // regions (after the logits), free once every CTA of the cluster has left
  // its main loop (copies landed, MMAs complete): arrive here, wait just
  // before the pushes.
  const bool list_barrier = p.direct && p.n_split > 1;
  constexpr uint32_t kListOff = (4 * BN + (KMAX == 8 ? BM * (BN + 4) : 0)) * 4;
  if (list_barrier) {
    cluster_arrive();
    if (warp < 2) cluster_wait();
  }

  if (p.direct) {
    // ------------------------------------------------------------ direct epilogue
    if (warp >= 2) {
      float tv[KMAX], tw[KMAX];
      int ti[KMAX];
      list_init<KMAX>(tv, ti, tw);
      const bool router = p.epilogue != NVFP4_EPILOGUE_IDENTITY;
      const float* bias_s = reinterpret_cast<const float*>(rowmem + p.bias_off);  // staged during the main loop
      const bool live = row < vr;
      if constexpr (KMAX == 8) {
        // The logits stay in shared memory (row stride BN + 4 floats).
        float* zrow = reinterpret_cast<float*>(smem) + 4 * BN + row * (BN + 4);
        if (router) {
          // Router: only the top 8 of f(z) + bias[n], f = sqrt(softplus),
          // matter, and f is increasing.  At least 8 columns have a logit
          // >= zlo = the 8th largest of the two largest logits of each
          // 16-column group, so the 8th best score is >= f(zlo) + min(bias);
          // a column can reach it only if f(z) >= f(zlo) - (max(bias) -
          // min(bias)).  That bound (less a safety margin for the
          // approximate functions) gives a logit threshold; the few columns
          // above it are scored exactly, eight at a time (independent
          // exponentials and logarithms overlap), and kept in a sorted list
          // in column order, so equal scores keep the lower column.  No
          // column that can be selected is skipped, so the result equals
          // scoring every column.
          float blo = __int_as_float(0x7F800000), bhi = -__int_as_float(0x7F800000);
          for (int c = lane; c < ncols; c += 32) {
            blo = fminf(blo, bias_s[c]);
            bhi = fmaxf(bhi, bias_s[c]);
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            blo = fminf(blo, __shfl_xor_sync(0xFFFFFFFFu, blo, o));
            bhi = fmaxf(bhi, __shfl_xor_sync(0xFFFFFFFFu, bhi, o));
          }
          float gtop[8];  // the 8 largest of the groups' two largest logits, descending
#pragma unroll
          for (int i = 0; i < 8; ++i) gtop[i] = -__int_as_float(0x7F800000);
          if (acc_ready) {
            for (int c0 = 0; c0 < mma_n; c0 += 32) {
              uint32_t v[32];
              tmem_ld_32x32b_x32(tmem + c0 + (static_cast<uint32_t>(quarter * 32) << 16), v);
              tmem_wait_ld();
              float h[2][2];  // per 16-column group: largest, second largest
#pragma unroll
              for (int g = 0; g < 2; ++g) h[g][0] = h[g][1] = -__int_as_float(0x7F800000);
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const float z = __uint_as_float(v[j]) * gab;
                v[j] = __float_as_uint(z);
                if (p.logits != nullptr && live && c0 + j < ncols)
                  p.logits[static_cast<int64_t>(m0 + row) * p.N + n0 + c0 + j] = z;
                const float zv = c0 + j < ncols ? z : -__int_as_float(0x7F800000);
                float(&hg)[2] = h[j >> 4];
                hg[1] = fmaxf(hg[1], fminf(hg[0], zv));
                hg[0] = fmaxf(hg[0], zv);
              }
              // insert the four into the running 8 (a compare-exchange chain each)
#pragma unroll
              for (int g = 0; g < 4; ++g) {
                float x = h[g >> 1][g & 1];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  const float hi = fmaxf(gtop[i], x);
                  x = fminf(gtop[i], x);
                  gtop[i] = hi;
                }
              }
              if (live) {
                const uint32_t dst = smem_addr(zrow + c0);
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4)
                  st_shared_v4(dst + 16 * q4, v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
              }
            }
          }
          // logit threshold: f^-1(y) = softplus^-1(y^2) = log(exp(y^2) - 1), with
          // margins far above the functions' approximation error (a lower
          // threshold only admits more candidates)
          float zthr = -__int_as_float(0x7F800000);
          const float zlo = gtop[7];
          if (zlo > -__int_as_float(0x7F800000) && zlo < __int_as_float(0x7F800000)) {
            const float y = router_weight(zlo) - (bhi - blo);
            if (y > 0.0f) {
              const float ym = y - (1e-3f * y + 1e-6f);
              const float t = ym * ym;
              const float zt = t > 15.0f ? t : __logf(fmaxf(__expf(t) - 1.0f, 1e-30f));
              zthr = zt - (1e-3f * fabsf(zt) + 1e-3f);
            }
          }
          // candidate columns, one mask word per 32-column chunk
          constexpr int kChunks = BN / 32;
          uint32_t cm[kChunks];
#pragma unroll
          for (int ci = 0; ci < kChunks; ++ci) {
            const int c0 = 32 * ci;
            uint32_t m = 0u;
            if (acc_ready && live && c0 < mma_n) {
#pragma unroll
              for (int q4 = 0; q4 < 8; ++q4) {
                const float4 z4 = *reinterpret_cast<const float4*>(zrow + c0 + 4 * q4);
                m |= (z4.x >= zthr ? 1u : 0u) << (4 * q4);
                m |= (z4.y >= zthr ? 1u : 0u) << (4 * q4 + 1);
                m |= (z4.z >= zthr ? 1u : 0u) << (4 * q4 + 2);
                m |= (z4.w >= zthr ? 1u : 0u) << (4 * q4 + 3);
              }
              if (c0 + 32 > ncols) m &= ncols - c0 >= 32 ? 0xFFFFFFFFu : ((1u << (ncols - c0)) - 1u);
            }
            cm[ci] = m;
          }
          // rounds of up to eight candidates: exact scores as (score, column)
          // keys, sorted and merged into the best eight by networks
          uint64_t best[8];
          float bw[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            best[i] = 0ull;
            bw[i] = 0.0f;
          }
          auto any_left = [&]() {
            uint32_t o = 0u;
#pragma unroll
            for (int ci = 0; ci < kChunks; ++ci) o |= cm[ci];
            return o != 0u;
          };
          while (any_left()) {
            int cb[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              // lowest set bit of the first non-empty word (selects only: the
              // words stay in registers)
              int sel = -1;
#pragma unroll
              for (int ci = kChunks - 1; ci >= 0; --ci) sel = cm[ci] != 0u ? ci : sel;
              uint32_t w = 0u;
#pragma unroll
              for (int ci = 0; ci < kChunks; ++ci) w = ci == sel ? cm[ci] : w;
              cb[q] = sel >= 0 ? 32 * sel + __ffs(w) - 1 : -1;
#pragma unroll
              for (int ci = 0; ci < kChunks; ++ci) cm[ci] = ci == sel ? (cm[ci] & (cm[ci] - 1u)) : cm[ci];
            }
            uint64_t e[8];
            float ew[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const int c = cb[q] >= 0 ? cb[q] : 0;
              const float w = router_weight(zrow[c]);
              e[q] = cb[q] >= 0 ? entry(w + bias_s[c], n0 + c) : 0ull;
              ew[q] = cb[q] >= 0 ? w : 0.0f;
            }
            sort8_pay(e, ew);
            merge_top8_pay(best, bw, e, ew);
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            tv[i] = best[i] != 0ull ? entry_score(best[i]) : -__int_as_float(0x7F800000);
            ti[i] = best[i] != 0ull ? entry_col(best[i]) : -1;
            tw[i] = best[i] != 0ull ? bw[i] : 0.0f;
          }
        } else {
          // Identity: branch-free 32-bit keys (the score key's top 24 bits |
          // 255 - local column), each 32-column chunk sorted in groups of 8
          // and merged into the running best 8; the picks then get their
          // exact scores from the stored logits (keys closer than 2^-15
          // relative may trade places at the boundary, a near-tie; equal
          // scores still go to the lower column).
          uint32_t top[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) top[i] = 0u;
          if (acc_ready) {
            for (int c0 = 0; c0 < mma_n; c0 += 32) {
              uint32_t v[32];
              tmem_ld_32x32b_x32(tmem + c0 + (static_cast<uint32_t>(quarter * 32) << 16), v);
              tmem_wait_ld();
              uint32_t key[4][8];
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const float z = __uint_as_float(v[j]) * gab;
                v[j] = __float_as_uint(z);
                if (p.logits != nullptr && live && c0 + j < ncols)
                  p.logits[static_cast<int64_t>(m0 + row) * p.N + n0 + c0 + j] = z;
                key[j >> 3][j & 7] = (live && c0 + j < ncols)
                                         ? ((float_key(z) & 0xFFFFFF00u) | (255u - static_cast<uint32_t>(c0 + j)))
                                         : 0u;
              }
#pragma unroll
              for (int g = 0; g < 4; ++g) {
                sort8_desc(key[g]);
                merge_top8(top, key[g]);
              }
              if (live) {
                const uint32_t dst = smem_addr(zrow + c0);
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4)
                  st_shared_v4(dst + 16 * q4, v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
              }
            }
          }
          // exact score of each pick, then an exact sort (score descending,
          // lower column first)
          uint64_t e[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int c = 255 - static_cast<int>(top[i] & 0xFFu);
            e[i] = top[i] != 0u ? entry(zrow[c], n0 + c) : 0ull;
          }
          sort8_desc(e);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            tv[i] = e[i] != 0ull ? entry_score(e[i]) : -__int_as_float(0x7F800000);
            ti[i] = e[i] != 0ull ? entry_col(e[i]) : -1;
            tw[i] = e[i] != 0ull ? tv[i] : 0.0f;
          }
        }
      } else {
        const bool full_list = p.k == KMAX;  // k-th score is simply the last slot
        float kth = -__int_as_float(0x7F800000);
        if (acc_ready) {
          for (int c0 = 0; c0 < mma_n; c0 += 32) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(tmem + c0 + (static_cast<uint32_t>(quarter * 32) << 16), v);
            tmem_wait_ld();
            // Logits, then activations for the whole chunk, branch-free (ILP across columns).
            float w[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float z = __uint_as_float(v[j]) * gab;
              w[j] = router ? router_weight(z) : z;
              if (p.logits != nullptr && live && c0 + j < ncols)
                p.logits[static_cast<int64_t>(m0 + row) * p.N + n0 + c0 + j] = z;
            }
            if (live) {
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                if (c0 + j < ncols) {
                  const float sc = router ? w[j] + bias_s[c0 + j] : w[j];
                  if (sc > kth) {
                    list_insert<KMAX>(tv, ti, tw, sc, n0 + c0 + j, w[j]);
                    kth = full_list ? tv[KMAX - 1] : list_kth<KMAX>(tv, p.k);
                  }
                }
              }
            }
          }
        }
      }
      if (list_barrier) cluster_wait();
      if (p.n_split == 1) {
        if (row < vr) list_store<KMAX>(p, m0 + row, tv, ti, tw);
      } else if (row < vr) {
        // push the row's list to its owner: [n slice][slot][owned row] x 16
        // bytes (consecutive rows at consecutive addresses, so the owner's
        // threads read a slot without bank conflicts)
        const int owner = row / p.ro;
        const uint32_t dst = mapa_shared(sbase + kListOff, static_cast<uint32_t>(owner)) +
                             static_cast<uint32_t>((n_idx * KMAX * p.ro + (row - owner * p.ro)) * 16);
#pragma unroll
        for (int i = 0; i < KMAX; ++i)
          st_cluster_v4(dst + i * p.ro * 16, __float_as_uint(tv[i]), static_cast<uint32_t>(ti[i]),
                        __float_as_uint(tw[i]), 0u);
      }
    }
    if (p.n_split > 1) {
      tc_fence_before();
      cluster_sync();  // every CTA's lists have arrived at their owners
      tc_fence_after();
      const int r0 = rank * p.ro;
      const int owned = min(p.ro, vr - r0);
      const int t = static_cast<int>(threadIdx.x);
      if (KMAX == 8 && t < owned) {
        // sorted lists of 8 entries, merged slice by slice (slices in column
        // order; the entry order already puts the lower column first on ties)
        const uint32_t* lists = reinterpret_cast<const uint32_t*>(smem + kListOff);
        uint64_t r[8], g[8];
        float rw[8], gw[8];
        for (int ni = 0; ni < p.n_split; ++ni) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint4 q = *reinterpret_cast<const uint4*>(lists + ((ni * 8 + i) * p.ro + t) * 4);
            const int col = static_cast<int>(q.y);
            g[i] = col >= 0 ? entry(__uint_as_float(q.x), col) : 0ull;
            gw[i] = __uint_as_float(q.z);
          }
          if (ni == 0) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              r[i] = g[i];
              rw[i] = gw[i];
            }
          } else {
            merge_top8_pay(r, rw, g, gw);
          }
        }
        float tv[KMAX], tw[KMAX];
        int ti[KMAX];
#pragma unroll
        for (int i = 0; i < KMAX; ++i) {
          tv[i] = r[i] != 0ull ? entry_score(r[i]) : -__int_as_float(0x7F800000);
          ti[i] = r[i] != 0ull ? entry_col(r[i]) : -1;
          tw[i] = r[i] != 0ull ? rw[i] : 0.0f;
        }
        list_store<KMAX>(p, m0 + r0 + t, tv, ti, tw);
      } else if (t < owned) {
        float tv[KMAX], tw[KMAX];
        int ti[KMAX];
        list_init<KMAX>(tv, ti, tw);
        float kth = -__int_as_float(0x7F800000);
        const uint32_t* lists = reinterpret_cast<const uint32_t*>(smem + kListOff);
        for (int ni = 0; ni < p.n_split; ++ni) {  // slices in column order: ties stay by lower n
#pragma unroll
          for (int i = 0; i < KMAX; ++i) {
            const uint32_t* e = lists + ((ni * KMAX + i) * p.ro + t) * 4;
            const float s = __uint_as_float(e[0]);
            if (s > kth) {
              list_insert<KMAX>(tv, ti, tw, s, static_cast<int>(e[1]), __uint_as_float(e[2]));
              kth = list_kth<KMAX>(tv, p.k);
            }
          }
        }
        list_store<KMAX>(p, m0 + r0 + t, tv, ti, tw);
      }
    }
  } else {
    // ------------------------------------------------------------ reduce epilogue
    const int rs = p.n_split * BN;  // floats per received row
    if (p.bulk) {
      cluster_wait();
      // Stage this CTA's tile row-major (stride BN + 4 floats: 16-byte rows,
      // conflict-free vector stores) in its own stage region, then send each
      // row to its owner with one bulk copy counted on the owner's barrier.
      if (warp >= 2) {
        if (p.heads) {
          // Indexer head reduction: I[t, n] = sum_h w[t, h] * ReLU(logit[t*H + h, n]).
          // Each warp folds its 32 rows (heads) per column (warp reduce-scatter:
          // lane l ends with column c0 + l), the quarters of a token are added in
          // quarter order, and the token's row of I is staged for its owner.
          float* part = reinterpret_cast<float*>(smem) + vrow_cap_floats(BN);  // [4][BN] per-quarter sums
          if (acc_ready) {  // warp-uniform
            const int tok = static_cast<int>(out0) + row / p.heads;
            const float hw = row < vr ? __ldg(p.head_w + static_cast<int64_t>(tok) * p.heads + row % p.heads) : 0.0f;
            for (int c0 = 0; c0 < mma_n; c0 += 32) {
              uint32_t v[32];
              tmem_ld_32x32b_x32(tmem + c0 + (static_cast<uint32_t>(quarter * 32) << 16), v);
              tmem_wait_ld();
              float val[32];
  #pragma unroll
              for (int j = 0; j < 32; ++j) val[j] = hw * fmaxf(__uint_as_float(v[j]) * gab, 0.0f);
              part[quarter * BN + c0 + static_cast<int>(lane)] = warp_reduce_scatter32(val);
            }
          }
          asm volatile("bar.sync 1, 128;" ::: "memory");  // the four epilogue warps
          const int qpt = p.heads / 32;  // quarters per token
          for (int i = (warp - 2) * 32 + static_cast<int>(lane); i < vrow * BN; i += 128) {
            const int t = i / BN, cc = i - t * BN;
            float acc = 0.0f;
            for (int q = t * qpt; q < (t + 1) * qpt; ++q) acc += part[q * BN + cc];
            reinterpret_cast<float*>(smem)[t * (BN + 4) + cc] = acc;
          }
          fence_proxy_async_smem();  // staged rows are read by the async (bulk copy) proxy
        } else if (acc_ready && quarter * 32 < vr) {  // warp-uniform (tcgen05.ld is collective)
          for (int c0 = 0; c0 < mma_n; c0 += 64) {  // two 32-column loads in flight
            const bool two = c0 + 32 < mma_n;       // then c0 + 64 <= BN
            uint32_t v[32], u[32];
            tmem_ld_32x32b_x32(tmem + c0 + (static_cast<uint32_t>(quarter * 32) << 16), v);
            if (two) tmem_ld_32x32b_x32(tmem + c0 + 32 + (static_cast<uint32_t>(quarter * 32) << 16), u);
            tmem_wait_ld();
            if (row < vr) {
              const uint32_t dst = sbase + static_cast<uint32_t>((row * (BN + 4) + c0) * 4);
#pragma unroll
              for (int q4 = 0; q4 < 8; ++q4)
                st_shared_v4(dst + 16 * q4, v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
              if (two) {
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4)
                  st_shared_v4(dst + 128 + 16 * q4, u[4 * q4], u[4 * q4 + 1], u[4 * q4 + 2], u[4 * q4 + 3]);
              }
            }
          }
          fence_proxy_async_smem();  // staged rows are read by the async (bulk copy) proxy
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");  // the four epilogue warps
        if (acc_ready) {
          const uint32_t bytes = static_cast<uint32_t>(((ncols + 3) & ~3) * 4);
          const uint32_t recv_local = smem_addr(rowmem);
          const uint32_t bar_local = smem_addr(&bars[3 * kMaxStages + 2]);
          for (int r = (warp - 2) + 4 * static_cast<int>(lane); r < vrow; r += 128) {  // 4 warps share few rows
            const int o = r / p.ro;
            const int rr = r - o * p.ro;
            bulk_copy_to_peer(
                mapa_shared(recv_local, static_cast<uint32_t>(o)) +
                    static_cast<uint32_t>(((k_idx * p.ro + rr) * rs + n0) * 4),
                sbase + static_cast<uint32_t>(r * (BN + 4) * 4), bytes,
                mapa_shared(bar_local, static_cast<uint32_t>(o)));
          }
          bulk_commit();
          bulk_wait_read();
        }
      }
      if (!warp_wait(smem_addr(&bars[3 * kMaxStages + 2]), 0, abort) && lane == 0)
        record_timeout(p.status, abort);
    } else {
      // Receive area too large to sit beside the pipeline: it reuses the stage
      // region, so every main loop must be over before anything is sent.
      tc_fence_before();
      cluster_sync();
      tc_fence_after();
      if (warp >= 2 && acc_ready) {  // warp-uniform: tcgen05.ld is warp-collective
        const bool live = row < vr;
        const int owner = live ? row / p.ro : 0;
        const uint32_t base =
            mapa_shared(sbase, static_cast<uint32_t>(owner)) +
            static_cast<uint32_t>(((k_idx * p.ro + (live ? row - owner * p.ro : 0)) * rs + n0) * 4);
        for (int c0 = 0; c0 < mma_n; c0 += 32) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tmem + c0 + (static_cast<uint32_t>(quarter * 32) << 16), v);
          tmem_wait_ld();
          if (live) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (c0 + j < ncols) st_cluster_f32(base + static_cast<uint32_t>((c0 + j) * 4), __uint_as_float(v[j]));
          }
        }
      }
      tc_fence_before();
      cluster_sync();  // all partial sums of this CTA's rows have arrived
      tc_fence_after();
    }
    __syncthreads();  // staged biases are visible to every warp of the row phase
    RowCtx c;
    c.recv = reinterpret_cast<float*>(p.bulk ? rowmem : smem);
    c.bias = reinterpret_cast<const float*>(rowmem + p.bias_off);
    c.ro = p.ro;
    c.rs = rs;
    c.k_split = p.k_split;
    c.gab = p.heads ? 1.0f : gab;  // head-reduced scores are final
    const int r0 = rank * p.ro;
    const int owned = min(p.ro, vrow - r0);
    if (!p.large) {
      rows_small(p, c, owned, out0 + r0);
    } else {
      uint8_t* mine = rowmem + p.recv_bytes;
      rows_large(p, c, owned, out0 + r0, reinterpret_cast<uint32_t*>(mine),
                 reinterpret_cast<uint64_t*>(mine + p.row_bytes),
                 reinterpret_cast<uint32_t*>(mine + p.row_bytes + p.cand_cap * 8));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- host side

}  // namespace

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 2-D byte matrix [rows, width] (row stride = width), boxes of box_w x box_rows,
// optional 128-byte swizzle; reads past the matrix return zeros.
bool make_map(CUtensorMap* map, const uint8_t* base, int64_t rows, int64_t width, int box_w,
              int box_rows, bool swizzle128) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(width), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(width)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_w), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

int next_pow2(int v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

struct Plan {
  int bn, kmax;
  int n_split, k_split;
  int stages;
  int direct, ro, bulk;
  uint32_t recv_bytes, bias_off;
  int rpc, heads;
  int large, cand_cap;
  uint32_t row_bytes;
  uint32_t region;
  size_t smem;
};

// Pick the split, epilogue and shared-memory layout of one problem; false if
// it cannot be laid out.
bool make_plan(int64_t M, int64_t N, int64_t K, int k, int sms, int smem_optin, int smem_one_cta,
               int max_cluster, int rpc, int heads, Plan* out) {
  Plan pl{};
  pl.rpc = rpc;
  pl.heads = heads;
  const int64_t m_tiles = (M + rpc - 1) / rpc;
  const int kt = static_cast<int>((K / 2 + BKB * kSub - 1) / (BKB * kSub));  // pipeline stages of K
  if (N <= 128) {
    pl.bn = 128;
  } else if (N <= 256 && m_tiles * 2 >= sms / 2) {
    pl.bn = 128;  // many row tiles: two 128-column halves give twice the CTAs
  } else if ((k > 32 || N > 32 * kSmallCols) && N <= 128 * max_cluster && m_tiles * 16 <= sms) {
    pl.bn = 128;  // long rows, few tiles: twice the CTAs, half the rows per CTA to select
  } else {
    pl.bn = 256;
  }
  pl.n_split = static_cast<int>((N + pl.bn - 1) / pl.bn);
  if (pl.n_split > max_cluster) return false;
  pl.k_split = 1;
  // (head reduction takes ReLU of complete logits: no K split)
  if (heads == 0 && m_tiles * pl.n_split < sms / 2) {  // few tiles: spread K over the rest of the cluster
    const int64_t want = (sms + m_tiles * pl.n_split - 1) / (m_tiles * pl.n_split);
    int ks = static_cast<int>(want < max_cluster / pl.n_split ? want : max_cluster / pl.n_split);
    if (ks > kt) ks = kt;
    pl.k_split = ks < 1 ? 1 : ks;
  }
  const int csize = pl.n_split * pl.k_split;
  // rows the epilogue owns per tile: A rows, or tokens under head reduction
  const int vr_max = static_cast<int>(M < rpc ? M : rpc) / (heads ? heads : 1);
  pl.ro = (vr_max + csize - 1) / csize;
  pl.direct = (heads == 0 && pl.k_split == 1 && k <= 32) ? 1 : 0;
  pl.kmax = k <= 8 ? 8 : (k <= 16 ? 16 : 32);
  pl.large = (!pl.direct && (k > 32 || N > 32 * kSmallCols)) ? 1 : 0;
  pl.cand_cap = pl.large ? (k <= 64 ? 64 : next_pow2(k)) : 0;  // 2 .. 32 per lane of the sort
  pl.row_bytes = pl.large ? static_cast<uint32_t>((N * 4 + 15) & ~15) : 0u;
  const int nk_max = (kt + pl.k_split - 1) / pl.k_split;
  const uint32_t sb = pl.bn == 128 ? Layout<128>::kStage : Layout<256>::kStage;
  const uint32_t recv = static_cast<uint32_t>(pl.k_split) * static_cast<uint32_t>(pl.ro) *
                        static_cast<uint32_t>(pl.n_split * pl.bn) * 4u;
  const uint32_t staging =
      heads ? static_cast<uint32_t>(vrow_cap_floats(pl.bn) + 4 * pl.bn) * 4u  // token rows + quarter sums
            : static_cast<uint32_t>(vr_max) * static_cast<uint32_t>(pl.bn + 4) * 4u;
  const int smax = pl.bn == 128 ? Layout<128>::kStagesMax : Layout<256>::kStagesMax;
  pl.stages = nk_max < smax ? nk_max : smax;
  // After the main loop the stage region holds the direct epilogue's bias
  // copies, or the reduce epilogue's staged tile (bulk) / received partials.
  auto total = [&]() {
    // direct: four bias copies, and for k <= 8 the tile's logits (BM rows of BN + 4 floats)
    // direct, N split: then the per-row lists pushed by the cluster's CTAs
    const uint32_t reuse =
        pl.direct ? 4u * static_cast<uint32_t>(pl.bn) * 4u +
                        (pl.kmax == 8 ? static_cast<uint32_t>(BM) * static_cast<uint32_t>(pl.bn + 4) * 4u : 0u) +
                        (pl.n_split > 1 ? static_cast<uint32_t>(pl.n_split * pl.ro * pl.kmax) * 16u : 0u)
                  : (pl.bulk ? staging : recv);
    uint32_t region = pl.stages * sb > reuse ? pl.stages * sb : reuse;
    region = (region + 1023u) & ~1023u;
    pl.region = region;
    pl.recv_bytes = (!pl.direct && pl.bulk) ? recv : 0u;
    size_t extra = pl.recv_bytes;
    if (pl.large)
      extra += pl.row_bytes + static_cast<size_t>(pl.cand_cap) * 8 + 256;  // keys, candidates, block scratch
    pl.bias_off = static_cast<uint32_t>(extra);
    extra += pl.direct ? static_cast<size_t>(pl.bn) * 4 : static_cast<size_t>((N * 4 + 15) & ~15);  // staged biases
    return 1024 + static_cast<size_t>(region) + kCtrlBytes + extra;
  };
  pl.bulk = pl.direct ? 0 : 1;
  while (pl.bulk && total() > static_cast<size_t>(smem_optin) && pl.stages > 1) --pl.stages;
  if (pl.bulk && total() > static_cast<size_t>(smem_optin)) {  // receive in the stage region
    pl.bulk = 0;
    pl.stages = nk_max < smax ? nk_max : smax;
  }
  while (total() > static_cast<size_t>(smem_optin) && pl.stages > 1) --pl.stages;
  pl.smem = total();
  if (pl.smem > static_cast<size_t>(smem_optin)) return false;
  // Every CTA allocates all of tensor memory: keep two CTAs off one SM by
  // asking for more than half of the SM's shared memory.
  if (pl.smem < static_cast<size_t>(smem_one_cta)) pl.smem = static_cast<size_t>(smem_one_cta);
  if (pl.smem > static_cast<size_t>(smem_optin)) return false;
  if (heads && !pl.bulk) return false;  // head reduction stages token rows for bulk copies
  *out = pl;
  return true;
}

template <int BN, int KMAX>
cudaLaunchConfig_t launch_config(int grid, int cluster, size_t smem, cudaStream_t stream,
                                 cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // set-up (barriers, TMEM) may overlap the previous kernel; every thread
  // waits for it (pdl_wait) before touching global memory
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

// Function attributes the launch needs (idempotent).
template <int BN, int KMAX>
cudaError_t configure(size_t smem, int cluster) {
  auto kern = gemm_topk_kernel<BN, KMAX>;
  static std::mutex mu;
  static int configured = 0;  // largest dynamic smem size set so far for this variant
  static bool nonportable = false;
  std::lock_guard<std::mutex> lock(mu);
  if (static_cast<int>(smem) > configured) {
    const cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured = static_cast<int>(smem);
  }
  if (cluster > 8 && !nonportable) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    nonportable = true;
  }
  return cudaSuccess;
}

// Whether clusters of this size and shared-memory footprint can be resident
// at all (answers cached per device and configuration).
template <int BN, int KMAX>
int active_clusters(int cluster, size_t smem) {
  static std::mutex mu;
  static int cache_dev[64], cache_cluster[64];
  static size_t cache_smem[64];
  static int cache_ok[64];
  static int n_cache = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_cache; ++i)
    if (cache_dev[i] == dev && cache_cluster[i] == cluster && cache_smem[i] == smem) return cache_ok[i];
  int ok = 0;
  // Every CTA takes all of tensor memory, so a second CTA on one SM would
  // wait in its allocation: a footprint that lets two share an SM is refused.
  int per_sm = 0;
  if (configure<BN, KMAX>(smem, cluster) == cudaSuccess &&
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemm_topk_kernel<BN, KMAX>, kThreads, smem) ==
          cudaSuccess &&
      per_sm == 1) {
    if (cluster <= 1) {
      ok = sm_count();
    } else {
      cudaLaunchAttribute attr[2];
      cudaLaunchConfig_t cfg = launch_config<BN, KMAX>(cluster, cluster, smem, nullptr, attr);
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, gemm_topk_kernel<BN, KMAX>, &cfg) == cudaSuccess && n > 0) ok = n;
    }
  }
  cudaGetLastError();  // a refused query leaves no error behind
  if (n_cache < 64) {
    cache_dev[n_cache] = dev;
    cache_cluster[n_cache] = cluster;
    cache_smem[n_cache] = smem;
    cache_ok[n_cache] = ok;
    ++n_cache;
  }
  return ok;
}

template <int BN, int KMAX>
cudaError_t launch_variant(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& msa,
                           const CUtensorMap& msb, const Params& p, int grid, int cluster,
                           size_t smem, cudaStream_t stream) {
  const cudaError_t e = configure<BN, KMAX>(smem, cluster);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = launch_config<BN, KMAX>(grid, cluster, smem, stream, attr);
  count_launch();
  return cudaLaunchKernelEx(&cfg, gemm_topk_kernel<BN, KMAX>, ma, mb, msa, msb, p);
}

// Clusters of this plan that can be resident at once (0: none fits).
int active(const Plan& pl) {
  const int c = pl.n_split * pl.k_split;
  if (pl.bn == 128) {
    if (pl.kmax == 8) return active_clusters<128, 8>(c, pl.smem);
    if (pl.kmax == 16) return active_clusters<128, 16>(c, pl.smem);
    return active_clusters<128, 32>(c, pl.smem);
  }
  if (pl.kmax == 8) return active_clusters<256, 8>(c, pl.smem);
  if (pl.kmax == 16) return active_clusters<256, 16>(c, pl.smem);
  return active_clusters<256, 32>(c, pl.smem);
}

cudaError_t launch(const Plan& pl, const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& msa,
                   const CUtensorMap& msb, const Params& p, int grid, cudaStream_t stream) {
  const int c = pl.n_split * pl.k_split;
  if (pl.bn == 128) {
    if (pl.kmax == 8) return launch_variant<128, 8>(ma, mb, msa, msb, p, grid, c, pl.smem, stream);
    if (pl.kmax == 16) return launch_variant<128, 16>(ma, mb, msa, msb, p, grid, c, pl.smem, stream);
    return launch_variant<128, 32>(ma, mb, msa, msb, p, grid, c, pl.smem, stream);
  }
  if (pl.kmax == 8) return launch_variant<256, 8>(ma, mb, msa, msb, p, grid, c, pl.smem, stream);
  if (pl.kmax == 16) return launch_variant<256, 16>(ma, mb, msa, msb, p, grid, c, pl.smem, stream);
  return launch_variant<256, 32>(ma, mb, msa, msb, p, grid, c, pl.smem, stream);
}

}  // namespace

int launch_gemm_topk(const GemmTopkArgs& a, cudaStream_t stream, cudaError_t* err) {
  *err = cudaSuccess;
  if (a.M == 0) return NVFP4_OK;
  int dev = 0;
  cudaGetDevice(&dev);
  int smem_optin = 0, smem_sm = 0, smem_reserved = 0;
  cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  cudaDeviceGetAttribute(&smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
  // the least dynamic shared memory that leaves no room for a second CTA
  const int smem_one_cta = smem_sm / 2 - smem_reserved + 1;
  // Scales by TMA when their rows and base are 16-byte aligned.
  const bool sf_tma = a.K % 256 == 0 && reinterpret_cast<uintptr_t>(a.sfa) % 16 == 0 &&
                      reinterpret_cast<uintptr_t>(a.sfb) % 16 == 0;
  // Largest cluster (16, else 8, 4, ...) whose CTAs can be co-resident.
  Plan pl;
  int cap = kMaxCluster;
  for (;;) {
    if (!make_plan(a.M, a.N, a.K, a.k, sm_count(), smem_optin, smem_one_cta, cap, BM, a.heads, &pl))
      return NVFP4_ERR_UNSUPPORTED;
    if (active(pl) > 0) break;
    const int c = pl.n_split * pl.k_split;
    if (c <= 1 || cap <= 1) return NVFP4_ERR_UNSUPPORTED;
    cap = c / 2;
  }
  if (pl.large) {
    // Row selection dominates: spread the rows over every cluster that can
    // be resident (fewer rows per tile, so fewer rows per owning CTA).
    const int n_active = active(pl);
    const int64_t unit = a.heads ? a.heads : 1;  // tiles hold whole tokens under head reduction
    int64_t rpc = n_active > 0 ? (a.M + n_active - 1) / n_active : BM;
    rpc = (rpc + unit - 1) / unit * unit;
    Plan spread;
    if (rpc < BM &&
        make_plan(a.M, a.N, a.K, a.k, sm_count(), smem_optin, smem_one_cta, cap, static_cast<int>(rpc), a.heads,
                  &spread) &&
        spread.n_split == pl.n_split && spread.k_split == pl.k_split && active(spread) > 0)
      pl = spread;
  }

  CUtensorMap ma, mb, msa, msb;
  if (!make_map(&ma, a.qa, a.M, a.K / 2, BKB, BM, true) ||
      !make_map(&mb, a.qb, a.N, a.K / 2, BKB, pl.bn, true))
    return NVFP4_ERR_UNSUPPORTED;
  if (sf_tma) {
    if (!make_map(&msa, a.sfa, a.M, a.K / 16, 16 * kSub, BM, false) ||
        !make_map(&msb, a.sfb, a.N, a.K / 16, 16 * kSub, pl.bn, false))
      return NVFP4_ERR_UNSUPPORTED;
  } else {
    msa = ma;  // not read
    msb = mb;
  }
  Params p;
  std::memset(&p, 0, sizeof(p));
  p.sfa = a.sfa;
  p.sfb = a.sfb;
  p.gsa = a.gsa;
  p.gsb = a.gsb;
  p.bias = a.bias;
  p.topk_idx = a.topk_idx;
  p.topk_score = a.topk_score;
  p.topk_weight = a.topk_weight;
  p.logits = a.logits;
  p.status = &a.ws->status;
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.k = a.k;
  p.epilogue = a.epilogue;
  p.num_k_tiles = static_cast<int>((a.K / 2 + BKB * kSub - 1) / (BKB * kSub));  // pipeline stages of K
  p.n_split = pl.n_split;
  p.k_split = pl.k_split;
  p.stages = pl.stages;
  p.sf_tma = sf_tma ? 1 : 0;
  p.region_bytes = pl.region;
  p.direct = pl.direct;
  p.ro = pl.ro;
  p.bulk = pl.bulk;
  p.recv_bytes = pl.recv_bytes;
  p.bias_off = pl.bias_off;
  p.rpc = pl.rpc;
  p.heads = a.heads;
  p.head_w = a.head_w;
  p.large = pl.large;
  p.cand_cap = pl.cand_cap;
  p.row_bytes = pl.row_bytes;
  {
    const auto a16 = [](const void* q) { return q == nullptr || reinterpret_cast<uintptr_t>(q) % 16 == 0; };
    p.vec_out = (a.k == 8 && a16(a.topk_idx) && a16(a.topk_score) && a16(a.topk_weight)) ? 1 : 0;
  }
  const int grid = static_cast<int>((a.M + pl.rpc - 1) / pl.rpc) * pl.n_split * pl.k_split;
  const cudaError_t e = launch(pl, ma, mb, msa, msb, p, grid, stream);
  if (e != cudaSuccess) {
    *err = e;
    return NVFP4_ERR_CUDA;
  }
  return NVFP4_OK;
}

}  // namespace nvfp4
