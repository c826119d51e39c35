// NVFP4 block-scaled GEMM with a fused scoring epilogue and per-row top-k,
// for sm_103a (tcgen05 tensor cores, tensor memory, TMA).
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
// The FP32 logits never go to global memory (unless a debug buffer is given).
//
// Structure (one CTA per 128-row tile of A, 6 warps):
//   warp 0     producer: TMA loads of the A and B code tiles (128-byte rows,
//              128-byte swizzle) and cp.async of the E4M3 scale words, which
//              it scatters straight into the layout tcgen05.cp expects;
//              multi-stage ring of shared-memory buffers with mbarriers.
//   warp 1     MMA issuer (one thread): per stage, tcgen05.cp of the scale
//              factors into tensor memory, then four 128x128x64
//              kind::mxf4nvf4 block-scaled MMAs into a TMEM accumulator.
//              Two accumulators alternate over the N tiles, so the epilogue
//              of one tile overlaps the main loop of the next.
//   warps 2-5  epilogue: tcgen05.ld of the accumulator (thread = row),
//              scale by gsa*gsb, activation + bias, and either a register
//              top-k per thread (k <= 32), or scores kept in shared memory for
//              a few rows followed by a warp-level radix select + bitonic sort
//              (k > 32, e.g. the indexer's top-512).
//
// The design of the pages' WIP fused router kernel (TMA warp, MMA warp, four
// epilogue warps with per-thread heaps) is prior art; the tile sizes, the
// scale-factor path and the selection scheme here are this library's own.
//
// Every wait on an mbarrier is bounded: after ~1 s of SM clock it records
// NVFP4_DEVICE_TIMEOUT in the workspace, tells the other warps to stop, lets
// the copies already issued land, frees tensor memory and returns.

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

constexpr int BM = 128;                  // MMA M: rows of A per tile
constexpr int BN = 128;                  // MMA N: rows of B (output columns) per tile
constexpr int BKB = 128;                 // bytes of a K tile per row = 256 FP4 elements
constexpr int kThreads = 192;            // 6 warps
constexpr uint32_t kABytes = BM * BKB;   // 16 KB
constexpr uint32_t kBBytes = BN * BKB;   // 16 KB
constexpr uint32_t kSfChunk = 512;       // scales of 128 rows for one MMA (K = 64)
constexpr uint32_t kSfBytes = 4 * kSfChunk;
constexpr uint32_t kStageBytes = kABytes + kBBytes + 2 * kSfBytes;  // 36 KB, 1 KB multiple
constexpr int kMaxStages = 4;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = BN;                  // FP32 accumulator: one column per n
constexpr uint32_t kSfTmemBase = 2 * kAccCols;     // after the two accumulators
constexpr uint32_t kSfTmemPerStage = 32;           // 16 columns SFA + 16 columns SFB
constexpr uint32_t kCtrlBytes = 256;
constexpr long long kWaitLimit = 2000000000LL;     // SM cycles (~1 s)

static_assert(kSfTmemBase + kMaxStages * kSfTmemPerStage <= kTmemCols, "TMEM budget");

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
  int num_n_tiles;
  int stages;
  int rows_per_cta;  // select mode: rows whose scores this CTA keeps
  int cand_cap;      // select mode: power of two >= k
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

__device__ __forceinline__ void record_timeout(const Params& p, volatile uint32_t* abort) {
  *abort = 1u;
  atomicOr(p.status, NVFP4_DEVICE_TIMEOUT);
}

// Order-preserving map of a float to an unsigned key (larger float, larger key).
__device__ __forceinline__ uint32_t float_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

__device__ __forceinline__ void score_of(float logit, int epilogue, const float* bias, int n,
                                         float& score, float& weight) {
  if (epilogue == NVFP4_EPILOGUE_SQRT_SOFTPLUS_BIAS) {
    const float sp = logit > 20.0f ? logit : log1pf(expf(logit));
    weight = sqrtf(sp);
    score = weight + __ldg(bias + n);
  } else {
    weight = logit;
    score = logit;
  }
}

// Sorted (descending) insertion into a KMAX-entry register list; equal
// scores keep the earlier (lower) column ahead.
template <int KMAX>
__device__ __forceinline__ void topk_insert(float (&tv)[KMAX], int (&ti)[KMAX], float (&tw)[KMAX],
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

template <int KMAX>
__device__ __forceinline__ float kth_value(const float (&tv)[KMAX], int k) {
  float t = tv[0];
#pragma unroll
  for (int i = 1; i < KMAX; ++i)
    if (i == k - 1) t = tv[i];
  return t;
}

// Warp-level top-k of n scores held in shared memory (overwritten by their
// keys): 4-pass radix select of the k-th largest key, in-order compaction
// (keys above it, then the lowest-index ties), bitonic sort of the picks.
__device__ void select_row_topk(float* row_scores, int n, int k, uint32_t* hist, uint64_t* cand,
                                int cand_cap, const Params& p, int64_t row) {
  const uint32_t lane = lane_id();
  uint32_t* keys = reinterpret_cast<uint32_t*>(row_scores);
  for (int i = lane; i < n; i += 32) keys[i] = float_key(row_scores[i]);
  __syncwarp();
  const int want = k < n ? k : n;
  uint32_t prefix = 0, pmask = 0;
  int remaining = want;
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = lane; i < 256; i += 32) hist[i] = 0;
    __syncwarp();
    for (int i = lane; i < n; i += 32) {
      const uint32_t u = keys[i];
      if ((u & pmask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1u);
    }
    __syncwarp();
    // lane l owns digits 255-8l down to 248-8l
    uint32_t c[8];
    uint32_t local = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      c[j] = hist[255 - 8 * lane - j];
      local += c[j];
    }
    uint32_t incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= static_cast<uint32_t>(o)) incl += t;
    }
    const uint32_t excl = incl - local;
    const bool mine = excl < static_cast<uint32_t>(remaining) && incl >= static_cast<uint32_t>(remaining);
    uint32_t digit = 0, above = 0;
    if (mine) {
      uint32_t acc = excl;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (acc + c[j] >= static_cast<uint32_t>(remaining)) {
          digit = 255 - 8 * lane - j;
          above = acc;
          break;
        }
        acc += c[j];
      }
    }
    const uint32_t owner = __ffs(__ballot_sync(0xFFFFFFFFu, mine)) - 1;
    digit = __shfl_sync(0xFFFFFFFFu, digit, owner);
    above = __shfl_sync(0xFFFFFFFFu, above, owner);
    remaining -= static_cast<int>(above);
    prefix |= digit << shift;
    pmask |= 255u << shift;
    __syncwarp();
  }
  const uint32_t kth = prefix;
  const int need_eq = remaining;
  int out = 0, eq_seen = 0;
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int base = 0; base < n; base += 32) {
    const int i = base + static_cast<int>(lane);
    const uint32_t u = i < n ? keys[i] : 0u;
    const bool gt = i < n && u > kth;
    const bool eq = i < n && u == kth;
    const uint32_t beq = __ballot_sync(0xFFFFFFFFu, eq);
    const int eq_rank = eq_seen + __popc(beq & lt_mask);
    const bool take = gt || (eq && eq_rank < need_eq);
    const uint32_t btake = __ballot_sync(0xFFFFFFFFu, take);
    if (take)
      cand[out + __popc(btake & lt_mask)] =
          (static_cast<uint64_t>(u) << 32) | static_cast<uint32_t>(0xFFFFFFFFu - static_cast<uint32_t>(i));
    out += __popc(btake);
    eq_seen += __popc(beq);
  }
  for (int i = out + static_cast<int>(lane); i < cand_cap; i += 32) cand[i] = 0ull;
  __syncwarp();
  // Bitonic sort, descending on (key, -index).
  for (int size = 2; size <= cand_cap; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = lane; t < cand_cap / 2; t += 32) {
        const int lo = 2 * stride * (t / stride) + (t % stride);
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const uint64_t a = cand[lo], b = cand[hi];
        if ((a < b) == desc) {
          cand[lo] = b;
          cand[hi] = a;
        }
      }
      __syncwarp();
    }
  }
  for (int t = lane; t < k; t += 32) {
    int32_t idx = -1;
    float s = -__int_as_float(0x7F800000);
    float w = 0.0f;
    if (t < out) {
      const uint64_t v = cand[t];
      idx = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(v & 0xFFFFFFFFu));
      s = key_float(static_cast<uint32_t>(v >> 32));
      w = (p.epilogue == NVFP4_EPILOGUE_SQRT_SOFTPLUS_BIAS) ? s - __ldg(p.bias + idx) : s;
    }
    p.topk_idx[row * p.k + t] = idx;
    p.topk_score[row * p.k + t] = s;
    if (p.topk_weight) p.topk_weight[row * p.k + t] = w;
  }
  __syncwarp();
}

// Shared-memory bytes of the per-row score buffers in select mode (16-byte rounded).
__host__ __device__ inline size_t select_scores_bytes(int rows, int n) {
  return (static_cast<size_t>(rows) * n * 4 + 15) & ~static_cast<size_t>(15);
}

template <int KMAX, bool SELECT>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_topk_kernel(const __grid_constant__ CUtensorMap tma_a,
                     const __grid_constant__ CUtensorMap tma_b, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();
  const int S = p.stages;
  uint8_t* ctrl = smem + S * kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(ctrl);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 128);
  volatile uint32_t* abort = reinterpret_cast<volatile uint32_t*>(ctrl + 132);
  auto full_bar = [&](int s) { return smem_addr(&bars[s]); };
  auto empty_bar = [&](int s) { return smem_addr(&bars[kMaxStages + s]); };
  auto tfull_bar = [&](int b) { return smem_addr(&bars[2 * kMaxStages + b]); };
  auto tempty_bar = [&](int b) { return smem_addr(&bars[2 * kMaxStages + 2 + b]); };
  const uint32_t drain_bar = smem_addr(&bars[2 * kMaxStages + 4]);

  int m0, row_lo, row_hi;
  if (SELECT) {
    row_lo = blockIdx.x * p.rows_per_cta;
    row_hi = min(row_lo + p.rows_per_cta, p.M);
    m0 = (row_lo / BM) * BM;
  } else {
    m0 = blockIdx.x * BM;
    row_lo = m0;
    row_hi = min(m0 + BM, p.M);
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1 + 32);  // expect_tx arrival + one cp.async arrival per lane
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 4);
    }
    mbar_init(drain_bar, 1);
    *abort = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tma_a);
    prefetch_tensormap(&tma_b);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const int kk = lane & 3;        // which MMA (K = 64) of the tile this lane's scale words feed
    const int rsub = lane >> 2;     // row offset 0..7 within each group of 8 rows
    const int kwords = p.K / 64;    // 4-byte scale words per row
    const int sf_ld = p.K / 16;     // scale bytes per row
    int issued_phase[kMaxStages];
    bool issued[kMaxStages];
    for (int s = 0; s < kMaxStages; ++s) issued[s] = false, issued_phase[s] = 0;
    int it = 0;
    bool ok = true;
    for (int nt = 0; nt < p.num_n_tiles && ok; ++nt) {
      const int n0 = nt * BN;
      for (int kt = 0; kt < p.num_k_tiles; ++kt, ++it) {
        const int s = it % S;
        const uint32_t ph = (it / S) & 1;
        if (!warp_wait(empty_bar(s), ph ^ 1u, abort)) {
          if (lane == 0) record_timeout(p, abort);
          ok = false;
          break;
        }
        uint8_t* st = smem + s * kStageBytes;
        const uint32_t a_dst = smem_addr(st);
        const uint32_t b_dst = a_dst + kABytes;
        const uint32_t sfa_dst = b_dst + kBBytes + kk * kSfChunk;
        const uint32_t sfb_dst = sfa_dst + kSfBytes;
        if (lane == 0) {
          mbar_arrive_expect_tx(full_bar(s), kABytes + kBBytes);
          tma_load_2d(a_dst, &tma_a, full_bar(s), kt * BKB, m0);
          tma_load_2d(b_dst, &tma_b, full_bar(s), kt * BKB, n0);
        }
        // Scale word (row r, MMA kk) goes to byte (r % 32) * 16 + (r / 32) * 4
        // of chunk kk: the 32 x 128-bit matrix that tcgen05.cp 32x128b.warpx4
        // turns into the per-row scale columns of one MMA.
        const int kw = kt * 4 + kk;
        const bool kvalid = kw < kwords;
#pragma unroll 4
        for (int j = 0; j < 16; ++j) {
          const int r = rsub + 8 * j;
          const uint32_t off = (r & 31) * 16 + (r >> 5) * 4;
          const int ra = m0 + r;
          const bool va = kvalid && ra < p.M;
          cp_async_4(sfa_dst + off, va ? p.sfa + static_cast<int64_t>(ra) * sf_ld + kw * 4 : p.sfa,
                     va ? 4u : 0u);
          const int rb = n0 + r;
          const bool vb = kvalid && rb < p.N;
          cp_async_4(sfb_dst + off, vb ? p.sfb + static_cast<int64_t>(rb) * sf_ld + kw * 4 : p.sfb,
                     vb ? 4u : 0u);
        }
        cp_async_arrive_noinc(full_bar(s));
        issued[s] = true;
        issued_phase[s] = ph;
      }
    }
    // Let every copy this warp issued land before the CTA can exit.
    if (lane == 0) {
      uint32_t never = 0;
      for (int s = 0; s < S; ++s)
        if (issued[s] && !mbar_wait_bounded(full_bar(s), issued_phase[s], &never, kWaitLimit))
          record_timeout(p, abort);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc = make_idesc(BM, BN);
    int it = 0;
    bool ok = true;
    for (int nt = 0; nt < p.num_n_tiles && ok; ++nt) {
      const int buf = nt & 1;
      const uint32_t acc = tmem + buf * kAccCols;
      if (nt >= 2 && !warp_wait(tempty_bar(buf), ((nt >> 1) + 1) & 1u, abort)) {
        if (lane == 0) record_timeout(p, abort);
        break;
      }
      tc_fence_after();
      for (int kt = 0; kt < p.num_k_tiles; ++kt, ++it) {
        const int s = it % S;
        const uint32_t ph = (it / S) & 1;
        if (!warp_wait(full_bar(s), ph, abort)) {
          if (lane == 0) record_timeout(p, abort);
          ok = false;
          break;
        }
        if (lane == 0) {
          fence_proxy_async_smem();  // scale words arrived through cp.async (generic proxy)
          tc_fence_after();
          const uint32_t a_addr = smem_addr(smem + s * kStageBytes);
          const uint32_t b_addr = a_addr + kABytes;
          const uint32_t sfa_addr = b_addr + kBBytes;
          const uint32_t sfb_addr = sfa_addr + kSfBytes;
          const uint32_t sf_col = tmem + kSfTmemBase + s * kSfTmemPerStage;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            tc_cp_32x128b_warpx4(sf_col + kk * 4, smem_desc(sfa_addr + kk * kSfChunk, 0, 128, 0));
            tc_cp_32x128b_warpx4(sf_col + 16 + kk * 4, smem_desc(sfb_addr + kk * kSfChunk, 0, 128, 0));
          }
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = smem_desc(a_addr + kk * 32, 16, 1024, 2);
            const uint64_t bd = smem_desc(b_addr + kk * 32, 16, 1024, 2);
            tc_mma_nvf4(acc, ad, bd, idesc, sf_col + kk * 4, sf_col + 16 + kk * 4,
                        (kt | kk) != 0 ? 1u : 0u);
          }
          tc_commit(empty_bar(s));  // frees the stage once these MMAs have read it
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) tc_commit(tfull_bar(buf));
      __syncwarp();
    }
    if (lane == 0) {
      uint32_t never = 0;
      tc_commit(drain_bar);
      if (!mbar_wait_bounded(drain_bar, 0, &never, kWaitLimit)) record_timeout(p, abort);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;               // TMEM lanes 32*quarter .. +31
    const int row = m0 + quarter * 32 + static_cast<int>(lane);
    const float gab = __ldg(p.gsa) * __ldg(p.gsb);
    float* scores = reinterpret_cast<float*>(ctrl + kCtrlBytes);
    const bool keep = SELECT ? (row >= row_lo && row < row_hi) : (row < p.M);
    float tv[KMAX];
    int ti[KMAX];
    float tw[KMAX];
#pragma unroll
    for (int i = 0; i < KMAX; ++i) {
      tv[i] = -__int_as_float(0x7F800000);
      ti[i] = -1;
      tw[i] = 0.0f;
    }
    float thr = tv[0];
    bool ok = true;
    for (int nt = 0; nt < p.num_n_tiles; ++nt) {
      const int buf = nt & 1;
      if (!warp_wait(tfull_bar(buf), (nt >> 1) & 1u, abort)) {
        if (lane == 0) record_timeout(p, abort);
        ok = false;
        break;
      }
      tc_fence_after();
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem + buf * kAccCols + c * 32 + (static_cast<uint32_t>(quarter * 32) << 16), r);
        tmem_wait_ld();
        const int nbase = nt * BN + c * 32;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int n = nbase + j;
          if (n < p.N) {
            const float logit = __uint_as_float(r[j]) * gab;
            if (p.logits != nullptr && keep) p.logits[static_cast<int64_t>(row) * p.N + n] = logit;
            float s, w;
            score_of(logit, p.epilogue, p.bias, n, s, w);
            if (SELECT) {
              if (keep) scores[(row - row_lo) * p.N + n] = s;
            } else if (s > thr) {
              topk_insert<KMAX>(tv, ti, tw, s, n, w);
              thr = kth_value<KMAX>(tv, p.k);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(buf));
    }
    if (!SELECT) {
      if (ok && keep) {
        const int64_t o = static_cast<int64_t>(row) * p.k;
#pragma unroll
        for (int i = 0; i < KMAX; ++i) {
          if (i < p.k) {
            p.topk_idx[o + i] = ti[i];
            p.topk_score[o + i] = tv[i];
            if (p.topk_weight) p.topk_weight[o + i] = tw[i];
          }
        }
      }
    } else {
      asm volatile("bar.sync 1, 128;" ::: "memory");  // the four epilogue warps
      if (ok && !*abort) {
        const int ew = warp - 2;
        uint8_t* sel = ctrl + kCtrlBytes + select_scores_bytes(p.rows_per_cta, p.N);
        uint32_t* hist = reinterpret_cast<uint32_t*>(sel) + ew * 256;
        uint64_t* cand = reinterpret_cast<uint64_t*>(sel + 4 * 256 * 4) + static_cast<size_t>(ew) * p.cand_cap;
        for (int rr = ew; rr < row_hi - row_lo; rr += 4)
          select_row_topk(scores + static_cast<size_t>(rr) * p.N, p.N, p.k, hist, cand, p.cand_cap, p,
                          row_lo + rr);
      }
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

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

// 2-D map over a [rows, K/2]-byte code matrix, boxes of 128 bytes x box_rows
// rows with the 128-byte swizzle; reads past the matrix return zeros.
bool make_code_map(CUtensorMap* map, const uint8_t* base, int64_t rows, int64_t K, int box_rows) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(BKB), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int KMAX, bool SELECT>
cudaError_t launch_variant(const CUtensorMap& ma, const CUtensorMap& mb, const Params& p, int grid,
                           size_t smem, cudaStream_t stream) {
  auto kern = gemm_topk_kernel<KMAX, SELECT>;
  static int configured = 0;  // largest dynamic smem size set so far for this variant
  if (static_cast<int>(smem) > configured) {
    const cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured = static_cast<int>(smem);
  }
  kern<<<grid, kThreads, smem, stream>>>(ma, mb, p);
  return cudaGetLastError();
}

int next_pow2(int v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

}  // namespace

int launch_gemm_topk(const GemmTopkArgs& a, cudaStream_t stream, cudaError_t* err) {
  *err = cudaSuccess;
  if (a.M == 0) return NVFP4_OK;
  CUtensorMap ma, mb;
  if (!make_code_map(&ma, a.qa, a.M, a.K, BM) || !make_code_map(&mb, a.qb, a.N, a.K, BN))
    return NVFP4_ERR_UNSUPPORTED;
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
  p.num_k_tiles = static_cast<int>((a.K / 2 + BKB - 1) / BKB);
  p.num_n_tiles = static_cast<int>((a.N + BN - 1) / BN);

  int dev = 0;
  cudaGetDevice(&dev);
  int smem_optin = 0;
  cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  const size_t fixed = 1024 + kCtrlBytes;
  cudaError_t e = cudaSuccess;

  if (a.k <= 32) {
    p.stages = kMaxStages;
    const size_t smem = fixed + p.stages * kStageBytes;
    const int grid = static_cast<int>((a.M + BM - 1) / BM);
    if (a.k <= 8)
      e = launch_variant<8, false>(ma, mb, p, grid, smem, stream);
    else if (a.k <= 16)
      e = launch_variant<16, false>(ma, mb, p, grid, smem, stream);
    else
      e = launch_variant<32, false>(ma, mb, p, grid, smem, stream);
  } else {
    p.cand_cap = next_pow2(a.k);
    const size_t sel_bytes = 4 * 256 * 4 + 4 * static_cast<size_t>(p.cand_cap) * 8;
    // Fewer pipeline stages and as many rows as fit, at most 8 per CTA.
    int stages = 2, rows = 8;
    auto need = [&](int st, int r) {
      return fixed + st * kStageBytes + select_scores_bytes(r, static_cast<int>(a.N)) + sel_bytes;
    };
    while (rows > 1 && need(stages, rows) > static_cast<size_t>(smem_optin)) rows >>= 1;
    if (need(stages, rows) > static_cast<size_t>(smem_optin)) return NVFP4_ERR_UNSUPPORTED;
    while (stages < kMaxStages && need(stages + 1, rows) <= static_cast<size_t>(smem_optin)) ++stages;
    p.stages = stages;
    p.rows_per_cta = rows;
    const int grid = static_cast<int>((a.M + rows - 1) / rows);
    e = launch_variant<1, true>(ma, mb, p, grid, need(stages, rows), stream);
  }
  if (e != cudaSuccess) {
    *err = e;
    return NVFP4_ERR_CUDA;
  }
  return NVFP4_OK;
}

}  // namespace nvfp4
