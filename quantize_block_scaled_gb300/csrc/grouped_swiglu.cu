// Grouped NVFP4 block-scaled GEMM with a fused SwiGLU epilogue (the MoE
// first projection) for sm_103a: tcgen05 tensor cores with TMEM
// accumulators, TMA tile loads, one persistent CTA per SM.
//
// What it computes (compare view of the nvfp4-megamoe-kernel pages: the MoE
// kernel notes, "FusedSwiGLUScaledGroupedGemmKernel" — L1 weights with gate
// and up interleaved at granularity 8, SwiGLU and clamp applied between the
// TMEM read and the store; the model notes, "SwiGLU activation with
// swiglu_limit=10.0"; PERFORMANCE_AUDIT.md P1 — the fused kernel writes
// [silu(gate), silu(gate)*up] interleaved at the weights' granularity):
//
//   group e owns A rows offs[e] .. offs[e+1]-1 and the weight rows
//   e*2I .. e*2I + 2I - 1 of B (gate and up rows in alternating runs of g)
//   logit[m, n] = gsa * gsb[e] * sum_k A[m, k] B[e*2I + n, k]
//   a_j = silu(min(gate_j, limit)),  h_j = a_j * min(max(up_j, -limit), limit)
//   layout 0: out[m, j] = bf16(h_j)                              [M, I]
//   layout 1: out[m, n] = bf16(a or h), gate columns a, up columns h  [M, 2I]
// The logits never reach global memory.
//
// Work split.  A work item is one 128-row tile of one group times one
// 256-row slice of that group's weights (128 gate and 128 up columns).  The
// group offsets live on the device (the router writes them), so the CTAs
// derive the item list themselves: one warp of each scans the offsets into
// per-group tile starts in shared memory.  Items are dealt round-robin
// with the weight slice varying fastest, so the CTAs that work at the same
// time share each A tile through L2 and the row tiles of one group share its
// weight slices.
//
// Per CTA, 6 warps:
//   warp 0     producer: TMA loads of the A and B code tiles (128-byte rows,
//              128-byte swizzle) and the row-major E4M3 scale boxes into a
//              ring of 4 stages of 54 KB (3 when the group tables of more than
//              ~830 groups need the room) that runs on across work items.
//              The scale boxes complete on a barrier of their own, so their
//              rearrangement and copy into TMEM overlap the landing of the
//              code tiles; A comes in 32-row boxes, only those holding the
//              item's rows.
//   warp 1     MMA issuer (one thread): four 128 x 256 x 64 kind::mxf4nvf4
//              block-scaled MMAs per stage into one TMEM accumulator; before
//              the first MMA of an item it waits until the epilogue has read
//              the previous item's accumulator.
//   warps 2-5  rearrange each stage's scale boxes in place into the layout
//              tcgen05.cp reads (all four read, a named barrier, then each
//              writes the chunk of its MMA step) and copy them into TMEM;
//              after an item's last stage they are its epilogue: the thread
//              owning TMEM lane r reads row r 32 columns at a time (two
//              chunks in flight), scales by gsa * gsb[e], applies the clamp
//              and SwiGLU in registers and stores bf16 straight to global
//              memory (rows past the group's end are not stored).
//
// Every wait is bounded (~1 s of SM clock): on expiry the kernel records
// NVFP4_DEVICE_TIMEOUT in the workspace, stops the CTA's other warps, lets
// its issued copies land, frees TMEM and returns.  Offsets that break the
// contract (decreasing, outside [0, M]) are clamped, never dereferenced out
// of range, and flagged with NVFP4_DEVICE_BAD_GROUPS.

#include <cuda.h>

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
constexpr int BN = 256;              // MMA N: weight rows per slice
constexpr int BKB = 128;             // bytes of a K tile per row = 256 FP4 elements
constexpr int kThreads = 192;
constexpr int kMaxStages = 4;        // 4 when the group tables leave room, else 3
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfTmemBase = 256;  // scale factors after the 256-column accumulator
constexpr uint32_t kSfChunk = 512;     // scales of 128 rows for one MMA (K = 64)
constexpr uint32_t kCtrlBytes = 256;  // barriers, then the TMEM address at byte 192
constexpr long long kWaitLimit = 2000000000LL;  // SM cycles (~1 s)

// Stage layout: A codes, B codes, then the scale boxes as loaded (row-major
// 16 bytes per row), which the scale warps rearrange in place into the
// layout tcgen05.cp reads (each 2 KB atom of 128 rows becomes four 512-byte
// chunks, one per MMA step).
constexpr uint32_t kA = BM * BKB;                  // 16 KB
constexpr uint32_t kB = BN * BKB;                  // 32 KB
constexpr uint32_t kSfaStage = BM * 16;
constexpr uint32_t kSfbStage = BN * 16;
constexpr uint32_t offB = kA;
constexpr uint32_t offSfaStage = kA + kB;
constexpr uint32_t offSfbStage = offSfaStage + kSfaStage;
constexpr uint32_t kStage = offSfbStage + kSfbStage;  // 54 KB
constexpr uint32_t kSfTmemPerStage = 16 + 32;          // SFA: 4 x 4 columns, SFB: 4 x 8
// A and its scales arrive in boxes of 32 rows, only as many as the item's
// rows need (a decode-sized group fills one); the MMA still reads 128 rows,
// and rows past the loaded boxes only feed accumulator rows never stored.
constexpr int kABox = 32;
constexpr uint32_t kABoxBytes = kABox * BKB;
constexpr uint32_t kSfaBoxBytes = kABox * 16;
static_assert(kStage % 1024 == 0, "stages keep the 1 KB alignment of the 128-byte swizzle");
static_assert(kABoxBytes % 1024 == 0, "A boxes keep the 8-row swizzle pattern");
static_assert(kSfTmemBase + kMaxStages * kSfTmemPerStage <= kTmemCols, "TMEM budget");
static_assert((4 * kMaxStages + 4) * 8 <= 192, "barriers precede the TMEM slot");

struct Params {
  const float* gsa;
  const float* gsb;
  const int32_t* offs;
  uint16_t* out;
  uint32_t* status;
  int64_t ld_out;
  int M, E, two_i, K;
  int layout;
  float limit;
  int num_k_tiles;    // K / 256
  int n_tiles;        // 2I / 256
  int max_row_tiles;  // row tiles the item list may hold (a bound for valid offsets)
  int stages;         // pipeline depth (3 or 4)
};

// Instruction descriptor of kind::mxf4nvf4: E2M1 A and B, E4M3 scales, both
// operands K-major, N >> 3 at bit 17, M >> 4 at bit 24, dense K = 64.
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
                            (static_cast<uint32_t>(BM >> 4) << 24);

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile uint32_t* abort) {
  bool ok = true;
  if (lane_id() == 0) ok = mbar_wait_bounded(bar, parity, abort, kWaitLimit);
  return __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
}

__device__ __forceinline__ void record_timeout(uint32_t* status, volatile uint32_t* abort) {
  *abort = 1u;
  atomicOr(status, NVFP4_DEVICE_TIMEOUT);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void st_global_v4(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

// tcgen05.ld writes its registers asynchronously: after tcgen05.wait::ld,
// this empty asm marks them as (re)defined, so no use of them can be
// scheduled before the wait.
__device__ __forceinline__ void regs_after_wait(uint32_t (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) asm volatile("" : "+r"(v[i]));
}

// Clamp + SwiGLU of one 32-column accumulator chunk of row `orow` (TMEM
// words v), then the bf16 store: 16 values h (layout 0) at output column
// (n0 + c) / 2, or the chunk's 32 columns as a / h (layout 1) at n0 + c.
// exp and the quotient use the fast hardware approximations (a few ulp;
// far inside the epilogue's tolerance).
template <int G>
__device__ __forceinline__ void swiglu_chunk(const uint32_t (&v)[32], float gab, float limit, int layout,
                                             uint16_t* orow, int col) {
  float av[16], hv[16];
#pragma unroll
  for (int x = 0; x < 16; ++x) {
    // x-th (gate, up) pair of the chunk: run x / G, offset x % G
    const int gi = (x / G) * 2 * G + (x % G);
    const float gate = fminf(__uint_as_float(v[gi]) * gab, limit);
    const float up = fminf(fmaxf(__uint_as_float(v[gi + G]) * gab, -limit), limit);
    av[x] = __fdividef(gate, 1.0f + __expf(-gate));
    hv[x] = av[x] * up;
  }
  if (layout == 0) {
    uint16_t* dst = orow + col / 2;
    st_global_v4(dst, pack_bf16x2(hv[0], hv[1]), pack_bf16x2(hv[2], hv[3]), pack_bf16x2(hv[4], hv[5]),
                 pack_bf16x2(hv[6], hv[7]));
    st_global_v4(dst + 8, pack_bf16x2(hv[8], hv[9]), pack_bf16x2(hv[10], hv[11]), pack_bf16x2(hv[12], hv[13]),
                 pack_bf16x2(hv[14], hv[15]));
  } else {
    // column y of the chunk: run y / G (even: gate -> a, odd: up -> h)
    float o[32];
#pragma unroll
    for (int y = 0; y < 32; ++y) {
      const int x = (y / (2 * G)) * G + (y % G);
      o[y] = ((y / G) & 1) ? hv[x] : av[x];
    }
    uint16_t* dst = orow + col;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      st_global_v4(dst + 8 * q, pack_bf16x2(o[8 * q], o[8 * q + 1]), pack_bf16x2(o[8 * q + 2], o[8 * q + 3]),
                   pack_bf16x2(o[8 * q + 4], o[8 * q + 5]), pack_bf16x2(o[8 * q + 6], o[8 * q + 7]));
  }
}

// One work item: rows m0 .. m0 + vr - 1 of A against weight rows brow ..
// brow + 255 of group e (output columns n0 .. n0 + 255 of the 2I).
struct Item {
  int e, m0, vr, n0;
};

// Item w of the list: row tile w / n_tiles (found among the groups' tile
// starts by bisection), weight slice w % n_tiles.
__device__ __forceinline__ Item item_of(int w, const Params& p, const int* tstart, const int* lo,
                                        const int* hi) {
  const int rt = w / p.n_tiles;
  int a = 0, b = p.E;  // the last group e with tstart[e] <= rt (a non-empty one)
  while (b - a > 1) {
    const int mid = (a + b) >> 1;
    if (tstart[mid] <= rt) a = mid; else b = mid;
  }
  Item it;
  it.e = a;
  it.m0 = lo[a] + (rt - tstart[a]) * BM;
  it.vr = min(BM, hi[a] - it.m0);
  it.n0 = (w % p.n_tiles) * BN;
  return it;
}

template <int G>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_swiglu_kernel(const __grid_constant__ CUtensorMap tma_a,
                          const __grid_constant__ CUtensorMap tma_b,
                          const __grid_constant__ CUtensorMap tma_sfa,
                          const __grid_constant__ CUtensorMap tma_sfb, const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const int warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();
  const int S = p.stages;
  uint8_t* ctrl = smem + S * kStage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(ctrl);
  auto full_bar = [&](int s) { return smem_addr(&bars[s]); };
  auto empty_bar = [&](int s) { return smem_addr(&bars[kMaxStages + s]); };
  auto sfready_bar = [&](int s) { return smem_addr(&bars[2 * kMaxStages + s]); };
  auto sffull_bar = [&](int s) { return smem_addr(&bars[3 * kMaxStages + s]); };  // scale boxes landed
  const uint32_t tfull_bar = smem_addr(&bars[4 * kMaxStages]);       // accumulator complete
  const uint32_t tempty_bar = smem_addr(&bars[4 * kMaxStages + 1]);  // accumulator read out
  const uint32_t drain_bar = smem_addr(&bars[4 * kMaxStages + 2]);   // MMAs drained
  const uint32_t xdrain_bar = smem_addr(&bars[4 * kMaxStages + 3]);  // scale copies drained
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 192);
  volatile uint32_t* abort = reinterpret_cast<volatile uint32_t*>(ctrl + 196);
  int* tstart = reinterpret_cast<int*>(ctrl + kCtrlBytes);  // [E + 1] first row tile of each group
  int* glo = tstart + (p.E + 1);                              // [E] clamped first row
  int* ghi = glo + p.E;                                       // [E] clamped end row

  if (threadIdx.x == 32) {  // descriptor fetches overlap the set-up
    prefetch_tensormap(&tma_a);
    prefetch_tensormap(&tma_b);
    prefetch_tensormap(&tma_sfa);
    prefetch_tensormap(&tma_sfb);
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(sffull_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(sfready_bar(s), 4);  // one tcgen05.commit per scale-layout warp
    }
    mbar_init(tfull_bar, 1);
    mbar_init(tempty_bar, 4);  // one arrival per epilogue warp
    mbar_init(drain_bar, 1);
    mbar_init(xdrain_bar, 4);
    *abort = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 2) {
    // Per-group tile starts: an exclusive scan of ceil(rows / 128) over the
    // groups, each group's row range clamped into [0, M] and made non-empty
    // only when its end lies past its start.
    bool bad = false;
    int acc = 0;
    for (int base = 0; base < p.E; base += 32) {
      const int e = base + static_cast<int>(lane);
      int lo = 0, hi = 0;
      if (e < p.E) {
        const int o0 = __ldg(p.offs + e), o1 = __ldg(p.offs + e + 1);
        bad |= o1 < o0 || o0 < 0 || o1 > p.M;
        lo = min(max(o0, 0), p.M);
        hi = min(max(o1, lo), p.M);
        glo[e] = lo;
        ghi[e] = hi;
      }
      const int tiles = (hi - lo + BM - 1) / BM;
      int incl = tiles;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (static_cast<int>(lane) >= o) incl += t;
      }
      if (e < p.E) tstart[e] = acc + incl - tiles;
      acc += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    if (acc > p.max_row_tiles) {  // overlapping groups: keep the items the launch has room for
      acc = p.max_row_tiles;
      bad = true;
    }
    if (lane == 0) tstart[p.E] = acc;
    if (__any_sync(0xFFFFFFFFu, bad) && lane == 0 && blockIdx.x == 0) atomicOr(p.status, NVFP4_DEVICE_BAD_GROUPS);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total = tstart[p.E] * p.n_tiles;
  const int nk = p.num_k_tiles;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int i = 0;  // stages issued by this CTA (the ring runs on across items)
    bool ok = true;
    for (int w = blockIdx.x; ok && w < total; w += gridDim.x) {
      const Item it = item_of(w, p, tstart, glo, ghi);
      const int brow = it.e * p.two_i + it.n0;
      const int na = (it.vr + kABox - 1) / kABox;  // A boxes holding the item's rows
      for (int kt = 0; kt < nk; ++kt, ++i) {
        const int s = i % S;
        const uint32_t ph = (i / S) & 1;
        if (!warp_wait(empty_bar(s), ph ^ 1u, abort)) {
          if (lane == 0) record_timeout(p.status, abort);
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t st = sbase + s * kStage;
          mbar_arrive_expect_tx(sffull_bar(s), na * kSfaBoxBytes + kSfbStage);
          for (int q = 0; q < na; ++q)
            tma_load_2d(st + offSfaStage + q * kSfaBoxBytes, &tma_sfa, sffull_bar(s), kt * 16, it.m0 + q * kABox);
          tma_load_2d(st + offSfbStage, &tma_sfb, sffull_bar(s), kt * 16, brow);
          mbar_arrive_expect_tx(full_bar(s), na * kABoxBytes + kB);
          for (int q = 0; q < na; ++q)
            tma_load_2d(st + q * kABoxBytes, &tma_a, full_bar(s), kt * BKB, it.m0 + q * kABox);
          tma_load_2d(st + offB, &tma_b, full_bar(s), kt * BKB, brow);
        }
        __syncwarp();
      }
    }
    if (lane == 0) {  // let every copy issued here land before the CTA can exit
      uint32_t never = 0;
      const int last = i - 1;
      for (int s = 0; s < S; ++s) {
        const int i_s = last - (((last - s) % S) + S) % S;
        if (last >= 0 && i_s >= 0 &&
            (!mbar_wait_bounded(full_bar(s), (i_s / S) & 1, &never, kWaitLimit) ||
             !mbar_wait_bounded(sffull_bar(s), (i_s / S) & 1, &never, kWaitLimit)))
          record_timeout(p.status, abort);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    int i = 0, t = 0;
    bool ok = true;
    for (int w = blockIdx.x; ok && w < total; w += gridDim.x, ++t) {
      if (t > 0) {  // the epilogue has read the previous item's accumulator
        if (!warp_wait(tempty_bar, (t - 1) & 1, abort)) {
          if (lane == 0) record_timeout(p.status, abort);
          break;
        }
        tc_fence_after();
      }
      for (int kt = 0; kt < nk; ++kt, ++i) {
        const int s = i % S;
        const uint32_t ph = (i / S) & 1;
        if (!warp_wait(full_bar(s), ph, abort) || !warp_wait(sfready_bar(s), ph, abort)) {
          if (lane == 0) record_timeout(p.status, abort);
          ok = false;
          break;
        }
        if (lane == 0) {
          tc_fence_after();
          const uint32_t st = sbase + s * kStage;
          const uint32_t sf_col = tmem + kSfTmemBase + s * kSfTmemPerStage;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_nvf4(tmem, smem_desc(st + kk * 32, 16, 1024, 2), smem_desc(st + offB + kk * 32, 16, 1024, 2),
                        kIdesc, sf_col + kk * 4, sf_col + 16 + kk * 8, (kt | kk) != 0 ? 1u : 0u);
          tc_commit(empty_bar(s));  // frees the stage once these MMAs have read it
        }
        __syncwarp();
      }
      if (ok && lane == 0) tc_commit(tfull_bar);
      __syncwarp();
    }
    if (lane == 0) {
      uint32_t never = 0;
      tc_commit(drain_bar);
      if (!mbar_wait_bounded(drain_bar, 0, &never, kWaitLimit)) record_timeout(p.status, abort);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ scale layout + epilogue
    const int u = warp - 2;            // MMA step kk = u of every scale atom
    const int quarter = warp & 3;      // TMEM lanes 32 * quarter .. + 31
    const int row = quarter * 32 + static_cast<int>(lane);
    const float gsa = __ldg(p.gsa);
    int i = 0, t = 0;
    bool ok = true;
    for (int w = blockIdx.x; ok && w < total; w += gridDim.x, ++t) {
      for (int kt = 0; kt < nk; ++kt, ++i) {
        const int s = i % S;
        const uint32_t ph = (i / S) & 1;
        // the four warps leave together when any of them gave up waiting
        const bool failed = !warp_wait(sffull_bar(s), ph, abort);
        if (bar_any_128(failed)) {
          if (failed && lane == 0) record_timeout(p.status, abort);
          ok = false;
          break;
        }
        const uint32_t st = sbase + s * kStage;
        // Staged row r (16 bytes: MMA words 0..3) -> chunk u gets, at offset
        // 16 * r0, word u of rows r0, r0 + 32, r0 + 64, r0 + 96.  Chunk u
        // overwrites staged rows 32u .. 32u + 31 of the atom, so every warp
        // reads its words before any writes (the barrier in between).
        uint32_t sw[3][4];
#pragma unroll
        for (int a = 0; a < 3; ++a) {
          const uint32_t src = a == 0 ? st + offSfaStage : st + offSfbStage + (a - 1) * 2048;
#pragma unroll
          for (int q = 0; q < 4; ++q) sw[a][q] = ld_shared_u32(src + (q * 32 + lane) * 16 + u * 4);
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
#pragma unroll
        for (int a = 0; a < 3; ++a) {
          const uint32_t atom = a == 0 ? st + offSfaStage : st + offSfbStage + (a - 1) * 2048;
          st_shared_v4(atom + u * kSfChunk + lane * 16, sw[a][0], sw[a][1], sw[a][2], sw[a][3]);
        }
        fence_proxy_async_smem();  // read by tcgen05.cp through the async proxy
        __syncwarp();
        if (lane == 0) {
          tc_fence_after();
          const uint32_t sf_col = tmem + kSfTmemBase + s * kSfTmemPerStage;
          tc_cp_32x128b_warpx4(sf_col + u * 4, smem_desc(st + offSfaStage + u * kSfChunk, 0, 128, 0));
          tc_cp_32x128b_warpx4(sf_col + 16 + u * 8, smem_desc(st + offSfbStage + u * kSfChunk, 0, 128, 0));
          tc_cp_32x128b_warpx4(sf_col + 16 + u * 8 + 4,
                               smem_desc(st + offSfbStage + 2048 + u * kSfChunk, 0, 128, 0));
          tc_commit(sfready_bar(s));
        }
        __syncwarp();
      }
      if (!ok) break;
      const bool tfailed = !warp_wait(tfull_bar, t & 1, abort);
      if (bar_any_128(tfailed)) {  // (uniform: the next item's barriers need all four warps)
        if (tfailed && lane == 0) record_timeout(p.status, abort);
        break;
      }
      tc_fence_after();
      // ---- epilogue of item w: TMEM -> registers -> clamp + SwiGLU -> bf16 -> global
      const Item it = item_of(w, p, tstart, glo, ghi);
      if (quarter * 32 < it.vr) {
        const float gab = gsa * __ldg(p.gsb + it.e);
        const bool live = row < it.vr;
        uint16_t* orow = p.out + static_cast<int64_t>(it.m0 + (live ? row : 0)) * p.ld_out;
        const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        // two chunks in flight: the load of chunk c + 32 overlaps the math of chunk c
        uint32_t va[32], vb[32];
        tmem_ld_32x32b_x32(taddr, va);
#pragma unroll
        for (int c = 0; c < BN; c += 64) {
          tmem_wait_ld();
          regs_after_wait(va);
          tmem_ld_32x32b_x32(taddr + c + 32, vb);
          if (live) swiglu_chunk<G>(va, gab, p.limit, p.layout, orow, it.n0 + c);
          tmem_wait_ld();
          regs_after_wait(vb);
          if (c + 64 < BN) tmem_ld_32x32b_x32(taddr + c + 64, va);
          if (live) swiglu_chunk<G>(vb, gab, p.limit, p.layout, orow, it.n0 + c + 32);
        }
        tmem_wait_ld();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar);
    }
    if (lane == 0) {  // every copy of this warp has completed before TMEM can be freed
      uint32_t never = 0;
      tc_commit(xdrain_bar);
      if (!mbar_wait_bounded(xdrain_bar, 0, &never, kWaitLimit)) record_timeout(p.status, abort);
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

size_t smem_bytes(int stages, int64_t E) {
  return 1024 + static_cast<size_t>(stages) * kStage + kCtrlBytes + static_cast<size_t>(3 * E + 1) * 4;
}

template <int G>
cudaError_t launch_g(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& msa, const CUtensorMap& msb,
                     const Params& p, int grid, size_t smem, cudaStream_t stream) {
  auto kern = grouped_swiglu_kernel<G>;
  static std::mutex mu;
  static int configured = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (static_cast<int>(smem) > configured) {
      const cudaError_t e =
          cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      configured = static_cast<int>(smem);
    }
  }
  count_launch();
  kern<<<grid, kThreads, smem, stream>>>(ma, mb, msa, msb, p);
  return cudaGetLastError();
}

}  // namespace

int launch_grouped_swiglu(const GroupedSwigluArgs& a, cudaStream_t stream, cudaError_t* err) {
  *err = cudaSuccess;
  if (a.M == 0) return NVFP4_OK;
  const int64_t two_i = 2 * a.inter;
  CUtensorMap ma, mb, msa, msb;
  if (!make_map(&ma, a.qa, a.M, a.K / 2, BKB, kABox, true) ||
      !make_map(&mb, a.qb, a.E * two_i, a.K / 2, BKB, BN, true) ||
      !make_map(&msa, a.sfa, a.M, a.K / 16, 16, kABox, false) ||
      !make_map(&msb, a.sfb, a.E * two_i, a.K / 16, 16, BN, false))
    return NVFP4_ERR_UNSUPPORTED;
  Params p;
  std::memset(&p, 0, sizeof(p));
  p.gsa = a.gsa;
  p.gsb = a.gsb;
  p.offs = a.offsets;
  p.out = a.out;
  p.status = &a.ws->status;
  p.ld_out = a.ld_out;
  p.M = static_cast<int>(a.M);
  p.E = static_cast<int>(a.E);
  p.two_i = static_cast<int>(two_i);
  p.K = static_cast<int>(a.K);
  p.layout = a.layout;
  p.limit = a.limit;
  p.num_k_tiles = static_cast<int>(a.K / 256);
  p.n_tiles = static_cast<int>(two_i / BN);
  // Valid offsets give at most floor(M / 128) + min(E, M) row tiles.
  const int64_t row_tiles = a.M / BM + (a.E < a.M ? a.E : a.M);
  p.max_row_tiles = static_cast<int>(row_tiles);
  const int64_t items = row_tiles * p.n_tiles;
  const int grid = static_cast<int>(items < sm_count() ? items : sm_count());
  int smem_optin = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  p.stages = smem_bytes(kMaxStages, a.E) <= static_cast<size_t>(smem_optin) ? kMaxStages : kMaxStages - 1;
  const size_t smem = smem_bytes(p.stages, a.E);
  cudaError_t e;
  switch (a.granularity) {
    case 1: e = launch_g<1>(ma, mb, msa, msb, p, grid, smem, stream); break;
    case 2: e = launch_g<2>(ma, mb, msa, msb, p, grid, smem, stream); break;
    case 4: e = launch_g<4>(ma, mb, msa, msb, p, grid, smem, stream); break;
    case 8: e = launch_g<8>(ma, mb, msa, msb, p, grid, smem, stream); break;
    default: e = launch_g<16>(ma, mb, msa, msb, p, grid, smem, stream); break;
  }
  if (e != cudaSuccess) {
    *err = e;
    return NVFP4_ERR_CUDA;
  }
  return NVFP4_OK;
}


}  // namespace nvfp4
