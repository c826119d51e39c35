// NVFP4 activation quantize for sm_103a: grid-wide amax -> global scale, then
// E4M3 block scales and E2M1 codes.
//
// Two kernels, as the dsv4/ops/quantize.py commit of the nvfp4-megamoe-kernel
// pages settles on after a one-kernel version raced (a __syncthreads-only
// reduction does not order blocks): the amax kernel combines block maxima
// with atomics and the last block to finish (ticket counter after a device
// fence) writes gs to device memory; the quantize kernel then reads gs from
// that buffer.  No host synchronisation anywhere.
//
// Memory access: 16-byte vector loads of 8 bf16 (eight in flight per thread
// in the amax pass, two 16-element blocks per thread in the quantize pass),
// 8-byte stores of the packed code bytes, grid-stride loops over a grid
// sized to the SM count.  The element quotients x / den are exact (one FMA
// correction of x * (1/den)), so codes match the correctly rounded division.

#include <cstdint>

#include <cuda_bf16.h>

#include "internal.h"
#include "nvfp4.h"
#include "ptx.cuh"

namespace nvfp4 {
namespace {

constexpr int kThreads = 256;
constexpr float kGsDivisor = 2688.0f;  // 6 (E2M1 max) * 448 (E4M3 max)
constexpr float kAmaxFloor = 1e-8f;

// First pass (amax): the tail of the tensor that the second pass (which runs
// backwards) reads first, up to kL2KeepBytes, is loaded with an L2
// evict-last policy and the rest with evict-first, so the tail survives in
// L2.  Second pass: loads with an evict-first policy (last use: lines just
// consumed leave before the ones still to come), ordinary stores (the codes
// and scales stay in L2 for the GEMM that reads them next).
__device__ __forceinline__ uint4 ld_keep(const uint16_t* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ uint64_t l2_policy_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t l2_policy_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint4 ld_policy(const uint4* p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}
// Bytes of a large tensor's tail the amax pass marks to keep in L2 (of 126 MB).
constexpr int64_t kL2KeepBytes = 64ll << 20;
__device__ __forceinline__ uint4 ld_stream(const uint16_t* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}

// Per-16-bit-lane maximum of |bf16| over 8 values (bit patterns compare like
// the magnitudes they encode once the sign bit is cleared).
__device__ __forceinline__ uint32_t absmax8(uint4 v) {
  const uint32_t m = 0x7FFF7FFFu;
  return __vmaxu2(__vmaxu2(v.x & m, v.y & m), __vmaxu2(v.z & m, v.w & m));
}

__device__ __forceinline__ uint32_t fold16(uint32_t m2) { return max(m2 & 0xFFFFu, m2 >> 16); }

// ---------------------------------------------------------------- amax

constexpr int kAmaxUnroll = 8;  // 16-byte loads in flight per thread

__global__ void __launch_bounds__(kThreads, 4)
    amax_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t vpr, int64_t ld,
                float* __restrict__ gs_out, Workspace* __restrict__ ws) {
  ptx::pdl_launch_dependents();  // a dependent kernel may set up while this one runs
  uint32_t m2 = 0;
  const int64_t total = rows * vpr;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (ld == vpr * 8) {
    const uint4* xv = reinterpret_cast<const uint4*>(x);
    // Keep (at most) the last kL2KeepBytes in L2 for the quantize pass, which
    // starts from the end; the head streams through.
    const int64_t keep_from = total * 16 > kL2KeepBytes ? total - kL2KeepBytes / 16 : 0;
    {
      const uint64_t pol_first = l2_policy_first(), pol_last = l2_policy_last();
      for (; i + (kAmaxUnroll - 1) * stride < total; i += kAmaxUnroll * stride) {
        uint4 v[kAmaxUnroll];
#pragma unroll
        for (int u = 0; u < kAmaxUnroll; ++u) {
          const int64_t j = i + u * stride;
          v[u] = ld_policy(xv + j, j >= keep_from ? pol_last : pol_first);
        }
#pragma unroll
        for (int u = 0; u < kAmaxUnroll; ++u) m2 = __vmaxu2(m2, absmax8(v[u]));
      }
      for (; i < total; i += stride) m2 = __vmaxu2(m2, absmax8(ld_policy(xv + i, i >= keep_from ? pol_last : pol_first)));
    }
  } else if (i < total) {
    int64_t r = i / vpr, c = i % vpr;
    const int64_t sr = stride / vpr, sc = stride % vpr;
    while (r < rows) {
      m2 = __vmaxu2(m2, absmax8(ld_keep(x + r * ld + c * 8)));
      c += sc;
      r += sr;
      if (c >= vpr) {
        c -= vpr;
        ++r;
      }
    }
  }
  uint32_t m = fold16(m2);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  __shared__ uint32_t warp_max[kThreads / 32];
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kThreads / 32; ++w) m = max(m, warp_max[w]);
    // bf16 bits << 16 are the FP32 bits of the same value; non-negative FP32
    // values order like their bit patterns, so an integer max is a float max.
    atomicMax(&ws->amax_bits, m << 16);
    __threadfence();
    const uint32_t ticket = atomicAdd(&ws->done, 1u);
    if (ticket == gridDim.x - 1) {
      // Every block's atomicMax precedes its ticket, so the max is complete.
      const uint32_t bits = atomicAdd(&ws->amax_bits, 0u);
      const float amax = fmaxf(__uint_as_float(bits), kAmaxFloor);
      gs_out[0] = __fdiv_rn(amax, kGsDivisor);
      ws->amax_bits = 0;
      ws->done = 0;
    }
  }
}

// ---------------------------------------------------------------- block codec

// E4M3 (FN) code of s >= 0: round to nearest even, saturating at 448 (the
// hardware conversion, branch-free; subnormal codes are steps of 2^-9).
__device__ __forceinline__ uint32_t e4m3_encode(float s) {
  uint16_t pair;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(0.0f), "f"(s));
  return pair & 0xFFu;  // the second operand lands in the low byte
}

// Value of a non-negative E4M3 code (exact through FP16).
__device__ __forceinline__ float e4m3_decode(uint32_t c) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(c)));
  float f;
  asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(static_cast<uint16_t>(h2 & 0xFFFFu)));
  return f;
}

__device__ __forceinline__ float lo_bf16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Correctly rounded a / b from r = RN(1/b) by one FMA correction: q = RN(a r),
// e = a - q b (exact, one FMA), result RN(q + e r).  This is Markstein's
// division theorem (P. Markstein, "Computation of elementary functions on the
// IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990): with r the
// correctly rounded reciprocal and q within one ulp of a / b, the corrected
// quotient is the correctly rounded one.  (Results in the subnormal range can
// be off by an ulp; every such value encodes to a zero code and an E4M3 zero
// here, so the outputs do not change.)
__device__ __forceinline__ float div_rn(float a, float b, float r) {
  const float q = __fmul_rn(a, r);
  const float e = __fmaf_rn(-q, b, a);
  return __fmaf_rn(e, r, q);
}

// Per-code divisors of one tensor: entry c holds den = e4m3(c) * gs (one
// FP32 multiply) and RN(1 / den) (0 when den is 0).  One table per CTA in
// shared memory, filled once gs is known, replaces a decode, a multiply and a
// correctly rounded reciprocal per block with one shared-memory load.
struct Codec {
  float gs;            // global scale
  float r_gs;          // RN(1 / gs)
  float r_six;         // RN(1 / 6)
  const float2* tab;   // [128] {den, RN(1/den)} by E4M3 code
};

// Threads of the block fill the table (the caller then synchronises).
__device__ __forceinline__ void fill_codec(float2* tab, float gs) {
  for (int c = static_cast<int>(threadIdx.x); c < 128; c += static_cast<int>(blockDim.x)) {
    const float den = __fmul_rn(e4m3_decode(static_cast<uint32_t>(c)), gs);
    tab[c] = make_float2(den, den == 0.0f ? 0.0f : __frcp_rn(den));
  }
}

__device__ __forceinline__ Codec make_codec(float gs, const float2* tab) {
  Codec cd;
  cd.gs = gs;
  cd.r_gs = __frcp_rn(gs);
  cd.r_six = __frcp_rn(6.0f);
  cd.tab = tab;
  return cd;
}

// Bits of the largest |x| over 16 bf16 values (two vectors): bf16x2 maxima
// of magnitudes (the sign bits they leave are cleared at the end).
__device__ __forceinline__ uint32_t absmax16(uint4 a, uint4 b) {
  uint32_t m0, m1, m2, m3, m4, m5, m6;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m0) : "r"(a.x), "r"(a.y));
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m1) : "r"(a.z), "r"(a.w));
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m2) : "r"(b.x), "r"(b.y));
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m3) : "r"(b.z), "r"(b.w));
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m4) : "r"(m0), "r"(m1));
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m5) : "r"(m2), "r"(m3));
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m6) : "r"(m4), "r"(m5));
  return fold16(m6 & 0x7FFF7FFFu);
}

// E2M1 codes of the 8 bf16 values of v divided by den (element 0 in the low
// nibble).  Per pair of values x (packed FP32 arithmetic) with nr = -RN(1/den):
//   qn = RN(x nr) = -RN(x r),  e = RN(qn den + x) = x - q den (exact),
//   vn = RN(e nr + qn) = -RN(q + e r) = -(x / den correctly rounded),
// Markstein's correction carried out on the negated quotient.  The E2M1
// conversion of vn rounds to nearest even, saturates and keeps the sign of
// values that round to zero; flipping the four sign bits of each byte then
// gives the codes of x / den.  Signed zeros come out right: x = -0 gives
// vn = +0 (code 0x8 after the flip), x = +0 gives vn = -0 (code 0x0), and
// den = 0 (r = 0) gives vn = -0 * sign(x), a zero code of x's sign.
__device__ __forceinline__ uint32_t encode8(uint4 v, uint64_t nr2, uint64_t d2) {
  uint32_t out;
  asm("{\n\t.reg .b64 x, qn, e, vn;\n\t.reg .f32 lo, hi;\n\t.reg .b8 c0, c1, c2, c3;\n\t"
      "mov.b64 x, {%3, %4};\n\tmul.rn.f32x2 qn, x, %1;\n\tfma.rn.f32x2 e, qn, %2, x;\n\t"
      "fma.rn.f32x2 vn, e, %1, qn;\n\tmov.b64 {lo, hi}, vn;\n\tcvt.rn.satfinite.e2m1x2.f32 c0, hi, lo;\n\t"
      "mov.b64 x, {%5, %6};\n\tmul.rn.f32x2 qn, x, %1;\n\tfma.rn.f32x2 e, qn, %2, x;\n\t"
      "fma.rn.f32x2 vn, e, %1, qn;\n\tmov.b64 {lo, hi}, vn;\n\tcvt.rn.satfinite.e2m1x2.f32 c1, hi, lo;\n\t"
      "mov.b64 x, {%7, %8};\n\tmul.rn.f32x2 qn, x, %1;\n\tfma.rn.f32x2 e, qn, %2, x;\n\t"
      "fma.rn.f32x2 vn, e, %1, qn;\n\tmov.b64 {lo, hi}, vn;\n\tcvt.rn.satfinite.e2m1x2.f32 c2, hi, lo;\n\t"
      "mov.b64 x, {%9, %10};\n\tmul.rn.f32x2 qn, x, %1;\n\tfma.rn.f32x2 e, qn, %2, x;\n\t"
      "fma.rn.f32x2 vn, e, %1, qn;\n\tmov.b64 {lo, hi}, vn;\n\tcvt.rn.satfinite.e2m1x2.f32 c3, hi, lo;\n\t"
      "mov.b32 %0, {c0, c1, c2, c3};\n\t}"
      : "=r"(out)
      : "l"(nr2), "l"(d2), "f"(lo_bf16(v.x)), "f"(hi_bf16(v.x)), "f"(lo_bf16(v.y)),
        "f"(hi_bf16(v.y)), "f"(lo_bf16(v.z)), "f"(hi_bf16(v.z)), "f"(lo_bf16(v.w)), "f"(hi_bf16(v.w)));
  return out ^ 0x88888888u;
}

__device__ __forceinline__ uint64_t pair_f32(float a) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(a));
  return r;
}

// Quantize one 16-element block held in two vectors.
__device__ __forceinline__ void quantize_block(uint4 a, uint4 b, const Codec& cd, uint32_t& sbyte,
                                               uint2& codes) {
  const float bamax = __uint_as_float(absmax16(a, b) << 16);
  const float s = div_rn(div_rn(bamax, 6.0f, cd.r_six), cd.gs, cd.r_gs);  // (bamax / 6) / gs
  sbyte = e4m3_encode(s);
  const float2 t = cd.tab[sbyte];  // {den, RN(1 / den)}
  const uint64_t nr2 = pair_f32(-t.y), d2 = pair_f32(t.x);
  codes = make_uint2(encode8(a, nr2, d2), encode8(b, nr2, d2));
}

// ---------------------------------------------------------------- quantize

// Blocks are visited from the end of the tensor backwards: the amax pass that
// ran just before leaves the tail of a tensor larger than L2 in L2, so this
// pass finds that part there.  Loads and stores stream (evict first).
__global__ void __launch_bounds__(kThreads, 4)
    quantize_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t bpr, int64_t ld,
                    uint8_t* __restrict__ q, uint8_t* __restrict__ sf,
                    const float* __restrict__ gs_ptr) {
  ptx::pdl_launch_dependents();
  __shared__ float2 tab[128];
  const float gs = __ldg(gs_ptr);
  fill_codec(tab, gs);
  __syncthreads();
  const int64_t total = rows * bpr;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t0 >= total) return;
  const Codec sc = make_codec(gs, tab);
  if (ld == bpr * 16) {  // contiguous rows: one flat index
    const uint4* xv = reinterpret_cast<const uint4*>(x);
    uint2* qv = reinterpret_cast<uint2*>(q);
    const uint64_t pol = l2_policy_first();
    int64_t b = total - 1 - t0;
    for (; b - 3 * stride >= 0; b -= 4 * stride) {  // four blocks (8 loads) in flight
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        v[2 * u] = ld_policy(xv + 2 * (b - u * stride), pol);
        v[2 * u + 1] = ld_policy(xv + 2 * (b - u * stride) + 1, pol);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        uint32_t s0;
        uint2 k0;
        quantize_block(v[2 * u], v[2 * u + 1], sc, s0, k0);
        qv[b - u * stride] = k0;
        sf[b - u * stride] = static_cast<uint8_t>(s0);
      }
    }
    for (; b >= 0; b -= stride) {
      uint32_t s0;
      uint2 k0;
      quantize_block(ld_policy(xv + 2 * b, pol), ld_policy(xv + 2 * b + 1, pol), sc, s0, k0);
      qv[b] = k0;
      sf[b] = static_cast<uint8_t>(s0);
    }
    return;
  }
  const int64_t b0 = total - 1 - t0;
  int64_t r = b0 / bpr, c = b0 % bpr;
  const int64_t sr = stride / bpr, scol = stride % bpr;
  while (r >= 0) {
    const uint16_t* src = x + r * ld + c * 16;
    uint32_t sbyte;
    uint2 codes;
    quantize_block(ld_stream(src), ld_stream(src + 8), sc, sbyte, codes);
    *reinterpret_cast<uint2*>(q + r * (bpr * 8) + c * 8) = codes;
    sf[r * bpr + c] = static_cast<uint8_t>(sbyte);
    c -= scol;
    r -= sr;
    if (c < 0) {
      c += bpr;
      --r;
    }
  }
}

// ---------------------------------------------------------------- deinterleave

// Split 32 consecutive input elements (16 words of two bf16) into the 16
// gate and 16 up elements they hold when gate/up alternate every G columns.
template <int G>
__device__ __forceinline__ void split_gate_up(const uint32_t (&w)[16], uint32_t (&gate)[8],
                                              uint32_t (&up)[8]) {
  if constexpr (G == 1) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      gate[k] = __byte_perm(w[2 * k], w[2 * k + 1], 0x5410);  // low halves
      up[k] = __byte_perm(w[2 * k], w[2 * k + 1], 0x7632);    // high halves
    }
  } else {
    constexpr int GW = G / 2;  // words per group
    int ng = 0, nu = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if ((i / GW) % 2 == 0)
        gate[ng++] = w[i];
      else
        up[nu++] = w[i];
    }
  }
}

// Same visiting order as quantize_kernel (from the end backwards, streaming).
template <int G>
__global__ void __launch_bounds__(kThreads, 4)
    deinterleave_quantize_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t inter,
                                 uint8_t* __restrict__ q, uint8_t* __restrict__ sf,
                                 const float* __restrict__ gs_ptr) {
  ptx::pdl_launch_dependents();
  __shared__ float2 tab[128];
  const float gs = __ldg(gs_ptr);
  fill_codec(tab, gs);
  __syncthreads();
  const int64_t cpr = inter / 16;  // 32-element input chunks per row
  const int64_t total = rows * cpr;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t0 >= total) return;
  const Codec sc = make_codec(gs, tab);
  const int64_t b0 = total - 1 - t0;
  int64_t r = b0 / cpr, c = b0 % cpr;
  const int64_t sr = stride / cpr, scol = stride % cpr;
  while (r >= 0) {
    const uint4* src = reinterpret_cast<const uint4*>(x + r * (2 * inter) + c * 32);
    uint32_t w[16];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const uint4 t = __ldcs(src + v);
      w[4 * v] = t.x;
      w[4 * v + 1] = t.y;
      w[4 * v + 2] = t.z;
      w[4 * v + 3] = t.w;
    }
    uint32_t g[8], u[8];
    split_gate_up<G>(w, g, u);
    uint32_t sg, su;
    uint2 cg, cu;
    quantize_block(make_uint4(g[0], g[1], g[2], g[3]), make_uint4(g[4], g[5], g[6], g[7]), sc, sg,
                   cg);
    quantize_block(make_uint4(u[0], u[1], u[2], u[3]), make_uint4(u[4], u[5], u[6], u[7]), sc, su,
                   cu);
    uint8_t* qrow = q + r * inter;  // 2*inter codes -> inter bytes per row
    __stcs(reinterpret_cast<uint2*>(qrow + c * 8), cg);
    __stcs(reinterpret_cast<uint2*>(qrow + inter / 2 + c * 8), cu);
    uint8_t* srow = sf + r * (inter / 8);
    srow[c] = static_cast<uint8_t>(sg);
    srow[inter / 16 + c] = static_cast<uint8_t>(su);
    c -= scol;
    r -= sr;
    if (c < 0) {
      c += cpr;
      --r;
    }
  }
}

// ---------------------------------------------------------------- one pass

// For inputs that fit in the shared memory of the SMs (up to ~30 MB on a
// GB300): one cooperative launch, one CTA per SM.  Each CTA bulk-copies its
// slice of units (16-element blocks, or 32-element gate/up chunks for the
// deinterleave variant) into shared memory, reduces its |x| maximum into the
// workspace, meets the other CTAs at a grid barrier (an arrival counter; the
// launch guarantees the CTAs are co-resident; the wait is bounded), derives
// gs from the complete maximum exactly as the amax kernel does, and
// quantizes its slice from shared memory.  x is read from HBM once.  The
// last CTA to finish re-zeroes the workspace counters.
constexpr int kOnePassThreads = 512;
constexpr uint32_t kOnePassMaxBytes = 200 * 1024;  // input bytes one CTA holds
constexpr long long kBarrierCycles = 2000000000LL;  // ~1 s of SM clock

// kCluster: the grid is one thread-block cluster (<= 16 CTAs, small inputs);
// the maxima meet in distributed shared memory behind cluster barriers
// instead of the workspace counter.
template <int G, bool kCluster>  // G = 0: plain quantize (unit = 16 elements); else deinterleave granularity (unit = 32)
__global__ void __launch_bounds__(kOnePassThreads, 1)
    quantize_onepass_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t upr, int64_t ld,
                            int64_t units_per_cta, uint8_t* __restrict__ q, uint8_t* __restrict__ sf,
                            float* __restrict__ gs_out, Workspace* __restrict__ ws) {
  ptx::pdl_launch_dependents();
  constexpr int kUnitElems = G == 0 ? 16 : 32;
  constexpr uint32_t kUnitBytes = kUnitElems * 2;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t red[kOnePassThreads / 32];
  __shared__ float gs_sh;
  __shared__ float2 tab[128];
  const int64_t total = rows * upr;
  const int64_t u0 = static_cast<int64_t>(blockIdx.x) * units_per_cta;
  const int64_t u1 = u0 + units_per_cta < total ? u0 + units_per_cta : total;
  const int64_t n_units = u1 > u0 ? u1 - u0 : 0;
  const uint32_t bar_a = ptx::smem_addr(&bar);
  const uint32_t dst0 = ptx::smem_addr(smem);
  ptx::pdl_wait();  // launched early after the previous kernel: its writes are complete now
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar_a, 1);
    ptx::fence_mbar_init();
    ptx::mbar_arrive_expect_tx(bar_a, static_cast<uint32_t>(n_units * kUnitBytes));
    // one copy per row segment (rows may be strided), at most 64 KB each
    const int64_t row_units = ld == upr * kUnitElems ? total : upr;  // contiguous rows: one segment
    for (int64_t u = u0; u < u1;) {
      const int64_t seg_end0 = (u / row_units + 1) * row_units;
      const int64_t seg_end = seg_end0 < u1 ? seg_end0 : u1;
      const int64_t r = u / upr, c = u % upr;
      const uint8_t* src = reinterpret_cast<const uint8_t*>(x + r * ld + c * kUnitElems);
      int64_t left = (seg_end - u) * kUnitBytes;
      uint32_t dst = dst0 + static_cast<uint32_t>((u - u0) * kUnitBytes);
      while (left > 0) {
        const uint32_t n = left < 65536 ? static_cast<uint32_t>(left) : 65536u;
        ptx::bulk_load(dst, src, n, bar_a);
        src += n;
        dst += n;
        left -= n;
      }
      u = seg_end;
    }
  }
  __syncthreads();  // the barrier is initialised before anyone waits on it
  uint32_t never = 0;
  // A slice that did not land in time is left alone: the CTA still meets the
  // others (so none waits for it) but contributes no maximum and writes no
  // outputs, and the recorded NVFP4_DEVICE_TIMEOUT marks q, sf and gs as
  // undefined.
  const bool late_load = __syncthreads_or(!ptx::mbar_wait_bounded(bar_a, 0, &never, 2000000000LL)) != 0;
  if (late_load && threadIdx.x == 0) atomicOr(&ws->status, NVFP4_DEVICE_TIMEOUT);
  // local max of |x| over the slice
  const uint4* sv = reinterpret_cast<const uint4*>(smem);
  const int64_t n_vec = late_load ? 0 : n_units * (kUnitBytes / 16);
  uint32_t m2 = 0;
  for (int64_t i = threadIdx.x; i < n_vec; i += kOnePassThreads) m2 = __vmaxu2(m2, absmax8(sv[i]));
  uint32_t m = fold16(m2);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if constexpr (kCluster) {
    __shared__ float cta_max;
    if (threadIdx.x == 0) {
      for (int w = 1; w < kOnePassThreads / 32; ++w) m = max(m, red[w]);
      cta_max = __uint_as_float(m << 16);
    }
    ptx::cluster_sync();
    if (threadIdx.x < 32) {
      // lane r reads CTA r's maximum (the reads overlap), then a warp max
      const uint32_t r = threadIdx.x;
      float mx = r < gridDim.x ? ptx::ld_cluster_f32(ptx::mapa_shared(ptx::smem_addr(&cta_max), r)) : 0.0f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
      if (threadIdx.x == 0) {
        const float gs = __fdiv_rn(fmaxf(mx, kAmaxFloor), kGsDivisor);
        gs_sh = gs;
        if (blockIdx.x == 0) gs_out[0] = gs;
      }
    }
    ptx::cluster_sync();  // no CTA leaves while a peer may still read its maximum
  } else if (threadIdx.x == 0) {
    for (int w = 1; w < kOnePassThreads / 32; ++w) m = max(m, red[w]);
    atomicMax(&ws->amax_bits, m << 16);
    __threadfence();
    atomicAdd(&ws->done, 1u);
    // grid barrier: every CTA's maximum is in before gs is derived
    volatile uint32_t* arrived = &ws->done;
    const long long t0 = clock64();
    bool late = false;
    while (*arrived < gridDim.x) {
      if (clock64() - t0 > kBarrierCycles) {
        late = true;
        break;
      }
    }
    if (late) atomicOr(&ws->status, NVFP4_DEVICE_TIMEOUT);
    __threadfence();
    const uint32_t bits = atomicAdd(&ws->amax_bits, 0u);
    const float gs = __fdiv_rn(fmaxf(__uint_as_float(bits), kAmaxFloor), kGsDivisor);
    gs_sh = gs;
    if (blockIdx.x == 0) gs_out[0] = gs;
  }
  __syncthreads();
  fill_codec(tab, gs_sh);
  __syncthreads();
  const Codec sc = make_codec(gs_sh, tab);
  for (int64_t i = threadIdx.x; i < (late_load ? 0 : n_units); i += kOnePassThreads) {
    const int64_t u = u0 + i;
    if constexpr (G == 0) {
      uint32_t sbyte;
      uint2 codes;
      quantize_block(sv[2 * i], sv[2 * i + 1], sc, sbyte, codes);
      __stcs(reinterpret_cast<uint2*>(q) + u, codes);  // flat block index: [rows, cols/16]
      sf[u] = static_cast<uint8_t>(sbyte);
    } else {
      const int64_t inter = upr * 16;
      const int64_t r = u / upr, c = u % upr;
      uint32_t w[16];
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const uint4 t = sv[4 * i + v];
        w[4 * v] = t.x;
        w[4 * v + 1] = t.y;
        w[4 * v + 2] = t.z;
        w[4 * v + 3] = t.w;
      }
      uint32_t g[8], up[8];
      split_gate_up<G>(w, g, up);
      uint32_t sg, su;
      uint2 cg, cu;
      quantize_block(make_uint4(g[0], g[1], g[2], g[3]), make_uint4(g[4], g[5], g[6], g[7]), sc, sg, cg);
      quantize_block(make_uint4(up[0], up[1], up[2], up[3]), make_uint4(up[4], up[5], up[6], up[7]), sc, su,
                     cu);
      uint8_t* qrow = q + r * inter;
      __stcs(reinterpret_cast<uint2*>(qrow + c * 8), cg);
      __stcs(reinterpret_cast<uint2*>(qrow + inter / 2 + c * 8), cu);
      uint8_t* srow = sf + r * (inter / 8);
      srow[c] = static_cast<uint8_t>(sg);
      srow[inter / 16 + c] = static_cast<uint8_t>(su);
    }
  }
  // copies still in flight after a timeout get one more bounded wait
  if (late_load && threadIdx.x == 0) ptx::mbar_wait_bounded(bar_a, 0, &never, 2000000000LL);
  if constexpr (kCluster) return;
  __syncthreads();
  if (threadIdx.x == 0) {
    // Every CTA read the maximum before departing; the last one resets.
    if (atomicAdd(&ws->depart, 1u) == gridDim.x - 1) {
      atomicExch(&ws->amax_bits, 0u);
      atomicExch(&ws->done, 0u);
      atomicExch(&ws->depart, 0u);
    }
  }
}

// Launch the one-pass kernel if the input fits in the SMs' shared memory;
// false (nothing launched, no error left behind) otherwise.  Up to 512 KB a
// single cluster of up to 16 CTAs, beyond that a cooperative grid of one
// CTA per SM.
constexpr int64_t kClusterMaxBytes = 512 * 1024;

template <int G>
bool launch_onepass(const uint16_t* x, int64_t rows, int64_t upr, int64_t ld, uint8_t* q, uint8_t* sf,
                    float* gs, Workspace* ws, cudaStream_t stream, cudaError_t* err) {
  constexpr int64_t kUnitBytes = (G == 0 ? 16 : 32) * 2;
  const int64_t total = rows * upr;
  if (total == 0) return false;
  const int sms = sm_count();
  const int64_t max_units = kOnePassMaxBytes / kUnitBytes;
  if (total > max_units * sms) return false;
  const bool cluster = total * kUnitBytes <= kClusterMaxBytes;
  // at least 8 KB per CTA; one cluster of <= 16 CTAs, or at most one CTA per SM
  const int64_t min_units = 8192 / kUnitBytes;
  int64_t grid = (total + min_units - 1) / min_units;
  const int64_t cap = cluster ? 16 : sms;
  if (grid > cap) grid = cap;
  const int64_t per = (total + grid - 1) / grid;
  grid = (total + per - 1) / per;
  const size_t smem = static_cast<size_t>(per * kUnitBytes);
  auto kernel = cluster ? quantize_onepass_kernel<G, true> : quantize_onepass_kernel<G, false>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kOnePassMaxBytes)) != cudaSuccess ||
      (cluster && cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)) {
    cudaGetLastError();
    return false;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kOnePassThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  if (cluster) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(grid);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // the small cluster may start while the previous kernel finishes (the
    // kernel waits for it before touching global memory)
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
  } else {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = cluster ? 2 : 1;
  if (cluster) {
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n < 1) {
      cudaGetLastError();
      return false;
    }
  }
  count_launch();
  *err = cudaLaunchKernelEx(&cfg, kernel, x, rows, upr, ld, per, q, sf, gs, ws);
  return true;
}

// ---------------------------------------------------------------- RMSNorm + quantize

// The quantize input produced by an RMSNorm: y = bf16((x * inv_rms) * w[c])
// with inv_rms = 1 / sqrt(sum(x^2) / cols + eps), fused so that y never
// reaches HBM (the compare view's PERFORMANCE_AUDIT.md P4).  The sum of
// squares has no order: it is the exact sum rounded once to FP32.
//
// Exact sum.  A finite bf16 value is M * 2^q (M < 256 an integer, q =
// max(E, 1) - 134 from its exponent field E), so relative to the row's
// largest exponent Emax an element with d = Emax' - E' <= 17 (primes: at
// least 1) is the integer a = M << (17 - d) < 2^25 in units of
// 2^(qmax - 17), and its square a^2 < 2^50 is exact in a 64-bit sum of up to
// 2^14 terms.  Window w >= 1 holds the elements with 17w < d <= 17w + 17 in
// units 2^-17w smaller.  Windows 0 and 1 cover almost every row; what lies
// below them can only set the sticky bit of the rounding, unless window 1's
// low bits sit so close to a carry that the lower windows could cross it,
// in which case every window is summed (a slow pass per window, rare).
constexpr int kWinBits = 17;         // exponent steps per window; squares gain 34 bits
constexpr uint64_t kLow34 = (1ull << 34) - 1;

// Add the square of one bf16 value (bits h, exponent field e) to windows 0
// and 1, or flag it as lying below them.
__device__ __forceinline__ void sq_windows(uint32_t h, int emax, uint64_t& w0, uint64_t& w1, uint32_t& below) {
  const uint32_t e = (h >> 7) & 0xFFu;
  const uint32_t m = (h & 0x7Fu) | (e != 0 ? 0x80u : 0u);
  const int d = emax - max(static_cast<int>(e), 1);
  const bool in0 = d <= kWinBits, in1 = !in0 && d <= 2 * kWinBits;
  const uint32_t a = (in0 || in1) ? m << (in0 ? kWinBits - d : 2 * kWinBits - d) : 0u;
  const uint64_t sq = static_cast<uint64_t>(a) * a;
  w0 += in0 ? sq : 0ull;
  w1 += in1 ? sq : 0ull;
  below |= (in0 || in1) ? 0u : m;
}

// Shifts with PTX semantics: an amount of 32 or more (a negative int
// passed as unsigned) gives 0.
__device__ __forceinline__ uint32_t shl_sat(uint32_t v, uint32_t s) {
  uint32_t r;
  asm("shl.b32 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(s));
  return r;
}
__device__ __forceinline__ uint32_t shr_sat(uint32_t v, uint32_t s) {
  uint32_t r;
  asm("shr.b32 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(s));
  return r;
}

// Rows whose nonzero elements span at most two windows (d <= 34 for all):
// with s0 = e' + 17 - Emax' (e' = max(E, 1)), window 0 takes m << s0
// (s0 >= 0) and window 1 takes m << (s0 + 17) (s0 < 0), both written as
// clamped shifts so that each element lands in exactly one window with no
// selects; m = |h| + 128 - 128 e' is the significand with its hidden bit.
// kTwo = false: every element is in window 0 (span <= 17).
template <bool kTwo>
__device__ __forceinline__ void sq_fast(uint32_t h, int c0, uint64_t& w0, uint64_t& w1) {
  const uint32_t u = h & 0x7FFFu;
  const uint32_t ep = max(u >> 7, 1u);
  const uint32_t m = u + 128u - (ep << 7);
  const int s0 = static_cast<int>(ep) + c0;
  const uint32_t a0 = shl_sat(m, static_cast<uint32_t>(s0));
  w0 += static_cast<uint64_t>(a0) * a0;
  if constexpr (kTwo) {
    const uint32_t a1 = shr_sat(m << 16, static_cast<uint32_t>(-1 - s0));
    w1 += static_cast<uint64_t>(a1) * a1;
  }
}

template <bool kTwo>
__device__ __forceinline__ void sq_fast_rows(const uint4* v, int nv, int lane, int c0, uint64_t& w0, uint64_t& w1) {
  uint64_t x0 = 0, x1 = 0;  // a second pair of sums: two independent accumulation chains
  for (int i = lane; i < nv; i += 32) {
    const uint4 t = v[i];
    sq_fast<kTwo>(t.x & 0xFFFFu, c0, w0, w1);
    sq_fast<kTwo>(t.x >> 16, c0, x0, x1);
    sq_fast<kTwo>(t.y & 0xFFFFu, c0, w0, w1);
    sq_fast<kTwo>(t.y >> 16, c0, x0, x1);
    sq_fast<kTwo>(t.z & 0xFFFFu, c0, w0, w1);
    sq_fast<kTwo>(t.z >> 16, c0, x0, x1);
    sq_fast<kTwo>(t.w & 0xFFFFu, c0, w0, w1);
    sq_fast<kTwo>(t.w >> 16, c0, x0, x1);
  }
  w0 += x0;
  w1 += x1;
}

// Window w alone (slow pass): the squares of the elements with
// 17w < d <= 17w + 17 (w = 0: d <= 17), in that window's units.
__device__ __forceinline__ uint64_t sq_window(uint32_t h, int emax, int w) {
  const uint32_t e = (h >> 7) & 0xFFu;
  const uint32_t m = (h & 0x7Fu) | (e != 0 ? 0x80u : 0u);
  const int d = emax - max(static_cast<int>(e), 1);
  const int wd = d == 0 ? 0 : (d - 1) / kWinBits;
  const uint32_t a = wd == w ? m << (kWinBits * (w + 1) - d) : 0u;
  return static_cast<uint64_t>(a) * a;
}

__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// v * 2^e for a v whose product is on the FP32 grid (or beyond its range,
// giving inf), by multiplications with normal powers of two.
__device__ __forceinline__ float scale_pow2(float v, int e) {
  auto pow2 = [](int k) { return __int_as_float((k + 127) << 23); };  // -126 <= k <= 127
  if (e > 127) {
    v = __fmul_rn(v, pow2(127));
    e -= 127;
    if (e > 127) e = 127;  // the product is past FP32's range already
  } else if (e < -126) {
    v = __fmul_rn(v, pow2(-100));
    e += 100;
  }
  return __fmul_rn(v, pow2(e));
}

// FP32 nearest (top + t) * 2^e0 for an integer top >= 2^34 and 0 <= t < 1,
// where sticky says whether t > 0 (ties to even).
__device__ __forceinline__ float round_sum(uint64_t top, bool sticky, int e0) {
  const int h = 63 - __clzll(static_cast<long long>(top));
  const int p = max(h - 23, -149 - e0);  // lowest kept bit: 24 bits, or FP32's 2^-149 step
  if (p >= 64) return 0.0f;              // top * 2^e0 < 2^-150: nearest is zero
  const uint64_t keep = top >> p;
  const uint64_t rem = top & ((1ull << p) - 1ull);
  const uint64_t half = 1ull << (p - 1);  // p >= 11 (h >= 34)
  const bool up = rem > half || (rem == half && (sticky || (keep & 1ull)));
  return scale_pow2(static_cast<float>(keep + (up ? 1ull : 0ull)), p + e0);
}

// The FP32 sum of squares of one bf16 row (global or shared memory), one
// warp; every lane returns it.  cols is a multiple of 16.
__device__ float warp_sum_sq_exact(const uint16_t* xr, int64_t cols) {
  const int lane = static_cast<int>(threadIdx.x & 31);
  const uint4* v = reinterpret_cast<const uint4*>(xr);
  const int nv = static_cast<int>(cols / 8);
  // the largest |h| and the smallest nonzero |h| (zeros wrap to 0xFFFF in
  // the 16-bit subtraction and drop out of the minimum)
  uint32_t m2 = 0, n2 = 0xFFFFFFFFu;
  for (int i = lane; i < nv; i += 32) {
    const uint4 t = v[i];
    m2 = __vmaxu2(m2, absmax8(t));
    const uint32_t k = 0x7FFF7FFFu, one = 0x00010001u;
    n2 = __vminu2(n2, __vminu2(__vminu2(__vsub2(t.x & k, one), __vsub2(t.y & k, one)),
                               __vminu2(__vsub2(t.z & k, one), __vsub2(t.w & k, one))));
  }
  uint32_t mb = fold16(m2), nb = min(n2 & 0xFFFFu, n2 >> 16);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, o));
    nb = min(nb, __shfl_xor_sync(0xFFFFFFFFu, nb, o));
  }
  if (mb == 0) return 0.0f;
  const int emax = max(static_cast<int>(mb >> 7), 1);
  const int emin = max(static_cast<int>((nb + 1) >> 7), 1);  // exponent of the smallest nonzero |x|
  const int e0 = 2 * (emax - 134) - 2 * kWinBits;  // window 0's unit: 2^e0
  uint64_t w0 = 0, w1 = 0;
  if (emax - emin <= 2 * kWinBits) {
    // nothing below window 1: the two windows are the exact sum
    if (emax - emin <= kWinBits) sq_fast_rows<false>(v, nv, lane, kWinBits - emax, w0, w1);
    else sq_fast_rows<true>(v, nv, lane, kWinBits - emax, w0, w1);
    w0 = warp_sum_u64(w0);
    w1 = warp_sum_u64(w1);
    return round_sum(w0 + (w1 >> 34), (w1 & kLow34) != 0, e0);
  }
  uint32_t below = 0;
  for (int i = lane; i < nv; i += 32) {
    const uint4 t = v[i];
    const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      sq_windows(w[j] & 0xFFFFu, emax, w0, w1, below);
      sq_windows(w[j] >> 16, emax, w0, w1, below);
    }
  }
  w0 = warp_sum_u64(w0);
  w1 = warp_sum_u64(w1);
  below = __reduce_or_sync(0xFFFFFFFFu, below);
  // The windows below window 1 add less than 2^30 of window 1's units.
  if (below == 0 || (w1 & kLow34) < kLow34 + 1 - (1ull << 30))
    return round_sum(w0 + (w1 >> 34), (w1 & kLow34) != 0 || below != 0, e0);
  // Every window, from the bottom up: carry the whole part, keep the rest as sticky.
  const int n_win = (emax - 1) / kWinBits + 1;
  uint64_t carry = 0;
  bool sticky = false;
  for (int wi = n_win - 1; wi >= 0; --wi) {
    uint64_t acc = 0;
    for (int i = lane; i < nv; i += 32) {
      const uint4 t = v[i];
      const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) acc += sq_window(w[j] & 0xFFFFu, emax, wi) + sq_window(w[j] >> 16, emax, wi);
    }
    const uint64_t tot = warp_sum_u64(acc) + carry;
    if (wi == 0) return round_sum(tot, sticky, e0);
    sticky = sticky || (tot & kLow34) != 0;
    carry = tot >> 34;
  }
  return 0.0f;  // not reached
}

// inv_rms of one bf16 row, one warp (every lane gets it).
__device__ float warp_inv_rms(const uint16_t* xr, int64_t cols, float eps) {
  const float sum = warp_sum_sq_exact(xr, cols);
  const float mean = __fdiv_rn(sum, static_cast<float>(cols));
  return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
}

// bf16 bits of (x * inv) * w, round to nearest even, for the two halves of a word.
__device__ __forceinline__ uint32_t rms_word(uint32_t xw, uint32_t ww, float inv) {
  const float ylo = __fmul_rn(__fmul_rn(lo_bf16(xw), inv), lo_bf16(ww));
  const float yhi = __fmul_rn(__fmul_rn(hi_bf16(xw), inv), hi_bf16(ww));
  return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(ylo))) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(yhi))) << 16);
}

__device__ __forceinline__ uint4 rms_vec(uint4 x, uint4 w, float inv) {
  return make_uint4(rms_word(x.x, w.x, inv), rms_word(x.y, w.y, inv), rms_word(x.z, w.z, inv),
                    rms_word(x.w, w.w, inv));
}

// mHC pre-mix of one token (the layer input before the norm): x_in[c] =
// bf16(sum_i A[i] X_i[c]), FP32 accumulation over the streams in index order
// (each bf16 product is exact in FP32).  One warp, 8 elements per lane step;
// streams i at src + i * cols, result to dst (may alias stream 0: each lane
// reads its own vector of every stream before it writes it).
__device__ __forceinline__ void warp_mhc_mix(const uint16_t* src, int64_t cols, int n_hc, const uint16_t* a,
                                             uint16_t* dst) {
  const int lane = static_cast<int>(threadIdx.x & 31);
  float av[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    av[i] = 0.0f;
    if (i < n_hc) av[i] = lo_bf16(static_cast<uint32_t>(__ldg(a + i)));
  }
  const int nv = static_cast<int>(cols / 8);
  for (int v = lane; v < nv; v += 32) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i < n_hc) {
        const uint4 w = reinterpret_cast<const uint4*>(src + i * cols)[v];
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float p0 = __fmul_rn(av[i], lo_bf16(ww[j])), p1 = __fmul_rn(av[i], hi_bf16(ww[j]));
          acc[2 * j] = i == 0 ? p0 : __fadd_rn(acc[2 * j], p0);
          acc[2 * j + 1] = i == 0 ? p1 : __fadd_rn(acc[2 * j + 1], p1);
        }
      }
    }
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      o[j] = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * j]))) |
             (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * j + 1]))) << 16);
    reinterpret_cast<uint4*>(dst)[v] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  __syncwarp();
}

// ---- two passes (inputs larger than the SMs' shared memory): one CTA per row at a time
//
// Thread t of the CTA (NT threads) holds the row's 16-element blocks
// b = t + j NT (j < J) in registers: it loads them (with the mix, each stream's, summed
// in stream order), the CTA reduces the row's maximum and smallest nonzero
// |x|, then the exact sum of squares (two windows, or every window for rows
// of a very wide range), and every thread normalises its blocks.  Both passes
// recompute the row the same way, so the second quantizes exactly what the
// first measured.
constexpr int kRowWarpsMax = 16;
constexpr int kBlockRowsMax = 6;  // one-pass kernel: up to this many rows per CTA, all threads per row

struct RowScratch {
  uint32_t mx[kRowWarpsMax], mn[kRowWarpsMax], below[kRowWarpsMax];
  unsigned long long w0[kRowWarpsMax], w1[kRowWarpsMax];
};

// Sum over the CTA of two 64-bit values (and an OR of a flag); every thread
// gets the totals.  One barrier; the caller's next use of the same fields
// comes after another barrier.
template <int NT>
__device__ __forceinline__ void block_sum2(uint64_t& a, uint64_t& b, uint32_t& f, RowScratch& sc) {
  const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
  a = warp_sum_u64(a);
  b = warp_sum_u64(b);
  f = __reduce_or_sync(0xFFFFFFFFu, f);
  if (lane == 0) {
    sc.w0[warp] = a;
    sc.w1[warp] = b;
    sc.below[warp] = f;
  }
  __syncthreads();
  a = 0;
  b = 0;
  f = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    a += sc.w0[w];
    b += sc.w1[w];
    f |= sc.below[w];
  }
}

// Loads of a row's 16-byte vectors: global memory (read-only path) or shared.
template <bool kShared>
__device__ __forceinline__ uint4 ld_row(const uint16_t* p) {
  if constexpr (kShared) return *reinterpret_cast<const uint4*>(p);
  else return __ldg(reinterpret_cast<const uint4*>(p));
}

// y = bf16((x * inv_rms) * w) of this thread's blocks of row r (x: the
// row, or with the mix the token's first stream, streams cols apart; in
// global memory, or shared with kShared).
template <int NT, int J, bool kMix, bool kShared = false>
__device__ __forceinline__ void block_row_norm(const uint16_t* __restrict__ xr, int64_t cols,
                                               const uint16_t* __restrict__ wt, float eps,
                                               const uint16_t* __restrict__ arow, int n_hc, RowScratch& sc,
                                               uint4 (&y)[J][2]) {
  const int t = static_cast<int>(threadIdx.x), warp = t >> 5, lane = t & 31;
  const int nb = static_cast<int>(cols / 16);
  uint4 x[J][2];
  if constexpr (kMix) {
    float acc[J][16];
    // streams four at a time, all of their loads issued before the
    // arithmetic (an index past n_hc re-reads stream 0 and is not used)
#pragma unroll
    for (int i0 = 0; i0 < 8; i0 += 4) {
      if (i0 < n_hc) {
        uint4 v[4][J][2];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i0 + u < n_hc ? i0 + u : 0;
#pragma unroll
          for (int j = 0; j < J; ++j) {
            const int b = t + j * NT;
#pragma unroll
            for (int h = 0; h < 2; ++h)
              v[u][j][h] = b < nb ? ld_row<kShared>(xr + i * cols + b * 16 + h * 8) : make_uint4(0, 0, 0, 0);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i0 + u;
          if (i < n_hc) {
            const float ai = lo_bf16(static_cast<uint32_t>(__ldg(arow + i)));
#pragma unroll
            for (int j = 0; j < J; ++j)
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const uint32_t ww[4] = {v[u][j][h].x, v[u][j][h].y, v[u][j][h].z, v[u][j][h].w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const float p0 = __fmul_rn(ai, lo_bf16(ww[k])), p1 = __fmul_rn(ai, hi_bf16(ww[k]));
                  float& s0 = acc[j][h * 8 + 2 * k];
                  float& s1 = acc[j][h * 8 + 2 * k + 1];
                  s0 = i == 0 ? p0 : __fadd_rn(s0, p0);
                  s1 = i == 0 ? p1 : __fadd_rn(s1, p1);
                }
              }
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < J; ++j)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          o[k] = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc[j][h * 8 + 2 * k]))) |
                 (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc[j][h * 8 + 2 * k + 1]))) << 16);
        x[j][h] = make_uint4(o[0], o[1], o[2], o[3]);
      }
  } else {
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int b = t + j * NT;
#pragma unroll
      for (int h = 0; h < 2; ++h)
        x[j][h] = b < nb ? ld_row<kShared>(xr + b * 16 + h * 8) : make_uint4(0, 0, 0, 0);
    }
  }
  // the row's largest |h| and smallest nonzero |h| (blocks past the row are zeros)
  uint32_t m2 = 0, n2 = 0xFFFFFFFFu;
#pragma unroll
  for (int j = 0; j < J; ++j)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 v = x[j][h];
      m2 = __vmaxu2(m2, absmax8(v));
      const uint32_t k = 0x7FFF7FFFu, one = 0x00010001u;
      n2 = __vminu2(n2, __vminu2(__vminu2(__vsub2(v.x & k, one), __vsub2(v.y & k, one)),
                                 __vminu2(__vsub2(v.z & k, one), __vsub2(v.w & k, one))));
    }
  uint32_t mb = fold16(m2), nm = min(n2 & 0xFFFFu, n2 >> 16);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, o));
    nm = min(nm, __shfl_xor_sync(0xFFFFFFFFu, nm, o));
  }
  if (lane == 0) {
    sc.mx[warp] = mb;
    sc.mn[warp] = nm;
  }
  __syncthreads();
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    mb = max(mb, sc.mx[w]);
    nm = min(nm, sc.mn[w]);
  }
  float sum = 0.0f;
  if (mb != 0) {
    const int emax = max(static_cast<int>(mb >> 7), 1);
    const int emin = max(static_cast<int>((nm + 1) >> 7), 1);
    const int e0 = 2 * (emax - 134) - 2 * kWinBits;  // window 0's unit: 2^e0
    uint64_t w0 = 0, w1 = 0;
    uint32_t below = 0;
    if (emax - emin <= 2 * kWinBits) {  // nothing below window 1
#pragma unroll
      for (int j = 0; j < J; ++j)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t ww[4] = {x[j][h].x, x[j][h].y, x[j][h].z, x[j][h].w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            sq_fast<true>(ww[k] & 0xFFFFu, kWinBits - emax, w0, w1);
            sq_fast<true>(ww[k] >> 16, kWinBits - emax, w0, w1);
          }
        }
      block_sum2<NT>(w0, w1, below, sc);
      sum = round_sum(w0 + (w1 >> 34), (w1 & kLow34) != 0, e0);
    } else {
#pragma unroll
      for (int j = 0; j < J; ++j)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t ww[4] = {x[j][h].x, x[j][h].y, x[j][h].z, x[j][h].w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            sq_windows(ww[k] & 0xFFFFu, emax, w0, w1, below);
            sq_windows(ww[k] >> 16, emax, w0, w1, below);
          }
        }
      block_sum2<NT>(w0, w1, below, sc);
      if (below == 0 || (w1 & kLow34) < kLow34 + 1 - (1ull << 30)) {
        sum = round_sum(w0 + (w1 >> 34), (w1 & kLow34) != 0 || below != 0, e0);
      } else {
        // every window, from the bottom up (rare: a carry may cross window 1)
        const int n_win = (emax - 1) / kWinBits + 1;
        uint64_t carry = 0;
        bool sticky = false;
        for (int wi = n_win - 1; wi >= 0; --wi) {
          __syncthreads();  // the previous totals have been read
          uint64_t acc = 0, none = 0;
          uint32_t nf = 0;
#pragma unroll
          for (int j = 0; j < J; ++j)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint32_t ww[4] = {x[j][h].x, x[j][h].y, x[j][h].z, x[j][h].w};
#pragma unroll
              for (int k = 0; k < 4; ++k) acc += sq_window(ww[k] & 0xFFFFu, emax, wi) + sq_window(ww[k] >> 16, emax, wi);
            }
          block_sum2<NT>(acc, none, nf, sc);
          const uint64_t tot = acc + carry;
          if (wi == 0) {
            sum = round_sum(tot, sticky, e0);
          } else {
            sticky = sticky || (tot & kLow34) != 0;
            carry = tot >> 34;
          }
        }
      }
    }
  }
  const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(sum, static_cast<float>(cols)), eps)));
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int b = t + j * NT;
    const uint4* wv = reinterpret_cast<const uint4*>(wt + (b < nb ? b : 0) * 16);
    y[j][0] = rms_vec(x[j][0], __ldg(wv), inv);
    y[j][1] = rms_vec(x[j][1], __ldg(wv + 1), inv);
  }
}

// This CTA's rows r = blockIdx.x + k gridDim.x, each normalised (y into f).
// With row_bytes != 0 the rows come through two shared-memory buffers: the
// next row's bulk copy is in flight while a row is processed.  Returns false
// if a copy did not land in time (NVFP4_DEVICE_TIMEOUT is recorded).
template <int NT, int J, bool kMix, typename F>
__device__ __forceinline__ bool for_rows(const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t ld,
                                         const uint16_t* __restrict__ wt, float eps,
                                         const uint16_t* __restrict__ amap, int n_hc, uint32_t row_bytes,
                                         uint8_t* buf, uint64_t* bars, RowScratch& sc, uint32_t* status, F f) {
  if (row_bytes == 0) {
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
      uint4 y[J][2];
      block_row_norm<NT, J, kMix>(x + r * ld, cols, wt, eps, amap + r * n_hc, n_hc, sc, y);
      f(r, y);
    }
    return true;
  }
  const uint32_t bar[2] = {ptx::smem_addr(&bars[0]), ptx::smem_addr(&bars[1])};
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar[0], 1);
    ptx::mbar_init(bar[1], 1);
    ptx::fence_mbar_init();
    if (static_cast<int64_t>(blockIdx.x) < rows) {
      ptx::mbar_arrive_expect_tx(bar[0], row_bytes);
      ptx::bulk_load(ptx::smem_addr(buf), x + static_cast<int64_t>(blockIdx.x) * ld, row_bytes, bar[0]);
    }
  }
  __syncthreads();
  uint32_t never = 0;
  int it = 0;
  int64_t issued = blockIdx.x;  // the last row whose copy was issued
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x, ++it) {
    const int cur = it & 1;
    const int64_t rn = r + gridDim.x;
    if (threadIdx.x == 0 && rn < rows) {
      // the other buffer was read in the previous row, before its barriers
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive_expect_tx(bar[cur ^ 1], row_bytes);
      ptx::bulk_load(ptx::smem_addr(buf + (cur ^ 1) * row_bytes), x + rn * ld, row_bytes, bar[cur ^ 1]);
    }
    if (rn < rows) issued = rn;
    const bool late = __syncthreads_or(!ptx::mbar_wait_bounded(bar[cur], (it >> 1) & 1, &never, 2000000000LL)) != 0;
    if (late) {
      if (threadIdx.x == 0) {
        atomicOr(status, NVFP4_DEVICE_TIMEOUT);
        // let the copies in flight land before the CTA can exit
        ptx::mbar_wait_bounded(bar[cur], (it >> 1) & 1, &never, 2000000000LL);
        if (issued == rn) ptx::mbar_wait_bounded(bar[cur ^ 1], ((it + 1) >> 1) & 1, &never, 2000000000LL);
      }
      return false;
    }
    uint4 y[J][2];
    block_row_norm<NT, J, kMix, true>(reinterpret_cast<const uint16_t*>(buf + cur * row_bytes), cols, wt, eps,
                                      amap + r * n_hc, n_hc, sc, y);
    f(r, y);
  }
  return true;
}

// Pass 1: y's maximum |.|, then gs by the last block, exactly as the amax kernel does.
template <int NT, int J, bool kMix>
__global__ void __launch_bounds__(NT, 512 / NT)
    rmsnorm_amax_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t ld,
                        const uint16_t* __restrict__ wt, float eps, const uint16_t* __restrict__ amap, int n_hc,
                        uint32_t row_bytes, float* __restrict__ gs_out, Workspace* __restrict__ ws) {
  ptx::pdl_launch_dependents();
  extern __shared__ __align__(128) uint8_t rowbuf[];
  __shared__ RowScratch sc;
  __shared__ __align__(8) uint64_t bars[2];
  const int nb = static_cast<int>(cols / 16);
  uint32_t m2 = 0;
  for_rows<NT, J, kMix>(x, rows, cols, ld, wt, eps, amap, n_hc, row_bytes, rowbuf, bars, sc, &ws->status,
                        [&](int64_t, const uint4 (&y)[J][2]) {
#pragma unroll
                          for (int j = 0; j < J; ++j)
                            if (static_cast<int>(threadIdx.x) + j * NT < nb)
                              m2 = __vmaxu2(m2, __vmaxu2(absmax8(y[j][0]), absmax8(y[j][1])));
                        });
  uint32_t m = fold16(m2);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  __syncthreads();  // the last row's scratch has been read
  if ((threadIdx.x & 31) == 0) sc.mx[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < NT / 32; ++w) m = max(m, sc.mx[w]);
    atomicMax(&ws->amax_bits, m << 16);
    __threadfence();
    const uint32_t ticket = atomicAdd(&ws->done, 1u);
    if (ticket == gridDim.x - 1) {
      const uint32_t bits = atomicAdd(&ws->amax_bits, 0u);
      gs_out[0] = __fdiv_rn(fmaxf(__uint_as_float(bits), kAmaxFloor), kGsDivisor);
      ws->amax_bits = 0;
      ws->done = 0;
    }
  }
}

// Pass 2: recompute each row (same values) and quantize y.
template <int NT, int J, bool kMix>
__global__ void __launch_bounds__(NT, 512 / NT)
    rmsnorm_quantize_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t ld,
                            const uint16_t* __restrict__ wt, float eps, const uint16_t* __restrict__ amap,
                            int n_hc, uint32_t row_bytes, uint8_t* __restrict__ q, uint8_t* __restrict__ sf,
                            const float* __restrict__ gs_ptr, uint32_t* __restrict__ status) {
  ptx::pdl_launch_dependents();
  extern __shared__ __align__(128) uint8_t rowbuf[];
  __shared__ RowScratch sc;
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ float2 tab[128];
  const int nb = static_cast<int>(cols / 16);
  const float gs = __ldg(gs_ptr);
  fill_codec(tab, gs);
  __syncthreads();
  const Codec cd = make_codec(gs, tab);
  for_rows<NT, J, kMix>(x, rows, cols, ld, wt, eps, amap, n_hc, row_bytes, rowbuf, bars, sc, status,
                        [&](int64_t r, const uint4 (&y)[J][2]) {
#pragma unroll
                          for (int j = 0; j < J; ++j) {
                            const int b = static_cast<int>(threadIdx.x) + j * NT;
                            if (b < nb) {
                              uint32_t sbyte;
                              uint2 codes;
                              quantize_block(y[j][0], y[j][1], cd, sbyte, codes);
                              const int64_t blk = r * nb + b;
                              __stcs(reinterpret_cast<uint2*>(q) + blk, codes);
                              sf[blk] = static_cast<uint8_t>(sbyte);
                            }
                          }
                        });
}

// One pass for inputs that fit in the SMs' shared memory: each CTA holds
// whole rows and normalises them in place (y replaces x) -- a few rows one
// after the other with all its threads on each (the scheme of the two-pass
// kernels, from shared memory), more rows one warp each -- the CTAs exchange
// maxima as in
// quantize_onepass_kernel (one cluster, or a cooperative grid meeting at the
// workspace counter), then each CTA quantizes its rows from shared memory.
// kMix: each token's n_hc streams are copied on chip and mixed (mHC
// pre-mix) into the first stream's buffer before the norm.
template <bool kCluster, bool kMix, int J>
__global__ void __launch_bounds__(kOnePassThreads, 1)
    rmsnorm_quantize_onepass_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t ld,
                                    const uint16_t* __restrict__ wt, float eps, const uint16_t* __restrict__ amap,
                                    int n_hc, int64_t rows_per_cta, uint8_t* __restrict__ q,
                                    uint8_t* __restrict__ sf, float* __restrict__ gs_out,
                                    Workspace* __restrict__ ws) {
  ptx::pdl_launch_dependents();
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t red[kOnePassThreads / 32];
  __shared__ float gs_sh;
  __shared__ float2 tab[128];
  constexpr int kWarpsOp = kOnePassThreads / 32;
  const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
  const int nb = static_cast<int>(cols / 16);
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * rows_per_cta;
  const int64_t r1 = r0 + rows_per_cta < rows ? r0 + rows_per_cta : rows;
  const int64_t n_rows = r1 > r0 ? r1 - r0 : 0;
  const int64_t row_elems = kMix ? n_hc * cols : cols;  // shared-memory row: the token's streams
  const uint32_t row_bytes = static_cast<uint32_t>(row_elems * 2);
  uint16_t* data = reinterpret_cast<uint16_t*>(smem);
  const uint32_t bar_a = ptx::smem_addr(&bar);
  ptx::pdl_wait();
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar_a, 1);
    ptx::fence_mbar_init();
    ptx::mbar_arrive_expect_tx(bar_a, static_cast<uint32_t>(n_rows) * row_bytes);
    for (int64_t r = r0; r < r1; ++r)  // one copy per row (rows may be strided)
      ptx::bulk_load(ptx::smem_addr(data) + static_cast<uint32_t>((r - r0) * row_bytes), x + r * ld, row_bytes,
                     bar_a);
  }
  __syncthreads();
  uint32_t never = 0;
  // as in quantize_onepass_kernel: a late slice adds nothing and writes nothing
  const bool late_load = __syncthreads_or(!ptx::mbar_wait_bounded(bar_a, 0, &never, 2000000000LL)) != 0;
  if (late_load && threadIdx.x == 0) atomicOr(&ws->status, NVFP4_DEVICE_TIMEOUT);
  const int64_t n_rows_live = late_load ? 0 : n_rows;
  __shared__ RowScratch rsc;
  uint32_t m2 = 0;
  if (n_rows_live > kBlockRowsMax) {
    // many rows: one warp per row, the rows side by side
    for (int64_t rr = warp; rr < n_rows_live; rr += kWarpsOp) {
      uint16_t* yr = data + rr * row_elems;
      if constexpr (kMix) warp_mhc_mix(yr, cols, n_hc, amap + (r0 + rr) * n_hc, yr);
      const float inv = warp_inv_rms(yr, cols, eps);
      for (int b = lane; b < nb; b += 32) {
        uint4* v = reinterpret_cast<uint4*>(yr + b * 16);
        const uint4* wv = reinterpret_cast<const uint4*>(wt + b * 16);
        const uint4 y0 = rms_vec(v[0], __ldg(wv), inv), y1 = rms_vec(v[1], __ldg(wv + 1), inv);
        v[0] = y0;  // y replaces x: only this lane touches this block
        v[1] = y1;
        m2 = __vmaxu2(m2, __vmaxu2(absmax8(y0), absmax8(y1)));
      }
    }
  }
  // few rows: all the CTA's threads on each row in turn
  for (int64_t rr = 0; n_rows_live <= kBlockRowsMax && rr < n_rows_live; ++rr) {
    uint16_t* yr = data + rr * row_elems;
    uint4 y[J][2];
    block_row_norm<kOnePassThreads, J, kMix, true>(yr, cols, wt, eps, amap + (r0 + rr) * n_hc, n_hc, rsc, y);
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int b = static_cast<int>(threadIdx.x) + j * kOnePassThreads;
      if (b < nb) {  // y replaces x: only this thread touches block b (of every stream)
        reinterpret_cast<uint4*>(yr + b * 16)[0] = y[j][0];
        reinterpret_cast<uint4*>(yr + b * 16)[1] = y[j][1];
        m2 = __vmaxu2(m2, __vmaxu2(absmax8(y[j][0]), absmax8(y[j][1])));
      }
    }
  }
  uint32_t m = fold16(m2);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if (lane == 0) red[warp] = m;
  __syncthreads();
  if constexpr (kCluster) {
    __shared__ float cta_max;
    if (threadIdx.x == 0) {
      for (int w = 1; w < kWarpsOp; ++w) m = max(m, red[w]);
      cta_max = __uint_as_float(m << 16);
    }
    ptx::cluster_sync();
    if (threadIdx.x < 32) {
      // lane r reads CTA r's maximum (the reads overlap), then a warp max
      const uint32_t r = threadIdx.x;
      float mx = r < gridDim.x ? ptx::ld_cluster_f32(ptx::mapa_shared(ptx::smem_addr(&cta_max), r)) : 0.0f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
      if (threadIdx.x == 0) {
        const float gs = __fdiv_rn(fmaxf(mx, kAmaxFloor), kGsDivisor);
        gs_sh = gs;
        if (blockIdx.x == 0) gs_out[0] = gs;
      }
    }
    ptx::cluster_sync();  // no CTA leaves while a peer may still read its maximum
  } else if (threadIdx.x == 0) {
    for (int w = 1; w < kWarpsOp; ++w) m = max(m, red[w]);
    atomicMax(&ws->amax_bits, m << 16);
    __threadfence();
    atomicAdd(&ws->done, 1u);
    volatile uint32_t* arrived = &ws->done;
    const long long t0 = clock64();
    bool late = false;
    while (*arrived < gridDim.x) {
      if (clock64() - t0 > kBarrierCycles) {
        late = true;
        break;
      }
    }
    if (late) atomicOr(&ws->status, NVFP4_DEVICE_TIMEOUT);
    __threadfence();
    const uint32_t bits = atomicAdd(&ws->amax_bits, 0u);
    const float gs = __fdiv_rn(fmaxf(__uint_as_float(bits), kAmaxFloor), kGsDivisor);
    gs_sh = gs;
    if (blockIdx.x == 0) gs_out[0] = gs;
  }
  __syncthreads();
  fill_codec(tab, gs_sh);
  __syncthreads();
  const Codec sc = make_codec(gs_sh, tab);
  const uint4* sv = reinterpret_cast<const uint4*>(data);
  const int64_t n_blocks = n_rows_live * nb;
  for (int64_t i = threadIdx.x; i < n_blocks; i += kOnePassThreads) {
    uint32_t sbyte;
    uint2 codes;
    const int64_t rr = kMix ? i / nb : 0;
    const int64_t vi = kMix ? rr * (row_elems / 8) + 2 * (i - rr * nb) : 2 * i;  // the normalised row's block i
    quantize_block(sv[vi], sv[vi + 1], sc, sbyte, codes);
    const int64_t blk = r0 * nb + i;
    __stcs(reinterpret_cast<uint2*>(q) + blk, codes);
    sf[blk] = static_cast<uint8_t>(sbyte);
  }
  if (late_load && threadIdx.x == 0) ptx::mbar_wait_bounded(bar_a, 0, &never, 2000000000LL);
  if constexpr (kCluster) return;
  __syncthreads();
  if (threadIdx.x == 0) {
    if (atomicAdd(&ws->depart, 1u) == gridDim.x - 1) {
      atomicExch(&ws->amax_bits, 0u);
      atomicExch(&ws->done, 0u);
      atomicExch(&ws->depart, 0u);
    }
  }
}

// Launch RMSNorm + quantize: one pass when whole rows fit in the SMs'
// shared memory (one cluster up to 512 KB, else a cooperative grid of one
// CTA per SM), otherwise the two row-parallel passes.
// n_hc == 0: plain RMSNorm of the rows; n_hc >= 1: each row is first the
// mHC pre-mix of the token's n_hc streams (contiguous, cols apart) by amap.
template <bool kMix>
cudaError_t launch_rmsnorm_quantize_t(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                                      const uint16_t* wt, float eps, const uint16_t* amap, int n_hc, uint8_t* q,
                                      uint8_t* sf, float* gs, Workspace* ws, cudaStream_t stream) {
  const int64_t row_bytes = (kMix ? n_hc : 1) * cols * 2;  // on chip per token
  const int sms = sm_count();
  if (rows > 0) {
    const int64_t rows_cap = static_cast<int64_t>(kOnePassMaxBytes) / row_bytes;
    if (rows_cap >= 1 && rows <= rows_cap * sms) {
      const bool cluster = rows * row_bytes <= kClusterMaxBytes;
      const int64_t cap = cluster ? 16 : sms;
      int64_t grid = (rows * row_bytes + 8191) / 8192;
      if (grid > cap) grid = cap;
      if (grid > rows) grid = rows;
      int64_t per = (rows + grid - 1) / grid;
      if (per > rows_cap) per = rows_cap;
      grid = (rows + per - 1) / per;
      if (grid <= cap) {
        const size_t smem = static_cast<size_t>(per * row_bytes);
        // one 16-element block per thread per row (cols <= 8192; the mix always), else two
        auto kernel = cluster ? rmsnorm_quantize_onepass_kernel<true, kMix, 1> : rmsnorm_quantize_onepass_kernel<false, kMix, 1>;
        if constexpr (!kMix) {
          if (cols / 16 > kOnePassThreads)
            kernel = cluster ? rmsnorm_quantize_onepass_kernel<true, false, 2> : rmsnorm_quantize_onepass_kernel<false, false, 2>;
        }
        bool ok = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem)) == cudaSuccess;
        if (ok && cluster)
          ok = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
        cfg.blockDim = dim3(kOnePassThreads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[2];
        if (cluster) {
          attr[0].id = cudaLaunchAttributeClusterDimension;
          attr[0].val.clusterDim.x = static_cast<unsigned>(grid);
          attr[0].val.clusterDim.y = 1;
          attr[0].val.clusterDim.z = 1;
          attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
          attr[1].val.programmaticStreamSerializationAllowed = 1;
        } else {
          attr[0].id = cudaLaunchAttributeCooperative;
          attr[0].val.cooperative = 1;
        }
        cfg.attrs = attr;
        cfg.numAttrs = cluster ? 2 : 1;
        if (ok && cluster) {
          int n = 0;
          ok = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) == cudaSuccess && n >= 1;
        }
        if (ok) {
          count_launch();
          return cudaLaunchKernelEx(&cfg, kernel, x, rows, cols, ld, wt, eps, amap, n_hc, per, q, sf, gs, ws);
        }
        cudaGetLastError();  // fall through to the two passes
      }
    }
  }
  // two passes, one CTA per row at a time, the row's blocks in registers;
  // one 16-element block per thread (256 or 512 threads: cols <= 8192), else
  // two of 512 threads'.  Rows come through two shared-memory buffers
  // (the next row's bulk copy in flight) when two fit.
  const int nbk = static_cast<int>(cols / 16);
  const int variant = nbk <= 256 ? 0 : (nbk <= 512 ? 1 : 2);
  // (the mix takes cols <= 8192: variants 0 and 1)
  auto amax_k = variant == 0 ? rmsnorm_amax_kernel<256, 1, kMix> : rmsnorm_amax_kernel<512, 1, kMix>;
  auto quant_k = variant == 0 ? rmsnorm_quantize_kernel<256, 1, kMix> : rmsnorm_quantize_kernel<512, 1, kMix>;
  if constexpr (!kMix) {
    if (variant == 2) {
      amax_k = rmsnorm_amax_kernel<512, 2, false>;
      quant_k = rmsnorm_quantize_kernel<512, 2, false>;
    }
  }
  const unsigned nt = variant == 0 ? 256u : 512u;
  const uint32_t rb = static_cast<uint32_t>(row_bytes);
  const bool staged = 2 * row_bytes <= kOnePassMaxBytes;
  const size_t smem = staged ? 2 * static_cast<size_t>(rb) : 0;
  cudaError_t e = cudaSuccess;
  if (smem > 48 * 1024) {
    e = cudaFuncSetAttribute(amax_k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(quant_k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  // persistent: as many CTAs as can be resident, each walking its rows
  int per_sm = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, quant_k, static_cast<int>(nt), smem) != cudaSuccess ||
      per_sm < 1) {
    cudaGetLastError();
    per_sm = 1;
  }
  int64_t grid = static_cast<int64_t>(sms) * per_sm;
  if (grid > rows) grid = rows > 0 ? rows : 1;
  count_launch();
  amax_k<<<static_cast<unsigned>(grid), nt, smem, stream>>>(x, rows, cols, ld, wt, eps, amap, n_hc, staged ? rb : 0u,
                                                            gs, ws);
  e = cudaGetLastError();
  if (e != cudaSuccess || rows == 0) return e;
  count_launch();
  quant_k<<<static_cast<unsigned>(grid), nt, smem, stream>>>(x, rows, cols, ld, wt, eps, amap, n_hc,
                                                             staged ? rb : 0u, q, sf, gs, &ws->status);
  return cudaGetLastError();
}

int grid_for(int64_t work_items, int blocks_per_sm) {
  const int64_t need = (work_items + kThreads - 1) / kThreads;
  const int64_t cap = static_cast<int64_t>(sm_count()) * blocks_per_sm;
  int64_t g = need < cap ? need : cap;
  return static_cast<int>(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_rmsnorm_quantize(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                                    const uint16_t* weight, float eps, uint8_t* q, uint8_t* sf, float* gs,
                                    Workspace* ws, cudaStream_t stream) {
  return launch_rmsnorm_quantize_t<false>(x, rows, cols, ld, weight, eps, nullptr, 0, q, sf, gs, ws, stream);
}

cudaError_t launch_mhc_rmsnorm_quantize(const uint16_t* x, int64_t rows, int n_hc, int64_t cols, int64_t ld,
                                        const uint16_t* amap, const uint16_t* weight, float eps, uint8_t* q,
                                        uint8_t* sf, float* gs, Workspace* ws, cudaStream_t stream) {
  return launch_rmsnorm_quantize_t<true>(x, rows, cols, ld, weight, eps, amap, n_hc, q, sf, gs, ws, stream);
}

bool launch_quantize_onepass(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, uint8_t* q,
                             uint8_t* sf, float* gs, Workspace* ws, cudaStream_t stream, cudaError_t* err) {
  return launch_onepass<0>(x, rows, cols / 16, ld, q, sf, gs, ws, stream, err);
}

bool launch_deinterleave_onepass(const uint16_t* x, int64_t rows, int64_t inter, int g, uint8_t* q,
                                 uint8_t* sf, float* gs, Workspace* ws, cudaStream_t stream,
                                 cudaError_t* err) {
  const int64_t cpr = inter / 16;  // 32-element input chunks per row
  switch (g) {
    case 1: return launch_onepass<1>(x, rows, cpr, 2 * inter, q, sf, gs, ws, stream, err);
    case 2: return launch_onepass<2>(x, rows, cpr, 2 * inter, q, sf, gs, ws, stream, err);
    case 4: return launch_onepass<4>(x, rows, cpr, 2 * inter, q, sf, gs, ws, stream, err);
    case 8: return launch_onepass<8>(x, rows, cpr, 2 * inter, q, sf, gs, ws, stream, err);
    case 16: return launch_onepass<16>(x, rows, cpr, 2 * inter, q, sf, gs, ws, stream, err);
    default: return false;
  }
}

cudaError_t launch_amax(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, float* gs,
                        Workspace* ws, cudaStream_t stream) {
  const int64_t vpr = cols / 8;
  const int grid = grid_for((rows * vpr + kAmaxUnroll - 1) / kAmaxUnroll, 4);
  count_launch();
  amax_kernel<<<grid, kThreads, 0, stream>>>(x, rows, vpr, ld, gs, ws);
  return cudaGetLastError();
}

cudaError_t launch_quantize(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, uint8_t* q,
                            uint8_t* sf, const float* gs, cudaStream_t stream) {
  const int64_t bpr = cols / 16;
  if (rows * bpr == 0) return cudaSuccess;
  const int grid = grid_for((rows * bpr + 1) / 2, 4);
  count_launch();
  quantize_kernel<<<grid, kThreads, 0, stream>>>(x, rows, bpr, ld, q, sf, gs);
  return cudaGetLastError();
}

cudaError_t launch_deinterleave_quantize(const uint16_t* x, int64_t rows, int64_t inter, int g,
                                         uint8_t* q, uint8_t* sf, const float* gs,
                                         cudaStream_t stream) {
  const int64_t items = rows * (inter / 16);
  if (items == 0) return cudaSuccess;
  const int grid = grid_for(items, 4);
  count_launch();
  switch (g) {
    case 1: deinterleave_quantize_kernel<1><<<grid, kThreads, 0, stream>>>(x, rows, inter, q, sf, gs); break;
    case 2: deinterleave_quantize_kernel<2><<<grid, kThreads, 0, stream>>>(x, rows, inter, q, sf, gs); break;
    case 4: deinterleave_quantize_kernel<4><<<grid, kThreads, 0, stream>>>(x, rows, inter, q, sf, gs); break;
    case 8: deinterleave_quantize_kernel<8><<<grid, kThreads, 0, stream>>>(x, rows, inter, q, sf, gs); break;
    case 16: deinterleave_quantize_kernel<16><<<grid, kThreads, 0, stream>>>(x, rows, inter, q, sf, gs); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace nvfp4
