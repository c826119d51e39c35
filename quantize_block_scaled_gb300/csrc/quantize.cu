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
// Memory access: 16-byte vector loads of 8 bf16, one 16-element block (two
// vectors) per thread and iteration, 8-byte stores of the 8 packed code
// bytes, grid-stride loops over a grid sized to the SM count.

#include <cstdint>

#include "internal.h"

namespace nvfp4 {
namespace {

constexpr int kThreads = 256;
constexpr float kGsDivisor = 2688.0f;  // 6 (E2M1 max) * 448 (E4M3 max)
constexpr float kAmaxFloor = 1e-8f;

// First pass (amax): ordinary loads, so a tensor that fits in L2 is still
// there for the second pass.  Second pass: streaming loads (last use).
__device__ __forceinline__ uint4 ld_keep(const uint16_t* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}
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

__global__ void __launch_bounds__(kThreads)
    amax_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t vpr, int64_t ld,
                float* __restrict__ gs_out, Workspace* __restrict__ ws) {
  uint32_t m2 = 0;
  const int64_t total = rows * vpr;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (ld == vpr * 8) {
    for (; i + 3 * stride < total; i += 4 * stride) {
      const uint4 a = ld_keep(x + i * 8);
      const uint4 b = ld_keep(x + (i + stride) * 8);
      const uint4 c = ld_keep(x + (i + 2 * stride) * 8);
      const uint4 d = ld_keep(x + (i + 3 * stride) * 8);
      m2 = __vmaxu2(m2, __vmaxu2(__vmaxu2(absmax8(a), absmax8(b)), __vmaxu2(absmax8(c), absmax8(d))));
    }
    for (; i < total; i += stride) m2 = __vmaxu2(m2, absmax8(ld_keep(x + i * 8)));
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

// E4M3 (FN) code of s >= 0: round to nearest even, saturating at 448.
__device__ __forceinline__ uint32_t e4m3_encode(float s) {
  if (!(s < 448.0f)) return 0x7Eu;
  if (s < 0.015625f) {  // below 2^-6: subnormal grid, step 2^-9 (code = step count)
    return static_cast<uint32_t>(__float2int_rn(__fmul_rn(s, 512.0f)));
  }
  const uint32_t b = __float_as_uint(s);
  const uint32_t r = b + 0x7FFFFu + ((b >> 20) & 1u);  // round the mantissa to 3 bits
  const uint32_t code = (r >> 20) - (120u << 3);        // rebias exponent 127 -> 7
  return min(code, 0x7Eu);
}

// Value of a non-negative E4M3 code.
__device__ __forceinline__ float e4m3_decode(uint32_t c) {
  const uint32_t e = (c >> 3) & 0xFu, m = c & 7u;
  if (e == 0) return __fmul_rn(static_cast<float>(m), 0.001953125f);  // m * 2^-9
  return __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// Four E2M1 bytes (8 codes, element 0 in the low nibble) of 8 floats.
__device__ __forceinline__ uint32_t cvt_e2m1x8(float f0, float f1, float f2, float f3, float f4,
                                               float f5, float f6, float f7) {
  uint32_t out;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(out)
      : "f"(f0), "f"(f1), "f"(f2), "f"(f3), "f"(f4), "f"(f5), "f"(f6), "f"(f7));
  return out;
}

__device__ __forceinline__ float lo_bf16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Sign bits of 8 bf16 values, placed at the sign position of each nibble.
__device__ __forceinline__ uint32_t sign_nibbles(uint4 v) {
  return ((v.x >> 12) & 0x8u) | ((v.x >> 24) & 0x80u) | ((v.y >> 4) & 0x800u) |
         ((v.y >> 16) & 0x8000u) | ((v.z << 4) & 0x80000u) | ((v.z >> 8) & 0x800000u) |
         ((v.w << 12) & 0x8000000u) | (v.w & 0x80000000u);
}

__device__ __forceinline__ float nudge(float v, int ulps) {
  return __int_as_float(__float_as_int(v) + ulps);
}

// Codes of 8 values x / den, where the quotient is the correctly rounded
// FP32 division.  Fast path: x * (1/den) is within 2 ulps of that quotient,
// so if the codes of x*(1/den) moved 4 ulps down and 4 ulps up (in
// magnitude) agree, the code of the exact quotient lies between them and
// equals them.  Otherwise (a quotient next to an E2M1 rounding midpoint) the
// 8 quotients are divided exactly.
__device__ __forceinline__ uint32_t encode8(uint4 v, float inv, float den) {
  const float x0 = lo_bf16(v.x), x1 = hi_bf16(v.x), x2 = lo_bf16(v.y), x3 = hi_bf16(v.y);
  const float x4 = lo_bf16(v.z), x5 = hi_bf16(v.z), x6 = lo_bf16(v.w), x7 = hi_bf16(v.w);
  const float q0 = __fmul_rn(x0, inv), q1 = __fmul_rn(x1, inv), q2 = __fmul_rn(x2, inv),
              q3 = __fmul_rn(x3, inv), q4 = __fmul_rn(x4, inv), q5 = __fmul_rn(x5, inv),
              q6 = __fmul_rn(x6, inv), q7 = __fmul_rn(x7, inv);
  const uint32_t lo = cvt_e2m1x8(nudge(q0, -4), nudge(q1, -4), nudge(q2, -4), nudge(q3, -4),
                                 nudge(q4, -4), nudge(q5, -4), nudge(q6, -4), nudge(q7, -4));
  const uint32_t hi = cvt_e2m1x8(nudge(q0, 4), nudge(q1, 4), nudge(q2, 4), nudge(q3, 4),
                                 nudge(q4, 4), nudge(q5, 4), nudge(q6, 4), nudge(q7, 4));
  uint32_t codes = lo;
  if (lo != hi) {
    codes = cvt_e2m1x8(__fdiv_rn(x0, den), __fdiv_rn(x1, den), __fdiv_rn(x2, den),
                       __fdiv_rn(x3, den), __fdiv_rn(x4, den), __fdiv_rn(x5, den),
                       __fdiv_rn(x6, den), __fdiv_rn(x7, den));
  }
  // A negative value that rounds to zero keeps its sign bit.
  return codes | sign_nibbles(v);
}

// Quantize one 16-element block held in two vectors.
__device__ __forceinline__ void quantize_block(uint4 a, uint4 b, float gs, uint32_t& sbyte,
                                               uint2& codes) {
  const uint32_t m = fold16(__vmaxu2(absmax8(a), absmax8(b)));
  const float bamax = __uint_as_float(m << 16);
  const float s = __fdiv_rn(__fdiv_rn(bamax, 6.0f), gs);
  sbyte = e4m3_encode(s);
  const float den = __fmul_rn(e4m3_decode(sbyte), gs);
  if (den == 0.0f) {
    codes = make_uint2(sign_nibbles(a), sign_nibbles(b));
  } else {
    const float inv = __frcp_rn(den);
    codes = make_uint2(encode8(a, inv, den), encode8(b, inv, den));
  }
}

// ---------------------------------------------------------------- quantize

__global__ void __launch_bounds__(kThreads)
    quantize_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t bpr, int64_t ld,
                    uint8_t* __restrict__ q, uint8_t* __restrict__ sf,
                    const float* __restrict__ gs_ptr) {
  const int64_t total = rows * bpr;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= total) return;
  const float gs = __ldg(gs_ptr);
  int64_t r = i / bpr, c = i % bpr;
  const int64_t sr = stride / bpr, sc = stride % bpr;
  while (r < rows) {
    const uint16_t* src = x + r * ld + c * 16;
    const uint4 a = ld_stream(src);
    const uint4 b = ld_stream(src + 8);
    uint32_t sbyte;
    uint2 codes;
    quantize_block(a, b, gs, sbyte, codes);
    *reinterpret_cast<uint2*>(q + r * (bpr * 8) + c * 8) = codes;
    sf[r * bpr + c] = static_cast<uint8_t>(sbyte);
    c += sc;
    r += sr;
    if (c >= bpr) {
      c -= bpr;
      ++r;
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

template <int G>
__global__ void __launch_bounds__(kThreads)
    deinterleave_quantize_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t inter,
                                 uint8_t* __restrict__ q, uint8_t* __restrict__ sf,
                                 const float* __restrict__ gs_ptr) {
  const int64_t cpr = inter / 16;  // 32-element input chunks per row
  const int64_t total = rows * cpr;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= total) return;
  const float gs = __ldg(gs_ptr);
  int64_t r = i / cpr, c = i % cpr;
  const int64_t sr = stride / cpr, sc = stride % cpr;
  while (r < rows) {
    const uint16_t* src = x + r * (2 * inter) + c * 32;
    uint32_t w[16];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const uint4 t = ld_stream(src + 8 * v);
      w[4 * v] = t.x;
      w[4 * v + 1] = t.y;
      w[4 * v + 2] = t.z;
      w[4 * v + 3] = t.w;
    }
    uint32_t g[8], u[8];
    split_gate_up<G>(w, g, u);
    uint32_t sg, su;
    uint2 cg, cu;
    quantize_block(make_uint4(g[0], g[1], g[2], g[3]), make_uint4(g[4], g[5], g[6], g[7]), gs, sg,
                   cg);
    quantize_block(make_uint4(u[0], u[1], u[2], u[3]), make_uint4(u[4], u[5], u[6], u[7]), gs, su,
                   cu);
    uint8_t* qrow = q + r * inter;  // 2*inter codes -> inter bytes per row
    *reinterpret_cast<uint2*>(qrow + c * 8) = cg;
    *reinterpret_cast<uint2*>(qrow + inter / 2 + c * 8) = cu;
    uint8_t* srow = sf + r * (inter / 8);
    srow[c] = static_cast<uint8_t>(sg);
    srow[inter / 16 + c] = static_cast<uint8_t>(su);
    c += sc;
    r += sr;
    if (c >= cpr) {
      c -= cpr;
      ++r;
    }
  }
}

int grid_for(int64_t work_items, int blocks_per_sm) {
  const int64_t need = (work_items + kThreads - 1) / kThreads;
  const int64_t cap = static_cast<int64_t>(sm_count()) * blocks_per_sm;
  int64_t g = need < cap ? need : cap;
  return static_cast<int>(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_amax(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, float* gs,
                        Workspace* ws, cudaStream_t stream) {
  const int64_t vpr = cols / 8;
  const int grid = grid_for(rows * vpr, 8);
  amax_kernel<<<grid, kThreads, 0, stream>>>(x, rows, vpr, ld, gs, ws);
  return cudaGetLastError();
}

cudaError_t launch_quantize(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, uint8_t* q,
                            uint8_t* sf, const float* gs, cudaStream_t stream) {
  const int64_t bpr = cols / 16;
  if (rows * bpr == 0) return cudaSuccess;
  const int grid = grid_for(rows * bpr, 8);
  quantize_kernel<<<grid, kThreads, 0, stream>>>(x, rows, bpr, ld, q, sf, gs);
  return cudaGetLastError();
}

cudaError_t launch_deinterleave_quantize(const uint16_t* x, int64_t rows, int64_t inter, int g,
                                         uint8_t* q, uint8_t* sf, const float* gs,
                                         cudaStream_t stream) {
  const int64_t items = rows * (inter / 16);
  if (items == 0) return cudaSuccess;
  const int grid = grid_for(items, 8);
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
