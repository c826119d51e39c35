// NVFP4 block-scaled quantize and GEMM + top-k: the CPU oracle.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path links,
// loads or calls this file; only the tests, the smoke check and the bench's
// CPU-baseline leg do.  It shares no code, header, table or constant
// generator with the CUDA path.
//
// It is a plain, slow, single-threaded restatement of the definitions on the
// pages of the "nvfp4-megamoe-kernel" repository (DeepSeek-V4-Pro NVFP4
// inference), step by step:
//
//   E2M1 code table      page "commit 0d1cd1e / dsv4/kernels/indexer",
//                        commit message, "E2M1 encoding (bias=1)" table
//   activation gs        page "commit 107d62d / single_shot_inference.py",
//                        "Fix: compute gsa at runtime": gsa = max|x| / (6*448)
//   amax clamp           page "compare ... v-official-encoding-path",
//                        PERFORMANCE_AUDIT.md section P0 (clamp(min=1e-8))
//   16-element blocks    same page, README.md "NVFP4 throughout"
//                        (E4M3 scales, 16-element micro-blocks)
//   E4M3 / FP4 maxima    same page, CORRECTNESS_BACKLOG.md section 7
//                        (E4M3 max 448, FP4 max 6)
//   dequant formula      page "commit db07d17 / dsv4", weight_scale_2 fix
//                        (w = lut[w] * weight_scale * weight_scale_2)
//   GEMM scaling         page "commit 107d62d / single_shot_inference.py",
//                        global-scale commit ((A*SFA)@(B*SFB), then gsa*gsb)
//   router epilogue      same commit (sqrt(softplus(logit*gsa*gsb))) and
//                        CORRECTNESS_BACKLOG.md section 5 (+ e_bias, top-k);
//                        the V4-Pro router variant (384 experts, top-6) is
//                        in the compare view's model notes; its gating-weight
//                        normalisation is not spelled out (reading below)
//   deinterleave         page "commit 0d1cd1e", fused_deinterleave commit;
//                        docs/PERFORMANCE_AUDIT.md P1 (granularity 8)
//   grouped SwiGLU GEMM  compare view: MoE kernel notes (fused SwiGLU
//                        grouped GEMM, granularity-8 interleaved L1
//                        weights), model notes (swiglu_limit = 10),
//                        PERFORMANCE_AUDIT.md P1 ([silu(gate), silu(gate)*up]
//                        interleaved output)
//
// Readings where the pages are silent (each one is listed in the design
// notes): block scale s = (bamax / 6) / gs in FP32; E4M3 round-to-nearest-
// even with saturation to 448; element value v = x / (dec(s) * gs) in FP32;
// E2M1 round-to-nearest-even with saturation to 6, sign bit kept (a
// negative value that rounds to zero encodes as 0x8); a block whose scale
// byte is zero encodes every element as a signed zero; the even element of a
// pair goes to the low nibble; softplus(z) = z for z > 20; normalised
// router weights (epilogue 2) are the selected weights over their sum;
// the SwiGLU limit clamps the gate from above and the up value on both
// sides.
//
// Floating point: every FP32 step is one IEEE single operation (compile with
// -ffp-contract=off and without fast-math); the GEMM accumulates in double.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <vector>

namespace {

// E2M1 magnitudes for codes 0..7 (bias 1): 0b000=0, 0b001=0.5, 0b010=1,
// 0b011=1.5, 0b100=2, 0b101=3, 0b110=4, 0b111=6.
const double kE2M1Magnitude[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

float bf16_value(uint16_t bits) {
  uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, sizeof(f));
  return f;
}

// Value of a non-negative E4M3 (FN variant) code: 4 exponent bits with bias
// 7, 3 mantissa bits; exponent field 0 is subnormal (m * 2^-9).
double e4m3_value(uint8_t code) {
  const int e = (code >> 3) & 0xF;
  const int m = code & 0x7;
  if (e == 0xF && m == 0x7) return std::numeric_limits<double>::quiet_NaN();
  double mag = (e == 0) ? std::ldexp(static_cast<double>(m), -9)
                        : std::ldexp(1.0 + m / 8.0, e - 7);
  return (code & 0x80) ? -mag : mag;
}

// The 127 non-negative finite E4M3 values, code order (0 .. 448).
const std::vector<double>& e4m3_grid() {
  static const std::vector<double> grid = [] {
    std::vector<double> g(127);
    for (int c = 0; c < 127; ++c) g[c] = e4m3_value(static_cast<uint8_t>(c));
    return g;
  }();
  return grid;
}

}  // namespace

extern "C" {

float orc_bf16_to_f32(uint16_t bits) { return bf16_value(bits); }

double orc_e2m1_decode(uint8_t code) {
  const double mag = kE2M1Magnitude[code & 7];
  return (code & 8) ? -mag : mag;
}

// Nearest E2M1 magnitude to |v| by exhaustive search over the 8 magnitudes;
// on an exact tie the even code wins (round to nearest, ties to even).  The
// largest magnitude, 6, is the nearest for everything above 5, so values
// beyond 6 saturate.  The sign bit is copied from v.
uint8_t orc_e2m1_encode(float v) {
  const double a = std::fabs(static_cast<double>(v));
  const uint8_t sign = std::signbit(v) ? 8 : 0;
  if (a >= 6.0) return static_cast<uint8_t>(sign | 7);  // saturate (also keeps huge |v| exact)
  int best = 0;
  double best_err = a;  // distance to magnitude 0
  for (int c = 1; c < 8; ++c) {
    const double err = std::fabs(a - kE2M1Magnitude[c]);
    if (err < best_err || (err == best_err && (c % 2 == 0) && (best % 2 != 0))) {
      best = c;
      best_err = err;
    }
  }
  return static_cast<uint8_t>(sign | best);
}

float orc_e4m3_decode(uint8_t code) { return static_cast<float>(e4m3_value(code)); }

// Nearest non-negative finite E4M3 value (codes 0..126, max 448) to v >= 0 by
// exhaustive search; ties go to the even code (even mantissa).  Values above
// 448 saturate to 448 (code 126).
uint8_t orc_e4m3_encode(float v) {
  const double a = static_cast<double>(v);
  if (a >= 448.0) return 0x7E;  // saturate (also keeps huge values exact)
  const std::vector<double>& grid = e4m3_grid();
  int best = 0;
  double best_err = std::fabs(a);
  for (int c = 1; c <= 126; ++c) {
    const double err = std::fabs(a - grid[c]);
    if (err < best_err || (err == best_err && (c % 2 == 0) && (best % 2 != 0))) {
      best = c;
      best_err = err;
    }
  }
  return static_cast<uint8_t>(best);
}

// amax = max(max_i |x_i|, 1e-8); gs = amax / (6 * 448) in FP32.
float orc_global_scale(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld) {
  float amax = 0.0f;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) {
      const float a = std::fabs(bf16_value(x[r * ld + c]));
      if (a > amax) amax = a;
    }
  if (amax < 1e-8f) amax = 1e-8f;
  return amax / 2688.0f;
}

// Quantize rows [row_begin, row_end) of x (row stride ld elements) with a
// given global scale gs.  q has cols/2 bytes per row (element 2j in the low
// nibble of byte j, element 2j+1 in the high nibble); sf has cols/16 E4M3
// bytes per row.  Outputs are indexed from row_begin (row r goes to row
// r - row_begin of q and sf).
void orc_quantize_rows(const uint16_t* x, int64_t cols, int64_t ld, float gs,
                       int64_t row_begin, int64_t row_end, uint8_t* q, uint8_t* sf) {
  const int64_t nblocks = cols / 16;
  for (int64_t r = row_begin; r < row_end; ++r) {
    const uint16_t* xr = x + r * ld;
    uint8_t* qr = q + (r - row_begin) * (cols / 2);
    uint8_t* sr = sf + (r - row_begin) * nblocks;
    for (int64_t b = 0; b < nblocks; ++b) {
      float vals[16];
      float bamax = 0.0f;
      for (int j = 0; j < 16; ++j) {
        vals[j] = bf16_value(xr[b * 16 + j]);
        const float a = std::fabs(vals[j]);
        if (a > bamax) bamax = a;
      }
      const float s = (bamax / 6.0f) / gs;          // block scale before encoding
      const uint8_t sbyte = orc_e4m3_encode(s);
      sr[b] = sbyte;
      const float den = orc_e4m3_decode(sbyte) * gs;  // effective block step
      uint8_t codes[16];
      for (int j = 0; j < 16; ++j) {
        const float v = (den != 0.0f) ? vals[j] / den : std::copysign(0.0f, vals[j]);
        codes[j] = orc_e2m1_encode(v);
      }
      for (int j = 0; j < 8; ++j)
        qr[b * 8 + j] = static_cast<uint8_t>(codes[2 * j] | (codes[2 * j + 1] << 4));
    }
  }
}

// Whole-tensor quantize: gs from the tensor's own amax, then every row.
void orc_quantize(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                  uint8_t* q, uint8_t* sf, float* gs_out) {
  const float gs = orc_global_scale(x, rows, cols, ld);
  *gs_out = gs;
  orc_quantize_rows(x, cols, ld, gs, 0, rows, q, sf);
}

// bf16 bits of a float, rounded to nearest even (finite inputs).
uint16_t bf16_round(float f) {
  uint32_t u;
  std::memcpy(&u, &f, sizeof(u));
  const uint32_t rounded = u + 0x7FFFu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(rounded >> 16);
}

// Sum of the squares of one bf16 row, exactly, rounded once to FP32 (round
// to nearest, ties to even; inf when the exact sum is past FP32's range).
// The pages write the norm's denominator as an FP32 sum (or mean) of x^2
// over the row (x_f32.pow(2).sum(dim=-1) in mhc.py, _project_and_rms;
// pow(2).mean(dim=-1) in _dynamic_params) without an order, so the order-
// free reading is taken: the FP32 value nearest the exact sum.
//
// Every finite bf16 value is M * 2^q with an integer M < 256 and
// q = max(E, 1) - 134 (E the 8-bit exponent field), so every square is the
// integer M^2 times 2^(2q), 2q >= -266: the exact sum is an integer S times
// 2^-266, accumulated here in 32-bit limbs, then rounded to the FP32 grid.
float exact_sum_of_squares(const uint16_t* xr, int64_t cols) {
  constexpr int kLimbs = 20;  // 640 bits: 2^16 * 2^506 * 2^14 < 2^537
  uint32_t acc[kLimbs] = {};
  for (int64_t c = 0; c < cols; ++c) {
    const uint32_t e = (xr[c] >> 7) & 0xFFu;
    const uint64_t m = (xr[c] & 0x7Fu) | (e != 0 ? 0x80u : 0u);
    const int shift = 2 * ((e != 0 ? static_cast<int>(e) : 1) - 134) + 266;  // 0 .. 506
    // add m^2 << shift
    uint64_t carry = 0;
    const int limb = shift / 32, off = shift % 32;
    const uint64_t part = (m * m) << off;  // < 2^48
    for (int i = limb; i < kLimbs; ++i) {
      uint64_t add = carry;
      if (i == limb) add += part & 0xFFFFFFFFu;
      if (i == limb + 1) add += part >> 32;
      const uint64_t t = static_cast<uint64_t>(acc[i]) + add;
      acc[i] = static_cast<uint32_t>(t);
      carry = t >> 32;
      if (carry == 0 && i > limb) break;
    }
  }
  auto bit = [&](int i) { return (acc[i / 32] >> (i % 32)) & 1u; };
  int top = kLimbs * 32 - 1;
  while (top >= 0 && !bit(top)) --top;
  if (top < 0) return 0.0f;
  // Keep the bits from position p up: 24 significant bits, but no finer than
  // FP32's smallest step 2^-149 (position 266 - 149 = 117).
  const int p = std::max(top - 23, 117);
  uint64_t keep = 0;
  for (int i = top; i >= p; --i) keep = (keep << 1) | bit(i);
  if (p > 0) {
    const bool half = bit(p - 1) != 0;
    bool below = false;
    for (int i = p - 2; i >= 0 && !below; --i) below = bit(i) != 0;
    if (half && (below || (keep & 1u))) ++keep;  // round to nearest, ties to even
  }
  // keep * 2^(p - 266) is on the FP32 grid (or past its largest value)
  const double v = std::ldexp(static_cast<double>(keep), p - 266);
  return v > static_cast<double>(std::numeric_limits<float>::max())
             ? std::numeric_limits<float>::infinity()
             : static_cast<float>(v);
}

// RMSNorm of each row to bf16, as the producer of the quantize input (page
// "compare ... v-official-encoding-path": fused RMSNorm + NVFP4 quantize,
// PERFORMANCE_AUDIT.md P4; the norm is input * inv_rms * weight[c]).  The
// pages fix no epsilon; the readings taken:
//   sum of squares: exact, rounded once to FP32 (exact_sum_of_squares);
//   inv_rms = 1 / sqrt(sum / cols + eps), each step one FP32 operation;
//   y = (x * inv_rms) * weight[c] in FP32, rounded to bf16 (the model's
//     hidden-state type), which is what gets quantized.
void orc_rmsnorm(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, const uint16_t* weight,
                 float eps, uint16_t* out) {
  for (int64_t r = 0; r < rows; ++r) {
    const uint16_t* xr = x + r * ld;
    const float sum = exact_sum_of_squares(xr, cols);
    const float mean = sum / static_cast<float>(cols);
    const float inv_rms = 1.0f / std::sqrt(mean + eps);
    for (int64_t c = 0; c < cols; ++c) {
      const float y = (bf16_value(xr[c]) * inv_rms) * bf16_value(weight[c]);
      out[r * cols + c] = bf16_round(y);
    }
  }
}

// The FP32 sum of squares of each row, as orc_rmsnorm takes it.
void orc_rms_sum_of_squares(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, float* out) {
  for (int64_t r = 0; r < rows; ++r) out[r] = exact_sum_of_squares(x + r * ld, cols);
}

// RMSNorm, then quantize the [rows, cols] bf16 result as a whole.
void orc_rmsnorm_quantize(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                          const uint16_t* weight, float eps, uint8_t* q, uint8_t* sf, float* gs_out) {
  std::vector<uint16_t> tmp(static_cast<size_t>(rows * cols));
  orc_rmsnorm(x, rows, cols, ld, weight, eps, tmp.data());
  orc_quantize(tmp.data(), rows, cols, cols, q, sf, gs_out);
}

// The mHC layer input of each token: the mix of its n_hc residual streams
// by the token's input mapping A_l (compare view: mhc.py, the mHCLayer
// docstring "x_in, ctx = mhc.pre_block(X_l)" with X_l of shape (T, n_hc, d),
// and _dynamic_params, "A_l: (T, n_hc) sigmoid-constrained input mapping",
// returned as bf16; FINAL_STRETCH.md / PERFORMANCE_AUDIT.md P5 fuse this
// pre_block with the RMSNorm and the NVFP4 quantize).  The pages do not print
// pre_block's body; the reading taken: x_in[t, c] = sum_i A[t, i] X[t, i, c]
// accumulated in FP32 over the streams in index order (each bf16 x bf16
// product is exact in FP32, so only the additions round), rounded to bf16.
// x: token t's stream i is the row of cols elements at x + t * ld + i * cols.
void orc_mhc_mix(const uint16_t* x, int64_t rows, int64_t n_hc, int64_t cols, int64_t ld,
                 const uint16_t* a, uint16_t* out) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) {
      float acc = 0.0f;
      for (int64_t i = 0; i < n_hc; ++i) {
        const float prod = bf16_value(a[r * n_hc + i]) * bf16_value(x[r * ld + i * cols + c]);  // exact
        acc = (i == 0) ? prod : acc + prod;
      }
      out[r * cols + c] = bf16_round(acc);
    }
}

// mHC pre-mix, then RMSNorm (orc_rmsnorm), then quantize: the fused op.
void orc_mhc_rmsnorm_quantize(const uint16_t* x, int64_t rows, int64_t n_hc, int64_t cols, int64_t ld,
                              const uint16_t* a, const uint16_t* weight, float eps, uint8_t* q, uint8_t* sf,
                              float* gs_out) {
  std::vector<uint16_t> mixed(static_cast<size_t>(rows * cols));
  orc_mhc_mix(x, rows, n_hc, cols, ld, a, mixed.data());
  std::vector<uint16_t> normed(static_cast<size_t>(rows * cols));
  orc_rmsnorm(mixed.data(), rows, cols, cols, weight, eps, normed.data());
  orc_quantize(normed.data(), rows, cols, cols, q, sf, gs_out);
}

// Deinterleave one [rows, 2I] matrix whose gate/up columns alternate in
// groups of g: output column j < I is gate column j, taken from input column
// 2g*floor(j/g) + (j mod g); output column I + j is up column j, taken from
// input column 2g*floor(j/g) + g + (j mod g).
void orc_deinterleave(const uint16_t* x, int64_t rows, int64_t inter, int64_t g, uint16_t* out) {
  const int64_t w = 2 * inter;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t j = 0; j < inter; ++j) {
      const int64_t base = 2 * g * (j / g) + (j % g);
      out[r * w + j] = x[r * w + base];
      out[r * w + inter + j] = x[r * w + base + g];
    }
}

// Deinterleave, then quantize the [rows, 2I] result as a whole.
void orc_deinterleave_quantize(const uint16_t* x, int64_t rows, int64_t inter, int64_t g,
                               uint8_t* q, uint8_t* sf, float* gs_out) {
  std::vector<uint16_t> tmp(static_cast<size_t>(rows * 2 * inter));
  orc_deinterleave(x, rows, inter, g, tmp.data());
  orc_quantize(tmp.data(), rows, 2 * inter, 2 * inter, q, sf, gs_out);
}

// Dequantize rows of an NVFP4 tensor: out = lut[q] * e4m3(sf) * gs, in double.
void orc_dequantize(const uint8_t* q, const uint8_t* sf, float gs, int64_t rows, int64_t cols,
                    double* out) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) {
      const uint8_t byte = q[r * (cols / 2) + c / 2];
      const uint8_t code = (c % 2 == 0) ? (byte & 0xF) : (byte >> 4);
      out[r * cols + c] = orc_e2m1_decode(code) * e4m3_value(sf[r * (cols / 16) + c / 16]) *
                          static_cast<double>(gs);
    }
}

// Block-scaled GEMM logits for rows [row_begin, row_end):
//   acc[m,n] = sum_k lut(qa[m,k]) * sfa[m,k/16] * lut(qb[n,k]) * sfb[n,k/16]   (double)
//   logit[m,n] = float(acc * gsa * gsb)
// A is M x K (K/2 bytes per row), B is N x K; out is (row_end-row_begin) x N.
void orc_gemm_logits(const uint8_t* qa, const uint8_t* sfa, float gsa,
                     const uint8_t* qb, const uint8_t* sfb, float gsb,
                     int64_t N, int64_t K, int64_t row_begin, int64_t row_end, float* out) {
  // lut(q) * e4m3(sf) for every element of B, then for each row of A.
  std::vector<double> b(static_cast<size_t>(N * K));
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k) {
      const uint8_t byte = qb[n * (K / 2) + k / 2];
      const uint8_t code = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
      b[n * K + k] = orc_e2m1_decode(code) * e4m3_value(sfb[n * (K / 16) + k / 16]);
    }
  std::vector<double> a(static_cast<size_t>(K));
  for (int64_t m = row_begin; m < row_end; ++m) {
    for (int64_t k = 0; k < K; ++k) {
      const uint8_t byte = qa[m * (K / 2) + k / 2];
      const uint8_t code = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
      a[k] = orc_e2m1_decode(code) * e4m3_value(sfa[m * (K / 16) + k / 16]);
    }
    for (int64_t n = 0; n < N; ++n) {
      const double* bn = b.data() + n * K;
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k) acc += a[k] * bn[k];
      out[(m - row_begin) * N + n] =
          static_cast<float>(acc * static_cast<double>(gsa) * static_cast<double>(gsb));
    }
  }
}

// Full indexer score (page "commit 0d1cd1e", dsv4/_archive/kernels/indexer/
// csa_indexer.py docstring, paper eq. 13-17 as quoted there; the key is
// shared across heads):  I[t, s] = sum_h w[t, h] * ReLU(q[t, h] . K[s]).
// The query rows of token t are rows t * H .. t * H + H - 1 of A (head-major
// per token), the logits are those of orc_gemm_logits, the head sum is
// taken in double and stored as float.
void orc_indexer_scores(const uint8_t* qa, const uint8_t* sfa, float gsa, const uint8_t* qb,
                        const uint8_t* sfb, float gsb, int64_t T, int64_t H, int64_t N, int64_t K,
                        const float* head_w, float* out) {
  std::vector<float> logits(static_cast<size_t>(H * N));
  for (int64_t t = 0; t < T; ++t) {
    orc_gemm_logits(qa, sfa, gsa, qb, sfb, gsb, N, K, t * H, t * H + H, logits.data());
    for (int64_t s = 0; s < N; ++s) {
      double acc = 0.0;
      for (int64_t h = 0; h < H; ++h) {
        const double z = logits[h * N + s];
        acc += static_cast<double>(head_w[t * H + h]) * (z > 0.0 ? z : 0.0);
      }
      out[t * N + s] = static_cast<float>(acc);
    }
  }
}

// Epilogue on a rows x N logit matrix.
//   epilogue 0 (identity, indexer-shaped): score = weight = logit
//   epilogue 1 (router-shaped): weight = sqrt(softplus(logit)),
//                               score = weight + bias[n]
// softplus(z) = log(1 + e^z), taken as z itself above 20.  Double, then float.
void orc_epilogue(const float* logits, int64_t rows, int64_t N, int epilogue, const float* bias,
                  float* score, float* weight) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t n = 0; n < N; ++n) {
      const double z = logits[r * N + n];
      if (epilogue == 0) {
        score[r * N + n] = static_cast<float>(z);
        if (weight) weight[r * N + n] = static_cast<float>(z);
      } else {
        const double sp = (z > 20.0) ? z : std::log1p(std::exp(z));
        const double w = std::sqrt(sp);
        score[r * N + n] = static_cast<float>(w + static_cast<double>(bias[n]));
        if (weight) weight[r * N + n] = static_cast<float>(w);
      }
    }
}

// Per-row top-k of a rows x N score matrix: the k largest scores in
// descending order, equal scores ordered by lower column index.  Slots past
// N get index -1, score -inf, weight 0.
void orc_topk(const float* score, const float* weight, int64_t rows, int64_t N, int k,
              int32_t* idx_out, float* score_out, float* weight_out) {
  std::vector<int64_t> order(static_cast<size_t>(N));
  for (int64_t r = 0; r < rows; ++r) {
    const float* s = score + r * N;
    for (int64_t n = 0; n < N; ++n) order[n] = n;
    const int64_t take = std::min<int64_t>(k, N);
    std::partial_sort(order.begin(), order.begin() + take, order.end(),
                      [s](int64_t i, int64_t j) { return s[i] > s[j] || (s[i] == s[j] && i < j); });
    for (int64_t t = 0; t < k; ++t) {
      if (t < take) {
        idx_out[r * k + t] = static_cast<int32_t>(order[t]);
        score_out[r * k + t] = s[order[t]];
        if (weight_out) weight_out[r * k + t] = weight ? weight[r * N + order[t]] : 0.0f;
      } else {
        idx_out[r * k + t] = -1;
        score_out[r * k + t] = -std::numeric_limits<float>::infinity();
        if (weight_out) weight_out[r * k + t] = 0.0f;
      }
    }
  }
}

// Gating-weight normalisation of a router's top-k (epilogue 2): each row's
// selected weights divided by their sum, so they add up to one (the pages
// name the router variants but give no formula; this is the reading taken).
// Sum and quotients in double, stored as float; empty slots (index -1) stay
// 0 and do not count.
void orc_normalize_topk_weights(const int32_t* idx, float* weight, int64_t rows, int k) {
  for (int64_t r = 0; r < rows; ++r) {
    double sum = 0.0;
    for (int t = 0; t < k; ++t)
      if (idx[r * k + t] >= 0) sum += weight[r * k + t];
    if (sum <= 0.0) continue;
    for (int t = 0; t < k; ++t)
      if (idx[r * k + t] >= 0) weight[r * k + t] = static_cast<float>(weight[r * k + t] / sum);
  }
}

// The whole GEMM + epilogue + top-k for rows [row_begin, row_end).
void orc_gemm_topk_rows(const uint8_t* qa, const uint8_t* sfa, float gsa,
                        const uint8_t* qb, const uint8_t* sfb, float gsb,
                        int64_t N, int64_t K, int epilogue, const float* bias, int k,
                        int64_t row_begin, int64_t row_end,
                        int32_t* idx_out, float* score_out, float* weight_out) {
  const int64_t rows = row_end - row_begin;
  std::vector<float> logits(static_cast<size_t>(rows * N));
  std::vector<float> score(static_cast<size_t>(rows * N));
  std::vector<float> weight(static_cast<size_t>(rows * N));
  orc_gemm_logits(qa, sfa, gsa, qb, sfb, gsb, N, K, row_begin, row_end, logits.data());
  orc_epilogue(logits.data(), rows, N, epilogue == 2 ? 1 : epilogue, bias, score.data(), weight.data());
  orc_topk(score.data(), weight.data(), rows, N, k, idx_out, score_out, weight_out);
  if (epilogue == 2 && weight_out) orc_normalize_topk_weights(idx_out, weight_out, rows, k);
}

// Grouped block-scaled GEMM with the SwiGLU epilogue of the MoE first
// projection (compare view, MoE kernel notes "FusedSwiGLUScaledGroupedGemm-
// Kernel": SwiGLU and clamp applied between the TMEM read and the store,
// L1 weights with gate and up interleaved at granularity 8; model notes
// "SwiGLU activation with swiglu_limit=10.0"; the shared-expert fix (P1):
// the fused kernel writes [silu(gate), silu(gate) * up] interleaved at the
// weights' granularity).
//
// Group e owns the A rows [offs[e], offs[e+1]) and the 2I weight rows
// [e * 2I, (e + 1) * 2I) of B, whose rows hold gate and up columns in
// alternating runs of g (as orc_deinterleave reads them), and its own
// global scale gsb[e].  For a row m of group e:
//   logit[n]  = float(gsa * gsb[e] * sum_k A[m, k] B[e*2I + n, k])  (as orc_gemm_logits)
//   gate[j]   = logit[2g*floor(j/g) + j mod g],  up[j] = logit[2g*floor(j/g) + g + j mod g]
//   gate'     = min(gate, limit),  up' = min(max(up, -limit), limit)
//   a[j]      = silu(gate') = gate' / (1 + exp(-gate'))              (double)
//   h[j]      = a[j] * up'
// The clamp form (gate from above, up on both sides, one limit) is the
// reading taken: the pages name the limit but not where it applies.
// Outputs, double, [M, I] each: h (the SwiGLU result) and a (the SiLU of
// the clamped gate).  Rows outside every group are left untouched.
void orc_grouped_swiglu(const uint8_t* qa, const uint8_t* sfa, float gsa, const uint8_t* qb,
                        const uint8_t* sfb, const float* gsb, const int32_t* offs, int64_t E,
                        int64_t inter, int64_t K, int64_t g, double limit, double* h_out,
                        double* a_out) {
  const int64_t two_i = 2 * inter;
  for (int64_t e = 0; e < E; ++e) {
    const int64_t lo = offs[e], hi = offs[e + 1];
    if (hi <= lo) continue;
    std::vector<float> logits(static_cast<size_t>((hi - lo) * two_i));
    orc_gemm_logits(qa, sfa, gsa, qb + e * two_i * (K / 2), sfb + e * two_i * (K / 16), gsb[e],
                    two_i, K, lo, hi, logits.data());
    for (int64_t m = lo; m < hi; ++m) {
      const float* z = logits.data() + (m - lo) * two_i;
      for (int64_t j = 0; j < inter; ++j) {
        const int64_t base = 2 * g * (j / g) + (j % g);
        const double gate = std::min(static_cast<double>(z[base]), limit);
        const double up = std::min(std::max(static_cast<double>(z[base + g]), -limit), limit);
        const double a = gate / (1.0 + std::exp(-gate));
        h_out[m * inter + j] = a * up;
        if (a_out) a_out[m * inter + j] = a;
      }
    }
  }
}

// Round doubles to bf16 bit patterns (through float; both roundings to
// nearest even).
void orc_to_bf16(const double* v, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = bf16_round(static_cast<float>(v[i]));
}

}  // extern "C"
