/*
 * nvfp4.h — C ABI of the GB300 (sm_103a) NVFP4 block-scaled quantize and
 * GEMM + top-k library (libnvfp4.so).
 *
 * The operations are those of the NVFP4 inference path described on the
 * "nvfp4-megamoe-kernel" repository pages (DeepSeek-V4-Pro on Blackwell):
 *
 *   nvfp4_quantize               activation quantize: grid-wide amax ->
 *                                global scale, E4M3 block scales, E2M1 codes
 *   nvfp4_deinterleave_quantize  the same for an interleaved SwiGLU gate/up
 *                                output, deinterleaved to [gate | up] first
 *   nvfp4_rmsnorm_quantize       the same for RMSNorm(x) * weight, the
 *                                norm fused in
 *   nvfp4_mhc_rmsnorm_quantize   the same for the mHC pre-mix of n_hc
 *                                residual streams, mix and norm fused in
 *   nvfp4_gemm_topk              block-scaled FP4 GEMM with a fused scoring
 *                                epilogue and per-row top-k
 *   nvfp4_indexer_topk           the same GEMM with the indexer's weighted
 *                                ReLU head sum fused in, top-k per token
 *   nvfp4_grouped_swiglu_gemm    grouped (per-expert) block-scaled FP4 GEMM
 *                                with the MoE SwiGLU epilogue, bf16 out
 *
 * Conventions shared by every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the
 *     library never allocates, frees or keeps them.
 *   - Every call is asynchronous on the given stream (0 = legacy default
 *     stream) and performs no host synchronisation.  Global scales stay on
 *     the device.
 *   - Arguments are validated on the host before anything is launched; a
 *     call that returns an error has launched nothing.
 *   - bf16 data is passed as its 16-bit patterns (uint16_t).
 *   - NVFP4 tensor of logical shape [rows, cols]:
 *       q  : uint8 [rows, cols/2], row-major; element 2j of a row is the
 *            low nibble of byte j, element 2j+1 the high nibble; a nibble
 *            is sign bit (bit 3) + E2M1 magnitude code (bits 0-2)
 *       sf : uint8 [rows, cols/16], row-major E4M3 (FN) block scales, one
 *            per 16 consecutive elements of a row
 *       gs : one FP32 global scale (device)
 *     value(r, c) = e2m1(q nibble) * e4m3(sf[r, c/16]) * gs
 *   - Workspace: a small device buffer of nvfp4_workspace_bytes() bytes,
 *     zeroed once by nvfp4_workspace_init() (or cudaMemsetAsync) before its
 *     first use.  Each call leaves it as it found it.  Calls that share one
 *     workspace must be ordered (same stream or explicit events).
 *
 * Return value of every int function: an nvfp4_status.
 */
#ifndef NVFP4_H_
#define NVFP4_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum nvfp4_status {
  NVFP4_OK = 0,
  NVFP4_ERR_INVALID = 1,      /* null pointer, negative size, bad enum, k out of range */
  NVFP4_ERR_UNSUPPORTED = 2,  /* shape or alignment outside what the kernels take */
  NVFP4_ERR_WORKSPACE = 3,    /* ws null or ws_bytes < nvfp4_workspace_bytes() */
  NVFP4_ERR_CUDA = 4          /* a CUDA call failed; see nvfp4_last_cuda_error() */
} nvfp4_status;

typedef enum nvfp4_epilogue {
  /* score = logit (indexer-shaped scoring) */
  NVFP4_EPILOGUE_IDENTITY = 0,
  /* weight = sqrt(softplus(logit)), score = weight + bias[n] (router-shaped) */
  NVFP4_EPILOGUE_SQRT_SOFTPLUS_BIAS = 1,
  /* as 1, and each row's k output weights are divided by their sum (the
   * router variant with normalised gating weights; k <= 32) */
  NVFP4_EPILOGUE_SQRT_SOFTPLUS_BIAS_NORM = 2
} nvfp4_epilogue;

/* Device-side status bits a kernel may record in the workspace. */
#define NVFP4_DEVICE_TIMEOUT 0x1u /* a bounded wait inside a kernel gave up */
#define NVFP4_DEVICE_BAD_GROUPS 0x2u /* group offsets broke their contract (grouped GEMM) */

/* Operations, for nvfp4_workspace_bytes. */
typedef enum nvfp4_op {
  NVFP4_OP_QUANTIZE = 0,
  NVFP4_OP_DEINTERLEAVE_QUANTIZE = 1,
  NVFP4_OP_GEMM_TOPK = 2,
  NVFP4_OP_RMSNORM_QUANTIZE = 3,
  NVFP4_OP_INDEXER_TOPK = 4,
  NVFP4_OP_GROUPED_SWIGLU_GEMM = 5,
  NVFP4_OP_MHC_RMSNORM_QUANTIZE = 6
} nvfp4_op;

/*
 * Bytes of workspace a call of operation `op` needs for a problem of `rows`
 * x `cols` (quantize ops: the input's shape; GEMM ops: rows = M, cols = K,
 * n = N, k = top-k).  Every kernel keeps its cross-CTA state in a few
 * counters, so today the answer is the same small constant (256) for every
 * operation and shape, and one workspace serves every call of a stream.
 * Returns 0 for an unknown op or a negative size.
 */
size_t nvfp4_workspace_bytes(int op, int64_t rows, int64_t cols, int64_t n, int k);

/* Zero a workspace on `stream` (cudaMemsetAsync).  Needed once per buffer. */
int nvfp4_workspace_init(void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Activation quantize.  Source: commit 107d62d ("Fix: compute gsa at
 * runtime ... gsa = max(|x|) / (6.0 * 448.0)") and the dsv4/ops/quantize.py
 * commit ("Two-kernel approach (correct, zero CPU syncs)"); 16-element E4M3
 * blocks per the compare view's README "NVFP4 throughout"; the E2M1 table of
 * commit 0d1cd1e.
 *
 *   amax  = max(max |x|, 1e-8);  gs = amax / 2688                  (FP32)
 *   per 16-element block of a row: s = (max|x_block| / 6) / gs     (FP32)
 *     sf    = E4M3(s), round to nearest even, saturating at 448
 *     den   = e4m3(sf) * gs                                        (FP32)
 *     code  = sign(x) | E2M1(|x| / den), round to nearest even,
 *             saturating at 6; den == 0 gives signed zero codes
 *
 * x     : bf16 [rows, cols] with row stride ld_x elements; 16-byte aligned,
 *         ld_x a multiple of 8, ld_x >= cols.
 * cols  : multiple of 16.  rows >= 0 (rows == 0 still writes gs for amax 1e-8;
 *         x, q and sf may then be NULL).
 * q     : [rows, cols/2] bytes, 8-byte aligned.   sf : [rows, cols/16] bytes.
 * gs    : one float on the device, written by the call (4-byte aligned).
 * Launches: inputs that fit in the SMs' shared memory (up to about 30 MB)
 * take ONE launch: each CTA copies its slice on chip, the CTAs meet on the
 * grid-wide maximum (one thread-block cluster in distributed shared memory
 * up to 512 KB, else a cooperative grid at a bounded counter barrier), and
 * quantize from shared memory, so x crosses HBM once.  Larger inputs take
 * two kernels: a grid-wide amax whose last block writes gs, then the
 * quantize pass, which reads gs from device memory.
 */
int nvfp4_quantize(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld_x,
                   uint8_t* q, uint8_t* sf, float* gs,
                   void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Deinterleave + quantize for a SwiGLU output whose gate and up columns
 * alternate in groups of `granularity` (commit 0d1cd1e,
 * "fused_deinterleave_amax_quantize.cu"; the compare view's
 * docs/PERFORMANCE_AUDIT.md P1, granularity 8).
 *
 * x    : bf16 [rows, 2*inter], contiguous rows, 16-byte aligned.  Input
 *        column 2g*floor(j/g) + (j mod g) is gate column j, and
 *        2g*floor(j/g) + g + (j mod g) is up column j (g = granularity).
 * The result is nvfp4_quantize of the [rows, 2*inter] matrix
 * [gate_0 .. gate_{inter-1} | up_0 .. up_{inter-1}]:
 * q [rows, inter] bytes (8-byte aligned), sf [rows, inter/8], gs one float.
 * inter: multiple of 16.  granularity: 1, 2, 4, 8 or 16.
 */
int nvfp4_deinterleave_quantize(const uint16_t* x, int64_t rows, int64_t inter, int granularity,
                                uint8_t* q, uint8_t* sf, float* gs,
                                void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * RMSNorm fused into the activation quantize (the compare view's
 * PERFORMANCE_AUDIT.md P4, "fuse RMSNorm into the next NVFP4 quantize";
 * the norm is input * inv_rms * weight[c], as in the model notes' kv_norm):
 *
 *   per row: sum = the exact sum of x^2 over the row rounded once to FP32
 *            (round to nearest even; the pages give an FP32 sum of squares
 *            without an order, mhc.py _project_and_rms),
 *            inv_rms = 1 / sqrt(sum / cols + eps)                  (FP32)
 *   y[r, c] = bf16((x[r, c] * inv_rms) * weight[c])   (round to nearest even)
 *   then exactly nvfp4_quantize of the bf16 matrix y, which never reaches
 *   memory.
 *
 * x      : bf16 [rows, cols], row stride ld_x elements (16-byte aligned,
 *          ld_x a multiple of 8).  weight: bf16 [cols], 16-byte aligned.
 * cols   : multiple of 16, at most 16384.  eps >= 0 (finite).
 * q, sf, gs: as for nvfp4_quantize.  One launch when the rows fit in the
 *          SMs' shared memory (about 30 MB), else two row-parallel passes.
 */
int nvfp4_rmsnorm_quantize(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld_x,
                           const uint16_t* weight, float eps, uint8_t* q, uint8_t* sf, float* gs,
                           void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * mHC pre-mix, RMSNorm and the activation quantize in one op (the compare
 * view's FINAL_STRETCH.md / PERFORMANCE_AUDIT.md P5, "fuse mHC pre_block +
 * RMSNorm + NVFP4 quantize"; mhc.py: the layer input x_in = pre_block(X_l)
 * of the (T, n_hc, d) residual state, with the per-token input mapping A_l
 * of shape (T, n_hc) in bf16):
 *
 *   x_in[t, c] = bf16(sum_i A[t, i] * X[t, i, c])   FP32 accumulation over
 *                the streams in index order (each product is exact in FP32;
 *                the pages do not print pre_block's body: this is the reading)
 *   then exactly nvfp4_rmsnorm_quantize of the [rows, cols] bf16 matrix x_in
 *   (x_in and the normalised rows never reach memory).
 *
 * x      : bf16, token t's stream i is the row of cols elements at
 *          x + t * ld_x + i * cols (streams of a token contiguous); 16-byte
 *          aligned, ld_x a multiple of 8 and >= n_hc * cols.
 * a      : bf16 [rows, n_hc] (2-byte aligned).   n_hc: 1 .. 8.
 * weight : bf16 [cols], 16-byte aligned.  cols: multiple of 16, at most 8192.
 * eps, q, sf, gs: as for nvfp4_rmsnorm_quantize.  One launch when the tokens'
 *          streams fit in the SMs' shared memory (about 30 MB), else two
 *          row-parallel passes (each mixes its rows again).
 */
int nvfp4_mhc_rmsnorm_quantize(const uint16_t* x, int64_t rows, int n_hc, int64_t cols, int64_t ld_x,
                               const uint16_t* a, const uint16_t* weight, float eps, uint8_t* q, uint8_t* sf,
                               float* gs, void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Block-scaled FP4 GEMM + fused epilogue + per-row top-k.  Sources: the
 * dequant formula of commit db07d17 (w = lut[w] * weight_scale *
 * weight_scale_2), the global-scale commit of 107d62d ((A*SFA) @ (B*SFB),
 * then * gsa * gsb), the router score of the same commit and of the compare
 * view's CORRECTNESS_BACKLOG.md section 5 (sqrt(softplus) + e_bias, top-k),
 * and the fused router kernel of commit db07d17 (no FP32 logits in GMEM).
 *
 *   logit[m, n] = gsa * gsb * sum_k A[m, k] * B[n, k]      (A, B NVFP4 values
 *                 without their global scales; FP32 tensor-core accumulation)
 *   epilogue IDENTITY:           weight = score = logit
 *   epilogue SQRT_SOFTPLUS_BIAS: weight = sqrt(softplus(logit)),
 *                                score  = weight + bias[n]
 *   epilogue SQRT_SOFTPLUS_BIAS_NORM: as above, then the k selected weights
 *                                of a row are divided by their sum (the
 *                                pages name this router variant without a
 *                                formula; this is the reading taken)
 *   per row m: the k largest scores, in descending order; equal scores are
 *   ordered by lower n.
 *
 * A: qa [M, K/2] (16-byte aligned), sfa [M, K/16] (4-byte aligned), gsa.
 * B: qb [N, K/2] (16-byte aligned), sfb [N, K/16] (4-byte aligned), gsb.
 *    (B row n holds output column n: the checkpoint's N x K weight layout.)
 * M >= 0 (M == 0 launches nothing; qa, sfa and the outputs may then be NULL),
 * N >= 1, K a positive multiple of 64.  1 <= k <= 1024; for k > 32
 * the N scores of a row must fit on chip (N <= 4096).
 * bias: N floats, required for the SQRT_SOFTPLUS epilogues, ignored for
 * IDENTITY.  SQRT_SOFTPLUS_BIAS_NORM takes k <= 32.
 * Outputs, each [M, k] row-major: topk_idx (int32), topk_score (float),
 * topk_weight (float, may be NULL).  Slots beyond N hold idx -1,
 * score -inf, weight 0.
 * logits: NULL in production; if non-NULL, [M, N] FP32 logits are also
 * written (for testing the GEMM stage on its own).
 */
int nvfp4_gemm_topk(const uint8_t* qa, const uint8_t* sfa, const float* gsa,
                    const uint8_t* qb, const uint8_t* sfb, const float* gsb,
                    int64_t M, int64_t N, int64_t K,
                    int epilogue, const float* bias, int k,
                    int32_t* topk_idx, float* topk_score, float* topk_weight,
                    float* logits, void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * nvfp4_quantize for callers that must not allocate device memory: an engine
 * that gives all of HBM to its own arena up front, or a thread that may not
 * call cudaMalloc/cudaFree because they can block on or synchronise the
 * device.  The pages have no counterpart; it runs the same kernels as
 * nvfp4_quantize with the same arguments and results, minus the workspace.
 *
 * Scratch: a 256-byte static device array inside the library (one per GPU
 * that loads it, held until exit).  A call whose scratch need exceeds it
 * returns NVFP4_ERR_WORKSPACE (today every shape needs exactly 256 bytes).
 * Each call clears the words that must start at zero on `stream` before its
 * kernels.  All calls on a device share the array: calls that can overlap on
 * the GPU (different streams without ordering between them) race and give
 * wrong results.  The first call on a device, with that device current,
 * looks up the array's device address (cudaGetSymbolAddress) and keeps it
 * for that device (one CUDA context per device, the runtime's primary
 * context, is assumed); make that first call before any stream capture.  A
 * bounded wait that runs out inside the one-pass kernel records
 * NVFP4_DEVICE_TIMEOUT in the static scratch, where no caller can read it
 * (nvfp4_read_device_status takes a workspace): q, sf and gs are then
 * undefined and nothing reports it.  Allocates nothing.
 */
int nvfp4_quantize_noalloc(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld_x,
                           uint8_t* q, uint8_t* sf, float* gs, cudaStream_t stream);

/*
 * Full indexer score with head reduction, then per-token top-k (page
 * "commit 0d1cd1e", the csa_indexer.py docstring: I[t, s] = sum_h w[t, h] *
 * ReLU(q[t, h] . K[s]), the key shared across heads; Selected = TopK(I[t, :])):
 *
 *   logit[t*heads + h, s] = gsa * gsb * sum_k A[t*heads + h, k] * B[s, k]
 *   I[t, s] = sum_h head_w[t, h] * max(logit[t*heads + h, s], 0)     (FP32)
 *   per token t: the k largest I[t, s], descending, ties by lower s.
 *
 * A: qa [tokens*heads, K/2], sfa [tokens*heads, K/16], gsa (query rows
 *    head-major per token).  B: qb [N, K/2], sfb [N, K/16], gsb (the keys).
 * heads: 32, 64 or 128.  head_w: float [tokens, heads].  N <= 4096, K a
 * positive multiple of 64, 1 <= k <= 1024.  Outputs [tokens, k]: topk_idx
 * (int32), topk_score (float); slots beyond N hold -1 / -inf.  scores: NULL,
 * or float [tokens, N] to receive I (for testing).  The head sum is fused in
 * the GEMM epilogue; I does not reach memory unless `scores` is given.
 */
int nvfp4_indexer_topk(const uint8_t* qa, const uint8_t* sfa, const float* gsa,
                       const uint8_t* qb, const uint8_t* sfb, const float* gsb,
                       int64_t tokens, int heads, int64_t N, int64_t K, const float* head_w,
                       int k, int32_t* topk_idx, float* topk_score, float* scores,
                       void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Grouped block-scaled FP4 GEMM with the SwiGLU epilogue of the MoE first
 * projection (compare view: the MoE kernel notes, fused SwiGLU grouped GEMM
 * with L1 weights whose gate and up rows are interleaved at granularity 8;
 * the model notes, "SwiGLU activation with swiglu_limit=10.0";
 * PERFORMANCE_AUDIT.md P1, the [silu(gate), silu(gate)*up] interleaved
 * output):
 *
 *   group e: A rows offsets[e] .. offsets[e+1]-1, weights W_e = B rows
 *            e*2I .. e*2I + 2I - 1, global scale gsb[e]
 *   logit[m, n] = gsa * gsb[e] * sum_k A[m, k] * W_e[n, k]   (FP32 accumulate)
 *   gate_j = logit[m, 2g*floor(j/g) + j mod g],  up_j = the column g after it
 *   a_j = silu(min(gate_j, limit)) = gate' / (1 + exp(-gate'))
 *   h_j = a_j * min(max(up_j, -limit), limit)                  (FP32)
 *   layout 0: out[m, j] = bf16(h_j)                 out is [M, ld_out], j < inter
 *   layout 1: out[m, n] = bf16(a) where W row n is a gate row, bf16(h) where
 *             it is an up row (the pages' interleaved output, the input of
 *             nvfp4_deinterleave_quantize)             n < 2*inter
 * (where the limit applies is not spelled out on the pages: the gate is
 * clamped from above, the up value on both sides; pass INFINITY for none)
 *
 * A: qa [M, K/2], sfa [M, K/16], gsa (one quantize call for all rows; the
 *    rows of each group contiguous, groups in order).
 * B: qb [E*2I, K/2], sfb [E*2I, K/16] (the E experts' [2I, K] weights
 *    stacked), gsb: E floats.  All four code/scale pointers 16-byte aligned.
 * offsets: int32 [E+1] in DEVICE memory (written by the router on the GPU;
 *    the host never reads it): non-decreasing, offsets[0] >= 0,
 *    offsets[E] <= M.  Rows outside every group are not written.  Offsets
 *    that break this are clamped into [0, M] (no access leaves the
 *    buffers), the result is unspecified, and NVFP4_DEVICE_BAD_GROUPS is
 *    recorded in the workspace.
 * 1 <= E <= 1024.  inter (I): a positive multiple of 128.  K: a positive
 * multiple of 256.  granularity: 1, 2, 4, 8 or 16.  limit > 0 (may be
 * INFINITY).  out: bf16, 16-byte aligned, ld_out a multiple of 8 and at
 * least I (layout 0) or 2I (layout 1).  M == 0 launches nothing.
 * One persistent launch (one CTA per SM); FP32 logits never reach memory.
 */
int nvfp4_grouped_swiglu_gemm(const uint8_t* qa, const uint8_t* sfa, const float* gsa,
                              const uint8_t* qb, const uint8_t* sfb, const float* gsb,
                              const int32_t* offsets, int64_t M, int64_t E, int64_t inter, int64_t K,
                              int granularity, float limit, int layout, uint16_t* out, int64_t ld_out,
                              void* ws, size_t ws_bytes, cudaStream_t stream);
/*
 * Diagnostic: synchronise `stream`, copy the workspace's device status bits
 * (NVFP4_DEVICE_*) to *status, and clear them.  Not for the hot path.
 */
int nvfp4_read_device_status(void* ws, size_t ws_bytes, uint32_t* status, cudaStream_t stream);

/* Human-readable name of a status code (static string). */
const char* nvfp4_status_string(int status);

/* The cudaError_t of the last call that returned NVFP4_ERR_CUDA on this thread. */
int nvfp4_last_cuda_error(void);

/* Diagnostic: kernels this library has launched in this process (all threads;
 * a launch recorded into a CUDA graph counts once, at capture). */
uint64_t nvfp4_kernel_launches(void);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_H_ */
