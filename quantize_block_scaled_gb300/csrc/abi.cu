// The C ABI of libnvfp4: argument validation, then kernel launches on the
// caller's stream.  Nothing here allocates or synchronises (except the
// diagnostic nvfp4_read_device_status).

#include <atomic>
#include <cstdint>

#include "internal.h"
#include "nvfp4.h"

namespace {

thread_local int g_last_cuda_error = 0;
std::atomic<uint64_t> g_launches{0};

int cuda_failure(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return NVFP4_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_workspace(const void* ws, size_t ws_bytes) {
  if (ws == nullptr || ws_bytes < nvfp4::kWorkspaceBytes || !aligned(ws, 4)) return NVFP4_ERR_WORKSPACE;
  return NVFP4_OK;
}

constexpr int64_t kInt32Max = 2147483647;

}  // namespace

namespace nvfp4 {

int sm_count() {
  static int cache[128] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 152;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
    cache[dev] = n;
  }
  return cache[dev];
}

void set_last_cuda_error(int e) { g_last_cuda_error = e; }

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

}  // namespace nvfp4

extern "C" {

size_t nvfp4_workspace_bytes(int op, int64_t rows, int64_t cols, int64_t n, int k) {
  if (op < NVFP4_OP_QUANTIZE || op > NVFP4_OP_MHC_RMSNORM_QUANTIZE || rows < 0 || cols < 0 || n < 0 || k < 0)
    return 0;
  return nvfp4::kWorkspaceBytes;  // cross-CTA counters only, whatever the shape
}

int nvfp4_workspace_init(void* ws, size_t ws_bytes, cudaStream_t stream) {
  const int st = check_workspace(ws, ws_bytes);
  if (st != NVFP4_OK) return st;
  const cudaError_t e = cudaMemsetAsync(ws, 0, nvfp4::kWorkspaceBytes, stream);
  return e == cudaSuccess ? NVFP4_OK : cuda_failure(e);
}

int nvfp4_quantize(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld_x, uint8_t* q,
                   uint8_t* sf, float* gs, void* ws, size_t ws_bytes, cudaStream_t stream) {
  // With rows == 0 nothing is read from x or written to q/sf (they may be NULL); gs is written.
  if (gs == nullptr || (rows != 0 && (x == nullptr || q == nullptr || sf == nullptr)))
    return NVFP4_ERR_INVALID;
  if (rows < 0 || cols <= 0 || ld_x < cols) return NVFP4_ERR_INVALID;
  if (cols % 16 != 0 || ld_x % 8 != 0 || !aligned(x, 16) || !aligned(q, 8) || !aligned(gs, 4))
    return NVFP4_ERR_UNSUPPORTED;
  const int st = check_workspace(ws, ws_bytes);
  if (st != NVFP4_OK) return st;
  auto* w = static_cast<nvfp4::Workspace*>(ws);
  cudaError_t e = cudaSuccess;
  if (nvfp4::launch_quantize_onepass(x, rows, cols, ld_x, q, sf, gs, w, stream, &e))
    return e == cudaSuccess ? NVFP4_OK : cuda_failure(e);
  e = nvfp4::launch_amax(x, rows, cols, ld_x, gs, w, stream);
  if (e != cudaSuccess) return cuda_failure(e);
  e = nvfp4::launch_quantize(x, rows, cols, ld_x, q, sf, gs, stream);
  if (e != cudaSuccess) return cuda_failure(e);
  return NVFP4_OK;
}

int nvfp4_mhc_rmsnorm_quantize(const uint16_t* x, int64_t rows, int n_hc, int64_t cols, int64_t ld_x,
                               const uint16_t* a, const uint16_t* weight, float eps, uint8_t* q, uint8_t* sf,
                               float* gs, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (gs == nullptr || weight == nullptr ||
      (rows != 0 && (x == nullptr || a == nullptr || q == nullptr || sf == nullptr)))
    return NVFP4_ERR_INVALID;
  if (rows < 0 || n_hc < 1 || n_hc > 8 || cols <= 0 || ld_x < n_hc * cols || !(eps >= 0.0f) || eps > 3.4e38f)
    return NVFP4_ERR_INVALID;
  if (cols % 16 != 0 || cols > 8192 || ld_x % 8 != 0 || !aligned(x, 16) || !aligned(a, 2) ||
      !aligned(weight, 16) || !aligned(q, 8) || !aligned(gs, 4))
    return NVFP4_ERR_UNSUPPORTED;
  const int st = check_workspace(ws, ws_bytes);
  if (st != NVFP4_OK) return st;
  const cudaError_t e = nvfp4::launch_mhc_rmsnorm_quantize(x, rows, n_hc, cols, ld_x, a, weight, eps, q, sf, gs,
                                                           static_cast<nvfp4::Workspace*>(ws), stream);
  return e == cudaSuccess ? NVFP4_OK : cuda_failure(e);
}

int nvfp4_rmsnorm_quantize(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld_x,
                           const uint16_t* weight, float eps, uint8_t* q, uint8_t* sf, float* gs, void* ws,
                           size_t ws_bytes, cudaStream_t stream) {
  if (gs == nullptr || weight == nullptr || (rows != 0 && (x == nullptr || q == nullptr || sf == nullptr)))
    return NVFP4_ERR_INVALID;
  if (rows < 0 || cols <= 0 || ld_x < cols || !(eps >= 0.0f) || eps > 3.4e38f) return NVFP4_ERR_INVALID;
  if (cols % 16 != 0 || cols > 16384 || ld_x % 8 != 0 || !aligned(x, 16) || !aligned(weight, 16) ||
      !aligned(q, 8) || !aligned(gs, 4))
    return NVFP4_ERR_UNSUPPORTED;
  const int st = check_workspace(ws, ws_bytes);
  if (st != NVFP4_OK) return st;
  const cudaError_t e = nvfp4::launch_rmsnorm_quantize(x, rows, cols, ld_x, weight, eps, q, sf, gs,
                                                       static_cast<nvfp4::Workspace*>(ws), stream);
  return e == cudaSuccess ? NVFP4_OK : cuda_failure(e);
}

int nvfp4_deinterleave_quantize(const uint16_t* x, int64_t rows, int64_t inter, int granularity,
                                uint8_t* q, uint8_t* sf, float* gs, void* ws, size_t ws_bytes,
                                cudaStream_t stream) {
  if (gs == nullptr || (rows != 0 && (x == nullptr || q == nullptr || sf == nullptr)))
    return NVFP4_ERR_INVALID;
  if (rows < 0 || inter <= 0) return NVFP4_ERR_INVALID;
  if (granularity != 1 && granularity != 2 && granularity != 4 && granularity != 8 &&
      granularity != 16)
    return NVFP4_ERR_UNSUPPORTED;
  if (inter % 16 != 0 || !aligned(x, 16) || !aligned(q, 8) || !aligned(gs, 4))
    return NVFP4_ERR_UNSUPPORTED;
  const int st = check_workspace(ws, ws_bytes);
  if (st != NVFP4_OK) return st;
  auto* w = static_cast<nvfp4::Workspace*>(ws);
  cudaError_t e = cudaSuccess;
  if (nvfp4::launch_deinterleave_onepass(x, rows, inter, granularity, q, sf, gs, w, stream, &e))
    return e == cudaSuccess ? NVFP4_OK : cuda_failure(e);
  e = nvfp4::launch_amax(x, rows, 2 * inter, 2 * inter, gs, w, stream);
  if (e != cudaSuccess) return cuda_failure(e);
  e = nvfp4::launch_deinterleave_quantize(x, rows, inter, granularity, q, sf, gs, stream);
  if (e != cudaSuccess) return cuda_failure(e);
  return NVFP4_OK;
}

int nvfp4_gemm_topk(const uint8_t* qa, const uint8_t* sfa, const float* gsa, const uint8_t* qb,
                    const uint8_t* sfb, const float* gsb, int64_t M, int64_t N, int64_t K,
                    int epilogue, const float* bias, int k, int32_t* topk_idx, float* topk_score,
                    float* topk_weight, float* logits, void* ws, size_t ws_bytes,
                    cudaStream_t stream) {
  // With M == 0 the A operand and the outputs are never touched (they may be NULL).
  if (gsa == nullptr || qb == nullptr || sfb == nullptr || gsb == nullptr) return NVFP4_ERR_INVALID;
  if (M != 0 && (qa == nullptr || sfa == nullptr || topk_idx == nullptr || topk_score == nullptr))
    return NVFP4_ERR_INVALID;
  if (M < 0 || N < 1 || K < 1 || M > kInt32Max || N > kInt32Max || K > kInt32Max)
    return NVFP4_ERR_INVALID;
  if (epilogue != NVFP4_EPILOGUE_IDENTITY && epilogue != NVFP4_EPILOGUE_SQRT_SOFTPLUS_BIAS &&
      epilogue != NVFP4_EPILOGUE_SQRT_SOFTPLUS_BIAS_NORM)
    return NVFP4_ERR_INVALID;
  if (epilogue != NVFP4_EPILOGUE_IDENTITY && bias == nullptr) return NVFP4_ERR_INVALID;
  if (k < 1 || k > 1024) return NVFP4_ERR_INVALID;
  if (K % 64 != 0) return NVFP4_ERR_UNSUPPORTED;
  if (k > 32 && N > 4096) return NVFP4_ERR_UNSUPPORTED;
  if (epilogue == NVFP4_EPILOGUE_SQRT_SOFTPLUS_BIAS_NORM && k > 32) return NVFP4_ERR_UNSUPPORTED;
  if (!aligned(qa, 16) || !aligned(qb, 16) || !aligned(sfa, 4) || !aligned(sfb, 4) ||
      !aligned(gsa, 4) || !aligned(gsb, 4) || !aligned(topk_idx, 4) || !aligned(topk_score, 4) ||
      (topk_weight != nullptr && !aligned(topk_weight, 4)) || (logits != nullptr && !aligned(logits, 4)) ||
      (bias != nullptr && !aligned(bias, 4)))
    return NVFP4_ERR_UNSUPPORTED;
  const int st = check_workspace(ws, ws_bytes);
  if (st != NVFP4_OK) return st;
  nvfp4::GemmTopkArgs a;
  a.qa = qa;
  a.sfa = sfa;
  a.gsa = gsa;
  a.qb = qb;
  a.sfb = sfb;
  a.gsb = gsb;
  a.M = M;
  a.N = N;
  a.K = K;
  a.epilogue = epilogue;
  a.bias = bias;
  a.k = k;
  a.topk_idx = topk_idx;
  a.topk_score = topk_score;
  a.topk_weight = topk_weight;
  a.logits = logits;
  a.ws = static_cast<nvfp4::Workspace*>(ws);
  cudaError_t e = cudaSuccess;
  const int rc = nvfp4::launch_gemm_topk(a, stream, &e);
  if (rc == NVFP4_ERR_CUDA) return cuda_failure(e);
  return rc;
}

int nvfp4_indexer_topk(const uint8_t* qa, const uint8_t* sfa, const float* gsa, const uint8_t* qb,
                       const uint8_t* sfb, const float* gsb, int64_t tokens, int heads, int64_t N, int64_t K,
                       const float* head_w, int k, int32_t* topk_idx, float* topk_score, float* scores,
                       void* ws, size_t ws_bytes, cudaStream_t stream) {
  // With tokens == 0 nothing is launched (queries, weights and outputs may be NULL).
  if (gsa == nullptr || qb == nullptr || sfb == nullptr || gsb == nullptr) return NVFP4_ERR_INVALID;
  if (tokens != 0 && (qa == nullptr || sfa == nullptr || head_w == nullptr || topk_idx == nullptr ||
                      topk_score == nullptr))
    return NVFP4_ERR_INVALID;
  if (tokens < 0 || N < 1 || K < 1 || N > kInt32Max || K > kInt32Max) return NVFP4_ERR_INVALID;
  if (heads != 32 && heads != 64 && heads != 128) return NVFP4_ERR_UNSUPPORTED;
  if (tokens > kInt32Max || tokens * heads > kInt32Max) return NVFP4_ERR_INVALID;
  if (k < 1 || k > 1024) return NVFP4_ERR_INVALID;
  if (K % 64 != 0 || N > 4096) return NVFP4_ERR_UNSUPPORTED;
  if (!aligned(qa, 16) || !aligned(qb, 16) || !aligned(sfa, 4) || !aligned(sfb, 4) || !aligned(gsa, 4) ||
      !aligned(gsb, 4) || !aligned(head_w, 4) || !aligned(topk_idx, 4) || !aligned(topk_score, 4) ||
      (scores != nullptr && !aligned(scores, 4)))
    return NVFP4_ERR_UNSUPPORTED;
  const int st = check_workspace(ws, ws_bytes);
  if (st != NVFP4_OK) return st;
  nvfp4::GemmTopkArgs a;
  a.qa = qa;
  a.sfa = sfa;
  a.gsa = gsa;
  a.qb = qb;
  a.sfb = sfb;
  a.gsb = gsb;
  a.M = tokens * heads;
  a.N = N;
  a.K = K;
  a.epilogue = NVFP4_EPILOGUE_IDENTITY;
  a.bias = nullptr;
  a.k = k;
  a.topk_idx = topk_idx;
  a.topk_score = topk_score;
  a.topk_weight = nullptr;
  a.logits = scores;
  a.ws = static_cast<nvfp4::Workspace*>(ws);
  a.heads = heads;
  a.head_w = head_w;
  cudaError_t e = cudaSuccess;
  const int rc = nvfp4::launch_gemm_topk(a, stream, &e);
  if (rc == NVFP4_ERR_CUDA) return cuda_failure(e);
  return rc;
}

int nvfp4_grouped_swiglu_gemm(const uint8_t* qa, const uint8_t* sfa, const float* gsa, const uint8_t* qb,
                              const uint8_t* sfb, const float* gsb, const int32_t* offsets, int64_t M, int64_t E,
                              int64_t inter, int64_t K, int granularity, float limit, int layout, uint16_t* out,
                              int64_t ld_out, void* ws, size_t ws_bytes, cudaStream_t stream) {
  // With M == 0 nothing is launched (A, the offsets and out may be NULL).
  if (gsa == nullptr || qb == nullptr || sfb == nullptr || gsb == nullptr) return NVFP4_ERR_INVALID;
  if (M != 0 && (qa == nullptr || sfa == nullptr || offsets == nullptr || out == nullptr))
    return NVFP4_ERR_INVALID;
  if (M < 0 || M > kInt32Max || E < 1 || inter < 1 || inter > kInt32Max || K < 1 || K > kInt32Max)
    return NVFP4_ERR_INVALID;
  if (E > 1024) return NVFP4_ERR_UNSUPPORTED;
  if (layout != 0 && layout != 1) return NVFP4_ERR_INVALID;
  if (!(limit > 0.0f)) return NVFP4_ERR_INVALID;  // also rejects NaN
  if (granularity != 1 && granularity != 2 && granularity != 4 && granularity != 8 && granularity != 16)
    return NVFP4_ERR_UNSUPPORTED;
  if (inter % 128 != 0 || K % 256 != 0) return NVFP4_ERR_UNSUPPORTED;
  if (E * 2 * inter > kInt32Max) return NVFP4_ERR_UNSUPPORTED;
  if (ld_out < (layout == 0 ? inter : 2 * inter) || ld_out % 8 != 0) return NVFP4_ERR_UNSUPPORTED;
  if ((M / 128 + E) * (2 * inter / 256) > kInt32Max) return NVFP4_ERR_UNSUPPORTED;
  if (!aligned(qa, 16) || !aligned(sfa, 16) || !aligned(qb, 16) || !aligned(sfb, 16) || !aligned(gsa, 4) ||
      !aligned(gsb, 4) || !aligned(offsets, 4) || !aligned(out, 16))
    return NVFP4_ERR_UNSUPPORTED;
  const int st = check_workspace(ws, ws_bytes);
  if (st != NVFP4_OK) return st;
  nvfp4::GroupedSwigluArgs a;
  a.qa = qa;
  a.sfa = sfa;
  a.gsa = gsa;
  a.qb = qb;
  a.sfb = sfb;
  a.gsb = gsb;
  a.offsets = offsets;
  a.M = M;
  a.E = E;
  a.inter = inter;
  a.K = K;
  a.granularity = granularity;
  a.limit = limit;
  a.layout = layout;
  a.out = out;
  a.ld_out = ld_out;
  a.ws = static_cast<nvfp4::Workspace*>(ws);
  cudaError_t e = cudaSuccess;
  const int rc = nvfp4::launch_grouped_swiglu(a, stream, &e);
  if (rc == NVFP4_ERR_CUDA) return cuda_failure(e);
  return rc;
}

int nvfp4_read_device_status(void* ws, size_t ws_bytes, uint32_t* status, cudaStream_t stream) {
  if (status == nullptr) return NVFP4_ERR_INVALID;
  const int st = check_workspace(ws, ws_bytes);
  if (st != NVFP4_OK) return st;
  auto* w = static_cast<nvfp4::Workspace*>(ws);
  uint32_t host = 0;
  cudaError_t e = cudaMemcpyAsync(&host, &w->status, sizeof(host), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(&w->status, 0, sizeof(uint32_t), stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_failure(e);
  *status = host;
  return NVFP4_OK;
}

const char* nvfp4_status_string(int status) {
  switch (status) {
    case NVFP4_OK: return "ok";
    case NVFP4_ERR_INVALID: return "invalid argument";
    case NVFP4_ERR_UNSUPPORTED: return "unsupported shape or alignment";
    case NVFP4_ERR_WORKSPACE: return "workspace missing or too small";
    case NVFP4_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

int nvfp4_last_cuda_error(void) { return g_last_cuda_error; }

uint64_t nvfp4_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
