// Internal declarations shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime_api.h>

namespace nvfp4 {

// Layout of the caller's workspace.  Every kernel that touches a field puts
// it back to zero before it finishes, so the buffer stays zeroed between
// calls.
struct Workspace {
  uint32_t amax_bits;  // running max of |x| as FP32 bits (valid for x >= 0)
  uint32_t done;       // blocks of the amax kernel that have finished (one-pass kernel: arrived)
  uint32_t depart;     // one-pass quantize kernel: blocks that have finished
  uint32_t status;     // NVFP4_DEVICE_* bits; cleared by nvfp4_read_device_status
  uint32_t reserved[60];
};
static_assert(sizeof(Workspace) == 256, "workspace layout");
constexpr size_t kWorkspaceBytes = sizeof(Workspace);

int sm_count();
// Record a cudaError_t for nvfp4_last_cuda_error on this thread.
void set_last_cuda_error(int e);
// Count one kernel launch issued by the library (nvfp4_kernel_launches).
void count_launch();

// One-pass quantize (single cooperative launch) for inputs that fit in the
// SMs' shared memory.  Returns false, having launched nothing, when the input
// is empty or too large; otherwise *err is the launch status.
bool launch_quantize_onepass(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, uint8_t* q,
                             uint8_t* sf, float* gs, Workspace* ws, cudaStream_t stream, cudaError_t* err);
bool launch_deinterleave_onepass(const uint16_t* x, int64_t rows, int64_t inter, int g, uint8_t* q,
                                 uint8_t* sf, float* gs, Workspace* ws, cudaStream_t stream,
                                 cudaError_t* err);

// RMSNorm (bf16 out) fused into the quantize: one pass when the rows fit on
// chip, else two row-parallel passes.
cudaError_t launch_rmsnorm_quantize(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                                    const uint16_t* weight, float eps, uint8_t* q, uint8_t* sf, float* gs,
                                    Workspace* ws, cudaStream_t stream);

// mHC pre-mix of n_hc streams per token (x: token stride ld, streams cols
// apart) by amap [rows, n_hc], then the same RMSNorm + quantize.
cudaError_t launch_mhc_rmsnorm_quantize(const uint16_t* x, int64_t rows, int n_hc, int64_t cols, int64_t ld,
                                        const uint16_t* amap, const uint16_t* weight, float eps, uint8_t* q,
                                        uint8_t* sf, float* gs, Workspace* ws, cudaStream_t stream);

cudaError_t launch_amax(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, float* gs,
                        Workspace* ws, cudaStream_t stream);

cudaError_t launch_quantize(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, uint8_t* q,
                            uint8_t* sf, const float* gs, cudaStream_t stream);

cudaError_t launch_deinterleave_quantize(const uint16_t* x, int64_t rows, int64_t inter, int g,
                                         uint8_t* q, uint8_t* sf, const float* gs,
                                         cudaStream_t stream);

struct GemmTopkArgs {
  const uint8_t* qa;
  const uint8_t* sfa;
  const float* gsa;
  const uint8_t* qb;
  const uint8_t* sfb;
  const float* gsb;
  int64_t M, N, K;
  int epilogue;
  const float* bias;
  int k;
  int32_t* topk_idx;
  float* topk_score;
  float* topk_weight;
  float* logits;
  Workspace* ws;
  int heads = 0;                  // indexer head reduction (A rows per token), 0 = off
  const float* head_w = nullptr;  // [M / heads, heads]
};

// Returns an nvfp4_status; on NVFP4_ERR_CUDA the CUDA error is in *err.
int launch_gemm_topk(const GemmTopkArgs& a, cudaStream_t stream, cudaError_t* err);

// Tensor map of a 2-D byte matrix [rows, width] (row stride = width) with
// boxes of box_w bytes x box_rows rows, optional 128-byte swizzle; reads past
// the matrix return zeros.  False if the driver refuses it.
bool make_map(CUtensorMap* map, const uint8_t* base, int64_t rows, int64_t width, int box_w,
              int box_rows, bool swizzle128);

struct GroupedSwigluArgs {
  const uint8_t* qa;
  const uint8_t* sfa;
  const float* gsa;
  const uint8_t* qb;
  const uint8_t* sfb;
  const float* gsb;        // [E]
  const int32_t* offsets;  // [E + 1], device
  int64_t M, E, inter, K;
  int granularity;
  float limit;
  int layout;
  uint16_t* out;
  int64_t ld_out;
  Workspace* ws;
};

int launch_grouped_swiglu(const GroupedSwigluArgs& a, cudaStream_t stream, cudaError_t* err);

}  // namespace nvfp4
