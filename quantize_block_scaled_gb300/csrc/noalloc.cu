// nvfp4_quantize_noalloc: nvfp4_quantize with its scratch in a static
// device array instead of a caller-supplied workspace.
//
// Who needs it: a caller that may not allocate device memory at all, such
// as an engine that hands every byte of HBM to its own arena at start-up
// (a cudaMalloc from a library then fails or eats into that budget), or a
// latency-critical thread where cudaMalloc/cudaFree are off limits because
// they can block on, or synchronise, the whole device.  Such a caller still
// owns its inputs and outputs; only the scratch moves into the library.
//
// The scratch is the same 256-byte block the workspace path uses: the
// grid-wide amax slot and the block counters of the amax and one-pass kernels
// (zero when a kernel starts) and the device status word.  It lives in
// one file-scope array per device, so every call on a device shares it and
// calls that run at the same time on the GPU (two streams, no ordering)
// race on it.

#include <cstddef>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "nvfp4.h"

namespace {

// Maximum scratch one call may use; the array is held by every GPU that
// loads the library, until the process exits.
constexpr size_t kNoallocScratchBytes = 256;
static_assert(kNoallocScratchBytes >= nvfp4::kWorkspaceBytes, "static scratch too small");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of this device's copy of the array (set up on first use;
// host code may not use the symbol itself as an address).  Cached per device
// ordinal: the runtime's primary context is the one context per device.
int scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return static_cast<int>(e);
  if (dev < 0 || dev >= kMaxDevices) return static_cast<int>(cudaErrorInvalidDevice);
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return static_cast<int>(e);
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return 0;
}

}  // namespace

extern "C" int nvfp4_quantize_noalloc(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld_x,
                                      uint8_t* q, uint8_t* sf, float* gs, cudaStream_t stream) {
  if (nvfp4_workspace_bytes(NVFP4_OP_QUANTIZE, rows, cols, 0, 0) > kNoallocScratchBytes) return NVFP4_ERR_WORKSPACE;
  // nvfp4_quantize's own argument checks, made here first so that a refused
  // call touches neither the scratch nor the stream.
  const auto misaligned = [](const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a != 0; };
  if (gs == nullptr || (rows != 0 && (x == nullptr || q == nullptr || sf == nullptr)))
    return NVFP4_ERR_INVALID;
  if (rows < 0 || cols <= 0 || ld_x < cols) return NVFP4_ERR_INVALID;
  if (cols % 16 != 0 || ld_x % 8 != 0 || misaligned(x, 16) || misaligned(q, 8) || misaligned(gs, 4))
    return NVFP4_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const int rc = scratch_for_current_device(&scratch);
  if (rc != 0) {
    nvfp4::set_last_cuda_error(rc);
    return NVFP4_ERR_CUDA;
  }
  // The amax slot and the two block counters (the first three words) must
  // start at zero; the kernels leave them zeroed, but a call that never
  // finished could have left anything behind, so they are cleared on the
  // caller's stream.
  static_assert(offsetof(nvfp4::Workspace, amax_bits) == 0 && offsetof(nvfp4::Workspace, done) == 4 &&
                    offsetof(nvfp4::Workspace, depart) == 8,
                "cleared words");
  const cudaError_t e = cudaMemsetAsync(scratch, 0, 3 * sizeof(uint32_t), stream);
  if (e != cudaSuccess) {
    nvfp4::set_last_cuda_error(static_cast<int>(e));
    return NVFP4_ERR_CUDA;
  }
  return nvfp4_quantize(x, rows, cols, ld_x, q, sf, gs, scratch, kNoallocScratchBytes, stream);
}
