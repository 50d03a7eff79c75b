// fa_noalloc.cu -- fa_bwd_noalloc: the backward for callers that cannot
// allocate device memory.
//
// Some callers are handed only their input and output buffers and may not
// allocate device memory on their own: plugins inside inference engines that
// enqueue work into buffers the engine planned in advance, or code that must
// not call cudaMalloc while it submits work.  fa_bwd needs a workspace for
// D = rowsum(O o dO) and the log2-domain LSE; this entry point takes that
// scratch from a fixed, statically sized device array owned by the library
// instead, so the caller passes only inputs and outputs.
//
// The array below lives in every GPU that loads the library until the process
// exits.  Host code must not use its name as a device address (on the host it
// is only a stand-in); the device address is looked up once per device with
// cudaGetSymbolAddress, with that device current, and handed to the kernels.
#include "../../include/fa.h"

#include <cuda_runtime.h>

#include <mutex>

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;   // FA_NOALLOC_SCRATCH_BYTES
static_assert(kScratchBytes == FA_NOALLOC_SCRATCH_BYTES, "keep the header limit in step");

// D and log2-LSE of the backward, [B*H][ceil(Nq/128)*128] float32 each.
static __device__ __align__(256) float g_bwd_scratch[kScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices];

// Device address of this device's copy of g_bwd_scratch (looked up on the
// first call made with that device current).
fa_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_bwd_scratch) != cudaSuccess || ptr == nullptr) return FA_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return FA_OK;
}

}  // namespace

extern "C" fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                                    const float* lse, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk,
                                    int d, float sm_scale, int causal, fa_dtype dtype, void* stream) {
  // Reject problems whose scratch does not fit before touching the device.
  // The scratch holds the two-pass backward's D and log2-LSE only, so this
  // entry point always takes that path.
  if (fa_bwd_workspace_bytes_path(B, H, Nq, Nk, d, FA_BWD_PATH_TWO_PASS) > kScratchBytes) return FA_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (B > 0 && H > 0 && Nq > 0) {
    const fa_status st = scratch_for_current_device(&scratch);
    if (st != FA_OK) return st;
  }
  // The preprocess launch overwrites every scratch entry the two later
  // launches read (padding rows included), so stale contents from an earlier
  // call need no clearing.
  return fa_bwd_ex(FA_BWD_PATH_TWO_PASS, 0, q, k, v, o, dout, lse, dq, dk, dv, B, H, Nq, Nk, d, sm_scale, causal,
                   dtype, nullptr, scratch, kScratchBytes, stream);
}
