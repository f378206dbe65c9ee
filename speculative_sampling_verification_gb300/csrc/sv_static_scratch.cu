// spec_verify_static: the verification step for callers that cannot allocate
// device memory, with its scratch in a fixed array inside this library.
//
// Some callers cannot obtain a workspace for spec_verify:
//   - code running while a stream is being captured into a CUDA graph in the
//     global or thread-local capture mode, where cudaMalloc is not permitted;
//   - plugins and custom operators inside a host framework whose device
//     memory must all come from the framework's own pool, where a raw
//     cudaMalloc would escape its accounting;
//   - latency-critical decode loops, where cudaMalloc may synchronise the
//     device and stall the loop.
// This entry point needs no workspace: the scratch is a file-scope array of
// kStaticScratchBytes in device memory, which every GPU that loads the
// library holds until the process exits.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/spec_verify.h"

namespace {

constexpr size_t kStaticScratchBytes = SV_STATIC_SCRATCH_BYTES;

// The scratch itself. In host code this name is only a stand-in for the
// device array: the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

void* g_scratch_ptr[64] = {};
std::mutex g_scratch_mu;

// Device address of the scratch on `device` (which must be current). The
// address belongs to the current context, so outside stream capture it is
// looked up afresh on every call: a context created after cudaDeviceReset, or
// another context made current by the driver API, gets its own address. While
// `stream` is being captured the last address looked up on this device is
// used instead, so that the capture makes no lookup; a call made outside
// capture on the same device and context must come first.
cudaError_t scratch_address(int device, cudaStream_t stream, void** out) {
  if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[device] = p;
  } else if (!g_scratch_ptr[device]) {
    return cudaErrorStreamCaptureUnsupported;
  }
  *out = g_scratch_ptr[device];
  return cudaSuccess;
}

}  // namespace

extern "C" int spec_verify_static(const void* target_logits, const void* draft_logits,
                                  const int32_t* draft_tokens, const float* uniforms, int B,
                                  int K, int V, int dtype, float temperature,
                                  int32_t* out_tokens, int32_t* n_accepted, void* stream) {
  const size_t need = sv_workspace_size(B, K, V, dtype);
  if (need > kStaticScratchBytes) return SV_ERR_SCRATCH_LIMIT;
  if (need == 0 || B == 0) {
    // Invalid sizes, or nothing to do: spec_verify reports which, touching no device.
    return spec_verify(target_logits, draft_logits, draft_tokens, uniforms, B, K, V, dtype,
                       temperature, out_tokens, n_accepted, nullptr, 0, stream);
  }
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return SV_ERR_CUDA;
  void* scratch = nullptr;
  if (scratch_address(device, static_cast<cudaStream_t>(stream), &scratch) != cudaSuccess)
    return SV_ERR_CUDA;
  return spec_verify(target_logits, draft_logits, draft_tokens, uniforms, B, K, V, dtype,
                     temperature, out_tokens, n_accepted, scratch, kStaticScratchBytes, stream);
}
