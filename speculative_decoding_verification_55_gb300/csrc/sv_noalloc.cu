// spec_verify_noalloc: the verifier for callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: engines whose device memory is fully
// planned at start-up and that forbid any allocation on the serving path, host code that cannot
// afford the device-wide synchronisation of cudaMalloc, and plugin interfaces that pass only the
// input and output buffers. This entry point serves them. It runs the same kernels as spec_verify,
// with the kernels' scratch (per-position records, per-row arrival counters, status word) in a
// file-scope static device array of SV_NOALLOC_SCRATCH_BYTES instead of a caller workspace.
//
// The array is part of the loaded library: every GPU that loads it holds it until the process
// exits. In host code `g_noalloc_scratch` is only a host-side stand-in for the device array, never
// a device address; the device address comes from cudaGetSymbolAddress, called once per device at
// set-up with that device current.

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/spec_verify.h"
#include "sv_common.cuh"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[SV_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64];                 // device address of the array, per device (set-up done)

// Set-up for the current device: the array's device address, looked up once per device.
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return SV_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return SV_OK;
}

}  // namespace

extern "C" int spec_verify_noalloc(const void* target_logits, const void* draft_logits,
                                   const int32_t* draft_tokens, const int32_t* draft_len,
                                   const float* temperature, const float* uniforms,
                                   int32_t* out_tokens, int32_t* out_num_emitted, float* out_alpha,
                                   float* out_p_draft, float* out_q_draft,
                                   int32_t B, int32_t gamma_max, int32_t V, int32_t dtype,
                                   void* cuda_stream) {
  const size_t need = spec_verify_workspace_size(B, gamma_max, V, dtype);
  if (need == 0) {
    if (dtype != SV_DTYPE_F32 && dtype != SV_DTYPE_BF16) return SV_ERR_BAD_DTYPE;
    return SV_ERR_BAD_SHAPE;
  }
  if (need > SV_NOALLOC_SCRATCH_BYTES) return SV_ERR_SCRATCH_TOO_SMALL;
  // The checks spec_verify_ex makes, first: a rejected call enqueues nothing and returns the status
  // spec_verify_ex would return.
  const int args = sv::verify_args_status(target_logits, draft_logits, draft_tokens, draft_len,
                                          temperature, uniforms, out_tokens, out_num_emitted,
                                          out_alpha, out_p_draft, out_q_draft, B, gamma_max, V,
                                          dtype);
  if (args != SV_OK) return args;
  void* scratch = nullptr;
  const int st = noalloc_scratch(&scratch);
  if (st != SV_OK) return st;
  // The array keeps whatever the previous call left: per-position records, row counters and the
  // status word must start at zero, and a call that gave up part-way leaves stale records. Clear
  // this call's whole layout on the caller's stream before the launch.
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  if (cudaMemsetAsync(scratch, 0, need, stream) != cudaSuccess) return SV_ERR_CUDA;
  return spec_verify_ex(target_logits, draft_logits, draft_tokens, draft_len, temperature, uniforms,
                        out_tokens, out_num_emitted, out_alpha, out_p_draft, out_q_draft, B,
                        gamma_max, V, dtype, scratch, SV_NOALLOC_SCRATCH_BYTES, cuda_stream);
}
