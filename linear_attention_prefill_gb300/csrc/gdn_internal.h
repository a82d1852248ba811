// gdn_internal.h - launch parameters shared by the C ABI layer and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

// One chunked-prefill forward call (sizes already validated by the ABI layer).
struct FwdParams {
  const void* q;      // [B, T, Hqk, dk]
  const void* k;      // [B, T, Hqk, dk]
  const void* v;      // [B, T, Hv, dv]
  const float* g;     // [B, T, Hv]
  const float* beta;  // [B, T, Hv]
  const float* h0;    // [N, Hv, dk, dv] or nullptr
  void* o;            // [B, T, Hv, dv]
  float* hT;          // [N, Hv, dk, dv] or nullptr
  const int32_t* cu_seqlens;  // [N + 1] or nullptr
  int N;              // sequences
  int T;              // tokens per row (packed total with cu_seqlens)
  int Hqk, Hv, dk, dv, chunk;
  float scale;
};

// One decode step.
struct StepParams {
  const void* q;      // [N, Hqk, dk]
  const void* k;      // [N, Hqk, dk]
  const void* v;      // [N, Hv, dv]
  const float* g;     // [N, Hv]
  const float* beta;  // [N, Hv]
  float* h;           // [N, Hv, dk, dv], in place
  void* o;            // [N, Hv, dv]
  int N, Hqk, Hv, dk, dv;
  float scale;
};

// Launchers: return cudaSuccess or the launch error.  Each validates nothing.
cudaError_t launch_fwd_bf16(const FwdParams& p, cudaStream_t stream);
cudaError_t launch_fwd_f32(const FwdParams& p, cudaStream_t stream);
cudaError_t launch_step_bf16(const StepParams& p, cudaStream_t stream);
cudaError_t launch_step_f32(const StepParams& p, cudaStream_t stream);

// The device error word (bounded waits); defined in gdn_abi.cu.
cudaError_t read_and_clear_device_error(unsigned* out, cudaStream_t stream);

}  // namespace gdn
