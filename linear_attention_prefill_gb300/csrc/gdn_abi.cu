// gdn_abi.cu - the extern "C" boundary of libgdn.so (declared in include/gdn.h).
//
// Validates arguments, maps them onto launch parameters and enqueues the kernels
// on the caller's stream.  It owns no tensors and allocates nothing.
#include <stdarg.h>
#include <stdlib.h>
#include <stdio.h>
#include <string.h>

#include "../../include/gdn.h"
#include "gdn_common.cuh"
#include "gdn_internal.h"

#ifdef GDN_PROFILE
__device__ unsigned long long g_gdn_phase[64];
#endif

namespace gdn {

__device__ unsigned g_device_error = 0u;

cudaError_t read_and_clear_device_error(unsigned* out, cudaStream_t stream) {
  unsigned zero = 0u;
  cudaError_t err = cudaMemcpyFromSymbolAsync(out, g_device_error, sizeof(unsigned), 0,
                                              cudaMemcpyDeviceToHost, stream);
  if (err == cudaSuccess) err = cudaStreamSynchronize(stream);
  if (err == cudaSuccess && *out != 0u)
    err = cudaMemcpyToSymbolAsync(g_device_error, &zero, sizeof(unsigned), 0,
                                  cudaMemcpyHostToDevice, stream);
  if (err == cudaSuccess) err = cudaStreamSynchronize(stream);
  return err;
}

// Diagnostic: one warp waits on an mbarrier that nothing ever completes, with a
// limit of `limit` cycles; the expired wait records kErrWaitTimeout in the error
// word and the kernel returns normally (no trap, no fault, nothing left pending).
__global__ void selftest_expired_wait_kernel(unsigned* err, long long limit) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) mbar_wait_limit(&bar, 0, err, limit);
}

// Input check of an _ex call: every log-decay g <= 0 and finite (with the fused
// prologue the raw gate only finite), every beta in [0, 1] (raw: finite), and
// cu_seqlens running from 0 to T without going down.  The first violation records
// kErrInput in the error word; nothing is modified.
__global__ void check_inputs_kernel(const float* g, long long n_g, const float* beta, long long n_b,
                                    const int32_t* cu, int N, int T, int raw, unsigned* err) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  bool ok = true;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n_g; i += stride) {
    const float x = g[i];
    ok &= raw ? isfinite(x) : (isfinite(x) && x <= 0.f);
  }
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n_b; i += stride) {
    const float x = beta[i];
    ok &= raw ? isfinite(x) : (x >= 0.f && x <= 1.f);
  }
  if (cu) {
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i <= N; i += stride) {
      const int a = cu[i];
      if (i == 0) ok &= a == 0;
      if (i == N) ok &= a == T;
      if (i > 0) ok &= a >= cu[i - 1];
    }
  }
  if (!ok) record_error(err, kErrInput);
}

cudaError_t launch_check_inputs(const FwdParams& p, cudaStream_t stream) {
  const long long rows = p.cu_seqlens ? 1ll : (long long)p.N;
  const long long n_b = rows * p.T * p.Hv;
  const long long n_g = n_b * (p.kda ? p.dk : 1);
  int blocks = (int)((n_g + 255) / 256);
  if (blocks > 1216) blocks = 1216;
  if (blocks < 1) blocks = 1;
  check_inputs_kernel<<<blocks, 256, 0, stream>>>(p.g, n_g, p.beta, n_b, p.cu_seqlens, p.N, p.T,
                                                  p.prologue, p.err);
  return cudaGetLastError();
}

}  // namespace gdn

namespace {

thread_local char t_last_error[512] = "";

gdn_status fail(gdn_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
  va_end(ap);
  return s;
}

gdn_status cuda_fail(cudaError_t e, const char* what) {
  return fail(GDN_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool head_dim_ok(int d) { return d == 64 || d == 128; }

// Shared validation of the forward; fills FwdParams.  elem = bytes of q/k/v/o.
gdn_status check_fwd(const void* q, const void* k, const void* v, const float* g,
                     const float* beta, const float* h0, void* o, float* hT, int B, int T,
                     int Hqk, int Hv, int dk, int dv, int chunk, float scale,
                     const int32_t* cu_seqlens, int elem, gdn::FwdParams* p) {
  if (B < 0 || T < 0) return fail(GDN_ERR_INVALID_ARG, "B=%d and T=%d must be >= 0", B, T);
  if (Hqk <= 0 || Hv <= 0) return fail(GDN_ERR_INVALID_ARG, "Hqk=%d, Hv=%d must be > 0", Hqk, Hv);
  if (Hv % Hqk != 0) return fail(GDN_ERR_INVALID_ARG, "Hv=%d is not a multiple of Hqk=%d", Hv, Hqk);
  if (!head_dim_ok(dk) || !head_dim_ok(dv))
    return fail(GDN_ERR_UNSUPPORTED, "dk=%d, dv=%d: supported head dims are 64 and 128", dk, dv);
  if (chunk != 64 && chunk != 128)
    return fail(GDN_ERR_UNSUPPORTED, "chunk=%d: supported chunk lengths are 64 and 128", chunk);
  if (!(scale == scale)) return fail(GDN_ERR_INVALID_ARG, "scale is NaN");
  if (cu_seqlens && B < 1) return fail(GDN_ERR_INVALID_ARG, "cu_seqlens needs B >= 1 sequences");
  const long long rows = cu_seqlens ? 1 : (long long)B;
  const long long tokens = rows * (long long)T;
  // every element index must fit comfortably in 63 bits and the grid in 2^31
  if (tokens > (1ll << 40) || (long long)B * Hv * 2 > 0x7fffffffll)
    return fail(GDN_ERR_INVALID_ARG, "problem too large: B=%d T=%d Hv=%d", B, T, Hv);
  if (tokens > 0) {
    if (!q || !k || !v || !g || !beta || !o)
      return fail(GDN_ERR_INVALID_ARG, "q, k, v, g, beta and o must be non-NULL when T > 0");
  }
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
    return fail(GDN_ERR_INVALID_ARG, "q, k, v and o must be 16-byte aligned");
  if (!aligned(g, 4) || !aligned(beta, 4))
    return fail(GDN_ERR_INVALID_ARG, "g and beta must be 4-byte aligned");
  if (!aligned(h0, 16) || !aligned(hT, 16) || !aligned(cu_seqlens, 4))
    return fail(GDN_ERR_INVALID_ARG, "h0 and hT must be 16-byte aligned, cu_seqlens 4-byte");
  (void)elem;
  p->q = q; p->k = k; p->v = v; p->g = g; p->beta = beta; p->h0 = h0; p->o = o; p->hT = hT;
  p->cu_seqlens = cu_seqlens;
  p->err = nullptr;
  p->N = B; p->T = T; p->Hqk = Hqk; p->Hv = Hv; p->dk = dk; p->dv = dv; p->chunk = chunk;
  p->scale = scale;
  p->delta_rule = 1;
  p->prologue = 0;
  p->A_log = nullptr;
  p->dt_bias = nullptr;
  p->kda = 0;
  p->head_map = 0;
  p->tc_chain = 0;
  return GDN_OK;
}

constexpr unsigned kFwdFlags =
    GDN_FLAG_HEAD_MAP_MODULO | GDN_FLAG_CHECK_INPUTS | GDN_FLAG_TC_CHAIN | GDN_FLAG_DV_TILE_CHAIN;

// Applies the flags of an _ex forward to p; `tc_ok` says whether the tcgen05 chain
// exists for this operation.
gdn_status apply_flags(unsigned flags, bool tc_ok, gdn::FwdParams* p) {
  if (flags & ~kFwdFlags) return fail(GDN_ERR_INVALID_ARG, "unknown flag bits 0x%x", flags & ~kFwdFlags);
  if ((flags & GDN_FLAG_TC_CHAIN) && (flags & GDN_FLAG_DV_TILE_CHAIN))
    return fail(GDN_ERR_INVALID_ARG, "GDN_FLAG_TC_CHAIN and GDN_FLAG_DV_TILE_CHAIN together");
  if ((flags & GDN_FLAG_TC_CHAIN) && !tc_ok)
    return fail(GDN_ERR_UNSUPPORTED, "GDN_FLAG_TC_CHAIN: no tensor-memory chain for this operation");
  p->head_map = (flags & GDN_FLAG_HEAD_MAP_MODULO) ? 1 : 0;
  p->tc_chain = (flags & GDN_FLAG_TC_CHAIN) ? 1 : (flags & GDN_FLAG_DV_TILE_CHAIN) ? -1 : 0;
  return GDN_OK;
}

// T == 0 without cu_seqlens: no tokens, the final state is the initial one.
gdn_status empty_forward(const gdn::FwdParams& p, cudaStream_t stream) {
  if (!p.hT || p.N == 0) return GDN_OK;
  const size_t bytes = (size_t)p.N * p.Hv * p.dk * p.dv * sizeof(float);
  cudaError_t e = p.h0 ? (p.h0 == p.hT ? cudaSuccess
                                       : cudaMemcpyAsync(p.hT, p.h0, bytes,
                                                         cudaMemcpyDeviceToDevice, stream))
                       : cudaMemsetAsync(p.hT, 0, bytes, stream);
  if (e != cudaSuccess) return cuda_fail(e, "copying h0 to hT");
  return GDN_OK;
}

gdn_status check_step(const void* q, const void* k, const void* v, const float* g,
                      const float* beta, float* h, void* o, int N, int Hqk, int Hv, int dk,
                      int dv, float scale, gdn::StepParams* p) {
  if (N < 0) return fail(GDN_ERR_INVALID_ARG, "N=%d must be >= 0", N);
  if (Hqk <= 0 || Hv <= 0) return fail(GDN_ERR_INVALID_ARG, "Hqk=%d, Hv=%d must be > 0", Hqk, Hv);
  if (Hv % Hqk != 0) return fail(GDN_ERR_INVALID_ARG, "Hv=%d is not a multiple of Hqk=%d", Hv, Hqk);
  if (!head_dim_ok(dk) || !head_dim_ok(dv))
    return fail(GDN_ERR_UNSUPPORTED, "dk=%d, dv=%d: supported head dims are 64 and 128", dk, dv);
  if (!(scale == scale)) return fail(GDN_ERR_INVALID_ARG, "scale is NaN");
  if ((long long)N * Hv * 4 > 0x7fffffffll) return fail(GDN_ERR_INVALID_ARG, "N=%d too large", N);
  if (N > 0 && (!q || !k || !v || !g || !beta || !h || !o))
    return fail(GDN_ERR_INVALID_ARG, "q, k, v, g, beta, h and o must be non-NULL");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(h, 16) || !aligned(g, 4) || !aligned(beta, 4))
    return fail(GDN_ERR_INVALID_ARG, "misaligned pointer (16 bytes for tensors, 4 for g, beta)");
  p->q = q; p->k = k; p->v = v; p->g = g; p->beta = beta; p->h = h; p->o = o;
  p->N = N; p->Hqk = Hqk; p->Hv = Hv; p->dk = dk; p->dv = dv; p->scale = scale;
  p->delta_rule = 1;
  p->prologue = 0;
  p->A_log = nullptr;
  p->dt_bias = nullptr;
  p->kda = 0;
  p->head_map = 0;
  return GDN_OK;
}

// Kimi Delta Attention: the forward's checks plus dk = 128 and a 16-byte aligned
// per-channel gate g [B, T, Hv, dk].
gdn_status check_kda(const void* q, const void* k, const void* v, const float* g,
                     const float* beta, const float* h0, void* o, float* hT, int B, int T,
                     int Hqk, int Hv, int dk, int dv, int chunk, float scale,
                     const int32_t* cu_seqlens, gdn::FwdParams* p) {
  gdn_status s = check_fwd(q, k, v, g, beta, h0, o, hT, B, T, Hqk, Hv, dk, dv, chunk, scale,
                           cu_seqlens, 2, p);
  if (s != GDN_OK) return s;
  if (dk != 128) return fail(GDN_ERR_UNSUPPORTED, "dk=%d: the KDA forward takes dk = 128", dk);
  if (!aligned(g, 16)) return fail(GDN_ERR_INVALID_ARG, "g must be 16-byte aligned for KDA");
  p->kda = 1;
  return GDN_OK;
}

// fp32 forward: the chunk-parallel prep and the chain, on fp32 records in a workspace
// taken from the stream-ordered pool and given back after.
gdn_status run_fwd_f32(const gdn::FwdParams& p, cudaStream_t stream) {
  if (p.N == 0) return GDN_OK;
  if (!p.cu_seqlens && p.T == 0) return empty_forward(p, stream);
  gdn::WsLayout w = gdn::ws_layout(p, nullptr);
  const size_t bytes = (size_t)w.n_slots * p.Hv * gdn::f32_rec_bytes(p);
  void* ws = nullptr;
  cudaError_t e = cudaMallocAsync(&ws, bytes, stream);
  if (e != cudaSuccess) return cuda_fail(e, "allocating the workspace");
  w = gdn::ws_layout(p, ws);
  e = gdn::launch_fwd_f32(p, w, stream);
  const cudaError_t ef = cudaFreeAsync(ws, stream);
  if (e != cudaSuccess) return cuda_fail(e, "launching the forward kernels");
  if (ef != cudaSuccess) return cuda_fail(ef, "freeing the workspace");
  return GDN_OK;
}

gdn_status launch_pipeline(const gdn::FwdParams& p, const gdn::WsLayout& w, cudaStream_t stream);

// bf16 forward: the chunk-parallel prep launch, then the chunk-serial chain launch
// (which also writes the output).
gdn_status run_fwd_bf16(const gdn::FwdParams& p, void* ws, size_t ws_size, cudaStream_t stream,
                        bool check = false) {
  if (p.N == 0) return GDN_OK;
  if (!p.cu_seqlens && p.T == 0) return empty_forward(p, stream);
  // tensor-map row coordinates are 32-bit
  if ((p.cu_seqlens ? 1ll : (long long)p.N) * p.T > 0x7fffffffll)
    return fail(GDN_ERR_UNSUPPORTED, "%lld tokens: the bf16 path takes at most 2^31 - 1",
                (p.cu_seqlens ? 1ll : (long long)p.N) * p.T);
  gdn::FwdParams q = p;
  // the chain kind: forced by a flag (1 / -1), else by the number of chains
  q.tc_chain = q.tc_chain > 0 || (q.tc_chain == 0 && gdn::tc_chain_pays(q)) ? 1 : 0;
  const gdn::WsLayout w = gdn::ws_layout(q, ws);
  if (!ws || (reinterpret_cast<uintptr_t>(ws) % 256) != 0 || ws_size < gdn::ws_bytes(w, p.Hv))
    return fail(GDN_ERR_INVALID_ARG, "workspace %p of %zu bytes: need %zu bytes, 256-byte aligned",
                ws, ws_size, gdn::ws_bytes(w, p.Hv));
  cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&q.err), gdn::g_device_error);
  if (e != cudaSuccess) return cuda_fail(e, "locating the device error word");
  if (check) {
    e = gdn::launch_check_inputs(q, stream);
    if (e != cudaSuccess) return cuda_fail(e, "launching the input check");
  }
  return launch_pipeline(q, w, stream);
}

gdn_status launch_pipeline(const gdn::FwdParams& p, const gdn::WsLayout& w, cudaStream_t stream) {
  if (p.tc_chain) {  // lookahead records, the tcgen05 chain
    cudaError_t e = gdn::launch_prep_tc(p, w, stream);
    if (e != cudaSuccess) return cuda_fail(e, "launching the prep kernel");
    e = gdn::launch_chain_tc(p, w, stream);
    if (e != cudaSuccess) return cuda_fail(e, "launching the chain kernel");
    return GDN_OK;
  }
  if (p.kda) {  // Kimi Delta Attention: its own prep, the mma.sync chain
    cudaError_t e = gdn::launch_kda_prep(p, w, stream);
    if (e != cudaSuccess) return cuda_fail(e, "launching the KDA prep kernel");
    e = gdn::launch_chain(p, w, stream);
    if (e != cudaSuccess) return cuda_fail(e, "launching the KDA chain kernel");
    return GDN_OK;
  }
  cudaError_t e = gdn::launch_prep(p, w, stream);
  if (e != cudaSuccess) return cuda_fail(e, "launching the prep kernel");
  e = gdn::launch_chain(p, w, stream);
  if (e != cudaSuccess) return cuda_fail(e, "launching the chain kernel");
  return GDN_OK;
}

// bf16 forward on a workspace taken from the stream-ordered pool and given back after.
gdn_status fwd_bf16_pooled(const gdn::FwdParams& p, cudaStream_t st) {
  if (p.N == 0 || (!p.cu_seqlens && p.T == 0)) return run_fwd_bf16(p, nullptr, 0, st);
  const size_t bytes = gdn::ws_bytes_any(p);
  void* ws = nullptr;
  cudaError_t e = cudaMallocAsync(&ws, bytes, st);
  if (e != cudaSuccess) return cuda_fail(e, "allocating the workspace");
  gdn_status s = run_fwd_bf16(p, ws, bytes, st);
  e = cudaFreeAsync(ws, st);
  if (s == GDN_OK && e != cudaSuccess) return cuda_fail(e, "freeing the workspace");
  return s;
}

gdn_status run_step(const gdn::StepParams& p, bool f32, cudaStream_t st, bool check = false) {
  if (p.N == 0) return GDN_OK;
  cudaError_t e;
  if (check) {  // the step's gates: one token of N rows
    gdn::FwdParams c{};
    c.g = p.g;
    c.beta = p.beta;
    c.N = p.N;
    c.T = 1;
    c.Hv = p.Hv;
    c.dk = p.dk;
    c.kda = p.kda;
    c.prologue = p.prologue;
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&c.err), gdn::g_device_error);
    if (e == cudaSuccess) e = gdn::launch_check_inputs(c, st);
    if (e != cudaSuccess) return cuda_fail(e, "launching the input check");
  }
  e = f32 ? gdn::launch_step_f32(p, st) : gdn::launch_step_bf16(p, st);
  return e == cudaSuccess ? GDN_OK : cuda_fail(e, "launching the decode step");
}

}  // namespace

extern "C" {

gdn_status gdn_chunk_fwd_ex(const void* q, const void* k, const void* v, const float* g,
                            const float* beta, const float* h0, void* o, float* hT, int B, int T,
                            int Hqk, int Hv, int dk, int dv, int chunk, float scale,
                            const int32_t* cu_seqlens, unsigned flags, void* workspace,
                            size_t workspace_bytes, gdn_stream_t stream) {
  gdn::FwdParams p;
  gdn_status s = check_fwd(q, k, v, g, beta, h0, o, hT, B, T, Hqk, Hv, dk, dv, chunk, scale,
                           cu_seqlens, 2, &p);
  if (s != GDN_OK) return s;
  s = apply_flags(flags, true, &p);
  if (s != GDN_OK) return s;
  return run_fwd_bf16(p, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream),
                      (flags & GDN_FLAG_CHECK_INPUTS) != 0);
}

size_t gdn_chunk_fwd_workspace_size(int B, int T, int Hqk, int Hv, int dk, int dv, int chunk,
                                    int has_cu_seqlens) {
  gdn::FwdParams p;
  static const int32_t fake_cu = 0;
  const void* A = reinterpret_cast<const void*>(static_cast<uintptr_t>(256));
  if (check_fwd(A, A, A, static_cast<const float*>(A), static_cast<const float*>(A), nullptr,
                const_cast<void*>(A), nullptr, B, T, Hqk, Hv, dk, dv, chunk, 1.0f,
                has_cu_seqlens ? &fake_cu : nullptr, 2, &p) != GDN_OK)
    return 0;
  return gdn::ws_bytes_any(p);
}

int gdn_chunk_fwd_chain_kind(int n_seqs, int Hv, int dk, int dv, int delta_rule, unsigned flags) {
  if (n_seqs < 0 || Hv <= 0 || (dk != 64 && dk != 128) || (dv != 64 && dv != 128)) return -1;
  if ((flags & ~kFwdFlags) ||
      ((flags & GDN_FLAG_TC_CHAIN) && (flags & GDN_FLAG_DV_TILE_CHAIN)))
    return -1;
  if (flags & GDN_FLAG_TC_CHAIN) return 1;
  if (flags & GDN_FLAG_DV_TILE_CHAIN) return 0;
  gdn::FwdParams p{};
  p.N = n_seqs;
  p.Hv = Hv;
  p.dk = dk;
  p.dv = dv;
  p.delta_rule = delta_rule ? 1 : 0;
  return gdn::tc_chain_pays(p) ? 1 : 0;
}

gdn_status gdn_chunk_fwd(const void* q, const void* k, const void* v, const float* g,
                         const float* beta, const float* h0, void* o, float* hT, int B, int T,
                         int Hqk, int Hv, int dk, int dv, int chunk, float scale,
                         const int32_t* cu_seqlens, gdn_stream_t stream) {
  gdn::FwdParams p;
  gdn_status s = check_fwd(q, k, v, g, beta, h0, o, hT, B, T, Hqk, Hv, dk, dv, chunk, scale,
                           cu_seqlens, 2, &p);
  if (s != GDN_OK) return s;
  return fwd_bf16_pooled(p, reinterpret_cast<cudaStream_t>(stream));
}

gdn_status gdn_chunk_fwd_f32(const float* q, const float* k, const float* v, const float* g,
                             const float* beta, const float* h0, float* o, float* hT, int B,
                             int T, int Hqk, int Hv, int dk, int dv, int chunk, float scale,
                             const int32_t* cu_seqlens, gdn_stream_t stream) {
  gdn::FwdParams p;
  gdn_status s = check_fwd(q, k, v, g, beta, h0, o, hT, B, T, Hqk, Hv, dk, dv, chunk, scale,
                           cu_seqlens, 4, &p);
  if (s != GDN_OK) return s;
  return run_fwd_f32(p, reinterpret_cast<cudaStream_t>(stream));
}

gdn_status gdn_recurrent_step(const void* q, const void* k, const void* v, const float* g,
                              const float* beta, float* h, void* o, int N, int Hqk, int Hv,
                              int dk, int dv, float scale, gdn_stream_t stream) {
  gdn::StepParams p;
  gdn_status s = check_step(q, k, v, g, beta, h, o, N, Hqk, Hv, dk, dv, scale, &p);
  if (s != GDN_OK) return s;
  return run_step(p, false, reinterpret_cast<cudaStream_t>(stream));
}

gdn_status gdn_recurrent_step_ex(const void* q, const void* k, const void* v, const float* g,
                                 const float* beta, float* h, void* o, int N, int Hqk, int Hv,
                                 int dk, int dv, float scale, unsigned flags,
                                 gdn_stream_t stream) {
  gdn::StepParams p;
  gdn_status s = check_step(q, k, v, g, beta, h, o, N, Hqk, Hv, dk, dv, scale, &p);
  if (s != GDN_OK) return s;
  constexpr unsigned kStepFlags = GDN_FLAG_HEAD_MAP_MODULO | GDN_FLAG_CHECK_INPUTS;
  if (flags & ~kStepFlags)
    return fail(GDN_ERR_INVALID_ARG, "flag bits 0x%x do not apply to the decode step",
                flags & ~kStepFlags);
  p.head_map = (flags & GDN_FLAG_HEAD_MAP_MODULO) ? 1 : 0;
  return run_step(p, false, reinterpret_cast<cudaStream_t>(stream),
                  (flags & GDN_FLAG_CHECK_INPUTS) != 0);
}

gdn_status gdn_recurrent_step_f32(const float* q, const float* k, const float* v,
                                  const float* g, const float* beta, float* h, float* o, int N,
                                  int Hqk, int Hv, int dk, int dv, float scale,
                                  gdn_stream_t stream) {
  gdn::StepParams p;
  gdn_status s = check_step(q, k, v, g, beta, h, o, N, Hqk, Hv, dk, dv, scale, &p);
  if (s != GDN_OK) return s;
  return run_step(p, true, reinterpret_cast<cudaStream_t>(stream));
}

// ---- the forward with the fused prologue ---------------------------------------
gdn_status gdn_chunk_fwd_prologue_ex(const void* q, const void* k, const void* v, const float* a,
                                     const float* b, const float* A_log, const float* dt_bias,
                                     const float* h0, void* o, float* hT, int B, int T, int Hqk,
                                     int Hv, int dk, int dv, int chunk, float scale,
                                     const int32_t* cu_seqlens, unsigned flags, void* workspace,
                                     size_t workspace_bytes, gdn_stream_t stream) {
  gdn::FwdParams p;
  gdn_status s = check_fwd(q, k, v, a, b, h0, o, hT, B, T, Hqk, Hv, dk, dv, chunk, scale,
                           cu_seqlens, 2, &p);
  if (s != GDN_OK) return s;
  if (!aligned(A_log, 4) || !aligned(dt_bias, 4))
    return fail(GDN_ERR_INVALID_ARG, "A_log and dt_bias must be 4-byte aligned");
  s = apply_flags(flags, true, &p);
  if (s != GDN_OK) return s;
  p.prologue = 1;
  p.A_log = A_log;
  p.dt_bias = dt_bias;
  return run_fwd_bf16(p, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream),
                      (flags & GDN_FLAG_CHECK_INPUTS) != 0);
}

gdn_status gdn_chunk_fwd_prologue(const void* q, const void* k, const void* v, const float* a,
                                  const float* b, const float* A_log, const float* dt_bias,
                                  const float* h0, void* o, float* hT, int B, int T, int Hqk,
                                  int Hv, int dk, int dv, int chunk, float scale,
                                  const int32_t* cu_seqlens, gdn_stream_t stream) {
  gdn::FwdParams p;
  gdn_status s = check_fwd(q, k, v, a, b, h0, o, hT, B, T, Hqk, Hv, dk, dv, chunk, scale,
                           cu_seqlens, 2, &p);
  if (s != GDN_OK) return s;
  if (!aligned(A_log, 4) || !aligned(dt_bias, 4))
    return fail(GDN_ERR_INVALID_ARG, "A_log and dt_bias must be 4-byte aligned");
  p.prologue = 1;
  p.A_log = A_log;
  p.dt_bias = dt_bias;
  return fwd_bf16_pooled(p, reinterpret_cast<cudaStream_t>(stream));
}

gdn_status gdn_recurrent_step_prologue(const void* q, const void* k, const void* v,
                                       const float* a, const float* b, const float* A_log,
                                       const float* dt_bias, float* h, void* o, int N, int Hqk,
                                       int Hv, int dk, int dv, float scale, gdn_stream_t stream) {
  gdn::StepParams p;
  gdn_status s = check_step(q, k, v, a, b, h, o, N, Hqk, Hv, dk, dv, scale, &p);
  if (s != GDN_OK) return s;
  if (!aligned(A_log, 4) || !aligned(dt_bias, 4))
    return fail(GDN_ERR_INVALID_ARG, "A_log and dt_bias must be 4-byte aligned");
  p.prologue = 1;
  p.A_log = A_log;
  p.dt_bias = dt_bias;
  return run_step(p, false, reinterpret_cast<cudaStream_t>(stream));
}

// ---- the same kernels without the erase term: Mamba-2 SSD ---------------------
gdn_status ssd_chunk_fwd(const void* q, const void* k, const void* v, const float* g,
                         const float* beta, const float* h0, void* o, float* hT, int B, int T,
                         int Hqk, int Hv, int dk, int dv, int chunk, float scale,
                         const int32_t* cu_seqlens, gdn_stream_t stream) {
  gdn::FwdParams p;
  gdn_status s = check_fwd(q, k, v, g, beta, h0, o, hT, B, T, Hqk, Hv, dk, dv, chunk, scale,
                           cu_seqlens, 2, &p);
  if (s != GDN_OK) return s;
  p.delta_rule = 0;
  return fwd_bf16_pooled(p, reinterpret_cast<cudaStream_t>(stream));
}

gdn_status ssd_chunk_fwd_ex(const void* q, const void* k, const void* v, const float* g,
                            const float* beta, const float* h0, void* o, float* hT, int B, int T,
                            int Hqk, int Hv, int dk, int dv, int chunk, float scale,
                            const int32_t* cu_seqlens, unsigned flags, void* workspace,
                            size_t workspace_bytes, gdn_stream_t stream) {
  gdn::FwdParams p;
  gdn_status s = check_fwd(q, k, v, g, beta, h0, o, hT, B, T, Hqk, Hv, dk, dv, chunk, scale,
                           cu_seqlens, 2, &p);
  if (s != GDN_OK) return s;
  s = apply_flags(flags, true, &p);
  if (s != GDN_OK) return s;
  p.delta_rule = 0;
  return run_fwd_bf16(p, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream),
                      (flags & GDN_FLAG_CHECK_INPUTS) != 0);
}

gdn_status ssd_chunk_fwd_f32(const float* q, const float* k, const float* v, const float* g,
                             const float* beta, const float* h0, float* o, float* hT, int B,
                             int T, int Hqk, int Hv, int dk, int dv, int chunk, float scale,
                             const int32_t* cu_seqlens, gdn_stream_t stream) {
  gdn::FwdParams p;
  gdn_status s = check_fwd(q, k, v, g, beta, h0, o, hT, B, T, Hqk, Hv, dk, dv, chunk, scale,
                           cu_seqlens, 4, &p);
  if (s != GDN_OK) return s;
  p.delta_rule = 0;
  return run_fwd_f32(p, reinterpret_cast<cudaStream_t>(stream));
}

gdn_status ssd_recurrent_step(const void* q, const void* k, const void* v, const float* g,
                              const float* beta, float* h, void* o, int N, int Hqk, int Hv,
                              int dk, int dv, float scale, gdn_stream_t stream) {
  gdn::StepParams p;
  gdn_status s = check_step(q, k, v, g, beta, h, o, N, Hqk, Hv, dk, dv, scale, &p);
  if (s != GDN_OK) return s;
  p.delta_rule = 0;
  return run_step(p, false, reinterpret_cast<cudaStream_t>(stream));
}

gdn_status ssd_recurrent_step_f32(const float* q, const float* k, const float* v,
                                  const float* g, const float* beta, float* h, float* o, int N,
                                  int Hqk, int Hv, int dk, int dv, float scale,
                                  gdn_stream_t stream) {
  gdn::StepParams p;
  gdn_status s = check_step(q, k, v, g, beta, h, o, N, Hqk, Hv, dk, dv, scale, &p);
  if (s != GDN_OK) return s;
  p.delta_rule = 0;
  return run_step(p, true, reinterpret_cast<cudaStream_t>(stream));
}

// ---- Kimi Delta Attention: the delta rule with a per-channel gate ------------------
gdn_status kda_chunk_fwd_ex(const void* q, const void* k, const void* v, const float* g,
                            const float* beta, const float* h0, void* o, float* hT, int B, int T,
                            int Hqk, int Hv, int dk, int dv, int chunk, float scale,
                            const int32_t* cu_seqlens, unsigned flags, void* workspace,
                            size_t workspace_bytes, gdn_stream_t stream) {
  gdn::FwdParams p;
  gdn_status s = check_kda(q, k, v, g, beta, h0, o, hT, B, T, Hqk, Hv, dk, dv, chunk, scale,
                           cu_seqlens, &p);
  if (s != GDN_OK) return s;
  s = apply_flags(flags, false, &p);
  if (s != GDN_OK) return s;
  return run_fwd_bf16(p, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream),
                      (flags & GDN_FLAG_CHECK_INPUTS) != 0);
}

gdn_status kda_chunk_fwd(const void* q, const void* k, const void* v, const float* g,
                         const float* beta, const float* h0, void* o, float* hT, int B, int T,
                         int Hqk, int Hv, int dk, int dv, int chunk, float scale,
                         const int32_t* cu_seqlens, gdn_stream_t stream) {
  gdn::FwdParams p;
  gdn_status s = check_kda(q, k, v, g, beta, h0, o, hT, B, T, Hqk, Hv, dk, dv, chunk, scale,
                           cu_seqlens, &p);
  if (s != GDN_OK) return s;
  return fwd_bf16_pooled(p, reinterpret_cast<cudaStream_t>(stream));
}

size_t kda_chunk_fwd_workspace_size(int B, int T, int Hqk, int Hv, int dk, int dv, int chunk,
                                    int has_cu_seqlens) {
  gdn::FwdParams p;
  static const int32_t fake_cu = 0;
  const void* A = reinterpret_cast<const void*>(static_cast<uintptr_t>(256));
  if (check_kda(A, A, A, static_cast<const float*>(A), static_cast<const float*>(A), nullptr,
                const_cast<void*>(A), nullptr, B, T, Hqk, Hv, dk, dv, chunk, 1.0f,
                has_cu_seqlens ? &fake_cu : nullptr, &p) != GDN_OK)
    return 0;
  return gdn::ws_bytes_any(p);
}

gdn_status kda_recurrent_step(const void* q, const void* k, const void* v, const float* g,
                              const float* beta, float* h, void* o, int N, int Hqk, int Hv,
                              int dk, int dv, float scale, gdn_stream_t stream) {
  gdn::StepParams p;
  gdn_status s = check_step(q, k, v, g, beta, h, o, N, Hqk, Hv, dk, dv, scale, &p);
  if (s != GDN_OK) return s;
  p.kda = 1;
  return run_step(p, false, reinterpret_cast<cudaStream_t>(stream));
}

gdn_status gdn_selftest_expired_wait(long long limit_cycles, gdn_stream_t stream) {
  if (limit_cycles < 0 || limit_cycles > (1ll << 31))
    return fail(GDN_ERR_INVALID_ARG, "limit_cycles=%lld must be in [0, 2^31]", limit_cycles);
  unsigned* err = nullptr;
  cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&err), gdn::g_device_error);
  if (e != cudaSuccess) return cuda_fail(e, "locating the device error word");
  gdn::selftest_expired_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      err, limit_cycles);
  e = cudaGetLastError();
  return e == cudaSuccess ? GDN_OK : cuda_fail(e, "launching the expired-wait self-test");
}

gdn_status gdn_device_status(gdn_stream_t stream) {
  unsigned word = 0u;
  cudaError_t e = gdn::read_and_clear_device_error(&word, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  if (word == gdn::kErrWaitTimeout)
    return fail(GDN_ERR_TIMEOUT, "a bounded device-side wait gave up");
  if (word == gdn::kErrGateRange)
    return fail(GDN_ERR_INVALID_ARG,
                "a KDA log-decay was below -10 or not a number: that call's result is not exact");
  if (word == gdn::kErrOperandRange)
    return fail(GDN_ERR_INVALID_ARG,
                "an on-chip fp16 operand (V_new or the state) left fp16's range (|x| > 65504 or "
                "not a number): that call's result is not exact");
  if (word == gdn::kErrInput)
    return fail(GDN_ERR_INVALID_ARG,
                "input check: a gate outside its domain (g > 0, beta outside [0, 1], or not a "
                "number) or cu_seqlens not ordered from 0 to T");
  if (word != 0u) return fail(GDN_ERR_TIMEOUT, "device error word 0x%x", word);
  return GDN_OK;
}

}  // extern "C"

// ---- forward without any allocation ------------------------------------------
// A fixed workspace compiled into the library: the device keeps these bytes
// from the moment the library's device code is first used until the process
// exits, on every GPU it runs on.  Host code must not use the array's name as a
// device address; every call looks the address up for the current device
// (cudaGetSymbolAddress allocates nothing), so nothing stale survives a device
// reset.
namespace {
constexpr size_t kNoAllocWorkspaceBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_noalloc_workspace[kNoAllocWorkspaceBytes];
}  // namespace

extern "C" {

gdn_status gdn_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const float* g,
                                 const float* beta, const float* h0, void* o, float* hT, int B,
                                 int T, int Hqk, int Hv, int dk, int dv, int chunk, float scale,
                                 const int32_t* cu_seqlens, gdn_stream_t stream) {
  gdn::FwdParams p;
  gdn_status s = check_fwd(q, k, v, g, beta, h0, o, hT, B, T, Hqk, Hv, dk, dv, chunk, scale,
                           cu_seqlens, 2, &p);
  if (s != GDN_OK) return s;
  const size_t need = gdn::ws_bytes_any(p);
  if (need > kNoAllocWorkspaceBytes)
    return fail(GDN_ERR_INVALID_ARG,
                "these sizes need %zu bytes of workspace; the built-in workspace holds %zu "
                "(use gdn_chunk_fwd_ex with a caller buffer)",
                need, kNoAllocWorkspaceBytes);
  void* ws = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&ws, g_noalloc_workspace);
  if (e != cudaSuccess) return cuda_fail(e, "locating the built-in workspace");
  return run_fwd_bf16(p, ws, kNoAllocWorkspaceBytes, reinterpret_cast<cudaStream_t>(stream));
}

const char* gdn_status_string(gdn_status s) {
  switch (s) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
    case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT";
  }
  return "GDN_ERR_UNKNOWN";
}

const char* gdn_last_error(void) { return t_last_error; }

int gdn_abi_version(void) { return 2; }

}  // extern "C"
