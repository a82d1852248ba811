// gdn_step.cu - one decode token: the gated delta rule applied once per
// (sequence, v head), continuing from the state the prefill left behind
// ("Empowering Hybrid Attention Models on NPUs", §7.3: decoding runs the
// token-by-token recurrence; "Exp 2026-07-13 — Linear-Attention Scans on the
// NPU", §4: the per-token recurrence needs no (I + A)^-1).
//
// Per token, with h = S^T of shape [dk, dv]:
//   h <- exp(g) h;  u = beta (v - h^T k);  h <- h + k u^T;  o = h^T (scale q)
// and, without the erase term (the Mamba-2 SSD recurrence of "Exp 2026-07-13 —
// Linear-Attention Scans on the NPU", §1 and §3), u = beta v.  For Kimi Delta
// Attention the decay is per key channel: h <- diag(exp g) h with g [dk].
// The state is read once and written once, so the step is bound by HBM
// bandwidth: each CTA streams a [dk, 32] column tile of h with 128-byte
// coalesced rows, keeps it in registers between the two column reductions.
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kCols = 32;    // dv columns per CTA (one per lane)
constexpr int kWarps = 4;    // warps split the dk rows

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void store(float* p, float x) { *p = x; }
__device__ __forceinline__ void store(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

template <typename TIn, int DK>
__global__ void __launch_bounds__(kWarps * 32) gdn_step_kernel(const StepParams p) {
  __shared__ float sk[DK], sq[DK], sa[DK];  // sa: KDA's per-channel decay
  __shared__ float red1[kWarps][kCols], red2[kWarps][kCols];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ntile = p.dv / kCols;
  const int tile = blockIdx.x % ntile;
  const int hv = (blockIdx.x / ntile) % p.Hv;
  const int n = blockIdx.x / (ntile * p.Hv);
  const int hq = qk_head(hv, p.Hqk, p.Hv, p.head_map);
  const TIn* q = static_cast<const TIn*>(p.q) + ((long long)n * p.Hqk + hq) * DK;
  const TIn* k = static_cast<const TIn*>(p.k) + ((long long)n * p.Hqk + hq) * DK;
  const long long nh = (long long)n * p.Hv + hv;
  const int col = tile * kCols + lane;
  // the state tile is requested first: its loads are in flight while k, q and the
  // gates arrive (rows warp + 4 i of column col)
  constexpr int R = DK / kWarps;  // rows per thread
  float* h = p.h + nh * DK * p.dv + col;
  float hr[R];
#pragma unroll
  for (int i = 0; i < R; ++i) hr[i] = h[(long long)(warp + kWarps * i) * p.dv];
  for (int i = tid; i < DK; i += kWarps * 32) {
    sk[i] = to_f(k[i]);
    sq[i] = to_f(q[i]);
  }
  float rk = 1.f, rq = 1.f;
  if (p.prologue) {  // fused prologue: unit k and q rows (divided by sqrt(sum x^2 + eps))
    __shared__ float s_inv[2];
    __syncthreads();
    if (warp == 0) {
      float kk = 0.f, qq = 0.f;
      for (int i = lane; i < DK; i += 32) {
        kk = fmaf(sk[i], sk[i], kk);
        qq = fmaf(sq[i], sq[i], qq);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        kk += __shfl_xor_sync(0xffffffffu, kk, off);
        qq += __shfl_xor_sync(0xffffffffu, qq, off);
      }
      if (lane == 0) {
        s_inv[0] = rsqrtf(kk + kNormEps);
        s_inv[1] = rsqrtf(qq + kNormEps);
      }
    }
    __syncthreads();
    rk = s_inv[0];
    rq = s_inv[1];
  }
  for (int i = tid; i < DK; i += kWarps * 32) {  // each thread rescales the entries it loaded
    sk[i] *= rk;
    sq[i] *= rq * p.scale;
  }
  float gate = p.kda ? 0.f : p.g[nh], b = p.beta[nh];
  if (p.prologue) {  // raw gates: g = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b)
    const float x = gate + (p.dt_bias ? p.dt_bias[hv] : 0.f);
    gate = -(p.A_log ? expf(p.A_log[hv]) : 1.f) * (x > 20.f ? x : log1pf(expf(x)));
    b = 1.f / (1.f + expf(-b));
  }
  const float alpha = p.kda ? 0.f : expf(gate);
  if (p.kda)  // Kimi Delta Attention: row r of h decays by exp(g[r])
    for (int i = tid; i < DK; i += kWarps * 32) sa[i] = expf(p.g[nh * DK + i]);
  const float vcol = to_f(static_cast<const TIn*>(p.v)[nh * p.dv + col]);
  __syncthreads();

  float part = 0.f;
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int r = warp + kWarps * i;
    hr[i] *= p.kda ? sa[r] : alpha;
    part += hr[i] * sk[r];
  }
  red1[warp][lane] = part;
  __syncthreads();
  float kh = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) kh += red1[w][lane];
  const float u = b * (p.delta_rule ? vcol - kh : vcol);  // no erase term: u = beta v
  part = 0.f;
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int r = warp + kWarps * i;
    hr[i] += sk[r] * u;
    h[(long long)r * p.dv] = hr[i];
    part += hr[i] * sq[r];
  }
  red2[warp][lane] = part;
  __syncthreads();
  if (warp == 0) {
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) o += red2[w][lane];
    store(static_cast<TIn*>(p.o) + nh * p.dv + col, o);
  }
}

template <typename TIn>
cudaError_t launch_t(const StepParams& p, cudaStream_t stream) {
  const long long grid = (long long)p.N * p.Hv * (p.dv / kCols);
  if (p.dk == 128)
    gdn_step_kernel<TIn, 128><<<(unsigned)grid, kWarps * 32, 0, stream>>>(p);
  else
    gdn_step_kernel<TIn, 64><<<(unsigned)grid, kWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_step_bf16(const StepParams& p, cudaStream_t stream) {
  return launch_t<__nv_bfloat16>(p, stream);
}
cudaError_t launch_step_f32(const StepParams& p, cudaStream_t stream) {
  return launch_t<float>(p, stream);
}

}  // namespace gdn
