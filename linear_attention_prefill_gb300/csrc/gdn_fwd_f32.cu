// gdn_fwd_f32.cu - chunked-prefill forward with fp32 q/k/v/o (fp32 throughout).
//
// Same chain mapping as the bf16 kernel: one CTA per (sequence, v head, dv tile),
// chunks walked in order, the fp32 state tile resident on chip.  Every product
// is an fp32 FMA on the CUDA cores (the fp32 path keeps fp32 operands).  The
// state read uses the rewrite of "Empowering Hybrid Attention Models on NPUs",
// §5 (Intra-Chunk, Figure 11): V_new = Tm (diag(beta) V - diag(beta gamma) K h),
// i.e. A^-1 (V - K S) with the scalings folded in, which drops the W operand
// and its shared-memory tile.  Operator list and order as in §2.1 / Figure 1(b)
// and the chunk-first state update of §5 (Figure 10(b)).
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kC = 64;
constexpr int kThreads = 256;
constexpr int kDVT = 64;  // dv columns per CTA

template <int DK>
struct SmemF32 {
  static constexpr int LDK = DK + 1;    // odd strides: conflict-free column walks
  static constexpr int LDV = kDVT + 1;
  static constexpr int LDA = kC + 1;
  float K[kC * LDK];
  float Q[kC * LDK];
  float V[kC * LDV];
  float H[DK * LDV];     // state tile h[:, tile]
  float A[kC * LDA];     // strictly lower A, later reused for R
  float Tm[kC * LDA];
  float P[kC * LDA];
  float Vn[kC * LDV];
  float X[3 * 256];
  float g[kC], beta[kC], G[kC], gam[kC], e[kC];
};

template <int DK>
__global__ void __launch_bounds__(kThreads, 1) gdn_fwd_f32_kernel(const FwdParams p) {
  using S = SmemF32<DK>;
  constexpr int LDK = S::LDK, LDV = S::LDV, LDA = S::LDA;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  S& s = *reinterpret_cast<S*>(smem_raw);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ti = tid >> 4, tj = tid & 15;  // 16 x 16 thread grid for register tiles
  const int n_dvt = p.dv / kDVT;
  const int dvt = blockIdx.x % n_dvt;
  const int hv = (blockIdx.x / n_dvt) % p.Hv;
  const int n = blockIdx.x / (n_dvt * p.Hv);
  const int hq = qk_head(hv, p.Hqk, p.Hv, p.head_map);

  long long t_begin, t_end;
  if (p.cu_seqlens) {
    t_begin = p.cu_seqlens[n];
    t_end = p.cu_seqlens[n + 1];
  } else {
    t_begin = (long long)n * p.T;
    t_end = t_begin + p.T;
  }
  const long long len = t_end - t_begin;
  const int n_chunks = (int)((len + kC - 1) / kC);
  const long long qk_tok = (long long)p.Hqk * DK, v_tok = (long long)p.Hv * p.dv;
  const float* qg = static_cast<const float*>(p.q) + (long long)hq * DK;
  const float* kg = static_cast<const float*>(p.k) + (long long)hq * DK;
  const float* vg = static_cast<const float*>(p.v) + (long long)hv * p.dv + dvt * kDVT;
  float* og = static_cast<float*>(p.o) + (long long)hv * p.dv + dvt * kDVT;
  const long long hoff = ((long long)(n * p.Hv + hv) * DK) * p.dv + dvt * kDVT;

  for (int i = tid; i < DK * kDVT; i += kThreads) {
    const int r = i / kDVT, cc = i % kDVT;
    s.H[r * LDV + cc] = p.h0 ? p.h0[hoff + (long long)r * p.dv + cc] : 0.f;
  }

  for (int c = 0; c < n_chunks; ++c) {
    const long long t0 = t_begin + (long long)c * kC;
    const int L = (int)min((long long)kC, len - (long long)c * kC);
    __syncthreads();  // previous chunk fully consumed
    for (int i = tid; i < kC * DK; i += kThreads) {
      const int r = i / DK, d = i % DK;
      const bool ok = r < L;
      s.K[r * LDK + d] = ok ? kg[(t0 + r) * qk_tok + d] : 0.f;
      s.Q[r * LDK + d] = ok ? qg[(t0 + r) * qk_tok + d] : 0.f;
    }
    for (int i = tid; i < kC * kDVT; i += kThreads) {
      const int r = i / kDVT, d = i % kDVT;
      s.V[r * LDV + d] = r < L ? vg[(t0 + r) * v_tok + d] : 0.f;
    }
    if (tid < kC) {
      const bool ok = tid < L;
      s.g[tid] = ok ? p.g[(t0 + tid) * p.Hv + hv] : 0.f;
      s.beta[tid] = ok ? p.beta[(t0 + tid) * p.Hv + hv] : 0.f;
    }
    __syncthreads();

    // #1 Gate
    if (warp == 0) {
      const float g0 = s.g[2 * lane], g1 = s.g[2 * lane + 1];
      float incl = g0 + g1;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      const float G1 = incl, G0 = incl - g1;
      const float Glast = __shfl_sync(0xffffffffu, G1, 31);
      s.G[2 * lane] = G0;
      s.G[2 * lane + 1] = G1;
      s.gam[2 * lane] = expf(G0);
      s.gam[2 * lane + 1] = expf(G1);
      s.e[2 * lane] = expf(Glast - G0);
      s.e[2 * lane + 1] = expf(Glast - G1);
    }
    __syncthreads();

    // #2 KKT and QK^T: thread (ti, tj) owns rows ti + 16a, columns tj + 16b
    {
      float sk[4][4] = {}, sq[4][4] = {};
      for (int d = 0; d < DK; ++d) {
        float kr[4], qr[4], kc[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          kr[a] = s.K[(ti + 16 * a) * LDK + d];
          qr[a] = s.Q[(ti + 16 * a) * LDK + d];
          kc[a] = s.K[(tj + 16 * a) * LDK + d];
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            sk[a][b] += kr[a] * kc[b];
            sq[a][b] += qr[a] * kc[b];
          }
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int r = ti + 16 * a, cc = tj + 16 * b;
          const bool low = r >= cc && r < L;
          const float m = low ? expf(s.G[r] - s.G[cc]) : 0.f;
          s.A[r * LDA + cc] = (low && r > cc && p.delta_rule) ? s.beta[r] * m * sk[a][b] : 0.f;
          s.P[r * LDA + cc] = low ? p.scale * m * sq[a][b] : 0.f;
        }
    }
    __syncthreads();

    // #3 Solve
    solve_unit_lower_64_f32<kThreads>(s.A, LDA, s.Tm, LDA, s.X);

    // #5 read (rewritten): R = diag(beta) V - diag(beta gamma) K h   -> s.A
    //   and the inter-chunk part of #6: O1 = diag(scale gamma) Q h     -> registers
    float o1[4][4] = {};
    {
      float kh[4][4] = {};
      for (int d = 0; d < DK; ++d) {
        float kr[4], qr[4], hc[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          kr[a] = s.K[(ti + 16 * a) * LDK + d];
          qr[a] = s.Q[(ti + 16 * a) * LDK + d];
          hc[a] = s.H[d * LDV + tj + 16 * a];
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            kh[a][b] += kr[a] * hc[b];
            o1[a][b] += qr[a] * hc[b];
          }
      }
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int r = ti + 16 * a;
        const float br = s.beta[r], sg = p.scale * s.gam[r];
        const float bgr = p.delta_rule ? s.beta[r] * s.gam[r] : 0.f;  // no K h term without the erase
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int cc = tj + 16 * b;
          s.A[r * LDA + cc] = br * s.V[r * LDV + cc] - bgr * kh[a][b];
          o1[a][b] *= sg;
        }
      }
    }
    __syncthreads();
    // V_new = Tm R
    {
      float vn[4][4] = {};
      for (int j = 0; j < kC; ++j) {
        float tr[4], rc[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          tr[a] = s.Tm[(ti + 16 * a) * LDA + j];
          rc[a] = s.A[j * LDA + tj + 16 * a];
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) vn[a][b] += tr[a] * rc[b];
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) s.Vn[(ti + 16 * a) * LDV + tj + 16 * b] = vn[a][b];
    }
    __syncthreads();
    // #6 O = O1 + P V_new
    {
      for (int j = 0; j < kC; ++j) {
        float pr[4], vc[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          pr[a] = s.P[(ti + 16 * a) * LDA + j];
          vc[a] = s.Vn[j * LDV + tj + 16 * a];
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) o1[a][b] += pr[a] * vc[b];
      }
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int r = ti + 16 * a;
        if (r < L)
#pragma unroll
          for (int b = 0; b < 4; ++b) og[(t0 + r) * v_tok + tj + 16 * b] = o1[a][b];
      }
    }
    // #5 update: h = gamma_last h + K^T diag(e) V_new; thread owns rows ti + 16a
    {
      constexpr int RA = DK / 16;
      float hn[RA][4] = {};
      for (int j = 0; j < kC; ++j) {
        const float ej = s.e[j];
        float kc[RA], vc[4];
#pragma unroll
        for (int a = 0; a < RA; ++a) kc[a] = s.K[j * LDK + ti + 16 * a];
#pragma unroll
        for (int b = 0; b < 4; ++b) vc[b] = ej * s.Vn[j * LDV + tj + 16 * b];
#pragma unroll
        for (int a = 0; a < RA; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) hn[a][b] += kc[a] * vc[b];
      }
      const float gl = s.gam[kC - 1];
      __syncthreads();  // all reads of s.H for this chunk are done
#pragma unroll
      for (int a = 0; a < RA; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          float& hr = s.H[(ti + 16 * a) * LDV + tj + 16 * b];
          hr = gl * hr + hn[a][b];
        }
    }
  }
  __syncthreads();
  if (p.hT) {
    for (int i = tid; i < DK * kDVT; i += kThreads) {
      const int r = i / kDVT, cc = i % kDVT;
      p.hT[hoff + (long long)r * p.dv + cc] = s.H[r * LDV + cc];
    }
  }
}

template <int DK>
cudaError_t launch_t(const FwdParams& p, cudaStream_t stream) {
  const size_t smem = sizeof(SmemF32<DK>);
  cudaError_t err = cudaFuncSetAttribute(gdn_fwd_f32_kernel<DK>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const long long grid = (long long)p.N * p.Hv * (p.dv / kDVT);
  gdn_fwd_f32_kernel<DK><<<(unsigned)grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_f32(const FwdParams& p, cudaStream_t stream) {
  if (p.dk == 128) return launch_t<128>(p, stream);
  return launch_t<64>(p, stream);
}

}  // namespace gdn
