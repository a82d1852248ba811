// gdn_prep.cu - the chunk-parallel Map phase of the chunkwise forward.
//
// "Empowering Hybrid Attention Models on NPUs", §2.1, Figure 1(b): operators
// #1-#4 (Gate, KKT, Solve, W/U) depend only on one chunk's q, k, v, g, beta,
// so every (chunk, v head) is an independent task here:
//   #1 Gate   G = cumsum(g), gamma = exp(G), e_j = exp(G_last - G_j)
//   #2 KKT    A = tril_strict(beta_i exp(G_i - G_j) k_i.k_j)
//      QK^T   P = tril(scale exp(G_i - G_j) q_i.k_j)
//   #3 Solve  Tm = (I + A)^-1   (diagonal blocks by substitution, merges on tensor cores)
//   #4 W/U    W = Tm diag(beta gamma) K,  U = Tm diag(beta) V
// plus the two scaled copies the later launches consume: Kt = diag(e) K (the
// state update's left factor) and Qt = diag(scale gamma) Q (the output's
// inter-chunk term).  The serial Reduce (#5) runs in gdn_chain.cu, the final
// Map (#6) in gdn_out.cu; both read this kernel's workspace records.
//
// Tensor-core products accumulate in fp32.  The grams and W = (Tm diag(beta
// gamma)) K take the bf16 inputs as they are (W's left factor rounded to bf16:
// its share of the error is below 1e-3 of RMS); U = Tm diag(beta) V takes fp16
// operands (v rewritten in place, exact in fp16's normal range), since U's
// rounding feeds V_new and the output directly.
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kC = 64;
constexpr int kThreads = 256;

template <int DK, int DV>
struct PrepSmem {
  static constexpr int LDK = DK + 8;   // 16-bit row strides (conflict-free ldmatrix)
  static constexpr int LDV = DV + 8;
  static constexpr int LDC = kC + 8;
  static constexpr int LDA = kC + 4;   // fp32 row stride of A and Tm
  __half K[kC * LDK];                  // bf16 bits (grams and W take bf16 operands)
  union {                              // Q (bf16 bits) until the grams are done, then A, then U staging
    __half Q[kC * LDK];
    float A[kC * LDA];
    __half Ust[kC * LDV];
  };
  __half V[kC * LDV];
  union {                              // Tm until Tw/Tu are built, then W staging
    float Tm[kC * LDA];
    __half Wst[kC * LDK];
  };
  __half Ah[kC * LDC];
  __half Th[kC * LDC];
  union {                              // P staging for its bulk store, then Tw (bf16 bits)
    __half Pst[kC * kC];
    __half Tw[kC * LDC];
  };
  __half Tu[kC * LDC];
  float g[kC], beta[kC], G[kC], gam[kC], e[kC];
};

// 8 bf16 values at p (16-byte aligned) times `scale`, rounded once to fp16.
__device__ __forceinline__ uint4 scale_bf16x8_to_f16(const __half* p, float scale) {
  uint4 raw = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
  uint4 out;
  __half2* o = reinterpret_cast<__half2*>(&out);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    o[i] = __floats2half2_rn(f.x * scale, f.y * scale);
  }
  return out;
}

template <int DK, int DV>
__global__ void __launch_bounds__(kThreads, 2) gdn_prep_kernel(const FwdParams p, WsLayout ws) {
  using S = PrepSmem<DK, DV>;
  constexpr int LDK = S::LDK, LDV = S::LDV, LDC = S::LDC, LDA = S::LDA;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  S& s = *reinterpret_cast<S*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;

  GDN_PHASE_INIT;
  // task -> (chunk slot, v head) -> (sequence, chunk within it)
  const int hv = blockIdx.x % p.Hv;
  const long long slot = blockIdx.x / p.Hv;
  int n, c;
  if (!locate_chunk(p, ws, slot, &n, &c)) return;
  const long long t_seq = p.cu_seqlens ? (long long)p.cu_seqlens[n] : (long long)n * p.T;
  const long long len =
      p.cu_seqlens ? (long long)p.cu_seqlens[n + 1] - t_seq : (long long)p.T;
  const long long t0 = t_seq + (long long)c * kC;
  const int L = (int)min((long long)kC, len - (long long)c * kC);
  const int hq = hv / (p.Hv / p.Hqk);

  // ---- staging (cp.async, zero-filled past the sequence end) ---------------
  {
    const long long qk_tok = (long long)p.Hqk * DK, v_tok = (long long)p.Hv * DV;
    const __nv_bfloat16* kg = static_cast<const __nv_bfloat16*>(p.k) + (long long)hq * DK;
    const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(p.q) + (long long)hq * DK;
    const __nv_bfloat16* vg = static_cast<const __nv_bfloat16*>(p.v) + (long long)hv * DV;
    for (int i = tid; i < kC * (DK / 8); i += kThreads) {
      const int r = i / (DK / 8), sg = i % (DK / 8);
      const bool ok = r < L;
      const long long tok = t0 + (ok ? r : 0);
      cp_async16(&s.K[r * LDK + sg * 8], kg + tok * qk_tok + sg * 8, ok);
      cp_async16(&s.Q[r * LDK + sg * 8], qg + tok * qk_tok + sg * 8, ok);
    }
    for (int i = tid; i < kC * (DV / 8); i += kThreads) {
      const int r = i / (DV / 8), sg = i % (DV / 8);
      const bool ok = r < L;
      const long long tok = t0 + (ok ? r : 0);
      cp_async16(&s.V[r * LDV + sg * 8], vg + tok * v_tok + sg * 8, ok);
    }
    if (tid < kC) {
      const bool ok = tid < L;
      const long long tok = t0 + (ok ? tid : 0);
      cp_async4(&s.g[tid], p.g + tok * p.Hv + hv, ok);
      cp_async4(&s.beta[tid], p.beta + tok * p.Hv + hv, ok);
    }
    cp_async_commit();
    cp_async_wait<0>();
  }
  __syncthreads();
  GDN_PHASE(0);  // staging
  for (int i = tid; i < kC * (DV / 8); i += kThreads) {  // V -> fp16 (U takes fp16 operands)
    const int r = i / (DV / 8), sg = i % (DV / 8);
    bf16x8_to_f16x8(&s.V[r * LDV + sg * 8]);
  }
  // ---- #1 Gate (padded rows carry g = 0, so G[63] = G_last) ------------------
  if (warp == 0) {
    const float g0 = s.g[2 * lane], g1 = s.g[2 * lane + 1];
    float incl = g0 + g1;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    const float Glast = __shfl_sync(0xffffffffu, incl, 31);
    s.G[2 * lane] = incl - g1;
    s.G[2 * lane + 1] = incl;
    s.gam[2 * lane] = expf(incl - g1);
    s.gam[2 * lane + 1] = expf(incl);
    s.e[2 * lane] = expf(Glast - (incl - g1));
    s.e[2 * lane + 1] = expf(Glast - incl);
    if (lane == 31) *ws.gl(slot, hv, p.Hv) = expf(Glast);
  }
  __syncthreads();
  GDN_PHASE(1);  // convert + gate

  // ---- #2 KKT and QK^T grams (lower triangle) -------------------------------
  __half* Pout = ws.P(slot, hv, p.Hv);
  {
    const int rb = warp >> 1, ch = warp & 1;
    float aK[4][4], aQ[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int x = 0; x < 4; ++x) aK[j][x] = aQ[j][x] = 0.f;
    const bool need0 = 2 * ch <= rb, need1 = 2 * ch + 1 <= rb;
    if (need0) {
#pragma unroll 2
      for (int kk = 0; kk < DK; kk += 16) {
        uint32_t ak[4], aq[4], b[4];
        load_a(ak, s.K, LDK, 16 * rb, kk, lane);
        load_a(aq, s.Q, LDK, 16 * rb, kk, lane);
        load_b_nk(b, s.K, LDK, 32 * ch, kk, lane);
        mma_bf16(aK[0], ak, b[0], b[1]);
        mma_bf16(aK[1], ak, b[2], b[3]);
        mma_bf16(aQ[0], aq, b[0], b[1]);
        mma_bf16(aQ[1], aq, b[2], b[3]);
        if (need1) {
          load_b_nk(b, s.K, LDK, 32 * ch + 16, kk, lane);
          mma_bf16(aK[2], ak, b[0], b[1]);
          mma_bf16(aK[3], ak, b[2], b[3]);
          mma_bf16(aQ[2], aq, b[0], b[1]);
          mma_bf16(aQ[3], aq, b[2], b[3]);
        }
      }
    }
    GDN_PHASE(2);  // grams
    // the scaled copies Qt = diag(scale gamma) Q and Kt = diag(e) K
    __half* Qt = ws.Qt(slot, hv, p.Hv);
    __half* Kt = ws.Kt(slot, hv, p.Hv);
    for (int i = tid; i < kC * (DK / 8); i += kThreads) {
      const int r = i / (DK / 8), sg = i % (DK / 8);
      *reinterpret_cast<uint4*>(Qt + swz<DK>(r, sg * 8)) =
          scale_bf16x8_to_f16(&s.Q[r * LDK + sg * 8], p.scale * s.gam[r]);
      *reinterpret_cast<uint4*>(Kt + swz<DK>(r, sg * 8)) =
          scale_bf16x8_to_f16(&s.K[r * LDK + sg * 8], s.e[r]);
    }
    __syncthreads();  // Q is dead: its storage becomes A
    GDN_PHASE(3);  // Qt, Kt
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
      for (int x = 0; x < 4; x += 2) {
        const int r = 16 * rb + gq + ((x >> 1) << 3);
        const int c0 = 32 * ch + 8 * j + 2 * tq;
        float pv[2], av[2];
#pragma unroll
        for (int y = 0; y < 2; ++y) {
          const int cc = c0 + y;
          const bool low = r >= cc && r < L;
          const float m = low ? expf(s.G[r] - s.G[cc]) : 0.f;
          av[y] = (low && r > cc) ? s.beta[r] * m * aK[j][x + y] : 0.f;
          pv[y] = low ? p.scale * m * aQ[j][x + y] : 0.f;
          s.A[r * LDA + cc] = av[y];
        }
        *reinterpret_cast<uint32_t*>(&s.Ah[r * LDC + c0]) = pack_f16(av[0], av[1]);
        *reinterpret_cast<uint32_t*>(&s.Pst[swz<kC>(r, c0)]) = pack_f16(pv[0], pv[1]);
      }
    }
    fence_proxy_async();  // P staging is read by a bulk store
  }
  __syncthreads();

  GDN_PHASE(4);  // masks
  // ---- #3 Solve and the scaled operands --------------------------------------
  if (tid == 0) {  // P leaves in one bulk store while the solve runs
    fence_proxy_async();
    bulk_s2g(Pout, s.Pst, kC * kC * 2);
    bulk_commit();
  }
  solve_unit_lower_64(s.A, LDA, s.Ah, s.Tm, LDA, s.Th, LDC);
  if (tid == 0) bulk_wait_read<0>();
  __syncthreads();  // P staging is free: Tw takes its place
  GDN_PHASE(5);  // solve
  for (int e = tid; e < kC * (kC / 8); e += kThreads) {  // 8 columns per item, 16-byte stores
    const int r = e >> 3, c0 = (e & 7) * 8;
    uint4 w, u;
    __nv_bfloat162* wp = reinterpret_cast<__nv_bfloat162*>(&w);
    __half2* up = reinterpret_cast<__half2*>(&u);
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int cc = c0 + 2 * x;
      const float t0 = s.Tm[r * LDA + cc], t1 = s.Tm[r * LDA + cc + 1];
      const float b0 = s.beta[cc], b1 = s.beta[cc + 1];
      wp[x] = __floats2bfloat162_rn(t0 * b0 * s.gam[cc], t1 * b1 * s.gam[cc + 1]);
      up[x] = __floats2half2_rn(t0 * b0, t1 * b1);
    }
    *reinterpret_cast<uint4*>(&s.Tw[r * LDC + c0]) = w;
    *reinterpret_cast<uint4*>(&s.Tu[r * LDC + c0]) = u;
  }
  __syncthreads();
  GDN_PHASE(6);  // Tw, Tu

  // ---- #4 W = Tw K, U = Tu V (lower-triangular Tw/Tu: k <= row block) -------
  {
    const int rb = warp & 3, nh = warp >> 2;
    constexpr int WNT = DK / 16, UNT = DV / 16;  // n8 tiles per warp (half the columns)
    float aW[WNT][4], aU[UNT][4];
#pragma unroll
    for (int j = 0; j < WNT; ++j)
#pragma unroll
      for (int x = 0; x < 4; ++x) aW[j][x] = 0.f;
#pragma unroll
    for (int j = 0; j < UNT; ++j)
#pragma unroll
      for (int x = 0; x < 4; ++x) aU[j][x] = 0.f;
    for (int kk = 0; kk <= 16 * rb; kk += 16) {
      uint32_t a[4], b[4];
      load_a(a, s.Tw, LDC, 16 * rb, kk, lane);
#pragma unroll
      for (int j = 0; j < WNT; j += 2) {
        load_b_kn(b, s.K, LDK, nh * (DK / 2) + 8 * j, kk, lane);
        mma_bf16(aW[j], a, b[0], b[1]);
        mma_bf16(aW[j + 1], a, b[2], b[3]);
      }
      load_a(a, s.Tu, LDC, 16 * rb, kk, lane);
#pragma unroll
      for (int j = 0; j < UNT; j += 2) {
        load_b_kn(b, s.V, LDV, nh * (DV / 2) + 8 * j, kk, lane);
        mma_f16(aU[j], a, b[0], b[1]);
        mma_f16(aU[j + 1], a, b[2], b[3]);
      }
    }
    __syncthreads();  // Tm and A/Q storage are dead: stage W and U there
    const int r0 = 16 * rb + gq;
#pragma unroll
    for (int j = 0; j < WNT; ++j) {
      const int col = nh * (DK / 2) + 8 * j + 2 * tq;
      *reinterpret_cast<uint32_t*>(&s.Wst[r0 * LDK + col]) = pack_f16(aW[j][0], aW[j][1]);
      *reinterpret_cast<uint32_t*>(&s.Wst[(r0 + 8) * LDK + col]) = pack_f16(aW[j][2], aW[j][3]);
    }
#pragma unroll
    for (int j = 0; j < UNT; ++j) {
      const int col = nh * (DV / 2) + 8 * j + 2 * tq;
      *reinterpret_cast<uint32_t*>(&s.Ust[r0 * LDV + col]) = pack_f16(aU[j][0], aU[j][1]);
      *reinterpret_cast<uint32_t*>(&s.Ust[(r0 + 8) * LDV + col]) = pack_f16(aU[j][2], aU[j][3]);
    }
  }
  __syncthreads();
  GDN_PHASE(7);  // W/U products
  __half* Wout = ws.W(slot, hv, p.Hv);
  __half* Uout = ws.U(slot, hv, p.Hv);
  for (int i = tid; i < kC * (DK / 8); i += kThreads) {
    const int r = i / (DK / 8), sg = i % (DK / 8);
    *reinterpret_cast<uint4*>(Wout + swz<DK>(r, sg * 8)) =
        *reinterpret_cast<const uint4*>(&s.Wst[r * LDK + sg * 8]);
  }
  const int dvt = ws.dvt;
  for (int i = tid; i < kC * (DV / 8); i += kThreads) {  // U tile-major: [dv/t][64][t]
    const int r = i / (DV / 8), sg = i % (DV / 8);
    const int col = sg * 8, t = col / dvt, w = col % dvt;
    *reinterpret_cast<uint4*>(Uout + (t * kC + r) * dvt + w) =
        *reinterpret_cast<const uint4*>(&s.Ust[r * LDV + col]);
  }
  GDN_PHASE(8);  // W/U stores
}

template <int DK, int DV>
cudaError_t launch_t(const FwdParams& p, const WsLayout& ws, cudaStream_t stream) {
  const size_t smem = sizeof(PrepSmem<DK, DV>);
  cudaError_t e = cudaFuncSetAttribute(gdn_prep_kernel<DK, DV>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const long long grid = ws.n_slots * p.Hv;
  gdn_prep_kernel<DK, DV><<<(unsigned)grid, kThreads, smem, stream>>>(p, ws);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prep(const FwdParams& p, const WsLayout& ws, cudaStream_t stream) {
  if (p.dk == 128) {
    if (p.dv == 128) return launch_t<128, 128>(p, ws, stream);
    return launch_t<128, 64>(p, ws, stream);
  }
  if (p.dv == 128) return launch_t<64, 128>(p, ws, stream);
  return launch_t<64, 64>(p, ws, stream);
}

}  // namespace gdn
