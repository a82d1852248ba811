// gdn_fwd_bf16.cu - fused chunked-prefill forward, bf16 q/k/v/o, fp32 gates and state.
//
// One CTA owns one (sequence, value head, dv tile) chain and walks its chunks in
// order, keeping the fp32 state tile h[:, tile] in registers for the whole
// sequence.  Per chunk it runs the operators of the chunkwise form
// ("Empowering Hybrid Attention Models on NPUs", §2.1, Figure 1(b)) all on chip:
//   #1 Gate     G = cumsum(g), gamma = exp(G), e_j = exp(G_last - G_j)
//   #2 KKT      A = tril_strict(beta_i exp(G_i - G_j) k_i.k_j)
//      QK^T     P = tril(scale exp(G_i - G_j) q_i.k_j)
//   #3 Solve    Tm = (I + A)^-1            (blocked forward substitution, fp32)
//   #4 W/U      W = Tm diag(beta gamma) K,  U = Tm diag(beta) V
//   #5 read     V_new = U - W h
//   #6 O        O = diag(scale gamma) Q h + P V_new
//   #5 update   h = gamma_last h + K^T diag(e) V_new
// in the chunk-first order of §5 (Figure 10(b)): the state is read for the
// output before it is overwritten in place, so only one copy of it exists.
// Head-resident mapping with cross-operator fusion (§4, Figure 7(c)) and the
// column split of the state for parallelism without a reduction (§4,
// Figure 8(b)) decide the grid: one CTA per (sequence, v head, dv tile).
//
// Contractions run on fp16 tensor cores (mma.sync m16n8k16, fp32 accumulate).
// The bf16 q/k/v tiles are rewritten as fp16 once staged (exact in fp16's
// normal range), and every on-chip operand (Tm scaled by beta (gamma), W,
// V_new, e*V_new, the state copy, P) is fp16: its 11-bit significand keeps the
// operand rounding 8x below bf16's at the same tensor-core rate.  The fp32
// state itself never leaves the registers until the end.  Chunk tiles are staged
// into padded shared memory with cp.async, double-buffered one chunk ahead.
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kC = 64;          // chunk length
constexpr int kThreads = 256;   // 8 warps

template <int DK, int DVT>
struct SmemBf16 {
  static constexpr int LDK = DK + 8;   // 16-bit row stride of K, Q, -W (272 B for DK=128)
  static constexpr int LDV = DVT + 8;  // 16-bit row stride of V, V_new, e*V_new, h
  static constexpr int LDC = kC + 8;   // 16-bit row stride of the 64x64 Tw, Tu, P
  static constexpr int LDA = kC + 4;   // fp32 row stride of A and Tm
  __half K[2][kC * LDK];   // staged as bf16, converted in place to fp16
  __half Q[2][kC * LDK];
  __half V[2][kC * LDV];
  float g[2][kC];
  float beta[2][kC];
  float G[kC], gam[kC], e[kC];
  float A[kC * LDA];
  float Tm[kC * LDA];
  float X[3 * 256];
  __half Tw[kC * LDC];
  __half Tu[kC * LDC];
  __half P[kC * LDC];
  __half Wn[kC * LDK];  // -W
  __half H[DK * LDV];   // fp16 copy of the state tile
  __half Vn[kC * LDV];  // V_new
  __half Ve[kC * LDV];  // diag(e) V_new
};

template <int DK, int DVT>
__global__ void __launch_bounds__(kThreads, 1) gdn_fwd_bf16_kernel(const FwdParams p) {
  using S = SmemBf16<DK, DVT>;
  constexpr int LDK = S::LDK, LDV = S::LDV, LDC = S::LDC, LDA = S::LDA;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  S& s = *reinterpret_cast<S*>(smem_raw);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;  // mma fragment row group / thread-in-group
  const int n_dvt = p.dv / DVT;
  const int dvt = blockIdx.x % n_dvt;
  const int hv = (blockIdx.x / n_dvt) % p.Hv;
  const int n = blockIdx.x / (n_dvt * p.Hv);
  const int hq = hv / (p.Hv / p.Hqk);

  long long t_begin, t_end;  // token range in the flattened [rows * T] index
  if (p.cu_seqlens) {
    t_begin = p.cu_seqlens[n];
    t_end = p.cu_seqlens[n + 1];
  } else {
    t_begin = (long long)n * p.T;
    t_end = t_begin + p.T;
  }
  const long long len = t_end - t_begin;
  const int n_chunks = (int)((len + kC - 1) / kC);

  const long long qk_tok = (long long)p.Hqk * DK;  // elements between tokens
  const long long v_tok = (long long)p.Hv * p.dv;
  const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(p.q) + (long long)hq * DK;
  const __nv_bfloat16* kg = static_cast<const __nv_bfloat16*>(p.k) + (long long)hq * DK;
  const __nv_bfloat16* vg =
      static_cast<const __nv_bfloat16*>(p.v) + (long long)hv * p.dv + dvt * DVT;
  __nv_bfloat16* og = static_cast<__nv_bfloat16*>(p.o) + (long long)hv * p.dv + dvt * DVT;
  const float* gg = p.g + hv;
  const float* bg = p.beta + hv;

  auto issue_loads = [&](int c, int buf) {
    const long long t0 = t_begin + (long long)c * kC;
    const int L = (int)min((long long)kC, len - (long long)c * kC);
    constexpr int SEGK = DK / 8;
    for (int i = tid; i < kC * SEGK; i += kThreads) {
      const int r = i / SEGK, sg = i % SEGK;
      const bool valid = r < L;
      const long long tok = t0 + (valid ? r : 0);
      cp_async16(&s.K[buf][r * LDK + sg * 8], kg + tok * qk_tok + sg * 8, valid);
      cp_async16(&s.Q[buf][r * LDK + sg * 8], qg + tok * qk_tok + sg * 8, valid);
    }
    constexpr int SEGV = DVT / 8;
    for (int i = tid; i < kC * SEGV; i += kThreads) {
      const int r = i / SEGV, sg = i % SEGV;
      const bool valid = r < L;
      const long long tok = t0 + (valid ? r : 0);
      cp_async16(&s.V[buf][r * LDV + sg * 8], vg + tok * v_tok + sg * 8, valid);
    }
    if (tid < kC) {
      const bool valid = tid < L;
      const long long tok = t0 + (valid ? tid : 0);
      cp_async4(&s.g[buf][tid], gg + tok * p.Hv, valid);
      cp_async4(&s.beta[buf][tid], bg + tok * p.Hv, valid);
    }
    cp_async_commit();
  };

  // ---- state tile in registers: warp -> (dk m-tile, column part) ----------
  constexpr int MT = DK / 16;              // m16 tiles over dk
  constexpr int WPM = (kThreads / 32) / MT;  // warps sharing one m-tile
  constexpr int HCOLS = DVT / WPM;         // columns per warp
  constexpr int HNT = HCOLS / 8;           // n8 tiles per warp
  static_assert(MT * WPM == kThreads / 32 && HNT % 2 == 0, "state tiling");
  const int hmt = warp / WPM, hcol0 = (warp % WPM) * HCOLS;
  float hacc[HNT][4];
  {
    const float* h0 = p.h0 ? p.h0 + ((long long)(n * p.Hv + hv) * DK) * p.dv + dvt * DVT : nullptr;
#pragma unroll
    for (int j = 0; j < HNT; ++j) {
      const int r0 = 16 * hmt + gq, col = hcol0 + 8 * j + 2 * tq;
      float2 a = make_float2(0.f, 0.f), b = make_float2(0.f, 0.f);
      if (h0) {
        a = *reinterpret_cast<const float2*>(h0 + (long long)r0 * p.dv + col);
        b = *reinterpret_cast<const float2*>(h0 + (long long)(r0 + 8) * p.dv + col);
      }
      hacc[j][0] = a.x; hacc[j][1] = a.y; hacc[j][2] = b.x; hacc[j][3] = b.y;
      *reinterpret_cast<uint32_t*>(&s.H[r0 * LDV + col]) = pack_f16(a.x, a.y);
      *reinterpret_cast<uint32_t*>(&s.H[(r0 + 8) * LDV + col]) = pack_f16(b.x, b.y);
    }
  }

  if (n_chunks > 0) issue_loads(0, 0);
  for (int c = 0; c < n_chunks; ++c) {
    const int buf = c & 1;
    const long long t0 = t_begin + (long long)c * kC;
    const int L = (int)min((long long)kC, len - (long long)c * kC);
    if (c + 1 < n_chunks) {
      issue_loads(c + 1, buf ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    // bf16 -> fp16 in place (16 bytes per thread per step), then every product is fp16
    for (int i = tid; i < kC * (DK / 8); i += kThreads) {
      const int r = i / (DK / 8), sg = i % (DK / 8);
      bf16x8_to_f16x8(&s.K[buf][r * LDK + sg * 8]);
      bf16x8_to_f16x8(&s.Q[buf][r * LDK + sg * 8]);
    }
    for (int i = tid; i < kC * (DVT / 8); i += kThreads) {
      const int r = i / (DVT / 8), sg = i % (DVT / 8);
      bf16x8_to_f16x8(&s.V[buf][r * LDV + sg * 8]);
    }
    __syncthreads();
    const __half* Ks = s.K[buf];
    const __half* Qs = s.Q[buf];

    // ---- #1 Gate (padded rows carry g = 0, so G[kC-1] = G[L-1]) ----------
    if (warp == 0) {
      const float g0 = s.g[buf][2 * lane], g1 = s.g[buf][2 * lane + 1];
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

    // ---- #2 KKT and QK^T grams (lower triangle only) ------------------------
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
          load_a(ak, Ks, LDK, 16 * rb, kk, lane);
          load_a(aq, Qs, LDK, 16 * rb, kk, lane);
          load_b_nk(b, Ks, LDK, 32 * ch, kk, lane);
          mma_f16(aK[0], ak, b[0], b[1]);
          mma_f16(aK[1], ak, b[2], b[3]);
          mma_f16(aQ[0], aq, b[0], b[1]);
          mma_f16(aQ[1], aq, b[2], b[3]);
          if (need1) {
            load_b_nk(b, Ks, LDK, 32 * ch + 16, kk, lane);
            mma_f16(aK[2], ak, b[0], b[1]);
            mma_f16(aK[3], ak, b[2], b[3]);
            mma_f16(aQ[2], aq, b[0], b[1]);
            mma_f16(aQ[3], aq, b[2], b[3]);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const int r = 16 * rb + gq + ((x >> 1) << 3);
          const int cc = 32 * ch + 8 * j + 2 * tq + (x & 1);
          const bool low = r >= cc && r < L;
          const float m = low ? expf(s.G[r] - s.G[cc]) : 0.f;
          s.A[r * LDA + cc] = (low && r > cc) ? s.beta[buf][r] * m * aK[j][x] : 0.f;
          s.P[r * LDC + cc] = __float2half_rn(low ? p.scale * m * aQ[j][x] : 0.f);
        }
      }
    }
    __syncthreads();

    // ---- #3 Solve: Tm = (I + A)^-1, then the bf16 operands Tw, Tu ----------
    solve_unit_lower_64<kThreads>(s.A, LDA, s.Tm, LDA, s.X);
    for (int e = tid; e < kC * kC; e += kThreads) {
      const int r = e >> 6, cc = e & 63;
      const float tv = s.Tm[r * LDA + cc];
      const float b = s.beta[buf][cc];
      s.Tw[r * LDC + cc] = __float2half_rn(tv * b * s.gam[cc]);
      s.Tu[r * LDC + cc] = __float2half_rn(tv * b);
    }
    __syncthreads();

    // ---- #4 W/U: W = Tw K (stored negated), U = Tu V (kept in registers) ----
    const int rb = warp & 3, nq = warp >> 2;  // 16 token rows, half the columns
    constexpr int WNT = DK / 16;              // n8 tiles of W per warp
    constexpr int UNT = DVT / 16;             // n8 tiles of U / V_new / O per warp
    float acc[UNT][4];
#pragma unroll
    for (int j = 0; j < UNT; ++j)
#pragma unroll
      for (int x = 0; x < 4; ++x) acc[j][x] = 0.f;
    {
      float aW[WNT][4];
#pragma unroll
      for (int j = 0; j < WNT; ++j)
#pragma unroll
        for (int x = 0; x < 4; ++x) aW[j][x] = 0.f;
      for (int kk = 0; kk <= 16 * rb; kk += 16) {  // Tw, Tu are lower triangular
        uint32_t a[4], b[4];
        load_a(a, s.Tw, LDC, 16 * rb, kk, lane);
#pragma unroll
        for (int j = 0; j < WNT; j += 2) {
          load_b_kn(b, Ks, LDK, nq * (DK / 2) + 8 * j, kk, lane);
          mma_f16(aW[j], a, b[0], b[1]);
          mma_f16(aW[j + 1], a, b[2], b[3]);
        }
        load_a(a, s.Tu, LDC, 16 * rb, kk, lane);
#pragma unroll
        for (int j = 0; j < UNT; j += 2) {
          load_b_kn(b, s.V[buf], LDV, nq * (DVT / 2) + 8 * j, kk, lane);
          mma_f16(acc[j], a, b[0], b[1]);
          mma_f16(acc[j + 1], a, b[2], b[3]);
        }
      }
#pragma unroll
      for (int j = 0; j < WNT; ++j) {
        const int r0 = 16 * rb + gq, col = nq * (DK / 2) + 8 * j + 2 * tq;
        *reinterpret_cast<uint32_t*>(&s.Wn[r0 * LDK + col]) = pack_f16(-aW[j][0], -aW[j][1]);
        *reinterpret_cast<uint32_t*>(&s.Wn[(r0 + 8) * LDK + col]) =
            pack_f16(-aW[j][2], -aW[j][3]);
      }
    }
    __syncthreads();

    // ---- #5 read: V_new = U + (-W) h ----------------------------------------
#pragma unroll 2
    for (int kk = 0; kk < DK; kk += 16) {
      uint32_t a[4], b[4];
      load_a(a, s.Wn, LDK, 16 * rb, kk, lane);
#pragma unroll
      for (int j = 0; j < UNT; j += 2) {
        load_b_kn(b, s.H, LDV, nq * (DVT / 2) + 8 * j, kk, lane);
        mma_f16(acc[j], a, b[0], b[1]);
        mma_f16(acc[j + 1], a, b[2], b[3]);
      }
    }
    {
      const int r0 = 16 * rb + gq;
      const float e0 = s.e[r0], e1 = s.e[r0 + 8];
#pragma unroll
      for (int j = 0; j < UNT; ++j) {
        const int col = nq * (DVT / 2) + 8 * j + 2 * tq;
        *reinterpret_cast<uint32_t*>(&s.Vn[r0 * LDV + col]) = pack_f16(acc[j][0], acc[j][1]);
        *reinterpret_cast<uint32_t*>(&s.Vn[(r0 + 8) * LDV + col]) =
            pack_f16(acc[j][2], acc[j][3]);
        *reinterpret_cast<uint32_t*>(&s.Ve[r0 * LDV + col]) =
            pack_f16(e0 * acc[j][0], e0 * acc[j][1]);
        *reinterpret_cast<uint32_t*>(&s.Ve[(r0 + 8) * LDV + col]) =
            pack_f16(e1 * acc[j][2], e1 * acc[j][3]);
      }
    }
    __syncthreads();

    // ---- #6 O = diag(scale gamma) Q h + P V_new -----------------------------
    {
#pragma unroll
      for (int j = 0; j < UNT; ++j)
#pragma unroll
        for (int x = 0; x < 4; ++x) acc[j][x] = 0.f;
#pragma unroll 2
      for (int kk = 0; kk < DK; kk += 16) {
        uint32_t a[4], b[4];
        load_a(a, Qs, LDK, 16 * rb, kk, lane);
#pragma unroll
        for (int j = 0; j < UNT; j += 2) {
          load_b_kn(b, s.H, LDV, nq * (DVT / 2) + 8 * j, kk, lane);
          mma_f16(acc[j], a, b[0], b[1]);
          mma_f16(acc[j + 1], a, b[2], b[3]);
        }
      }
      const int r0 = 16 * rb + gq;
      const float s0 = p.scale * s.gam[r0], s1 = p.scale * s.gam[r0 + 8];
#pragma unroll
      for (int j = 0; j < UNT; ++j) {
        acc[j][0] *= s0; acc[j][1] *= s0; acc[j][2] *= s1; acc[j][3] *= s1;
      }
      for (int kk = 0; kk <= 16 * rb; kk += 16) {  // P is lower triangular
        uint32_t a[4], b[4];
        load_a(a, s.P, LDC, 16 * rb, kk, lane);
#pragma unroll
        for (int j = 0; j < UNT; j += 2) {
          load_b_kn(b, s.Vn, LDV, nq * (DVT / 2) + 8 * j, kk, lane);
          mma_f16(acc[j], a, b[0], b[1]);
          mma_f16(acc[j + 1], a, b[2], b[3]);
        }
      }
#pragma unroll
      for (int j = 0; j < UNT; ++j) {
        const int col = nq * (DVT / 2) + 8 * j + 2 * tq;
        if (r0 < L)
          *reinterpret_cast<uint32_t*>(og + (t0 + r0) * v_tok + col) =
              pack_bf16(acc[j][0], acc[j][1]);
        if (r0 + 8 < L)
          *reinterpret_cast<uint32_t*>(og + (t0 + r0 + 8) * v_tok + col) =
              pack_bf16(acc[j][2], acc[j][3]);
      }
    }

    // ---- #5 update: h = gamma_last h + K^T diag(e) V_new ---------------------
    {
      const float gl = s.gam[kC - 1];
#pragma unroll
      for (int j = 0; j < HNT; ++j)
#pragma unroll
        for (int x = 0; x < 4; ++x) hacc[j][x] *= gl;
#pragma unroll
      for (int kk = 0; kk < kC; kk += 16) {
        uint32_t a[4], b[4];
        load_a_trans(a, Ks, LDK, 16 * hmt, kk, lane);
#pragma unroll
        for (int j = 0; j < HNT; j += 2) {
          load_b_kn(b, s.Ve, LDV, hcol0 + 8 * j, kk, lane);
          mma_f16(hacc[j], a, b[0], b[1]);
          mma_f16(hacc[j + 1], a, b[2], b[3]);
        }
      }
    }
    __syncthreads();  // every warp is done reading s.H for this chunk
#pragma unroll
    for (int j = 0; j < HNT; ++j) {
      const int r0 = 16 * hmt + gq, col = hcol0 + 8 * j + 2 * tq;
      *reinterpret_cast<uint32_t*>(&s.H[r0 * LDV + col]) = pack_f16(hacc[j][0], hacc[j][1]);
      *reinterpret_cast<uint32_t*>(&s.H[(r0 + 8) * LDV + col]) = pack_f16(hacc[j][2], hacc[j][3]);
    }
    __syncthreads();  // buffers of this chunk are free, s.H holds the new state
  }

  if (p.hT) {
    float* hT = p.hT + ((long long)(n * p.Hv + hv) * DK) * p.dv + dvt * DVT;
#pragma unroll
    for (int j = 0; j < HNT; ++j) {
      const int r0 = 16 * hmt + gq, col = hcol0 + 8 * j + 2 * tq;
      *reinterpret_cast<float2*>(hT + (long long)r0 * p.dv + col) =
          make_float2(hacc[j][0], hacc[j][1]);
      *reinterpret_cast<float2*>(hT + (long long)(r0 + 8) * p.dv + col) =
          make_float2(hacc[j][2], hacc[j][3]);
    }
  }
}

template <int DK, int DVT>
cudaError_t launch_t(const FwdParams& p, cudaStream_t stream) {
  const size_t smem = sizeof(SmemBf16<DK, DVT>);
  static cudaError_t attr = cudaFuncSetAttribute(
      gdn_fwd_bf16_kernel<DK, DVT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (attr != cudaSuccess) return attr;
  const long long grid = (long long)p.N * p.Hv * (p.dv / DVT);
  gdn_fwd_bf16_kernel<DK, DVT><<<(unsigned)grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_bf16(const FwdParams& p, cudaStream_t stream) {
  if (p.dk == 128) return launch_t<128, 64>(p, stream);
  return launch_t<64, 64>(p, stream);
}

}  // namespace gdn
