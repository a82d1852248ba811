// gdn_fwd_f32.cu - chunked-prefill forward with fp32 q/k/v/o (fp32 throughout).
//
// The operators of "Empowering Hybrid Attention Models on NPUs", §2.1 / Figure
// 1(b), in two launches like the bf16 path, every product an fp32 FMA on the
// CUDA cores:
//
//  * gdn_prep_f32_kernel - one CTA per (64-token chunk, v head), all chunks in
//    parallel: #1 Gate (cumsum of g, gamma, e), #2 KKT and the QK^T gram P, #3
//    Solve Tm = (I + A)^-1, #4 W = Tm diag(beta gamma) K and U = Tm diag(beta) V,
//    plus Kt^T = (diag(e) K)^T and Q~ = diag(scale gamma) Q; one fp32 record per
//    task in the workspace.
//  * gdn_chain_f32_kernel - one CTA per (sequence, v head, 16 dv columns), the
//    chunks in order with the state tile h[:, tile] on chip and the next chunk's
//    record loading meanwhile: #5 V_new = U - W h,
//    #6 O = Q~ h + P V_new, then the in-place update h = gamma_last h + Kt^T V_new
//    (the chunk-first order of §5, Figure 10(b)).
//
// Without the delta rule's erase term (the Mamba-2 scan) A = 0, so Tm = I and the
// chain takes V_new = U = diag(beta) V.
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kC = 64;
constexpr int kThreads = 256;
constexpr int kTile = 16;  // dv columns per chain CTA

// fp32 record of one (chunk slot, v head), offsets in floats; every piece is a
// multiple of 4 floats (16 bytes) long.
template <int DK, int DV>
struct RecF32 {
  static constexpr int W = 0;                   // W [64][DK]
  static constexpr int KtT = W + kC * DK;       // (diag(e) K)^T [DK][64]
  static constexpr int Qt = KtT + DK * kC;      // diag(scale gamma) Q [64][DK]
  static constexpr int P = Qt + kC * DK;        // P [64][64]
  static constexpr int U = P + kC * kC;         // U [64][DV]
  static constexpr int Gl = U + kC * DV;        // gamma_last, 3 pad
  static constexpr int kFloats = (Gl + 4 + 31) / 32 * 32;
};

// ---------------------------------------------------------------------------
// prep: one chunk of one v head
template <int DK, int DV>
struct PrepSmem {
  static constexpr int LDK = DK + 1, LDV = DV + 1, LDA = kC + 1;  // odd strides
  float K[kC * LDK];
  float Q[kC * LDK];
  float V[kC * LDV];
  float A[kC * LDA];  // strictly lower A
  float Tm[kC * LDA];
  float P[kC * LDA];
  float X[3 * 256];   // solve scratch
  float g[kC], beta[kC], G[kC], gam[kC], e[kC];
};

template <int DK, int DV>
__global__ void __launch_bounds__(kThreads) gdn_prep_f32_kernel(const FwdParams p, const WsLayout ws) {
  using S = PrepSmem<DK, DV>;
  using R = RecF32<DK, DV>;
  constexpr int LDK = S::LDK, LDV = S::LDV, LDA = S::LDA;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  S& s = *reinterpret_cast<S*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ti = tid >> 4, tj = tid & 15;  // 16 x 16 thread grid for register tiles

  const int hv = blockIdx.x % p.Hv;
  const long long slot = blockIdx.x / p.Hv;
  int n, c;
  if (!locate_chunk(p, ws, slot, &n, &c)) return;
  const long long t_seq = p.cu_seqlens ? (long long)p.cu_seqlens[n] : (long long)n * p.T;
  const long long len = p.cu_seqlens ? (long long)p.cu_seqlens[n + 1] - t_seq : (long long)p.T;
  const long long t0 = t_seq + (long long)c * kC;
  const int L = (int)min((long long)kC, len - (long long)c * kC);
  const int hq = qk_head(hv, p.Hqk, p.Hv, p.head_map);
  const bool delta = p.delta_rule != 0;
  const long long qk_tok = (long long)p.Hqk * DK, v_tok = (long long)p.Hv * DV;
  const float* qg = static_cast<const float*>(p.q) + (long long)hq * DK;
  const float* kg = static_cast<const float*>(p.k) + (long long)hq * DK;
  const float* vg = static_cast<const float*>(p.v) + (long long)hv * DV;
  float* rec = reinterpret_cast<float*>(ws.base) + (slot * p.Hv + hv) * (long long)R::kFloats;

  // ---- loads (rows past the sequence are zero; their g and beta are 0): every load of
  // a thread is issued before its first shared-memory store, 16 bytes at a time
  {
    constexpr int NK = kC * DK / 4 / kThreads, NV = kC * DV / 4 / kThreads;
    float4 kr[NK], qr[NK], vr[NV];
#pragma unroll
    for (int i = 0; i < NK; ++i) {
      const int e4 = tid + i * kThreads, rr = (4 * e4) / DK, d = (4 * e4) % DK;
      const bool ok = rr < L;
      kr[i] = ok ? __ldg(reinterpret_cast<const float4*>(kg + (t0 + rr) * qk_tok + d))
                 : make_float4(0.f, 0.f, 0.f, 0.f);
      qr[i] = ok ? __ldg(reinterpret_cast<const float4*>(qg + (t0 + rr) * qk_tok + d))
                 : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e4 = tid + i * kThreads, rr = (4 * e4) / DV, d = (4 * e4) % DV;
      vr[i] = rr < L ? __ldg(reinterpret_cast<const float4*>(vg + (t0 + rr) * v_tok + d))
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float gv = 0.f, bv = 0.f;
    if (tid < kC && tid < L) {
      gv = __ldg(p.g + (t0 + tid) * p.Hv + hv);
      bv = __ldg(p.beta + (t0 + tid) * p.Hv + hv);
    }
#pragma unroll
    for (int i = 0; i < NK; ++i) {
      const int e4 = tid + i * kThreads, rr = (4 * e4) / DK, d = (4 * e4) % DK;
      float* kd = &s.K[rr * LDK + d];
      float* qd = &s.Q[rr * LDK + d];
      kd[0] = kr[i].x, kd[1] = kr[i].y, kd[2] = kr[i].z, kd[3] = kr[i].w;
      qd[0] = qr[i].x, qd[1] = qr[i].y, qd[2] = qr[i].z, qd[3] = qr[i].w;
    }
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e4 = tid + i * kThreads, rr = (4 * e4) / DV, d = (4 * e4) % DV;
      float* vd = &s.V[rr * LDV + d];
      vd[0] = vr[i].x, vd[1] = vr[i].y, vd[2] = vr[i].z, vd[3] = vr[i].w;
    }
    if (tid < kC) {
      s.g[tid] = gv;
      s.beta[tid] = bv;
    }
  }
  __syncthreads();

  // ---- #1 Gate: G = cumsum(g), gamma = exp(G), e = exp(G_last - G)
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
    if (lane == 31) rec[R::Gl] = expf(Glast);
  }
  __syncthreads();

  // ---- #2 KK^T and QK^T: thread (ti, tj) owns rows ti + 16a, columns tj + 16b
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
        s.A[r * LDA + cc] = (low && r > cc && delta) ? s.beta[r] * m * sk[a][b] : 0.f;
        const float pv = low ? p.scale * m * sq[a][b] : 0.f;
        s.P[r * LDA + cc] = pv;
        rec[R::P + r * kC + cc] = pv;
      }
  }
  // Kt^T and Q~ go out while the grams are formed
  for (int i = tid; i < kC * DK; i += kThreads) {
    const int r = i / DK, d = i % DK;  // token r, channel d
    rec[R::Qt + r * DK + d] = p.scale * s.gam[r] * s.Q[r * LDK + d];
    const int dd = i / kC, j = i % kC;  // channel dd, token j: coalesced transposed store
    rec[R::KtT + dd * kC + j] = s.e[j] * s.K[j * LDK + dd];
  }
  __syncthreads();

  // ---- #3 Solve: Tm = (I + A)^-1
  solve_unit_lower_64_f32<kThreads>(s.A, LDA, s.Tm, LDA, s.X);

  // ---- #4 W = Tm diag(beta gamma) K, U = Tm diag(beta) V: rows ti + 16a, columns tj + 16b
  if (delta) {
    constexpr int NB = DK / 16;
    float w[4][NB] = {};
    for (int j = 0; j < kC; ++j) {
      const float f = s.beta[j] * s.gam[j];
      float tr[4], kc[NB];
#pragma unroll
      for (int a = 0; a < 4; ++a) tr[a] = s.Tm[(ti + 16 * a) * LDA + j];
#pragma unroll
      for (int b = 0; b < NB; ++b) kc[b] = f * s.K[j * LDK + tj + 16 * b];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < NB; ++b) w[a][b] += tr[a] * kc[b];
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < NB; ++b) rec[R::W + (ti + 16 * a) * DK + tj + 16 * b] = w[a][b];
  }
  {
    constexpr int NB = DV / 16;
    float u[4][NB] = {};
    for (int j = 0; j < kC; ++j) {
      const float f = s.beta[j];
      float tr[4], vc[NB];
#pragma unroll
      for (int a = 0; a < 4; ++a) tr[a] = s.Tm[(ti + 16 * a) * LDA + j];
#pragma unroll
      for (int b = 0; b < NB; ++b) vc[b] = f * s.V[j * LDV + tj + 16 * b];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < NB; ++b) u[a][b] += tr[a] * vc[b];
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < NB; ++b) rec[R::U + (ti + 16 * a) * DV + tj + 16 * b] = u[a][b];
  }
}

// ---------------------------------------------------------------------------
// chain: one (sequence, v head, 16-column dv tile), chunks in order
template <int DK>
struct ChainRec {  // one chunk's record pieces in shared memory
  static constexpr int LDK = DK + 4, LDC = kC + 4;  // float4 rows, banks spread
  float W[kC * LDK];
  float Qt[kC * LDK];
  float KtT[DK * LDC];
  float P[kC * LDC];
  float U[kC * kTile];
};
// two record buffers where they fit (dk = 64): the next chunk's pieces load while
// this chunk computes
template <int DK>
struct ChainSmem {
  static constexpr int kBufs = DK == 64 ? 2 : 1;
  ChainRec<DK> rec[kBufs];
  float H[DK * kTile];   // h[:, tile]
  float Vn[kC * kTile];  // V_new[:, tile]
};

__device__ __forceinline__ float4 lds4(const float* a) { return *reinterpret_cast<const float4*>(a); }
__device__ __forceinline__ void fma4(float4& acc, float a, const float4& b) {
  acc.x = fmaf(a, b.x, acc.x);
  acc.y = fmaf(a, b.y, acc.y);
  acc.z = fmaf(a, b.z, acc.z);
  acc.w = fmaf(a, b.w, acc.w);
}
// A[row][0..K) x B[0..K)[cg..cg+4), A row-major, B [K][kTile]; two accumulators (even
// and odd groups of four k) halve the dependent FMA chain
template <int K>
__device__ __forceinline__ float4 row_times_tile(const float* arow, const float* B, int cg) {
  float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
#pragma unroll 2
  for (int k = 0; k < K; k += 8) {
    const float4 x = lds4(arow + k), y = lds4(arow + k + 4);
    fma4(a0, x.x, lds4(B + (k + 0) * kTile + cg));
    fma4(a1, y.x, lds4(B + (k + 4) * kTile + cg));
    fma4(a0, x.y, lds4(B + (k + 1) * kTile + cg));
    fma4(a1, y.y, lds4(B + (k + 5) * kTile + cg));
    fma4(a0, x.z, lds4(B + (k + 2) * kTile + cg));
    fma4(a1, y.z, lds4(B + (k + 6) * kTile + cg));
    fma4(a0, x.w, lds4(B + (k + 3) * kTile + cg));
    fma4(a1, y.w, lds4(B + (k + 7) * kTile + cg));
  }
  return make_float4(a0.x + a1.x, a0.y + a1.y, a0.z + a1.z, a0.w + a1.w);
}

// issue the cp.async copies of one chunk's record pieces (the caller commits)
template <int DK, int DV, bool DELTA>
__device__ __forceinline__ void load_rec(ChainRec<DK>& d, const float* rec, int tile, int tid) {
  using R = RecF32<DK, DV>;
  constexpr int LDK = ChainRec<DK>::LDK, LDC = ChainRec<DK>::LDC;
  if (DELTA)
    for (int i = tid; i < kC * DK / 4; i += kThreads) {
      const int rr = (4 * i) / DK, dd = (4 * i) % DK;
      cp_async16(&d.W[rr * LDK + dd], rec + R::W + 4 * i, true);
    }
  for (int i = tid; i < kC * DK / 4; i += kThreads) {
    const int rr = (4 * i) / DK, dd = (4 * i) % DK;
    cp_async16(&d.Qt[rr * LDK + dd], rec + R::Qt + 4 * i, true);
    const int kk = (4 * i) / kC, j = (4 * i) % kC;
    cp_async16(&d.KtT[kk * LDC + j], rec + R::KtT + 4 * i, true);
  }
  for (int i = tid; i < kC * kC / 4; i += kThreads) {
    const int rr = (4 * i) / kC, j = (4 * i) % kC;
    cp_async16(&d.P[rr * LDC + j], rec + R::P + 4 * i, true);
  }
  {
    const int rr = tid >> 2, q4 = tid & 3;  // U[:, tile]: 64 rows of 16 floats
    cp_async16(&d.U[rr * kTile + 4 * q4], rec + R::U + rr * DV + tile * kTile + 4 * q4, true);
  }
}

template <int DK, int DV, bool DELTA>
__global__ void __launch_bounds__(kThreads) gdn_chain_f32_kernel(const FwdParams p, const WsLayout ws) {
  using S = ChainSmem<DK>;
  using R = RecF32<DK, DV>;
  constexpr int LDK = ChainRec<DK>::LDK, LDC = ChainRec<DK>::LDC;
  constexpr int RA = DK / 64;  // state rows of a thread in the update
  extern __shared__ __align__(16) unsigned char smem_raw[];
  S& s = *reinterpret_cast<S*>(smem_raw);
  const int tid = threadIdx.x;
  const int r = tid >> 2, cg = (tid & 3) * 4;  // token row and first column of this thread

  constexpr int n_tiles = DV / kTile;
  const int tile = blockIdx.x % n_tiles;
  const int hv = (blockIdx.x / n_tiles) % p.Hv;
  const int n = blockIdx.x / (n_tiles * p.Hv);
  const long long t_seq = p.cu_seqlens ? (long long)p.cu_seqlens[n] : (long long)n * p.T;
  const long long len = p.cu_seqlens ? (long long)p.cu_seqlens[n + 1] - t_seq : (long long)p.T;
  const int n_chunks = (int)((len + kC - 1) / kC);
  const long long slot0 = ws.first_slot(p, n);
  const long long hoff = (long long)(n * p.Hv + hv) * DK * DV + tile * kTile;
  const float* recs = reinterpret_cast<const float*>(ws.base);
  auto rec_of = [&](int c) { return recs + ((slot0 + c) * p.Hv + hv) * (long long)R::kFloats; };
  float* og = static_cast<float*>(p.o) + (long long)hv * DV + tile * kTile;
  const long long v_tok = (long long)p.Hv * DV;

  for (int i = tid; i < DK * kTile; i += kThreads) {
    const int d = i / kTile, cc = i % kTile;
    s.H[i] = p.h0 ? p.h0[hoff + (long long)d * DV + cc] : 0.f;
  }
  if (n_chunks > 0) {
    load_rec<DK, DV, DELTA>(s.rec[0], rec_of(0), tile, tid);
    cp_async_commit();
  }

  for (int c = 0; c < n_chunks; ++c) {
    ChainRec<DK>& b = s.rec[c % S::kBufs];
    const int L = (int)min((long long)kC, len - (long long)c * kC);
    const float gl = rec_of(c)[R::Gl];
    cp_async_wait<0>();
    __syncthreads();  // this chunk's pieces are in; the other buffer is free
    if (S::kBufs == 2 && c + 1 < n_chunks) {
      load_rec<DK, DV, DELTA>(s.rec[(c + 1) % S::kBufs], rec_of(c + 1), tile, tid);
      cp_async_commit();
    }

    // ---- #5 V_new = U - W h   (row r, columns cg..cg+3)
    {
      float4 v = lds4(&b.U[r * kTile + cg]);
      if (DELTA) {
        const float4 wh = row_times_tile<DK>(&b.W[r * LDK], s.H, cg);
        v.x -= wh.x;
        v.y -= wh.y;
        v.z -= wh.z;
        v.w -= wh.w;
      }
      *reinterpret_cast<float4*>(&s.Vn[r * kTile + cg]) = v;
    }
    __syncthreads();
    // ---- #6 O = Q~ h + P V_new, and the update's products (h is still the old state)
    {
      const float4 o1 = row_times_tile<DK>(&b.Qt[r * LDK], s.H, cg);
      const float4 o2 = row_times_tile<kC>(&b.P[r * LDC], s.Vn, cg);
      if (r < L)
        *reinterpret_cast<float4*>(og + (t_seq + (long long)c * kC + r) * v_tok + cg) =
            make_float4(o1.x + o2.x, o1.y + o2.y, o1.z + o2.z, o1.w + o2.w);
    }
    float4 hn[RA];
#pragma unroll
    for (int a = 0; a < RA; ++a) hn[a] = row_times_tile<kC>(&b.KtT[(r + 64 * a) * LDC], s.Vn, cg);
    __syncthreads();  // every read of h and of this chunk's pieces is done
#pragma unroll
    for (int a = 0; a < RA; ++a) {
      float* hp = &s.H[(r + 64 * a) * kTile + cg];
      const float4 h = lds4(hp);
      *reinterpret_cast<float4*>(hp) =
          make_float4(fmaf(gl, h.x, hn[a].x), fmaf(gl, h.y, hn[a].y), fmaf(gl, h.z, hn[a].z),
                      fmaf(gl, h.w, hn[a].w));
    }
    if (S::kBufs == 1 && c + 1 < n_chunks) {
      __syncthreads();  // the single buffer is free again
      load_rec<DK, DV, DELTA>(s.rec[0], rec_of(c + 1), tile, tid);
      cp_async_commit();
    }
  }
  __syncthreads();
  if (p.hT) {
    for (int i = tid; i < DK * kTile; i += kThreads) {
      const int d = i / kTile, cc = i % kTile;
      p.hT[hoff + (long long)d * DV + cc] = s.H[i];
    }
  }
}

template <int DK, int DV>
cudaError_t launch_dd(const FwdParams& p, const WsLayout& ws, cudaStream_t stream) {
  const size_t sp = sizeof(PrepSmem<DK, DV>), sc = sizeof(ChainSmem<DK>);
  cudaError_t e = cudaFuncSetAttribute(gdn_prep_f32_kernel<DK, DV>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sp);
  if (e != cudaSuccess) return e;
  gdn_prep_f32_kernel<DK, DV><<<(unsigned)(ws.n_slots * p.Hv), kThreads, sp, stream>>>(p, ws);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)((long long)p.N * p.Hv * (DV / kTile));
  if (p.delta_rule) {
    e = cudaFuncSetAttribute(gdn_chain_f32_kernel<DK, DV, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sc);
    if (e != cudaSuccess) return e;
    gdn_chain_f32_kernel<DK, DV, true><<<grid, kThreads, sc, stream>>>(p, ws);
  } else {
    e = cudaFuncSetAttribute(gdn_chain_f32_kernel<DK, DV, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sc);
    if (e != cudaSuccess) return e;
    gdn_chain_f32_kernel<DK, DV, false><<<grid, kThreads, sc, stream>>>(p, ws);
  }
  return cudaGetLastError();
}

template <int DK, int DV>
size_t rec_bytes() {
  return (size_t)RecF32<DK, DV>::kFloats * 4;
}

}  // namespace

size_t f32_rec_bytes(const FwdParams& p) {
  if (p.dk == 128) return p.dv == 128 ? rec_bytes<128, 128>() : rec_bytes<128, 64>();
  return p.dv == 128 ? rec_bytes<64, 128>() : rec_bytes<64, 64>();
}

cudaError_t launch_fwd_f32(const FwdParams& p, const WsLayout& ws, cudaStream_t stream) {
  if (p.dk == 128) return p.dv == 128 ? launch_dd<128, 128>(p, ws, stream) : launch_dd<128, 64>(p, ws, stream);
  return p.dv == 128 ? launch_dd<64, 128>(p, ws, stream) : launch_dd<64, 64>(p, ws, stream);
}

}  // namespace gdn
