// gdn_fwd_f32.cu - chunked-prefill forward with fp32 q/k/v/o (fp32 throughout).
//
// The operators of "Empowering Hybrid Attention Models on NPUs", §2.1 / Figure
// 1(b), in two launches like the bf16 path:
//
//  * gdn_prep_f32_kernel - one CTA per (64-token chunk, v head), all chunks in
//    parallel: #1 Gate (cumsum of g, gamma, e), #2 KKT and the QK^T gram P, #3
//    Solve Tm = (I + A)^-1, #4 W = Tm diag(beta gamma) K and U = Tm diag(beta) V,
//    plus Kt^T = (diag(e) K)^T and Q~ = diag(scale gamma) Q; one fp32 record per
//    task in the workspace.
//  * gdn_chain_f32_kernel - one CTA per (sequence, v head, 16 dv columns), the
//    chunks in order with the state tile h[:, tile] on chip and the next chunk's
//    record loading meanwhile: #5 V_new = U - W h, #6 O = Q~ h + P V_new, then
//    the in-place update h = gamma_last h + Kt^T V_new (the chunk-first order of
//    §5, Figure 10(b)).
//
// Every matrix product runs on the tensor cores in three tf32 MMAs (m16n8k8)
// per step: each fp32 operand is split into a tf32 part and a tf32 remainder,
// x = hi + lo, and A B ~ A_hi B_hi + A_hi B_lo + A_lo B_hi with fp32
// accumulation (the split-precision method of Ootomo and Yokota, "Recovering
// single precision accuracy from Tensor Cores while surpassing the FP32
// theoretical peak performance", 2022): about 21 significant bits per product,
// well inside the fp32 path's tolerance.  The gates and the solve's four diagonal
// 16 x 16 blocks stay fp32 on the CUDA cores; the solve's block merges are products
// like the rest.  Triangular operands are multiplied by their nonzero blocks only.
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

// ---- split-precision tf32 MMA ------------------------------------------------
__device__ __forceinline__ uint32_t f2tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;\n" : "=r"(r) : "f"(x));
  return r;
}
// x = hi + lo: hi = tf32(x), lo = tf32(x - hi)
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
  hi = f2tf32(x);
  lo = f2tf32(x - __uint_as_float(hi));
}
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4],
                                         const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
// Fragment layout of the tf32 MMA (g = lane / 4, t = lane % 4): a = A[g][t], A[g+8][t],
// A[g][t+4], A[g+8][t+4]; b = B[t][g], B[t+4][g]; d = D[g][2t], D[g][2t+1], D[g+8][2t],
// D[g+8][2t+1].
// operands split once and reused: hi/lo of an A fragment (4) or a B fragment (2)
template <int N>
struct Split {
  uint32_t h[N], l[N];
};
template <int N>
__device__ __forceinline__ Split<N> split(const float (&x)[N]) {
  Split<N> r;
#pragma unroll
  for (int i = 0; i < N; ++i) split_tf32(x[i], r.h[i], r.l[i]);
  return r;
}
// d += A_hi B_hi and dx += A_lo B_hi + A_hi B_lo: the big and the small terms in two
// accumulators, so a k-step adds one MMA to each dependence chain of d and two to dx
__device__ __forceinline__ void mma3s(float (&d)[4], float (&dx)[4], const Split<4>& a,
                                      const Split<2>& b) {
  mma_tf32(dx, a.l, b.h);
  mma_tf32(dx, a.h, b.l);
  mma_tf32(d, a.h, b.h);
}
// A fragment of rows r0.., columns k0.. of a row-major matrix with row stride ld
__device__ __forceinline__ void frag_a(float (&a)[4], const float* A, int ld, int r0, int k0,
                                       int g, int t) {
  a[0] = A[(r0 + g) * ld + k0 + t];
  a[1] = A[(r0 + g + 8) * ld + k0 + t];
  a[2] = A[(r0 + g) * ld + k0 + t + 4];
  a[3] = A[(r0 + g + 8) * ld + k0 + t + 4];
}
// B fragment of B[k][n] stored row-major [k][n] (stride ld), rows k0.., columns n0..
__device__ __forceinline__ void frag_b_kn(float (&b)[2], const float* B, int ld, int k0, int n0,
                                          int g, int t) {
  b[0] = B[(k0 + t) * ld + n0 + g];
  b[1] = B[(k0 + t + 4) * ld + n0 + g];
}
// B fragment of B[k][n] = M[n][k] for M stored row-major [n][k] (stride ld)
__device__ __forceinline__ void frag_b_nk(float (&b)[2], const float* M, int ld, int k0, int n0,
                                          int g, int t) {
  b[0] = M[(n0 + g) * ld + k0 + t];
  b[1] = M[(n0 + g) * ld + k0 + t + 4];
}

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
  // row strides: 4 mod 32 for the A-operand rows (fragment rows g, columns t), 8 mod 32
  // for V, read as a [k][n] B operand (rows t, columns g)
  static constexpr int LDK = DK + 4, LDV = DV + 8, LDA = kC + 4;
  float K[kC * LDK];
  float Q[kC * LDK];
  float V[kC * LDV];
  float A[kC * LDA];  // strictly lower A
  float Tm[kC * LDA];
  float X[32 * 40];   // solve scratch: the products Y of the block merges
  float g[kC], beta[kC], G[kC], gam[kC], e[kC];
};

// The 20 gram tiles on and below the diagonal, 5 per warp j: nA column tiles from ntA
// in row block rbA, then 5 - nA from ntB in row block rbB.
struct GramTiles {
  int rbA, ntA, nA, rbB, ntB;
};
__device__ __forceinline__ GramTiles gram_tiles(int j) {
  switch (j) {
    case 0: return {0, 0, 2, 3, 0};  // row block 0: 0-1;  row block 3: 0-2
    case 1: return {1, 0, 4, 3, 3};  // row block 1: 0-3;  row block 3: 3
    case 2: return {2, 0, 5, 2, 5};  // row block 2: 0-4
    default: return {2, 5, 1, 3, 4}; // row block 2: 5;    row block 3: 4-7
  }
}

// Tm = (I + A)^-1 for the strictly lower 64 x 64 A (row stride LD; only the blocks on
// and below the diagonal are read), by 16 x 16 blocks: the four diagonal blocks by
// substitution on the CUDA cores, then two levels of merges on the tensor cores (split
// tf32).  For a unit lower triangular [[L_a, 0], [A_ba, L_b]] the inverse has the
// off-diagonal block -L_b^-1 A_ba L_a^-1: level 1 forms it for the 16-row pairs
// (blocks 1,0 and 3,2), level 2 for the 32-row halves.  X: 32 x 40 floats of scratch.
template <int LD>
__device__ __forceinline__ void solve_f32(const float* A, float* T, float* X, int warp, int lane) {
  const int fg = lane >> 2, ft = lane & 3;
  if (warp < 4) {
    if (lane < 16) {  // diagonal block b, column l: once x_m is final it updates every x_i, i > m
      const int b = warp, l = lane;
      const float* Ab = A + 16 * b * LD + 16 * b;
      float x[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = (i == l) ? 1.f : 0.f;
#pragma unroll
      for (int m = 0; m < 15; ++m)
#pragma unroll
        for (int i = m + 1; i < 16; ++i) x[i] = fmaf(-Ab[i * LD + m], x[m], x[i]);
#pragma unroll
      for (int i = 0; i < 16; ++i) T[(16 * b + i) * LD + 16 * b + l] = x[i];
    }
  } else {
    for (int e = (warp - 4) * 32 + lane; e < 64 * 16; e += 128) {  // 4-column groups
      const int r = e >> 4, c = 4 * (e & 15);
      if ((c >> 4) > (r >> 4))
        *reinterpret_cast<float4*>(&T[r * LD + c]) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  __syncthreads();
  if (warp < 4) {  // level 1: T_IJ = -T_II (A_IJ T_JJ), (I, J) = (1, 0) or (3, 2); 8 columns a warp
    const int I = 2 * (warp >> 1) + 1, J = I - 1, n0 = 16 * J + 8 * (warp & 1);
    float y[4] = {}, yx[4] = {};
#pragma unroll
    for (int k0 = 0; k0 < 16; k0 += 8) {
      float a[4], b[2];
      frag_a(a, A, LD, 16 * I, 16 * J + k0, fg, ft);
      frag_b_kn(b, T, LD, 16 * J + k0, n0, fg, ft);
      mma3s(y, yx, split(a), split(b));
    }
    float* Y = X + warp * 128;  // 16 x 8, row stride 8
#pragma unroll
    for (int i = 0; i < 4; ++i) Y[(fg + 8 * (i >> 1)) * 8 + 2 * ft + (i & 1)] = y[i] + yx[i];
    __syncwarp();
    float t[4] = {}, tx[4] = {};
#pragma unroll
    for (int k0 = 0; k0 < 16; k0 += 8) {
      float a[4], b[2];
      frag_a(a, T, LD, 16 * I, 16 * I + k0, fg, ft);
      frag_b_kn(b, Y, 8, k0, 0, fg, ft);
      mma3s(t, tx, split(a), split(b));
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
      T[(16 * I + fg + 8 * (i >> 1)) * LD + n0 + 2 * ft + (i & 1)] = -(t[i] + tx[i]);
  }
  __syncthreads();
  // level 2: rows 32-63 x columns 0-31 = -T_bb (A_ba T_aa); warp: 16 rows rb, 8 columns n0
  const int rb = warp >> 2, n0 = 8 * (warp & 3);
  {
    float y[4] = {}, yx[4] = {};
    for (int k0 = n0; k0 < 32; k0 += 8) {  // T_aa[k][n] = 0 for k < n
      float a[4], b[2];
      frag_a(a, A, LD, 32 + 16 * rb, k0, fg, ft);
      frag_b_kn(b, T, LD, k0, n0, fg, ft);
      mma3s(y, yx, split(a), split(b));
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) X[(16 * rb + fg + 8 * (i >> 1)) * 40 + n0 + 2 * ft + (i & 1)] = y[i] + yx[i];
  }
  __syncthreads();
  {
    float t[4] = {}, tx[4] = {};
    for (int k0 = 0; k0 < 16 * (rb + 1); k0 += 8) {  // T_bb[r][k] = 0 for k > r
      float a[4], b[2];
      frag_a(a, T, LD, 32 + 16 * rb, 32 + k0, fg, ft);
      frag_b_kn(b, X, 40, k0, n0, fg, ft);
      mma3s(t, tx, split(a), split(b));
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
      T[(32 + 16 * rb + fg + 8 * (i >> 1)) * LD + n0 + 2 * ft + (i & 1)] = -(t[i] + tx[i]);
  }
  __syncthreads();
}

// One of the prep's products out = Tm diag(f) B for a [64][N] operand B (row stride LDB)
// with f = beta gamma (gam given) or beta: this warp's column tiles of row blocks rbs[0]
// and rbs[1], N / 32 tiles of 8 columns each, in half `half` of the columns; out is
// row-major [64][N].
template <int N, int LDB>
__device__ __forceinline__ void wu_product(const float* Tm, int lda, const float* B,
                                           const float* beta, const float* gam,
                                           const int (&rbs)[2], int half, float* out, int fg,
                                           int ft) {
  constexpr int NQ = N / 32;
  float acc[2][NQ][4] = {}, accx[2][NQ][4] = {};
#pragma unroll
  for (int k0 = 0; k0 < kC; k0 += 8) {
    const float f0 = gam ? beta[k0 + ft] * gam[k0 + ft] : beta[k0 + ft];
    const float f1 = gam ? beta[k0 + ft + 4] * gam[k0 + ft + 4] : beta[k0 + ft + 4];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (k0 >= 16 * (rbs[u] + 1)) continue;  // above the diagonal block
      float a[4];
      frag_a(a, Tm, lda, 16 * rbs[u], k0, fg, ft);
      const Split<4> sa = split(a);
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        float b[2];
        frag_b_kn(b, B, LDB, k0, half * (N / 2) + 8 * (u * NQ + q), fg, ft);
        b[0] *= f0;
        b[1] *= f1;
        mma3s(acc[u][q], accx[u][q], sa, split(b));
      }
    }
  }
#pragma unroll
  for (int u = 0; u < 2; ++u)
#pragma unroll
    for (int q = 0; q < NQ; ++q)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r = 16 * rbs[u] + fg + 8 * h, cc = half * (N / 2) + 8 * (u * NQ + q) + 2 * ft;
        *reinterpret_cast<float2*>(&out[r * N + cc]) =
            make_float2(acc[u][q][2 * h] + accx[u][q][2 * h],
                        acc[u][q][2 * h + 1] + accx[u][q][2 * h + 1]);
      }
}

template <int DK, int DV>
__global__ void __launch_bounds__(kThreads) gdn_prep_f32_kernel(const FwdParams p, const WsLayout ws) {
  using S = PrepSmem<DK, DV>;
  using R = RecF32<DK, DV>;
  constexpr int LDK = S::LDK, LDV = S::LDV, LDA = S::LDA;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  S& s = *reinterpret_cast<S*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int fg = lane >> 2, ft = lane & 3;  // MMA fragment row / column group

  const int hv = blockIdx.x % p.Hv;
  const long long slot = blockIdx.x / p.Hv;
  int n, c;
  // the chain launch may come in now: it waits for this grid before reading a record
  griddep_launch_dependents();
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
      *reinterpret_cast<float4*>(&s.K[rr * LDK + d]) = kr[i];
      *reinterpret_cast<float4*>(&s.Q[rr * LDK + d]) = qr[i];
    }
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e4 = tid + i * kThreads, rr = (4 * e4) / DV, d = (4 * e4) % DV;
      *reinterpret_cast<float4*>(&s.V[rr * LDV + d]) = vr[i];
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

  // ---- #2 KK^T and QK^T (warps 0-3: K rows, warps 4-7: Q rows).  Both grams are
  // needed on and below the diagonal only: of the 4 x 8 tiles (16 rows x 8 columns) the
  // 20 with columns below 16 (rb + 1) are formed, 5 per warp, a warp taking the tiles
  // of one or two row blocks (gram_tiles)
  {
    const bool isQ = warp >= 4;
    const int j = warp & 3;
    const GramTiles gt = gram_tiles(j);
    const int rbA = gt.rbA, ntA = gt.ntA, nA = gt.nA, rbB = gt.rbB, ntB = gt.ntB;
    const float* Arows = isQ ? s.Q : s.K;
    float acc[5][4] = {}, accx[5][4] = {};
#pragma unroll 2
    for (int k0 = 0; k0 < DK; k0 += 8) {
      float a[4];
      frag_a(a, Arows, LDK, 16 * rbA, k0, fg, ft);
      const Split<4> sa = split(a);
      frag_a(a, Arows, LDK, 16 * rbB, k0, fg, ft);
      const Split<4> sb = split(a);
#pragma unroll
      for (int t = 0; t < 5; ++t) {
        const bool inA = t < nA;
        float b[2];
        frag_b_nk(b, s.K, LDK, k0, 8 * (inA ? ntA + t : ntB + t - nA), fg, ft);
        mma3s(acc[t], accx[t], inA ? sa : sb, split(b));
      }
    }
#pragma unroll
    for (int t = 0; t < 5; ++t) {
      const bool inA = t < nA;
      const int rb = inA ? rbA : rbB, nt = inA ? ntA + t : ntB + t - nA;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = 16 * rb + fg + 8 * (i >> 1), cc = 8 * nt + 2 * ft + (i & 1);
        const float x = acc[t][i] + accx[t][i];
        const bool low = r >= cc && r < L;
        const float m = low ? expf(s.G[r] - s.G[cc]) : 0.f;
        if (isQ)
          rec[R::P + r * kC + cc] = low ? p.scale * m * x : 0.f;
        else
          s.A[r * LDA + cc] = (low && r > cc && delta) ? s.beta[r] * m * x : 0.f;
      }
    }
  }
  // P above the formed tiles is zero (the chain reads P whole); A there is never read
  for (int i = tid; i < kC * kC / 4; i += kThreads) {
    const int r = (4 * i) / kC, cc = (4 * i) % kC;
    if (cc >= 16 * ((r >> 4) + 1))
      *reinterpret_cast<float4*>(&rec[R::P + r * kC + cc]) = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // Q~ and Kt^T go out while the others finish the grams, 16 bytes a store
  for (int i = tid; i < kC * DK / 4; i += kThreads) {
    const int r = (4 * i) / DK, d = (4 * i) % DK;  // token r, channels d..d+3
    const float f = p.scale * s.gam[r];
    const float4 x = *reinterpret_cast<const float4*>(&s.Q[r * LDK + d]);
    *reinterpret_cast<float4*>(&rec[R::Qt + r * DK + d]) =
        make_float4(f * x.x, f * x.y, f * x.z, f * x.w);
    const int dd = i % DK, j = 4 * (i / DK);  // channel dd, tokens j..j+3
    *reinterpret_cast<float4*>(&rec[R::KtT + dd * kC + j]) =
        make_float4(s.e[j] * s.K[j * LDK + dd], s.e[j + 1] * s.K[(j + 1) * LDK + dd],
                    s.e[j + 2] * s.K[(j + 2) * LDK + dd], s.e[j + 3] * s.K[(j + 3) * LDK + dd]);
  }
  __syncthreads();

  // ---- #3 Solve: Tm = (I + A)^-1
  solve_f32<LDA>(s.A, s.Tm, s.X, warp, lane);

  // ---- #4 W = Tm diag(beta gamma) K, U = Tm diag(beta) V.  Tm is lower triangular, so
  // row block rb needs the k-steps up to 2 rb + 1 only; warp w pairs row blocks j = w % 4
  // and 3 - j (10 k-steps of work per column tile either way) over a quarter of the
  // columns of half w / 4 each
  {
    const int j = warp & 3, half = warp >> 2;
    const int rbs[2] = {j, 3 - j};
    if (delta) wu_product<DK, LDK>(s.Tm, LDA, s.K, s.beta, s.gam, rbs, half, rec + R::W, fg, ft);
    wu_product<DV, LDV>(s.Tm, LDA, s.V, s.beta, nullptr, rbs, half, rec + R::U, fg, ft);
  }
}

// ---------------------------------------------------------------------------
// chain: one (sequence, v head, 16-column dv tile), chunks in order
template <int DK>
struct ChainRec {  // one chunk's record pieces in shared memory
  static constexpr int LDK = DK + 4, LDC = kC + 4;  // A-operand rows: stride 4 mod 32
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
  static constexpr int LDT = kTile + 8;  // B-operand rows [k][n]: stride 8 mod 32 (24)
  ChainRec<DK> rec[kBufs];
  float H[DK * LDT];   // h[:, tile]
  float Vn[kC * LDT];  // V_new[:, tile]
};

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
  constexpr int LDK = ChainRec<DK>::LDK, LDC = ChainRec<DK>::LDC, LDT = S::LDT;
  constexpr int RT = DK / 64;  // update tiles per warp
  extern __shared__ __align__(16) unsigned char smem_raw[];
  S& s = *reinterpret_cast<S*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int fg = lane >> 2, ft = lane & 3;
  // the 16 x 8 output tile of this warp in the 64 x 16 products: rows 16 rb, columns 8 nt
  const int rb = warp >> 1, nt = warp & 1;

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
    s.H[d * LDT + cc] = p.h0 ? p.h0[hoff + (long long)d * DV + cc] : 0.f;
  }
  griddep_wait();  // the records are the prep launch's output
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

    // ---- #5 V_new = U - W h and the Q~ h half of #6 O, both from the old state
    // (rows 16 rb.., columns 8 nt..; each split B fragment of h serves both)
    float ao[4] = {}, aox[4] = {};
    {
      float av[4] = {}, avx[4] = {};
#pragma unroll 4
      for (int k0 = 0; k0 < DK; k0 += 8) {
        float a[4], bb[2];
        frag_b_kn(bb, s.H, LDT, k0, 8 * nt, fg, ft);
        const Split<2> sb = split(bb);
        if (DELTA) {
          frag_a(a, b.W, LDK, 16 * rb, k0, fg, ft);
          mma3s(av, avx, split(a), sb);
        }
        frag_a(a, b.Qt, LDK, 16 * rb, k0, fg, ft);
        mma3s(ao, aox, split(a), sb);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = 16 * rb + fg + 8 * (i >> 1), cc = 8 * nt + 2 * ft + (i & 1);
        s.Vn[r * LDT + cc] = b.U[r * kTile + cc] - (av[i] + avx[i]);
      }
    }
    __syncthreads();
    // ---- #6 O += P V_new (P is zero right of the diagonal block) and the update's
    // product Kt^T V_new (h is still the old state); each split B fragment of V_new
    // serves both
    float hn[RT][4] = {}, hnx[RT][4] = {};
#pragma unroll 2
    for (int k0 = 0; k0 < kC; k0 += 8) {
      float a[4], bb[2];
      frag_b_kn(bb, s.Vn, LDT, k0, 8 * nt, fg, ft);
      const Split<2> sb = split(bb);
      if (k0 < 16 * (rb + 1)) {
        frag_a(a, b.P, LDC, 16 * rb, k0, fg, ft);
        mma3s(ao, aox, split(a), sb);
      }
#pragma unroll
      for (int a2 = 0; a2 < RT; ++a2) {
        frag_a(a, b.KtT, LDC, 16 * rb + 64 * a2, k0, fg, ft);
        mma3s(hn[a2], hnx[a2], split(a), sb);
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = 16 * rb + fg + 8 * h;
      if (r < L)
        *reinterpret_cast<float2*>(og + (t_seq + (long long)c * kC + r) * v_tok + 8 * nt + 2 * ft) =
            make_float2(ao[2 * h] + aox[2 * h], ao[2 * h + 1] + aox[2 * h + 1]);
    }
    __syncthreads();  // every read of h and of this chunk's pieces is done
#pragma unroll
    for (int a2 = 0; a2 < RT; ++a2)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int d = 16 * rb + 64 * a2 + fg + 8 * (i >> 1), cc = 8 * nt + 2 * ft + (i & 1);
        float& hr = s.H[d * LDT + cc];
        hr = fmaf(gl, hr, hn[a2][i] + hnx[a2][i]);
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
      p.hT[hoff + (long long)d * DV + cc] = s.H[d * LDT + cc];
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
    e = launch_after(gdn_chain_f32_kernel<DK, DV, true>, grid, kThreads, sc, stream, p, ws);
  } else {
    e = cudaFuncSetAttribute(gdn_chain_f32_kernel<DK, DV, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sc);
    if (e != cudaSuccess) return e;
    e = launch_after(gdn_chain_f32_kernel<DK, DV, false>, grid, kThreads, sc, stream, p, ws);
  }
  return e;
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
