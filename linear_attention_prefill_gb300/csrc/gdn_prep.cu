// gdn_prep.cu - the chunk-parallel Map phase of the chunkwise forward.
//
// "Empowering Hybrid Attention Models on NPUs", §2.1, Figure 1(b): operators
// #1-#4 (Gate, KKT, Solve, W/U) depend only on one chunk's q, k, v, g, beta,
// so every (chunk, v head) is an independent task here:
//   #1 Gate   G = cumsum(g), gamma = exp(G), e_j = exp(G_last - G_j)
//   #2 KKT    A = tril_strict(beta_i exp(G_i - G_j) k_i.k_j)
//      QK^T   P = tril(scale exp(G_i - G_j) q_i.k_j)
//   #3 Solve  Tm = (I + A)^-1   (diagonal blocks by substitution, merges on mma.sync)
//   #4 W/U    W = Tm diag(beta gamma) K,  U = Tm diag(beta) V
// plus the scaled copies Kt = diag(e) K (the state update's left factor) and
// Q~ = diag(scale gamma) Q (the output's left factor, fp16), and the row
// factors gamma.  The serial Reduce (#5) and the final Map (#6) run in
// gdn_chain.cu, which reads this kernel's workspace records.
//
// Blackwell mapping.  K and Q arrive by TMA in 128-byte-swizzled tiles stacked
// as one 128-row operand [K; Q], so a single M = 128 tcgen05 MMA chain gives
// both grams (K K^T in tensor-memory lanes 0-63, Q K^T in lanes 64-127).  The
// same K tile, read MN-major, is the left factor of W^T = K^T (Tm diag(beta
// gamma))^T, and V (loaded into the Q rows once Q is consumed) that of U^T:
// the products come out transposed, one d index per tensor-memory lane, so each
// thread writes whole 16-byte row segments of W^T and U^T.  Accumulators stay
// in 128 tensor-memory columns and shared memory in ~54 KB (the Q rows hold the
// solve's fp16 tiles, then V), so four tasks share an SM.  The triangular solve
// keeps its fp32 diagonal blocks and fp16 mma.sync merges, and writes the
// scaled MMA operands directly.
//
// Precision: products accumulate in fp32.  The grams and W take the bf16
// inputs as they are (W's left factor rounded to bf16: its share of the error
// is below 1e-3 of RMS); U takes fp16 operands (v rewritten in place, exact in
// fp16's normal range), since U's rounding feeds V_new and the output directly.
#include <cudaTypedefs.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

constexpr int kC = 64;
constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;

// Shared-memory map (byte offsets from a 1024-aligned base), ~54 KB at d = 128
// so that four tasks share an SM.  The Q rows are reused twice: once the grams
// have read Q they hold the solve's fp16 copies Ah and Th, and once the solve
// is done they take V.
template <int DK, int DV>
struct PrepLayout {
  // [DK/64][128 rows][64] bf16, 128-byte swizzle: rows 0-63 K, rows 64-127 Q
  static constexpr int kKQBytes = (DK / 64) * 16384;
  static constexpr bool kThInQ = DK == 128;             // Th in the second block's Q rows
  static constexpr bool kVinQ = DV <= DK;               // V in the Q rows after the solve
  static constexpr int kAh = 8192;                      // fp16 [64][64] swz<64>, first Q rows
  static constexpr int kTh = kThInQ ? 24576 : kKQBytes; // fp16 [64][64] swz<64>
  static constexpr int kAfterTh = kKQBytes + (kThInQ ? 0 : 8192);
  static constexpr int kV = kVinQ ? 8192 : kAfterTh;
  static constexpr int kVStride = kVinQ ? 16384 : 8192;  // bytes between 64-column blocks
  static constexpr int kTw = kAfterTh + (kVinQ ? 0 : (DV / 64) * 8192);  // bf16 [64][64] sw128
  static constexpr int kTu = kTw + 8192;                                   // fp16 [64][64] sw128
  static constexpr int kAd = kTu + 8192;               // fp32 diagonal blocks of A [4][16][16]
  static constexpr int kVec = kAd + 4 * 256 * 4;  // beta, G (log2 units), gamma, e, beta*gamma, 1/|k|, 1/|q|
  static constexpr int kBar = kVec + 7 * kC * 4;  // 5 mbarriers, tmem address, abort flag
  static constexpr int kBytes = kBar + 64;
  static constexpr int kAlloc = kBytes + 1024;         // slack to align the base
  static_assert(kTw % 1024 == 0 && kTh % 1024 == 0 && kAd % 16 == 0 && kVec % 16 == 0, "alignment");
};

// 8 bf16 values at p (16-byte aligned) times `scale`, rounded once to fp16.
__device__ __forceinline__ uint4 scale_bf16x8_to_f16(const void* p, float scale) {
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

__device__ __forceinline__ uint4 pack8_f16(const float* x) {
  return make_uint4(pack_f16(x[0], x[1]), pack_f16(x[2], x[3]), pack_f16(x[4], x[5]),
                    pack_f16(x[6], x[7]));
}

// Store T(r, c) and T(r, c + 1) (c even) into the solve's outputs: the fp16
// copy Th (when given) and the MMA operands Tw = T diag(beta gamma) (bf16) and
// Tu = T diag(beta) (fp16).
__device__ __forceinline__ void put_t2(__half* Th, __half* Tw, __half* Tu, const float* bg,
                                       const float* beta, int r, int c, float t0, float t1) {
  if (Th) *reinterpret_cast<uint32_t*>(&Th[swz<kC>(r, c)]) = pack_f16(t0, t1);
  *reinterpret_cast<uint32_t*>(&Tw[sw128(r, c)]) = pack_bf16(t0 * bg[c], t1 * bg[c + 1]);
  *reinterpret_cast<uint32_t*>(&Tu[sw128(r, c)]) = pack_f16(t0 * beta[c], t1 * beta[c + 1]);
}

template <int DK, int DV>
__global__ void __launch_bounds__(kThreads, 4)
    gdn_prep_kernel(const FwdParams p, const WsLayout ws, const __grid_constant__ CUtensorMap tmq,
                    const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
  using Lo = PrepLayout<DK, DV>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(sm);
  __half* Tw = reinterpret_cast<__half*>(sm + Lo::kTw);  // bf16 bits
  __half* Tu = reinterpret_cast<__half*>(sm + Lo::kTu);
  __half* Ah = reinterpret_cast<__half*>(sm + Lo::kAh);
  __half* Th = reinterpret_cast<__half*>(sm + Lo::kTh);
  float* Ad = reinterpret_cast<float*>(sm + Lo::kAd);
  float* s_beta = reinterpret_cast<float*>(sm + Lo::kVec);
  float* s_G = s_beta + kC;
  float* s_gam = s_G + kC;
  float* s_e = s_gam + kC;
  float* s_bg = s_e + kC;
  float* s_rk = s_bg + kC;  // 1/|k_r| with the fused prologue, else 1
  float* s_rq = s_rk + kC;  // 1/|q_r| likewise
  uint64_t* bar_kq = reinterpret_cast<uint64_t*>(sm + Lo::kBar);
  uint64_t* bar_v = bar_kq + 1;
  uint64_t* bar_mma = bar_kq + 2;  // grams
  uint64_t* bar_w = bar_kq + 3;    // W^T product
  uint64_t* bar_u = bar_kq + 4;    // U^T product
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bar_kq + 5);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;

  GDN_PHASE_INIT;
  // task -> (chunk slot, v head) -> (sequence, chunk within it)
  const int hv = blockIdx.x % p.Hv;
  const long long slot = blockIdx.x / p.Hv;
  int n, c;
  // the chain launch may come in now: it waits for this grid before reading a record
  griddep_launch_dependents();
  if (!locate_chunk(p, ws, slot, &n, &c)) return;  // before any allocation
  const long long t_seq = p.cu_seqlens ? (long long)p.cu_seqlens[n] : (long long)n * p.T;
  const long long len =
      p.cu_seqlens ? (long long)p.cu_seqlens[n + 1] - t_seq : (long long)p.T;
  const int t0 = (int)(t_seq + (long long)c * kC);  // row in the flattened [tokens, H d] maps
  const int L = (int)min((long long)kC, len - (long long)c * kC);
  const int hq = qk_head(hv, p.Hqk, p.Hv, p.head_map);

  // ---- setup: barriers, the K/Q (and a separate V) loads, tensor memory -----
  if (tid == 0) {
    mbar_init(bar_kq, 1);
    mbar_init(bar_v, 1);
    mbar_init(bar_mma, 1);
    mbar_init(bar_w, 1);
    mbar_init(bar_u, 1);
    *s_abort = 0;
    mbar_fence_init();
    mbar_expect_tx(bar_kq, 2u * kC * DK * 2);
#pragma unroll
    for (int kb = 0; kb < DK / 64; ++kb) {
      tma_load_2d(sm + kb * 16384, &tmk, hq * DK + kb * 64, t0, bar_kq);
      tma_load_2d(sm + kb * 16384 + 8192, &tmq, hq * DK + kb * 64, t0, bar_kq);
    }
    if (!Lo::kVinQ) {
      mbar_expect_tx(bar_v, (unsigned)kC * DV * 2);
#pragma unroll
      for (int vb = 0; vb < DV / 64; ++vb)
        tma_load_2d(sm + Lo::kV + vb * Lo::kVStride, &tmv, hv * DV + vb * 64, t0, bar_v);
    } else {  // V's shared-memory slot frees up only after the grams: stage it in L2 now
#pragma unroll
      for (int vb = 0; vb < DV / 64; ++vb) tma_prefetch_2d(&tmv, hv * DV + vb * 64, t0);
    }
  }
  __syncwarp();
  if (warp == 0) tmem_alloc(s_tmem, 128);
  // ---- #1 Gate (rows past the sequence carry g = beta = 0, so G[63] = G_last)
  if (warp == 1) {
    const int r0 = 2 * lane, r1 = 2 * lane + 1;
    const float* gp = p.g + (long long)t0 * p.Hv + hv;
    const float* bp = p.beta + (long long)t0 * p.Hv + hv;
    float g0 = r0 < L ? gp[(long long)r0 * p.Hv] : 0.f;
    float g1 = r1 < L ? gp[(long long)r1 * p.Hv] : 0.f;
    float b0 = r0 < L ? bp[(long long)r0 * p.Hv] : 0.f;
    float b1 = r1 < L ? bp[(long long)r1 * p.Hv] : 0.f;
    if (p.prologue) {  // raw gates: g = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b)
      const float amul = p.A_log ? expf(p.A_log[hv]) : 1.f;
      const float abias = p.dt_bias ? p.dt_bias[hv] : 0.f;
      auto softplus = [](float x) { return x > 20.f ? x : log1pf(expf(x)); };
      g0 = r0 < L ? -amul * softplus(g0 + abias) : 0.f;
      g1 = r1 < L ? -amul * softplus(g1 + abias) : 0.f;
      b0 = r0 < L ? 1.f / (1.f + expf(-b0)) : 0.f;
      b1 = r1 < L ? 1.f / (1.f + expf(-b1)) : 0.f;
    }
    float incl = g0 + g1;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    const float Glast = __shfl_sync(0xffffffffu, incl, 31);
    const float G0 = incl - g1, G1 = incl;
    const float gam0 = expf(G0), gam1 = expf(G1);
    s_G[r0] = G0 * kLog2e;  // log2 units: the masks' exponent
    s_G[r1] = G1 * kLog2e;
    s_gam[r0] = gam0;
    s_gam[r1] = gam1;
    s_e[r0] = expf(Glast - G0);
    s_e[r1] = expf(Glast - G1);
    s_beta[r0] = b0;
    s_beta[r1] = b1;
    s_bg[r0] = p.delta_rule ? b0 * gam0 : 0.f;  // W's column factor: 0 without the erase
    s_bg[r1] = p.delta_rule ? b1 * gam1 : 0.f;
    s_rk[r0] = s_rk[r1] = s_rq[r0] = s_rq[r1] = 1.f;
    float* gv = ws.gv(slot, hv, p.Hv);  // gamma_last, then gamma of every row
    if (lane == 31) gv[0] = expf(Glast);
    if (!p.prologue) {
      *reinterpret_cast<float2*>(gv + 4 + r0) = make_float2(gam0, gam1);
      *reinterpret_cast<float2*>(gv + 68 + r0) = make_float2(s_e[r0], s_e[r1]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  GDN_PHASE(0);  // setup + gate

  // ---- #2 grams: one M = 128 MMA chain, [K; Q] K^T -> tensor columns 0-63 ----
  // One thread spins on each barrier; the others block in bar.sync and then
  // observe the completed phase with a single test.
  if (tid == 0 && !mbar_wait(bar_kq, 0, p.err)) *s_abort = 1;
  __syncthreads();
  if (!*s_abort) mbar_wait(bar_kq, 0, p.err);
  GDN_STAMP(32, 0);  // K, Q landed
  if (L < kC) {  // ragged chunk: rows past the sequence end are zero
    for (int i = tid; i < (DK / 64) * 2 * (kC - L) * 8; i += kThreads) {
      const int ch = i & 7, rr = L + ((i >> 3) % (kC - L)), blk = (i >> 3) / (kC - L);
      *reinterpret_cast<uint4*>(sm + blk * 8192 + rr * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async();
    __syncthreads();
  }
  if (p.prologue) {
    // fused prologue: 1/sqrt(sum x^2 + eps) of every k and q row (two threads a row,
    // 8 of its 16-byte chunks each), folded into the factors the later steps apply:
    // Kt's row factor e, W's column factor beta gamma, and the gamma the output
    // stage multiplies q rows by
    const int R = tid >> 1, half = tid & 1;  // R < 64: k row, else q row R - 64
    const int r = R & (kC - 1);
    float ss = 0.f;
    for (int ch = half * (DK / 16); ch < (half + 1) * (DK / 16); ++ch) {
      const uint4 raw = *reinterpret_cast<const uint4*>(
          sm + (ch >> 3) * 16384 + (R >= kC ? 8192 : 0) + r * 128 + (((ch & 7) ^ (r & 7)) << 4));
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(b2[i]);
        ss = fmaf(f.x, f.x, fmaf(f.y, f.y, ss));
      }
    }
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    const float inv = rsqrtf(ss + kNormEps);
    if (half == 0) {
      if (R < kC) {
        s_rk[r] = inv;
        s_e[r] *= inv;
        s_bg[r] *= inv;
        ws.gv(slot, hv, p.Hv)[68 + r] = s_e[r];
      } else {
        s_rq[r] = inv;
        ws.gv(slot, hv, p.Hv)[4 + r] = s_gam[r] * inv;
      }
    }
    __syncthreads();
  }
  if (tid == 0 && !*s_abort) {
    constexpr uint32_t idg = idesc_f16(128, 64, true, false, false);
#pragma unroll
    for (int s = 0; s < DK / 16; ++s) {
      const uint32_t a = sbase + (s >> 2) * 16384 + (s & 3) * 32;
      tc_mma(tmem, sw128_desc(a, 16, 1024), sw128_desc(a, 16, 1024), idg, s > 0);
    }
    tc_commit(bar_mma);
  }
  // meanwhile: the scaled copy Kt = diag(e) K
  {
    __half* Kt = ws.Kt(slot, hv, p.Hv);
    constexpr int kRowChunks = DK / 8;
    for (int i = tid; i < kC * kRowChunks; i += kThreads) {
      const int r = i / kRowChunks, ch = i % kRowChunks;
      const unsigned char* src = sm + (ch >> 3) * 16384 + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
      *reinterpret_cast<uint4*>(Kt + swzb<kC>(r, ch * 8)) = scale_bf16x8_to_f16(src, s_e[r]);
    }
    {  // the output's left factor diag(scale gamma) Q (norm folded in), fp16
      __half* Qt = ws.Qt(slot, hv, p.Hv);
      for (int i = tid; i < kC * kRowChunks; i += kThreads) {
        const int r = i / kRowChunks, ch = i % kRowChunks;
        const unsigned char* src =
            sm + (ch >> 3) * 16384 + 8192 + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
        *reinterpret_cast<uint4*>(Qt + swzb<kC>(r, ch * 8)) =
            scale_bf16x8_to_f16(src, p.scale * s_gam[r] * s_rq[r]);
      }
    }
  }
  GDN_STAMP(33, 0);  // Kt written (thread 0's share)
  if (tid == 0 && !*s_abort && !mbar_wait(bar_mma, 0, p.err)) *s_abort = 1;
  __syncthreads();  // grams landed: the Q rows are free for Ah and Th
  if (!*s_abort) mbar_wait(bar_mma, 0, p.err);
  tc_fence_after();
  GDN_PHASE(1);  // grams + Kt

  // ---- masks: A (fp16 + fp32 diagonal blocks) and P, from the grams ---------
  if (!*s_abort) {
    const int q4 = warp & 3, h = warp >> 2;
    const int R = 32 * q4 + lane;  // gram row: 0-63 K K^T, 64-127 Q K^T
    const bool isP = R >= kC;
    const int r = R & (kC - 1), c0 = 32 * h;
    float x[32];
    tmem_ld32(tmem + ((uint32_t)(32 * q4) << 16) + c0, x);
    const float rowf = isP ? p.scale * s_rq[r] : s_beta[r] * s_rk[r];
    // last column kept; without the erase term (SSD) A is zero, so Tm = I and U = diag(beta) V
    const int lim = isP ? r : (p.delta_rule ? r - 1 : -1);
    if (p.prologue) mask_row32<true>(x, s_G, s_rk, c0, s_G[r], rowf, lim, r < L);
    else mask_row32<false>(x, s_G, nullptr, c0, s_G[r], rowf, lim, r < L);
    if (isP) {
      __half* P = ws.P(slot, hv, p.Hv);
#pragma unroll
      for (int m = 0; m < 4; ++m)
        *reinterpret_cast<uint4*>(P + swz<kC>(r, c0 + 8 * m)) = pack8_f16(x + 8 * m);
    } else {
#pragma unroll
      for (int m = 0; m < 4; ++m)
        *reinterpret_cast<uint4*>(Ah + swz<kC>(r, c0 + 8 * m)) = pack8_f16(x + 8 * m);
      const int b = r >> 4;  // diagonal block of this row, kept in fp32 for the substitution
      if ((b >> 1) == h) {
        float4* dst = reinterpret_cast<float4*>(Ad + b * 256 + (r & 15) * 16);
        const bool hi = b & 1;  // columns 16-31 of this half (selects keep indices static)
#pragma unroll
        for (int m = 0; m < 4; ++m)
          dst[m] = make_float4(hi ? x[16 + 4 * m] : x[4 * m], hi ? x[17 + 4 * m] : x[4 * m + 1],
                               hi ? x[18 + 4 * m] : x[4 * m + 2], hi ? x[19 + 4 * m] : x[4 * m + 3]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  GDN_PHASE(2);  // masks

  // ---- #3 Solve: Tm = (I + A)^-1, written as Th (fp16), Tw and Tu ------------
  // Diagonal 16x16 blocks in fp32 (warp b, lane l = column l of block b), by
  // right-looking substitution: once x_m is final it updates every x_i, i > m,
  // so the dependent chain is 15 FMAs deep.  Warps 4-7 zero the strictly upper
  // blocks meanwhile.  Without the erase term (SSD) A = 0: Tm = I, so only
  // Tu = diag(beta) is needed (W is zero and never formed).
  const bool delta = p.delta_rule != 0;  // uniform over the grid
  if (!*s_abort && !delta) {
    for (int e = tid; e < kC * 8; e += kThreads) {  // 16-byte chunks of Tu, diagonal inside
      const int rr = e >> 3, ch = e & 7;
      __align__(16) __half z[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) z[i] = __float2half_rn(rr == 8 * ch + i ? s_beta[rr] : 0.f);
      *reinterpret_cast<uint4*>(&Tu[sw128(rr, 8 * ch)]) = *reinterpret_cast<const uint4*>(z);
    }
  }
  if (!*s_abort && delta) {
    if (warp < 4) {
      if (lane < 16) {
        const int b = warp, l = lane;
        const float* Ab = Ad + b * 256;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = (i == l) ? 1.f : 0.f;
#pragma unroll
        for (int m = 0; m < 15; ++m)
#pragma unroll
          for (int i = m + 1; i < 16; ++i) x[i] = fmaf(-Ab[i * 16 + m], x[m], x[i]);
        const int cc = 16 * b + l;
        const float fw = s_bg[cc], fu = s_beta[cc];
        __nv_bfloat16* Twb = reinterpret_cast<__nv_bfloat16*>(Tw);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int rr = 16 * b + i;
          Th[swz<kC>(rr, cc)] = __float2half_rn(x[i]);
          Twb[sw128(rr, cc)] = __float2bfloat16_rn(x[i] * fw);
          Tu[sw128(rr, cc)] = __float2half_rn(x[i] * fu);
        }
      }
    } else {
      for (int e = tid - 128; e < kC * 8; e += 128) {  // 16-byte chunks of the upper blocks
        const int rr = e >> 3, ch = e & 7;
        if ((ch >> 1) > (rr >> 4)) {
          const uint4 z = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(&Th[swz<kC>(rr, 8 * ch)]) = z;
          *reinterpret_cast<uint4*>(&Tw[sw128(rr, 8 * ch)]) = z;
          *reinterpret_cast<uint4*>(&Tu[sw128(rr, 8 * ch)]) = z;
        }
      }
    }
  }
  __syncthreads();
  GDN_STAMP(34, 0);  // diagonal blocks done
  GDN_STAMP(40, 128);
  if (!*s_abort && delta) {
    if (warp < 2) {
      // level 1: T10 = -(T11 A10) T00 (warp 0), T32 = -(T33 A32) T22 (warp 1)
      {
        const int i0 = 16 + 32 * warp, j0 = 32 * warp;
        float y[2][4] = {}, t[2][4] = {};
        uint32_t a[4], b[4];
        load_a_sw<kC>(a, Th, i0, i0, lane);     // T_II
        load_b_kn_sw<kC>(b, Ah, j0, i0, lane);  // A_IJ as [k][n]
        mma_f16(y[0], a, b[0], b[1]);
        mma_f16(y[1], a, b[2], b[3]);
        c_to_a(a, y[0], y[1]);
        load_b_kn_sw<kC>(b, Th, j0, j0, lane);  // T_JJ as [k][n]
        mma_f16(t[0], a, b[0], b[1]);
        mma_f16(t[1], a, b[2], b[3]);
#pragma unroll
        for (int jn = 0; jn < 2; ++jn)
#pragma unroll
          for (int xh = 0; xh < 2; ++xh) {
            const int rr = i0 + gq + 8 * xh, cc = j0 + 8 * jn + 2 * tq;
            put_t2(Th, Tw, Tu, s_bg, s_beta, rr, cc, -t[jn][2 * xh], -t[jn][2 * xh + 1]);
          }
      }
      named_sync(1, 64);
      // level 2: rows 32..63 x columns 0..31 = -(T_BB A_BA) T_AA; warp w takes 16 rows
      {
        const int i0 = 32 + 16 * warp;
        float y[4][4] = {}, t[4][4] = {};
        uint32_t a[4], b[4];
        for (int k0 = 32; k0 <= i0; k0 += 16) {  // T_BB is lower triangular
          load_a_sw<kC>(a, Th, i0, k0, lane);
          load_b_kn_sw<kC>(b, Ah, 0, k0, lane);
          mma_f16(y[0], a, b[0], b[1]);
          mma_f16(y[1], a, b[2], b[3]);
          load_b_kn_sw<kC>(b, Ah, 16, k0, lane);
          mma_f16(y[2], a, b[0], b[1]);
          mma_f16(y[3], a, b[2], b[3]);
        }
#pragma unroll
        for (int s = 0; s < 2; ++s) {  // k over the 32 columns of Y
          c_to_a(a, y[2 * s], y[2 * s + 1]);
          load_b_kn_sw<kC>(b, Th, 0, 16 * s, lane);
          mma_f16(t[0], a, b[0], b[1]);
          mma_f16(t[1], a, b[2], b[3]);
          load_b_kn_sw<kC>(b, Th, 16, 16 * s, lane);
          mma_f16(t[2], a, b[0], b[1]);
          mma_f16(t[3], a, b[2], b[3]);
        }
#pragma unroll
        for (int jn = 0; jn < 4; ++jn)
#pragma unroll
          for (int xh = 0; xh < 2; ++xh) {
            const int rr = i0 + gq + 8 * xh, cc = 8 * jn + 2 * tq;
            put_t2(nullptr, Tw, Tu, s_bg, s_beta, rr, cc, -t[jn][2 * xh], -t[jn][2 * xh + 1]);
          }
      }
      GDN_STAMP(35, 0);  // merges done
    }
  }
  fence_proxy_async();  // Tw, Tu are read by the tensor cores; the Q rows take V next
  tc_fence_before();
  __syncthreads();  // the solve is done: Ah and Th are dead
  GDN_PHASE(3);  // solve

  // ---- #4 W^T = K^T Tw^T (bf16, tensor columns 64-127) while V lands in the Q
  // rows; then U^T = V^T Tu^T (fp16, columns 0-63) -------------------------------
  if (tid == 0 && !*s_abort) {
    if (Lo::kVinQ) {
      mbar_expect_tx(bar_v, (unsigned)kC * DV * 2);
#pragma unroll
      for (int vb = 0; vb < DV / 64; ++vb)
        tma_load_2d(sm + Lo::kV + vb * Lo::kVStride, &tmv, hv * DV + vb * 64, t0, bar_v);
    }
    if (delta) {
      tc_fence_after();
      constexpr uint32_t idw = idesc_f16(DK, 64, true, true, false);
#pragma unroll
      for (int s = 0; s < kC / 16; ++s)
        tc_mma(tmem + 64, sw128_desc(sbase + s * 2048, 16384, 1024),
               sw128_desc(sbase + Lo::kTw + s * 32, 16, 1024), idw, s > 0);
      tc_commit(bar_w);
    }
  }
  // tensor-memory lane -> d: lane d for M = 128; rows 16q + i sit in lanes 32q + i for M = 64
  const int q4 = warp & 3, h = warp >> 2;
  const uint32_t lane_base = tmem + ((uint32_t)(32 * q4) << 16);
  if (delta && tid == 0 && !*s_abort && !mbar_wait(bar_w, 0, p.err)) *s_abort = 1;
  if (delta) __syncthreads();
  if (!*s_abort && delta) {
    mbar_wait(bar_w, 0, p.err);
    tc_fence_after();
    float x[32];
    tmem_ld32(lane_base + 64 + 32 * h, x);
    if (DK == 128 || lane < 16) {
      const int d = DK == 128 ? 32 * q4 + lane : 16 * q4 + lane;
      __half* Wt = ws.W(slot, hv, p.Hv);  // [dk][64], swz<64>
#pragma unroll
      for (int m = 0; m < 4; ++m)
        *reinterpret_cast<uint4*>(Wt + swz<kC>(d, 32 * h + 8 * m)) = pack8_f16(x + 8 * m);
    }
  }
  GDN_STAMP(36, 0);  // W stored
  // V: zero its rows past the sequence end, rewrite it as fp16 for the U product
  if (tid == 0 && !*s_abort && !mbar_wait(bar_v, 0, p.err)) *s_abort = 1;
  __syncthreads();
  if (!*s_abort) {
    mbar_wait(bar_v, 0, p.err);
    for (int i = tid; i < (DV / 64) * kC * 8; i += kThreads) {
      const int ch = i & 7, rr = (i >> 3) & (kC - 1), vb = i >> 9;
      unsigned char* q = sm + Lo::kV + vb * Lo::kVStride + rr * 128 + ch * 16;
      if (rr >= L) *reinterpret_cast<uint4*>(q) = make_uint4(0, 0, 0, 0);
      else bf16x8_to_f16x8(q);
    }
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && !*s_abort) {
    tc_fence_after();
    constexpr uint32_t idu = idesc_f16(DV, 64, false, true, false);
#pragma unroll
    for (int s = 0; s < kC / 16; ++s)
      tc_mma(tmem, sw128_desc(sbase + Lo::kV + s * 2048, Lo::kVStride, 1024),
             sw128_desc(sbase + Lo::kTu + s * 32, 16, 1024), idu, s > 0);
    tc_commit(bar_u);
  }
  if (tid == 0 && !*s_abort && !mbar_wait(bar_u, 0, p.err)) *s_abort = 1;
  __syncthreads();
  if (!*s_abort) {
    mbar_wait(bar_u, 0, p.err);
    tc_fence_after();
    float x[32];
    tmem_ld32(lane_base + 32 * h, x);
    if (DV == 128 || lane < 16) {
      const int d = DV == 128 ? 32 * q4 + lane : 16 * q4 + lane;
      __half* Ut = ws.U(slot, hv, p.Hv);  // [dv][64], plain
#pragma unroll
      for (int m = 0; m < 4; ++m)
        *reinterpret_cast<uint4*>(Ut + swz<kC>(d, 32 * h + 8 * m)) = pack8_f16(x + 8 * m);
    }
  }
  GDN_PHASE(4);  // W/U
  GDN_STAMP(37, 0);  // W, U stored
  // ---- teardown: after an expired wait, let copies in flight land first ------
  if (*s_abort && tid == 0) {  // bounded: a copy never issued just times out
    mbar_wait(bar_kq, 0, nullptr);
    mbar_wait(bar_v, 0, nullptr);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 128);
}

// ---- host: tensor maps -------------------------------------------------------
using EncodeTiled = PFN_cuTensorMapEncodeTiled_v12000;

EncodeTiled encode_fn() {
  static const EncodeTiled fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<EncodeTiled>(f);
  }();
  return fn;
}

}  // namespace

bool make_tensor_map_bf16(CUtensorMap* m, const void* base, long long rows, long long cols) {
  EncodeTiled fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {64, 64};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tensor_map_bf16_3d(CUtensorMap* m, const void* base, long long planes, long long rows,
                             long long cols) {
  EncodeTiled fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)planes};
  const cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)(cols * rows * 2)};
  const cuuint32_t box[3] = {64, 64, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

template <int DK, int DV>
cudaError_t launch_t(const FwdParams& p, const WsLayout& ws, cudaStream_t stream) {
  using Lo = PrepLayout<DK, DV>;
  const long long rows = p.cu_seqlens ? (long long)p.T : (long long)p.N * p.T;
  CUtensorMap mq, mk, mv;
  if (!make_tensor_map_bf16(&mq, p.q, rows, (long long)p.Hqk * DK) ||
      !make_tensor_map_bf16(&mk, p.k, rows, (long long)p.Hqk * DK) ||
      !make_tensor_map_bf16(&mv, p.v, rows, (long long)p.Hv * DV))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(gdn_prep_kernel<DK, DV>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, Lo::kAlloc);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gdn_prep_kernel<DK, DV>,
                             cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  const long long grid = ws.n_slots * p.Hv;
  gdn_prep_kernel<DK, DV><<<(unsigned)grid, kThreads, Lo::kAlloc, stream>>>(p, ws, mq, mk, mv);
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
