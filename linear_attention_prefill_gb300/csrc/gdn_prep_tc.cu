// gdn_prep_tc.cu - the chunk-parallel Map phase for the tensor-memory chain (lookahead records).
//
// "Empowering Hybrid Attention Models on NPUs", §2.1, Figure 1(b): operators
// #1-#4 (Gate, KKT, Solve, W/U) depend only on one chunk's q, k, v, g, beta,
// so every (chunk, v head) is an independent task here:
//   #1 Gate   G = cumsum(g), gamma = exp(G), e_j = exp(G_last - G_j)
//   #2 KKT    A = tril_strict(beta_i exp(G_i - G_j) k_i.k_j)
//      QK^T   P = tril(scale exp(G_i - G_j) q_i.k_j)
//   #3 Solve  Tm = (I + A)^-1   (diagonal blocks by substitution, merges on mma.sync)
//   #4 W/U    W = Tm diag(beta gamma) K,  U = Tm diag(beta) V
// plus what the chain's one-chunk lookahead needs from the previous chunk c - 1
// of the same sequence (its keys and gates, re-read here rather than passed
// between tasks): W'(c) = gamma_last(c-1) W(c) and X(c) = W(c) Kt(c-1)^T, so
// that the chain can form V_new(c) = U(c) - W'(c) h(c-1) - X(c) V_new(c-1)
// while the state entering chunk c is still being produced.  The scaled copies
// Kt = diag(e) K (the state update's factor) and Q~ = diag(scale gamma) Q (the
// output's) complete the record (layout in gdn_internal.h).  The serial Reduce
// (#5) and the final Map (#6) run in gdn_chain_tc.cu.
//
// Blackwell mapping.  K and Q arrive by TMA in 128-byte-swizzled tiles stacked
// as one 128-row operand [K; Q], so a single M = 128 tcgen05 MMA chain gives
// both grams (K K^T in tensor-memory lanes 0-63, Q K^T in lanes 64-127); the
// same launch forms Y = K(c-1) K(c)^T (M = 64).  The K tile read MN-major is the
// left factor of W^T = K^T (Tm diag(beta gamma))^T (one d index per lane), Y
// that of X^T = Y (Tm diag(beta gamma))^T, and V (loaded into the Q rows once
// Q is consumed) that of U^T.  W and P leave transposed from tensor memory: each
// pair of neighbouring lanes swaps one value so that both store 4-byte pairs of
// the record's row-major tile.  Accumulators stay in 128 tensor-memory columns
// and shared memory in ~67 KB, so three tasks share an SM.
//
// Precision: products accumulate in fp32.  The grams, Y, W and X take bf16
// operands (the inputs as they are; Tm diag(beta gamma) and Y rounded to bf16);
// U takes fp16 operands (v rewritten in place, exact in fp16's normal range).
#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

constexpr int kC = 64;
constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;

// Shared-memory map (byte offsets from a 1024-aligned base), ~67 KB at d = 128
// so that three tasks share an SM.  The Q rows are reused twice: once the grams
// have read Q they hold the solve's fp16 copies Ah and Th, and once the solve is
// done they take V.  The previous chunk's K tile is read only by the Y product;
// its space then holds Y (bf16, X's left factor) and A's fp32 diagonal blocks.
template <int DK, int DV>
struct PrepLayout {
  // [DK/64][128 rows][64] bf16, 128-byte swizzle: rows 0-63 K, rows 64-127 Q
  static constexpr int kKQBytes = (DK / 64) * 16384;
  static constexpr int kPrev = kKQBytes;  // K(c-1) [DK/64][64][64] bf16, then Y, Ad
  static constexpr int kY = kPrev;                                // bf16 [64][64] sw128
  static constexpr int kAd = kPrev + 8192;  // fp32 diagonal blocks of A [4][16][16]
  static constexpr int kPrevBytes = DK == 128 ? 16384 : 12288;
  static constexpr int kAfterPrev = kPrev + kPrevBytes;
  static constexpr bool kThInQ = DK == 128;             // Th in the second block's Q rows
  static constexpr bool kVinQ = DV <= DK;               // V in the Q rows after the solve
  static constexpr int kAh = 8192;                      // fp16 [64][64] swz<64>, first Q rows
  static constexpr int kTh = kThInQ ? 24576 : kAfterPrev;  // fp16 [64][64] swz<64>
  static constexpr int kAfterTh = kAfterPrev + (kThInQ ? 0 : 8192);
  static constexpr int kV = kVinQ ? 8192 : kAfterTh;
  static constexpr int kVStride = kVinQ ? 16384 : 8192;  // bytes between 64-column blocks
  static constexpr int kTw = kAfterTh + (kVinQ ? 0 : (DV / 64) * 8192);  // bf16 [64][64] sw128
  static constexpr int kTu = kTw + 8192;                                   // fp16 [64][64] sw128
  // beta, G, gamma, e, beta*gamma, 1/|k|, 1/|q|, e(c-1)
  static constexpr int kVec = kTu + 8192;
  static constexpr int kBar = kVec + 8 * kC * 4;  // 7 mbarriers, tmem address, flags
  static constexpr int kBytes = kBar + 128;
  static constexpr int kAlloc = kBytes + 1024;  // slack to align the base
  static_assert(kTw % 1024 == 0 && kTh % 1024 == 0 && kY % 1024 == 0 && kAd % 16 == 0 &&
                kVec % 16 == 0,
                "alignment");
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
__device__ __forceinline__ uint4 pack8_bf16(const float* x) {
  return make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]),
                    pack_bf16(x[6], x[7]));
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

// Transposed store of a tensor-memory row block.  This thread holds x[m] =
// M[row][col0 + m] (m < 32) of a matrix whose rows sit in consecutive lanes; the
// record tile is its transpose, Mt[col][row], at `dst` (element offset `off(r, c)`
// of (row r, column c) of Mt).  Lanes row and row ^ 1 trade one value per column
// pair, so that each stores 4-byte pairs: the even lane (col, row..row + 1), the
// odd lane (col + 1, row - 1..row).  `active` is false on lanes that hold no row
// (their values are not stored, but they still take part in the shuffles).
template <typename Off>
__device__ __forceinline__ void store_transposed(__half* dst, const float (&x)[32], int row,
                                                 int col0, float scale, bool active, Off off) {
  const bool odd = row & 1;
#pragma unroll
  for (int m = 0; m < 32; m += 2) {
    const float a0 = x[m] * scale, a1 = x[m + 1] * scale;
    const float b0 = __shfl_xor_sync(0xffffffffu, a0, 1);
    const float b1 = __shfl_xor_sync(0xffffffffu, a1, 1);
    if (active) {
      if (!odd)
        *reinterpret_cast<uint32_t*>(dst + off(col0 + m, row)) = pack_f16(a0, b0);
      else
        *reinterpret_cast<uint32_t*>(dst + off(col0 + m + 1, row - 1)) = pack_f16(b1, a1);
    }
  }
}

// Log-decay of one token and v head from the stored gate: g itself, or with the
// fused prologue -exp(A_log) softplus(a + dt_bias) of the raw gate a.
__device__ __forceinline__ float decay_of(const FwdParams& p, float raw, float amul, float abias) {
  if (!p.prologue) return raw;
  const float x = raw + abias;
  return -amul * (x > 20.f ? x : log1pf(expf(x)));
}

template <int DK, int DV>
__global__ void __launch_bounds__(kThreads, 3)
    gdn_prep_tc_kernel(const FwdParams p, const WsLayout ws, const __grid_constant__ CUtensorMap tmq,
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
  float* s_rk = s_bg + kC;   // 1/|k_r| with the fused prologue, else 1
  float* s_rq = s_rk + kC;   // 1/|q_r| likewise
  float* s_ep = s_rq + kC;   // e_s(c-1) = exp(G_last(c-1) - G_s(c-1)) (norm folded in)
  uint64_t* bar_kq = reinterpret_cast<uint64_t*>(sm + Lo::kBar);
  uint64_t* bar_v = bar_kq + 1;
  uint64_t* bar_mma = bar_kq + 2;  // grams and Y
  uint64_t* bar_w = bar_kq + 3;    // W^T and X^T products
  uint64_t* bar_u = bar_kq + 4;    // U^T product
  uint64_t* bar_kp = bar_kq + 5;   // K(c-1)
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bar_kq + 6);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  float* s_glp = reinterpret_cast<float*>(s_tmem + 2);  // gamma_last(c-1) (1 for chunk 0)

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
  const bool delta = p.delta_rule != 0;  // uniform over the grid
  const bool prev = delta && c > 0;      // the lookahead terms of chunk c - 1 exist
  const float amul = (p.prologue && p.A_log) ? expf(p.A_log[hv]) : 1.f;
  const float abias = (p.prologue && p.dt_bias) ? p.dt_bias[hv] : 0.f;

  // ---- setup: barriers, the K/Q (K(c-1), and a separate V) loads, tensor memory
  if (tid == 0) {
    mbar_init(bar_kq, 1);
    mbar_init(bar_v, 1);
    mbar_init(bar_mma, 1);
    mbar_init(bar_w, 1);
    mbar_init(bar_u, 1);
    mbar_init(bar_kp, 1);
    *s_abort = 0;
    mbar_fence_init();
    mbar_expect_tx(bar_kq, 2u * kC * DK * 2);
#pragma unroll
    for (int kb = 0; kb < DK / 64; ++kb) {
      tma_load_2d(sm + kb * 16384, &tmk, hq * DK + kb * 64, t0, bar_kq);
      tma_load_2d(sm + kb * 16384 + 8192, &tmq, hq * DK + kb * 64, t0, bar_kq);
    }
    if (prev) {  // the previous chunk is whole: only a sequence's last chunk is ragged
      mbar_expect_tx(bar_kp, (unsigned)kC * DK * 2);
#pragma unroll
      for (int kb = 0; kb < DK / 64; ++kb)
        tma_load_2d(sm + Lo::kPrev + kb * 8192, &tmk, hq * DK + kb * 64, t0 - kC, bar_kp);
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
    float g0 = r0 < L ? decay_of(p, gp[(long long)r0 * p.Hv], amul, abias) : 0.f;
    float g1 = r1 < L ? decay_of(p, gp[(long long)r1 * p.Hv], amul, abias) : 0.f;
    float b0 = r0 < L ? bp[(long long)r0 * p.Hv] : 0.f;
    float b1 = r1 < L ? bp[(long long)r1 * p.Hv] : 0.f;
    if (p.prologue) {  // raw beta: sigmoid(b)
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
    s_bg[r0] = delta ? b0 * gam0 : 0.f;  // W's column factor: 0 without the erase
    s_bg[r1] = delta ? b1 * gam1 : 0.f;
    s_rk[r0] = s_rk[r1] = s_rq[r0] = s_rq[r1] = 1.f;
    float* gv = ws.gv(slot, hv, p.Hv);  // gamma_last, then gamma of every row
    if (lane == 31) gv[0] = expf(Glast);
    if (!p.prologue) {
      *reinterpret_cast<float2*>(gv + 4 + r0) = make_float2(gam0, gam1);
      *reinterpret_cast<float2*>(gv + 68 + r0) = make_float2(s_e[r0], s_e[r1]);
    }
  } else if (warp == 2 && !prev) {
    if (lane == 0) *s_glp = 1.f;
  } else if (warp == 2) {
    // the previous chunk's gates: e_s(c-1) and gamma_last(c-1)
    const int r0 = 2 * lane, r1 = 2 * lane + 1;
    const float* gp = p.g + (long long)(t0 - kC) * p.Hv + hv;
    const float g0 = decay_of(p, gp[(long long)r0 * p.Hv], amul, abias);
    const float g1 = decay_of(p, gp[(long long)r1 * p.Hv], amul, abias);
    float incl = g0 + g1;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    const float Glast = __shfl_sync(0xffffffffu, incl, 31);
    s_ep[r0] = expf(Glast - (incl - g1));
    s_ep[r1] = expf(Glast - incl);
    if (lane == 0) *s_glp = expf(Glast);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  GDN_PHASE(0);  // setup + gate

  // ---- #2 grams: one M = 128 MMA chain, [K; Q] K^T -> tensor columns 0-63, and
  // Y = K(c-1) K^T (M = 64) -> columns 64-127.  One thread spins on each barrier;
  // the others block in bar.sync and then observe the completed phase with one test.
  if (tid == 0 && !mbar_wait(bar_kq, 0, p.err)) *s_abort = 1;
  if (tid == 0 && prev && !*s_abort && !mbar_wait(bar_kp, 0, p.err)) *s_abort = 1;
  __syncthreads();
  if (!*s_abort) {
    mbar_wait(bar_kq, 0, p.err);
    if (prev) mbar_wait(bar_kp, 0, p.err);
  }
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
    // Kt's row factor e, W's column factor beta gamma, the gamma the output stage
    // multiplies q rows by, and X's row factor e(c-1) for the previous chunk's keys
    for (int pass = 0; pass < (prev ? 2 : 1); ++pass) {
      const int R = tid >> 1, half = tid & 1;  // pass 0: R < 64 k row, else q row R - 64
      if (pass == 1 && R >= kC) break;         // pass 1: the 64 rows of K(c-1)
      const int r = R & (kC - 1);
      float ss = 0.f;
      for (int ch = half * (DK / 16); ch < (half + 1) * (DK / 16); ++ch) {
        const unsigned char* src =
            pass == 0 ? sm + (ch >> 3) * 16384 + (R >= kC ? 8192 : 0) + r * 128
                      : sm + Lo::kPrev + (ch >> 3) * 8192 + r * 128;
        const uint4 raw = *reinterpret_cast<const uint4*>(src + (((ch & 7) ^ (r & 7)) << 4));
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
        if (pass == 1) {
          s_ep[r] *= inv;
        } else if (R < kC) {
          s_rk[r] = inv;
          s_e[r] *= inv;
          s_bg[r] *= inv;
          ws.gv(slot, hv, p.Hv)[68 + r] = s_e[r];
        } else {
          s_rq[r] = inv;
          ws.gv(slot, hv, p.Hv)[4 + r] = s_gam[r] * inv;
        }
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
    if (prev) {
      constexpr uint32_t idy = idesc_f16(64, 64, true, false, false);
#pragma unroll
      for (int s = 0; s < DK / 16; ++s)
        tc_mma(tmem + 64, sw128_desc(sbase + Lo::kPrev + (s >> 2) * 8192 + (s & 3) * 32, 16, 1024),
               sw128_desc(sbase + (s >> 2) * 16384 + (s & 3) * 32, 16, 1024), idy, s > 0);
    }
    tc_commit(bar_mma);
  }
  // meanwhile: the scaled copies Kt = diag(e) K and Q~ = diag(scale gamma) Q (fp16)
  {
    __half* Kt = ws.Kt(slot, hv, p.Hv);
    __half* Qt = ws.Qt(slot, hv, p.Hv);
    constexpr int kRowChunks = DK / 8;
    for (int i = tid; i < 2 * kC * kRowChunks; i += kThreads) {
      const int isq = i >= kC * kRowChunks;
      const int j = i - isq * kC * kRowChunks;
      const int r = j / kRowChunks, ch = j % kRowChunks;
      const unsigned char* src =
          sm + (ch >> 3) * 16384 + isq * 8192 + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
      const float f = isq ? p.scale * s_gam[r] * s_rq[r] : s_e[r];
      *reinterpret_cast<uint4*>((isq ? Qt : Kt) + swzb<kC>(r, ch * 8)) = scale_bf16x8_to_f16(src, f);
    }
  }
  GDN_STAMP(33, 0);  // Kt written (thread 0's share)
  if (tid == 0 && !*s_abort && !mbar_wait(bar_mma, 0, p.err)) *s_abort = 1;
  __syncthreads();  // grams landed: the Q rows are free for Ah and Th
  if (!*s_abort) mbar_wait(bar_mma, 0, p.err);
  tc_fence_after();
  GDN_PHASE(1);  // grams + Kt

  // ---- masks: A (fp16 + fp32 diagonal blocks) and P^T, from the grams; Y -> bf16
  if (!*s_abort) {
    const int q4 = warp & 3, h = warp >> 2;
    const int R = 32 * q4 + lane;  // gram row: 0-63 K K^T, 64-127 Q K^T
    const bool isP = R >= kC;
    const int r = R & (kC - 1), c0 = 32 * h;
    float x[32];
    tmem_ld32(tmem + ((uint32_t)(32 * q4) << 16) + c0, x);
    const float rowf = isP ? p.scale * s_rq[r] : s_beta[r] * s_rk[r];
    // last column kept; without the erase term (SSD) A is zero, so Tm = I and U = diag(beta) V
    const int lim = isP ? r : (delta ? r - 1 : -1);
    if (p.prologue) mask_row32<true>(x, s_G, s_rk, c0, s_G[r], rowf, lim, r < L);
    else mask_row32<false>(x, s_G, nullptr, c0, s_G[r], rowf, lim, r < L);
    if (isP) {  // q4 = 2, 3: lanes hold P rows r = R - 64; the record holds P^T
      store_transposed(ws.P(slot, hv, p.Hv), x, r, c0, 1.f, true,
                       [](int rr, int cc) { return swz<kC>(rr, cc); });
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
    if (prev) {  // Y (M = 64: row s = 16 q4 + i in lane 32 q4 + i) -> bf16 over K(c-1)
      float y[32];
      tmem_ld32(tmem + ((uint32_t)(32 * q4) << 16) + 64 + c0, y);
      if (lane < 16) {
        const int s = 16 * q4 + lane;
        __half* Y = reinterpret_cast<__half*>(sm + Lo::kY);
#pragma unroll
        for (int m = 0; m < 4; ++m)
          *reinterpret_cast<uint4*>(Y + sw128(s, c0 + 8 * m)) = pack8_bf16(y + 8 * m);
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
  fence_proxy_async();  // Tw, Tu, Y are read by the tensor cores; the Q rows take V next
  tc_fence_before();
  __syncthreads();  // the solve is done: Ah and Th are dead
  GDN_PHASE(3);  // solve

  // ---- #4 W^T = K^T Tw^T (columns 64-127) and X^T = Y Tw^T (columns 0-63) while V
  // lands in the Q rows; then U^T = V^T Tu^T (fp16, columns 0-63) -------------------
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
      if (prev) {
        constexpr uint32_t idx = idesc_f16(64, 64, true, false, false);
#pragma unroll
        for (int s = 0; s < kC / 16; ++s)
          tc_mma(tmem, sw128_desc(sbase + Lo::kY + s * 32, 16, 1024),
                 sw128_desc(sbase + Lo::kTw + s * 32, 16, 1024), idx, s > 0);
      }
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
    // W'(c) = gamma_last(c-1) W(c), stored [64][dk] (row t, column d)
    const int d = DK == 128 ? 32 * q4 + lane : 16 * q4 + lane;
    store_transposed(ws.W(slot, hv, p.Hv), x, d, 32 * h, *s_glp, DK == 128 || lane < 16,
                     [](int rr, int cc) { return swzb<kC>(rr, cc); });
    if (prev) {  // X^T[s][t] = e_s(c-1) (Y Tw^T)[s][t], M = 64: row s = 16 q4 + i
      float xt[32];
      tmem_ld32(lane_base + 32 * h, xt);
      if (lane < 16) {
        const int s = 16 * q4 + lane;
        const float f = s_ep[s];
#pragma unroll
        for (int j = 0; j < 32; ++j) xt[j] *= f;
        __half* Xt = ws.Xt(slot, hv, p.Hv);
#pragma unroll
        for (int m = 0; m < 4; ++m)
          *reinterpret_cast<uint4*>(Xt + swz<kC>(s, 32 * h + 8 * m)) = pack8_f16(xt + 8 * m);
      }
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
  __syncthreads();  // also: X^T has been read out of columns 0-63
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
      __half* Ut = ws.U(slot, hv, p.Hv);  // [dv][64]
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
    if (prev) mbar_wait(bar_kp, 0, nullptr);
    mbar_wait(bar_v, 0, nullptr);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 128);
}

}  // namespace

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
  cudaError_t e = cudaFuncSetAttribute(gdn_prep_tc_kernel<DK, DV>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, Lo::kAlloc);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gdn_prep_tc_kernel<DK, DV>,
                             cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  const long long grid = ws.n_slots * p.Hv;
  gdn_prep_tc_kernel<DK, DV><<<(unsigned)grid, kThreads, Lo::kAlloc, stream>>>(p, ws, mq, mk, mv);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prep_tc(const FwdParams& p, const WsLayout& ws, cudaStream_t stream) {
  if (p.dk == 128) {
    if (p.dv == 128) return launch_t<128, 128>(p, ws, stream);
    return launch_t<128, 64>(p, ws, stream);
  }
  if (p.dv == 128) return launch_t<64, 128>(p, ws, stream);
  return launch_t<64, 64>(p, ws, stream);
}

}  // namespace gdn
