// gdn_chain.cu - the serial Reduce (#5 H) and the final Map (#6 O) of the
// chunkwise forward ("Empowering Hybrid Attention Models on NPUs", §2.1,
// Figure 1(b)), the state update split as in §5 (Figure 10(b)) into the state
// read and the in-place update:
//   #5 read    V_new = U - W h
//   #5 update  h = gamma_last h + Kt^T V_new        (Kt = diag(e) K)
//   #6 O       O = Q~ h + P V_new  (Q~ = diag(scale gamma) Q; h: the state entering the chunk)
// One CTA per (sequence, v head, dv tile) walks the chunks of its sequence in
// order with its fp32 state tile h[:, tile] in registers: the column split of
// the state (§4, Figure 8(b)) gives parallelism without any reduction.
//
// Warp roles.  Warps 0-3 run the chain: two warp-level fp16 tensor-core
// products per chunk (mma.sync, the state as accumulator) and two CTA-local
// barriers - nothing else sits on the serial path.  They leave the state
// entering each chunk (fp16) and V_new in a 3-deep shared-memory ring, from
// which warps 4-7 compute that chunk's output tile one or two chunks behind,
// so neither ever travels through HBM.  Warp 8 is the producer: it stages W^T,
// Kt, P, the U^T tile, the gate factors and Q~ of chunk c + 3 with bulk copies
// into a 3-deep ring.  The roles meet only at mbarriers; every wait is bounded
// and an expired wait ends the CTA cleanly.
//
// Precision: every product takes fp16 operands with fp32 accumulation.  Q~ is
// formed by the prep kernel (scale gamma_i, and the norm with the fused
// prologue, applied to the bf16 q rows and rounded once to fp16), so the output
// warps feed it to the tensor cores as it is.
//
// KDA mode (Kimi Delta Attention, the per-channel gate; records from
// kda_prep.cu): the decay of the state update is one factor per state row,
// h <- diag(exp G_last) h + Kt^T V_new, and Q~ = scale Q * exp(G) carries the
// per-channel decay.
#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

constexpr int kC = 64;
constexpr int kComputeThreads = 128;  // warps 0-3: the chain
constexpr int kOutWarp0 = 4;          // warps 4-7: the output
constexpr int kProducerWarp = 8;
constexpr int kThreads = 288;
constexpr int kStages = 3;
constexpr int kPub = 3;  // state / V_new buffers shared with the output warps

// Shared-memory map (byte offsets from a 1024-aligned base).  NOW: a run without
// the erase term (Mamba-2 SSD), whose stages carry no W tile.
template <int DK, int DVT, bool NOW = false>
struct ChainLayout {
  // one stage: the record's Q~ rows (fp16, swzb<64>: [DK/64][64][64], the
  // 128-byte swizzle) first, then the other record pieces
  static constexpr int kQ = 0;
  static constexpr int kWt = kQ + kC * DK * 2;   // W^T [DK][64] swz<64>
  static constexpr int kKt = kWt + (NOW ? 0 : kC * DK * 2);  // Kt [64][DK] swzb<64>
  static constexpr int kP = kKt + kC * DK * 2;   // P [64][64] swz<64>
  static constexpr int kUt = kP + kC * kC * 2;   // U^T [DVT][64] swz<64>
  static constexpr int kGv = kUt + DVT * kC * 2; // gamma_last, pad, gamma[64], e[64]
  static constexpr int kStageBytes = (kGv + kGvFloats * 4 + 1023) / 1024 * 1024;
  static constexpr int kH = kStages * kStageBytes;      // [kPub][DK][DVT] fp16 swz<DVT>
  static constexpr int kVn = kH + kPub * DK * DVT * 2;  // [kPub][64][DVT] fp16 swz<DVT>
  static constexpr int kBar = kVn + kPub * kC * DVT * 2;
  static constexpr int kBytes = kBar + 8 * (2 * kStages + 2 * kPub) + 16;
  static constexpr int kAlloc = kBytes + 1024;  // slack to align the base
  static constexpr unsigned kTx =
      (NOW ? 2 : 3) * kC * DK * 2 + kC * kC * 2 + DVT * kC * 2 + kGvFloats * 4;
};

// A fragment (16x16) of a bf16 tile in the 128-byte-swizzled [k/64][rows][64] layout.
__device__ __forceinline__ void load_a_sw128(uint32_t (&a)[4], const unsigned char* base, int m0,
                                             int k0, int lane) {
  const int r = m0 + (lane & 15), k = k0 + ((lane >> 4) << 3);
  ldsm_x4(a[0], a[1], a[2], a[3],
          base + (k >> 6) * 8192 + r * 128 + ((((k & 63) >> 3) ^ (r & 7)) << 4));
}

template <int DK, int DVT, bool KDA, bool NOW = false>
__global__ void __launch_bounds__(kThreads, 1)
    gdn_chain_kernel(const FwdParams p, const WsLayout ws) {
  using Lo = ChainLayout<DK, DVT, NOW>;
  const bool delta = !NOW && p.delta_rule;  // the erase term (W) takes part
  constexpr int NT = DVT / 8;          // n8 tiles over the dv tile
  constexpr int MTW = DK / 64;         // m16 tiles of the state per chain warp
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __half* Hring = reinterpret_cast<__half*>(sm + Lo::kH);
  __half* Vring = reinterpret_cast<__half*>(sm + Lo::kVn);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + Lo::kBar);  // producer -> consumers
  uint64_t* empty = full + kStages;  // 4 chain + 4 output warp arrivals: stage consumed
  uint64_t* pub = empty + kStages;   // chain -> output: H[b], Vn[b] ready
  uint64_t* pubd = pub + kPub;       // output -> chain: H[b], Vn[b] consumed (4 arrivals)
  volatile int* s_abort = reinterpret_cast<volatile int*>(pubd + kPub);  // any wait expired
  // the chain warps' stop decision: written by thread 0 before a named barrier and
  // read by all four warps after it, so they never split at a barrier
  volatile int* s_cstop = s_abort + 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;

  GDN_PHASE_INIT;
  const int n_dvt = p.dv / DVT;
  const int dvt = blockIdx.x % n_dvt;
  const int hv = (blockIdx.x / n_dvt) % p.Hv;
  const int n = blockIdx.x / (n_dvt * p.Hv);
  const long long t_seq = p.cu_seqlens ? (long long)p.cu_seqlens[n] : (long long)n * p.T;
  const long long len = p.cu_seqlens ? (long long)p.cu_seqlens[n + 1] - t_seq : (long long)p.T;
  const int n_chunks = (int)((len + kC - 1) / kC);
  const long long slot0 = ws.first_slot(p, n);

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 8);
    }
    for (int i = 0; i < kPub; ++i) {
      mbar_init(&pub[i], 1);
      mbar_init(&pubd[i], 4);
    }
    *s_abort = 0;
    *s_cstop = 0;
    mbar_fence_init();
  }

  // ---- initial state (chain warps) --------------------------------------------
  float hacc[MTW][NT][4];
  if (warp < 4) {
    const float* h0 =
        p.h0 ? p.h0 + ((long long)(n * p.Hv + hv) * DK) * p.dv + dvt * DVT : nullptr;
#pragma unroll
    for (int mt = 0; mt < MTW; ++mt)
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int r0 = 16 * (MTW * warp + mt) + gq, col = 8 * j + 2 * tq;
        float2 a = make_float2(0.f, 0.f), b = make_float2(0.f, 0.f);
        if (h0) {
          a = *reinterpret_cast<const float2*>(h0 + (long long)r0 * p.dv + col);
          b = *reinterpret_cast<const float2*>(h0 + (long long)(r0 + 8) * p.dv + col);
        }
        hacc[mt][j][0] = a.x; hacc[mt][j][1] = a.y; hacc[mt][j][2] = b.x; hacc[mt][j][3] = b.y;
        *reinterpret_cast<uint32_t*>(&Hring[swz<DVT>(r0, col)]) = pack_f16(a.x, a.y);
        *reinterpret_cast<uint32_t*>(&Hring[swz<DVT>(r0 + 8, col)]) = pack_f16(b.x, b.y);
      }
  }
  __syncthreads();  // barriers initialised, H[0] written

  if (warp == kProducerWarp) {
    // ======================= producer ======================================
    if (lane == 0) {
      griddep_wait();  // the records are the prep launch's output
      auto issue = [&](int c) {
        unsigned char* st = sm + (c % kStages) * Lo::kStageBytes;
        uint64_t* bar = &full[c % kStages];
        const long long slot = slot0 + c;
        // without the erase term (SSD) W is zero: it is neither formed nor loaded
        mbar_expect_tx(bar, (delta || NOW) ? Lo::kTx : Lo::kTx - kC * DK * 2);
        if (delta) bulk_g2s(st + Lo::kWt, ws.W(slot, hv, p.Hv), kC * DK * 2, bar);
        bulk_g2s(st + Lo::kKt, ws.Kt(slot, hv, p.Hv), kC * DK * 2, bar);
        bulk_g2s(st + Lo::kP, ws.P(slot, hv, p.Hv), kC * kC * 2, bar);
        bulk_g2s(st + Lo::kUt, ws.U(slot, hv, p.Hv) + dvt * kC * DVT, kC * DVT * 2, bar);
        bulk_g2s(st + Lo::kGv, ws.gv(slot, hv, p.Hv), kGvFloats * 4, bar);
        bulk_g2s(st + Lo::kQ, ws.Qt(slot, hv, p.Hv), kC * DK * 2, bar);
      };
      for (int c = 0; c < kStages && c < n_chunks; ++c) issue(c);
      for (int c = 0; c + kStages < n_chunks; ++c) {
        // refill the stage chunk c used with chunk c + 3 once both roles are done with it
        if (!mbar_wait(&empty[c % kStages], (c / kStages) & 1, p.err)) { *s_abort = 1; break; }
        if (*s_abort) break;
        issue(c + kStages);
      }
    }
    return;
  }

  if (warp >= kOutWarp0) {
    // ======================= output (warps 4-7) =============================
    // O[16 ow .. 16 ow + 15][tile] = diag(scale gamma) Q h + P V_new
    const int ow = warp - kOutWarp0, m0 = 16 * ow;
    __nv_bfloat16* og = static_cast<__nv_bfloat16*>(p.o) + (long long)hv * p.dv + dvt * DVT;
    const long long o_tok = (long long)p.Hv * p.dv;
    for (int c = 0; c < n_chunks; ++c) {
      const unsigned char* st = sm + (c % kStages) * Lo::kStageBytes;
      const int hb = c % kPub;
      if (!mbar_wait(&full[c % kStages], (c / kStages) & 1, p.err)) *s_abort = 1;
      if (!*s_abort && !mbar_wait(&pub[hb], (c / kPub) & 1, p.err)) *s_abort = 1;
      if (*s_abort) break;
      const __half* H = Hring + hb * DK * DVT;
      const __half* Vn = Vring + hb * kC * DVT;
      float acc[NT][4];
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int x = 0; x < 4; ++x) acc[j][x] = 0.f;
      // inter-chunk term Q~ h (Q~ already scaled, fp16)
#pragma unroll
      for (int ks = 0; ks < DK / 16; ++ks) {
        uint32_t a[4];
        load_a_sw128(a, st + Lo::kQ, m0, 16 * ks, lane);
#pragma unroll
        for (int j = 0; j < NT; j += 2) {
          uint32_t bb[4];
          load_b_kn_sw<DVT>(bb, H, 8 * j, 16 * ks, lane);
          mma_f16(acc[j], a, bb[0], bb[1]);
          mma_f16(acc[j + 1], a, bb[2], bb[3]);
        }
      }
      // intra-chunk term P V_new (P lower triangular: k <= this row block)
      const __half* P = reinterpret_cast<const __half*>(st + Lo::kP);
      for (int kk = 0; kk <= m0; kk += 16) {
        uint32_t a[4];
        load_a_sw<kC>(a, P, m0, kk, lane);
#pragma unroll
        for (int j = 0; j < NT; j += 2) {
          uint32_t bb[4];
          load_b_kn_sw<DVT>(bb, Vn, 8 * j, kk, lane);
          mma_f16(acc[j], a, bb[0], bb[1]);
          mma_f16(acc[j + 1], a, bb[2], bb[3]);
        }
      }
      __syncwarp();
      if (lane == 0) {  // this warp is done with H[hb], Vn[hb] and the stage
        mbar_arrive(&pubd[hb]);
        mbar_arrive(&empty[c % kStages]);
      }
      const long long t0 = t_seq + (long long)c * kC;
      const int L = (int)min((long long)kC, len - (long long)c * kC);
      const int r0 = m0 + gq, r1 = r0 + 8;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int col = 8 * j + 2 * tq;
        if (r0 < L)
          *reinterpret_cast<uint32_t*>(og + (t0 + r0) * o_tok + col) = pack_bf16(acc[j][0], acc[j][1]);
        if (r1 < L)
          *reinterpret_cast<uint32_t*>(og + (t0 + r1) * o_tok + col) = pack_bf16(acc[j][2], acc[j][3]);
      }
    }
    return;
  }

  // ========================= chain (warps 0-3) ===============================
  // Per chunk: V_new (depth-4 accumulation chains: K split in two halves), one
  // barrier, the state update straight into the next H buffer, one barrier.
  // The A fragments of W and Kt are read before the state they multiply is ready.
  // any fp16 copy of V_new or of the state that rounded to infinity (|x| past 65504)
  // or is not a number: the fp16 operands are no longer exact and the call is reported
  uint32_t f16bad = 0u;
  int c = 0;
  for (; c < n_chunks; ++c) {
    const unsigned char* st = sm + (c % kStages) * Lo::kStageBytes;
    const __half* Wt = reinterpret_cast<const __half*>(st + Lo::kWt);
    const __half* Kt = reinterpret_cast<const __half*>(st + Lo::kKt);
    const __half* Ut = reinterpret_cast<const __half*>(st + Lo::kUt);
    const int hb = c % kPub, hn = (c + 1) % kPub;
    __half* Hc = Hring + hb * DK * DVT;
    __half* Hn = Hring + hn * DK * DVT;
    __half* Vc = Vring + hb * kC * DVT;
    GDN_PHASE(16);  // loop top
    if (!mbar_wait(&full[c % kStages], (c / kStages) & 1, p.err)) *s_abort = 1;
    GDN_PHASE(17);  // wait for staging
    uint32_t wa[DK / 16][4];  // W rows of this warp, all k steps
    if (delta) {
#pragma unroll
      for (int ks = 0; ks < DK / 16; ++ks) load_a_trans_sw<kC>(wa[ks], Wt, 16 * warp, 16 * ks, lane);
    }
    uint32_t ka[kC / 16][MTW][4];  // Kt^T rows of this warp, all k steps
#pragma unroll
    for (int ks = 0; ks < kC / 16; ++ks)
#pragma unroll
      for (int mt = 0; mt < MTW; ++mt)
        load_a_trans_blk<kC>(ka[ks][mt], Kt, 16 * (MTW * warp + mt), 16 * ks, lane);

    // #5 read: V_new = U - W h   (warp: 16 token rows x the dv tile)
    const int r0 = 16 * warp + gq;
    {
      float wh[2][NT][4];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int x = 0; x < 4; ++x) wh[hh][j][x] = 0.f;
      if (delta) {  // SSD: V_new = U
#pragma unroll
      for (int ks = 0; ks < DK / 32; ++ks) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int kk = 16 * (ks + hh * (DK / 32));
#pragma unroll
          for (int j = 0; j < NT; j += 2) {
            uint32_t bb[4];
            load_b_kn_sw<DVT>(bb, Hc, 8 * j, kk, lane);
            mma_f16(wh[hh][j], wa[kk / 16], bb[0], bb[1]);
            mma_f16(wh[hh][j + 1], wa[kk / 16], bb[2], bb[3]);
          }
        }
      }
      }
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int col = 8 * j + 2 * tq;
        const float2 u0 = make_float2(__half2float(Ut[swz<kC>(col, r0)]),
                                      __half2float(Ut[swz<kC>(col + 1, r0)]));
        const float2 u1 = make_float2(__half2float(Ut[swz<kC>(col, r0 + 8)]),
                                      __half2float(Ut[swz<kC>(col + 1, r0 + 8)]));
        const uint32_t va =
            pack_f16(u0.x - wh[0][j][0] - wh[1][j][0], u0.y - wh[0][j][1] - wh[1][j][1]);
        const uint32_t vb =
            pack_f16(u1.x - wh[0][j][2] - wh[1][j][2], u1.y - wh[0][j][3] - wh[1][j][3]);
        *reinterpret_cast<uint32_t*>(&Vc[swz<DVT>(r0, col)]) = va;
        *reinterpret_cast<uint32_t*>(&Vc[swz<DVT>(r0 + 8, col)]) = vb;
        f16bad |= f16_inf_or_nan(va) | f16_inf_or_nan(vb);
      }
    }
    if (tid == 0) *s_cstop = *s_abort;
    named_sync(1, kComputeThreads);  // V_new complete (H[hb] was complete before)
    GDN_PHASE(20);  // V_new
    if (*s_cstop) break;
    if (tid == 0) mbar_arrive(&pub[hb]);

    // #5 update: h = gamma_last h + Kt^T V_new, written straight into H[hn]
    // (KDA: row r of h decays by exp(G_last) of key channel r)
    {
      const float* gvs = reinterpret_cast<const float*>(st + Lo::kGv);
#pragma unroll
      for (int mt = 0; mt < MTW; ++mt) {
        const int hr = 16 * (MTW * warp + mt) + gq;
        const float g0 = KDA ? gvs[4 + hr] : gvs[0], g1 = KDA ? gvs[4 + hr + 8] : gvs[0];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          hacc[mt][j][0] *= g0;
          hacc[mt][j][1] *= g0;
          hacc[mt][j][2] *= g1;
          hacc[mt][j][3] *= g1;
        }
      }
#pragma unroll
      for (int ks = 0; ks < kC / 16; ++ks) {
#pragma unroll
        for (int j = 0; j < NT; j += 2) {
          uint32_t bb[4];
          load_b_kn_sw<DVT>(bb, Vc, 8 * j, 16 * ks, lane);
#pragma unroll
          for (int mt = 0; mt < MTW; ++mt) {
            mma_f16(hacc[mt][j], ka[ks][mt], bb[0], bb[1]);
            mma_f16(hacc[mt][j + 1], ka[ks][mt], bb[2], bb[3]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[c % kStages]);  // this warp is done with the stage
    GDN_PHASE(22);  // update
    // H[hn] last held the state entering chunk c - 2: the output warps must be done with it
    if (c >= 2 && !mbar_wait(&pubd[hn], ((c - 2) / kPub) & 1, p.err)) *s_abort = 1;
#pragma unroll
    for (int mt = 0; mt < MTW; ++mt)
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int hr = 16 * (MTW * warp + mt) + gq, col = 8 * j + 2 * tq;
        const uint32_t ha = pack_f16(hacc[mt][j][0], hacc[mt][j][1]);
        const uint32_t hb = pack_f16(hacc[mt][j][2], hacc[mt][j][3]);
        *reinterpret_cast<uint32_t*>(&Hn[swz<DVT>(hr, col)]) = ha;
        *reinterpret_cast<uint32_t*>(&Hn[swz<DVT>(hr + 8, col)]) = hb;
        f16bad |= f16_inf_or_nan(ha) | f16_inf_or_nan(hb);
      }
    named_sync(1, kComputeThreads);  // next state copy complete
    GDN_PHASE(23);  // state copy
  }
  if (__any_sync(0xffffffffu, f16bad != 0u) && lane == 0) record_error(p.err, kErrOperandRange);
  if (tid == 0 && *s_abort) {  // a wait gave up: let the copies already issued land
    for (int cc = c + 1; cc < min(c + kStages, n_chunks); ++cc)
      mbar_wait(&full[cc % kStages], (cc / kStages) & 1, nullptr);
  }
  if (p.hT && !*s_abort) {
    float* hT = p.hT + ((long long)(n * p.Hv + hv) * DK) * p.dv + dvt * DVT;
#pragma unroll
    for (int mt = 0; mt < MTW; ++mt)
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int r0 = 16 * (MTW * warp + mt) + gq, col = 8 * j + 2 * tq;
        *reinterpret_cast<float2*>(hT + (long long)r0 * p.dv + col) =
            make_float2(hacc[mt][j][0], hacc[mt][j][1]);
        *reinterpret_cast<float2*>(hT + (long long)(r0 + 8) * p.dv + col) =
            make_float2(hacc[mt][j][2], hacc[mt][j][3]);
      }
  }
}

template <int DK, int DVT>
cudaError_t launch_t(const FwdParams& p, const WsLayout& ws, cudaStream_t stream) {
  using Lo = ChainLayout<DK, DVT>;
  const long long grid = (long long)p.N * p.Hv * (p.dv / DVT);
  if constexpr (DVT == 64) {  // 64-column tiles: only without the erase term (no W stage)
    using L64 = ChainLayout<DK, 64, true>;
    if (p.delta_rule || p.kda) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(gdn_chain_kernel<DK, 64, false, true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L64::kAlloc);
    if (e != cudaSuccess) return e;
    return launch_after(gdn_chain_kernel<DK, 64, false, true>, (unsigned)grid, kThreads,
                        L64::kAlloc, stream, p, ws);
  } else {
    if (p.kda) {  // KDA records exist for dk = 128 only
      if constexpr (DK == 128) {
        cudaError_t e = cudaFuncSetAttribute(gdn_chain_kernel<DK, DVT, true>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, Lo::kAlloc);
        if (e != cudaSuccess) return e;
        return launch_after(gdn_chain_kernel<DK, DVT, true>, (unsigned)grid, kThreads, Lo::kAlloc,
                            stream, p, ws);
      }
      return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaFuncSetAttribute(gdn_chain_kernel<DK, DVT, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Lo::kAlloc);
    if (e != cudaSuccess) return e;
    return launch_after(gdn_chain_kernel<DK, DVT, false>, (unsigned)grid, kThreads, Lo::kAlloc,
                        stream, p, ws);
  }
}

template <int DK>
cudaError_t launch_dk(const FwdParams& p, const WsLayout& ws, cudaStream_t stream) {
  if (ws.dvt == 16) return launch_t<DK, 16>(p, ws, stream);
  if (ws.dvt == 64) return launch_t<DK, 64>(p, ws, stream);
  return launch_t<DK, 32>(p, ws, stream);
}

}  // namespace

cudaError_t launch_chain(const FwdParams& p, const WsLayout& ws, cudaStream_t stream) {
  if (p.dk == 128) return launch_dk<128>(p, ws, stream);
  return launch_dk<64>(p, ws, stream);
}

}  // namespace gdn
