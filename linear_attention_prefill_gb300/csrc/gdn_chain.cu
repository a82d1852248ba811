// gdn_chain.cu - the serial Reduce (#5 H) of the chunkwise forward
// ("Empowering Hybrid Attention Models on NPUs", §2.1, Figure 1(b)), split as in
// §5 (Figure 10(b)) into the state read and the in-place update:
//   #5 read    V_new = U - W h
//   #5 update  h = gamma_last h + Kt^T V_new        (Kt = diag(e) K)
// One CTA per (sequence, v head, dv tile) walks the chunks of its sequence in
// order with its fp32 state tile h[:, tile] in registers: the column split of
// the state (§4, Figure 8(b)) gives parallelism without any reduction.
//
// Warp roles.  Warps 0-3 run the chain: two warp-level fp16 tensor-core
// products per chunk (mma.sync, the state as accumulator) and two CTA-local
// barriers - nothing else sits on the serial path.  Warp 4 is the producer: it
// stages W, Kt, the U tile and gamma_last of chunk c + 3 with bulk copies into a
// 3-deep ring (36 KB per chunk at d = 128: one SM takes in about 64 bytes per
// clock from L2, which bounds the step), and publishes the state entering each
// chunk (H) and V_new with bulk stores for gdn_out.  The roles meet only at
// mbarriers; every wait is bounded and an expired wait ends the CTA cleanly.
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kC = 64;
constexpr int kComputeThreads = 128;  // warps 0-3
constexpr int kThreads = 160;         // + producer warp
constexpr int kStages = 3;
constexpr int kPub = 3;  // H / V_new buffers: the store of chunk c - 1 has a whole step to finish

template <int DK, int DVT>
struct ChainSmem {
  struct Stage {
    __half W[kC * DK];    // swz<DK>
    __half Kt[kC * DK];   // swz<DK>
    __half U[kC * DVT];   // plain
    float gl[4];
  };
  Stage st[kStages];
  __half H[kPub][DK * DVT];   // swz<DVT>: state entering the chunk (ring for the stores)
  __half Vn[kPub][kC * DVT];  // swz<DVT>
  uint64_t full[kStages];     // producer -> chain: chunk staged (transaction bytes)
  uint64_t empty[kStages];    // chain -> producer: stage consumed (4 warp arrivals)
  uint64_t pub[kPub];         // chain -> producer: H[b], Vn[b] ready to store
  uint64_t pubd[kPub];        // producer -> chain: H[b], Vn[b] read by the store
  int abort;
};

template <int DK, int DVT>
__global__ void __launch_bounds__(kThreads, 1) gdn_chain_kernel(const FwdParams p, WsLayout ws) {
  using S = ChainSmem<DK, DVT>;
  constexpr int NT = DVT / 8;          // n8 tiles over the dv tile
  constexpr int MTW = DK / 64;         // m16 tiles of the state per warp
  constexpr unsigned kStageBytes = 2 * kC * DK * 2 + kC * DVT * 2 + 16;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  S& s = *reinterpret_cast<S*>(smem_raw);
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
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 4);
    }
    for (int i = 0; i < kPub; ++i) {
      mbar_init(&s.pub[i], 1);
      mbar_init(&s.pubd[i], 1);
    }
    s.abort = 0;
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
        *reinterpret_cast<uint32_t*>(&s.H[0][swz<DVT>(r0, col)]) = pack_f16(a.x, a.y);
        *reinterpret_cast<uint32_t*>(&s.H[0][swz<DVT>(r0 + 8, col)]) = pack_f16(b.x, b.y);
      }
  }
  __syncthreads();  // barriers initialised, H[0] written

  if (warp == 4) {
    // ======================= producer ======================================
    if (lane == 0) {
      auto issue = [&](int c) {
        typename S::Stage& b = s.st[c % kStages];
        uint64_t* bar = &s.full[c % kStages];
        mbar_expect_tx(bar, kStageBytes);
        bulk_g2s(b.W, ws.W(slot0 + c, hv, p.Hv), kC * DK * 2, bar);
        bulk_g2s(b.Kt, ws.Kt(slot0 + c, hv, p.Hv), kC * DK * 2, bar);
        bulk_g2s(b.U, ws.U(slot0 + c, hv, p.Hv) + dvt * kC * DVT, kC * DVT * 2, bar);
        bulk_g2s(b.gl, ws.gl(slot0 + c, hv, p.Hv), 16, bar);
      };
      for (int c = 0; c < kStages && c < n_chunks; ++c) issue(c);
      for (int c = 0; c < n_chunks; ++c) {
        const int hb = c % kPub;
        // publish the state entering chunk c and its V_new
        if (!mbar_wait(&s.pub[hb], (c / kPub) & 1, p.err)) { s.abort = 1; break; }
        bulk_s2g(ws.H(slot0 + c, hv, p.Hv) + dvt * DK * DVT, s.H[hb], DK * DVT * 2);
        bulk_s2g(ws.Vn(slot0 + c, hv, p.Hv) + dvt * kC * DVT, s.Vn[hb], kC * DVT * 2);
        bulk_commit();
        bulk_wait_read<0>();
        mbar_arrive(&s.pubd[hb]);
        // refill the stage chunk c used with chunk c + 3
        if (c + kStages < n_chunks) {
          if (!mbar_wait(&s.empty[c % kStages], (c / kStages) & 1, p.err)) { s.abort = 1; break; }
          issue(c + kStages);
        }
        if (s.abort) break;
      }
      bulk_wait<0>();
    }
    return;
  }

  // ========================= chain (warps 0-3) ===============================
  // Per chunk: V_new (depth-4 accumulation chains: K split in two halves), one
  // barrier, the state update straight into the next H buffer, one barrier.
  // The A fragments of W and Kt are read before the state they multiply is ready.
  int c = 0;
  for (; c < n_chunks; ++c) {
    typename S::Stage& b = s.st[c % kStages];
    const int hb = c % kPub, hn = (c + 1) % kPub;
    GDN_PHASE(16);  // loop top
    if (!mbar_wait(&s.full[c % kStages], (c / kStages) & 1, p.err)) s.abort = 1;
    GDN_PHASE(17);  // wait for staging
    uint32_t wa[DK / 16][4];  // W rows of this warp, all k steps
#pragma unroll
    for (int ks = 0; ks < DK / 16; ++ks) load_a_sw<DK>(wa[ks], b.W, 16 * warp, 16 * ks, lane);
    uint32_t ka[kC / 16][MTW][4];  // Kt^T rows of this warp, all k steps
#pragma unroll
    for (int ks = 0; ks < kC / 16; ++ks)
#pragma unroll
      for (int mt = 0; mt < MTW; ++mt)
        load_a_trans_sw<DK>(ka[ks][mt], b.Kt, 16 * (MTW * warp + mt), 16 * ks, lane);

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
#pragma unroll
      for (int ks = 0; ks < DK / 32; ++ks) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int kk = 16 * (ks + hh * (DK / 32));
#pragma unroll
          for (int j = 0; j < NT; j += 2) {
            uint32_t bb[4];
            load_b_kn_sw<DVT>(bb, s.H[hb], 8 * j, kk, lane);
            mma_f16(wh[hh][j], wa[kk / 16], bb[0], bb[1]);
            mma_f16(wh[hh][j + 1], wa[kk / 16], bb[2], bb[3]);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int col = 8 * j + 2 * tq;
        const float2 u0 = __half22float2(*reinterpret_cast<const __half2*>(&b.U[r0 * DVT + col]));
        const float2 u1 =
            __half22float2(*reinterpret_cast<const __half2*>(&b.U[(r0 + 8) * DVT + col]));
        *reinterpret_cast<uint32_t*>(&s.Vn[hb][swz<DVT>(r0, col)]) =
            pack_f16(u0.x - wh[0][j][0] - wh[1][j][0], u0.y - wh[0][j][1] - wh[1][j][1]);
        *reinterpret_cast<uint32_t*>(&s.Vn[hb][swz<DVT>(r0 + 8, col)]) =
            pack_f16(u1.x - wh[0][j][2] - wh[1][j][2], u1.y - wh[0][j][3] - wh[1][j][3]);
      }
    }
    fence_proxy_async();
    named_sync(1, kComputeThreads);  // V_new complete (H[hb] was complete before)
    GDN_PHASE(20);  // V_new
    if (s.abort) break;
    if (tid == 0) mbar_arrive(&s.pub[hb]);

    // #5 update: h = gamma_last h + Kt^T V_new, written straight into H[hn]
    {
      const float gl = b.gl[0];
#pragma unroll
      for (int mt = 0; mt < MTW; ++mt)
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int x = 0; x < 4; ++x) hacc[mt][j][x] *= gl;
#pragma unroll
      for (int ks = 0; ks < kC / 16; ++ks) {
#pragma unroll
        for (int j = 0; j < NT; j += 2) {
          uint32_t bb[4];
          load_b_kn_sw<DVT>(bb, s.Vn[hb], 8 * j, 16 * ks, lane);
#pragma unroll
          for (int mt = 0; mt < MTW; ++mt) {
            mma_f16(hacc[mt][j], ka[ks][mt], bb[0], bb[1]);
            mma_f16(hacc[mt][j + 1], ka[ks][mt], bb[2], bb[3]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&s.empty[c % kStages]);  // this warp is done with the stage
    GDN_PHASE(22);  // update
    // H[hn] last held the state entering chunk c - 2: its store must have read it
    if (c >= 2 && !mbar_wait(&s.pubd[hn], ((c - 2) / kPub) & 1, p.err)) s.abort = 1;
#pragma unroll
    for (int mt = 0; mt < MTW; ++mt)
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int hr = 16 * (MTW * warp + mt) + gq, col = 8 * j + 2 * tq;
        *reinterpret_cast<uint32_t*>(&s.H[hn][swz<DVT>(hr, col)]) =
            pack_f16(hacc[mt][j][0], hacc[mt][j][1]);
        *reinterpret_cast<uint32_t*>(&s.H[hn][swz<DVT>(hr + 8, col)]) =
            pack_f16(hacc[mt][j][2], hacc[mt][j][3]);
      }
    named_sync(1, kComputeThreads);  // next state copy complete
    GDN_PHASE(23);  // state copy
  }
  if (tid == 0 && s.abort) {  // a wait gave up: let the copies already issued land
    for (int cc = c + 1; cc < min(c + kStages, n_chunks); ++cc)
      mbar_wait(&s.full[cc % kStages], (cc / kStages) & 1, nullptr);
  }
  if (p.hT && !s.abort) {
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
  const size_t smem = sizeof(ChainSmem<DK, DVT>);
  cudaError_t e = cudaFuncSetAttribute(gdn_chain_kernel<DK, DVT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)p.N * p.Hv * (p.dv / DVT);
  gdn_chain_kernel<DK, DVT><<<(unsigned)grid, kThreads, smem, stream>>>(p, ws);
  return cudaGetLastError();
}

template <int DK>
cudaError_t launch_dk(const FwdParams& p, const WsLayout& ws, cudaStream_t stream) {
  if (ws.dvt == 16) return launch_t<DK, 16>(p, ws, stream);
  if (ws.dvt == 32) return launch_t<DK, 32>(p, ws, stream);
  return launch_t<DK, 64>(p, ws, stream);
}

}  // namespace

cudaError_t launch_chain(const FwdParams& p, const WsLayout& ws, cudaStream_t stream) {
  if (p.dk == 128) return launch_dk<128>(p, ws, stream);
  return launch_dk<64>(p, ws, stream);
}

}  // namespace gdn
