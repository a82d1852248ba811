// gdn_chain.cu - the serial Reduce (#5 H) of the chunkwise forward
// ("Empowering Hybrid Attention Models on NPUs", §2.1, Figure 1(b)), split as in
// §5 (Figure 10(b)) into the state read and the in-place update:
//   #5 read    V_new = U - W h
//   #5 update  h = gamma_last h + Kt^T V_new        (Kt = diag(e) K)
// One CTA per (sequence, v head, 32-column dv tile) walks the chunks of its
// sequence in order with its fp32 state tile h[:, tile] in registers: the
// column split of the state (§4, Figure 8(b)) gives parallelism without any
// reduction.  Per chunk it reads only W, Kt and its U tile (36 KB at d = 128,
// about what one SM can pull from L2 in a chain step) from gdn_prep's record,
// and publishes the state entering the chunk (H) and V_new for gdn_out, which
// forms the outputs chunk-parallel.  The chain's two products are warp-level
// fp16 tensor-core MMAs (mma.sync; the state is their accumulator).
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kC = 64;
constexpr int kThreads = 128;  // 4 warps
constexpr int kStages = 3;
constexpr int DVT = kDvTile;

template <int DK>
struct ChainSmem {
  static constexpr int LDK = DK + 8;
  static constexpr int LDT = DVT + 8;
  struct Stage {
    __half W[kC * LDK];
    __half Kt[kC * LDK];
    __half U[kC * LDT];
    float gl[4];
  };
  Stage st[kStages];
  __half H[DK * LDT];     // fp16 copy of the state tile entering the chunk
  __half Vn[kC * LDT];    // V_new
};

template <int DK>
__global__ void __launch_bounds__(kThreads, 1) gdn_chain_kernel(const FwdParams p, WsLayout ws) {
  using S = ChainSmem<DK>;
  constexpr int LDK = S::LDK, LDT = S::LDT;
  constexpr int NT = DVT / 8;          // n8 tiles over the dv tile (4)
  constexpr int MTW = DK / 64;         // m16 tiles of the state per warp
  extern __shared__ __align__(128) unsigned char smem_raw[];
  S& s = *reinterpret_cast<S*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;

  const int n_dvt = p.dv / DVT;
  const int dvt = blockIdx.x % n_dvt;
  const int hv = (blockIdx.x / n_dvt) % p.Hv;
  const int n = blockIdx.x / (n_dvt * p.Hv);
  const long long t_seq = p.cu_seqlens ? (long long)p.cu_seqlens[n] : (long long)n * p.T;
  const long long len = p.cu_seqlens ? (long long)p.cu_seqlens[n + 1] - t_seq : (long long)p.T;
  const int n_chunks = (int)((len + kC - 1) / kC);
  const long long slot0 = ws.first_slot(p, n);

  auto issue = [&](int c) {
    if (c < n_chunks) {
      typename S::Stage& b = s.st[c % kStages];
      const __half* Wg = ws.W(slot0 + c, hv, p.Hv);
      const __half* Kg = ws.Kt(slot0 + c, hv, p.Hv);
      const __half* Ug = ws.U(slot0 + c, hv, p.Hv) + dvt * kC * DVT;
      for (int i = tid; i < kC * (DK / 8); i += kThreads) {
        const int r = i / (DK / 8), sg = i % (DK / 8);
        cp_async16(&b.W[r * LDK + sg * 8], Wg + r * DK + sg * 8, true);
        cp_async16(&b.Kt[r * LDK + sg * 8], Kg + r * DK + sg * 8, true);
      }
      for (int i = tid; i < kC * (DVT / 8); i += kThreads) {
        const int r = i / (DVT / 8), sg = i % (DVT / 8);
        cp_async16(&b.U[r * LDT + sg * 8], Ug + r * DVT + sg * 8, true);
      }
      if (tid == 0) cp_async4(&b.gl[0], ws.gl(slot0 + c, hv, p.Hv), true);
    }
    cp_async_commit();  // possibly empty: one group per chunk keeps the counting uniform
  };

  // ---- initial state ---------------------------------------------------------
  float hacc[MTW][NT][4];
  {
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
        *reinterpret_cast<uint32_t*>(&s.H[r0 * LDT + col]) = pack_f16(a.x, a.y);
        *reinterpret_cast<uint32_t*>(&s.H[(r0 + 8) * LDT + col]) = pack_f16(b.x, b.y);
      }
  }
  for (int i = 0; i < kStages - 1; ++i) issue(i);

  for (int c = 0; c < n_chunks; ++c) {
    typename S::Stage& b = s.st[c % kStages];
    const long long slot = slot0 + c;
    cp_async_wait<kStages - 2>();
    __syncthreads();  // chunk c staged; s.H holds the state entering chunk c
    issue(c + kStages - 1);

    // publish the state entering the chunk for the output launch (fp16 tile)
    {
      __half* Hg = ws.H(slot, hv, p.Hv) + dvt * DK * DVT;
      for (int i = tid; i < DK * (DVT / 8); i += kThreads) {
        const int r = i / (DVT / 8), sg = i % (DVT / 8);
        *reinterpret_cast<uint4*>(Hg + r * DVT + sg * 8) =
            *reinterpret_cast<const uint4*>(&s.H[r * LDT + sg * 8]);
      }
    }

    // #5 read: V_new = U - W h   (warp: 16 token rows x the dv tile)
    const int r0 = 16 * warp + gq;
    {
      float wh[NT][4];
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int x = 0; x < 4; ++x) wh[j][x] = 0.f;
#pragma unroll
      for (int kk = 0; kk < DK; kk += 16) {
        uint32_t a[4], bb[4];
        load_a(a, b.W, LDK, 16 * warp, kk, lane);
#pragma unroll
        for (int j = 0; j < NT; j += 2) {
          load_b_kn(bb, s.H, LDT, 8 * j, kk, lane);
          mma_f16(wh[j], a, bb[0], bb[1]);
          mma_f16(wh[j + 1], a, bb[2], bb[3]);
        }
      }
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int col = 8 * j + 2 * tq;
        const float2 u0 = __half22float2(*reinterpret_cast<const __half2*>(&b.U[r0 * LDT + col]));
        const float2 u1 =
            __half22float2(*reinterpret_cast<const __half2*>(&b.U[(r0 + 8) * LDT + col]));
        *reinterpret_cast<uint32_t*>(&s.Vn[r0 * LDT + col]) =
            pack_f16(u0.x - wh[j][0], u0.y - wh[j][1]);
        *reinterpret_cast<uint32_t*>(&s.Vn[(r0 + 8) * LDT + col]) =
            pack_f16(u1.x - wh[j][2], u1.y - wh[j][3]);
      }
    }
    __syncthreads();  // V_new complete; every warp is done reading s.H

    // publish V_new; #5 update: h = gamma_last h + Kt^T V_new
    {
      __half* Vg = ws.Vn(slot, hv, p.Hv) + dvt * kC * DVT;
      for (int i = tid; i < kC * (DVT / 8); i += kThreads) {
        const int r = i / (DVT / 8), sg = i % (DVT / 8);
        *reinterpret_cast<uint4*>(Vg + r * DVT + sg * 8) =
            *reinterpret_cast<const uint4*>(&s.Vn[r * LDT + sg * 8]);
      }
      const float gl = b.gl[0];
#pragma unroll
      for (int mt = 0; mt < MTW; ++mt)
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int x = 0; x < 4; ++x) hacc[mt][j][x] *= gl;
#pragma unroll
      for (int kk = 0; kk < kC; kk += 16) {
        uint32_t bb[4];
        uint32_t a[MTW][4];
#pragma unroll
        for (int mt = 0; mt < MTW; ++mt)
          load_a_trans(a[mt], b.Kt, LDK, 16 * (MTW * warp + mt), kk, lane);
#pragma unroll
        for (int j = 0; j < NT; j += 2) {
          load_b_kn(bb, s.Vn, LDT, 8 * j, kk, lane);
#pragma unroll
          for (int mt = 0; mt < MTW; ++mt) {
            mma_f16(hacc[mt][j], a[mt], bb[0], bb[1]);
            mma_f16(hacc[mt][j + 1], a[mt], bb[2], bb[3]);
          }
        }
      }
#pragma unroll
      for (int mt = 0; mt < MTW; ++mt)
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const int hr = 16 * (MTW * warp + mt) + gq, col = 8 * j + 2 * tq;
          *reinterpret_cast<uint32_t*>(&s.H[hr * LDT + col]) =
              pack_f16(hacc[mt][j][0], hacc[mt][j][1]);
          *reinterpret_cast<uint32_t*>(&s.H[(hr + 8) * LDT + col]) =
              pack_f16(hacc[mt][j][2], hacc[mt][j][3]);
        }
    }
  }
  cp_async_wait<0>();

  if (p.hT) {
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

template <int DK>
cudaError_t launch_t(const FwdParams& p, const WsLayout& ws, cudaStream_t stream) {
  const size_t smem = sizeof(ChainSmem<DK>);
  cudaError_t e = cudaFuncSetAttribute(gdn_chain_kernel<DK>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)p.N * p.Hv * (p.dv / DVT);
  gdn_chain_kernel<DK><<<(unsigned)grid, kThreads, smem, stream>>>(p, ws);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chain(const FwdParams& p, const WsLayout& ws, cudaStream_t stream) {
  if (p.dk == 128) return launch_t<128>(p, ws, stream);
  return launch_t<64>(p, ws, stream);
}

}  // namespace gdn
