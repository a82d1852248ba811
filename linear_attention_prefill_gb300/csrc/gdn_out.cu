// gdn_out.cu - the final Map (#6 O) of the chunkwise forward
// ("Empowering Hybrid Attention Models on NPUs", §2.1, Figure 1(b)):
//   O = diag(scale gamma) Q h + P V_new   = Qt h + P V_new
// with h the state entering the chunk and V_new = U - W h, both published by
// gdn_chain.  Every (chunk, v head) is independent once the chain has passed
// it, so this launch is chunk-parallel over the whole GPU.  Products on fp16
// tensor cores (mma.sync) with fp32 accumulation; o is rounded once to bf16.
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kC = 64;
constexpr int kThreads = 256;

template <int DK, int DV>
struct OutSmem {
  static constexpr int LDK = DK + 8;
  static constexpr int LDV = DV + 8;
  static constexpr int LDC = kC + 8;
  union {
    __half Qt[kC * LDK];
    __nv_bfloat16 O[kC * LDV];  // output staging once the products are done
  };
  __half P[kC * LDC];
  __half H[DK * LDV];
  __half Vn[kC * LDV];
};

template <int DK, int DV>
__global__ void __launch_bounds__(kThreads, 2) gdn_out_kernel(const FwdParams p, WsLayout ws) {
  using S = OutSmem<DK, DV>;
  constexpr int LDK = S::LDK, LDV = S::LDV, LDC = S::LDC;
  constexpr int T32 = kDvTile;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  S& s = *reinterpret_cast<S*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;

  const int hv = blockIdx.x % p.Hv;
  const long long slot = blockIdx.x / p.Hv;
  int n, c;
  if (!locate_chunk(p, ws, slot, &n, &c)) return;
  const long long t_seq = p.cu_seqlens ? (long long)p.cu_seqlens[n] : (long long)n * p.T;
  const long long len =
      p.cu_seqlens ? (long long)p.cu_seqlens[n + 1] - t_seq : (long long)p.T;
  const long long t0 = t_seq + (long long)c * kC;
  const int L = (int)min((long long)kC, len - (long long)c * kC);

  {
    const __half* Qg = ws.Qt(slot, hv, p.Hv);
    const __half* Pg = ws.P(slot, hv, p.Hv);
    const __half* Hg = ws.H(slot, hv, p.Hv);
    const __half* Vg = ws.Vn(slot, hv, p.Hv);
    for (int i = tid; i < kC * (DK / 8); i += kThreads) {
      const int r = i / (DK / 8), sg = i % (DK / 8);
      cp_async16(&s.Qt[r * LDK + sg * 8], Qg + r * DK + sg * 8, true);
    }
    for (int i = tid; i < kC * (kC / 8); i += kThreads) {
      const int r = i / (kC / 8), sg = i % (kC / 8);
      cp_async16(&s.P[r * LDC + sg * 8], Pg + r * kC + sg * 8, true);
    }
    for (int i = tid; i < DK * (DV / 8); i += kThreads) {  // [dv/32][dk][32] -> [dk][dv]
      const int r = i / (DV / 8), col = (i % (DV / 8)) * 8;
      const int t = col / T32, w = col % T32;
      cp_async16(&s.H[r * LDV + col], Hg + (t * DK + r) * T32 + w, true);
    }
    for (int i = tid; i < kC * (DV / 8); i += kThreads) {  // [dv/32][64][32] -> [64][dv]
      const int r = i / (DV / 8), col = (i % (DV / 8)) * 8;
      const int t = col / T32, w = col % T32;
      cp_async16(&s.Vn[r * LDV + col], Vg + (t * kC + r) * T32 + w, true);
    }
    cp_async_commit();
    cp_async_wait<0>();
  }
  __syncthreads();

  const int rb = warp & 3, nh = warp >> 2;
  constexpr int NT = DV / 16;  // n8 tiles per warp (half the columns)
  float acc[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int x = 0; x < 4; ++x) acc[j][x] = 0.f;
#pragma unroll 2
  for (int kk = 0; kk < DK; kk += 16) {
    uint32_t a[4], b[4];
    load_a(a, s.Qt, LDK, 16 * rb, kk, lane);
#pragma unroll
    for (int j = 0; j < NT; j += 2) {
      load_b_kn(b, s.H, LDV, nh * (DV / 2) + 8 * j, kk, lane);
      mma_f16(acc[j], a, b[0], b[1]);
      mma_f16(acc[j + 1], a, b[2], b[3]);
    }
  }
  for (int kk = 0; kk <= 16 * rb; kk += 16) {  // P is lower triangular
    uint32_t a[4], b[4];
    load_a(a, s.P, LDC, 16 * rb, kk, lane);
#pragma unroll
    for (int j = 0; j < NT; j += 2) {
      load_b_kn(b, s.Vn, LDV, nh * (DV / 2) + 8 * j, kk, lane);
      mma_f16(acc[j], a, b[0], b[1]);
      mma_f16(acc[j + 1], a, b[2], b[3]);
    }
  }
  __syncthreads();  // Qt is dead: stage O in its place
  const int r0 = 16 * rb + gq;
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int col = nh * (DV / 2) + 8 * j + 2 * tq;
    *reinterpret_cast<uint32_t*>(&s.O[r0 * LDV + col]) = pack_bf16(acc[j][0], acc[j][1]);
    *reinterpret_cast<uint32_t*>(&s.O[(r0 + 8) * LDV + col]) = pack_bf16(acc[j][2], acc[j][3]);
  }
  __syncthreads();
  const long long v_tok = (long long)p.Hv * DV;
  __nv_bfloat16* og = static_cast<__nv_bfloat16*>(p.o) + (long long)hv * DV;
  for (int i = tid; i < L * (DV / 8); i += kThreads) {
    const int r = i / (DV / 8), sg = i % (DV / 8);
    *reinterpret_cast<uint4*>(og + (t0 + r) * v_tok + sg * 8) =
        *reinterpret_cast<const uint4*>(&s.O[r * LDV + sg * 8]);
  }
}

template <int DK, int DV>
cudaError_t launch_t(const FwdParams& p, const WsLayout& ws, cudaStream_t stream) {
  const size_t smem = sizeof(OutSmem<DK, DV>);
  cudaError_t e = cudaFuncSetAttribute(gdn_out_kernel<DK, DV>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const long long grid = ws.n_slots * p.Hv;
  gdn_out_kernel<DK, DV><<<(unsigned)grid, kThreads, smem, stream>>>(p, ws);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_out(const FwdParams& p, const WsLayout& ws, cudaStream_t stream) {
  if (p.dk == 128) {
    if (p.dv == 128) return launch_t<128, 128>(p, ws, stream);
    return launch_t<128, 64>(p, ws, stream);
  }
  if (p.dv == 128) return launch_t<64, 128>(p, ws, stream);
  return launch_t<64, 64>(p, ws, stream);
}

}  // namespace gdn
