// gdn_out.cu - the final Map (#6 O) of the chunkwise forward
// ("Empowering Hybrid Attention Models on NPUs", §2.1, Figure 1(b)):
//   O = diag(scale gamma) Q h + P V_new   = Qt h + P V_new
// with h the state entering the chunk and V_new = U - W h, both published by
// gdn_chain.  Every (chunk, v head) is independent once the chain has passed
// it, so this launch is chunk-parallel over the whole GPU: one persistent CTA
// per SM walks tasks blockIdx.x, blockIdx.x + gridDim.x, ...; thread 0 stages
// the next task's record (72 KB at d = 128) with bulk copies while the eight
// warps multiply the current one (fp16 tensor cores, mma.sync, fp32
// accumulation); o is rounded once to bf16 and written row by row.
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kC = 64;
constexpr int kThreads = 256;

template <int DK, int DV, int T32>
struct OutSmem {
  static constexpr int LDO = DV + 8;
  struct Stage {
    __half Qt[kC * DK];             // swz<DK>
    __half P[kC * kC];              // swz<64>
    __half H[DV / T32][DK * T32];   // swz<T32> per dv tile
    __half Vn[DV / T32][kC * T32];  // swz<T32> per dv tile
  };
  Stage st[2];
  __nv_bfloat16 O[kC * LDO];        // output staging
  uint64_t full[2];
  int abort;
};

template <int DK, int DV, int T32>
__global__ void __launch_bounds__(kThreads, 1) gdn_out_kernel(const FwdParams p, WsLayout ws) {
  using S = OutSmem<DK, DV, T32>;
  constexpr int LDO = S::LDO;
  constexpr unsigned kBytes = kC * DK * 2 + kC * kC * 2 + DK * DV * 2 + kC * DV * 2;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  S& s = *reinterpret_cast<S*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const long long n_tasks = ws.n_slots * p.Hv;

  if (tid == 0) {
    s.abort = 0;
    mbar_init(&s.full[0], 1);
    mbar_init(&s.full[1], 1);
    mbar_fence_init();
  }
  __syncthreads();
  // thread 0 stages task t into buffer b (tasks on unused slots stage nothing)
  auto stage = [&](long long t, int b) {
    const long long slot = t / p.Hv;
    const int hv = (int)(t % p.Hv);
    int n, c;
    uint64_t* bar = &s.full[b];
    if (!locate_chunk(p, ws, slot, &n, &c)) {
      mbar_arrive(bar);
      return;
    }
    mbar_expect_tx(bar, kBytes);
    bulk_g2s(s.st[b].Qt, ws.Qt(slot, hv, p.Hv), kC * DK * 2, bar);
    bulk_g2s(s.st[b].P, ws.P(slot, hv, p.Hv), kC * kC * 2, bar);
    bulk_g2s(s.st[b].H[0], ws.H(slot, hv, p.Hv), DK * DV * 2, bar);
    bulk_g2s(s.st[b].Vn[0], ws.Vn(slot, hv, p.Hv), kC * DV * 2, bar);
  };
  if (tid == 0 && blockIdx.x < n_tasks) stage(blockIdx.x, 0);

  int it = 0;
  for (long long t = blockIdx.x; t < n_tasks; t += gridDim.x, ++it) {
    const int b = it & 1;
    // every thread is past the previous task, so buffer b ^ 1 is free: stage the next task
    if (tid == 0 && t + gridDim.x < n_tasks) stage(t + gridDim.x, b ^ 1);
    if (!mbar_wait(&s.full[b], (it >> 1) & 1, p.err)) s.abort = 1;
    const long long slot = t / p.Hv;
    const int hv = (int)(t % p.Hv);
    int n, c;
    const bool real = locate_chunk(p, ws, slot, &n, &c);
    if (real) {
      const typename S::Stage& st = s.st[b];
      const int rb = warp & 3, nh = warp >> 2;
      constexpr int NT = DV / 16;  // n8 tiles per warp (half the columns)
      float acc[NT][4];
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int x = 0; x < 4; ++x) acc[j][x] = 0.f;
#pragma unroll 2
      for (int kk = 0; kk < DK; kk += 16) {
        uint32_t a[4], bb[4];
        load_a_sw<DK>(a, st.Qt, 16 * rb, kk, lane);
#pragma unroll
        for (int j = 0; j < NT; j += 2) {
          const int n0 = nh * (DV / 2) + 8 * j;
          load_b_kn_sw<T32>(bb, st.H[n0 / T32], n0 % T32, kk, lane);
          mma_f16(acc[j], a, bb[0], bb[1]);
          mma_f16(acc[j + 1], a, bb[2], bb[3]);
        }
      }
      for (int kk = 0; kk <= 16 * rb; kk += 16) {  // P is lower triangular
        uint32_t a[4], bb[4];
        load_a_sw<kC>(a, st.P, 16 * rb, kk, lane);
#pragma unroll
        for (int j = 0; j < NT; j += 2) {
          const int n0 = nh * (DV / 2) + 8 * j;
          load_b_kn_sw<T32>(bb, st.Vn[n0 / T32], n0 % T32, kk, lane);
          mma_f16(acc[j], a, bb[0], bb[1]);
          mma_f16(acc[j + 1], a, bb[2], bb[3]);
        }
      }
      const int r0 = 16 * rb + gq;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int col = nh * (DV / 2) + 8 * j + 2 * tq;
        *reinterpret_cast<uint32_t*>(&s.O[r0 * LDO + col]) = pack_bf16(acc[j][0], acc[j][1]);
        *reinterpret_cast<uint32_t*>(&s.O[(r0 + 8) * LDO + col]) = pack_bf16(acc[j][2], acc[j][3]);
      }
    }
    __syncthreads();  // O staged; every warp is done with buffer b
    if (s.abort) break;
    if (real) {
      const long long t_seq = p.cu_seqlens ? (long long)p.cu_seqlens[n] : (long long)n * p.T;
      const long long len =
          p.cu_seqlens ? (long long)p.cu_seqlens[n + 1] - t_seq : (long long)p.T;
      const long long t0 = t_seq + (long long)c * kC;
      const int L = (int)min((long long)kC, len - (long long)c * kC);
      const long long v_tok = (long long)p.Hv * DV;
      __nv_bfloat16* og = static_cast<__nv_bfloat16*>(p.o) + (long long)hv * DV;
      for (int i = tid; i < L * (DV / 8); i += kThreads) {
        const int r = i / (DV / 8), sg = i % (DV / 8);
        *reinterpret_cast<uint4*>(og + (t0 + r) * v_tok + sg * 8) =
            *reinterpret_cast<const uint4*>(&s.O[r * LDO + sg * 8]);
      }
    }
    __syncthreads();  // O is free again
  }
  if (tid == 0 && s.abort) {  // let a copy already issued land before exiting
    const int b = (it + 1) & 1;
    mbar_wait(&s.full[b], ((it + 1) >> 1) & 1, nullptr);
  }
}

template <int DK, int DV, int T>
cudaError_t launch_t(const FwdParams& p, const WsLayout& ws, cudaStream_t stream) {
  const size_t smem = sizeof(OutSmem<DK, DV, T>);
  cudaError_t e = cudaFuncSetAttribute(gdn_out_kernel<DK, DV, T>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long tasks = ws.n_slots * p.Hv;
  const long long grid = tasks < sms ? tasks : sms;
  gdn_out_kernel<DK, DV, T><<<(unsigned)grid, kThreads, smem, stream>>>(p, ws);
  return cudaGetLastError();
}

template <int DK, int DV>
cudaError_t launch_dv(const FwdParams& p, const WsLayout& ws, cudaStream_t stream) {
  if (ws.dvt == 16) return launch_t<DK, DV, 16>(p, ws, stream);
  if (ws.dvt == 32) return launch_t<DK, DV, 32>(p, ws, stream);
  return launch_t<DK, DV, 64>(p, ws, stream);
}

}  // namespace

cudaError_t launch_out(const FwdParams& p, const WsLayout& ws, cudaStream_t stream) {
  if (p.dk == 128) {
    if (p.dv == 128) return launch_dv<128, 128>(p, ws, stream);
    return launch_dv<128, 64>(p, ws, stream);
  }
  if (p.dv == 128) return launch_dv<64, 128>(p, ws, stream);
  return launch_dv<64, 64>(p, ws, stream);
}

}  // namespace gdn
