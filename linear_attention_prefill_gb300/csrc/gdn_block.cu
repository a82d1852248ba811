// gdn_block.cu - the chunkwise forward on 128-token blocks (gated delta rule,
// dk = dv = 128): the state-passing Reduce (#5) as an affine recurrence with
// one tensor-core product per block, and the final Map (#6) fully parallel.
//
// "Empowering Hybrid Attention Models on NPUs", §2.1 (Figure 1(b)) splits the
// chunkwise form into chunk-local Map operators #1-#4, the serial Reduce #5
// and the output Map #6.  With W = Tm diag(beta gamma) K, U = Tm diag(beta) V
// and Kt = diag(e) K of one chunk (from gdn_prep.cu), #5 is
//     h <- gamma_last h + Kt^T (U - W h) = gamma_last h - N h + B,
//     N = Kt^T W (dk x dk),  B = Kt^T U (dk x dv),
// an affine map whose matrices depend on the chunk alone.  Two consecutive
// 64-token chunks compose into one such map for their 128-token block: with
// X = W2 Kt1^T,
//     W2' = gamma_last1 W2 - X W1,   U2' = U2 - X U1,
//     N = [Kt1; Kt2]^T [gamma_last2 W1; W2'],  B = [Kt1; Kt2]^T [gamma_last2 U1; U2'],
//     gamma = gamma_last1 gamma_last2,
// and the block's values V_new = [U1; U2'] - [W1; W2'] h read the state only
// at the block start (W2', U2' fold the first chunk's update into the second
// chunk's state read: the coupling block of the blocked UT transform).  The
// block output is
//     O = diag(scale gamma') Q h + P' V_new,
// gamma' the gate products from the block start and P' the 128 x 128 causal
// intra-block matrix: the two chunks' P on the diagonal and
//     Y_ij = scale gamma2_i e1_j q_i.k_j
// (chunk-2 rows, chunk-1 columns) below it.  These are the UT-transform
// identities of "Exp 2026-07-13 — Linear-Attention Scans on the NPU", §1,
// applied to a chunk of twice the length.
//
// Three launches:
//   gdn_pair_kernel  (block, v head): X, W2', U2' (written back into the second
//                    chunk's record), N, B, gamma -> the block record
//   gdn_scan_kernel  (sequence, v head, 64-column dv tile): walks the blocks in
//                    order, fp32 state tile in registers, one M = 128, N = 64,
//                    K = 128 tcgen05 product per block; stores the fp16 state
//                    entering each block
//   gdn_out_kernel   (block, v head): V_new, Y, then O in one accumulator
// All products are tcgen05 (kind::f16, fp32 accumulation in tensor memory) on
// 128-byte-swizzled shared-memory operands; tiles arrive by bulk copy or TMA.
#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

constexpr int kC = 64;   // chunk
constexpr int kD = 128;  // dk = dv

__device__ __forceinline__ unsigned char* align1024(unsigned char* p) {
  return reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
}
// K-major operand: rows of 64 halves, 8-row atoms 1024 bytes apart.
__device__ __forceinline__ uint64_t kdesc(uint32_t a) { return sw128_desc(a, 16, 1024); }
// MN-major operand: k rows of 64 halves; 64-element MN blocks `lbo` bytes apart.
__device__ __forceinline__ uint64_t mdesc(uint32_t a, uint32_t lbo) {
  return sw128_desc(a, lbo, 1024);
}
// Byte offset of 16-byte chunk c (< 8) of row r in a 128-byte-swizzled tile.
__device__ __forceinline__ int sw_chunk(int r, int c) { return r * 128 + (((c ^ r) & 7) << 4); }

__device__ __forceinline__ void zero_bytes(unsigned char* p, int bytes, int tid, int nthreads) {
  for (int i = tid * 16; i < bytes; i += nthreads * 16)
    *reinterpret_cast<uint4*>(p + i) = make_uint4(0, 0, 0, 0);
}

// Eight fp16 values (one 16-byte chunk) as floats.
__device__ __forceinline__ void unpack8(const uint4& u, float* f) {
  const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 x = __half22float2(h[i]);
    f[2 * i] = x.x;
    f[2 * i + 1] = x.y;
  }
}

// Block-local context shared by the pair and output kernels.
struct BlockCtx {
  int n, b, hv, hq;
  long long t_seq, len, s1;
  bool has2;
  int rows;  // valid tokens in this block
};
__device__ __forceinline__ bool block_ctx(const FwdParams& p, const WsLayout& ws, BlockCtx* x) {
  x->hv = blockIdx.x % p.Hv;
  const long long bslot = blockIdx.x / p.Hv;
  if (!locate_block(p, ws, bslot, &x->n, &x->b)) return false;
  x->t_seq = p.cu_seqlens ? (long long)p.cu_seqlens[x->n] : (long long)x->n * p.T;
  x->len = p.cu_seqlens ? (long long)p.cu_seqlens[x->n + 1] - x->t_seq : (long long)p.T;
  const long long n_chunks = (x->len + kC - 1) / kC;
  x->has2 = 2ll * x->b + 1 < n_chunks;
  x->s1 = ws.first_slot(p, x->n) + 2ll * x->b;
  x->rows = (int)min((long long)kBlock, x->len - (long long)kBlock * x->b);
  x->hq = x->hv / (p.Hv / p.Hqk);
  return true;
}

// =============================================================================
// gdn_pair_kernel: one CTA (128 threads, thread d = tensor-memory lane d) per
// (block, v head).
// =============================================================================
struct PairLayout {
  static constexpr int kW2 = 0;        // W2^T [128][64] -> W2'^T; [W2; W1] is one M = 128 operand
  static constexpr int kW1 = 16384;    // W1^T [128][64]
  static constexpr int kK1 = 32768;    // Kt1 [2][64][64]
  static constexpr int kK2 = 49152;    // Kt2
  static constexpr int kU1 = 65536;    // U1^T [128][64]
  static constexpr int kU2 = 81920;    // U2^T -> U2'^T
  static constexpr int kX = 98304;     // X [64][64] fp16
  static constexpr int kBar = 106496;  // 2 mbarriers, tensor-memory address, abort flag
  static constexpr int kAlloc = kBar + 64 + 1024;
};

__global__ void __launch_bounds__(128, 2) gdn_pair_kernel(const FwdParams p, const WsLayout ws) {
  using Lo = PairLayout;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = align1024(smem_raw);
  const uint32_t sb = smem_u32(sm);
  uint64_t* bar_ld = reinterpret_cast<uint64_t*>(sm + Lo::kBar);
  uint64_t* bar_mma = bar_ld + 1;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bar_ld + 2);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  const int tid = threadIdx.x, warp = tid >> 5;

  GDN_PHASE_INIT;
  BlockCtx x;
  if (!block_ctx(p, ws, &x)) return;  // before any allocation
  const int Hv = p.Hv, hv = x.hv;
  const long long s1 = x.s1, s2 = x.s1 + 1;
  const float gl1 = ws.gv(s1, hv, Hv)[0];
  const float gl2 = x.has2 ? ws.gv(s2, hv, Hv)[0] : 1.f;

  if (tid == 0) {
    mbar_init(bar_ld, 1);
    mbar_init(bar_mma, 1);
    *s_abort = 0;
    mbar_fence_init();
    mbar_expect_tx(bar_ld, (x.has2 ? 6u : 3u) * 16384u);
    bulk_g2s(sm + Lo::kW1, ws.W(s1, hv, Hv), 16384, bar_ld);
    bulk_g2s(sm + Lo::kK1, ws.Kt(s1, hv, Hv), 16384, bar_ld);
    bulk_g2s(sm + Lo::kU1, ws.U(s1, hv, Hv), 16384, bar_ld);
    if (x.has2) {
      bulk_g2s(sm + Lo::kW2, ws.W(s2, hv, Hv), 16384, bar_ld);
      bulk_g2s(sm + Lo::kK2, ws.Kt(s2, hv, Hv), 16384, bar_ld);
      bulk_g2s(sm + Lo::kU2, ws.U(s2, hv, Hv), 16384, bar_ld);
    }
  }
  if (!x.has2) {  // a lone last chunk: the second chunk's tiles are zero
    zero_bytes(sm + Lo::kW2, 16384, tid, 128);
    zero_bytes(sm + Lo::kK2, 16384, tid, 128);
    zero_bytes(sm + Lo::kU2, 16384, tid, 128);
    fence_proxy_async();
  }
  __syncwarp();
  if (warp == 0) tmem_alloc(s_tmem, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t lane_addr = tmem + ((uint32_t)(32 * warp) << 16);
  const int d = tid;  // tensor-memory lane = row of every M = 128 result

  if (tid == 0 && !mbar_wait(bar_ld, 0, p.err)) *s_abort = 1;
  __syncthreads();
  if (!*s_abort) mbar_wait(bar_ld, 0, p.err);
  GDN_PHASE(53);  // records landed

  // ---- X' = [W2; W1] Kt1^T (M = 128, N = 64, K = dk): rows 0-63 are X -------
  if (tid == 0 && !*s_abort) {
    tc_fence_after();
    constexpr uint32_t id = idesc_f16(128, 64, false, true, false);
#pragma unroll
    for (int s = 0; s < kD / 16; ++s)
      tc_mma(tmem, mdesc(sb + Lo::kW2 + s * 2048, 16384),
             kdesc(sb + Lo::kK1 + (s >> 2) * 8192 + (s & 3) * 32), id, s > 0);
    tc_commit(bar_mma);
  }
  if (tid == 0 && !*s_abort && !mbar_wait(bar_mma, 0, p.err)) *s_abort = 1;
  __syncthreads();
  GDN_PHASE(54);  // X product
  if (!*s_abort) {
    mbar_wait(bar_mma, 0, p.err);
    tc_fence_after();
    if (warp < 2) {  // X row i = d (a chunk-2 token), 64 columns (chunk-1 tokens)
      float v[32];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        tmem_ld32(lane_addr + 32 * hh, v);
#pragma unroll
        for (int m = 0; m < 4; ++m)
          *reinterpret_cast<uint4*>(sm + Lo::kX + sw_chunk(d, 4 * hh + m)) =
              make_uint4(pack_f16(v[8 * m], v[8 * m + 1]), pack_f16(v[8 * m + 2], v[8 * m + 3]),
                         pack_f16(v[8 * m + 4], v[8 * m + 5]),
                         pack_f16(v[8 * m + 6], v[8 * m + 7]));
      }
    }
    fence_proxy_async();
  }
  tc_fence_before();
  __syncthreads();

  // ---- D_w = W1^T X^T, D_u = U1^T X^T (M = 128, N = 64, K = 64) -------------
  if (tid == 0 && !*s_abort) {
    tc_fence_after();
    constexpr uint32_t id = idesc_f16(128, 64, false, false, false);
#pragma unroll
    for (int s = 0; s < kC / 16; ++s)
      tc_mma(tmem, kdesc(sb + Lo::kW1 + s * 32), kdesc(sb + Lo::kX + s * 32), id, s > 0);
#pragma unroll
    for (int s = 0; s < kC / 16; ++s)
      tc_mma(tmem + 64, kdesc(sb + Lo::kU1 + s * 32), kdesc(sb + Lo::kX + s * 32), id, s > 0);
    tc_commit(bar_mma);
  }
  GDN_PHASE(55);  // X stored
  if (tid == 0 && !*s_abort && !mbar_wait(bar_mma, 1, p.err)) *s_abort = 1;
  __syncthreads();
  GDN_PHASE(56);  // D_w, D_u products
  if (!*s_abort) {
    mbar_wait(bar_mma, 1, p.err);
    tc_fence_after();
    // row d: W2'^T = gamma_last1 W2^T - D_w, U2'^T = U2^T - D_u in place (then
    // copied to the second chunk's record); W1^T, U1^T scaled by gamma_last2
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float dw[32], du[32];
      tmem_ld32(lane_addr + 32 * hh, dw);
      tmem_ld32(lane_addr + 64 + 32 * hh, du);
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int c = 4 * hh + m, off = sw_chunk(d, c);
        float f[8];
        uint4* w2 = reinterpret_cast<uint4*>(sm + Lo::kW2 + off);
        unpack8(*w2, f);
        const uint4 w2n = make_uint4(pack_f16(gl1 * f[0] - dw[8 * m], gl1 * f[1] - dw[8 * m + 1]),
                                     pack_f16(gl1 * f[2] - dw[8 * m + 2], gl1 * f[3] - dw[8 * m + 3]),
                                     pack_f16(gl1 * f[4] - dw[8 * m + 4], gl1 * f[5] - dw[8 * m + 5]),
                                     pack_f16(gl1 * f[6] - dw[8 * m + 6], gl1 * f[7] - dw[8 * m + 7]));
        *w2 = w2n;
        uint4* u2 = reinterpret_cast<uint4*>(sm + Lo::kU2 + off);
        unpack8(*u2, f);
        const uint4 u2n = make_uint4(pack_f16(f[0] - du[8 * m], f[1] - du[8 * m + 1]),
                                     pack_f16(f[2] - du[8 * m + 2], f[3] - du[8 * m + 3]),
                                     pack_f16(f[4] - du[8 * m + 4], f[5] - du[8 * m + 5]),
                                     pack_f16(f[6] - du[8 * m + 6], f[7] - du[8 * m + 7]));
        *u2 = u2n;
        uint4* w1 = reinterpret_cast<uint4*>(sm + Lo::kW1 + off);
        unpack8(*w1, f);
        *w1 = make_uint4(pack_f16(gl2 * f[0], gl2 * f[1]), pack_f16(gl2 * f[2], gl2 * f[3]),
                         pack_f16(gl2 * f[4], gl2 * f[5]), pack_f16(gl2 * f[6], gl2 * f[7]));
        uint4* u1 = reinterpret_cast<uint4*>(sm + Lo::kU1 + off);
        unpack8(*u1, f);
        *u1 = make_uint4(pack_f16(gl2 * f[0], gl2 * f[1]), pack_f16(gl2 * f[2], gl2 * f[3]),
                         pack_f16(gl2 * f[4], gl2 * f[5]), pack_f16(gl2 * f[6], gl2 * f[7]));
      }
    }
    fence_proxy_async();
  }
  tc_fence_before();
  __syncthreads();

  // ---- N = [Kt1; Kt2]^T R, B = [Kt1; Kt2]^T U' (M = 128, N = 128, K = 128) ----
  if (tid == 0 && !*s_abort) {
    if (x.has2) {  // W2', U2' into the second chunk's record (the output kernel reads them)
      bulk_s2g(ws.W(s2, hv, Hv), sm + Lo::kW2, 16384);
      bulk_s2g(ws.U(s2, hv, Hv), sm + Lo::kU2, 16384);
      bulk_commit();
    }
    tc_fence_after();
    constexpr uint32_t id = idesc_f16(128, 128, false, true, false);
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const uint32_t kt = sb + (s < 4 ? Lo::kK1 : Lo::kK2) + (s & 3) * 2048;
      tc_mma(tmem, mdesc(kt, 8192), kdesc(sb + (s < 4 ? Lo::kW1 : Lo::kW2) + (s & 3) * 32), id,
             s > 0);
    }
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const uint32_t kt = sb + (s < 4 ? Lo::kK1 : Lo::kK2) + (s & 3) * 2048;
      tc_mma(tmem + 128, mdesc(kt, 8192), kdesc(sb + (s < 4 ? Lo::kU1 : Lo::kU2) + (s & 3) * 32),
             id, s > 0);
    }
    tc_commit(bar_mma);
  }
  GDN_PHASE(57);  // W2', U2' formed
  if (tid == 0 && !*s_abort && !mbar_wait(bar_mma, 0, p.err)) *s_abort = 1;
  if (tid == 0) bulk_wait_read<0>();  // W2', U2' tiles read out: the staging may reuse them
  __syncthreads();
  GDN_PHASE(58);  // N, B products
  const long long bs = ws.first_bslot(p, x.n) + x.b;
  if (!*s_abort) {
    mbar_wait(bar_mma, 0, p.err);
    tc_fence_after();
    // staged in the dead operand tiles in the record layout, then one bulk store each
    unsigned char* ng = sm + Lo::kW2;  // 32 KB: W2^T, W1^T
    unsigned char* bg = sm + Lo::kK1;  // 32 KB: Kt1, Kt2
#pragma unroll
    for (int q4 = 0; q4 < 8; ++q4) {  // 32 columns at a time: N (0-127), then B (128-255)
      float v[32];
      tmem_ld32(lane_addr + 32 * q4, v);
      unsigned char* dst = q4 < 4 ? ng : bg;
      const int col0 = 32 * (q4 & 3);  // column within the 128-wide matrix
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int col = col0 + 8 * m;
        *reinterpret_cast<uint4*>(dst + (col >> 6) * 16384 + sw_chunk(d, (col & 63) >> 3)) =
            make_uint4(pack_f16(v[8 * m], v[8 * m + 1]), pack_f16(v[8 * m + 2], v[8 * m + 3]),
                       pack_f16(v[8 * m + 4], v[8 * m + 5]), pack_f16(v[8 * m + 6], v[8 * m + 7]));
      }
    }
    fence_proxy_async();
  }
  __syncthreads();
  if (tid == 0 && !*s_abort) {
    bulk_s2g(ws.PN(bs, hv, Hv), sm + Lo::kW2, 32768);
    bulk_s2g(ws.PB(bs, hv, Hv), sm + Lo::kK1, 32768);
    bulk_commit();
    *ws.PG(bs, hv, Hv) = gl1 * gl2;
  }
  if (tid == 0) bulk_wait<0>();
  GDN_PHASE(59);  // N, B stored
  if (*s_abort && tid == 0) mbar_wait(bar_ld, 0, nullptr);  // copies in flight land first
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

// =============================================================================
// gdn_scan_kernel: one CTA per (sequence, v head, 64-column dv tile).  Warps
// 0-3: thread d holds row d of the fp32 state tile; warp 4 stages each block's
// N, B tile and gamma three blocks ahead.  Per block: one elected thread issues
// D = N h (8 MMAs, the fp16 state tile as the MN-major B operand) and then a
// bulk store of that same tile (the state entering the block, for the output
// kernel), which runs beside the product; every thread then forms
// h <- gamma h - D + B in fp32 and writes the fp16 copy into the next of three
// tile buffers.  One CTA barrier per block.
// =============================================================================
struct ScanLayout {
  static constexpr int kStages = 3;
  static constexpr int kHBufs = 3;
  static constexpr int kN = 0;          // per stage: N [2][128][64] fp16
  static constexpr int kB = 32768;      //            B tile [128][64] fp16
  static constexpr int kG = 49152;      //            gamma (16 bytes)
  static constexpr int kStage = 50176;  // 49 KB, 1024-aligned
  static constexpr int kH = kStages * kStage;  // fp16 state tiles [kHBufs][128][64]
  static constexpr int kBar = kH + kHBufs * 16384;
  static constexpr int kAlloc = kBar + 8 * (2 * kStages + 1) + 16 + 1024;
  static constexpr unsigned kTx = 32768 + 16384 + 16;
};

__device__ __forceinline__ uint4 pack8_h(const float* h) {
  return make_uint4(pack_f16(h[0], h[1]), pack_f16(h[2], h[3]), pack_f16(h[4], h[5]),
                    pack_f16(h[6], h[7]));
}

__global__ void __launch_bounds__(160, 1) gdn_scan_kernel(const FwdParams p, const WsLayout ws) {
  using Lo = ScanLayout;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = align1024(smem_raw);
  const uint32_t sb = smem_u32(sm);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + Lo::kBar);
  uint64_t* empty = full + Lo::kStages;
  uint64_t* bar_mma = empty + Lo::kStages;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bar_mma + 1);
  volatile int* s_stop = reinterpret_cast<volatile int*>(s_tmem + 1);  // any wait gave up
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  GDN_PHASE_INIT;
  const int j = blockIdx.x & 1;
  const int hv = (blockIdx.x >> 1) % p.Hv;
  const int n = (blockIdx.x >> 1) / p.Hv;
  const int Hv = p.Hv;
  const long long t_seq = p.cu_seqlens ? (long long)p.cu_seqlens[n] : (long long)n * p.T;
  const long long len = p.cu_seqlens ? (long long)p.cu_seqlens[n + 1] - t_seq : (long long)p.T;
  const int n_blocks = (int)((len + kBlock - 1) / kBlock);
  const long long bs0 = ws.first_bslot(p, n);

  if (tid == 0) {
    for (int i = 0; i < Lo::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 4);
    }
    mbar_init(bar_mma, 1);
    *s_stop = 0;
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(s_tmem, 64);

  // ---- initial state: registers and the first fp16 tile ---------------------
  float h[64];
  const int d = tid;
  if (warp < 4) {
    const float* h0 = p.h0 ? p.h0 + ((long long)(n * Hv + hv) * kD + d) * kD + 64 * j : nullptr;
#pragma unroll
    for (int c = 0; c < 64; c += 4) {
      const float4 v = h0 ? *reinterpret_cast<const float4*>(h0 + c) : make_float4(0, 0, 0, 0);
      h[c] = v.x; h[c + 1] = v.y; h[c + 2] = v.z; h[c + 3] = v.w;
    }
#pragma unroll
    for (int c = 0; c < 8; ++c)
      *reinterpret_cast<uint4*>(sm + Lo::kH + sw_chunk(d, c)) = pack8_h(h + 8 * c);
    fence_proxy_async();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  GDN_PHASE(44);  // setup

  if (warp == 4) {
    // ======================= producer =======================================
    if (lane == 0) {
      for (int bb = 0; bb < n_blocks; ++bb) {
        const int st = bb % Lo::kStages;
        if (bb >= Lo::kStages && !mbar_wait(&empty[st], ((bb / Lo::kStages) - 1) & 1, p.err)) {
          *s_stop = 1;
          break;
        }
        unsigned char* stage = sm + st * Lo::kStage;
        mbar_expect_tx(&full[st], Lo::kTx);
        bulk_g2s(stage + Lo::kN, ws.PN(bs0 + bb, hv, Hv), 32768, &full[st]);
        bulk_g2s(stage + Lo::kB, reinterpret_cast<unsigned char*>(ws.PB(bs0 + bb, hv, Hv)) + j * 16384,
                 16384, &full[st]);
        bulk_g2s(stage + Lo::kG, ws.PG(bs0 + bb, hv, Hv), 16, &full[st]);
      }
    }
    return;
  }

  // ========================= state warps ====================================
  // A thread whose wait gives up raises s_stop; every state thread reads it
  // after the step's barrier, so all leave the loop together.
  constexpr uint32_t id = idesc_f16(128, 64, false, false, true);
  const uint32_t lane_addr = tmem + ((uint32_t)(32 * warp) << 16);
  bool ok = true;
  int bb = 0;
  for (; bb < n_blocks; ++bb) {
    const int st = bb % Lo::kStages;
    const unsigned char* stage = sm + st * Lo::kStage;
    const int hb = bb % Lo::kHBufs;
    ok = mbar_wait(&full[st], (bb / Lo::kStages) & 1, p.err);
    GDN_PHASE(45);  // staged block landed
    if (warp == 0) {  // the rest of warp 0 waits here, not in a spin beside the issuer
      if (lane == 0 && ok) {
        tc_fence_after();
        const uint32_t hcur = sb + Lo::kH + hb * 16384;
#pragma unroll
        for (int s = 0; s < kD / 16; ++s)
          tc_mma(tmem, kdesc(sb + st * Lo::kStage + Lo::kN + (s >> 2) * 16384 + (s & 3) * 32),
                 mdesc(hcur + s * 2048, 16384), id, s > 0);
        tc_commit(bar_mma);
        // the state entering this block, for the output kernel (beside the product)
        bulk_s2g(reinterpret_cast<unsigned char*>(ws.PH(bs0 + bb, hv, Hv)) + j * 16384,
                 sm + Lo::kH + hb * 16384, 16384);
        bulk_commit();
      }
      __syncwarp();
    }
    GDN_PHASE(46);  // product issued
    // B row d and gamma while the product runs
    uint4 braw[8];
#pragma unroll
    for (int c = 0; c < 8; ++c)
      braw[c] = *reinterpret_cast<const uint4*>(stage + Lo::kB + sw_chunk(d, c));
    const float gam = *reinterpret_cast<const float*>(stage + Lo::kG);
    GDN_PHASE(47);  // B loaded
    if (ok) ok = mbar_wait(bar_mma, bb & 1, p.err);
    GDN_PHASE(48);  // product complete
    // the stage is consumed (N by the product, B and gamma by this warp)
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
    tc_fence_after();
    uint32_t dr[2][32];
    tmem_ld32_async(lane_addr, dr[0]);
    tmem_ld32_async(lane_addr + 32, dr[1]);
    tmem_ld_wait();
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        float bf[8];
        unpack8(braw[4 * hh + m], bf);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int c = 32 * hh + 8 * m + i;
          h[c] = fmaf(gam, h[c], bf[i] - __uint_as_float(dr[hh][8 * m + i]));
        }
      }
    GDN_PHASE(50);  // state update
    if (bb + 1 < n_blocks) {
      unsigned char* hnext = sm + Lo::kH + ((bb + 1) % Lo::kHBufs) * 16384;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(hnext + sw_chunk(d, c)) = pack8_h(h + 8 * c);
      fence_proxy_async();
    }
    GDN_PHASE(51);  // fp16 state tile written
    if (!ok) *s_stop = 1;
    // the tile written next step held the state entering block bb - 1: its bulk
    // store (issued a step ago) must have read it
    if (tid == 0) bulk_wait_read<1>();
    tc_fence_before();
    named_sync(1, 128);  // the fp16 tile is complete; tensor memory has been read
    GDN_PHASE(52);  // barrier
    if (*s_stop) break;
  }
  if (tid == 0 && *s_stop) {  // a wait gave up: let the copies already issued land
    for (int c = bb + 1; c < min(bb + Lo::kStages, n_blocks); ++c)
      mbar_wait(&full[c % Lo::kStages], (c / Lo::kStages) & 1, nullptr);
  }
  if (p.hT && !*s_stop) {
    float* hT = p.hT + ((long long)(n * Hv + hv) * kD + d) * kD + 64 * j;
#pragma unroll
    for (int c = 0; c < 64; c += 4)
      *reinterpret_cast<float4*>(hT + c) = make_float4(h[c], h[c + 1], h[c + 2], h[c + 3]);
  }
  if (tid == 0) bulk_wait<0>();
  tc_fence_before();
  named_sync(1, 128);
  if (warp == 0) tmem_dealloc(tmem, 64);
}

// =============================================================================
// gdn_out_kernel: one CTA (256 threads) per (block, v head).  Warp w reads
// tensor-memory lanes 32 (w % 4) + [0, 32) and column half w / 4.
// =============================================================================
struct OutLayout {
  static constexpr int kQ = 0;          // q [2][128][64] bf16 (TMA) -> fp16 * row scale
  static constexpr int kK1 = 32768;     // k of chunk 1 [2][64][64] bf16 (TMA)
  static constexpr int kH = 49152;      // state entering the block [2][128][64] fp16
  static constexpr int kW1 = 81920;     // W1^T [128][64]; W2'^T at +16384
  static constexpr int kW2 = 98304;
  static constexpr int kU1 = 114688;    // U1^T [128][64] -> V1^T; U2'^T -> V2^T at +16384
  static constexpr int kU2 = 131072;
  static constexpr int kP = 147456;     // P' [2][128][64] fp16
  static constexpr int kVec = 180224;   // row scales [128], e1 [64], Y row scales [64]
  static constexpr int kOPitch = 272;   // o staging rows (in the q and k tiles)
  static constexpr int kBar = kVec + 1024;
  static constexpr int kAlloc = kBar + 64 + 1024;
};

__global__ void __launch_bounds__(256, 1)
    gdn_out_kernel(const FwdParams p, const WsLayout ws, const __grid_constant__ CUtensorMap tmq,
                   const __grid_constant__ CUtensorMap tmk) {
  using Lo = OutLayout;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = align1024(smem_raw);
  const uint32_t sb = smem_u32(sm);
  float* s_rs = reinterpret_cast<float*>(sm + Lo::kVec);  // scale gamma' (q rows)
  float* s_e1 = s_rs + 128;                               // e of chunk 1 (k columns)
  float* s_ys = s_e1 + 64;                                // scale gamma2 (Y rows)
  uint64_t* bar_ld = reinterpret_cast<uint64_t*>(sm + Lo::kBar);  // operands of the first products
  uint64_t* bar_ld2 = bar_ld + 1;                                   // U tiles and P
  uint64_t* bar_mma = bar_ld + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bar_ld + 3);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  GDN_PHASE_INIT;
  BlockCtx x;
  if (!block_ctx(p, ws, &x)) return;
  const int Hv = p.Hv, hv = x.hv;
  const long long s1 = x.s1, s2 = x.s1 + 1;
  const long long bs = ws.first_bslot(p, x.n) + x.b;
  const int tok0 = (int)(x.t_seq + (long long)kBlock * x.b);  // row of the q/k tensor maps

  if (tid == 0) {
    mbar_init(bar_ld, 1);
    mbar_init(bar_ld2, 1);
    mbar_init(bar_mma, 1);
    *s_abort = 0;
    mbar_fence_init();
    mbar_expect_tx(bar_ld, 32768u + 16384u + 32768u + 16384u + (x.has2 ? 16384u : 0u));
    mbar_expect_tx(bar_ld2, 16384u + 8192u + (x.has2 ? 24576u : 0u));
#pragma unroll
    for (int kb = 0; kb < 2; ++kb) {
      tma_load_2d(sm + Lo::kQ + kb * 16384, &tmq, x.hq * kD + kb * 64, tok0, bar_ld);
      tma_load_2d(sm + Lo::kQ + kb * 16384 + 8192, &tmq, x.hq * kD + kb * 64, tok0 + 64, bar_ld);
      tma_load_2d(sm + Lo::kK1 + kb * 8192, &tmk, x.hq * kD + kb * 64, tok0, bar_ld);
    }
    bulk_g2s(sm + Lo::kH, ws.PH(bs, hv, Hv), 32768, bar_ld);
    bulk_g2s(sm + Lo::kW1, ws.W(s1, hv, Hv), 16384, bar_ld);
    if (x.has2) bulk_g2s(sm + Lo::kW2, ws.W(s2, hv, Hv), 16384, bar_ld);
    bulk_g2s(sm + Lo::kU1, ws.U(s1, hv, Hv), 16384, bar_ld2);
    bulk_g2s(sm + Lo::kP, ws.P(s1, hv, Hv), 8192, bar_ld2);
    if (x.has2) {
      bulk_g2s(sm + Lo::kU2, ws.U(s2, hv, Hv), 16384, bar_ld2);
      bulk_g2s(sm + Lo::kP + 16384 + 8192, ws.P(s2, hv, Hv), 8192, bar_ld2);
    }
  }
  // P' upper-right block (chunk-1 rows, chunk-2 columns) is zero; so is every
  // chunk-2 tile of a lone last chunk
  zero_bytes(sm + Lo::kP + 16384, 8192, tid, 256);
  if (!x.has2) {
    zero_bytes(sm + Lo::kW2, 16384, tid, 256);
    zero_bytes(sm + Lo::kU2, 16384, tid, 256);
    zero_bytes(sm + Lo::kP + 16384 + 8192, 8192, tid, 256);
  }
  if (tid < 64) {
    const float* gv1 = ws.gv(s1, hv, Hv);
    const float gl1 = gv1[0];
    s_rs[tid] = p.scale * gv1[4 + tid];
    s_e1[tid] = gv1[68 + tid];
    if (x.has2) {
      const float g2 = ws.gv(s2, hv, Hv)[4 + tid];
      s_rs[64 + tid] = p.scale * g2 * gl1;
      s_ys[tid] = p.scale * g2;
    } else {
      s_rs[64 + tid] = 0.f;
      s_ys[tid] = 0.f;
    }
  }
  fence_proxy_async();
  __syncwarp();
  if (warp == 0) tmem_alloc(s_tmem, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const int q4 = warp & 3, hh = warp >> 2;
  const uint32_t lane_addr = tmem + ((uint32_t)(32 * q4) << 16);

  if (tid == 0 && !mbar_wait(bar_ld, 0, p.err)) *s_abort = 1;
  __syncthreads();
  if (!*s_abort) mbar_wait(bar_ld, 0, p.err);
  GDN_PHASE(60);  // tiles landed

  // ---- D_V = h^T W'^T (M = dv, N = 128 tokens); Z = Q2 K1^T (M = 64, bf16) ---
  if (tid == 0 && !*s_abort) {
    tc_fence_after();
    constexpr uint32_t idv = idesc_f16(128, 128, false, true, true);
#pragma unroll
    for (int s = 0; s < kD / 16; ++s)
      tc_mma(tmem, mdesc(sb + Lo::kH + s * 2048, 16384), mdesc(sb + Lo::kW1 + s * 2048, 16384), idv,
             s > 0);
    constexpr uint32_t idz = idesc_f16(64, 64, true, false, false);
#pragma unroll
    for (int s = 0; s < kD / 16; ++s)
      tc_mma(tmem + 128, kdesc(sb + Lo::kQ + (s >> 2) * 16384 + 8192 + (s & 3) * 32),
             kdesc(sb + Lo::kK1 + (s >> 2) * 8192 + (s & 3) * 32), idz, s > 0);
    tc_commit(bar_mma);
  }
  // meanwhile: q rows 0-63 -> fp16 times scale gamma' (rows 64-127 still feed Z)
  if (!*s_abort) {
    for (int e = tid; e < 64 * 16; e += 256) {
      const int r = e >> 4, c = e & 15;
      bf16x8_to_f16x8_scaled(sm + Lo::kQ + (c >> 3) * 16384 + sw_chunk(r, c & 7), s_rs[r]);
    }
  }
  if (tid == 0 && !*s_abort && !mbar_wait(bar_mma, 0, p.err)) *s_abort = 1;
  if (tid == 0 && !*s_abort && !mbar_wait(bar_ld2, 0, p.err)) *s_abort = 1;
  __syncthreads();
  GDN_PHASE(61);  // V, Z products (and q rows 0-63)
  if (!*s_abort) {
    mbar_wait(bar_mma, 0, p.err);
    mbar_wait(bar_ld2, 0, p.err);
    tc_fence_after();
    {  // V^T row dv = 32 q4 + lane, tokens of chunk hh: V^T = U'^T - D_V, in place
      const int dvr = 32 * q4 + lane;
      unsigned char* ut = sm + (hh ? Lo::kU2 : Lo::kU1);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float v[32];
        tmem_ld32(lane_addr + 64 * hh + 32 * half, v);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          uint4* u = reinterpret_cast<uint4*>(ut + sw_chunk(dvr, 4 * half + m));
          float f[8];
          unpack8(*u, f);
          *u = make_uint4(pack_f16(f[0] - v[8 * m], f[1] - v[8 * m + 1]),
                          pack_f16(f[2] - v[8 * m + 2], f[3] - v[8 * m + 3]),
                          pack_f16(f[4] - v[8 * m + 4], f[5] - v[8 * m + 5]),
                          pack_f16(f[6] - v[8 * m + 6], f[7] - v[8 * m + 7]));
        }
      }
    }
    {  // Y (M = 64 layout: lanes 32 q4 + i, i < 16, hold row 16 q4 + i); columns 32 hh..
      float v[32];
      tmem_ld32(lane_addr + 128 + 32 * hh, v);
      if (lane < 16) {
        const int i2 = 16 * q4 + lane, r = 64 + i2;
        const float ys = s_ys[i2];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int c0 = 32 * hh + 8 * m;
          float y[8];
#pragma unroll
          for (int t = 0; t < 8; ++t) y[t] = ys * v[8 * m + t] * s_e1[c0 + t];
          *reinterpret_cast<uint4*>(sm + Lo::kP + sw_chunk(r, c0 >> 3)) =
              make_uint4(pack_f16(y[0], y[1]), pack_f16(y[2], y[3]), pack_f16(y[4], y[5]),
                         pack_f16(y[6], y[7]));
        }
      }
    }
    for (int e = tid; e < 64 * 16; e += 256) {  // q rows 64-127 (Z has read them)
      const int r = 64 + (e >> 4), c = e & 15;
      bf16x8_to_f16x8_scaled(sm + Lo::kQ + (c >> 3) * 16384 + sw_chunk(r, c & 7), s_rs[r]);
    }
    fence_proxy_async();
  }
  tc_fence_before();
  __syncthreads();

  // ---- O = (diag(scale gamma') Q) h + P' V (M = 128 tokens, N = dv) ----------
  if (tid == 0 && !*s_abort) {
    tc_fence_after();
    constexpr uint32_t idq = idesc_f16(128, 128, false, false, true);
#pragma unroll
    for (int s = 0; s < kD / 16; ++s)
      tc_mma(tmem, kdesc(sb + Lo::kQ + (s >> 2) * 16384 + (s & 3) * 32),
             mdesc(sb + Lo::kH + s * 2048, 16384), idq, s > 0);
    constexpr uint32_t idp = idesc_f16(128, 128, false, false, false);
#pragma unroll
    for (int s = 0; s < kBlock / 16; ++s)
      tc_mma(tmem, kdesc(sb + Lo::kP + (s >> 2) * 16384 + (s & 3) * 32),
             kdesc(sb + Lo::kU1 + (s >> 2) * 16384 + (s & 3) * 32), idp, true);
    tc_commit(bar_mma);
  }
  GDN_PHASE(62);  // V, Y, q rows 64-127 stored
  if (tid == 0 && !*s_abort && !mbar_wait(bar_mma, 1, p.err)) *s_abort = 1;
  __syncthreads();
  GDN_PHASE(63);  // O product
  if (!*s_abort) {
    mbar_wait(bar_mma, 1, p.err);
    tc_fence_after();
    // o rows staged in the dead q / k tiles (272-byte row pitch: conflict-free),
    // then one 256-byte bulk store per valid token row
    const int i = 32 * q4 + lane;  // token row of the block
    unsigned char* row = sm + Lo::kQ + i * Lo::kOPitch + 128 * hh;
    uint32_t r[2][32];
    tmem_ld32_async(lane_addr + 64 * hh, r[0]);
    tmem_ld32_async(lane_addr + 64 * hh + 32, r[1]);
    tmem_ld_wait();
#pragma unroll
    for (int half = 0; half < 2; ++half)
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const uint32_t* v = r[half] + 8 * m;
        *reinterpret_cast<uint4*>(row + 64 * half + 16 * m) = make_uint4(
            pack_bf16(__uint_as_float(v[0]), __uint_as_float(v[1])),
            pack_bf16(__uint_as_float(v[2]), __uint_as_float(v[3])),
            pack_bf16(__uint_as_float(v[4]), __uint_as_float(v[5])),
            pack_bf16(__uint_as_float(v[6]), __uint_as_float(v[7])));
      }
    fence_proxy_async();
  }
  __syncthreads();
  if (!*s_abort && tid < x.rows) {
    bulk_s2g(static_cast<__nv_bfloat16*>(p.o) + ((long long)(tok0 + tid) * Hv + hv) * kD,
             sm + Lo::kQ + tid * Lo::kOPitch, 256);
    bulk_commit();
    bulk_wait<0>();
  }
  GDN_PHASE(39);  // O stored
  if (*s_abort && tid == 0) {
    mbar_wait(bar_ld, 0, nullptr);
    mbar_wait(bar_ld2, 0, nullptr);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

}  // namespace

cudaError_t launch_pair(const FwdParams& p, const WsLayout& ws, cudaStream_t stream) {
  cudaError_t e = set_smem(gdn_pair_kernel, PairLayout::kAlloc);
  if (e != cudaSuccess) return e;
  const long long grid = ws.n_bslots * p.Hv;
  gdn_pair_kernel<<<(unsigned)grid, 128, PairLayout::kAlloc, stream>>>(p, ws);
  return cudaGetLastError();
}

cudaError_t launch_scan(const FwdParams& p, const WsLayout& ws, cudaStream_t stream) {
  cudaError_t e = set_smem(gdn_scan_kernel, ScanLayout::kAlloc);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)p.N * p.Hv * 2;
  gdn_scan_kernel<<<(unsigned)grid, 160, ScanLayout::kAlloc, stream>>>(p, ws);
  return cudaGetLastError();
}

cudaError_t launch_out(const FwdParams& p, const WsLayout& ws, cudaStream_t stream) {
  const long long rows = p.cu_seqlens ? (long long)p.T : (long long)p.N * p.T;
  CUtensorMap mq, mk;
  if (!make_tensor_map_bf16(&mq, p.q, rows, (long long)p.Hqk * kD) ||
      !make_tensor_map_bf16(&mk, p.k, rows, (long long)p.Hqk * kD))
    return cudaErrorInvalidValue;
  cudaError_t e = set_smem(gdn_out_kernel, OutLayout::kAlloc);
  if (e != cudaSuccess) return e;
  const long long grid = ws.n_bslots * p.Hv;
  gdn_out_kernel<<<(unsigned)grid, 256, OutLayout::kAlloc, stream>>>(p, ws, mq, mk);
  return cudaGetLastError();
}

}  // namespace gdn
