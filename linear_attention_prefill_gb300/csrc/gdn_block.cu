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
// Three stages, as three launches or (fixed-length rows) one:
//   pair task   (block, v head): X, W2', U2' (written back into the second
//               chunk's record), N, B, gamma -> the block record
//   scan chain  (sequence, v head, 64-column dv tile): walks the blocks in
//               order, fp32 state tile in registers, one M = 128, N = 64,
//               K = 128 tcgen05 product per block; stores the fp16 state
//               entering each block
//   out task    (block, v head): V_new, Y, then O in one accumulator
// gdn_pair_kernel, gdn_scan_kernel and gdn_out_kernel run one stage each;
// gdn_scanout_kernel runs the scan chains beside worker CTAs that take the
// pair and out tasks in block order, synchronised by per-block flags.
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

__device__ __forceinline__ uint4 pack8_h(const float* h) {
  return make_uint4(pack_f16(h[0], h[1]), pack_f16(h[2], h[3]), pack_f16(h[4], h[5]),
                    pack_f16(h[6], h[7]));
}

// Release store / acquire load of a flag word in global memory, and the
// generic <-> async proxy ordering for global memory.
__device__ __forceinline__ void flag_release(unsigned* f, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;\n" ::"l"(f), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned flag_acquire(const unsigned* f) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(f) : "memory");
  return v;
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;\n" ::: "memory");
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
// Pair transition: one task per (block, v head), 128 or 256 threads.  Thread
// (warp w, lane l) owns tensor-memory lane / result row d = 32 (w % 4) + l;
// with 256 threads warps w and w + 4 split each row's columns (or its tiles).
// =============================================================================
struct PairLayout {
  static constexpr int kW2 = 0;        // W2^T [128][64] -> W2'^T; [W2; W1] is one M = 128 operand
  static constexpr int kW1 = 16384;    // W1^T [128][64]
  static constexpr int kK1 = 32768;    // Kt1 [2][64][64]
  static constexpr int kK2 = 49152;    // Kt2
  static constexpr int kU1 = 65536;    // U1^T [128][64]
  static constexpr int kU2 = 81920;    // U2^T -> U2'^T
  static constexpr int kX = 98304;     // X [64][64] fp16
  static constexpr int kBar = 106496;  // barriers of the stand-alone kernel
  static constexpr int kAlloc = kBar + 64 + 1024;
};

struct PairBars {
  uint64_t* ld;
  uint64_t* mma;  // three completions per task
  volatile int* abort;
};

// Scales the 8 fp16 values of a 16-byte chunk in place.
__device__ __forceinline__ void scale_chunk(uint4* c, float g) {
  float f[8];
  unpack8(*c, f);
  *c = make_uint4(pack_f16(g * f[0], g * f[1]), pack_f16(g * f[2], g * f[3]),
                  pack_f16(g * f[4], g * f[5]), pack_f16(g * f[6], g * f[7]));
}

// One pair task.  With `pending` (worker CTAs), thread 0 leaves the block's
// flag in *pending: it is set (flush_pending) once the block record and the
// rewritten chunk-2 tiles are complete in global memory, at the start of the
// worker's next task, when the stores have normally long landed.
__device__ __forceinline__ void pair_task(const FwdParams& p, const WsLayout& ws, unsigned char* sm,
                                          const PairBars& bars, uint32_t tmem, const BlockCtx& x,
                                          int it, unsigned** pending) {
  using Lo = PairLayout;
  const uint32_t sb = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nt = blockDim.x;           // 128 or 256
  const int q4 = warp & 3, ch = warp >> 2;
  const bool split = nt >= 256;        // column halves shared by warps w and w + 4
  GDN_PHASE_INIT;
  const int Hv = p.Hv, hv = x.hv;
  const long long s1 = x.s1, s2 = x.s1 + 1;
  const float gl1 = ws.gv(s1, hv, Hv)[0];
  const float gl2 = x.has2 ? ws.gv(s2, hv, Hv)[0] : 1.f;
  const unsigned ph = it & 1, m0 = (3 * it) & 1;  // load phase, first mma phase

  if (tid == 0) {
    *bars.abort = 0;
    mbar_expect_tx(bars.ld, (x.has2 ? 6u : 3u) * 16384u);
    bulk_g2s(sm + Lo::kW1, ws.W(s1, hv, Hv), 16384, bars.ld);
    bulk_g2s(sm + Lo::kK1, ws.Kt(s1, hv, Hv), 16384, bars.ld);
    bulk_g2s(sm + Lo::kU1, ws.U(s1, hv, Hv), 16384, bars.ld);
    if (x.has2) {
      bulk_g2s(sm + Lo::kW2, ws.W(s2, hv, Hv), 16384, bars.ld);
      bulk_g2s(sm + Lo::kK2, ws.Kt(s2, hv, Hv), 16384, bars.ld);
      bulk_g2s(sm + Lo::kU2, ws.U(s2, hv, Hv), 16384, bars.ld);
    }
  }
  if (!x.has2) {  // a lone last chunk: the second chunk's tiles are zero
    zero_bytes(sm + Lo::kW2, 16384, tid, nt);
    zero_bytes(sm + Lo::kK2, 16384, tid, nt);
    zero_bytes(sm + Lo::kU2, 16384, tid, nt);
    fence_proxy_async();
  }
  const uint32_t lane_addr = tmem + ((uint32_t)(32 * q4) << 16);
  const int d = 32 * q4 + lane;  // tensor-memory lane = row of every M = 128 result

  if (tid == 0 && !mbar_wait(bars.ld, ph, p.err)) *bars.abort = 1;
  __syncthreads();
  if (!*bars.abort) mbar_wait(bars.ld, ph, p.err);
  GDN_PHASE(53);  // records landed

  // ---- X' = [W2; W1] Kt1^T (M = 128, N = 64, K = dk): rows 0-63 are X -------
  if (tid == 0 && !*bars.abort) {
    tc_fence_after();
    constexpr uint32_t id = idesc_f16(128, 64, false, true, false);
#pragma unroll
    for (int s = 0; s < kD / 16; ++s)
      tc_mma(tmem, mdesc(sb + Lo::kW2 + s * 2048, 16384),
             kdesc(sb + Lo::kK1 + (s >> 2) * 8192 + (s & 3) * 32), id, s > 0);
    tc_commit(bars.mma);
  }
  if (tid == 0 && !*bars.abort && !mbar_wait(bars.mma, m0, p.err)) *bars.abort = 1;
  __syncthreads();
  GDN_PHASE(54);  // X product
  if (!*bars.abort) {
    mbar_wait(bars.mma, m0, p.err);
    tc_fence_after();
    if (q4 < 2) {  // X row i = d (a chunk-2 token), 64 columns (chunk-1 tokens)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        if (split && hh != ch) continue;
        float v[32];
        tmem_ld32(lane_addr + 32 * hh, v);
#pragma unroll
        for (int m = 0; m < 4; ++m)
          *reinterpret_cast<uint4*>(sm + Lo::kX + sw_chunk(d, 4 * hh + m)) = pack8_h(v + 8 * m);
      }
    }
    fence_proxy_async();
  }
  tc_fence_before();
  __syncthreads();
  GDN_PHASE(55);  // X stored

  // ---- D_w = W1^T X^T, D_u = U1^T X^T (M = 128, N = 64, K = 64) -------------
  if (tid == 0 && !*bars.abort) {
    tc_fence_after();
    constexpr uint32_t id = idesc_f16(128, 64, false, false, false);
#pragma unroll
    for (int s = 0; s < kC / 16; ++s)
      tc_mma(tmem, kdesc(sb + Lo::kW1 + s * 32), kdesc(sb + Lo::kX + s * 32), id, s > 0);
#pragma unroll
    for (int s = 0; s < kC / 16; ++s)
      tc_mma(tmem + 64, kdesc(sb + Lo::kU1 + s * 32), kdesc(sb + Lo::kX + s * 32), id, s > 0);
    tc_commit(bars.mma);
  }
  if (tid == 0 && !*bars.abort && !mbar_wait(bars.mma, m0 ^ 1, p.err)) *bars.abort = 1;
  __syncthreads();
  GDN_PHASE(56);  // D_w, D_u products
  if (!*bars.abort) {
    mbar_wait(bars.mma, m0 ^ 1, p.err);
    tc_fence_after();
    // row d: W2'^T = gamma_last1 W2^T - D_w, U2'^T = U2^T - D_u in place (then
    // copied to the second chunk's record); W1^T, U1^T scaled by gamma_last2
#pragma unroll
    for (int t = 0; t < 2; ++t) {  // t = 0: the W tiles, t = 1: the U tiles
      if (split && t != ch) continue;
      uint32_t r[2][32];
      tmem_ld32_async(lane_addr + 64 * t, r[0]);
      tmem_ld32_async(lane_addr + 64 * t + 32, r[1]);
      tmem_ld_wait();
      unsigned char* t2 = sm + (t ? Lo::kU2 : Lo::kW2);
      unsigned char* t1 = sm + (t ? Lo::kU1 : Lo::kW1);
      const float g2 = t ? 1.f : gl1;
      uint4 c2[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) c2[c] = *reinterpret_cast<const uint4*>(t2 + sw_chunk(d, c));
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        float f[8];
        unpack8(c2[c], f);
        const uint32_t* v = r[c >> 2] + 8 * (c & 3);
        *reinterpret_cast<uint4*>(t2 + sw_chunk(d, c)) =
            make_uint4(pack_f16(g2 * f[0] - __uint_as_float(v[0]), g2 * f[1] - __uint_as_float(v[1])),
                       pack_f16(g2 * f[2] - __uint_as_float(v[2]), g2 * f[3] - __uint_as_float(v[3])),
                       pack_f16(g2 * f[4] - __uint_as_float(v[4]), g2 * f[5] - __uint_as_float(v[5])),
                       pack_f16(g2 * f[6] - __uint_as_float(v[6]), g2 * f[7] - __uint_as_float(v[7])));
        scale_chunk(reinterpret_cast<uint4*>(t1 + sw_chunk(d, c)), gl2);
      }
    }
    fence_proxy_async();
  }
  tc_fence_before();
  __syncthreads();
  GDN_PHASE(57);  // W2', U2' formed

  // ---- N = [Kt1; Kt2]^T R, B = [Kt1; Kt2]^T U' (M = 128, N = 128, K = 128) ----
  if (tid == 0 && !*bars.abort) {
    if (x.has2) {  // W2', U2' into the second chunk's record (the output stage reads them)
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
    tc_commit(bars.mma);
  }
  if (tid == 0 && !*bars.abort && !mbar_wait(bars.mma, m0, p.err)) *bars.abort = 1;
  if (tid == 0) bulk_wait_read<0>();  // W2', U2' tiles read out: the staging may reuse them
  __syncthreads();
  GDN_PHASE(58);  // N, B products
  const long long bs = ws.first_bslot(p, x.n) + x.b;
  if (!*bars.abort) {
    mbar_wait(bars.mma, m0, p.err);
    tc_fence_after();
    // staged in the dead operand tiles in the record layout, then one bulk store each
#pragma unroll
    for (int t = 0; t < 2; ++t) {  // t = 0: N (columns 0-127), t = 1: B (128-255)
      if (split && t != ch) continue;
      unsigned char* dst = sm + (t ? Lo::kK1 : Lo::kW2);  // 32 KB each: W2^T W1^T / Kt1 Kt2
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t r[2][32];
        tmem_ld32_async(lane_addr + 128 * t + 64 * q, r[0]);
        tmem_ld32_async(lane_addr + 128 * t + 64 * q + 32, r[1]);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t* v = r[c >> 2] + 8 * (c & 3);
          *reinterpret_cast<uint4*>(dst + q * 16384 + sw_chunk(d, c)) =
              make_uint4(pack_f16(__uint_as_float(v[0]), __uint_as_float(v[1])),
                         pack_f16(__uint_as_float(v[2]), __uint_as_float(v[3])),
                         pack_f16(__uint_as_float(v[4]), __uint_as_float(v[5])),
                         pack_f16(__uint_as_float(v[6]), __uint_as_float(v[7])));
        }
      }
    }
    fence_proxy_async();
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && !*bars.abort) {
    bulk_s2g(ws.PN(bs, hv, Hv), sm + Lo::kW2, 32768);
    bulk_s2g(ws.PB(bs, hv, Hv), sm + Lo::kK1, 32768);
    bulk_commit();
    *ws.PG(bs, hv, Hv) = gl1 * gl2;
  }
  if (tid == 0) {
    if (pending) {
      if (!*bars.abort) *pending = ws.pair_flags() + bs * Hv + hv;
      bulk_wait_read<0>();
    } else {
      bulk_wait_read<0>();  // the stand-alone kernel: only the staging must outlive the reads
    }
  }
  GDN_PHASE(59);  // N, B stored
  if (*bars.abort && tid == 0) mbar_wait(bars.ld, ph, nullptr);  // copies in flight land first
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

__global__ void __launch_bounds__(256, 2) gdn_pair_kernel(const FwdParams p, const WsLayout ws) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = align1024(smem_raw);
  BlockCtx x;
  if (!block_ctx(p, ws, &x)) return;  // before any allocation
  PairBars bars;
  bars.ld = reinterpret_cast<uint64_t*>(sm + PairLayout::kBar);
  bars.mma = bars.ld + 1;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars.ld + 2);
  bars.abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  if (threadIdx.x == 0) {
    mbar_init(bars.ld, 1);
    mbar_init(bars.mma, 1);
    mbar_fence_init();
  }
  if (threadIdx.x < 32) tmem_alloc(s_tmem, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pair_task(p, ws, sm, bars, *s_tmem, x, 0, nullptr);
  if (threadIdx.x < 32) tmem_dealloc(*s_tmem, 256);
}

// =============================================================================
// The block scan: one chain per (sequence, v head, 64-column dv tile).  Warps
// 0-3: thread d holds row d of the fp32 state tile; warp 4 stages each block's
// N, B tile and gamma three blocks ahead; warp 5 stores each fp16 state tile
// (the state entering a block, for the output stage) with a bulk copy.  Per
// block: one elected thread issues D = N h (8 MMAs, the fp16 state tile as the
// MN-major B operand); every state thread then forms h <- gamma h - D + B in
// fp32 and writes the fp16 copy into the next of three tile buffers.  One
// barrier among the state warps per block.  Tile k % 3 holding the state
// entering block k is handed to warp 5 through hrdy[k % 3] and handed back
// through hfree[k % 3]; each completes one phase per use of its tile, so no
// side can run two phases ahead.  With `flags`, warp 5 sets the word of
// (block, head, tile) once that block's stored state is complete in global
// memory (the output work may run concurrently).
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
  static constexpr int kBars = 2 * kStages + 1 + 2 * kHBufs;  // full, empty, mma, hrdy, hfree
  static constexpr int kAlloc = kBar + 8 * kBars + 16 + 1024;
  static constexpr unsigned kTx = 32768 + 16384 + 16;
  static constexpr int kThreads = 192;
};

// Flag waits: spin (bounded) until every word is non-zero; then order the
// async-proxy reads that follow.  Returns false (and records a timeout) if
// the words stay zero.
__device__ __forceinline__ bool wait_flags(const unsigned* f, int count, unsigned* err) {
  const long long t0 = clock64();
  for (int i = 0; i < count; ++i) {
    while (!flag_acquire(f + i)) {
      if (clock64() - t0 > (1ll << 31)) {
        if (err) atomicExch(err, kErrWaitTimeout);
        return false;
      }
    }
  }
  fence_proxy_async_global();
  return true;
}

// Sets the flag a finished pair task left behind, once its stores completed.
__device__ __forceinline__ void flush_pending(unsigned** pending) {
  if (*pending) {
    bulk_wait<0>();
    fence_proxy_async_global();
    flag_release(*pending, 1u);
    *pending = nullptr;
  }
}

// Threads 0-191 of the CTA take part; others must not call this.  With
// `pair_flags` the block records come from concurrent pair tasks: each block
// is staged only after its flag is set.
__device__ __forceinline__ void scan_chain(const FwdParams& p, const WsLayout& ws, unsigned char* sm,
                                           int chain, unsigned* flags, const unsigned* pair_flags) {
  using Lo = ScanLayout;
  const uint32_t sb = smem_u32(sm);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + Lo::kBar);
  uint64_t* empty = full + Lo::kStages;
  uint64_t* bar_mma = empty + Lo::kStages;
  uint64_t* hrdy = bar_mma + 1;
  uint64_t* hfree = hrdy + Lo::kHBufs;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(hfree + Lo::kHBufs);
  volatile int* s_stop = reinterpret_cast<volatile int*>(s_tmem + 1);  // any wait gave up
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  GDN_PHASE_INIT;
  const int j = chain & 1;
  const int hv = (chain >> 1) % p.Hv;
  const int n = (chain >> 1) / p.Hv;
  const int Hv = p.Hv;
  const long long t_seq = p.cu_seqlens ? (long long)p.cu_seqlens[n] : (long long)n * p.T;
  const long long len = p.cu_seqlens ? (long long)p.cu_seqlens[n + 1] - t_seq : (long long)p.T;
  const int n_blocks = (int)((len + kBlock - 1) / kBlock);
  const long long bs0 = ws.first_bslot(p, n);
  auto flag_of = [&](int bb) { return flags + ((bs0 + bb) * Hv + hv) * 2 + j; };

  if (tid == 0) {
    for (int i = 0; i < Lo::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 4);
    }
    mbar_init(bar_mma, 1);
    for (int i = 0; i < Lo::kHBufs; ++i) {
      mbar_init(&hrdy[i], 1);
      mbar_init(&hfree[i], 1);
    }
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
  named_sync(2, Lo::kThreads);
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  if (tid == 0 && n_blocks > 0) mbar_arrive(&hrdy[0]);  // tile 0 holds the initial state
  GDN_PHASE(44);  // setup

  if (warp == 5) {
    // ======================= state stores ===================================
    if (lane == 0) {
      for (int k = 0; k < n_blocks; ++k) {
        const int x = k % Lo::kHBufs, u = k / Lo::kHBufs;
        if (!mbar_wait(&hrdy[x], u & 1, p.err)) {
          *s_stop = 1;
          break;
        }
        bulk_s2g(reinterpret_cast<unsigned char*>(ws.PH(bs0 + k, hv, Hv)) + j * 16384,
                 sm + Lo::kH + x * 16384, 16384);
        bulk_commit();
        bulk_wait_read<0>();
        mbar_arrive(&hfree[x]);
        if (flags && k > 0) {  // the previous block's stored state is complete
          bulk_wait<1>();
          fence_proxy_async_global();
          flag_release(flag_of(k - 1), 1u);
        }
      }
      bulk_wait<0>();
      if (flags && n_blocks > 0 && !*s_stop) {
        fence_proxy_async_global();
        flag_release(flag_of(n_blocks - 1), 1u);
      }
    }
    return;
  }

  if (warp == 4) {
    // ======================= producer =======================================
    if (lane == 0) {
      for (int bb = 0; bb < n_blocks; ++bb) {
        const int st = bb % Lo::kStages;
        if (bb >= Lo::kStages && !mbar_wait(&empty[st], ((bb / Lo::kStages) - 1) & 1, p.err)) {
          *s_stop = 1;
          break;
        }
        if (pair_flags && !wait_flags(pair_flags + (bs0 + bb) * Hv + hv, 1, p.err)) {
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
      const int x = (bb + 1) % Lo::kHBufs;
      unsigned char* hnext = sm + Lo::kH + x * 16384;
      // the tile's previous state (entering block bb - 2) must have been read out
      if (bb >= 2 && ok) ok = mbar_wait(&hfree[x], ((bb + 1) / Lo::kHBufs - 1) & 1, p.err);
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(hnext + sw_chunk(d, c)) = pack8_h(h + 8 * c);
      fence_proxy_async();
    }
    GDN_PHASE(51);  // fp16 state tile written
    if (!ok) *s_stop = 1;
    tc_fence_before();
    named_sync(1, 128);  // the fp16 tile is complete; tensor memory has been read
    GDN_PHASE(52);  // barrier
    if (tid == 0 && bb + 1 < n_blocks) mbar_arrive(&hrdy[(bb + 1) % Lo::kHBufs]);
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
  tc_fence_before();
  named_sync(1, 128);
  if (warp == 0) tmem_dealloc(tmem, 64);
}

__global__ void __launch_bounds__(ScanLayout::kThreads, 1) gdn_scan_kernel(const FwdParams p,
                                                                          const WsLayout ws) {
  extern __shared__ unsigned char smem_raw[];
  scan_chain(p, ws, align1024(smem_raw), blockIdx.x, nullptr, nullptr);
}

// =============================================================================
// Block output: one task per (block, v head), 256 threads; warp w reads
// tensor-memory lanes 32 (w % 4) + [0, 32) and column half w / 4.  The caller
// owns the barriers and the 256 tensor-memory columns; `it` counts the tasks
// this CTA ran before (barrier phases).
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
  static constexpr int kAlloc = kBar + 128 + 1024;
};

struct OutBars {
  uint64_t* ld;    // W', q and k tiles
  uint64_t* ld2;   // U tiles and P
  uint64_t* ldh;   // the stored state entering the block
  uint64_t* mma;
  volatile int* abort;
};

__device__ __forceinline__ OutBars out_bars(unsigned char* sm) {
  OutBars b;
  b.ld = reinterpret_cast<uint64_t*>(sm + OutLayout::kBar);
  b.ld2 = b.ld + 1;
  b.ldh = b.ld + 2;
  b.mma = b.ld + 3;
  b.abort = reinterpret_cast<volatile int*>(b.ld + 5);
  return b;
}
__device__ __forceinline__ uint32_t* out_tmem_slot(unsigned char* sm) {
  return reinterpret_cast<uint32_t*>(sm + OutLayout::kBar + 32);
}
// The worker CTAs' pair-task barriers (beside the output ones).
__device__ __forceinline__ PairBars worker_pair_bars(unsigned char* sm) {
  PairBars b;
  b.ld = reinterpret_cast<uint64_t*>(sm + OutLayout::kBar + 48);
  b.mma = b.ld + 1;
  b.abort = reinterpret_cast<volatile int*>(b.ld + 2);
  return b;
}

// One block-output task; all 256 threads.  With `scan_flags` the state entering
// the block is loaded only once the scan has flagged it (every other operand is
// loaded first; with `pair_flags` those wait for the block's pair task), and
// `tmo` (a [N][T][Hv dv] map of o) stores the output tile by TMA; otherwise
// rows are stored one by one.  Returns false if a wait gave up.
__device__ __forceinline__ bool out_task(const FwdParams& p, const WsLayout& ws,
                                         const CUtensorMap* tmq, const CUtensorMap* tmk,
                                         const CUtensorMap* tmo, unsigned char* sm,
                                         const OutBars& bars, uint32_t tmem, const BlockCtx& x,
                                         int it, const unsigned* scan_flags,
                                         const unsigned* pair_flags) {
  using Lo = OutLayout;
  const uint32_t sb = smem_u32(sm);
  float* s_rs = reinterpret_cast<float*>(sm + Lo::kVec);  // scale gamma' (q rows)
  float* s_e1 = s_rs + 128;                               // e of chunk 1 (k columns)
  float* s_ys = s_e1 + 64;                                // scale gamma2 (Y rows)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  GDN_PHASE_INIT;
  const int Hv = p.Hv, hv = x.hv;
  const long long s1 = x.s1, s2 = x.s1 + 1;
  const long long bs = ws.first_bslot(p, x.n) + x.b;
  const int tok0 = (int)(x.t_seq + (long long)kBlock * x.b);  // row of the q/k tensor maps
  const unsigned ph = it & 1;

  if (tid == 0) {
    *bars.abort = 0;
    if (pair_flags && !wait_flags(pair_flags + bs * Hv + hv, 1, p.err)) *bars.abort = 1;
  }
  __syncthreads();
  if (*bars.abort) return false;
  if (tid == 0) {
    mbar_expect_tx(bars.ld, 32768u + 16384u + 16384u + (x.has2 ? 16384u : 0u));
    mbar_expect_tx(bars.ld2, 16384u + 8192u + (x.has2 ? 24576u : 0u));
#pragma unroll
    for (int kb = 0; kb < 2; ++kb) {
      tma_load_2d(sm + Lo::kQ + kb * 16384, tmq, x.hq * kD + kb * 64, tok0, bars.ld);
      tma_load_2d(sm + Lo::kQ + kb * 16384 + 8192, tmq, x.hq * kD + kb * 64, tok0 + 64, bars.ld);
      tma_load_2d(sm + Lo::kK1 + kb * 8192, tmk, x.hq * kD + kb * 64, tok0, bars.ld);
    }
    bulk_g2s(sm + Lo::kW1, ws.W(s1, hv, Hv), 16384, bars.ld);
    if (x.has2) bulk_g2s(sm + Lo::kW2, ws.W(s2, hv, Hv), 16384, bars.ld);
    bulk_g2s(sm + Lo::kU1, ws.U(s1, hv, Hv), 16384, bars.ld2);
    bulk_g2s(sm + Lo::kP, ws.P(s1, hv, Hv), 8192, bars.ld2);
    if (x.has2) {
      bulk_g2s(sm + Lo::kU2, ws.U(s2, hv, Hv), 16384, bars.ld2);
      bulk_g2s(sm + Lo::kP + 16384 + 8192, ws.P(s2, hv, Hv), 8192, bars.ld2);
    }
    // the scan may store this block's entering state concurrently
    const bool ready = !scan_flags || wait_flags(scan_flags + (bs * Hv + hv) * 2, 2, p.err);
    mbar_expect_tx(bars.ldh, 32768u);
    if (ready) {
      bulk_g2s(sm + Lo::kH, ws.PH(bs, hv, Hv), 32768, bars.ldh);
    } else {  // nothing to load: release the barrier without data
      *bars.abort = 1;
      mbar_complete_tx(bars.ldh, 32768u);
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
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int q4 = warp & 3, hh = warp >> 2;
  const uint32_t lane_addr = tmem + ((uint32_t)(32 * q4) << 16);

  if (tid == 0 && !mbar_wait(bars.ld, ph, p.err)) *bars.abort = 1;
  if (tid == 0 && !mbar_wait(bars.ldh, ph, p.err)) *bars.abort = 1;
  __syncthreads();
  if (!*bars.abort) {
    mbar_wait(bars.ld, ph, p.err);
    mbar_wait(bars.ldh, ph, p.err);
  }
  GDN_PHASE(60);  // tiles landed

  // ---- D_V = h^T W'^T (M = dv, N = 128 tokens); Z = Q2 K1^T (M = 64, bf16) ---
  if (tid == 0 && !*bars.abort) {
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
    tc_commit(bars.mma);
  }
  // meanwhile: q rows 0-63 -> fp16 times scale gamma' (rows 64-127 still feed Z)
  if (!*bars.abort) {
    for (int e = tid; e < 64 * 16; e += 256) {
      const int r = e >> 4, c = e & 15;
      bf16x8_to_f16x8_scaled(sm + Lo::kQ + (c >> 3) * 16384 + sw_chunk(r, c & 7), s_rs[r]);
    }
  }
  if (tid == 0 && !*bars.abort && !mbar_wait(bars.mma, 0, p.err)) *bars.abort = 1;
  if (tid == 0 && !*bars.abort && !mbar_wait(bars.ld2, ph, p.err)) *bars.abort = 1;
  __syncthreads();
  GDN_PHASE(61);  // V, Z products (and q rows 0-63)
  if (!*bars.abort) {
    mbar_wait(bars.mma, 0, p.err);
    mbar_wait(bars.ld2, ph, p.err);
    tc_fence_after();
    {  // V^T row dv = 32 q4 + lane, tokens of chunk hh: V^T = U'^T - D_V, in place
      const int dvr = 32 * q4 + lane;
      unsigned char* ut = sm + (hh ? Lo::kU2 : Lo::kU1);
      uint32_t r[2][32];
      tmem_ld32_async(lane_addr + 64 * hh, r[0]);
      tmem_ld32_async(lane_addr + 64 * hh + 32, r[1]);
      tmem_ld_wait();
#pragma unroll
      for (int half = 0; half < 2; ++half)
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          uint4* u = reinterpret_cast<uint4*>(ut + sw_chunk(dvr, 4 * half + m));
          float f[8];
          unpack8(*u, f);
          const uint32_t* v = r[half] + 8 * m;
          *u = make_uint4(pack_f16(f[0] - __uint_as_float(v[0]), f[1] - __uint_as_float(v[1])),
                          pack_f16(f[2] - __uint_as_float(v[2]), f[3] - __uint_as_float(v[3])),
                          pack_f16(f[4] - __uint_as_float(v[4]), f[5] - __uint_as_float(v[5])),
                          pack_f16(f[6] - __uint_as_float(v[6]), f[7] - __uint_as_float(v[7])));
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
  if (tid == 0 && !*bars.abort) {
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
    tc_commit(bars.mma);
  }
  GDN_PHASE(62);  // V, Y, q rows 64-127 stored
  if (tid == 0 && !*bars.abort && !mbar_wait(bars.mma, 1, p.err)) *bars.abort = 1;
  __syncthreads();
  GDN_PHASE(63);  // O product
  if (!*bars.abort) {
    mbar_wait(bars.mma, 1, p.err);
    tc_fence_after();
    const int i = 32 * q4 + lane;  // token row of the block
    uint32_t r[2][32];
    tmem_ld32_async(lane_addr + 64 * hh, r[0]);
    tmem_ld32_async(lane_addr + 64 * hh + 32, r[1]);
    tmem_ld_wait();
    // o staged in the dead q / k tiles: as four 64 x 64 TMA boxes (128-byte
    // swizzle) for the tensor store, else rows of 272 bytes (conflict-free)
    // for one 256-byte bulk store per valid row
    unsigned char* box = sm + Lo::kQ + ((i >> 6) * 2 + hh) * 8192;
    unsigned char* row = sm + Lo::kQ + i * Lo::kOPitch + 128 * hh;
#pragma unroll
    for (int half = 0; half < 2; ++half)
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const uint32_t* v = r[half] + 8 * m;
        const uint4 val = make_uint4(pack_bf16(__uint_as_float(v[0]), __uint_as_float(v[1])),
                                     pack_bf16(__uint_as_float(v[2]), __uint_as_float(v[3])),
                                     pack_bf16(__uint_as_float(v[4]), __uint_as_float(v[5])),
                                     pack_bf16(__uint_as_float(v[6]), __uint_as_float(v[7])));
        if (tmo)
          *reinterpret_cast<uint4*>(box + sw_chunk(i & 63, 4 * half + m)) = val;
        else
          *reinterpret_cast<uint4*>(row + 64 * half + 16 * m) = val;
      }
    fence_proxy_async();
  }
  tc_fence_before();
  __syncthreads();
  if (!*bars.abort) {
    if (tmo) {
      if (tid == 0) {
#pragma unroll
        for (int bx = 0; bx < 4; ++bx)
          tma_store_3d(tmo, hv * kD + 64 * (bx & 1), kBlock * x.b + 64 * (bx >> 1), x.n,
                       sm + Lo::kQ + bx * 8192);
        bulk_commit();
      }
    } else if (tid < x.rows) {
      bulk_s2g(static_cast<__nv_bfloat16*>(p.o) + ((long long)(tok0 + tid) * Hv + hv) * kD,
               sm + Lo::kQ + tid * Lo::kOPitch, 256);
      bulk_commit();
    }
  }
  bulk_wait_read<0>();  // the staging is read before the next task's loads land there
  GDN_PHASE(39);  // O stored
  const bool ok = !*bars.abort;
  if (!ok && tid == 0) {
    mbar_wait(bars.ld, ph, nullptr);
    mbar_wait(bars.ld2, ph, nullptr);
    mbar_wait(bars.ldh, ph, nullptr);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  return ok;
}

__device__ __forceinline__ void out_setup(unsigned char* sm) {
  const OutBars bars = out_bars(sm);
  if (threadIdx.x == 0) {
    mbar_init(bars.ld, 1);
    mbar_init(bars.ld2, 1);
    mbar_init(bars.ldh, 1);
    mbar_init(bars.mma, 1);
    const PairBars pb = worker_pair_bars(sm);
    mbar_init(pb.ld, 1);
    mbar_init(pb.mma, 1);
    *bars.abort = 0;
    mbar_fence_init();
  }
  if (threadIdx.x < 32) tmem_alloc(out_tmem_slot(sm), 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}
__device__ __forceinline__ void out_teardown(unsigned char* sm) {
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) tmem_dealloc(*out_tmem_slot(sm), 256);
}

__global__ void __launch_bounds__(256, 1)
    gdn_out_kernel(const FwdParams p, const WsLayout ws, const __grid_constant__ CUtensorMap tmq,
                   const __grid_constant__ CUtensorMap tmk) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = align1024(smem_raw);
  BlockCtx x;
  if (!block_ctx(p, ws, &x)) return;
  out_setup(sm);
  out_task(p, ws, &tmq, &tmk, nullptr, sm, out_bars(sm), *out_tmem_slot(sm), x, 0, nullptr,
           nullptr);
  out_teardown(sm);
}

// =============================================================================
// gdn_scanout_kernel (fixed-length rows): CTAs [0, n_chains) run the scan
// chains; every other CTA takes tasks in block order from a shared counter:
// first the pair tasks (when `pairs`), then the block-output tasks, each
// waiting for the flags of what it reads (the pair task of its block, the
// scan's stored state).  All CTAs are resident at once (one per SM) and a
// task only waits for work handed out before it or for the scan, so every
// flag waited for is eventually set; every wait is also bounded.
// =============================================================================
struct ScanOutSmem {
  static constexpr int kAlloc = ScanLayout::kAlloc > OutLayout::kAlloc ? ScanLayout::kAlloc
                                                                        : OutLayout::kAlloc;
};

__device__ __forceinline__ BlockCtx fixed_block(const FwdParams& p, const WsLayout& ws, long long t) {
  const int per_block = p.N * p.Hv;
  BlockCtx x;
  x.b = (int)(t / per_block);
  x.n = (int)((t % per_block) / p.Hv);
  x.hv = (int)(t % p.Hv);
  x.t_seq = (long long)x.n * p.T;
  x.len = p.T;
  x.has2 = 2ll * x.b + 1 < (x.len + kC - 1) / kC;
  x.s1 = ws.first_slot(p, x.n) + 2ll * x.b;
  x.rows = (int)min((long long)kBlock, x.len - (long long)kBlock * x.b);
  x.hq = x.hv / (p.Hv / p.Hqk);
  return x;
}

__global__ void __launch_bounds__(256, 1)
    gdn_scanout_kernel(const FwdParams p, const WsLayout ws, const __grid_constant__ CUtensorMap tmq,
                       const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmo, int n_chains, int pairs) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = align1024(smem_raw);
  unsigned* pflags = pairs ? ws.pair_flags() : nullptr;
  if ((int)blockIdx.x < n_chains) {
    if (threadIdx.x < ScanLayout::kThreads) scan_chain(p, ws, sm, blockIdx.x, ws.scan_flags(), pflags);
    return;
  }
  __shared__ int s_task;
  const long long n_blk = ws.bslots_per_seq * p.N * p.Hv;  // tasks of each kind
  const long long n_tasks = pairs ? 2 * n_blk : n_blk;
  out_setup(sm);
  const OutBars bars = out_bars(sm);
  const PairBars pbars = worker_pair_bars(sm);
  const uint32_t tmem = *out_tmem_slot(sm);
  unsigned* pending = nullptr;  // thread 0: the last pair task's flag, not yet set
  int it_pair = 0, it_out = 0;
  while (true) {
    if (threadIdx.x == 0) {
      flush_pending(&pending);
      s_task = (int)atomicAdd(ws.task_counter(), 1u);
    }
    __syncthreads();
    const long long t = s_task;
    if (t >= n_tasks) break;
    if (pairs && t < n_blk) {
      pair_task(p, ws, sm, pbars, tmem, fixed_block(p, ws, t), it_pair++, &pending);
      if (*pbars.abort) break;
    } else {
      const BlockCtx x = fixed_block(p, ws, pairs ? t - n_blk : t);
      if (!out_task(p, ws, &tmq, &tmk, &tmo, sm, bars, tmem, x, it_out++, ws.scan_flags(), pflags))
        break;
    }
  }
  if (threadIdx.x == 0) flush_pending(&pending);
  out_teardown(sm);
}

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

}  // namespace

cudaError_t launch_pair(const FwdParams& p, const WsLayout& ws, cudaStream_t stream) {
  if (!ws.blocks) return cudaErrorInvalidValue;  // the workspace has no block records
  cudaError_t e = set_smem(gdn_pair_kernel, PairLayout::kAlloc);
  if (e != cudaSuccess) return e;
  const long long grid = ws.n_bslots * p.Hv;
  gdn_pair_kernel<<<(unsigned)grid, 256, PairLayout::kAlloc, stream>>>(p, ws);
  return cudaGetLastError();
}

cudaError_t launch_scan(const FwdParams& p, const WsLayout& ws, cudaStream_t stream) {
  if (!ws.blocks) return cudaErrorInvalidValue;  // the workspace has no block records
  cudaError_t e = set_smem(gdn_scan_kernel, ScanLayout::kAlloc);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)p.N * p.Hv * 2;
  gdn_scan_kernel<<<(unsigned)grid, ScanLayout::kThreads, ScanLayout::kAlloc, stream>>>(p, ws);
  return cudaGetLastError();
}

namespace {
int sm_count() {
  static const int n = [] {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return 0;
    return v;
  }();
  return n;
}
}  // namespace

cudaError_t launch_out(const FwdParams& p, const WsLayout& ws, cudaStream_t stream) {
  if (!ws.blocks) return cudaErrorInvalidValue;  // the workspace has no block records
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

bool scan_out_fused(const FwdParams& p) {
  const int sms = sm_count();
  return !p.cu_seqlens && sms >= 64 && (long long)p.N * p.Hv * 2 <= sms - 32;
}

cudaError_t launch_scan_out(const FwdParams& p, const WsLayout& ws, cudaStream_t stream,
                            bool pairs) {
  if (!ws.blocks) return cudaErrorInvalidValue;  // the workspace has no block records
  const long long rows = (long long)p.N * p.T;
  CUtensorMap mq, mk, mo;
  if (!make_tensor_map_bf16(&mq, p.q, rows, (long long)p.Hqk * kD) ||
      !make_tensor_map_bf16(&mk, p.k, rows, (long long)p.Hqk * kD) ||
      !make_tensor_map_bf16_3d(&mo, p.o, p.N, p.T, (long long)p.Hv * kD))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(ws.pair_flags(), 0, ws.flag_bytes, stream);
  if (e != cudaSuccess) return e;
  e = set_smem(gdn_scanout_kernel, ScanOutSmem::kAlloc);
  if (e != cudaSuccess) return e;
  const int n_chains = p.N * p.Hv * 2;
  gdn_scanout_kernel<<<(unsigned)sm_count(), 256, ScanOutSmem::kAlloc, stream>>>(
      p, ws, mq, mk, mo, n_chains, pairs ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace gdn
