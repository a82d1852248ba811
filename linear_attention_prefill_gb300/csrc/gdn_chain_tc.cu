// gdn_chain_tc.cu - the serial Reduce (#5 H) and the final Map (#6 O) of the
// chunkwise forward ("Empowering Hybrid Attention Models on NPUs", §2.1,
// Figure 1(b)) on the 5th-generation tensor cores.
//
// One CTA walks the chunks of one (sequence, v head) chain.  The products run
// transposed (tensor-memory lane = dv index j) so that their left factors, the
// state entering the chunk and V_new, are read straight from tensor memory (the
// "TS" MMA form: A in tensor memory, B in shared memory), and every accumulator
// lands in tensor memory.  The fp32 state itself lives in the registers of eight
// state warps (thread j of warpgroup g holds half g of column j of h, i.e. of row
// j of h^T).  Per chunk c, with the records of gdn_prep_tc.cu, three product
// groups:
//
//   G_A(c):  [O(c) | Vacc(c+1)]  = h(c)^T     x [Q~(c) | W'(c+1)]^T
//   G_D(c):  D                  = V_new(c)^T x Kt(c)
//   G_V(c):  [O(c) | Vacc(c+1)] += V_new(c)^T x [P^T(c) | X^T(c+1)]
//   h(c+1)     = gamma_last(c) h(c) + D^T        (state warps, fp32)
//   V_new(c+1) = U(c+1) - Vacc(c+1)              (V warps)
//
// so the state is read (W h, Q~ h) before it is updated (the chunk-first order
// of §5, Figure 10(b)).  The state read of the next chunk is split by the
// one-chunk lookahead, W(c+1) h(c+1) = W'(c+1) h(c) + X(c+1) V_new(c), which
// leaves two dependence cycles: V_new(c) -> G_V(c) -> V_new(c+1) (one chunk) and
// V_new(c) -> G_D(c) -> h(c+1) -> G_A(c+1) -> V_new(c+2) (two chunks).  G_A(c) is
// issued as soon as the fp16 copy of h(c) is in tensor memory, G_D(c) and then
// G_V(c) as soon as V_new(c) is, each group with its own commit, and the [O |
// Vacc] accumulators and V_new alternate between two tensor-memory buffers, so
// that neither cycle waits for the other's products.  Per chunk at d = 128: 16
// MMAs of K = 16 and N = 128.
//
// Warp roles, in four warpgroups (setmaxnreg moves registers from the first to
// the others).  Warp 0: producer - stages the record pieces of step c (chunk c's
// Q~, Kt, P^T and chunk c+1's W', X^T, U^T and gates) into a 2-deep ring with
// bulk copies, laid out so that each product group is one MMA chain.  Warp 1:
// allocates tensor memory; its lane 0 issues the MMAs.  Warps 4-7: V_new (U^T
// read ahead, the V accumulator, fp16 out to tensor memory) and then the output
// (-> bf16 -> shared memory -> TMA tile store).  Warps 8-15: the fp32 state (h0
// in, the update, its fp16 copy out to tensor memory, hT at the end).  The roles
// meet only at mbarriers; every wait is bounded and an expired wait ends the CTA
// cleanly.
//
// Precision: products take fp16 operands (the state and V_new rounded once per
// chunk) with fp32 accumulation; the state itself stays fp32.  An fp16 copy
// outside fp16's finite range is recorded in the device error word.
#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

constexpr int kC = 64;
constexpr int kThreads = 512;
constexpr int kStages = 2;
constexpr float kF16Max = 65504.f;
// registers per thread after setmaxnreg (launch: 128): warpgroup 0 (producer, MMA
// issue) gives, the V and state warpgroups take; 128 x (56 + 168 + 136 + 136) =
// 63488 stays within the 512 x 128 = 65536 the block is launched with
constexpr int kRegsLow = 56;
constexpr int kRegsV = 168;
constexpr int kRegsState = 136;

// Stage map (byte offsets; every piece 1024-aligned).
template <int DK, int DV>
struct ChainTcLayout {
  static constexpr int kKB = DK / 64;             // 64-column blocks of a [64][DK] tile
  static constexpr int kB1 = 0;                   // [kKB][Q~ rows | W' rows] (K-major, N = 128)
  static constexpr int kB2 = kKB * 16384;         // [Kt blocks | P^T | X^T] (MN-major)
  static constexpr int kU = kB2 + (kKB + 2) * 8192;  // U^T [DV][64]
  static constexpr int kGv = kU + DV * 128;          // gate factors (132 fp32)
  static constexpr int kStage = (kGv + kGvFloats * 4 + 1023) / 1024 * 1024;
  // output staging: the TMA boxes of one output tile: [DV/64][64 rows][64 columns]
  // bf16, 128-byte swizzled
  static constexpr int kOstBuf = DV * kC * 2;
  static constexpr int kOst = kStages * kStage;
  static constexpr int kBar = kOst + kOstBuf;
  static constexpr int kBytes = kBar + 256;
  static constexpr int kAlloc = kBytes + 1024;  // slack to align the base
  // tensor-memory columns
  static constexpr uint32_t cOV0 = 0;              // [O^T | Vacc] buffer 0: [DV][64 | 64]
  static constexpr uint32_t cOV1 = 128;            // buffer 1
  static constexpr uint32_t cD = 256;              // increment Kt^T V_new, transposed [DV][DK]
  static constexpr uint32_t cHf = 256 + DK;        // h^T fp16, 2 per column [DV][DK/2]
  static constexpr uint32_t cVf0 = 256 + DK + DK / 2;  // V_new^T fp16 [DV][32], buffer 0
  static constexpr uint32_t cVf1 = cVf0 + 32;          // buffer 1
  static constexpr uint32_t kCols = 512;
  static_assert(cVf1 + 32 <= kCols, "tensor memory");
};

struct ChainBars {
  uint64_t full[kStages], empty[kStages];
  uint64_t mma_done;    // commit after G_A(c), G_D(c), G_V(c) (prologue: phase 0)
  uint64_t d_ready;     // commit after G_D(c)
  uint64_t hf_ready;    // 8 state-warp arrivals: the fp16 copy of h(c) is in tensor memory
  uint64_t d_free;      // 8 state-warp arrivals: the increment has been read
  uint64_t v_ready;     // 4 V-warp arrivals: V_new(c) in fp16
  uint64_t ob_free[2];  // 4 V-warp arrivals: [O | Vacc] buffer b has been read
  uint64_t fin;         // teardown: every issued MMA has completed
  uint64_t ost_free;    // the output store thread: the staging buffer may be rewritten
  uint64_t ost_full;    // 4 V-warp arrivals: the output staging buffer is written
  uint32_t tmem;
  int abort;
};

// Bounded wait that also gives up as soon as another role has given up: try_wait
// blocks for a while (a system-dependent time) unless the phase completes; the clock
// is read only once the first try has failed.
__device__ __forceinline__ bool try_wait_bar(uint64_t* bar, unsigned parity) {
  unsigned done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}
__device__ __forceinline__ bool wait_bar(uint64_t* bar, unsigned parity, volatile int* abort,
                                         unsigned* err) {
  if (try_wait_bar(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (try_wait_bar(bar, parity)) return true;
    if (*abort) return false;
    if (clock64() - t0 > (1ll << 31)) {
      record_error(err, kErrWaitTimeout);
      *abort = 1;
      return false;
    }
  }
}

// wait_bar for all lanes of a warp, with one outcome for the whole warp (a lane
// that timed out makes the warp give up), so warp-collective code after it never
// runs with lanes missing.
__device__ __forceinline__ bool wait_warp(uint64_t* bar, unsigned parity, volatile int* abort,
                                          unsigned* err) {
  return __all_sync(0xffffffffu, wait_bar(bar, parity, abort, err));
}

// per-thread register budget of the calling warpgroup (every warp of it executes the
// same one)
template <int N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(N));
}

template <int DK, int DV, bool DELTA>
__global__ void __launch_bounds__(kThreads, 1)
    gdn_chain_tc_kernel(const FwdParams p, const WsLayout ws,
                        const __grid_constant__ CUtensorMap tmo) {
  using Lo = ChainTcLayout<DK, DV>;
  constexpr int HK = DK / 2;  // state rows per state warpgroup
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  ChainBars* B = reinterpret_cast<ChainBars*>(sm + Lo::kBar);
  volatile int* abort = &B->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int hv = blockIdx.x % p.Hv;
  const int n = blockIdx.x / p.Hv;
  const long long t_seq = p.cu_seqlens ? (long long)p.cu_seqlens[n] : (long long)n * p.T;
  const long long len = p.cu_seqlens ? (long long)p.cu_seqlens[n + 1] - t_seq : (long long)p.T;
  const int n_chunks = (int)((len + kC - 1) / kC);
  const long long slot0 = ws.first_slot(p, n);
  const long long hoff = (long long)(n * p.Hv + hv) * DK * DV;

  if (n_chunks == 0) {  // an empty sequence: hT = h0 (or zeros)
    if (p.hT)
      for (int i = tid; i < DK * DV; i += kThreads) p.hT[hoff + i] = p.h0 ? p.h0[hoff + i] : 0.f;
    return;
  }

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&B->full[i], 1);
      mbar_init(&B->empty[i], 13);  // the MMA commit + 4 V warps + 8 state warps
    }
    mbar_init(&B->mma_done, 1);
    mbar_init(&B->d_ready, 1);
    mbar_init(&B->hf_ready, 8);
    mbar_init(&B->d_free, 8);
    mbar_init(&B->v_ready, 4);
    mbar_init(&B->ob_free[0], 4);
    mbar_init(&B->ob_free[1], 4);
    mbar_init(&B->fin, 1);
    mbar_init(&B->ost_free, 1);
    mbar_init(&B->ost_full, 4);
    B->abort = 0;
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(&B->tmem, Lo::kCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = B->tmem;
  // epilogue warps: lanes of quadrant warp % 4; the state column j this thread owns
  const int quad = warp & 3;
  const uint32_t lane_base = tmem + ((uint32_t)(32 * quad) << 16);
  const int j = DV == 128 ? 32 * quad + lane : 16 * quad + lane;
  const bool jact = DV == 128 || lane < 16;

  if (warp < 4) {
    regs_dec<kRegsLow>();
    if (warp == 0 && lane == 0) {
      // ======================= producer =======================================
      // Stage jj holds chunk jj-1's Q~, Kt, P^T (jj >= 1) and chunk jj's W', X^T, U^T,
      // gates (jj < n_chunks): everything step jj-1 and the V / state epilogues after
      // it read.  The prologue reads stage 0.
      griddep_wait();  // the records are the prep launch's output
      int issued = 0;
      for (int jj = 0; jj <= n_chunks; ++jj) {
        const int s = jj % kStages;
        if (jj >= kStages && !wait_bar(&B->empty[s], ((jj / kStages) - 1) & 1, abort, p.err)) break;
        unsigned char* st = sm + s * Lo::kStage;
        uint64_t* bar = &B->full[s];
        const bool has_prev = jj >= 1, has_cur = jj < n_chunks;
        unsigned bytes = 0;
        if (has_prev) bytes += 2 * kC * DK * 2 + kC * kC * 2;  // Q~, Kt, P^T
        if (has_cur) {
          bytes += DV * kC * 2 + kGvFloats * 4;  // U^T, gates
          if (DELTA) bytes += kC * DK * 2 + (has_prev ? kC * kC * 2 : 0);  // W', X^T
        }
        mbar_expect_tx(bar, bytes);
        if (has_prev) {
          const long long rs = slot0 + jj - 1;
          const __half* q = ws.Qt(rs, hv, p.Hv);
#pragma unroll
          for (int kb = 0; kb < Lo::kKB; ++kb)
            bulk_g2s(st + Lo::kB1 + kb * 16384, q + kb * kC * 64, kC * 128, bar);
          bulk_g2s(st + Lo::kB2, ws.Kt(rs, hv, p.Hv), kC * DK * 2, bar);
          bulk_g2s(st + Lo::kB2 + Lo::kKB * 8192, ws.P(rs, hv, p.Hv), kC * kC * 2, bar);
        }
        if (has_cur) {
          const long long rs = slot0 + jj;
          if (DELTA) {
            const __half* w = ws.W(rs, hv, p.Hv);
#pragma unroll
            for (int kb = 0; kb < Lo::kKB; ++kb)
              bulk_g2s(st + Lo::kB1 + kb * 16384 + 8192, w + kb * kC * 64, kC * 128, bar);
            if (has_prev)
              bulk_g2s(st + Lo::kB2 + (Lo::kKB + 1) * 8192, ws.Xt(rs, hv, p.Hv), kC * kC * 2, bar);
          }
          bulk_g2s(st + Lo::kU, ws.U(rs, hv, p.Hv), DV * kC * 2, bar);
          bulk_g2s(st + Lo::kGv, ws.gv(rs, hv, p.Hv), kGvFloats * 4, bar);
        }
        issued = jj + 1;
        if (jj + kStages < n_chunks)  // the record two stages ahead: into L2 now
          bulk_prefetch_l2(ws.rec(slot0 + jj + kStages, hv, p.Hv), (unsigned)ws.task_bytes);
      }
      // let every copy this thread issued land before the CTA can exit
      for (int jj = max(0, issued - kStages); jj < issued; ++jj)
        mbar_wait_limit(&B->full[jj % kStages], (jj / kStages) & 1, nullptr, 1ll << 31);
    } else if (warp == 1 && lane == 0) {
      // ======================= MMA issue (one thread) =========================
      bool issued_any = false;  // any product issued (then `fin` tracks their completion)
      // G_A's B operand: k step s of [Q~ | W'] (N = 128) - or of one of them (N = 64)
      auto b1 = [&](int s, int stage, bool wrows) {
        return sw128_desc(smem_u32(sm + stage * Lo::kStage + Lo::kB1 + (s >> 2) * 16384 +
                                   (wrows ? 8192 : 0)) + (s & 3) * 32, 16, 1024);
      };
      // G_D's and G_V's B operand: k step s (16 tokens) of the MN-major [Kt | P^T | X^T]
      // from 64-column block nb on
      auto b2 = [&](int s, int stage, int nb) {
        return sw128_desc(smem_u32(sm + stage * Lo::kStage + Lo::kB2 + nb * 8192) + s * 2048,
                          8192, 1024);
      };
      if (wait_bar(&B->full[0], 0, abort, p.err) && wait_bar(&B->hf_ready, 0, abort, p.err)) {
        tc_fence_after();
        if (DELTA) {  // prologue: Vacc(0) = h(0)^T W'(0)^T, into buffer 1 (step -1)
          constexpr uint32_t id = idesc_f16(DV, 64, false, false, false);
#pragma unroll
          for (int s = 0; s < DK / 16; ++s)
            tc_mma_ts(tmem + Lo::cOV1 + 64, tmem + Lo::cHf + 8 * s, b1(s, 0, true), id, s > 0);
          tc_commit(&B->mma_done);
          tc_commit(&B->empty[0]);
          issued_any = true;
        } else {  // no product in the prologue: release its waiters directly
          mbar_arrive(&B->mma_done);
          mbar_arrive(&B->empty[0]);
        }
        for (int c = 0; c < n_chunks; ++c) {
          const int jj = c + 1, s = jj % kStages, b = c & 1;
          const int use = (c + b) / 2;  // earlier uses of [O | Vacc] buffer b: steps c-2, c-4, ..
          const uint32_t cOV = b ? Lo::cOV1 : Lo::cOV0, cVf = b ? Lo::cVf1 : Lo::cVf0;
          if (!wait_bar(&B->full[s], (jj / kStages) & 1, abort, p.err)) break;
          if (use >= 1 && !wait_bar(&B->ob_free[b], (use - 1) & 1, abort, p.err)) break;
          if (!wait_bar(&B->hf_ready, c & 1, abort, p.err)) break;
          tc_fence_after();
          const bool more = DELTA && c + 1 < n_chunks;  // the lookahead terms of chunk c + 1
          const uint32_t id_ov = more ? idesc_f16(DV, 128, false, false, false)
                                      : idesc_f16(DV, 64, false, false, false);
          // G_A: [O | Vacc] = h^T [Q~ | W']^T  (fresh)
#pragma unroll
          for (int k = 0; k < DK / 16; ++k)
            tc_mma_ts(tmem + cOV, tmem + Lo::cHf + 8 * k, b1(k, s, false), id_ov, k > 0);
          issued_any = true;
          if (!wait_bar(&B->v_ready, c & 1, abort, p.err)) break;
          if (!wait_bar(&B->d_free, c & 1, abort, p.err)) break;
          tc_fence_after();
          // G_D: D = V_new^T Kt  (fresh), then its own commit for the state warps
          constexpr uint32_t id_d = idesc_f16(DV, DK, false, false, true);
#pragma unroll
          for (int k = 0; k < kC / 16; ++k)
            tc_mma_ts(tmem + Lo::cD, tmem + cVf + 8 * k, b2(k, s, 0), id_d, k > 0);
          tc_commit(&B->d_ready);
          // G_V: [O | Vacc] += V_new^T [P^T | X^T]
          const uint32_t id_v = more ? idesc_f16(DV, 128, false, false, true)
                                     : idesc_f16(DV, 64, false, false, true);
#pragma unroll
          for (int k = 0; k < kC / 16; ++k)
            tc_mma_ts(tmem + cOV, tmem + cVf + 8 * k, b2(k, s, Lo::kKB), id_v, true);
          tc_commit(&B->mma_done);
          tc_commit(&B->empty[s]);
        }
      }
      // every product issued has completed before tensor memory is released
      if (issued_any) {
        tc_commit(&B->fin);
        mbar_wait_limit(&B->fin, 0, nullptr, 1ll << 31);
      }
    }
  } else if (warp < 8) {
    // ======================= V_new and the output (warps 4-7) =================
    // The output tile goes through shared memory and leaves by TMA tile stores, one
    // per 64 columns, issued by lane 0 of warp 4.
    regs_inc<kRegsV>();
    const int vw = warp - 4;  // 0..3
    __nv_bfloat16* og = static_cast<__nv_bfloat16*>(p.o) + (long long)hv * p.dv;
    const long long o_tok = (long long)p.Hv * p.dv;
    __half2 vmax = __floats2half2_rn(0.f, 0.f);  // max |V_new| (NaN sticks)
    for (int step = -1; step < n_chunks; ++step) {
      // step -1: the prologue's Vacc(0); step c: O(c) and Vacc(c+1) of G_A(c) + G_V(c)
      const int jj = step + 1;  // the chunk whose V_new this step forms
      const bool has_v = jj < n_chunks;
      const bool has_acc = DELTA && has_v;
      const int b = step & 1;  // [O | Vacc] buffer of this step (step -1: buffer 1)
      const uint32_t cOV = b ? Lo::cOV1 : Lo::cOV0;
      // this thread's row j of U^T(jj) (128 bytes, swizzled), read ahead of the products
      uint4 u[8];
      if (has_v) {
        const int s = jj % kStages;
        if (!wait_warp(&B->full[s], (jj / kStages) & 1, abort, p.err)) break;
        const unsigned char* urow = sm + s * Lo::kStage + Lo::kU + j * 128;
#pragma unroll
        for (int m = 0; m < 8; ++m)
          u[m] = jact ? *reinterpret_cast<const uint4*>(urow + ((m ^ (j & 7)) << 4))
                      : make_uint4(0, 0, 0, 0);
      }
      if (!wait_warp(&B->mma_done, (step + 1) & 1, abort, p.err)) break;
      tc_fence_after();
      if (has_v) {
        // V_new(jj) = U(jj) - Vacc(jj)
        uint32_t b0[32], b1[32];
        if (has_acc) {
          tmem_ld32_async(lane_base + cOV + 64, b0);
          tmem_ld32_async(lane_base + cOV + 96, b1);
          tmem_ld_wait();
        }
        uint32_t pk[32];
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const __half2* h2 = reinterpret_cast<const __half2*>(&u[m]);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int c0 = 8 * m + 2 * i;  // tokens c0, c0 + 1 (static after unrolling)
            const float2 uu = __half22float2(h2[i]);
            const float va = c0 < 32 ? __uint_as_float(b0[c0]) : __uint_as_float(b1[c0 - 32]);
            const float vb = c0 < 32 ? __uint_as_float(b0[c0 + 1]) : __uint_as_float(b1[c0 - 31]);
            // (lanes past dv = 64 hold no row: their accumulator lanes are not written)
            const float x0 = !jact ? 0.f : has_acc ? uu.x - va : uu.x;
            const float x1 = !jact ? 0.f : has_acc ? uu.y - vb : uu.y;
            pk[4 * m + i] = pack_f16(x0, x1);
            vmax = __hmax2_nan(vmax, __habs2(*reinterpret_cast<const __half2*>(&pk[4 * m + i])));
          }
        }
        tmem_st32(lane_base + ((jj & 1) ? Lo::cVf1 : Lo::cVf0), pk);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&B->v_ready);
          mbar_arrive(&B->empty[jj % kStages]);
        }
        // reconverge right after lane 0's arrivals, so that they are issued now and not
        // after the work below (they release the next products)
        __syncwarp();
      } else if (lane == 0) {
        mbar_arrive(&B->empty[jj % kStages]);
      }
      uint32_t ob[32];  // O(step) as bf16 pairs: ob[m] = (o[2m], o[2m + 1])
      if (step >= 0) {
        uint32_t a0[32], a1[32];
        tmem_ld32_async(lane_base + cOV, a0);
        tmem_ld32_async(lane_base + cOV + 32, a1);
        tmem_ld_wait();
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          ob[m] = pack_bf16(__uint_as_float(a0[2 * m]), __uint_as_float(a0[2 * m + 1]));
          ob[16 + m] = pack_bf16(__uint_as_float(a1[2 * m]), __uint_as_float(a1[2 * m + 1]));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&B->ob_free[b]);  // G_A(step + 2) may overwrite buffer b
      __syncwarp();
      if (step >= 0) {
        const int L = (int)min((long long)kC, len - (long long)step * kC);
        const bool odd = j & 1;
        if (p.cu_seqlens && L < kC) {
          // a packed sequence's ragged last chunk: a tile store would reach into the next
          // sequence's rows, so these rows are stored directly (lanes j and j ^ 1 trade
          // one bf16 pair per token pair: the even lane writes (t, j..j+1), the odd lane
          // (t+1, j-1..j))
          __nv_bfloat16* orow = og + (t_seq + (long long)step * kC) * o_tok;
#pragma unroll
          for (int m = 0; m < 32; ++m) {
            const int t = 2 * m;
            const uint32_t other = __shfl_xor_sync(0xffffffffu, ob[m], 1);
            if (jact) {
              if (!odd) {
                if (t < L)
                  *reinterpret_cast<uint32_t*>(orow + (long long)t * o_tok + j) =
                      __byte_perm(ob[m], other, 0x5410);
              } else if (t + 1 < L) {
                *reinterpret_cast<uint32_t*>(orow + (long long)(t + 1) * o_tok + j - 1) =
                    __byte_perm(ob[m], other, 0x3276);
              }
            }
          }
          continue;  // always the last step
        }
        // O(step) through the staging buffer (free once the previous tile store has read
        // it) and one TMA tile store per 64 columns
        unsigned char* ostage = sm + Lo::kOst;
        if (vw == 0 && lane == 0) {
          bulk_wait_read<0>();
          mbar_arrive(&B->ost_free);
        }
        if (!wait_warp(&B->ost_free, step & 1, abort, p.err)) break;
#pragma unroll
        for (int m = 0; m < 32; ++m) {
          const int t = 2 * m;
          const uint32_t other = __shfl_xor_sync(0xffffffffu, ob[m], 1);
          if (jact) {
            const int tt = odd ? t + 1 : t, jj0 = odd ? j - 1 : j;  // row, even column
            *reinterpret_cast<uint32_t*>(ostage + (jj0 >> 6) * 8192 + tt * 128 +
                                         ((((jj0 & 63) >> 3) ^ (tt & 7)) << 4) + (jj0 & 7) * 2) =
                __byte_perm(ob[m], other, odd ? 0x3276 : 0x5410);
          }
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(&B->ost_full);
        if (vw == 0) {
          if (!wait_warp(&B->ost_full, step & 1, abort, p.err)) break;
          if (lane == 0) {
#pragma unroll
            for (int bb = 0; bb < DV / 64; ++bb) {
              if (p.cu_seqlens)
                tma_store_2d(&tmo, hv * DV + 64 * bb, (int)(t_seq + (long long)step * kC),
                             ostage + bb * 8192);
              else
                tma_store_3d(&tmo, hv * DV + 64 * bb, step * kC, n, ostage + bb * 8192);
            }
            bulk_commit();
          }
        }
      }
    }
    if (vw == 0 && lane == 0) bulk_wait<0>();  // the output has left shared memory and landed
    const float2 vm = __half22float2(vmax);
    if (!__all_sync(0xffffffffu, vm.x <= kF16Max && vm.y <= kF16Max) && lane == 0)
      record_error(p.err, kErrOperandRange);
  } else {
    // ======================= state (warps 8-15) ===============================
    // Thread j of state warpgroup g keeps rows [g HK, (g + 1) HK) of column j of h
    // (fp32) in registers for the whole chain.
    regs_inc<kRegsState>();
    const int g = (warp - 8) >> 2;
    __half2 hmax = __floats2half2_rn(0.f, 0.f);  // max |h| in its fp16 copy (NaN sticks)
    float h[HK];
#pragma unroll
    for (int i = 0; i < HK; ++i)
      h[i] = (p.h0 && jact) ? p.h0[hoff + (long long)(g * HK + i) * DV + j] : 0.f;
    float gl = 1.f;  // gamma_last of the chunk whose increment comes next
    for (int step = -1; step < n_chunks; ++step) {
      // step -1: h(0) = h0; step c: h(c+1) = gamma_last(c) h(c) + (Kt(c)^T V_new(c))^T
      if (step >= 0) {
        if (!wait_warp(&B->d_ready, step & 1, abort, p.err)) break;
        tc_fence_after();
#pragma unroll
        for (int b = 0; b < HK / 32; ++b) {
          uint32_t r[32];
          tmem_ld32_async(lane_base + Lo::cD + g * HK + 32 * b, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i)  // (lanes past dv = 64 hold no row: kept at 0)
            h[32 * b + i] = fmaf(gl, h[32 * b + i], jact ? __uint_as_float(r[i]) : 0.f);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&B->d_free);  // G_D(step + 1) may overwrite the increment
        __syncwarp();
      }
      const int jj = step + 1;  // the chunk the state now enters
      if (jj == n_chunks) {
        if (p.hT && jact) {
#pragma unroll
          for (int i = 0; i < HK; ++i) p.hT[hoff + (long long)(g * HK + i) * DV + j] = h[i];
        }
        break;
      }
      // the fp16 copy of h(jj): G_A(jj)'s left factor
#pragma unroll
      for (int b = 0; b < HK / 32; ++b) {
        uint32_t hf[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          hf[i] = pack_f16(h[32 * b + 2 * i], h[32 * b + 2 * i + 1]);
          hmax = __hmax2_nan(hmax, __habs2(*reinterpret_cast<const __half2*>(&hf[i])));
        }
        tmem_st16(lane_base + Lo::cHf + g * (HK / 2) + 16 * b, hf);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&B->hf_ready);
      __syncwarp();
      // gamma_last(jj) for the next update, from stage jj
      const int s = jj % kStages;
      if (!wait_warp(&B->full[s], (jj / kStages) & 1, abort, p.err)) break;
      gl = reinterpret_cast<const float*>(sm + s * Lo::kStage + Lo::kGv)[0];
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&B->empty[s]);
        if (step < 0) mbar_arrive(&B->d_free);  // nothing to read before G_D(0)
      }
    }
    const float2 hm = __half22float2(hmax);
    if (!__all_sync(0xffffffffu, hm.x <= kF16Max && hm.y <= kF16Max) && lane == 0)
      record_error(p.err, kErrOperandRange);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, Lo::kCols);
}

template <int DK, int DV, bool DELTA>
cudaError_t launch_t(const FwdParams& p, const WsLayout& ws, cudaStream_t stream) {
  using Lo = ChainTcLayout<DK, DV>;
  // the output as TMA tiles of 64 tokens x 64 columns: [N][T][Hv dv] for fixed-length
  // rows (a ragged last chunk clips at T), [T][Hv dv] for packed sequences
  CUtensorMap mo;
  const bool ok = p.cu_seqlens
                      ? make_tensor_map_bf16(&mo, p.o, (long long)p.T, (long long)p.Hv * DV)
                      : make_tensor_map_bf16_3d(&mo, p.o, (long long)p.N, (long long)p.T,
                                                (long long)p.Hv * DV);
  if (!ok) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(gdn_chain_tc_kernel<DK, DV, DELTA>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, Lo::kAlloc);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)p.N * p.Hv;
  return launch_after(gdn_chain_tc_kernel<DK, DV, DELTA>, (unsigned)grid, kThreads, Lo::kAlloc,
                      stream, p, ws, mo);
}

template <int DK, int DV>
cudaError_t launch_dd(const FwdParams& p, const WsLayout& ws, cudaStream_t stream) {
  return p.delta_rule ? launch_t<DK, DV, true>(p, ws, stream) : launch_t<DK, DV, false>(p, ws, stream);
}

}  // namespace

cudaError_t launch_chain_tc(const FwdParams& p, const WsLayout& ws, cudaStream_t stream) {
  if (p.kda) return cudaErrorInvalidValue;  // KDA records run the mma.sync chain
  if (p.dk == 128) return p.dv == 128 ? launch_dd<128, 128>(p, ws, stream) : launch_dd<128, 64>(p, ws, stream);
  return p.dv == 128 ? launch_dd<64, 128>(p, ws, stream) : launch_dd<64, 64>(p, ws, stream);
}

}  // namespace gdn
