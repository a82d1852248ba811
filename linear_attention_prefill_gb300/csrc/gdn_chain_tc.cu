// gdn_chain_tc.cu - the serial Reduce (#5 H) and the final Map (#6 O) of the
// chunkwise forward ("Empowering Hybrid Attention Models on NPUs", §2.1,
// Figure 1(b)) on the 5th-generation tensor cores, with the fp32 state resident
// in tensor memory.
//
// One CTA walks the chunks of one (sequence, v head) chain.  The state is kept
// transposed, h^T [dv][dk] (tensor-memory lane = dv index, column = dk index), so
// that the products whose left factor is the state or V_new read it straight
// from tensor memory (the "TS" MMA form: A in tensor memory, B in shared memory)
// and every accumulator lands in tensor memory; nothing of the state goes
// through shared memory.  Per chunk c, with the records of gdn_prep.cu:
//
//   G_A(c):  [O(c) | Vacc(c+1)]      = h(c)^T     x [Q~(c) | W'(c+1)]^T
//   G_B(c):  [h | O(c) | Vacc(c+1)] += V_new(c)^T x [Kt(c) | P^T(c) | X^T(c+1)]
//   V_new(c+1) = U(c+1) - Vacc(c+1)
//
// G_B accumulates onto gamma_last(c) h(c), so it performs the in-place update
// h(c+1) = gamma_last(c) h(c) + Kt(c)^T V_new(c) after the state read and the
// output (the chunk-first order of §5, Figure 10(b)).  The state read of the
// next chunk is split by the one-chunk lookahead, W(c+1) h(c+1) = W'(c+1) h(c) +
// X(c+1) V_new(c): both halves come from the operands of chunk c, so one
// commit per chunk covers the read, the output and the update (12 MMAs of K =
// 16 at d = 128: 8 with N = 128 and 4 with N = 256).
//
// Warp roles.  Warp 0: producer - stages the record pieces of step c (chunk c's
// Q~, Kt, P^T and chunk c+1's W', X^T, U^T and gates) into a 2-deep ring with
// bulk copies, B operands laid out so that each group is one MMA chain.  Warp
// 1: allocates tensor memory; its lane 0 issues the MMAs.  Warps 2-5: read the
// output and V accumulators (output -> bf16 -> o; V_new -> fp16 -> tensor memory).
// Warps 6-9: read the new state, store its fp16 copy (G_A's left factor) and
// write it back scaled by the next chunk's gamma_last; after the last chunk they
// write hT.  The roles meet only at mbarriers; every wait is bounded and an
// expired wait ends the CTA cleanly.
//
// Precision: products take fp16 operands (the state and V_new rounded once per
// chunk) with fp32 accumulation; the state itself stays fp32 in tensor memory.
// An operand outside fp16's finite range is recorded in the device error word.
#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

constexpr int kC = 64;
constexpr int kThreads = 320;
constexpr int kStages = 2;
constexpr float kF16Max = 65504.f;

// Stage map (byte offsets; every piece 1024-aligned).
template <int DK, int DV>
struct ChainTcLayout {
  static constexpr int kKB = DK / 64;             // 64-column blocks of a [64][DK] tile
  static constexpr int kB1 = 0;                   // [kKB][Q~ rows | W' rows] (K-major, N = 128)
  static constexpr int kB2 = kKB * 16384;         // [Kt blocks | P^T | X^T] (MN-major)
  static constexpr int kU = kB2 + (kKB + 2) * 8192;  // U^T [DV][64]
  static constexpr int kGv = kU + DV * 128;          // gate factors (132 fp32)
  static constexpr int kStage = (kGv + kGvFloats * 4 + 1023) / 1024 * 1024;
  // output staging: 2 buffers, each the TMA boxes of one output tile: [DV/64][64 rows]
  // [64 columns] bf16, 128-byte swizzled
  static constexpr int kOstBuf = DV * kC * 2;
  static constexpr int kOst = kStages * kStage;
  static constexpr int kBar = kOst + 2 * kOstBuf;
  static constexpr int kBytes = kBar + 128;
  static constexpr int kAlloc = kBytes + 1024;  // slack to align the base
  // tensor-memory columns
  static constexpr uint32_t cH = 0;                // h^T fp32 [DV lanes][DK]
  static constexpr uint32_t cO = DK;               // O^T accumulator [DV][64]
  static constexpr uint32_t cV = DK + 64;          // V accumulator [DV][64]
  static constexpr uint32_t cHf = DK + 128;        // h^T fp16, 2 per column [DV][DK/2]
  static constexpr uint32_t cVf = DK + 128 + DK / 2;  // V_new^T fp16 [DV][32]
  static constexpr uint32_t kCols = DK == 128 ? 512 : 256;
  static_assert(cVf + 32 <= kCols, "tensor memory");
};

struct ChainBars {
  uint64_t full[kStages], empty[kStages];
  uint64_t mma_done;  // tcgen05.commit after each step's products (prologue: phase 0)
  uint64_t h_ready;   // 4 warp arrivals: h(c) in fp16 and gamma h(c) in place
  uint64_t v_ready;   // 4 warp arrivals: V_new(c) in fp16
  uint64_t ov_free;   // 4 warp arrivals: the O / V accumulators have been read
  uint64_t fin;       // teardown: every issued MMA has completed
  uint64_t ost_free;  // the output store thread: the staging buffer may be rewritten
  uint64_t ost_full;  // 4 V-warp arrivals: the output staging buffer is written
  uint32_t tmem;
  int abort;
};

// Bounded wait that also gives up as soon as another role has given up.  Each
// try_wait lets the hardware suspend the thread until the phase completes (up to
// kSuspendNs), so waiting warps take no issue slots from the working ones.
constexpr unsigned kSuspendNs = 100000;
__device__ __forceinline__ bool wait_bar(uint64_t* bar, unsigned parity, volatile int* abort,
                                         unsigned* err) {
  const long long t0 = clock64();
  while (true) {
    unsigned done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendNs)
        : "memory");
    if (done) return true;
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

template <int DK, int DV, bool DELTA>
__global__ void __launch_bounds__(kThreads, 1)
    gdn_chain_tc_kernel(const FwdParams p, const WsLayout ws,
                        const __grid_constant__ CUtensorMap tmo) {
  using Lo = ChainTcLayout<DK, DV>;
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
      mbar_init(&B->empty[i], 9);  // the MMA commit + 4 V warps + 4 state warps
    }
    mbar_init(&B->mma_done, 1);
    mbar_init(&B->h_ready, 4);
    mbar_init(&B->v_ready, 4);
    mbar_init(&B->ov_free, 4);
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

  if (warp == 0) {
    // ======================= producer =========================================
    // Stage jj holds chunk jj-1's Q~, Kt, P^T (jj >= 1) and chunk jj's W', X^T, U^T,
    // gates (jj < n_chunks): everything step jj-1 and the V / state epilogues after
    // it read.  The prologue reads stage 0.
    int issued = 0;
    if (lane == 0) {
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
    }
  } else if (warp == 1) {
    // ======================= MMA issue (one thread) ===========================
    if (lane == 0) {
      bool issued_any = false;  // any product issued (then `fin` tracks their completion)
      // G_A's B operand: k step s of [Q~ | W'] (N = 128) - or of one of them (N = 64)
      auto b1 = [&](int s, int stage, bool wrows) {
        return sw128_desc(smem_u32(sm + stage * Lo::kStage + Lo::kB1 + (s >> 2) * 16384 +
                                   (wrows ? 8192 : 0)) + (s & 3) * 32, 16, 1024);
      };
      // G_B's B operand: k step s (16 tokens) of [Kt | P^T | X^T], MN-major
      auto b2 = [&](int s, int stage) {
        return sw128_desc(smem_u32(sm + stage * Lo::kStage + Lo::kB2) + s * 2048, 8192, 1024);
      };
      bool ok = wait_bar(&B->full[0], 0, abort, p.err) && wait_bar(&B->h_ready, 0, abort, p.err);
      if (ok) {
        tc_fence_after();
        if (DELTA) {  // prologue: Vacc(0) = h(0)^T W'(0)^T
          constexpr uint32_t id = idesc_f16(DV, 64, false, false, false);
#pragma unroll
          for (int s = 0; s < DK / 16; ++s)
            tc_mma_ts(tmem + Lo::cV, tmem + Lo::cHf + 8 * s, b1(s, 0, true), id, s > 0);
        }
        if (DELTA) {
          tc_commit(&B->mma_done);
          tc_commit(&B->empty[0]);
        } else {  // no product in the prologue: release its waiters directly
          mbar_arrive(&B->mma_done);
          mbar_arrive(&B->empty[0]);
        }
        issued_any = DELTA;
        for (int c = 0; c < n_chunks; ++c) {
          const int jj = c + 1, s = jj % kStages;
          if (!wait_bar(&B->full[s], (jj / kStages) & 1, abort, p.err)) break;
          if (!wait_bar(&B->h_ready, c & 1, abort, p.err)) break;
          if (!wait_bar(&B->v_ready, c & 1, abort, p.err)) break;
          if (!wait_bar(&B->ov_free, c & 1, abort, p.err)) break;
          tc_fence_after();
          const bool more = DELTA && c + 1 < n_chunks;  // the lookahead terms of chunk c + 1
          // G_A: [O | Vacc] = h^T [Q~ | W']^T
          const uint32_t ida = more ? idesc_f16(DV, 128, false, false, false)
                                    : idesc_f16(DV, 64, false, false, false);
#pragma unroll
          for (int k = 0; k < DK / 16; ++k)
            tc_mma_ts(tmem + Lo::cO, tmem + Lo::cHf + 8 * k, b1(k, s, false), ida, k > 0);
          // G_B: [h | O | Vacc] += V_new^T [Kt | P^T | X^T]
          const uint32_t idb = more ? idesc_f16(DV, DK + 128, false, false, true)
                                    : idesc_f16(DV, DK + 64, false, false, true);
#pragma unroll
          for (int k = 0; k < kC / 16; ++k)
            tc_mma_ts(tmem + Lo::cH, tmem + Lo::cVf + 8 * k, b2(k, s), idb, true);
          tc_commit(&B->mma_done);
          tc_commit(&B->empty[s]);
          issued_any = true;
        }
      }
      // every product issued has completed before tensor memory is released
      if (issued_any) {
        tc_commit(&B->fin);
        mbar_wait_limit(&B->fin, 0, nullptr, 1ll << 31);
      }
    }
  } else if (warp < 6) {
    // ======================= output and V_new (warps 2-5) =====================
    // The output tile goes through shared memory (row t of the staging buffer is
    // o[t][hv][0..DV), padded to spread the banks) and leaves by bulk copies, one row
    // each, issued by lane 0 of every V warp for its quarter of the rows.
    const int vw = warp - 2;  // 0..3
    __nv_bfloat16* og = static_cast<__nv_bfloat16*>(p.o) + (long long)hv * p.dv;
    const long long o_tok = (long long)p.Hv * p.dv;
    __half2 vmax = __floats2half2_rn(0.f, 0.f);  // max |V_new| (NaN sticks)
    for (int step = -1; step < n_chunks; ++step) {
      // step -1: the prologue's Vacc(0); step c: G_A(c), G_B(c)
      if (!wait_warp(&B->mma_done, (step + 1) & 1, abort, p.err)) break;
      tc_fence_after();
      const int jj = step + 1;  // the stage whose U^T this step's V_new takes
      const bool has_v = jj < n_chunks;
      const bool has_acc = DELTA && has_v;
      uint32_t ob[32];  // O(step) as bf16 pairs: ob[m] = (o[2m], o[2m + 1])
      if (step >= 0) {
        uint32_t a0[32], a1[32];
        tmem_ld32_async(lane_base + Lo::cO, a0);
        tmem_ld32_async(lane_base + Lo::cO + 32, a1);
        tmem_ld_wait();
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          ob[m] = pack_bf16(__uint_as_float(a0[2 * m]), __uint_as_float(a0[2 * m + 1]));
          ob[16 + m] = pack_bf16(__uint_as_float(a1[2 * m]), __uint_as_float(a1[2 * m + 1]));
        }
      }
      uint32_t b0[32], b1[32];
      if (has_acc) {
        tmem_ld32_async(lane_base + Lo::cV, b0);
        tmem_ld32_async(lane_base + Lo::cV + 32, b1);
        tmem_ld_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&B->ov_free);  // G_A(step + 1) may overwrite O and Vacc
      if (has_v) {
        // V_new(jj) = U(jj) - Vacc(jj), this thread's row j of U^T (128 bytes, swizzled)
        const int s = jj % kStages;
        if (!wait_warp(&B->full[s], (jj / kStages) & 1, abort, p.err)) break;
        const unsigned char* urow = sm + s * Lo::kStage + Lo::kU + j * 128;
        uint32_t pk[32];
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const uint4 raw = jact ? *reinterpret_cast<const uint4*>(urow + ((m ^ (j & 7)) << 4))
                                 : make_uint4(0, 0, 0, 0);
          const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int c0 = 8 * m + 2 * i;  // tokens c0, c0 + 1 (static after unrolling)
            const float2 u = __half22float2(h2[i]);
            const float va = c0 < 32 ? __uint_as_float(b0[c0]) : __uint_as_float(b1[c0 - 32]);
            const float vb = c0 < 32 ? __uint_as_float(b0[c0 + 1]) : __uint_as_float(b1[c0 - 31]);
            const float x0 = has_acc ? u.x - va : u.x;
            const float x1 = has_acc ? u.y - vb : u.y;
            pk[4 * m + i] = pack_f16(x0, x1);
            vmax = __hmax2_nan(vmax, __habs2(*reinterpret_cast<const __half2*>(&pk[4 * m + i])));
          }
        }
        tmem_st32(lane_base + Lo::cVf, pk);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&B->v_ready);
          mbar_arrive(&B->empty[s]);
        }
      } else if (lane == 0) {
        mbar_arrive(&B->empty[jj % kStages]);
      }
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
        // O(step) through staging buffer step & 1 (free once the store of step - 2 has
        // read it) and one TMA tile store per 64 columns
        unsigned char* ostage = sm + Lo::kOst + (step & 1) * Lo::kOstBuf;
        if (vw == 0 && lane == 0) {
          bulk_wait_read<1>();
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
            for (int b = 0; b < DV / 64; ++b) {
              if (p.cu_seqlens)
                tma_store_2d(&tmo, hv * DV + 64 * b, (int)(t_seq + (long long)step * kC),
                             ostage + b * 8192);
              else
                tma_store_3d(&tmo, hv * DV + 64 * b, step * kC, n, ostage + b * 8192);
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
    // ======================= state (warps 6-9) ================================
    __half2 hmax = __floats2half2_rn(0.f, 0.f);  // max |h| in its fp16 copy (NaN sticks)
    // h(0): h0 column j (or zeros); then per step the new state
    for (int step = -1; step < n_chunks; ++step) {
      const int jj = step + 1;  // the stage with gamma_last(jj)
      if (step >= 0) {
        if (!wait_warp(&B->mma_done, (step + 1) & 1, abort, p.err)) break;
        tc_fence_after();
      }
      const bool last = jj == n_chunks;
      float gl = 1.f;
      if (!last) {
        const int s = jj % kStages;
        if (!wait_warp(&B->full[s], (jj / kStages) & 1, abort, p.err)) break;
        gl = reinterpret_cast<const float*>(sm + s * Lo::kStage + Lo::kGv)[0];
      }
      // 64 columns (dk indices 64 hb ..) at a time
#pragma unroll
      for (int hb = 0; hb < DK / 64; ++hb) {
        float h[64];
        if (step < 0) {
#pragma unroll
          for (int i = 0; i < 64; ++i)
            h[i] = (p.h0 && jact) ? p.h0[hoff + (long long)(64 * hb + i) * DV + j] : 0.f;
        } else {
          uint32_t r0[32], r1[32];
          tmem_ld32_async(lane_base + Lo::cH + 64 * hb, r0);
          tmem_ld32_async(lane_base + Lo::cH + 64 * hb + 32, r1);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            h[i] = __uint_as_float(r0[i]);
            h[32 + i] = __uint_as_float(r1[i]);
          }
        }
        if (last) {
          if (p.hT && jact) {
#pragma unroll
            for (int i = 0; i < 64; ++i) p.hT[hoff + (long long)(64 * hb + i) * DV + j] = h[i];
          }
          continue;
        }
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          uint32_t hs[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) hs[i] = __float_as_uint(gl * h[32 * b + i]);
          tmem_st32(lane_base + Lo::cH + 64 * hb + 32 * b, hs);
        }
        uint32_t hf[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          hf[i] = pack_f16(h[2 * i], h[2 * i + 1]);
          hmax = __hmax2_nan(hmax, __habs2(*reinterpret_cast<const __half2*>(&hf[i])));
        }
        tmem_st32(lane_base + Lo::cHf + 32 * hb, hf);
      }
      if (last) break;
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&B->h_ready);
        mbar_arrive(&B->empty[jj % kStages]);
      }
      // the prologue's commit (phase 0) is waited for here, so that every later wait
      // names the phase right after the last one observed (a parity wait on a phase
      // two ahead would pass at once)
      if (step < 0 && !wait_warp(&B->mma_done, 0, abort, p.err)) break;
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
  gdn_chain_tc_kernel<DK, DV, DELTA><<<(unsigned)grid, kThreads, Lo::kAlloc, stream>>>(p, ws, mo);
  return cudaGetLastError();
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
