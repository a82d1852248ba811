// gdn_internal.h - launch parameters shared by the C ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

// One chunked-prefill forward call (sizes already validated by the ABI layer).
struct FwdParams {
  const void* q;      // [B, T, Hqk, dk]
  const void* k;      // [B, T, Hqk, dk]
  const void* v;      // [B, T, Hv, dv]
  const float* g;     // [B, T, Hv]
  const float* beta;  // [B, T, Hv]
  const float* h0;    // [N, Hv, dk, dv] or nullptr
  void* o;            // [B, T, Hv, dv]
  float* hT;          // [N, Hv, dk, dv] or nullptr
  const int32_t* cu_seqlens;  // [N + 1] or nullptr
  int N;              // sequences
  int T;              // tokens per row (packed total with cu_seqlens)
  int Hqk, Hv, dk, dv, chunk;
  float scale;
  unsigned* err;      // device error word: bounded waits record a timeout here
  int delta_rule;     // 1: gated delta rule (GDN); 0: no erase term (Mamba-2 SSD scan)
  // Fused prologue (prologue != 0): q and k arrive unnormalised and are divided by
  // sqrt(sum x^2 + kNormEps) per head vector; g holds the raw gate a and beta the raw
  // b, turned into g = -exp(A_log[h]) softplus(a + dt_bias[h]) and beta = sigmoid(b)
  // (A_log, dt_bias: [Hv] fp32 or nullptr for zeros).
  int prologue;
  const float* A_log;
  const float* dt_bias;
  // Kimi Delta Attention (kda != 0, dk = 128): g is [B, T, Hv, dk], one log-decay per
  // key channel; h_t = (I - beta k k^T) diag(exp g_t) h_{t-1} + beta k v^T.
  int kda;
  // GQA map: 0 grouped (v head hv reads q/k head hv / (Hv / Hqk)), 1 modulo (hv % Hqk)
  int head_map;
  // the chain kind: 1 the tcgen05 chain (one CTA per chain, the fp32 state in the
  // registers of its state warps, products in tensor memory, lookahead records); 0 the
  // mma.sync chain (dv tiles, one CTA each); as a flag of a call, -1 forces the
  // mma.sync chain and 0 leaves the choice to tc_chain_pays
  int tc_chain;
};
constexpr float kNormEps = 1e-6f;

// The q/k head that v head hv reads.
__host__ __device__ inline int qk_head(int hv, int Hqk, int Hv, int head_map) {
  return head_map ? hv % Hqk : hv / (Hv / Hqk);
}

// One decode step.
struct StepParams {
  const void* q;      // [N, Hqk, dk]
  const void* k;      // [N, Hqk, dk]
  const void* v;      // [N, Hv, dv]
  const float* g;     // [N, Hv]
  const float* beta;  // [N, Hv]
  float* h;           // [N, Hv, dk, dv], in place
  void* o;            // [N, Hv, dv]
  int N, Hqk, Hv, dk, dv;
  float scale;
  int delta_rule;     // 1: gated delta rule; 0: no erase term (Mamba-2 SSD)
  int prologue;       // as in FwdParams: raw q, k, gates a (in g) and b (in beta)
  const float* A_log;
  const float* dt_bias;
  int kda;            // 1: g is [N, Hv, dk], a per-channel decay of the state rows
  int head_map;       // as in FwdParams
};

// Workspace of the bf16 forward: one record per (chunk slot, v head), written
// by a prep kernel and read by a chain kernel.  16-bit tiles are row-major with
// their 16-byte chunks XOR-swizzled per row (the tensor cores' 128-byte swizzle:
// gdn::swz<64> for 64-column tiles, gdn::swzb<64> for [dk] wide ones, stored as
// 64-column blocks of 64 rows), so a verbatim bulk copy lands in shared memory
// as a ready tcgen05 operand.  Chunk c of a sequence, tokens t, s in [0, 64):
//
// Lookahead records (gated delta rule / Mamba-2 SSD on the tcgen05 chain:
// gdn_prep_tc.cu -> gdn_chain_tc.cu), the one-chunk lookahead form of the state read:
//   Wn   [64][dk]  W'(c) = gamma_last(c-1) W(c), W = Tm diag(beta gamma) K  (W'(0) = W(0))
//   Xt   [64][64]  X(c)^T: Xt[s][t] = X[t][s], X(c) = W(c) Kt(c-1)^T         (chunk 0: unused)
//   U    [dv][64]  U^T, U = Tm diag(beta) V; dv row j is the state column j
//   gv   fp32[132] gamma_last, 3 pad, gamma_i (64), e_j (64)
//   Qt   [64][dk]  Q~ = diag(scale gamma) Q (norm folded in with the prologue)
//   Kt   [64][dk]  Kt = diag(e) K, e_j = exp(G_last - G_j)
//   Pt   [64][64]  P^T: Pt[s][t] = P[t][s], P = tril(scale exp(G_t - G_s) q_t.k_s)
// so that V_new(c) = U(c) - W'(c) h(c-1) - X(c) V_new(c-1) needs only the state
// entering chunk c - 1 and chunk c - 1's V_new, and h(c + 1) = gamma_last(c)
// h(c) + Kt(c)^T V_new(c), O(c) = Q~(c) h(c) + P(c) V_new(c).  Without the erase
// term (SSD) Wn and Xt are zero and neither written nor read.
//
// Direct records (the mma.sync chain, gdn_chain.cu; written by gdn_prep.cu for the
// gated delta rule and SSD, by kda_prep.cu for Kimi Delta Attention):
//   W    [dk][64]  W^T, W = Tm diag(beta gamma) K (KDA: Tm diag(beta) (K * exp G)), swz<64>
//   Kt   [64][dk]  diag(e) K (KDA: K * exp(G_last - G)), swzb<64>
//   P    [64][64]  tril(scale exp(G_t - G_s) q_t.k_s) (KDA: the decay inside the channel
//                  sum), swz<64>
//   U    [dv][64]  U^T
//   gv   fp32[132] gamma_last, 3 pad, gamma (64), e (64) (KDA: [4 + c] = exp(G_last,c))
//   Qt   [64][dk]  Q~ = diag(scale gamma) Q (KDA: scale Q * exp(G))
// The mma.sync chain's dv tile t (16, 32 or 64 columns, one chain CTA each) is picked
// per call by dv_tile().
//
// Sequence n's chunk c lives in slot first_slot(n) + c: n * ceil(T / 64) for
// fixed-length rows; floor(cu[n] / 64) + n with cu_seqlens, which never
// overlaps because floor((a + L) / 64) - floor(a / 64) + 1 >= ceil(L / 64), and
// ends below floor(T / 64) + N + 1.
constexpr int kChunk = 64;
constexpr int kGvFloats = 132;

struct WsLayout {
  char* base;
  int dvt;                  // dv tile width of the mma.sync chain launch
  int look;                 // 1: lookahead records (tcgen05 chain); 0: direct records
  long long n_slots;        // chunk slots per v head
  long long slots_per_seq;  // fixed-length rows: ceil(T / 64); 0 with cu_seqlens
  long long task_bytes;     // bytes per record (a multiple of 128)
  // piece offsets within a record
  long long w_off, xt_off, u_off, gv_off, qt_off, kt_off, p_off;

  __host__ __device__ char* rec(long long slot, int hv, int Hv) const {
    return base + (slot * Hv + hv) * task_bytes;
  }
  // W'(c) (lookahead layout) or W^T (KDA layout)
  __host__ __device__ __half* W(long long s, int hv, int Hv) const {
    return reinterpret_cast<__half*>(rec(s, hv, Hv) + w_off);
  }
  __host__ __device__ __half* Xt(long long s, int hv, int Hv) const {
    return reinterpret_cast<__half*>(rec(s, hv, Hv) + xt_off);
  }
  __host__ __device__ __half* U(long long s, int hv, int Hv) const {
    return reinterpret_cast<__half*>(rec(s, hv, Hv) + u_off);
  }
  __host__ __device__ float* gv(long long s, int hv, int Hv) const {
    return reinterpret_cast<float*>(rec(s, hv, Hv) + gv_off);
  }
  __host__ __device__ __half* Qt(long long s, int hv, int Hv) const {
    return reinterpret_cast<__half*>(rec(s, hv, Hv) + qt_off);
  }
  __host__ __device__ __half* Kt(long long s, int hv, int Hv) const {
    return reinterpret_cast<__half*>(rec(s, hv, Hv) + kt_off);
  }
  // P^T (lookahead layout) or P (KDA layout)
  __host__ __device__ __half* P(long long s, int hv, int Hv) const {
    return reinterpret_cast<__half*>(rec(s, hv, Hv) + p_off);
  }
  __device__ long long first_slot(const FwdParams& p, int n) const {
    if (p.cu_seqlens) return (long long)(p.cu_seqlens[n] / kChunk) + n;
    return (long long)n * slots_per_seq;
  }
};

// dv tile of the mma.sync chain launch: 16 columns while chains x dv/16 CTAs fit on
// the 152 SMs, else 32 (and never wider than dv); without the erase term (no W stage)
// a 64-column tile where 32-column CTAs would need a second wave but whole-dv ones fit
// (dv = 64).
inline int dv_tile(const FwdParams& p) {
  const long long chains = (long long)p.N * p.Hv;
  if (chains * (p.dv / 16) <= 152) return 16;
  if (!p.delta_rule && !p.kda && p.dv == 64 && chains * 2 > 152 && chains <= 152) return 64;
  return 32;
}

// Which chain runs when the caller forces neither: the mma.sync chain walks one CTA
// per (chain, dv tile) at ~0.93 us a chunk, the tcgen05 chain one CTA per chain at
// ~1.72 us a chunk (both measured on GB300 at d = 128), so the tcgen05 chain is taken
// when the mma.sync chain would need about twice as many waves of CTAs over the SMs.
// KDA records exist for the mma.sync chain only.
inline bool tc_chain_pays(const FwdParams& p) {
  if (p.kda) return false;
  const long long chains = (long long)p.N * p.Hv;
  const long long tiles = p.dv / dv_tile(p);
  const long long waves_mma = (chains * tiles + 151) / 152, waves_tc = (chains + 151) / 152;
  return 172 * waves_tc < 93 * waves_mma;
}

// Layout for one call (sizes validated); base may be null when only sizing.
inline WsLayout ws_layout(const FwdParams& p, void* base) {
  WsLayout w;
  w.base = static_cast<char*>(base);
  w.dvt = dv_tile(p);
  w.look = (p.tc_chain && !p.kda) ? 1 : 0;
  if (p.cu_seqlens) {
    w.slots_per_seq = 0;
    w.n_slots = (long long)p.T / kChunk + p.N + 1;
  } else {
    w.slots_per_seq = ((long long)p.T + kChunk - 1) / kChunk;
    w.n_slots = w.slots_per_seq * p.N;
  }
  const long long wk = (long long)kChunk * p.dk * 2, wv = (long long)kChunk * p.dv * 2;
  const long long sq = (long long)kChunk * kChunk * 2;
  auto up = [](long long x, long long a) { return (x + a - 1) / a * a; };
  if (!w.look) {
    w.w_off = 0;
    w.kt_off = wk;
    w.p_off = 2 * wk;
    w.u_off = w.p_off + sq;
    w.gv_off = w.u_off + wv;
    w.qt_off = up(w.gv_off + kGvFloats * 4, 128);
    w.xt_off = 0;  // no X tile
    w.task_bytes = up(w.qt_off + wk, 128);
  } else {
    // the pieces of chunk c the chain stages with chunk c - 1's (W', X, U, gates),
    // then the rest (Q~, Kt, P^T)
    w.w_off = 0;
    w.xt_off = wk;
    w.u_off = w.xt_off + sq;
    w.gv_off = w.u_off + wv;
    w.qt_off = up(w.gv_off + kGvFloats * 4, 128);
    w.kt_off = w.qt_off + wk;
    w.p_off = w.kt_off + wk;
    w.task_bytes = up(w.p_off + sq, 128);
  }
  return w;
}
inline size_t ws_bytes(const WsLayout& w, int Hv) { return (size_t)(w.n_slots * Hv * w.task_bytes); }
// Workspace bytes for either record layout of these sizes (the size functions of the
// ABI report this, so one buffer serves every path).
inline size_t ws_bytes_any(const FwdParams& p) {
  FwdParams a = p, b = p;
  a.tc_chain = 0;
  b.tc_chain = 1;
  const size_t x = ws_bytes(ws_layout(a, nullptr), p.Hv), y = ws_bytes(ws_layout(b, nullptr), p.Hv);
  return x > y ? x : y;
}

// Slot -> (sequence, chunk of that sequence); false for a slot no chunk uses.
__device__ inline bool locate_chunk(const FwdParams& p, const WsLayout& ws, long long slot, int* n,
                                    int* c) {
  if (!p.cu_seqlens) {
    *n = (int)(slot / ws.slots_per_seq);
    *c = (int)(slot % ws.slots_per_seq);
    return *n < p.N;
  }
  int lo = 0, hi = p.N - 1;  // largest n with first_slot(n) <= slot
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((long long)(p.cu_seqlens[mid] / kChunk) + mid <= slot) lo = mid; else hi = mid - 1;
  }
  const long long first = (long long)(p.cu_seqlens[lo] / kChunk) + lo;
  const long long len = (long long)p.cu_seqlens[lo + 1] - p.cu_seqlens[lo];
  if (slot < first || slot - first >= (len + kChunk - 1) / kChunk) return false;
  *n = lo;
  *c = (int)(slot - first);
  return true;
}

// Tensor map of a row-major [rows, cols] bf16 matrix, boxes of 64 x 64 with the
// 128-byte swizzle (gdn_prep.cu); false if the driver refuses it.
bool make_tensor_map_bf16(CUtensorMap* m, const void* base, long long rows, long long cols);
// Tensor map of a row-major [planes, rows, cols] bf16 tensor, boxes of 64 x 64 x 1
// with the 128-byte swizzle; a store clips at each plane's `rows`.
bool make_tensor_map_bf16_3d(CUtensorMap* m, const void* base, long long planes, long long rows,
                             long long cols);

// Launchers: return cudaSuccess or the launch error.  Each validates nothing.
cudaError_t launch_prep(const FwdParams& p, const WsLayout& ws, cudaStream_t stream);
// Kimi Delta Attention records (kda_prep.cu; p.kda, dk = 128).
cudaError_t launch_kda_prep(const FwdParams& p, const WsLayout& ws, cudaStream_t stream);
// Lookahead records for the tcgen05 chain (gated delta rule / SSD).
cudaError_t launch_prep_tc(const FwdParams& p, const WsLayout& ws, cudaStream_t stream);
// The mma.sync chain (dv tiles; direct records).
cudaError_t launch_chain(const FwdParams& p, const WsLayout& ws, cudaStream_t stream);
// The tcgen05 chain (one CTA per chain; lookahead records).
cudaError_t launch_chain_tc(const FwdParams& p, const WsLayout& ws, cudaStream_t stream);
// Input check of an _ex call (g, beta in their domains, cu_seqlens ordered): records
// kErrInput in the device error word.
cudaError_t launch_check_inputs(const FwdParams& p, cudaStream_t stream);
// The fp32 forward (gdn_fwd_f32.cu): fp32 records of f32_rec_bytes(p) per (chunk slot,
// v head) in the slots of ws_layout(p, base), then the chain.
size_t f32_rec_bytes(const FwdParams& p);
cudaError_t launch_fwd_f32(const FwdParams& p, const WsLayout& ws, cudaStream_t stream);
cudaError_t launch_step_bf16(const StepParams& p, cudaStream_t stream);
cudaError_t launch_step_f32(const StepParams& p, cudaStream_t stream);

// The device error word (bounded waits); defined in gdn_abi.cu.
cudaError_t read_and_clear_device_error(unsigned* out, cudaStream_t stream);

}  // namespace gdn
