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
};
constexpr float kNormEps = 1e-6f;

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
};

// Workspace of the bf16 forward: one record per (chunk slot, v head), written
// by gdn_prep and read by gdn_chain.  16-bit tiles are row-major with their
// 16-byte chunks XOR-swizzled per row (gdn::swz<width>), so a verbatim bulk
// copy lands in shared memory ready for conflict-free ldmatrix:
//   W    [dk][64]   W^T, W = Tm diag(beta gamma) K, swz<64>, fp16
//   Kt   [64][dk]   diag(e) K, e_j = exp(G_last - G_j), swzb<64> (64-column
//                   blocks), fp16
//   P    [64][64]   tril(scale exp(G_i - G_j) q_i.k_j), swz<64>, fp16
//   U    [dv][64]   U^T, U = Tm diag(beta) V, swz<64>, fp16: the t-column dv
//                   tile j is the contiguous rows [j t, (j + 1) t)
//   gv   fp32 [132] gamma_last, 3 pad, gamma_i = exp(G_i) for the 64 rows, then
//                   e_j for the 64 rows (norm factors folded in with the prologue)
//   Qt   [64][dk]   Q~ = diag(scale gamma) Q (norm folded in), swzb<64>, fp16: the
//                   output's left factor, in the layout the chain stages q in
// Kimi Delta Attention records (kda_prep.cu, dk = 128) are the same tiles with
// the per-channel gate inside (W = Tm diag(beta) (K * exp G), Kt = K *
// exp(G_last - G), P with exp(G_i - G_j) inside the channel sum, Qt = scale Q *
// exp(G)) and gv[4 + c] = exp(G_last,c) for the 128 key channels.
// The block path (ws.blocks) reads q itself and its chunk records carry no Qt.
// Every 16-bit tile is in the tensor cores' 128-byte-swizzled layout, so the
// same bytes serve ldmatrix loads and tcgen05 operand descriptors.
// The dv tile t (16 or 32 columns, one chain CTA each) is picked per call by
// dv_tile(): the narrowest that still leaves at most ~one CTA per SM, since
// every chain CTA must take in the whole W, Kt, P and q of each chunk.
// Sequence n's chunk c lives in slot first_slot(n) + c: n * ceil(T / 64) for
// fixed-length rows; floor(cu[n] / 64) + n with cu_seqlens, which never
// overlaps because floor((a + L) / 64) - floor(a / 64) + 1 >= ceil(L / 64), and
// ends below floor(T / 64) + N + 1.
constexpr int kChunk = 64;
constexpr int kGvFloats = 132;

// The block path (gdn_pair.cu; gated delta rule, dk = dv = 128) adds one pair
// record per (128-token block slot, v head) after the chunk records: block b of
// a sequence is its chunks 2b and 2b + 1, and its record holds
//   N    [2][dk][64]     N = Kb^T Wb, the block's state transition h <- gamma h
//                        - N h + B (swzb<dk>, fp16; K-major over the input dk)
//   B    [dv/64][dk][64] B = Kb^T Ub (swzb<dk>, fp16)
//   H    [dv/64][dk][64] the fp16 state entering the block (swzb<dk>)
//   gp   fp32            gamma_last of the block (16 bytes)
// Block slots follow the chunk slots' rule with 128 tokens: n * ceil(T / 128),
// or floor(cu[n] / 128) + n.
constexpr int kBlock = 128;

struct WsLayout {
  char* base;
  int dvt;                  // dv tile width of the chain launch
  long long n_slots;        // chunk slots per v head
  long long slots_per_seq;  // fixed-length rows: ceil(T / 64); 0 with cu_seqlens
  long long task_bytes, kt_off, p_off, u_off, gv_off, qt_off;
  int qrec;                 // 1: the records carry the Qt tile (every chunk-chain run)
  int blocks;               // 1: the block path runs (pair records present)
  long long n_bslots, bslots_per_seq, pair_off, pair_bytes, pb_off, ph_off, pg_off;
  // fused scan launch: [n_bslots][Hv] pair-done flags, [n_bslots][Hv][2]
  // stored-state flags, then the task counter (zeroed before each launch)
  long long flag_off, flag_bytes;
  int hv_count;

  __host__ __device__ unsigned* pair_flags() const {
    return reinterpret_cast<unsigned*>(base + flag_off);
  }
  __host__ __device__ unsigned* scan_flags() const { return pair_flags() + n_bslots * hv_count; }
  __host__ __device__ unsigned* task_counter() const {
    return pair_flags() + n_bslots * hv_count * 3;
  }

  __host__ __device__ char* prec(long long bslot, int hv, int Hv) const {
    return base + pair_off + (bslot * Hv + hv) * pair_bytes;
  }
  __host__ __device__ __half* PN(long long b, int hv, int Hv) const {
    return reinterpret_cast<__half*>(prec(b, hv, Hv));
  }
  __host__ __device__ __half* PB(long long b, int hv, int Hv) const {
    return reinterpret_cast<__half*>(prec(b, hv, Hv) + pb_off);
  }
  __host__ __device__ __half* PH(long long b, int hv, int Hv) const {
    return reinterpret_cast<__half*>(prec(b, hv, Hv) + ph_off);
  }
  __host__ __device__ float* PG(long long b, int hv, int Hv) const {
    return reinterpret_cast<float*>(prec(b, hv, Hv) + pg_off);
  }
  __device__ long long first_bslot(const FwdParams& p, int n) const {
    if (p.cu_seqlens) return (long long)(p.cu_seqlens[n] / kBlock) + n;
    return (long long)n * bslots_per_seq;
  }

  __host__ __device__ char* rec(long long slot, int hv, int Hv) const {
    return base + (slot * Hv + hv) * task_bytes;
  }
  __host__ __device__ __half* W(long long s, int hv, int Hv) const {
    return reinterpret_cast<__half*>(rec(s, hv, Hv));
  }
  __host__ __device__ __half* Kt(long long s, int hv, int Hv) const {
    return reinterpret_cast<__half*>(rec(s, hv, Hv) + kt_off);
  }
  __host__ __device__ __half* P(long long s, int hv, int Hv) const {
    return reinterpret_cast<__half*>(rec(s, hv, Hv) + p_off);
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
  __device__ long long first_slot(const FwdParams& p, int n) const {
    if (p.cu_seqlens) return (long long)(p.cu_seqlens[n] / kChunk) + n;
    return (long long)n * slots_per_seq;
  }
};

// dv tile of the chain launch: 16 columns while chains x dv/16 CTAs fit on the
// 152 SMs, else 32 (and never wider than dv); without the erase term (no W stage)
// a 64-column tile where 32-column CTAs would need a second wave but whole-dv
// ones fit (dv = 64).
inline int dv_tile(const FwdParams& p) {
  const long long chains = (long long)p.N * p.Hv;
  if (chains * (p.dv / 16) <= 152) return 16;
  if (!p.delta_rule && !p.kda && p.dv == 64 && chains * 2 > 152 && chains <= 152) return 64;
  return 32;
}

// Whether the 128-token block path (gdn_block.cu) runs for the shapes it covers:
// on when the environment variable GDN_BLOCK_PATH is "1" at first use (gdn_abi.cu).
bool block_path_enabled();

// Layout for one call (sizes validated); base may be null when only sizing.
inline WsLayout ws_layout(const FwdParams& p, void* base) {
  WsLayout w;
  w.base = static_cast<char*>(base);
  w.dvt = dv_tile(p);
  if (p.cu_seqlens) {
    w.slots_per_seq = 0;
    w.n_slots = (long long)p.T / kChunk + p.N + 1;
  } else {
    w.slots_per_seq = ((long long)p.T + kChunk - 1) / kChunk;
    w.n_slots = w.slots_per_seq * p.N;
  }
  const long long wk = (long long)kChunk * p.dk * 2, wv = (long long)kChunk * p.dv * 2;
  w.kt_off = wk;
  w.p_off = 2 * wk;
  w.u_off = w.p_off + (long long)kChunk * kChunk * 2;
  w.gv_off = w.u_off + wv;
  w.qt_off = (w.gv_off + kGvFloats * 4 + 127) / 128 * 128;
  w.blocks = !p.kda && p.delta_rule && p.dk == 128 && p.dv == 128 && block_path_enabled();
  // records on 128-byte lines; a chain run's records add the Qt tile
  w.qrec = p.kda || !w.blocks;
  w.task_bytes = w.qrec ? (w.qt_off + wk + 127) / 128 * 128 : w.qt_off;
  if (p.cu_seqlens) {
    w.bslots_per_seq = 0;
    w.n_bslots = (long long)p.T / kBlock + p.N + 1;
  } else {
    w.bslots_per_seq = ((long long)p.T + kBlock - 1) / kBlock;
    w.n_bslots = w.bslots_per_seq * p.N;
  }
  w.pair_off = w.n_slots * p.Hv * w.task_bytes;
  w.pb_off = (long long)p.dk * p.dk * 2;
  w.ph_off = w.pb_off + (long long)p.dk * p.dv * 2;
  w.pg_off = w.ph_off + (long long)p.dk * p.dv * 2;
  w.pair_bytes = w.blocks ? (w.pg_off + 16 + 127) / 128 * 128 : 0;
  w.hv_count = p.Hv;
  w.flag_off = w.pair_off + w.n_bslots * p.Hv * w.pair_bytes;
  w.flag_bytes = w.blocks ? (w.n_bslots * p.Hv * 3 * 4 + 4 + 127) / 128 * 128 : 0;
  return w;
}
inline size_t ws_bytes(const WsLayout& w, int Hv) {
  return (size_t)(w.n_slots * Hv * w.task_bytes + w.n_bslots * Hv * w.pair_bytes + w.flag_bytes);
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

// Block slot -> (sequence, block of that sequence); false for a slot no block uses.
__device__ inline bool locate_block(const FwdParams& p, const WsLayout& ws, long long bslot, int* n,
                                    int* b) {
  if (!p.cu_seqlens) {
    *n = (int)(bslot / ws.bslots_per_seq);
    *b = (int)(bslot % ws.bslots_per_seq);
    return *n < p.N;
  }
  int lo = 0, hi = p.N - 1;  // largest n with first_bslot(n) <= bslot
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((long long)(p.cu_seqlens[mid] / kBlock) + mid <= bslot) lo = mid; else hi = mid - 1;
  }
  const long long first = (long long)(p.cu_seqlens[lo] / kBlock) + lo;
  const long long len = (long long)p.cu_seqlens[lo + 1] - p.cu_seqlens[lo];
  if (bslot < first || bslot - first >= (len + kBlock - 1) / kBlock) return false;
  *n = lo;
  *b = (int)(bslot - first);
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
cudaError_t launch_chain(const FwdParams& p, const WsLayout& ws, cudaStream_t stream);
// The block path (ws.blocks): pair transitions, the block scan, the block output.
cudaError_t launch_pair(const FwdParams& p, const WsLayout& ws, cudaStream_t stream);
cudaError_t launch_scan(const FwdParams& p, const WsLayout& ws, cudaStream_t stream);
cudaError_t launch_out(const FwdParams& p, const WsLayout& ws, cudaStream_t stream);
// The scan and the block output in one launch (fixed-length rows, few enough
// chains to leave SMs for the output work); scan_out_fused says when.
bool scan_out_fused(const FwdParams& p);
cudaError_t launch_scan_out(const FwdParams& p, const WsLayout& ws, cudaStream_t stream,
                            bool pairs);
cudaError_t launch_fwd_f32(const FwdParams& p, cudaStream_t stream);
cudaError_t launch_step_bf16(const StepParams& p, cudaStream_t stream);
cudaError_t launch_step_f32(const StepParams& p, cudaStream_t stream);

// The device error word (bounded waits); defined in gdn_abi.cu.
cudaError_t read_and_clear_device_error(unsigned* out, cudaStream_t stream);

}  // namespace gdn
