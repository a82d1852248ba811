/*
 * gdn.h - C ABI of libgdn.so: Gated DeltaNet chunked-prefill forward and the
 * one-token decode step on an sm_103a GPU.
 *
 * The operation (per sequence n and value head hv, tokens t in order):
 *
 *     S_t = exp(g_t) * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *     o_t = S_t (scale * q_t)
 *
 * the gated delta rule of Gated DeltaNet, which "Empowering Hybrid Attention
 * Models on NPUs" (§2.1, "Architecture of Linear-Attention Hybrids") describes
 * as a fixed-size per-head state updated from K_t and V_t, then read with Q_t.
 * The forward computes it chunkwise as that page's Map-Reduce-Map operators
 * #1 Gate, #2 KKT, #3 Solve, #4 W/U, #5 H, #6 O (§2.1, Figure 1(b)), reading
 * the state before updating it in place (§5, chunk-first order, Figure 10(b)).
 * The state is stored transposed: h = S^T, [dk][dv] row-major.
 *
 * Conventions shared by every entry point
 *  - Every tensor pointer is DEVICE memory of the current device, dense
 *    row-major in the stated shape, 16-byte aligned.  The caller owns every
 *    buffer; the library keeps no pointer and no allocation after a call
 *    (only gdn_chunk_fwd takes a temporary workspace, see gdn_chunk_fwd_ex).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream).  GDN_OK means the launch was enqueued.  Kernel faults
 *    show up on the stream like any CUDA error.
 *  - GQA: value head hv reads query/key head hv / (Hv / Hqk) ("grouped");
 *    gdn_chunk_fwd_ex and gdn_recurrent_step_ex also take hv % Hqk ("modulo",
 *    GDN_FLAG_HEAD_MAP_MODULO).
 *  - q and k are expected L2-normalised per head vector, beta in [0, 1] and
 *    g <= 0 (a log-decay).  The host does not read them; GDN_FLAG_CHECK_INPUTS
 *    of the _ex entry points adds a device pass that checks g, beta and
 *    cu_seqlens and reports a violation through gdn_device_status.
 *  - Range of the bf16 path: the on-chip products take fp16 operands (the
 *    state entering each chunk, V_new = U - W h and the scaled copies of q, k
 *    and v are rounded to fp16 once), so |v|, the state and V_new must stay
 *    below fp16's 65504.  A value outside that range (or not a number) in the
 *    state or V_new is recorded and reported by the next gdn_device_status as
 *    GDN_ERR_INVALID_ARG: that call's result is not exact.
 *  - Errors: a non-OK status means nothing was launched (except GDN_ERR_CUDA,
 *    which reports a failed launch).  gdn_last_error() gives a one-line
 *    description, per calling thread.  Nothing prints, aborts or throws.
 *  - No environment variable or other process state changes what a call does.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* gdn_stream_t; /* ABI-identical to cudaStream_t */

/* Flags of the _ex entry points (gdn_chunk_fwd_ex, gdn_chunk_fwd_prologue_ex,
 * ssd_chunk_fwd_ex, kda_chunk_fwd_ex, gdn_recurrent_step_ex): bitwise or, 0 = the
 * plain call.  An unknown bit is GDN_ERR_INVALID_ARG. */
enum {
  /* GQA map hv % Hqk instead of hv / (Hv / Hqk) (the replication of the GQA
   * marshaller in "Exp 2026-07-13 — Linear-Attention Scans on the NPU", §4) */
  GDN_FLAG_HEAD_MAP_MODULO = 1u,
  /* before the forward (or step), one device pass checks every g <= 0 and
   * finite, every beta in [0, 1], and cu_seqlens running from 0 to T without
   * going down; a violation is reported by the next gdn_device_status as
   * GDN_ERR_INVALID_ARG (the call itself still runs) */
  GDN_FLAG_CHECK_INPUTS = 2u,
  /* the chunk-serial operators on the 5th-generation tensor cores: one CTA per
   * (sequence, v head), the fp32 state in registers, every product's left
   * factor and accumulator in tensor memory, the one-chunk lookahead form of
   * the state read (the forwards' _ex entry points; KDA returns
   * GDN_ERR_UNSUPPORTED).  Same function and tolerances; uses one SM per chain
   * where the dv-tile chain uses dv / 16 (or / 32), so it pays off when many
   * chains share the GPU.  Without either chain flag every forward picks one
   * by itself from the number of chains (the tensor-memory chain once the
   * dv-tile chain would need more waves of CTAs over the SMs than it saves
   * per chunk). */
  GDN_FLAG_TC_CHAIN = 4u,
  /* the dv-tile chain (warp-level MMAs, dv / 16 or dv / 32 CTAs per chain)
   * whatever the automatic choice; with GDN_FLAG_TC_CHAIN as well the call is
   * GDN_ERR_INVALID_ARG */
  GDN_FLAG_DV_TILE_CHAIN = 8u
};

typedef enum {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = 1, /* NULL pointer, bad size, misaligned pointer, Hv % Hqk != 0 */
  GDN_ERR_UNSUPPORTED = 2, /* valid but not built: dk, dv or chunk not in {64, 128} */
  GDN_ERR_CUDA = 3,        /* a CUDA call failed (launch error, no device) */
  GDN_ERR_TIMEOUT = 4      /* a bounded device-side wait gave up (see gdn_device_status) */
} gdn_status;

/*
 * gdn_chunk_fwd - chunked-prefill forward, bf16 q/k/v/o, fp32 gates and state.
 *
 *   q, k   [B, T, Hqk, dk] bf16       (with cu_seqlens: [1, T, Hqk, dk])
 *   v      [B, T, Hv, dv]  bf16
 *   g      [B, T, Hv] fp32  log-decay per token and value head
 *   beta   [B, T, Hv] fp32
 *   h0     [N, Hv, dk, dv] fp32 initial state, or NULL for zeros
 *   o      [B, T, Hv, dv]  bf16 output (written; fp32 accumulation, rounded
 *          to nearest even once)
 *   hT     [N, Hv, dk, dv] fp32 final state, or NULL to skip; may equal h0
 *          (each state tile is read before it is overwritten)
 *   B      number of sequences N.  Without cu_seqlens the batch is B rows of
 *          T tokens; with cu_seqlens it is one packed row of T tokens.
 *   T      tokens per row (packed total with cu_seqlens); T = 0 is a no-op
 *          that copies h0 (or zeros) to hT
 *   chunk  chunk length C of the chunkwise form, 64 or 128; chunks restart
 *          at every sequence start, the last one may be partial.  The chunked
 *          recurrence gives the same o and hT for any C (it is exact, not an
 *          approximation), so a 128-token chunk is computed as two 64-token
 *          chunks: both values give identical results and timings here.
 *   scale  multiplies q (o_t = S_t (scale q_t)), usually dk^-0.5
 *   cu_seqlens  NULL, or DEVICE int32 [B + 1]: 0 = cu[0] <= cu[1] <= ... <=
 *          cu[B] = T (not checked on the host; empty sequences allowed)
 *
 * Supported: dk, dv in {64, 128}; Hv a multiple of Hqk.
 */
gdn_status gdn_chunk_fwd(const void* q, const void* k, const void* v, const float* g,
                         const float* beta, const float* h0, void* o, float* hT, int B, int T,
                         int Hqk, int Hv, int dk, int dv, int chunk, float scale,
                         const int32_t* cu_seqlens, gdn_stream_t stream);

/*
 * gdn_chunk_fwd_workspace_size - bytes of device workspace gdn_chunk_fwd_ex
 * needs for these sizes with any flags (has_cu_seqlens: 1 if cu_seqlens will
 * be passed).  The bf16 forward runs in two launches: the chunk-parallel
 * operators #1-#4 (Gate, KKT, Solve, W/U) write one record per (64-token
 * chunk, v head) - W, diag(e) K, P, U^T and diag(scale gamma) Q in fp16 plus
 * the gate factors (72.6 KiB at d = 128; 80.6 KiB for the tensor-memory chain,
 * whose records add the lookahead tile X) - and the chunk-serial launch (#5 H
 * with #6 O) reads them.  Returns 0 for sizes gdn_chunk_fwd would reject.
 */
size_t gdn_chunk_fwd_workspace_size(int B, int T, int Hqk, int Hv, int dk, int dv, int chunk,
                                    int has_cu_seqlens);

/*
 * gdn_chunk_fwd_chain_kind - which chunk-serial kernel a bf16 forward runs for
 * n_seqs sequences (B, or the number of packed sequences) of Hv v heads with
 * these head dims and flags: 1 the tensor-memory chain, 0 the dv-tile chain,
 * -1 for sizes or flags the forward would reject.  delta_rule: 1 for
 * gdn_chunk_fwd(_prologue)(_ex), 0 for ssd_chunk_fwd(_ex).  Host only; KDA
 * forwards always run the dv-tile chain.
 */
int gdn_chunk_fwd_chain_kind(int n_seqs, int Hv, int dk, int dv, int delta_rule, unsigned flags);

/*
 * gdn_chunk_fwd_ex - gdn_chunk_fwd with `flags` (GDN_FLAG_*: the GQA map, the
 * input check, the tensor-memory chain) and a caller-provided device workspace
 * of at least gdn_chunk_fwd_workspace_size(...) bytes, 256-byte aligned.  The
 * workspace is overwritten; calls sharing it must be ordered on one stream.
 * Returns GDN_ERR_INVALID_ARG if it is NULL, misaligned or too small, or for
 * an unknown flag bit.  (gdn_chunk_fwd itself takes the workspace from the
 * device's stream-ordered memory pool with cudaMallocAsync/cudaFreeAsync on
 * `stream`.)
 */
gdn_status gdn_chunk_fwd_ex(const void* q, const void* k, const void* v, const float* g,
                            const float* beta, const float* h0, void* o, float* hT, int B, int T,
                            int Hqk, int Hv, int dk, int dv, int chunk, float scale,
                            const int32_t* cu_seqlens, unsigned flags, void* workspace,
                            size_t workspace_bytes, gdn_stream_t stream);

/*
 * gdn_chunk_fwd_noalloc - gdn_chunk_fwd for callers that must not allocate
 * device memory: it runs on a workspace of 32 MiB compiled into the library
 * (a static device array) and makes no allocation call of any kind.  No
 * passage of the pages corresponds to it; it exists for callers such as a
 * serving loop that may not take an allocator's locks or risk the device
 * synchronisation an allocation can imply, or code embedded in a runtime that
 * owns all device memory through its own pool.
 *  - Limit: gdn_chunk_fwd_workspace_size(...) must be at most 32 MiB (about
 *    406 chunk-and-v-head records at dk = dv = 128: the size covers the
 *    larger, 80.6 KiB record of the tensor-memory chain; e.g. 4096 tokens x 6
 *    v heads); larger sizes return GDN_ERR_INVALID_ARG and launch nothing.
 *  - Every GPU that runs the library's device code keeps those 32 MiB until
 *    the process exits.
 *  - Every call looks up the array's device address on the current device
 *    (cudaGetSymbolAddress, which allocates nothing); the first call on a
 *    device also loads the library's device code there, so make it before any
 *    stream capture.
 *  - All calls share the one array and its contents persist between calls;
 *    each call rewrites every byte it later reads, so nothing needs clearing,
 *    but calls that overlap on the GPU (different streams, or different host
 *    threads without ordering) race on it.
 * Arguments, results and other errors are those of gdn_chunk_fwd.
 */
gdn_status gdn_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const float* g,
                                 const float* beta, const float* h0, void* o, float* hT, int B,
                                 int T, int Hqk, int Hv, int dk, int dv, int chunk, float scale,
                                 const int32_t* cu_seqlens, gdn_stream_t stream);

/* gdn_chunk_fwd_f32 - as gdn_chunk_fwd with fp32 q, k, v and o (fp32 throughout).
 * One fused launch per call; no workspace. */
gdn_status gdn_chunk_fwd_f32(const float* q, const float* k, const float* v, const float* g,
                             const float* beta, const float* h0, float* o, float* hT, int B,
                             int T, int Hqk, int Hv, int dk, int dv, int chunk, float scale,
                             const int32_t* cu_seqlens, gdn_stream_t stream);

/*
 * gdn_recurrent_step - one decode token per sequence, continuing from a state
 * (the rule above applied once; the decode path of "Empowering Hybrid
 * Attention Models on NPUs", §7.3, and the per-token recurrence of "Exp
 * 2026-07-13 — Linear-Attention Scans on the NPU", §4).
 *
 *   q, k  [N, Hqk, dk] bf16;  v [N, Hv, dv] bf16;  g, beta [N, Hv] fp32
 *   h     [N, Hv, dk, dv] fp32, read and overwritten in place
 *   o     [N, Hv, dv] bf16 output
 */
gdn_status gdn_recurrent_step(const void* q, const void* k, const void* v, const float* g,
                              const float* beta, float* h, void* o, int N, int Hqk, int Hv,
                              int dk, int dv, float scale, gdn_stream_t stream);

/*
 * gdn_recurrent_step_ex - gdn_recurrent_step with `flags`:
 * GDN_FLAG_HEAD_MAP_MODULO (the GQA map, as the prefill that produced h used)
 * and GDN_FLAG_CHECK_INPUTS (g and beta of this token checked on the device).
 */
gdn_status gdn_recurrent_step_ex(const void* q, const void* k, const void* v, const float* g,
                                 const float* beta, float* h, void* o, int N, int Hqk, int Hv,
                                 int dk, int dv, float scale, unsigned flags,
                                 gdn_stream_t stream);

/* gdn_recurrent_step_f32 - as gdn_recurrent_step with fp32 q, k, v and o. */
gdn_status gdn_recurrent_step_f32(const float* q, const float* k, const float* v,
                                  const float* g, const float* beta, float* h, float* o, int N,
                                  int Hqk, int Hv, int dk, int dv, float scale,
                                  gdn_stream_t stream);

/*
 * gdn_chunk_fwd_prologue(_ex) - gdn_chunk_fwd with the projection-side
 * elementwise steps fused into the first kernel: q and k arrive unnormalised
 * and each head vector is divided by sqrt(sum x^2 + 1e-6); the gates arrive
 * raw, as a (in the g slot) and b (in the beta slot), [B, T, Hv] fp32:
 *
 *   g_t = -exp(A_log[h]) * softplus(a_t + dt_bias[h]),   beta_t = sigmoid(b_t)
 *
 * with A_log, dt_bias [Hv] fp32 per v head, or NULL for zeros (g_t =
 * -softplus(a_t)).  The pages state only that the projection-side operators
 * are fused ("Empowering Hybrid Attention Models on NPUs", §7 Implementation:
 * operator fusion of the projections); this form is the GDN gate with a
 * per-head decay rate and step bias.  The norms never materialise normalised
 * tensors: they are folded into the row and column factors the kernels apply
 * anyway.  Other arguments, the workspace and errors as gdn_chunk_fwd(_ex).
 * gdn_recurrent_step_prologue is the decode step with the same prologue.
 */
gdn_status gdn_chunk_fwd_prologue(const void* q, const void* k, const void* v, const float* a,
                                  const float* b, const float* A_log, const float* dt_bias,
                                  const float* h0, void* o, float* hT, int B, int T, int Hqk,
                                  int Hv, int dk, int dv, int chunk, float scale,
                                  const int32_t* cu_seqlens, gdn_stream_t stream);
gdn_status gdn_chunk_fwd_prologue_ex(const void* q, const void* k, const void* v, const float* a,
                                     const float* b, const float* A_log, const float* dt_bias,
                                     const float* h0, void* o, float* hT, int B, int T, int Hqk,
                                     int Hv, int dk, int dv, int chunk, float scale,
                                     const int32_t* cu_seqlens, unsigned flags, void* workspace,
                                     size_t workspace_bytes, gdn_stream_t stream);
gdn_status gdn_recurrent_step_prologue(const void* q, const void* k, const void* v,
                                       const float* a, const float* b, const float* A_log,
                                       const float* dt_bias, float* h, void* o, int N, int Hqk,
                                       int Hv, int dk, int dv, float scale, gdn_stream_t stream);

/*
 * Mamba-2 SSD scan - the same chunked scan without the delta rule's erase term
 * ("Exp 2026-07-13 — Linear-Attention Scans on the NPU", §1 and §3: the SSM
 * scan's four matrix stages per chunk - the C B^T gram, the intra-chunk output,
 * the chunk state and the inter-chunk output).  Per (sequence, v head), tokens
 * in order, with C -> q, B -> k, x -> v, the per-token log-decay dt A -> g and
 * the input step dt -> beta:
 *
 *   S_t = exp(g_t) S_{t-1} + beta_t v_t k_t^T,      o_t = S_t (scale q_t)
 *
 * (the gated delta rule above with (I - beta_t k_t k_t^T) replaced by I; the
 * state is h = S^T, [dk = d_state][dv = head_dim]).  Arguments, layouts, sizes,
 * grouping of q/k heads (B/C groups), workspace (gdn_chunk_fwd_workspace_size)
 * and errors are those of the gdn_* counterpart; beta may exceed 1 here.  The
 * same kernels run with the KKT gram and the W term switched off (Tm = I,
 * W = 0, U = diag(beta) V).
 */
gdn_status ssd_chunk_fwd(const void* q, const void* k, const void* v, const float* g,
                         const float* beta, const float* h0, void* o, float* hT, int B, int T,
                         int Hqk, int Hv, int dk, int dv, int chunk, float scale,
                         const int32_t* cu_seqlens, gdn_stream_t stream);
gdn_status ssd_chunk_fwd_ex(const void* q, const void* k, const void* v, const float* g,
                            const float* beta, const float* h0, void* o, float* hT, int B, int T,
                            int Hqk, int Hv, int dk, int dv, int chunk, float scale,
                            const int32_t* cu_seqlens, unsigned flags, void* workspace,
                            size_t workspace_bytes, gdn_stream_t stream);
gdn_status ssd_chunk_fwd_f32(const float* q, const float* k, const float* v, const float* g,
                             const float* beta, const float* h0, float* o, float* hT, int B,
                             int T, int Hqk, int Hv, int dk, int dv, int chunk, float scale,
                             const int32_t* cu_seqlens, gdn_stream_t stream);
/* one decode token of the SSD recurrence: h <- exp(g) h + beta k v^T; o = h^T (scale q) */
gdn_status ssd_recurrent_step(const void* q, const void* k, const void* v, const float* g,
                              const float* beta, float* h, void* o, int N, int Hqk, int Hv,
                              int dk, int dv, float scale, gdn_stream_t stream);
gdn_status ssd_recurrent_step_f32(const float* q, const float* k, const float* v,
                                  const float* g, const float* beta, float* h, float* o, int N,
                                  int Hqk, int Hv, int dk, int dv, float scale,
                                  gdn_stream_t stream);

/*
 * Kimi Delta Attention (KDA) - the delta rule with a per-key-channel gate.
 * "Empowering Hybrid Attention Models on NPUs" runs GDN and KDA through the same
 * Map-Reduce-Map chunkwise paradigm (§2.1, Figure 1); KDA's gate is one fp32
 * log-decay per token, head and key channel (Figure 4(a) prices it at 31.33 MiB
 * against GDN's 21.41 MiB at T = 2048, H = 10).  The pages print no formula; the
 * reading implemented here replaces GDN's scalar decay by a diagonal one over the
 * key channels, applied before the delta rule reads the state.  Per (sequence,
 * v head), tokens in order, with h = S^T [dk][dv]:
 *
 *   h_t = (I - beta_t k_t k_t^T) diag(exp g_t) h_{t-1} + beta_t k_t v_t^T,
 *   o_t = h_t^T (scale q_t),                      g_t in R^dk, g_t <= 0.
 *
 * Arguments, layouts, ownership, streams and errors are those of gdn_chunk_fwd
 * (bf16 q, k, v, o; fp32 state; GQA; cu_seqlens), except:
 *   g     [B, T, Hv, dk] fp32, one log-decay per key channel, 16-byte aligned;
 *         exact to the tolerance for g >= -10 per token and channel (the chunk
 *         grams split exp(G_i - G_j) around each 16-token block's middle token,
 *         and a factor must stay a normal fp32 number); a value below -10 (or
 *         NaN) is reported by the next gdn_device_status as GDN_ERR_INVALID_ARG
 *   dk    128 only (GDN_ERR_UNSUPPORTED otherwise); dv 64 or 128
 * kda_chunk_fwd_ex takes a caller-owned device workspace of at least
 * kda_chunk_fwd_workspace_size(...) bytes, 256-byte aligned (0 for rejected
 * sizes); kda_chunk_fwd takes one from the stream-ordered pool.
 * kda_recurrent_step: one decode token (g [N, Hv, dk]; dk 64 or 128), as
 * gdn_recurrent_step otherwise.
 */
gdn_status kda_chunk_fwd(const void* q, const void* k, const void* v, const float* g,
                         const float* beta, const float* h0, void* o, float* hT, int B, int T,
                         int Hqk, int Hv, int dk, int dv, int chunk, float scale,
                         const int32_t* cu_seqlens, gdn_stream_t stream);
gdn_status kda_chunk_fwd_ex(const void* q, const void* k, const void* v, const float* g,
                            const float* beta, const float* h0, void* o, float* hT, int B, int T,
                            int Hqk, int Hv, int dk, int dv, int chunk, float scale,
                            const int32_t* cu_seqlens, unsigned flags, void* workspace,
                            size_t workspace_bytes, gdn_stream_t stream);
size_t kda_chunk_fwd_workspace_size(int B, int T, int Hqk, int Hv, int dk, int dv, int chunk,
                                    int has_cu_seqlens);
gdn_status kda_recurrent_step(const void* q, const void* k, const void* v, const float* g,
                              const float* beta, float* h, void* o, int N, int Hqk, int Hv,
                              int dk, int dv, float scale, gdn_stream_t stream);

/*
 * gdn_device_status - waits for `stream`, then reads and clears the device
 * error word.  The kernels record there (the first record stays until read):
 * a bounded device-side wait that gave up (GDN_ERR_TIMEOUT); a KDA log-decay
 * below -10 or not a number, an fp16 operand of the bf16 path out of range, or
 * a violation found by GDN_FLAG_CHECK_INPUTS (GDN_ERR_INVALID_ARG: the result
 * of that call is not exact).  Returns GDN_OK, one of those, or GDN_ERR_CUDA
 * if the stream itself failed.
 */
gdn_status gdn_device_status(gdn_stream_t stream);

/*
 * gdn_selftest_expired_wait - diagnostic for the timeout path: enqueues one
 * warp that waits on a device barrier nothing ever completes, giving up after
 * `limit_cycles` SM clock cycles (0 .. 2^31; the kernels' own waits use
 * 2^31, about a second).  The expired wait records the timeout in the device
 * error word, so the next gdn_device_status returns GDN_ERR_TIMEOUT (and
 * clears it); the kernel returns normally and leaves the context usable.
 * Returns GDN_OK once enqueued.
 */
gdn_status gdn_selftest_expired_wait(long long limit_cycles, gdn_stream_t stream);

/* Static description of a status code. */
const char* gdn_status_string(gdn_status s);

/* Description of the last non-OK status returned to this thread ("" if none). */
const char* gdn_last_error(void);

/* ABI version of this header: 2. */
int gdn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
