"""fp64 CPU oracle for the Gated DeltaNet chunked-prefill forward and decode step.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code, table or helper with the CUDA path.

What it computes
----------------
Gated DeltaNet keeps one state matrix per (sequence, value head).  The pages
describe the step in words ("Empowering Hybrid Attention Models on NPUs", §2.1
"Architecture of Linear-Attention Hybrids": at step t the previous state
S_{t-1} is updated with K_t and V_t, then the output is formed from Q_t and the
*updated* state S_t) and name Gated DeltaNet as the linear attention of the
Qwen3.5 family; they never print the update formula.  The oracle takes the
gated delta rule that defines GDN:

    S_t = exp(g_t) * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
    o_t = S_t (scale * q_t)

with S_t of shape [dv, dk].  It is stored transposed, h = S^T of shape
[dk, dv] (the "[dk x dv]" per-head state of the workloads; "Exp 2026-07-13 —
Linear-Attention Scans on the NPU", §4 notes that systems differ in the state's
key/value orientation).

Functions
---------
* ``gdn_dense``      - the rule above with explicit dk x dk matrices
                       (I - beta k k^T); tiny cases only.  Parity unpinned by
                       itself: it is the definition typed out, pinned by the
                       invariant tests.
* ``gdn_recurrent``  - the same rule as rank-1 steps (decay, erase-and-write
                       vector u, rank-1 add, read-out); the primary oracle.
* ``gdn_chunked``    - the chunkwise Map-Reduce-Map form: #1 Gate, #2 KKT,
                       #3 Solve, #4 W/U, #5 H-read, #6 O, #5 H-update
                       ("Empowering Hybrid Attention Models on NPUs", §2.1,
                       Figure 1(b); chunk-first order of §5, Figure 10(b)),
                       with a naive forward-substitution solve ("Exp
                       2026-07-13 — Linear-Attention Scans on the NPU", §1).
* ``gdn_step``       - one decode token, the rule above applied once.

Conventions (readings of the pages, listed with reasons in the design notes)
* q, k: [B, T, Hqk, dk]; v: [B, T, Hv, dv]; g, beta: [B, T, Hv];
  h0 / hT: [N, Hv, dk, dv].
* q and k arrive L2-normalised; beta arrives squashed; g arrives as log-decay.
* GQA: v head hv reads qk head hv // (Hv // Hqk) ("grouped"); "modulo"
  (hv % Hqk) is available for comparison.
* cu_seqlens (int [N+1]) packs N sequences into one row: tensors are
  [1, T_total, ...], each sequence starts from its own h0 and gets its own hT.
* h0 = None means zeros.
* Every input is upcast to float64 before any arithmetic.
"""
from __future__ import annotations

import numpy as np

__all__ = ["gdn_dense", "gdn_recurrent", "gdn_chunked", "gdn_step", "chains",
           "qk_head", "forward_substitution_inverse", "prologue"]


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):            # a torch tensor: take its exact values
        x = x.detach().to("cpu")
        if str(x.dtype) == "torch.bfloat16":
            x = x.float()
        x = x.numpy()
    return np.asarray(x, dtype=np.float64)


def qk_head(hv: int, Hqk: int, Hv: int, head_map: str = "grouped") -> int:
    """The qk head that v head ``hv`` reads (GQA).

    "grouped": consecutive v heads share a qk head.  "modulo": the
    ``hv % Hk`` replication of the GQA marshaller in "Exp 2026-07-13 —
    Linear-Attention Scans on the NPU", §4.
    """
    if Hv % Hqk:
        raise ValueError("Hv must be a multiple of Hqk")
    if head_map == "grouped":
        return hv // (Hv // Hqk)
    if head_map == "modulo":
        return hv % Hqk
    raise ValueError(head_map)


def chains(B: int, T: int, cu_seqlens=None):
    """(sequence index, row b, first token, end token) for every sequence."""
    if cu_seqlens is None:
        return [(b, b, 0, T) for b in range(B)]
    cu = [int(x) for x in np.asarray(_f64(cu_seqlens))]
    return [(n, 0, cu[n], cu[n + 1]) for n in range(len(cu) - 1)]


def _prepare(q, k, v, g, beta, h0, cu_seqlens):
    q, k, v, g, beta, h0 = map(_f64, (q, k, v, g, beta, h0))
    B, T, Hqk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    assert k.shape == q.shape and v.shape[:2] == (B, T) and g.shape == (B, T, Hv)
    assert beta.shape == g.shape
    ch = chains(B, T, cu_seqlens)
    N = len(ch)
    if h0 is None:
        h0 = np.zeros((N, Hv, dk, dv))
    assert h0.shape == (N, Hv, dk, dv)
    return q, k, v, g, beta, h0, ch


# --------------------------------------------------------------------------
# Definition, dense form (tiny inputs only)
# --------------------------------------------------------------------------
def gdn_dense(q, k, v, g, beta, scale, h0=None, cu_seqlens=None, head_map="grouped"):
    """S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T, o_t = S_t (scale q_t).

    Every product is a full matrix product; S is [dv, dk].  Returns (o, hT)
    with hT[n, hv] = S_T^T.
    """
    q, k, v, g, beta, h0, ch = _prepare(q, k, v, g, beta, h0, cu_seqlens)
    B, T, Hqk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    o = np.zeros((B, T, Hv, dv))
    hT = np.zeros_like(h0)
    eye = np.eye(dk)
    for n, b, t0, t1 in ch:
        for hv in range(Hv):
            hq = qk_head(hv, Hqk, Hv, head_map)
            S = h0[n, hv].T.copy()
            for t in range(t0, t1):
                kt = k[b, t, hq][:, None]            # [dk, 1]
                vt = v[b, t, hv][:, None]            # [dv, 1]
                erase = eye - beta[b, t, hv] * (kt @ kt.T)
                S = np.exp(g[b, t, hv]) * (S @ erase) + beta[b, t, hv] * (vt @ kt.T)
                o[b, t, hv] = S @ (scale * q[b, t, hq])
            hT[n, hv] = S.T
    return o, hT


# --------------------------------------------------------------------------
# Definition, rank-1 sequential form (the primary oracle)
# --------------------------------------------------------------------------
def recurrent_chain(qs, ks, vs, gs, betas, h, scale):
    """Run the rule over one chain (one sequence, one v head), in place on h.

    qs, ks: [L, dk]; vs: [L, dv]; gs, betas: [L]; h: [dk, dv] (= S^T).
    Per token: h <- exp(g) h; u = beta (v - h^T k); h <- h + k u^T;
    o = h^T (scale q).  Expanding S_t = exp(g) S (I - beta k k^T) + beta v k^T
    with S = h^T gives exactly these four lines.
    Returns o [L, dv].
    """
    L = qs.shape[0]
    o = np.zeros((L, h.shape[1]))
    for t in range(L):
        h *= np.exp(gs[t])
        u = betas[t] * (vs[t] - h.T @ ks[t])
        h += np.outer(ks[t], u)
        o[t] = h.T @ (scale * qs[t])
    return o


def gdn_recurrent(q, k, v, g, beta, scale, h0=None, cu_seqlens=None, head_map="grouped",
                  heads=None):
    """Token-by-token gated delta rule over every (sequence, v head) chain.

    ``heads`` (optional list of v heads) restricts the work to those heads;
    the other outputs stay zero.  Returns (o [B,T,Hv,dv], hT [N,Hv,dk,dv]).
    """
    q, k, v, g, beta, h0, ch = _prepare(q, k, v, g, beta, h0, cu_seqlens)
    B, T, Hqk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    o = np.zeros((B, T, Hv, dv))
    hT = np.zeros_like(h0)
    for n, b, t0, t1 in ch:
        for hv in (range(Hv) if heads is None else heads):
            hq = qk_head(hv, Hqk, Hv, head_map)
            h = h0[n, hv].copy()
            o[b, t0:t1, hv] = recurrent_chain(q[b, t0:t1, hq], k[b, t0:t1, hq],
                                              v[b, t0:t1, hv], g[b, t0:t1, hv],
                                              beta[b, t0:t1, hv], h, scale)
            hT[n, hv] = h
    return o, hT


def gdn_step(q, k, v, g, beta, h, scale, head_map="grouped"):
    """One decode token for N sequences: the rule applied once.

    q, k: [N, Hqk, dk]; v: [N, Hv, dv]; g, beta: [N, Hv]; h: [N, Hv, dk, dv].
    Returns (o [N, Hv, dv], h_new [N, Hv, dk, dv]); the inputs are not modified.
    """
    q, k, v, g, beta, h = map(_f64, (q, k, v, g, beta, h))
    N, Hqk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    o = np.zeros((N, Hv, dv))
    hn = h.copy()
    for n in range(N):
        for hv in range(Hv):
            hq = qk_head(hv, Hqk, Hv, head_map)
            o[n, hv] = recurrent_chain(q[n, hq][None], k[n, hq][None], v[n, hv][None],
                                       g[n, hv][None], beta[n, hv][None], hn[n, hv], scale)[0]
    return o, hn


# --------------------------------------------------------------------------
# Chunkwise Map-Reduce-Map form
# --------------------------------------------------------------------------
def forward_substitution_inverse(A):
    """(I + A)^-1 for strictly lower-triangular A, one row at a time.

    Row i of X = (I + A)^-1 satisfies X_i = e_i - sum_{j<i} A_ij X_j, which
    is forward substitution on the unit lower-triangular system (I + A) X = I
    (the UT transform's solve, "Exp 2026-07-13 — Linear-Attention Scans on
    the NPU", §1 and §4).
    """
    L = A.shape[0]
    X = np.zeros((L, L))
    for i in range(L):
        X[i, i] = 1.0
        for j in range(i):
            X[i] -= A[i, j] * X[j]
    return X


def chunked_chain(qs, ks, vs, gs, betas, h, scale, chunk):
    """Chunkwise form over one chain, in place on h ([dk, dv]); returns o [L, dv].

    For each chunk of L <= chunk tokens (local indices i, j), with
    q^ = scale q:
      #1 Gate:   G_i = sum_{s<=i} g_s,  gamma_i = exp(G_i),
                 M_ij = exp(G_i - G_j) for i >= j, else 0
      #2 KKT:    A_ij = beta_i M_ij (k_i . k_j) for i > j, else 0
      (QK^T)     P_ij = M_ij (q^_i . k_j) for i >= j, else 0
      #3 Solve:  Tm = (I + A)^-1
      #4 W/U:    W = Tm diag(beta*gamma) K,  U = Tm diag(beta) V
      #5 read:   V_new = U - W h
      #6 O:      O = diag(gamma) Q^ h + P V_new
      #5 update: h <- gamma_{L-1} h + K^T diag(e) V_new,  e_j = exp(G_{L-1} - G_j)
    ("Empowering Hybrid Attention Models on NPUs", §2.1 and Figure 1(b) for
    the operator list; §5 Figure 10(b) for reading the state before the
    in-place update.)  Derivation: unrolling the rule inside a chunk gives
    S_i = gamma_i S_0 + sum_{j<=i} M_ij u_j k_j^T with
    u_i = beta_i (v_i - exp(g_i) S_{i-1} k_i); substituting S_{i-1} turns the
    u's into the unit lower-triangular system (I + A) U_rows = diag(beta) V -
    diag(beta*gamma) K h, solved by Tm.
    """
    T_len = qs.shape[0]
    o = np.zeros((T_len, h.shape[1]))
    for c0 in range(0, T_len, chunk):
        c1 = min(c0 + chunk, T_len)
        Q = scale * qs[c0:c1]
        K = ks[c0:c1]
        V = vs[c0:c1]
        b = betas[c0:c1]
        L = c1 - c0
        # #1 Gate
        G = np.cumsum(gs[c0:c1])
        gamma = np.exp(G)
        M = np.zeros((L, L))
        for i in range(L):
            for j in range(i + 1):
                M[i, j] = np.exp(G[i] - G[j])
        # #2 KKT and the QK^T gram
        A = np.tril(b[:, None] * M * (K @ K.T), k=-1)
        P = np.tril(M * (Q @ K.T), k=0)
        # #3 Solve
        Tm = forward_substitution_inverse(A)
        # #4 W/U
        W = Tm @ ((b * gamma)[:, None] * K)
        U = Tm @ (b[:, None] * V)
        # #5 read, #6 O, #5 update
        V_new = U - W @ h
        o[c0:c1] = gamma[:, None] * (Q @ h) + P @ V_new
        e = np.exp(G[-1] - G)
        h *= gamma[-1]
        h += K.T @ (e[:, None] * V_new)
    return o


def gdn_chunked(q, k, v, g, beta, scale, h0=None, cu_seqlens=None, chunk=64,
                head_map="grouped", heads=None):
    """Chunkwise form over every chain; chunks restart at every sequence start."""
    q, k, v, g, beta, h0, ch = _prepare(q, k, v, g, beta, h0, cu_seqlens)
    B, T, Hqk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    o = np.zeros((B, T, Hv, dv))
    hT = np.zeros_like(h0)
    for n, b, t0, t1 in ch:
        for hv in (range(Hv) if heads is None else heads):
            hq = qk_head(hv, Hqk, Hv, head_map)
            h = h0[n, hv].copy()
            o[b, t0:t1, hv] = chunked_chain(q[b, t0:t1, hq], k[b, t0:t1, hq], v[b, t0:t1, hv],
                                            g[b, t0:t1, hv], beta[b, t0:t1, hv], h, scale, chunk)
            hT[n, hv] = h
    return o, hT


# --------------------------------------------------------------------------
# The fused prologue's elementwise steps, written out on their own
# --------------------------------------------------------------------------
def prologue(q, k, a, b, A_log=None, dt_bias=None, eps=1e-6):
    """Unnormalised q, k and raw gates -> the inputs the rule takes.

    q_hat = q / sqrt(sum q^2 + eps) per head vector (likewise k);
    g = -exp(A_log[h]) * softplus(a + dt_bias[h]); beta = 1 / (1 + exp(-b)).
    A_log, dt_bias: [Hv] or None (zeros).  Returns (q_hat, k_hat, g, beta) in fp64.
    """
    q, k, a, b = map(_f64, (q, k, a, b))
    Hv = a.shape[-1]
    A_log = np.zeros(Hv) if A_log is None else _f64(A_log)
    dt_bias = np.zeros(Hv) if dt_bias is None else _f64(dt_bias)
    qh = q / np.sqrt(np.sum(q * q, axis=-1, keepdims=True) + eps)
    kh = k / np.sqrt(np.sum(k * k, axis=-1, keepdims=True) + eps)
    x = a + dt_bias
    softplus = np.where(x > 30.0, x, np.log1p(np.exp(np.minimum(x, 30.0))))
    g = -np.exp(A_log) * softplus
    beta = 1.0 / (1.0 + np.exp(-b))
    return qh, kh, g, beta
