"""fp64 CPU oracle for Kimi Delta Attention (KDA): the delta rule with a per-channel gate.

TEST INFRASTRUCTURE ONLY, like ``gdn_oracle``: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU legs of ``bench.py`` may use it, and it
shares no code with the CUDA path.

What it computes
----------------
"Empowering Hybrid Attention Models on NPUs" treats GDN and KDA as the two
delta-rule mechanisms of its Map-Reduce-Map paradigm (§2.1, Figure 1): KDA keeps
the delta rule's error-correcting update and gates it finely (§8 Related Work),
its gate is per key channel - the cumulative-gate tensor is 128x larger than
GDN's (§7.5, Figure 16, d = 128) - and Figure 4(a) prices that gate as one fp32
value per (token, head, channel): 31.33 MiB against GDN's 21.41 MiB at T = 2048,
H = 10.  The pages print no KDA formula.  The plainest reading that these facts
support, used here: GDN's scalar decay exp(g_t) becomes the diagonal matrix
diag(exp(g_t)) over the key channels, applied to the state before the delta
rule reads it.  With the state stored as h = S^T, [dk][dv], per (sequence, v
head) and tokens in order,

    h_t = (I - beta_t k_t k_t^T) diag(exp(g_t)) h_{t-1} + beta_t k_t v_t^T,
    o_t = h_t^T (scale q_t),                  g_t in R^dk, g_t <= 0.

With every g_t[c] equal this is the gated delta rule of ``gdn_oracle``.
Conventions (shapes, GQA "grouped" head map, cu_seqlens, h0 = None for zeros,
fp64 upcast) are those of ``gdn_oracle``; g is [B, T, Hv, dk] fp32.

Functions
---------
* ``kda_recurrent``  - the recurrence token by token (the definition).
* ``kda_transitions``- the same state written as products of the explicit
                       dk x dk transition matrices (tiny inputs; a pin).
* ``kda_chunked``    - the chunkwise Map-Reduce-Map form the kernels follow:
                       per chunk the per-channel cumulative gate, the KK^T and
                       QK^T grams with the decay exp(G_i - G_j) inside the
                       channel sum, the UT transform (I + A)^-1, W and U, then
                       V_new = U - W h, O = Q~ h + P V_new and the state carry.
* ``kda_step``       - one decode token.
"""
from __future__ import annotations

import numpy as np

from .gdn_oracle import _f64, chains, forward_substitution_inverse, qk_head

__all__ = ["kda_recurrent", "kda_transitions", "kda_chunked", "kda_step",
           "kda_recurrent_chain", "kda_chunked_chain"]


def _prepare(q, k, v, g, beta, h0, cu_seqlens):
    q, k, v, g, beta, h0 = map(_f64, (q, k, v, g, beta, h0))
    B, T, Hqk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    assert k.shape == q.shape and v.shape[:2] == (B, T)
    assert g.shape == (B, T, Hv, dk), "KDA takes one log-decay per key channel"
    assert beta.shape == (B, T, Hv)
    ch = chains(B, T, cu_seqlens)
    if h0 is None:
        h0 = np.zeros((len(ch), Hv, dk, dv))
    assert h0.shape == (len(ch), Hv, dk, dv)
    return q, k, v, g, beta, h0, ch


def _over_chains(fn, q, k, v, g, beta, scale, h0, cu_seqlens, head_map, heads, *extra):
    q, k, v, g, beta, h0, ch = _prepare(q, k, v, g, beta, h0, cu_seqlens)
    B, T, Hqk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    o = np.zeros((B, T, Hv, dv))
    hT = np.zeros_like(h0)
    for n, b, t0, t1 in ch:
        for hv in (range(Hv) if heads is None else heads):
            hq = qk_head(hv, Hqk, Hv, head_map)
            h = h0[n, hv].copy()
            o[b, t0:t1, hv] = fn(q[b, t0:t1, hq], k[b, t0:t1, hq], v[b, t0:t1, hv],
                                 g[b, t0:t1, hv], beta[b, t0:t1, hv], h, scale, *extra)
            hT[n, hv] = h
    return o, hT


# --------------------------------------------------------------------------
# Definition: the recurrence, token by token
# --------------------------------------------------------------------------
def kda_recurrent_chain(qs, ks, vs, gs, betas, h, scale):
    """One chain in place on h [dk, dv]; gs is [L, dk].

    Per token: the gate scales row c of h (key channel c) by exp(g_t[c]); the
    delta rule then reads the decayed state along k_t and writes the correction
    beta_t (v_t - h^T k_t) along k_t.
    """
    L = qs.shape[0]
    o = np.zeros((L, h.shape[1]))
    for t in range(L):
        h *= np.exp(gs[t])[:, None]
        u = betas[t] * (vs[t] - h.T @ ks[t])
        h += np.outer(ks[t], u)
        o[t] = h.T @ (scale * qs[t])
    return o


def kda_recurrent(q, k, v, g, beta, scale, h0=None, cu_seqlens=None, head_map="grouped",
                  heads=None):
    """Token-by-token KDA recurrence over every (sequence, v head) chain -> (o, hT)."""
    return _over_chains(kda_recurrent_chain, q, k, v, g, beta, scale, h0, cu_seqlens, head_map,
                        heads)


# --------------------------------------------------------------------------
# Explicit transition matrices (tiny inputs only)
# --------------------------------------------------------------------------
def _transitions_chain(qs, ks, vs, gs, betas, h, scale):
    """h_t = M_t h_{t-1} + beta_t k_t v_t^T with M_t = (I - beta_t k_t k_t^T) diag(exp g_t)
    formed as a full dk x dk matrix; o_t from the state so obtained."""
    L, dk = ks.shape
    eye = np.eye(dk)
    o = np.zeros((L, h.shape[1]))
    h0 = h.copy()
    for t in range(L):
        # h_t = (M_t ... M_1) h0 + sum_{s<=t} (M_t ... M_{s+1}) beta_s k_s v_s^T
        prod = eye.copy()
        acc = np.zeros_like(h0)
        for s in range(t, -1, -1):
            acc += prod @ (betas[s] * np.outer(ks[s], vs[s]))
            M = (eye - betas[s] * np.outer(ks[s], ks[s])) @ np.diag(np.exp(gs[s]))
            prod = prod @ M
        ht = prod @ h0 + acc
        o[t] = ht.T @ (scale * qs[t])
        if t == L - 1:
            h[...] = ht
    return o


def kda_transitions(q, k, v, g, beta, scale, h0=None, cu_seqlens=None, head_map="grouped"):
    """The recurrence as products of explicit transition matrices (O(T^2 dk^3): tiny only)."""
    return _over_chains(_transitions_chain, q, k, v, g, beta, scale, h0, cu_seqlens, head_map,
                        None)


# --------------------------------------------------------------------------
# Chunkwise form (Map #1-#4, Reduce #5, Map #6 of Figure 1(b), per-channel gate)
# --------------------------------------------------------------------------
def kda_chunked_chain(qs, ks, vs, gs, betas, h, scale, chunk):
    """One chain, chunk by chunk, in place on h.  Within a chunk (local i, j < L):

    #1 Gate   G_i = sum_{s<=i} g_s            (per channel, [L, dk])
    #2 KKT    A_ij = beta_i sum_c k_ic k_jc exp(G_ic - G_jc),  j < i  (else 0)
       QK^T   P_ij = scale sum_c q_ic k_jc exp(G_ic - G_jc),   j <= i (else 0)
    #3 Solve  Tm = (I + A)^-1
    #4 W/U    W = Tm diag(beta) (K * exp(G)),  U = Tm diag(beta) V
    #5 Reduce V_new = U - W h;  h <- diag(exp(G_L-1)) h + (K * exp(G_L-1 - G))^T V_new
    #6 Map    O = (scale Q * exp(G)) h + P V_new          (h: the state entering the chunk)

    Derivation: with u_j the correction written at token j, h_i = diag(exp G_i) h
    + sum_{j<=i} diag(exp(G_i - G_j)) k_j u_j^T, and u_j = beta_j (v_j - h_{j-1}^T
    diag(exp g_j) k_j) gives (I + A) u = diag(beta)(V - (K * exp G) h).
    """
    T = qs.shape[0]
    o = np.zeros((T, h.shape[1]))
    for c0 in range(0, T, chunk):
        c1 = min(T, c0 + chunk)
        Q, K, V = qs[c0:c1], ks[c0:c1], vs[c0:c1]
        G = np.cumsum(gs[c0:c1], axis=0)
        b = betas[c0:c1]
        L = c1 - c0
        decay = np.exp(G[:, None, :] - G[None, :, :])          # [i, j, c]
        KK = np.einsum("ic,jc,ijc->ij", K, K, decay)
        QK = np.einsum("ic,jc,ijc->ij", Q, K, decay)
        A = np.tril(b[:, None] * KK, -1)
        P = scale * np.tril(QK)
        Tm = forward_substitution_inverse(A)
        W = Tm @ (b[:, None] * (K * np.exp(G)))
        U = Tm @ (b[:, None] * V)
        Vn = U - W @ h
        O = (scale * Q * np.exp(G)) @ h + P @ Vn
        GL = G[L - 1]
        h[...] = np.exp(GL)[:, None] * h + (K * np.exp(GL[None, :] - G)).T @ Vn
        o[c0:c1] = O
    return o


def kda_chunked(q, k, v, g, beta, scale, h0=None, cu_seqlens=None, chunk=64, head_map="grouped",
                heads=None):
    """The chunkwise KDA forward over every chain; chunks restart at every sequence start."""
    return _over_chains(kda_chunked_chain, q, k, v, g, beta, scale, h0, cu_seqlens, head_map, heads,
                        chunk)


# --------------------------------------------------------------------------
# Decode
# --------------------------------------------------------------------------
def kda_step(q, k, v, g, beta, h, scale, head_map="grouped"):
    """One decode token for N sequences (q, k [N, Hqk, dk]; v [N, Hv, dv]; g [N, Hv, dk];
    beta [N, Hv]; h [N, Hv, dk, dv]) -> (o [N, Hv, dv], h_new); inputs unchanged."""
    q, k, v, g, beta, h = map(_f64, (q, k, v, g, beta, h))
    N, Hqk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    assert g.shape == (N, Hv, dk)
    o = np.zeros((N, Hv, dv))
    hn = h.copy()
    for n in range(N):
        for hv in range(Hv):
            hq = qk_head(hv, Hqk, Hv, head_map)
            s = hn[n, hv]
            o[n, hv] = kda_recurrent_chain(q[n, hq][None], k[n, hq][None], v[n, hv][None],
                                           g[n, hv][None], beta[n, hv][None], s, scale)[0]
    return o, hn
