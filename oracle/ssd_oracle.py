"""fp64 CPU oracle for the Mamba-2 SSD scan (the chunked scan without the erase).

TEST INFRASTRUCTURE ONLY, like ``gdn_oracle``: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU legs of ``bench.py`` may use it, and it
shares no code with the CUDA path.

What it computes
----------------
"Exp 2026-07-13 — Linear-Attention Scans on the NPU" (§1 Design, §3 Mamba-2 /
SSD) runs the Mamba-2 selective state-space scan with the same chunked
reformulation as the GDN scan: four matrix stages per chunk (the C B^T gram,
the intra-chunk output, the chunk state, the inter-chunk output) around a
per-chunk cumulative decay (softplus / cumsum / decay on the host).  Per
(sequence, head), with C -> q, B -> k, x -> v, the per-token log-decay dt*A ->
g and the input step dt -> beta, the recurrence is

    S_t = exp(g_t) S_{t-1} + beta_t v_t k_t^T,      o_t = S_t (scale * q_t)

i.e. the gated delta rule of ``gdn_oracle`` with the erase factor
(I - beta_t k_t k_t^T) replaced by the identity.  The state is stored as
h = S^T, [dk = d_state, dv = head_dim].  Conventions (shapes, GQA "grouped"
map of B/C groups to heads, cu_seqlens, h0 = None for zeros, fp64 upcast) are
those of ``gdn_oracle``.

Functions
---------
* ``ssd_recurrent`` - the recurrence token by token (primary oracle).
* ``ssd_unrolled``  - the recurrence unrolled into its closed form,
                      o_t = scale [exp(G_t) h0^T q_t + sum_{s<=t}
                      exp(G_t - G_s) beta_s (q_t . k_s) v_s], G the running
                      sum of g within the sequence; an independent pin.
* ``ssd_chunked``   - the four chunk stages in the page's order.
* ``ssd_step``      - one decode token.
"""
from __future__ import annotations

import numpy as np

from .gdn_oracle import _f64, _prepare, qk_head

__all__ = ["ssd_recurrent", "ssd_unrolled", "ssd_chunked", "ssd_step", "ssd_recurrent_chain"]


def ssd_recurrent_chain(qs, ks, vs, gs, betas, h, scale):
    """One chain in place on h [dk, dv]: h <- exp(g) h + beta k v^T; o = h^T (scale q)."""
    L = qs.shape[0]
    o = np.zeros((L, h.shape[1]))
    for t in range(L):
        h *= np.exp(gs[t])
        h += betas[t] * np.outer(ks[t], vs[t])
        o[t] = h.T @ (scale * qs[t])
    return o


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


def ssd_recurrent(q, k, v, g, beta, scale, h0=None, cu_seqlens=None, head_map="grouped",
                  heads=None):
    """Token-by-token SSD recurrence over every (sequence, head) chain."""
    return _over_chains(ssd_recurrent_chain, q, k, v, g, beta, scale, h0, cu_seqlens, head_map,
                        heads)


def _unrolled_chain(qs, ks, vs, gs, betas, h, scale):
    """Closed form of the unrolled recurrence over one chain (h: h0 in, hT out)."""
    L = qs.shape[0]
    G = np.cumsum(gs)
    o = np.zeros((L, h.shape[1]))
    for t in range(L):
        acc = np.exp(G[t]) * (h.T @ qs[t])
        for s in range(t + 1):
            acc = acc + np.exp(G[t] - G[s]) * betas[s] * (qs[t] @ ks[s]) * vs[s]
        o[t] = scale * acc
    hT = np.exp(G[-1]) * h if L else h.copy()
    for s in range(L):
        hT = hT + np.exp(G[-1] - G[s]) * betas[s] * np.outer(ks[s], vs[s])
    h[...] = hT
    return o


def ssd_unrolled(q, k, v, g, beta, scale, h0=None, cu_seqlens=None, head_map="grouped"):
    """The SSD recurrence in closed form (small inputs only)."""
    return _over_chains(_unrolled_chain, q, k, v, g, beta, scale, h0, cu_seqlens, head_map, None)


def _chunked_chain(qs, ks, vs, gs, betas, h, scale, chunk):
    """The four stages per chunk (local index i, j; L <= chunk tokens):

    cumulative decay  G = cumsum(g), gamma_i = exp(G_i), e_j = exp(G_L-1 - G_j)
    gram              P = tril(exp(G_i - G_j) (scale q_i) . k_j)         (C B^T)
    intra-chunk out   O = P diag(beta) V
    inter-chunk out   O += diag(gamma) (scale Q) h                       (state entering)
    chunk state       h <- gamma_L-1 h + K^T diag(e beta) V
    """
    T = qs.shape[0]
    o = np.zeros((T, h.shape[1]))
    for c0 in range(0, T, chunk):
        c1 = min(T, c0 + chunk)
        Q, K, V = scale * qs[c0:c1], ks[c0:c1], vs[c0:c1]
        G = np.cumsum(gs[c0:c1])
        b = betas[c0:c1]
        L = c1 - c0
        M = np.tril(np.exp(G[:, None] - G[None, :]))
        P = M * (Q @ K.T)
        O = P @ (b[:, None] * V)
        O += np.exp(G)[:, None] * (Q @ h)
        e = np.exp(G[L - 1] - G)
        h[...] = np.exp(G[L - 1]) * h + K.T @ ((e * b)[:, None] * V)
        o[c0:c1] = O
    return o


def ssd_chunked(q, k, v, g, beta, scale, h0=None, cu_seqlens=None, chunk=64, head_map="grouped",
                heads=None):
    """The chunked SSD scan over every chain; chunks restart at every sequence start."""
    return _over_chains(_chunked_chain, q, k, v, g, beta, scale, h0, cu_seqlens, head_map, heads,
                        chunk)


def ssd_step(q, k, v, g, beta, h, scale, head_map="grouped"):
    """One decode token for N sequences; returns (o [N, Hv, dv], h_new); inputs unchanged."""
    q, k, v, g, beta, h = map(_f64, (q, k, v, g, beta, h))
    N, Hqk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    o = np.zeros((N, Hv, dv))
    hn = h.copy()
    for n in range(N):
        for hv in range(Hv):
            hq = qk_head(hv, Hqk, Hv, head_map)
            o[n, hv] = ssd_recurrent_chain(q[n, hq][None], k[n, hq][None], v[n, hv][None],
                                           g[n, hv][None], beta[n, hv][None], hn[n, hv],
                                           scale)[0]
    return o, hn
