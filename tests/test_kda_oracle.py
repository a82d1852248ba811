"""Pins for the Kimi Delta Attention oracle, all on the CPU.

Each pin is fixed by something other than the oracle's own recurrence: the
gated delta rule (every channel of the gate equal, against the pinned GDN
oracle), pure per-channel decay (beta = 0), exact store and retrieval with
orthonormal keys and no decay, keys on one channel (the other rows only decay,
by their own channel's gate), explicit transition-matrix products, the
norm bound of a contraction, and the chunked form.  Planted mistakes in the
recurrence must each trip a pin.
"""
import numpy as np
import pytest

from oracle import (gdn_recurrent, kda_chunked, kda_recurrent, kda_step, kda_transitions)
from oracle.kda_oracle import _over_chains


def unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def rand_inputs(rng, B=1, T=9, Hqk=1, Hv=2, dk=5, dv=3, h0=True, g_scale=1.0):
    q = unit(rng.standard_normal((B, T, Hqk, dk)))
    k = unit(rng.standard_normal((B, T, Hqk, dk)))
    v = rng.standard_normal((B, T, Hv, dv))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, Hv))))
    g = -np.log1p(np.exp(rng.standard_normal((B, T, Hv, dk)))) * g_scale
    hz = rng.standard_normal((B, Hv, dk, dv)) * 0.5 if h0 else None
    return q, k, v, g, beta, hz


def close(a, b, tol=1e-11):
    return np.allclose(a, b, rtol=tol, atol=tol)


def pin_uniform_gate_is_gdn(fwd):
    """Every channel of g_t equal: KDA is the gated delta rule (GQA, two rows, h0)."""
    rng = np.random.default_rng(61)
    q, k, v, g, beta, h0 = rand_inputs(rng, B=2, T=12, Hqk=1, Hv=2, dk=6, dv=4)
    g[:] = g[..., :1]
    o, hT = fwd(q, k, v, g, beta, 0.7, h0, None)
    o2, hT2 = gdn_recurrent(q, k, v, g[..., 0], beta, 0.7, h0)
    return close(o, o2) and close(hT, hT2)


def pin_pure_channel_decay(fwd):
    """beta = 0: nothing is written; h_t = diag(exp G_t) h0, o_t = h_t^T (scale q_t)."""
    rng = np.random.default_rng(62)
    q, k, v, g, beta, h0 = rand_inputs(rng, T=7, Hqk=1, Hv=1, dk=5, dv=3)
    beta[:] = 0.0
    o, hT = fwd(q, k, v, g, beta, 0.8, h0, None)
    G = np.cumsum(g[0, :, 0], axis=0)                    # [T, dk]
    ok = all(close(o[0, t, 0], (np.exp(G[t])[:, None] * h0[0, 0]).T @ (0.8 * q[0, t, 0]))
             for t in range(7))
    return ok and close(hT[0, 0], np.exp(G[-1])[:, None] * h0[0, 0])


def pin_orthonormal_store_retrieve(fwd):
    """g = 0, beta = 1, keys distinct basis vectors: token t overwrites row pi(t) of h
    with v_t exactly, and a query on basis vector pi(s), s <= t, reads scale * v_s."""
    rng = np.random.default_rng(63)
    dk, dv, T = 6, 4, 5
    perm = rng.permutation(dk)[:T]
    q, k, v, g, beta, h0 = rand_inputs(rng, T=T, Hqk=1, Hv=1, dk=dk, dv=dv)
    k[0, :, 0] = np.eye(dk)[perm]
    qsel = rng.integers(0, np.arange(T) + 1)             # a token s <= t for every t
    q[0, :, 0] = np.eye(dk)[perm[qsel]]
    g[:] = 0.0
    beta[:] = 1.0
    o, hT = fwd(q, k, v, g, beta, 0.5, h0, None)
    want_h = h0[0, 0].copy()
    want_h[perm] = v[0, :, 0]
    ok = all(close(o[0, t, 0], 0.5 * v[0, qsel[t], 0]) for t in range(T))
    return ok and close(hT[0, 0], want_h)


def pin_one_channel_keys(fwd):
    """Every key is +-e_c: rows r != c only decay by their own channel's gate; row c
    follows the scalar delta rule x <- (1 - beta) exp(g_c) x + beta (+-v)."""
    rng = np.random.default_rng(64)
    dk, dv, T, c = 5, 3, 8, 2
    q, k, v, g, beta, h0 = rand_inputs(rng, T=T, Hqk=1, Hv=1, dk=dk, dv=dv)
    sign = rng.choice([-1.0, 1.0], size=T)
    k[0, :, 0] = 0.0
    k[0, :, 0, c] = sign
    _, hT = fwd(q, k, v, g, beta, 1.0, h0, None)
    G = np.cumsum(g[0, :, 0], axis=0)
    want = np.exp(G[-1])[:, None] * h0[0, 0]
    x = h0[0, 0, c].copy()
    for t in range(T):
        b = beta[0, t, 0]
        x = (1.0 - b) * np.exp(g[0, t, 0, c]) * x + b * sign[t] * v[0, t, 0]
    want[c] = x
    return close(hT[0, 0], want)


def pin_transition_products(fwd):
    """The state equals (M_T...M_1) h0 + sum_s (M_T...M_{s+1}) beta_s k_s v_s^T with the
    full matrices M_t = (I - beta_t k_t k_t^T) diag(exp g_t), T <= 4."""
    rng = np.random.default_rng(65)
    q, k, v, g, beta, h0 = rand_inputs(rng, B=1, T=4, Hqk=1, Hv=2, dk=4, dv=3)
    o, hT = fwd(q, k, v, g, beta, 0.9, h0, None)
    o2, hT2 = kda_transitions(q, k, v, g, beta, 0.9, h0)
    return close(o, o2) and close(hT, hT2)


def pin_contraction_bound(fwd):
    """||k|| = 1, beta in (0, 1], g <= 0: each M_t has spectral norm <= 1, so
    ||h_t||_2 <= ||h_{t-1}||_2 + beta_t ||v_t|| (checked along the sequence)."""
    rng = np.random.default_rng(66)
    q, k, v, g, beta, h0 = rand_inputs(rng, T=10, Hqk=1, Hv=1, dk=6, dv=4)
    prev = np.linalg.norm(h0[0, 0], 2)
    for t in range(10):
        _, ht = fwd(q[:, :t + 1], k[:, :t + 1], v[:, :t + 1], g[:, :t + 1], beta[:, :t + 1], 1.0,
                    h0, None)
        now = np.linalg.norm(ht[0, 0], 2)
        if now > prev + beta[0, t, 0] * np.linalg.norm(v[0, t, 0]) + 1e-12:
            return False
        prev = now
    return True


PINS = [pin_uniform_gate_is_gdn, pin_pure_channel_decay, pin_orthonormal_store_retrieve,
        pin_one_channel_keys, pin_transition_products, pin_contraction_bound]


def _recurrent(q, k, v, g, beta, scale, h0, cu):
    return kda_recurrent(q, k, v, g, beta, scale, h0, cu)


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_recurrent_oracle_meets_pin(pin):
    assert pin(_recurrent)


@pytest.mark.parametrize("chunk", [16, 64])
def test_chunked_matches_sequential_d128(chunk):
    rng = np.random.default_rng(67)
    q, k, v, g, beta, h0 = rand_inputs(rng, B=1, T=150, Hqk=1, Hv=2, dk=128, dv=32)
    o1, t1 = kda_recurrent(q, k, v, g, beta, 128 ** -0.5, h0)
    o2, t2 = kda_chunked(q, k, v, g, beta, 128 ** -0.5, h0, chunk=chunk)
    assert np.abs(o1 - o2).max() / np.sqrt(np.mean(o1 ** 2)) < 1e-10
    assert np.abs(t1 - t2).max() / np.sqrt(np.mean(t1 ** 2)) < 1e-10


def test_chunked_weak_decay_and_varlen_match_sequential():
    rng = np.random.default_rng(68)
    lens = [70, 0, 5, 129]
    q, k, v, g, beta, _ = rand_inputs(rng, B=1, T=sum(lens), Hqk=2, Hv=4, dk=16, dv=8,
                                      h0=False, g_scale=0.02)
    h0 = rng.standard_normal((len(lens), 4, 16, 8)) * 0.3
    cu = np.concatenate([[0], np.cumsum(lens)])
    o1, t1 = kda_recurrent(q, k, v, g, beta, 0.5, h0, cu)
    o2, t2 = kda_chunked(q, k, v, g, beta, 0.5, h0, cu, chunk=64)
    assert close(o1, o2, 1e-10) and close(t1, t2, 1e-10)


def test_split_sequence_with_carried_state_equals_one_call():
    rng = np.random.default_rng(69)
    q, k, v, g, beta, h0 = rand_inputs(rng, T=40, Hqk=1, Hv=2, dk=8, dv=4)
    o, hT = kda_recurrent(q, k, v, g, beta, 0.6, h0)
    oa, ha = kda_recurrent(q[:, :17], k[:, :17], v[:, :17], g[:, :17], beta[:, :17], 0.6, h0)
    ob, hb = kda_recurrent(q[:, 17:], k[:, 17:], v[:, 17:], g[:, 17:], beta[:, 17:], 0.6, ha)
    assert close(np.concatenate([oa, ob], axis=1), o, 1e-12) and close(hb, hT, 1e-12)


def test_prefill_then_step_equals_one_pass():
    rng = np.random.default_rng(70)
    q, k, v, g, beta, h0 = rand_inputs(rng, T=10, Hqk=1, Hv=2, dk=6, dv=4)
    o, hT = kda_recurrent(q, k, v, g, beta, 0.7, h0)
    _, h9 = kda_recurrent(q[:, :9], k[:, :9], v[:, :9], g[:, :9], beta[:, :9], 0.7, h0)
    o_last, h_new = kda_step(q[:, 9], k[:, 9], v[:, 9], g[:, 9], beta[:, 9], h9, 0.7)
    assert close(o_last, o[:, 9], 1e-12) and close(h_new, hT, 1e-12)


# ---------------------------------------------------------------------------
# Planted mistakes: each must fail at least one pin
# ---------------------------------------------------------------------------
def _mutant(kind):
    def chain(qs, ks, vs, gs, betas, h, scale):
        L = qs.shape[0]
        o = np.zeros((L, h.shape[1]))
        for t in range(L):
            dec = np.exp(gs[t])
            if kind == "decay_on_dv":            # gate applied to the value columns
                h *= dec[: h.shape[1]][None, :] if h.shape[1] <= h.shape[0] else 1.0
            elif kind == "decay_after_update":
                pass
            elif kind == "scalar_mean_gate":
                h *= np.exp(gs[t].mean())
            else:
                h *= dec[:, None]
            if kind == "read_before_decay":      # delta rule reads the undecayed state
                u = betas[t] * (vs[t] - (h / dec[:, None]).T @ ks[t])
            else:
                u = betas[t] * (vs[t] - h.T @ ks[t])
            h += np.outer(ks[t], u)
            if kind == "decay_after_update":
                h *= dec[:, None]
            o[t] = h.T @ (scale * qs[t])
        return o

    def fwd(q, k, v, g, beta, scale, h0, cu):
        return _over_chains(chain, q, k, v, g, beta, scale, h0, cu, "grouped", None)
    return fwd


@pytest.mark.parametrize("kind", ["decay_on_dv", "decay_after_update", "scalar_mean_gate",
                                  "read_before_decay"])
def test_planted_mistake_is_caught(kind):
    fwd = _mutant(kind)
    assert not all(pin(fwd) for pin in PINS), kind
