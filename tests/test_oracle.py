"""Pins for the fp64 oracle, all on the CPU.

Each pin is fixed by something other than the oracle's own code: a closed form
worked by hand, an invariant of the gated delta rule, a library routine, or the
figures printed in "Empowering Hybrid Attention Models on NPUs" (Figure 4).
The mutant tests plant plausible mistakes in a copy of the recurrence and check
that every one of them trips at least one pin.
"""
import os

import numpy as np
import pytest

from oracle import (gdn_chunked, gdn_dense, gdn_recurrent, gdn_step, forward_substitution_inverse,
                    qk_head)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def rand_inputs(rng, B=1, T=7, Hqk=1, Hv=1, dk=5, dv=3, h0=True, g_mu=0.0):
    q = _unit(rng.standard_normal((B, T, Hqk, dk)))
    k = _unit(rng.standard_normal((B, T, Hqk, dk)))
    v = rng.standard_normal((B, T, Hv, dv))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, Hv))))
    g = -np.log1p(np.exp(rng.standard_normal((B, T, Hv)) + g_mu))
    hz = rng.standard_normal((B, Hv, dk, dv)) * 0.5 if h0 else None
    return q, k, v, g, beta, hz


# ---------------------------------------------------------------------------
# Pins, written against a generic forward fwd(q,k,v,g,beta,scale,h0,cu_seqlens)
# ---------------------------------------------------------------------------
def pin_pure_decay(fwd):
    """beta = 0: nothing is written, the state only decays.

    o_t = exp(G_t) h0^T (scale q_t), hT = exp(G_T) h0, G_t = sum_{s<=t} g_s.
    dk != dv, so a transposed state also fails here.
    """
    rng = np.random.default_rng(11)
    q, k, v, g, beta, h0 = rand_inputs(rng, T=6, dk=5, dv=3)
    beta[:] = 0.0
    scale = 0.7
    o, hT = fwd(q, k, v, g, beta, scale, h0, None)
    G = np.cumsum(g[0, :, 0])
    for t in range(6):
        want = np.exp(G[t]) * (h0[0, 0].T @ (scale * q[0, t, 0]))
        if not np.allclose(o[0, t, 0], want, rtol=1e-12, atol=1e-14):
            return False
    return np.allclose(hT[0, 0], np.exp(G[-1]) * h0[0, 0], rtol=1e-12, atol=1e-14)


def pin_store_retrieve(fwd):
    """g = 0, beta = 1, orthonormal keys, h0 = 0: the state stores v_j under key k_j.

    Then S_t k_j = v_j for every j <= t, so querying with q_t = k_j / scale
    returns v_j exactly, and the final state maps every key to its value.
    """
    rng = np.random.default_rng(12)
    dk, dv, T = 8, 3, 6
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    keys = Qm[:T]                                   # orthonormal rows
    scale = 0.5
    k = keys[None, :, None, :].copy()
    v = rng.standard_normal((1, T, 1, dv))
    which = [0, 0, 2, 1, 4, 3]                      # query token t asks for key which[t] <= t
    q = (keys[which] / scale)[None, :, None, :]
    g = np.zeros((1, T, 1))
    beta = np.ones((1, T, 1))
    o, hT = fwd(q, k, v, g, beta, scale, None, None)
    for t in range(T):
        if not np.allclose(o[0, t, 0], v[0, which[t], 0], atol=1e-12):
            return False
    for j in range(T):
        if not np.allclose(hT[0, 0].T @ keys[j], v[0, j, 0], atol=1e-12):
            return False
    return True


def pin_reset(fwd):
    """exp(g) = 0 (g very negative): the old state is wiped every step.

    S_t = beta_t v_t k_t^T, so o_t = beta_t (k_t . scale q_t) v_t and
    hT = beta_T k_T v_T^T.
    """
    rng = np.random.default_rng(13)
    q, k, v, g, beta, h0 = rand_inputs(rng, T=5, dk=4, dv=3)
    g[:] = -800.0                                   # exp(-800) == 0.0 in fp64
    scale = 0.9
    o, hT = fwd(q, k, v, g, beta, scale, h0, None)
    for t in range(5):
        want = beta[0, t, 0] * np.dot(k[0, t, 0], scale * q[0, t, 0]) * v[0, t, 0]
        if not np.allclose(o[0, t, 0], want, rtol=1e-12, atol=1e-14):
            return False
    want_h = beta[0, -1, 0] * np.outer(k[0, -1, 0], v[0, -1, 0])
    return np.allclose(hT[0, 0], want_h, rtol=1e-12, atol=1e-14)


def pin_scalar(fwd):
    """dk = dv = 1 with k_t = +-1: s_t = exp(g_t) (1 - beta_t) s_{t-1} + beta_t v_t k_t.

    Worked by hand from the rule (k_t^2 = 1); o_t = s_t scale q_t.
    """
    rng = np.random.default_rng(14)
    T = 9
    k = rng.choice([-1.0, 1.0], size=(1, T, 1, 1))
    q = rng.choice([-1.0, 1.0], size=(1, T, 1, 1))
    v = rng.standard_normal((1, T, 1, 1))
    beta = rng.uniform(0.1, 0.9, size=(1, T, 1))
    g = -rng.uniform(0.0, 1.0, size=(1, T, 1))
    h0 = np.array([[[[0.8]]]])
    scale = 1.3
    o, hT = fwd(q, k, v, g, beta, scale, h0, None)
    s = 0.8
    for t in range(T):
        s = np.exp(g[0, t, 0]) * (1 - beta[0, t, 0]) * s + beta[0, t, 0] * v[0, t, 0, 0] * k[0, t, 0, 0]
        if not np.isclose(o[0, t, 0, 0], s * scale * q[0, t, 0, 0], rtol=1e-12, atol=1e-14):
            return False
    return np.isclose(hT[0, 0, 0, 0], s, rtol=1e-12)


def pin_affine_in_h0(fwd):
    """o and hT are affine in h0: f(a + b) - f(0) = (f(a) - f(0)) + (f(b) - f(0))."""
    rng = np.random.default_rng(15)
    q, k, v, g, beta, ha = rand_inputs(rng, T=8, dk=4, dv=3)
    hb = rng.standard_normal(ha.shape)
    z = np.zeros_like(ha)
    oa, ta = fwd(q, k, v, g, beta, 0.6, ha, None)
    ob, tb = fwd(q, k, v, g, beta, 0.6, hb, None)
    oab, tab = fwd(q, k, v, g, beta, 0.6, ha + hb, None)
    o0, t0 = fwd(q, k, v, g, beta, 0.6, z, None)
    return (np.allclose(oab - o0, (oa - o0) + (ob - o0), atol=1e-12)
            and np.allclose(tab - t0, (ta - t0) + (tb - t0), atol=1e-12))


def pin_gqa_grouped(fwd):
    """Hqk = 2, Hv = 4: v head hv must equal a one-head run on qk head hv // 2."""
    rng = np.random.default_rng(16)
    q, k, v, g, beta, h0 = rand_inputs(rng, T=6, Hqk=2, Hv=4, dk=4, dv=3)
    o, hT = fwd(q, k, v, g, beta, 0.5, h0, None)
    for hv in range(4):
        hq = hv // 2
        o1, t1 = fwd(q[:, :, hq:hq + 1], k[:, :, hq:hq + 1], v[:, :, hv:hv + 1],
                     g[:, :, hv:hv + 1], beta[:, :, hv:hv + 1], 0.5, h0[:, hv:hv + 1], None)
        if not (np.allclose(o[:, :, hv], o1[:, :, 0], atol=1e-13)
                and np.allclose(hT[:, hv], t1[:, 0], atol=1e-13)):
            return False
    return True


def pin_varlen_equals_separate(fwd):
    """A packed batch (cu_seqlens) equals running each sequence alone from its own h0."""
    rng = np.random.default_rng(17)
    lens = [3, 1, 5]
    T = sum(lens)
    q, k, v, g, beta, _ = rand_inputs(rng, T=T, dk=4, dv=3)
    h0 = rng.standard_normal((3, 1, 4, 3))
    cu = np.array([0, 3, 4, 9])
    o, hT = fwd(q, k, v, g, beta, 0.8, h0, cu)
    for n in range(3):
        a, b = cu[n], cu[n + 1]
        o1, t1 = fwd(q[:, a:b], k[:, a:b], v[:, a:b], g[:, a:b], beta[:, a:b], 0.8,
                     h0[n:n + 1], None)
        if not (np.allclose(o[:, a:b], o1, atol=1e-13) and np.allclose(hT[n], t1[0], atol=1e-13)):
            return False
    return True


def pin_split_resume(fwd):
    """One pass over T equals two passes over [0, T1) and [T1, T) with hT carried as h0."""
    rng = np.random.default_rng(18)
    q, k, v, g, beta, h0 = rand_inputs(rng, T=9, dk=4, dv=3)
    o, hT = fwd(q, k, v, g, beta, 0.8, h0, None)
    T1 = 4
    oa, ta = fwd(q[:, :T1], k[:, :T1], v[:, :T1], g[:, :T1], beta[:, :T1], 0.8, h0, None)
    ob, tb = fwd(q[:, T1:], k[:, T1:], v[:, T1:], g[:, T1:], beta[:, T1:], 0.8, ta, None)
    return np.allclose(o, np.concatenate([oa, ob], axis=1), atol=1e-13) and np.allclose(hT, tb, atol=1e-13)


PINS = [pin_pure_decay, pin_store_retrieve, pin_reset, pin_scalar, pin_affine_in_h0,
        pin_gqa_grouped, pin_varlen_equals_separate, pin_split_resume]


def _fwd_recurrent(q, k, v, g, beta, scale, h0, cu):
    return gdn_recurrent(q, k, v, g, beta, scale, h0, cu)


def _fwd_dense(q, k, v, g, beta, scale, h0, cu):
    return gdn_dense(q, k, v, g, beta, scale, h0, cu)


def _fwd_chunked(chunk):
    def f(q, k, v, g, beta, scale, h0, cu):
        return gdn_chunked(q, k, v, g, beta, scale, h0, cu, chunk=chunk)
    return f


FORMS = {"recurrent": _fwd_recurrent, "dense": _fwd_dense, "chunked1": _fwd_chunked(1),
         "chunked2": _fwd_chunked(2), "chunked3": _fwd_chunked(3), "chunked64": _fwd_chunked(64)}


@pytest.mark.parametrize("form", list(FORMS))
@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_form_passes_pin(form, pin):
    assert pin(FORMS[form])


# ---------------------------------------------------------------------------
# Planted mistakes: each must trip at least one pin
# ---------------------------------------------------------------------------
def _step_ok(S, k, v, q, a, b, scale):
    S = a * (S @ (np.eye(len(k)) - b * np.outer(k, k))) + b * np.outer(v, k)
    return S, S @ (scale * q)


def _step_decay_on_write(S, k, v, q, a, b, scale):
    S = a * (S @ (np.eye(len(k)) - b * np.outer(k, k)) + b * np.outer(v, k))
    return S, S @ (scale * q)


def _step_read_old_state(S, k, v, q, a, b, scale):
    o = S @ (scale * q)
    S = a * (S @ (np.eye(len(k)) - b * np.outer(k, k))) + b * np.outer(v, k)
    return S, o


def _step_erase_without_beta(S, k, v, q, a, b, scale):
    S = a * (S @ (np.eye(len(k)) - np.outer(k, k))) + b * np.outer(v, k)
    return S, S @ (scale * q)


def _step_inverted_decay(S, k, v, q, a, b, scale):
    S = (1.0 / a if a > 0 else 0.0) * (S @ (np.eye(len(k)) - b * np.outer(k, k))) + b * np.outer(v, k)
    return S, S @ (scale * q)


def _step_scale_on_keys(S, k, v, q, a, b, scale):
    ks = scale * k
    S = a * (S @ (np.eye(len(k)) - b * np.outer(ks, ks))) + b * np.outer(v, ks)
    return S, S @ q


def _step_undecayed_read(S, k, v, q, a, b, scale):
    u = b * (v - S @ k)                              # reads S_{t-1} before the decay
    S = a * S + np.outer(u, k)
    return S, S @ (scale * q)


def _step_wrong_erase_sign(S, k, v, q, a, b, scale):
    S = a * (S @ (np.eye(len(k)) + b * np.outer(k, k))) + b * np.outer(v, k)
    return S, S @ (scale * q)


def _fwd_from_step(step, transpose_h0=False, head_map="grouped"):
    def fwd(q, k, v, g, beta, scale, h0, cu):
        B, T, Hqk, dk = q.shape
        Hv, dv = v.shape[2], v.shape[3]
        spans = ([(b, b, 0, T) for b in range(B)] if cu is None
                 else [(n, 0, int(cu[n]), int(cu[n + 1])) for n in range(len(cu) - 1)])
        o = np.zeros((B, T, Hv, dv))
        hT = np.zeros((len(spans), Hv, dk, dv))
        for n, b, t0, t1 in spans:
            for hv in range(Hv):
                hq = qk_head(hv, Hqk, Hv, head_map)
                if h0 is None:
                    S = np.zeros((dv, dk))
                else:
                    S = (h0[n, hv].copy() if transpose_h0 and dk == dv else h0[n, hv].T.copy())
                    if transpose_h0 and dk != dv:
                        S = h0[n, hv].reshape(dv, dk).copy()
                for t in range(t0, t1):
                    S, o[b, t, hv] = step(S, k[b, t, hq], v[b, t, hv], q[b, t, hq],
                                          np.exp(g[b, t, hv]), beta[b, t, hv], scale)
                hT[n, hv] = S.T
        return o, hT
    return fwd


def test_mutant_driver_is_sound():
    fwd = _fwd_from_step(_step_ok)
    for pin in PINS:
        assert pin(fwd), pin.__name__


MUTANTS = {
    "decay_on_write": _fwd_from_step(_step_decay_on_write),
    "read_old_state": _fwd_from_step(_step_read_old_state),
    "erase_without_beta": _fwd_from_step(_step_erase_without_beta),
    "inverted_decay": _fwd_from_step(_step_inverted_decay),
    "scale_on_keys": _fwd_from_step(_step_scale_on_keys),
    "undecayed_read": _fwd_from_step(_step_undecayed_read),
    "wrong_erase_sign": _fwd_from_step(_step_wrong_erase_sign),
    "transposed_h0": _fwd_from_step(_step_ok, transpose_h0=True),
    "modulo_head_map": _fwd_from_step(_step_ok, head_map="modulo"),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_planted_mistake_trips_a_pin(name):
    fwd = MUTANTS[name]
    failed = [p.__name__ for p in PINS if not p(fwd)]
    assert failed, f"mutant {name} passed every pin"


# ---------------------------------------------------------------------------
# Chunked form against the sequential definition (the chunked == sequential
# check of "Exp 2026-07-13 — Linear-Attention Scans on the NPU", §1, ~1e-11 at
# d=128, CS=64)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("chunk", [64, 16])
def test_chunked_matches_sequential_d128(chunk):
    rng = np.random.default_rng(21)
    q, k, v, g, beta, h0 = rand_inputs(rng, T=150, Hqk=1, Hv=2, dk=128, dv=128)
    o1, t1 = gdn_recurrent(q, k, v, g, beta, 128 ** -0.5, h0)
    o2, t2 = gdn_chunked(q, k, v, g, beta, 128 ** -0.5, h0, chunk=chunk)
    rms = np.sqrt(np.mean(o1 ** 2))
    assert np.abs(o1 - o2).max() <= 1e-10 * max(rms, 1.0)
    assert np.abs(t1 - t2).max() <= 1e-10 * max(np.sqrt(np.mean(t1 ** 2)), 1.0)


def test_chunk_size_invariance_strong_decay():
    """Strong decay (g ~ -softplus(N(1,1))): chunk 64 and 128 agree with the definition."""
    rng = np.random.default_rng(22)
    q, k, v, g, beta, _ = rand_inputs(rng, T=200, dk=32, dv=16, h0=False, g_mu=1.0)
    o1, t1 = gdn_recurrent(q, k, v, g, beta, 32 ** -0.5)
    for c in (64, 128):
        o2, t2 = gdn_chunked(q, k, v, g, beta, 32 ** -0.5, chunk=c)
        assert np.abs(o1 - o2).max() < 1e-10
        assert np.abs(t1 - t2).max() < 1e-10


def test_dense_definition_matches_recurrent_gqa_varlen():
    rng = np.random.default_rng(23)
    q, k, v, g, beta, _ = rand_inputs(rng, T=10, Hqk=2, Hv=4, dk=6, dv=5)
    h0 = rng.standard_normal((3, 4, 6, 5))
    cu = np.array([0, 4, 4, 10])                    # includes an empty sequence
    o1, t1 = gdn_dense(q, k, v, g, beta, 0.4, h0, cu)
    o2, t2 = gdn_recurrent(q, k, v, g, beta, 0.4, h0, cu)
    assert np.abs(o1 - o2).max() < 1e-13 and np.abs(t1 - t2).max() < 1e-13
    assert np.array_equal(t2[1], h0[1])             # empty sequence: hT = h0


def test_state_norm_bound():
    """||S_t||_F <= gamma_t ||S_0||_F + sum_{j<=t} beta_j ||v_j|| exp(G_t - G_j) for unit keys."""
    rng = np.random.default_rng(24)
    q, k, v, g, beta, h0 = rand_inputs(rng, T=40, dk=8, dv=6)
    from oracle import recurrent_chain
    h = h0[0, 0].copy()
    G = np.cumsum(g[0, :, 0])
    for t in range(40):
        recurrent_chain(q[0, t:t + 1, 0], k[0, t:t + 1, 0], v[0, t:t + 1, 0], g[0, t:t + 1, 0],
                        beta[0, t:t + 1, 0], h, 0.5)
        bound = np.exp(G[t]) * np.linalg.norm(h0[0, 0])
        bound += sum(beta[0, j, 0] * np.linalg.norm(v[0, j, 0]) * np.exp(G[t] - G[j]) for j in range(t + 1))
        assert np.linalg.norm(h) <= bound * (1 + 1e-12)


def test_prefill_then_decode_equals_one_pass():
    """Decode steps continuing from hT equal the definition over the concatenated tokens."""
    rng = np.random.default_rng(25)
    q, k, v, g, beta, h0 = rand_inputs(rng, T=12, Hqk=1, Hv=2, dk=6, dv=4)
    oa, hT = gdn_chunked(q[:, :9], k[:, :9], v[:, :9], g[:, :9], beta[:, :9], 0.5, h0, chunk=4)
    o_all, h_all = gdn_recurrent(q, k, v, g, beta, 0.5, h0)
    h = hT
    for t in range(9, 12):
        o_t, h = gdn_step(q[:, t], k[:, t], v[:, t], g[:, t], beta[:, t], h, 0.5)
        assert np.abs(o_t - o_all[:, t]).max() < 1e-12
    assert np.abs(h - h_all).max() < 1e-12


def test_forward_substitution_is_the_inverse():
    """Against the library inverse of the unit lower-triangular matrix."""
    rng = np.random.default_rng(26)
    for L in (1, 2, 17, 64):
        A = np.tril(rng.standard_normal((L, L)) * 0.3, k=-1)
        X = forward_substitution_inverse(A)
        assert np.allclose(X, np.linalg.inv(np.eye(L) + A), atol=1e-10)
        assert np.allclose(np.triu(X, 1), 0) and np.allclose(np.diag(X), 1)


def test_io_byte_model_matches_figure4():
    """The algorithmic byte model reproduces Figure 4(a)'s ideal-resident traffic."""
    from linear_attention_prefill_gb300.roofline import io_bytes
    rows = [l.split() for l in open(os.path.join(GOLDEN, "fig4_io_traffic.txt"))
            if l.strip() and not l.startswith("#")]
    assert len(rows) == 2
    for name, T, H, d, eb, gate, mib in rows:
        T, H, d, eb = int(T), int(H), int(d), int(eb)
        b = io_bytes(T, 1, H, H, d, d, eb, h0_read=True, hT_written=True,
                     gate_per_channel=(gate == "per_channel"))
        # the state term counts N * Hv states; Figure 4 is one sequence of H heads
        assert round(b / 2 ** 20, 2) == float(mib), (name, b / 2 ** 20)
