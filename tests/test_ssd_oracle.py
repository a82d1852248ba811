"""Pins for the Mamba-2 SSD oracle, all on the CPU.

Each pin is fixed by something other than the oracle's own recurrence: the
closed form of the unrolled recurrence, causal linear attention (g = 0,
beta = 1) as a plain masked matrix product, pure decay, the chunked form, and
prefill + decode == one pass.  Planted mistakes must each trip a pin.
"""
import numpy as np
import pytest

from oracle import ssd_chunked, ssd_recurrent, ssd_step, ssd_unrolled


def rand_inputs(rng, B=1, T=9, Hqk=1, Hv=2, dk=5, dv=3, h0=True):
    q = rng.standard_normal((B, T, Hqk, dk)) / np.sqrt(dk)
    k = rng.standard_normal((B, T, Hqk, dk)) / np.sqrt(dk)
    v = rng.standard_normal((B, T, Hv, dv))
    beta = np.log1p(np.exp(rng.standard_normal((B, T, Hv))))   # dt = softplus(.)
    g = -beta * np.exp(0.3 * rng.standard_normal((1, 1, Hv)))  # dt * A, A < 0 per head
    hz = rng.standard_normal((B, Hv, dk, dv)) * 0.5 if h0 else None
    return q, k, v, g, beta, hz


def pin_unrolled(fwd):
    """The recurrence equals its unrolled closed form (GQA groups, two rows, h0)."""
    rng = np.random.default_rng(31)
    q, k, v, g, beta, h0 = rand_inputs(rng, B=2, T=11, Hqk=1, Hv=2)
    o, hT = fwd(q, k, v, g, beta, 0.6, h0, None)
    o2, hT2 = ssd_unrolled(q, k, v, g, beta, 0.6, h0)
    return np.allclose(o, o2, rtol=1e-11, atol=1e-13) and np.allclose(hT, hT2, rtol=1e-11,
                                                                      atol=1e-13)


def pin_causal_linear_attention(fwd):
    """g = 0, beta = 1, h0 = 0: O = scale * tril(Q K^T) V, a masked matrix product."""
    rng = np.random.default_rng(32)
    q, k, v, g, beta, _ = rand_inputs(rng, T=8, Hqk=1, Hv=1, dk=4, dv=6)
    g[:] = 0.0
    beta[:] = 1.0
    o, hT = fwd(q, k, v, g, beta, 0.9, None, None)
    Q, K, V = q[0, :, 0], k[0, :, 0], v[0, :, 0]
    want = 0.9 * np.tril(Q @ K.T) @ V
    return np.allclose(o[0, :, 0], want, rtol=1e-12, atol=1e-13) and np.allclose(
        hT[0, 0], K.T @ V, rtol=1e-12, atol=1e-13)


def pin_pure_decay(fwd):
    """k = 0: nothing is written; o_t = exp(G_t) h0^T (scale q_t), hT = exp(G_T) h0."""
    rng = np.random.default_rng(33)
    q, k, v, g, beta, h0 = rand_inputs(rng, T=6, Hqk=1, Hv=1, dk=5, dv=3)
    k[:] = 0.0
    o, hT = fwd(q, k, v, g, beta, 0.8, h0, None)
    G = np.cumsum(g[0, :, 0])
    ok = all(np.allclose(o[0, t, 0], np.exp(G[t]) * (h0[0, 0].T @ (0.8 * q[0, t, 0])),
                         rtol=1e-12, atol=1e-14) for t in range(6))
    return ok and np.allclose(hT[0, 0], np.exp(G[-1]) * h0[0, 0], rtol=1e-12, atol=1e-14)


def pin_one_token_writes_beta_k_v(fwd):
    """One token from h0 = 0: hT = beta k v^T (k along the rows: [dk, dv])."""
    rng = np.random.default_rng(34)
    q, k, v, g, beta, _ = rand_inputs(rng, T=1, Hqk=1, Hv=1, dk=4, dv=4)
    _, hT = fwd(q, k, v, g, beta, 1.0, None, None)
    return np.allclose(hT[0, 0], beta[0, 0, 0] * np.outer(k[0, 0, 0], v[0, 0, 0]), rtol=1e-12)


PINS = [pin_unrolled, pin_causal_linear_attention, pin_pure_decay, pin_one_token_writes_beta_k_v]


def _recurrent(q, k, v, g, beta, scale, h0, cu):
    return ssd_recurrent(q, k, v, g, beta, scale, h0, cu)


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_recurrent_oracle_meets_pin(pin):
    assert pin(_recurrent)


@pytest.mark.parametrize("chunk", [16, 64])
def test_chunked_matches_sequential_d128(chunk):
    rng = np.random.default_rng(35)
    q, k, v, g, beta, h0 = rand_inputs(rng, B=1, T=200, Hqk=1, Hv=2, dk=128, dv=64)
    o1, t1 = ssd_recurrent(q, k, v, g, beta, 1.0, h0)
    o2, t2 = ssd_chunked(q, k, v, g, beta, 1.0, h0, chunk=chunk)
    rms = np.sqrt(np.mean(o1 ** 2))
    assert np.abs(o1 - o2).max() / rms < 1e-10
    assert np.abs(t1 - t2).max() / np.sqrt(np.mean(t1 ** 2)) < 1e-10


def test_chunked_varlen_matches_sequential():
    rng = np.random.default_rng(36)
    lens = [70, 0, 5, 129]
    T = sum(lens)
    q, k, v, g, beta, _ = rand_inputs(rng, B=1, T=T, Hqk=2, Hv=4, dk=16, dv=8, h0=False)
    h0 = rng.standard_normal((len(lens), 4, 16, 8)) * 0.3
    cu = np.concatenate([[0], np.cumsum(lens)])
    o1, t1 = ssd_recurrent(q, k, v, g, beta, 0.5, h0, cu)
    o2, t2 = ssd_chunked(q, k, v, g, beta, 0.5, h0, cu, chunk=64)
    assert np.allclose(o1, o2, rtol=1e-10, atol=1e-12) and np.allclose(t1, t2, rtol=1e-10,
                                                                       atol=1e-12)


def test_prefill_then_step_equals_one_pass():
    rng = np.random.default_rng(37)
    q, k, v, g, beta, h0 = rand_inputs(rng, T=10, Hqk=1, Hv=2, dk=6, dv=4)
    o, hT = ssd_recurrent(q, k, v, g, beta, 0.7, h0)
    _, h9 = ssd_recurrent(q[:, :9], k[:, :9], v[:, :9], g[:, :9], beta[:, :9], 0.7, h0)
    o_last, h_new = ssd_step(q[:, 9], k[:, 9], v[:, 9], g[:, 9], beta[:, 9], h9, 0.7)
    assert np.allclose(o_last, o[:, 9], rtol=1e-12) and np.allclose(h_new, hT, rtol=1e-12)


# ---------------------------------------------------------------------------
# Planted mistakes: each must fail at least one pin
# ---------------------------------------------------------------------------
def _mutant(kind):
    def chain(qs, ks, vs, gs, betas, h, scale):
        L = qs.shape[0]
        o = np.zeros((L, h.shape[1]))
        for t in range(L):
            b = 1.0 if kind == "no_beta" else betas[t]
            if kind == "decay_after_write":
                h += b * np.outer(ks[t], vs[t])
                h *= np.exp(gs[t])
            else:
                h *= np.exp(-gs[t] if kind == "inverted_decay" else gs[t])
                if kind == "read_old_state":
                    o[t] = h.T @ (scale * qs[t])
                h += b * np.outer(ks[t], vs[t])
            if kind != "read_old_state":
                o[t] = h.T @ (scale * qs[t])
        return o

    def fwd(q, k, v, g, beta, scale, h0, cu):
        from oracle.ssd_oracle import _over_chains
        return _over_chains(chain, q, k, v, g, beta, scale, h0, cu, "grouped", None)
    return fwd


@pytest.mark.parametrize("kind", ["decay_after_write", "no_beta", "inverted_decay",
                                  "read_old_state"])
def test_planted_mistake_is_caught(kind):
    fwd = _mutant(kind)
    assert not all(pin(fwd) for pin in PINS), kind
