"""The fused prologue (in-kernel L2 norm of q, k and the GDN gates from raw inputs).

CPU: the oracle's prologue is pinned by invariants of its formulas - per-row scale
invariance of the normalisation, the gate maps' closed values and their inverses.
GPU: gdn_chunk_fwd_prologue and gdn_recurrent_step_prologue against the fp64 oracle
applied to the same raw inputs."""
import numpy as np
import pytest
import torch

from helpers import TOL, rel_err, to_np
from oracle import gdn_recurrent, gdn_step, prologue


def test_normalisation_is_scale_invariant_per_row():
    rng = np.random.default_rng(60)
    q = rng.standard_normal((1, 9, 2, 16)) * 3
    k = rng.standard_normal((1, 9, 2, 16)) * 3
    a = rng.standard_normal((1, 9, 4))
    b = rng.standard_normal((1, 9, 4))
    s = np.exp(rng.standard_normal((1, 9, 2, 1)))
    q1, k1, g1, b1 = prologue(q, k, a, b)
    q2, k2, g2, b2 = prologue(q * s, k * s[..., ::-1, :], a, b)
    assert np.allclose(q1, q2, rtol=1e-6) and np.allclose(k1, k2, rtol=1e-6)
    assert np.allclose(np.linalg.norm(q1, axis=-1), 1.0, rtol=1e-6)


def test_gate_maps_closed_values():
    a = np.array([[[0.0, -40.0, 40.0]]])
    b = np.array([[[0.0, 50.0, -50.0]]])
    A_log = np.array([np.log(2.0), 0.0, 0.0])
    dt_bias = np.array([0.0, 0.0, 0.0])
    _, _, g, beta = prologue(np.ones((1, 1, 1, 4)), np.ones((1, 1, 1, 4)), a, b, A_log, dt_bias)
    assert np.isclose(g[0, 0, 0], -2.0 * np.log(2.0))   # softplus(0) = ln 2, exp(A_log) = 2
    assert abs(g[0, 0, 1]) < 1e-15                       # softplus(-40) ~ 0: no decay
    assert np.isclose(g[0, 0, 2], -40.0)                 # softplus(40) = 40
    assert np.isclose(beta[0, 0, 0], 0.5) and beta[0, 0, 1] > 1 - 1e-15 and beta[0, 0, 2] < 1e-20


def test_gate_maps_invert():
    """a = log(exp(-g) - 1), b = log(beta / (1 - beta)) give back g and beta."""
    rng = np.random.default_rng(61)
    g = -np.log1p(np.exp(rng.standard_normal((1, 7, 3))))
    beta = 1 / (1 + np.exp(-rng.standard_normal((1, 7, 3))))
    a = np.log(np.expm1(-g))
    b = np.log(beta / (1 - beta))
    _, _, g2, beta2 = prologue(np.ones((1, 7, 1, 4)), np.ones((1, 7, 1, 4)), a, b)
    assert np.allclose(g2, g, rtol=1e-12) and np.allclose(beta2, beta, rtol=1e-12)


def raw_inputs(T, Hqk=1, Hv=2, dk=128, dv=128, seed=62, device="cuda"):
    gen = torch.Generator(device=device).manual_seed(seed)

    def randn(*shape):
        return torch.randn(*shape, generator=gen, device=device)
    q = (randn(1, T, Hqk, dk) * torch.exp(randn(1, T, Hqk, 1))).to(torch.bfloat16)
    k = (randn(1, T, Hqk, dk) * torch.exp(randn(1, T, Hqk, 1))).to(torch.bfloat16)
    v = randn(1, T, Hv, dv).to(torch.bfloat16)
    a = randn(1, T, Hv).contiguous()
    b = randn(1, T, Hv).contiguous()
    A_log = (0.3 * randn(Hv)).contiguous()
    dt_bias = (0.3 * randn(Hv)).contiguous()
    h0 = randn(1, Hv, dk, dv) * 0.1
    return q, k, v, a, b, A_log, dt_bias, h0


@pytest.mark.gpu
@pytest.mark.parametrize("T", [1, 64, 150])
@pytest.mark.parametrize("with_params", [False, True])
def test_prologue_forward_parity(cuda_lib, T, with_params):
    q, k, v, a, b, A_log, dt_bias, h0 = raw_inputs(T, seed=62 + T)
    if not with_params:
        A_log = dt_bias = None
    o, hT = cuda_lib.gdn_chunk_fwd_prologue(q, k, v, a, b, A_log, dt_bias, h0)
    torch.cuda.synchronize()
    qh, kh, g, beta = prologue(q, k, a, b, A_log, dt_bias)
    o_ref, h_ref = gdn_recurrent(qh, kh, v, g, beta, 128 ** -0.5, h0)
    assert rel_err(to_np(o), o_ref, out_dtype="bf16") < TOL["bf16"]
    assert rel_err(to_np(hT), h_ref) < TOL["bf16"]


@pytest.mark.gpu
def test_prologue_decode_step_parity(cuda_lib):
    torch.manual_seed(63)
    N, Hqk, Hv, dk, dv = 3, 1, 4, 128, 128
    q = (torch.randn(N, Hqk, dk, device="cuda") * 2.5).to(torch.bfloat16)
    k = (torch.randn(N, Hqk, dk, device="cuda") * 0.4).to(torch.bfloat16)
    v = torch.randn(N, Hv, dv, device="cuda").to(torch.bfloat16)
    a = torch.randn(N, Hv, device="cuda")
    b = torch.randn(N, Hv, device="cuda")
    A_log = 0.3 * torch.randn(Hv, device="cuda")
    dt_bias = 0.3 * torch.randn(Hv, device="cuda")
    h = torch.randn(N, Hv, dk, dv, device="cuda") * 0.1
    h_in = h.clone()
    o = cuda_lib.gdn_recurrent_step_prologue(q, k, v, a, b, h, A_log, dt_bias)
    torch.cuda.synchronize()
    qh, kh, g, beta = prologue(q, k, a, b, A_log, dt_bias)
    o_ref, h_ref = gdn_step(qh, kh, v, g, beta, h_in, 128 ** -0.5)
    assert rel_err(to_np(o), o_ref, out_dtype="bf16") < TOL["bf16"]
    assert rel_err(to_np(h), h_ref) < TOL["bf16"]
