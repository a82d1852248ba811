"""GPU parity of Kimi Delta Attention (kda_chunk_fwd, kda_recurrent_step) through the C ABI
against the fp64 KDA oracle (the per-channel-gate recurrence), element by element on the
same seeded inputs: ragged chunks, GQA, packed sequences with an empty one, carried
state, weak and strong per-channel decay, the 16-head 4K layer on sampled heads, and the
decode step."""
import numpy as np
import pytest
import torch

from helpers import TOL, check_heads, rel_err, to_np
from linear_attention_prefill_gb300.workloads import WORKLOADS, Workload, make_inputs
from oracle import kda_recurrent, kda_step

pytestmark = pytest.mark.gpu


def kda_case(T, Hqk=2, Hv=2, dv=128, h0_std=0.1, seed=0, varlen=False, **kw):
    seqlens = T if isinstance(T, tuple) else (T,)
    return Workload("kda_case", seqlens, Hqk, Hv, 128, dv, 64, "bf16", h0_std=h0_std,
                    varlen=varlen, seed=seed, op="kda", **kw)


def run(lap, x, chunk=64, **kw):
    return lap.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], chunk=chunk,
                             scale=x["scale"], cu_seqlens=x["cu_seqlens"], **kw)


@pytest.mark.parametrize("T,dv", [(1, 128), (63, 64), (64, 128), (65, 128), (200, 64),
                                  (257, 128)])
def test_kda_ragged(cuda_lib, T, dv):
    """One sequence spanning several chunks and a ragged tail; both dv tiles."""
    x = make_inputs(kda_case(T, dv=dv, seed=80 + T), device="cuda")
    o, hT = run(cuda_lib, x)
    check_heads(x, o, hT, heads=range(2), dtype="bf16", op="kda")


def test_kda_gqa_batch_no_state(cuda_lib):
    """Two rows, each qk head shared by two v heads, no initial state."""
    x = make_inputs(kda_case((130, 130), Hqk=2, Hv=4, h0_std=None, seed=81), device="cuda")
    o, hT = run(cuda_lib, x)
    check_heads(x, o, hT, heads=range(4), dtype="bf16", op="kda")


def test_kda_varlen(cuda_lib):
    """Packed sequences (one empty, one of a single token) with per-sequence state."""
    x = make_inputs(kda_case((70, 0, 1, 129, 64), Hqk=2, Hv=4, seed=82, varlen=True),
                    device="cuda")
    o, hT = run(cuda_lib, x)
    check_heads(x, o, hT, heads=range(4), seqs=range(5), dtype="bf16", op="kda")


@pytest.mark.parametrize("g_mu,g_scale", [(0.0, 0.02), (1.0, 1.0), (-2.0, 3.0)])
def test_kda_decay_regimes(cuda_lib, g_mu, g_scale):
    """Weak decay (long memory), strong decay, and a wide spread of per-channel decays."""
    x = make_inputs(kda_case(600, seed=83, g_mu=g_mu, g_scale=g_scale), device="cuda")
    o, hT = run(cuda_lib, x)
    check_heads(x, o, hT, heads=range(2), dtype="bf16", op="kda")
    assert torch.isfinite(o.float()).all() and torch.isfinite(hT).all()


def test_kda_layer_sampled_heads(cuda_lib):
    """The 16-head 4K layer in the launch configuration the bench times; heads sampled."""
    x = make_inputs(WORKLOADS["kda_16h_4k"], device="cuda")
    o, hT = run(cuda_lib, x)
    check_heads(x, o, hT, heads=[0, 7, 15], dtype="bf16", op="kda")


def test_kda_chunk_128_is_the_same_function(cuda_lib):
    x = make_inputs(kda_case(300, seed=84), device="cuda")
    o64, h64 = run(cuda_lib, x, 64)
    o128, h128 = run(cuda_lib, x, 128)
    assert torch.equal(o64, o128) and torch.equal(h64, h128)


def test_kda_in_place_state_and_empty(cuda_lib):
    """hT may be h0 (each chain reads its state before writing it); T = 0 copies h0."""
    x = make_inputs(kda_case(150, seed=85), device="cuda")
    o_ref, h_ref = run(cuda_lib, x)
    h = x["h0"].clone()
    o, hT = run(cuda_lib, x, hT=h)
    assert hT.data_ptr() == h.data_ptr()
    assert torch.equal(o, o_ref) and torch.equal(h, h_ref)
    e = make_inputs(kda_case(0, seed=86), device="cuda")
    _, h_empty = run(cuda_lib, e)
    assert torch.equal(h_empty, e["h0"])


def test_kda_rejects_unsupported(cuda_lib):
    x = make_inputs(kda_case(64, seed=87), device="cuda")
    q64 = x["q"][..., :64].contiguous()
    with pytest.raises(cuda_lib.GdnError) as err:
        cuda_lib.kda_chunk_fwd(q64, q64.clone(), x["v"], x["g"][..., :64].contiguous(),
                               x["beta"], None)
    assert err.value.status == 2  # GDN_ERR_UNSUPPORTED: dk = 64


def test_kda_decode_step_and_continuation(cuda_lib):
    """Prefill, then one decode token: equals the oracle over the concatenated sequence."""
    w = kda_case(100, Hqk=1, Hv=2, seed=88)
    x = make_inputs(w, device="cuda")
    o, hT = run(cuda_lib, x)
    gen = torch.Generator(device="cuda").manual_seed(89)
    q1 = torch.nn.functional.normalize(torch.randn(1, 1, 128, generator=gen, device="cuda"),
                                       dim=-1).to(torch.bfloat16)
    k1 = torch.nn.functional.normalize(torch.randn(1, 1, 128, generator=gen, device="cuda"),
                                       dim=-1).to(torch.bfloat16)
    v1 = torch.randn(1, 2, 128, generator=gen, device="cuda").to(torch.bfloat16)
    g1 = -torch.nn.functional.softplus(torch.randn(1, 2, 128, generator=gen, device="cuda"))
    b1 = torch.sigmoid(torch.randn(1, 2, generator=gen, device="cuda"))
    h = hT.clone()
    o1 = cuda_lib.kda_recurrent_step(q1, k1, v1, g1.contiguous(), b1.contiguous(), h,
                                     scale=x["scale"])
    # the step alone against the oracle's step from the kernel's own prefill state
    o_ref, h_ref = kda_step(to_np(q1), to_np(k1), to_np(v1), to_np(g1), to_np(b1), to_np(hT),
                            x["scale"])
    assert rel_err(to_np(o1), o_ref, out_dtype="bf16") < TOL["bf16"]
    assert rel_err(to_np(h), h_ref) < 1e-5
    # prefill + step against one oracle pass over all 101 tokens
    cat = lambda a, b: np.concatenate([to_np(a), to_np(b)[:, None]], axis=1)
    o_all, h_all = kda_recurrent(cat(x["q"], q1), cat(x["k"], k1), cat(x["v"], v1),
                                 cat(x["g"], g1), cat(x["beta"], b1), x["scale"], to_np(x["h0"]))
    assert rel_err(to_np(o1), o_all[:, -1], out_dtype="bf16") < TOL["bf16"]
    assert rel_err(to_np(h), h_all) < TOL["bf16"]


def test_kda_gate_domain_edge(cuda_lib):
    """Log-decays down to -10 per token and channel (the stated domain of the GPU path):
    a tenth of the gate entries set to -10, runs of 8 strongly decaying tokens in some
    channels, the rest weak; the grams' block-referenced factors must stay in range."""
    x = make_inputs(kda_case(300, seed=90), device="cuda")
    gen = torch.Generator(device="cuda").manual_seed(91)
    g = x["g"] * 0.05
    g = torch.where(torch.rand(g.shape, generator=gen, device="cuda") < 0.1,
                    torch.full_like(g, -10.0), g)
    g[:, 40:48, :, :16] = -10.0   # eight consecutive tokens, sixteen channels
    x["g"] = g.contiguous()
    o, hT = run(cuda_lib, x)
    assert torch.isfinite(o.float()).all() and torch.isfinite(hT).all()
    check_heads(x, o, hT, heads=range(2), dtype="bf16", op="kda")


def test_kda_long_sequence_weak_decay(cuda_lib):
    """16K tokens (256 chunks) with weak per-channel decay: the carried state stays accurate
    over a long chain (one v head checked in full against the fp64 recurrence)."""
    x = make_inputs(kda_case(16384, Hqk=1, Hv=2, seed=92, g_scale=0.02), device="cuda")
    o, hT = run(cuda_lib, x)
    assert torch.isfinite(o.float()).all() and torch.isfinite(hT).all()
    check_heads(x, o, hT, heads=[1], dtype="bf16", op="kda")


def test_kda_gate_outside_range_is_reported(cuda_lib):
    """A log-decay below -10 is outside the range the GPU path is exact for: the prep
    records it in the device error word and gdn_device_status reports INVALID_ARG once;
    an in-range call afterwards reports nothing."""
    cuda_lib.gdn_device_status()  # clear anything earlier
    x = make_inputs(kda_case(130, seed=93), device="cuda")
    g = x["g"].clone()
    g[0, 70, 1, 5] = -12.0
    run(cuda_lib, dict(x, g=g.contiguous()))
    with pytest.raises(cuda_lib.GdnError) as err:
        cuda_lib.gdn_device_status()
    assert err.value.status == 1  # GDN_ERR_INVALID_ARG
    run(cuda_lib, x)
    cuda_lib.gdn_device_status()  # in range: no report


def test_kda_32_column_chain_tile(cuda_lib):
    """32 v heads: the KDA chain runs 32-column tiles (128 CTAs)."""
    x = make_inputs(kda_case(150, Hqk=8, Hv=32, seed=94), device="cuda")
    o, hT = run(cuda_lib, x)
    check_heads(x, o, hT, heads=[0, 15, 31], dtype="bf16", op="kda")


@pytest.mark.parametrize("dk", [64, 128])
def test_kda_decode_step_head_dims(cuda_lib, dk):
    """The decode step against the oracle's step at both key head dims (GQA, dv = 64)."""
    gen = torch.Generator(device="cuda").manual_seed(95 + dk)
    N, Hqk, Hv, dv = 3, 2, 4, 64
    unit = lambda x: torch.nn.functional.normalize(x, dim=-1).to(torch.bfloat16)
    q = unit(torch.randn(N, Hqk, dk, generator=gen, device="cuda"))
    k = unit(torch.randn(N, Hqk, dk, generator=gen, device="cuda"))
    v = torch.randn(N, Hv, dv, generator=gen, device="cuda").to(torch.bfloat16)
    g = -torch.nn.functional.softplus(torch.randn(N, Hv, dk, generator=gen, device="cuda"))
    b = torch.sigmoid(torch.randn(N, Hv, generator=gen, device="cuda"))
    h = torch.randn(N, Hv, dk, dv, generator=gen, device="cuda") * 0.1
    h_in = h.clone()
    o = cuda_lib.kda_recurrent_step(q, k, v, g.contiguous(), b.contiguous(), h)
    o_ref, h_ref = kda_step(to_np(q), to_np(k), to_np(v), to_np(g), to_np(b), to_np(h_in),
                            dk ** -0.5)
    assert rel_err(to_np(o), o_ref, out_dtype="bf16") < TOL["bf16"]
    assert rel_err(to_np(h), h_ref) < 1e-5
