"""GPU parity of gdn_recurrent_step (one decode token) and of prefill followed by
decode steps, against the fp64 oracle over the concatenated tokens."""
import numpy as np
import pytest
import torch

from helpers import TOL, rel_err, to_np
from linear_attention_prefill_gb300.workloads import WORKLOADS, Workload, make_decode_inputs, make_inputs
from oracle import gdn_recurrent, gdn_step, recurrent_chain

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 64), (128, 64), (64, 128)])
def test_single_step(cuda_lib, dtype, dk, dv):
    w = Workload("dec", (1, 1, 1), 2, 4, dk, dv, 64, dtype, seed=31)
    x = make_decode_inputs(w, 0, device="cuda")
    gen = torch.Generator(device="cuda").manual_seed(5)
    h = torch.randn((3, 4, dk, dv), generator=gen, device="cuda") * 0.3
    h_before = h.clone()
    o = cuda_lib.gdn_recurrent_step(x["q"], x["k"], x["v"], x["g"], x["beta"], h)
    torch.cuda.synchronize()
    o_ref, h_ref = gdn_step(x["q"], x["k"], x["v"], x["g"], x["beta"], h_before, x["scale"])
    assert rel_err(to_np(o), o_ref, out_dtype=dtype) < TOL[dtype]
    assert rel_err(to_np(h), h_ref) < TOL[dtype]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_prefill_then_decode(cuda_lib, dtype):
    w = Workload("pd", (200,), 1, 2, 128, 128, 64, dtype, h0_std=0.1, seed=32)
    x = make_inputs(w, device="cuda")
    o, hT = cuda_lib.gdn_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    h = hT.clone()
    outs, toks = [], []
    for s in range(20):
        d = make_decode_inputs(w, s, device="cuda")
        outs.append(cuda_lib.gdn_recurrent_step(d["q"], d["k"], d["v"], d["g"], d["beta"], h))
        toks.append(d)
    torch.cuda.synchronize()
    cat = {k_: torch.cat([x[k_]] + [d[k_][:, None] for d in toks], dim=1)
           for k_ in ("q", "k", "v", "g", "beta")}
    o_ref, h_ref = gdn_recurrent(cat["q"], cat["k"], cat["v"], cat["g"], cat["beta"], x["scale"],
                                 x["h0"])
    o_dec = torch.stack(outs, dim=1)
    assert rel_err(to_np(o_dec), o_ref[:, 200:], out_dtype=dtype) < TOL[dtype]
    assert rel_err(to_np(h), h_ref) < TOL[dtype]


def test_long_context_then_1000_steps(cuda_lib):
    """T = 65536 strong-decay prefill, then 1000 decode steps; one sampled head end to end."""
    w = WORKLOADS["long_64k_strong"]
    x = make_inputs(w, device="cuda")
    o, hT = cuda_lib.gdn_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                                   chunk=w.chunk)
    h = hT.clone()
    hv = 11
    steps = []
    o_last = None
    for s in range(w.decode_steps):
        d = make_decode_inputs(w, s, device="cuda")
        o_last = cuda_lib.gdn_recurrent_step(d["q"], d["k"], d["v"], d["g"], d["beta"], h)
        steps.append({k_: d[k_][0, hv].detach().cpu() for k_ in ("q", "k", "v", "g", "beta")})
    torch.cuda.synchronize()
    # oracle: this head's chain over prefill + decode tokens
    hs = to_np(hT[0, hv])
    chain = np.zeros((128, 128))
    recurrent_chain(to_np(x["q"][0, :, hv]), to_np(x["k"][0, :, hv]), to_np(x["v"][0, :, hv]),
                    to_np(x["g"][0, :, hv]), to_np(x["beta"][0, :, hv]), chain, w.scale)
    assert rel_err(hs, chain) < TOL["bf16"]
    q = np.stack([to_np(s_["q"]) for s_ in steps])
    k = np.stack([to_np(s_["k"]) for s_ in steps])
    v = np.stack([to_np(s_["v"]) for s_ in steps])
    g = np.array([float(s_["g"]) for s_ in steps])
    b = np.array([float(s_["beta"]) for s_ in steps])
    o_ref = recurrent_chain(q, k, v, g, b, chain, w.scale)
    assert rel_err(to_np(h[0, hv]), chain) < TOL["bf16"]
    assert rel_err(to_np(o_last[0, hv]), o_ref[-1], out_dtype="bf16") < TOL["bf16"]
