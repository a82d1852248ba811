"""GPU parity: gdn_chunk_fwd through the C ABI against the fp64 oracle.

Small cases compare every element; the full-size workloads (launched exactly as
bench.py launches them) compare every token of sampled (sequence, v head)
chains, which the oracle computes one by one.  Tolerance: max |x - ref| /
RMS(ref) <= 2e-2 for bf16 inputs with fp32 accumulation, 1e-4 for the fp32
path, on o and on the final state.  A bf16 o is first allowed the half-ulp
rounding of its own store (helpers.rel_err); the fp32 state gets no allowance.
"""
import numpy as np
import pytest
import torch

from helpers import TOL, check_heads, rel_err, to_np
from oracle import gdn_recurrent
from linear_attention_prefill_gb300.workloads import WORKLOADS, Workload, make_inputs

pytestmark = pytest.mark.gpu


def run(lap, x, chunk=64, hT=True):
    o, h = lap.gdn_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], chunk=chunk,
                             cu_seqlens=x["cu_seqlens"], output_final_state=hT)
    torch.cuda.synchronize()
    return o, h


def small(T, Hqk=1, Hv=2, dk=128, dv=128, dtype="bf16", h0=0.1, seed=0, g_mu=0.0, g_scale=1.0,
          seqlens=None):
    if seqlens is not None:
        return Workload("case", tuple(seqlens), Hqk, Hv, dk, dv, 64, dtype, g_mu=g_mu,
                        g_scale=g_scale, h0_std=h0, varlen=True, seed=seed)
    return Workload("case", (T,), Hqk, Hv, dk, dv, 64, dtype, g_mu=g_mu, g_scale=g_scale,
                    h0_std=h0, seed=seed)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 127, 128, 129, 200])
def test_ragged_lengths(cuda_lib, T, dtype):
    w = small(T, dtype=dtype, seed=T)
    x = make_inputs(w, device="cuda")
    o, hT = run(cuda_lib, x)
    check_heads(x, o, hT, heads=range(w.Hv), dtype=dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 64), (64, 128), (128, 128)])
def test_head_dims(cuda_lib, dk, dv, dtype):
    w = small(150, Hqk=2, Hv=4, dk=dk, dv=dv, dtype=dtype, seed=dk + dv)
    x = make_inputs(w, device="cuda")
    o, hT = run(cuda_lib, x)
    check_heads(x, o, hT, heads=range(w.Hv), dtype=dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_gqa_ratio_four_and_batch_rows(cuda_lib, dtype):
    w = Workload("rows", (100, 100), 1, 4, 128, 128, 64, dtype, h0_std=0.1, seed=9)
    x = make_inputs(w, device="cuda")
    assert x["q"].shape[0] == 2
    o, hT = run(cuda_lib, x)
    check_heads(x, o, hT, heads=range(4), dtype=dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_varlen_with_empty_and_short_sequences(cuda_lib, dtype):
    w = small(0, Hqk=2, Hv=4, dtype=dtype, seqlens=[0, 1, 64, 0, 130, 65], seed=10)
    x = make_inputs(w, device="cuda")
    o, hT = run(cuda_lib, x)
    check_heads(x, o, hT, heads=range(4), dtype=dtype)
    # empty sequences hand their initial state straight through
    assert torch.equal(hT[0], x["h0"][0]) and torch.equal(hT[3], x["h0"][3])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_no_initial_state_and_no_final_state(cuda_lib, dtype):
    w = small(100, h0=None, dtype=dtype, seed=11)
    x = make_inputs(w, device="cuda")
    o, hT = run(cuda_lib, x, hT=False)
    assert hT is None
    check_heads(x, o, None, heads=range(w.Hv), dtype=dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_final_state_in_place(cuda_lib, dtype):
    w = small(130, dtype=dtype, seed=12)
    x = make_inputs(w, device="cuda")
    o_ref, h_ref = run(cuda_lib, x)
    h = x["h0"].clone()
    o, h2 = cuda_lib.gdn_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], h, hT=h)
    torch.cuda.synchronize()
    assert h2.data_ptr() == h.data_ptr()
    assert torch.equal(h, h_ref) and torch.equal(o, o_ref)


def test_zero_length_copies_state(cuda_lib):
    w = small(0, seed=13)
    x = make_inputs(w, device="cuda")
    o, hT = run(cuda_lib, x)
    assert o.numel() == 0 and torch.equal(hT, x["h0"])
    w = small(0, h0=None, seed=13)
    x = make_inputs(w, device="cuda")
    o, hT = run(cuda_lib, x)
    assert torch.count_nonzero(hT) == 0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_split_resume_matches_one_call(cuda_lib, dtype):
    """hT of the first call as h0 of the second equals one call over all tokens."""
    w = small(300, dtype=dtype, seed=14)
    x = make_inputs(w, device="cuda")
    o, hT = run(cuda_lib, x)
    T1 = 128  # a chunk boundary, so both sides round identically
    a = {k_: (v_[:, :T1].contiguous() if k_ in ("q", "k", "v", "g", "beta") else v_)
         for k_, v_ in x.items()}
    oa, ha = run(cuda_lib, a)
    b = {k_: (v_[:, T1:].contiguous() if k_ in ("q", "k", "v", "g", "beta") else v_)
         for k_, v_ in x.items()}
    b["h0"] = ha
    ob, hb = run(cuda_lib, b)
    if dtype == "f32":  # the fp32 state passes from chunk to chunk as from call to call
        assert torch.equal(torch.cat([oa, ob], dim=1), o)
        assert torch.equal(hb, hT)
    else:
        # The bf16 chain reads the state of chunk c through the previous chunk's operands
        # (W'(c) h(c-1) + X(c) V_new(c-1)); a resumed call reads its first chunk's state
        # directly from h0, so the two round differently: the split is checked within the
        # tolerance, against the one call and against the oracle.
        ref_o, ref_h = gdn_recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"])
        split_o = to_np(torch.cat([oa, ob], dim=1))
        assert rel_err(split_o, to_np(o)) < TOL[dtype]
        assert rel_err(to_np(hb), to_np(hT)) < TOL[dtype]
        assert rel_err(split_o, ref_o, out_dtype=dtype) < TOL[dtype]
        assert rel_err(to_np(hb), ref_h) < TOL[dtype]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_pure_decay_when_beta_is_zero(cuda_lib, dtype):
    """beta = 0: o_t = exp(G_t) h0^T (scale q_t) and hT = exp(G_T) h0."""
    w = small(90, dtype=dtype, seed=15)
    x = make_inputs(w, device="cuda")
    x["beta"].zero_()
    o, hT = run(cuda_lib, x)
    G = torch.cumsum(x["g"][0].double(), dim=0)                       # [T, Hv]
    h0 = x["h0"][0].double()                                          # [Hv, dk, dv]
    q = x["q"][0].double()                                            # [T, Hqk, dk]
    want = torch.einsum("thd,hdv->thv", q[:, [0, 0]] * x["scale"], h0) * torch.exp(G)[..., None]
    assert rel_err(to_np(o[0]), want.cpu().numpy(), out_dtype=dtype) < TOL[dtype]
    assert rel_err(to_np(hT[0]), (torch.exp(G[-1])[:, None, None] * h0).cpu().numpy()) < TOL[dtype]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("decay", ["strong", "weak"])
def test_decay_regimes(cuda_lib, dtype, decay):
    g_mu, g_scale = (1.0, 1.0) if decay == "strong" else (0.0, 0.01)
    w = small(260, Hqk=1, Hv=2, dtype=dtype, g_mu=g_mu, g_scale=g_scale, seed=16)
    x = make_inputs(w, device="cuda")
    o, hT = run(cuda_lib, x)
    check_heads(x, o, hT, heads=range(2), dtype=dtype)


@pytest.mark.parametrize("B,T", [(1, 1100), (2, 2053)])
def test_long_rows_with_state(cuda_lib, B, T):
    """Several fixed-length rows of many chunks, a ragged last chunk and a carried h0."""
    w = Workload("case", (T,) * B, 1, 2, 128, 128, 64, "bf16", h0_std=0.1, seed=20 + B)
    x = make_inputs(w, device="cuda")
    o, hT = run(cuda_lib, x)
    check_heads(x, o, hT, heads=range(2), seqs=list(range(B)), dtype="bf16")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_chunk_128_is_the_same_function(cuda_lib, dtype):
    """chunk = 128 runs as two 64-token chunks: bit-identical to chunk = 64, and the
    oracle's own 128-token chunked form agrees with its recurrence."""
    w = small(0, Hqk=1, Hv=2, seqlens=[300, 0, 129], dtype=dtype, seed=19)
    x = make_inputs(w, device="cuda")
    o64, h64 = run(cuda_lib, x, chunk=64)
    o128, h128 = run(cuda_lib, x, chunk=128)
    assert torch.equal(o64, o128) and torch.equal(h64, h128)
    check_heads(x, o128, h128, heads=range(2), dtype=dtype)


def test_unsupported_chunk_is_reported(cuda_lib):
    w = small(64, seed=17)
    x = make_inputs(w, device="cuda")
    with pytest.raises(cuda_lib.GdnError) as e:
        run(cuda_lib, x, chunk=32)
    assert e.value.status == 2


# --------------------------------------------------------------------------
# The named workloads, launched as bench.py launches them
# --------------------------------------------------------------------------
SAMPLES = {
    "tiny_f32": dict(heads=[0, 1]),
    "layer_16h_4k": dict(heads=[0, 7, 15]),
    "gqa_32v_8k_state": dict(heads=[0, 1, 30, 31]),
    "varlen_8seq": dict(heads=[0, 13, 31], seqs=[0, 3, 7]),
    "long_64k_strong": dict(heads=[5]),
    "long_64k_weak": dict(heads=[26]),
}


@pytest.mark.parametrize("name", list(SAMPLES))
def test_workload(cuda_lib, name):
    w = WORKLOADS[name]
    x = make_inputs(w, device="cuda")
    o, hT = run(cuda_lib, x, chunk=w.chunk)
    eo, eh = check_heads(x, o, hT, dtype=w.dtype, **SAMPLES[name])
    print(f"{name}: err_o={eo:.3e} err_h={eh:.3e}")
    # properties that hold at any size: finite everywhere
    assert torch.isfinite(o.float()).all() and torch.isfinite(hT).all()


@pytest.mark.slow
@pytest.mark.parametrize("name", ["layer_16h_4k", "gqa_32v_8k_state"])
def test_workload_every_head(cuda_lib, name):
    """Every v head of the headline layer and of the GQA 8K layer against the oracle, as
    bench.py launches them (no sampling of heads)."""
    w = WORKLOADS[name]
    x = make_inputs(w, device="cuda")
    o, hT = run(cuda_lib, x, chunk=w.chunk)
    check_heads(x, o, hT, heads=range(w.Hv), dtype=w.dtype)


def test_allocating_entry_point_matches_workspace_entry_point(cuda_lib):
    """gdn_chunk_fwd (stream-ordered workspace) == gdn_chunk_fwd_ex, bit for bit."""
    import ctypes
    lib = cuda_lib.load_library()
    w = small(0, Hqk=2, Hv=4, seqlens=[70, 0, 130], seed=18)
    x = make_inputs(w, device="cuda")
    o_ref, h_ref = run(cuda_lib, x)
    o = torch.empty_like(o_ref)
    h = torch.empty_like(h_ref)
    st = torch.cuda.current_stream().cuda_stream
    rc = lib.gdn_chunk_fwd(x["q"].data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(),
                           x["g"].data_ptr(), x["beta"].data_ptr(), x["h0"].data_ptr(),
                           o.data_ptr(), h.data_ptr(), 3, x["q"].shape[1], 2, 4, 128, 128, 64,
                           ctypes.c_float(x["scale"]), x["cu_seqlens"].data_ptr(), st)
    torch.cuda.synchronize()
    assert rc == 0
    assert torch.equal(o, o_ref) and torch.equal(h, h_ref)


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 64)])
def test_many_heads_take_the_32_column_chain_tile(cuda_lib, dk, dv):
    """40 v heads of dv = 64: 160 CTAs of 16 columns would not fit the SMs, so the chain
    runs 32-column tiles (the instantiations the workloads reach only at dk = dv = 128)."""
    w = Workload("case", (150,), 4, 40, dk, dv, 64, "bf16", h0_std=0.1, seed=30 + dk)
    x = make_inputs(w, device="cuda")
    o, hT = run(cuda_lib, x)
    check_heads(x, o, hT, heads=[0, 17, 39], dtype="bf16")


@pytest.mark.parametrize("dtype,tc", [("bf16", False), ("bf16", True), ("f32", None)])
def test_cuda_graph_replay_matches_eager(cuda_lib, dtype, tc):
    """The prep and chain launches (the chain a programmatic dependent of the prep) and
    a decode step captured in one CUDA graph: replaying it gives bit for bit what the
    same calls give eagerly, and the state passes from the forward to the step."""
    lap = cuda_lib
    w = small(200, Hqk=2, Hv=4, dtype=dtype, seed=11)
    x = make_inputs(w, device="cuda")
    kw = {} if tc is None else {"tc_chain": tc}
    tok = {n: x[n][:, 199] for n in ("q", "k", "v", "g", "beta")}

    def calls(o, hT, o1):
        lap.gdn_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], o, hT,
                          chunk=64, scale=w.scale, **kw)
        lap.gdn_recurrent_step(tok["q"], tok["k"], tok["v"], tok["g"], tok["beta"], hT, o1,
                               scale=w.scale)

    o_e, h_e = torch.empty_like(x["v"]), torch.empty_like(x["h0"])
    o1_e = torch.empty_like(tok["v"])
    calls(o_e, h_e, o1_e)
    torch.cuda.synchronize()
    o_g, h_g = torch.empty_like(o_e), torch.empty_like(h_e)
    o1_g = torch.empty_like(o1_e)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        calls(o_g, h_g, o1_g)  # warm-up on the capture stream (workspace pools)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        calls(o_g, h_g, o1_g)
    for _ in range(3):
        o_g.zero_(), h_g.zero_(), o1_g.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o_g, o_e) and torch.equal(h_g, h_e) and torch.equal(o1_g, o1_e)
