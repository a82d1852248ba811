"""The _ex flags on the GPU: the tensor-memory chain (GDN_FLAG_TC_CHAIN) against the
oracle across shapes, the modulo GQA map, the input check and the fp16 range report."""
import pytest
import torch

from helpers import TOL, check_heads, record, to_np
from linear_attention_prefill_gb300.workloads import WORKLOADS, Workload, make_inputs
from oracle import gdn_recurrent, prologue, ssd_recurrent

pytestmark = pytest.mark.gpu


def run(lap, x, **kw):
    o, h = lap.gdn_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                             cu_seqlens=x["cu_seqlens"], **kw)
    torch.cuda.synchronize()
    return o, h


def clear_status(lap):
    try:
        lap.gdn_device_status()
    except lap.GdnError:
        pass


# ---- the tensor-memory chain ------------------------------------------------
@pytest.mark.parametrize("T", [1, 63, 64, 65, 129, 200])
def test_tc_chain_ragged_lengths(cuda_lib, T):
    w = Workload("tc", (T,), 1, 2, 128, 128, 64, "bf16", h0_std=0.1, seed=100 + T)
    x = make_inputs(w, device="cuda")
    o, hT = run(cuda_lib, x, tc_chain=True)
    check_heads(x, o, hT, heads=range(2), dtype="bf16")


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 64), (64, 128), (128, 128)])
def test_tc_chain_head_dims(cuda_lib, dk, dv):
    w = Workload("tc", (150,), 2, 4, dk, dv, 64, "bf16", h0_std=0.1, seed=dk + dv + 7)
    x = make_inputs(w, device="cuda")
    o, hT = run(cuda_lib, x, tc_chain=True)
    check_heads(x, o, hT, heads=range(4), dtype="bf16")


def test_tc_chain_rows_gqa_and_no_state(cuda_lib):
    w = Workload("tc", (333, 333), 1, 4, 128, 128, 64, "bf16", seed=111)
    x = make_inputs(w, device="cuda")
    assert x["h0"] is None
    o, hT = run(cuda_lib, x, tc_chain=True)
    check_heads(x, o, hT, heads=range(4), seqs=[0, 1], dtype="bf16")


def test_tc_chain_packed_sequences_with_empty_ones(cuda_lib):
    w = Workload("tc", (300, 0, 129, 1, 64), 2, 4, 128, 128, 64, "bf16", h0_std=0.1,
                 varlen=True, seed=112)
    x = make_inputs(w, device="cuda")
    o, hT = run(cuda_lib, x, tc_chain=True)
    check_heads(x, o, hT, heads=range(4), dtype="bf16")
    assert torch.equal(hT[1], x["h0"][1])  # the empty sequence keeps its state


@pytest.mark.parametrize("g_mu,g_scale", [(1.0, 1.0), (0.0, 0.01)])
def test_tc_chain_strong_and_weak_decay(cuda_lib, g_mu, g_scale):
    w = Workload("tc", (700,), 1, 2, 128, 128, 64, "bf16", g_mu=g_mu, g_scale=g_scale,
                 h0_std=0.1, seed=113)
    x = make_inputs(w, device="cuda")
    o, hT = run(cuda_lib, x, tc_chain=True)
    check_heads(x, o, hT, heads=range(2), dtype="bf16")


def test_tc_chain_matches_the_dv_tile_chain(cuda_lib):
    """Both chains compute the same function: within the tolerance of each other."""
    w = Workload("tc", (500,), 2, 4, 128, 128, 64, "bf16", h0_std=0.1, seed=114)
    x = make_inputs(w, device="cuda")
    o1, h1 = run(cuda_lib, x, tc_chain=False)
    o2, h2 = run(cuda_lib, x, tc_chain=True)
    assert record("tc_vs_default", "o", to_np(o2), to_np(o1)) < TOL["bf16"]
    assert record("tc_vs_default", "hT", to_np(h2), to_np(h1)) < TOL["bf16"]


def test_dv_tile_chain_forced_on_many_chains(cuda_lib):
    """256 packed chains pick the tensor-memory chain by themselves; forcing the dv-tile
    chain there gives the same function."""
    w = WORKLOADS["varlen_8seq"]
    assert cuda_lib.chain_kind(w.n_seqs, w.Hv, w.dk, w.dv) == "tc"
    x = make_inputs(w, device="cuda")
    o, hT = run(cuda_lib, x, tc_chain=False)
    check_heads(x, o, hT, [0, 31], "bf16", seqs=[0, 3, 7])


@pytest.mark.parametrize("name,heads", [("layer_16h_4k", [0, 9, 15]),
                                        ("gqa_32v_8k_state", [0, 1, 31]),
                                        ("varlen_8seq", [0, 17, 31])])
def test_tc_chain_workloads(cuda_lib, name, heads):
    w = WORKLOADS[name]
    x = make_inputs(w, device="cuda")
    o, hT = run(cuda_lib, x, tc_chain=True)
    seqs = [0, 4, 7] if w.varlen else None
    check_heads(x, o, hT, heads=heads, seqs=seqs, dtype="bf16")


def test_tc_chain_ssd(cuda_lib):
    w = Workload("tc_ssd", (200,), 1, 4, 128, 64, 64, "bf16", h0_std=0.1, seed=115, op="ssd")
    x = make_inputs(w, device="cuda")
    o, hT = cuda_lib.ssd_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                                   scale=x["scale"], tc_chain=True)
    torch.cuda.synchronize()
    check_heads(x, o, hT, heads=range(4), dtype="bf16", op="ssd")


def test_tc_chain_prologue(cuda_lib):
    w = Workload("tc_pro", (190,), 2, 4, 128, 128, 64, "bf16", h0_std=0.1, seed=116,
                 prologue=True)
    x = make_inputs(w, device="cuda")
    o, hT = cuda_lib.gdn_chunk_fwd_prologue(x["q"], x["k"], x["v"], x["g"], x["beta"], None,
                                            None, x["h0"], tc_chain=True)
    torch.cuda.synchronize()
    qn, kn, g, beta = prologue(x["q"], x["k"], x["g"], x["beta"])
    o_ref, h_ref = gdn_recurrent(qn, kn, x["v"], g, beta, x["scale"], x["h0"])
    assert record("tc_chain_prologue", "o", to_np(o), o_ref, out_dtype="bf16") < TOL["bf16"]
    assert record("tc_chain_prologue", "hT", to_np(hT), h_ref) < TOL["bf16"]


def test_kda_has_no_tc_chain(cuda_lib):
    w = Workload("kda", (64,), 1, 1, 128, 128, 64, "bf16", seed=117, op="kda")
    x = make_inputs(w, device="cuda")
    lib = cuda_lib.load_library()
    need = cuda_lib.kda_chunk_fwd_workspace_size(1, 64, 1, 1, 128, 128)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    o = torch.empty_like(x["v"])
    import ctypes
    rc = lib.kda_chunk_fwd_ex(x["q"].data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(),
                              x["g"].data_ptr(), x["beta"].data_ptr(), None, o.data_ptr(), None,
                              1, 64, 1, 1, 128, 128, 64, ctypes.c_float(x["scale"]), None, 4,
                              ws.data_ptr(), need, None)
    assert rc == 2


# ---- the modulo GQA map -------------------------------------------------------
@pytest.mark.parametrize("tc", [False, True])
def test_modulo_head_map(cuda_lib, tc):
    """v head hv reads q/k head hv % Hqk: matches the oracle's modulo map, and differs from
    the grouped call (with Hqk = 2, Hv = 4 the two maps disagree on heads 1 and 2)."""
    w = Workload("mod", (170,), 2, 4, 128, 128, 64, "bf16", h0_std=0.1, seed=118)
    x = make_inputs(w, device="cuda")
    o, hT = run(cuda_lib, x, head_map="modulo", tc_chain=tc)
    check_heads(x, o, hT, heads=range(4), dtype="bf16", head_map="modulo")
    og, _ = run(cuda_lib, x, tc_chain=tc)
    assert not torch.equal(o[:, :, 1], og[:, :, 1])
    assert torch.equal(o[:, :, 0], og[:, :, 0]) or tc  # head 0 reads q/k head 0 either way


def test_modulo_head_map_decode(cuda_lib):
    w = Workload("mod", (1,), 2, 4, 128, 128, 64, "bf16", h0_std=0.1, seed=119)
    x = make_inputs(w, device="cuda")
    q, k, v, g, beta = (x[n][:, 0].contiguous() for n in ("q", "k", "v", "g", "beta"))
    h = x["h0"].clone()
    o = cuda_lib.gdn_recurrent_step(q, k, v, g, beta, h, head_map="modulo")
    torch.cuda.synchronize()
    from oracle import gdn_step
    o_ref, h_ref = gdn_step(q, k, v, g, beta, x["h0"], x["scale"], head_map="modulo")
    assert record("modulo_decode", "o", to_np(o), o_ref, out_dtype="bf16") < TOL["bf16"]
    assert record("modulo_decode", "hT", to_np(h), h_ref) < TOL["bf16"]


# ---- the input check --------------------------------------------------------------
@pytest.mark.parametrize("tc", [False, True])
def test_input_check_passes_valid_inputs(cuda_lib, tc):
    w = Workload("chk", (300, 0, 129), 1, 2, 128, 128, 64, "bf16", h0_std=0.1, varlen=True,
                 seed=120)
    x = make_inputs(w, device="cuda")
    clear_status(cuda_lib)
    run(cuda_lib, x, check_inputs=True, tc_chain=tc)
    cuda_lib.gdn_device_status()  # raises on any record


@pytest.mark.parametrize("what", ["g_positive", "g_nan", "beta_above_one", "beta_negative",
                                  "cu_end"])
def test_input_check_reports_a_violation(cuda_lib, what):
    """Each violation is recorded and reported by gdn_device_status.  Only values the
    kernels compute through safely are planted (no cu_seqlens that would send a kernel
    out of its buffers): a gate outside its domain, and a cu_seqlens that ends before T."""
    w = Workload("chk", (100, 90), 1, 2, 128, 128, 64, "bf16", varlen=True, seed=121)
    x = make_inputs(w, device="cuda")
    if what == "g_positive":
        x["g"][0, 17, 1] = 0.5
    elif what == "g_nan":
        x["g"][0, 3, 0] = float("nan")
    elif what == "beta_above_one":
        x["beta"][0, 150, 0] = 1.5
    elif what == "beta_negative":
        x["beta"][0, 5, 1] = -0.25
    else:  # the packed sequences cover 180 of the 190 tokens
        x["cu_seqlens"] = torch.tensor([0, 100, 180], dtype=torch.int32, device="cuda")
    clear_status(cuda_lib)
    run(cuda_lib, x, check_inputs=True)
    with pytest.raises(cuda_lib.GdnError) as e:
        cuda_lib.gdn_device_status()
    assert e.value.status == 1 and "input check" in str(e.value)
    cuda_lib.gdn_device_status()  # the record was cleared by the read


def test_input_check_of_the_decode_step(cuda_lib):
    w = Workload("chk", (1,), 1, 2, 128, 128, 64, "bf16", h0_std=0.1, seed=122)
    x = make_inputs(w, device="cuda")
    q, k, v, g, beta = (x[n][:, 0].contiguous() for n in ("q", "k", "v", "g", "beta"))
    h = x["h0"].clone()
    clear_status(cuda_lib)
    cuda_lib.gdn_recurrent_step(q, k, v, g, beta, h, check_inputs=True)
    cuda_lib.gdn_device_status()
    g[0, 1] = 2.0
    cuda_lib.gdn_recurrent_step(q, k, v, g, beta, h, check_inputs=True)
    with pytest.raises(cuda_lib.GdnError):
        cuda_lib.gdn_device_status()


# ---- the fp16 range of the on-chip operands --------------------------------------
@pytest.mark.parametrize("tc", [False, True])
def test_fp16_operand_range_is_reported(cuda_lib, tc):
    """|v| beyond fp16's range makes U and V_new overflow their fp16 copies: the call
    completes and gdn_device_status reports it (GDN_ERR_INVALID_ARG)."""
    w = Workload("rng", (130,), 1, 2, 128, 128, 64, "bf16", seed=123)
    x = make_inputs(w, device="cuda")
    clear_status(cuda_lib)
    run(cuda_lib, x, tc_chain=tc)
    cuda_lib.gdn_device_status()  # in range: nothing recorded
    x["v"] = (x["v"].float() * 3e5).to(torch.bfloat16)
    run(cuda_lib, x, tc_chain=tc)
    with pytest.raises(cuda_lib.GdnError) as e:
        cuda_lib.gdn_device_status()
    assert e.value.status == 1 and "fp16" in str(e.value)
