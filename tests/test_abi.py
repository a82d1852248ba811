"""The C ABI on the CPU: the library loads, exports every declared symbol, and
rejects bad arguments before touching CUDA (no compute call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")


@pytest.fixture(scope="module")
def lib():
    from linear_attention_prefill_gb300 import _build, binding
    _build.build()
    return binding.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*((?:gdn|ssd|kda)_\w+)\s*\(", text,
                                 flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("gdn_chunk_fwd", "gdn_chunk_fwd_f32", "gdn_recurrent_step",
                 "gdn_recurrent_step_f32", "gdn_status_string", "gdn_last_error",
                 "gdn_device_status", "gdn_abi_version", "ssd_chunk_fwd", "ssd_chunk_fwd_ex",
                 "ssd_chunk_fwd_f32", "ssd_recurrent_step", "ssd_recurrent_step_f32",
                 "gdn_chunk_fwd_prologue", "gdn_chunk_fwd_prologue_ex",
                 "gdn_recurrent_step_prologue", "gdn_selftest_expired_wait", "kda_chunk_fwd",
                 "kda_chunk_fwd_ex", "kda_chunk_fwd_workspace_size", "kda_recurrent_step",
                 "gdn_chunk_fwd_chain_kind"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    from linear_attention_prefill_gb300.binding import SIGNATURES
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in SIGNATURES, f"binding lacks a signature for {name}"


def test_abi_version_and_status_strings(lib):
    assert lib.gdn_abi_version() == 2
    assert lib.gdn_status_string(0) == b"GDN_OK"
    assert lib.gdn_status_string(1) == b"GDN_ERR_INVALID_ARG"
    assert lib.gdn_status_string(2) == b"GDN_ERR_UNSUPPORTED"
    assert lib.gdn_status_string(3) == b"GDN_ERR_CUDA"
    assert lib.gdn_status_string(4) == b"GDN_ERR_TIMEOUT"


A = 0x10000  # an aligned fake address: never dereferenced, validation fails first


def fwd(lib, q=A, k=A, v=A, g=A, beta=A, h0=None, o=A, hT=None, B=1, T=128, Hqk=1, Hv=2,
        dk=128, dv=128, chunk=64, scale=0.088, cu=None, f32=False, op="gdn"):
    fn = getattr(lib, f"{op}_chunk_fwd" + ("_f32" if f32 else ""))
    return fn(q, k, v, g, beta, h0, o, hT, B, T, Hqk, Hv, dk, dv, chunk, scale, cu, None)


@pytest.mark.parametrize("op", ["gdn", "ssd"])
@pytest.mark.parametrize("f32", [False, True])
@pytest.mark.parametrize("case,status", [
    (dict(q=None), 1), (dict(k=None), 1), (dict(v=None), 1), (dict(g=None), 1),
    (dict(beta=None), 1), (dict(o=None), 1),
    (dict(B=-1), 1), (dict(T=-5), 1), (dict(Hqk=0), 1), (dict(Hv=0), 1),
    (dict(Hqk=3, Hv=4), 1),
    (dict(dk=96), 2), (dict(dv=32), 2), (dict(dk=256), 2), (dict(chunk=32), 2),
    (dict(chunk=100), 2),
    (dict(q=A + 8), 1), (dict(o=A + 2), 1), (dict(g=A + 2), 1), (dict(h0=A + 4), 1),
    (dict(hT=A + 8), 1), (dict(cu=A + 2), 1),
    (dict(scale=float("nan")), 1),
    (dict(T=1 << 30, B=4096), 1),
    (dict(cu=A, B=0), 1),
])
def test_forward_rejects_bad_arguments(lib, case, status, f32, op):
    assert fwd(lib, f32=f32, op=op, **case) == status
    assert lib.gdn_last_error() != b""


def step(lib, q=A, k=A, v=A, g=A, beta=A, h=A, o=A, N=2, Hqk=1, Hv=2, dk=128, dv=128,
         scale=0.088, f32=False, op="gdn"):
    fn = getattr(lib, f"{op}_recurrent_step" + ("_f32" if f32 else ""))
    return fn(q, k, v, g, beta, h, o, N, Hqk, Hv, dk, dv, scale, None)


@pytest.mark.parametrize("op", ["gdn", "ssd"])
@pytest.mark.parametrize("f32", [False, True])
@pytest.mark.parametrize("case,status", [
    (dict(q=None), 1), (dict(h=None), 1), (dict(o=None), 1), (dict(N=-1), 1),
    (dict(Hqk=2, Hv=3), 1), (dict(dk=80), 2), (dict(dv=256), 2), (dict(h=A + 4), 1),
    (dict(scale=float("nan")), 1),
])
def test_step_rejects_bad_arguments(lib, case, status, f32, op):
    assert step(lib, f32=f32, op=op, **case) == status


def test_no_op_calls_return_ok_without_a_device(lib):
    # B = 0 sequences and N = 0 decode rows enqueue nothing
    assert fwd(lib, B=0, T=0, q=None, k=None, v=None, g=None, beta=None, o=None) == 0
    assert step(lib, N=0, q=None, k=None, v=None, g=None, beta=None, h=None, o=None) == 0


def test_binding_raises_without_the_library(tmp_path):
    from linear_attention_prefill_gb300 import binding
    saved = binding._lib
    binding._lib = None
    try:
        with pytest.raises(RuntimeError, match="libgdn.so not found"):
            binding.load_library(str(tmp_path / "missing.so"))
    finally:
        binding._lib = saved


def test_binding_signatures_cover_the_header():
    from linear_attention_prefill_gb300.binding import SIGNATURES
    assert sorted(SIGNATURES) == declared_functions()


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "linear_attention_prefill_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f


def test_workspace_size_formula(lib):
    # gated delta rule record: W' [64][dk], X^T [64][64], U^T [dv][64] (fp16), 132 fp32 gate
    # factors, then (on a 128-byte line) Q~ [64][dk], Kt [64][dk], P^T [64][64] (fp16),
    # padded to a 128-byte multiple
    def rec(dk, dv):
        gv_end = 64 * dk * 2 + 64 * 64 * 2 + 64 * dv * 2 + 132 * 4
        qt = (gv_end + 127) // 128 * 128
        return (qt + 2 * 64 * dk * 2 + 64 * 64 * 2 + 127) // 128 * 128
    # fixed-length rows: N * ceil(T/64) chunk slots, x Hv
    assert lib.gdn_chunk_fwd_workspace_size(1, 4096, 16, 16, 128, 128, 64, 0) == 64 * 16 * rec(128, 128)
    assert lib.gdn_chunk_fwd_workspace_size(2, 100, 1, 4, 128, 64, 64, 0) == 2 * 2 * 4 * rec(128, 64)
    # packed rows: floor(T/64) + N + 1 chunk slots
    assert lib.gdn_chunk_fwd_workspace_size(8, 9849, 16, 32, 128, 128, 64, 1) == \
        (9849 // 64 + 9) * 32 * rec(128, 128)
    # Kimi Delta Attention record: W^T [dk][64], Kt [64][dk], P [64][64], U^T [dv][64], gates,
    # then Q~ [64][dk] on a 128-byte line
    kda = (2 * 64 * 128 * 2 + 64 * 64 * 2 + 64 * 128 * 2 + 132 * 4 + 127) // 128 * 128 + 64 * 128 * 2
    assert lib.kda_chunk_fwd_workspace_size(1, 4096, 16, 16, 128, 128, 64, 0) == 64 * 16 * kda
    # rejected sizes give 0
    assert lib.gdn_chunk_fwd_workspace_size(1, 64, 3, 4, 128, 128, 64, 0) == 0
    assert lib.gdn_chunk_fwd_workspace_size(1, 64, 1, 1, 96, 128, 64, 0) == 0


def test_ex_rejects_small_or_misaligned_workspace(lib):
    need = lib.gdn_chunk_fwd_workspace_size(1, 128, 1, 2, 128, 128, 64, 0)
    args = (A, A, A, A, A, None, A, None, 1, 128, 1, 2, 128, 128, 64, 0.088, None)
    # the size function covers every flag; a call checks what its own records need
    for flags in (0, 1, 2, 4, 7, 8, 11):
        assert lib.gdn_chunk_fwd_ex(*args, flags, None, need, None) == 1
        assert lib.gdn_chunk_fwd_ex(*args, flags, A, need // 2, None) == 1
        assert lib.gdn_chunk_fwd_ex(*args, flags, A + 16, need, None) == 1
        assert b"workspace" in lib.gdn_last_error()
    assert lib.gdn_chunk_fwd_ex(*args, 4, A, need - 1, None) == 1  # the larger records


def test_ex_rejects_unknown_flags(lib):
    need = lib.gdn_chunk_fwd_workspace_size(1, 128, 1, 2, 128, 128, 64, 0)
    args = (A, A, A, A, A, None, A, None, 1, 128, 1, 2, 128, 128, 64, 0.088, None)
    assert lib.gdn_chunk_fwd_ex(*args, 16, A, need, None) == 1
    assert b"flag" in lib.gdn_last_error()
    # the two chain flags exclude each other
    assert lib.gdn_chunk_fwd_ex(*args, 12, A, need, None) == 1
    assert b"together" in lib.gdn_last_error()
    # the decode step takes the head map and the input check, not the chain choice
    sargs = (A, A, A, A, A, A, A, 1, 1, 2, 128, 128, 0.088)
    assert lib.gdn_recurrent_step_ex(*sargs, 4, None) == 1
    assert lib.gdn_recurrent_step_ex(*sargs, 16, None) == 1
    assert lib.gdn_recurrent_step_ex(A, A, A, A, A, None, A, 1, 1, 2, 128, 128, 0.088, 1,
                                     None) == 1  # NULL state: the step's own checks run
    # KDA has no tensor-memory chain
    kargs = (A, A, A, A, A, None, A, None, 1, 128, 1, 2, 128, 128, 64, 0.088, None)
    kneed = lib.kda_chunk_fwd_workspace_size(1, 128, 1, 2, 128, 128, 64, 0)
    assert lib.kda_chunk_fwd_ex(*kargs, 4, A, kneed, None) == 2
    assert lib.ssd_chunk_fwd_ex(*kargs, 16, A, need, None) == 1


def test_chain_kind(lib):
    """The chain choice: forced by a flag, else the dv-tile chain while its CTAs fit in few
    waves over the 152 SMs and the tensor-memory chain once they do not; never for KDA."""
    kind = lib.gdn_chunk_fwd_chain_kind
    assert kind(1, 16, 128, 128, 1, 0) == 0      # 16 chains
    assert kind(1, 32, 128, 128, 1, 0) == 0      # 32 chains
    assert kind(8, 32, 128, 128, 1, 0) == 1      # 256 chains
    assert kind(1, 16, 128, 128, 1, 4) == 1      # forced
    assert kind(8, 32, 128, 128, 1, 8) == 0      # forced
    assert kind(1, 16, 128, 128, 1, 12) == -1    # both
    assert kind(1, 16, 128, 128, 1, 16) == -1    # unknown bit
    assert kind(1, 16, 96, 128, 1, 0) == -1      # unsupported head dim
    import linear_attention_prefill_gb300 as lap
    assert lap.chain_kind(8, 32, 128, 128, "kda") == "dv_tile"
    assert lap.chain_kind(8, 32, 128, 128) == "tc"
    assert lap.chain_kind(8, 32, 128, 128, tc_chain=False) == "dv_tile"


@pytest.mark.parametrize("case,status", [
    (dict(q=None), 1), (dict(g=None), 1), (dict(Hqk=3, Hv=4), 1), (dict(dv=32), 2),
    (dict(dk=64), 2), (dict(chunk=32), 2), (dict(g=A + 4), 1), (dict(q=A + 8), 1),
    (dict(scale=float("nan")), 1),
])
def test_kda_forward_rejects_bad_arguments(lib, case, status):
    """KDA adds dk = 128 only and a 16-byte aligned per-channel gate to the forward's checks."""
    assert fwd(lib, op="kda", **case) == status
    assert lib.gdn_last_error() != b""


def test_kda_step_rejects_bad_arguments(lib):
    assert step(lib, op="kda", h=None) == 1
    assert step(lib, op="kda", dk=80) == 2
    assert step(lib, op="kda", N=0, q=None, k=None, v=None, g=None, beta=None, h=None,
                o=None) == 0


def test_kda_workspace_size_formula(lib):
    # the GDN chunk record, then the fp16 Qt tile [64][dk] on a 128-byte line
    def rec(dk, dv):
        gv_end = 2 * 64 * dk * 2 + 64 * 64 * 2 + 64 * dv * 2 + 132 * 4
        qt_off = (gv_end + 127) // 128 * 128
        return (qt_off + 64 * dk * 2 + 127) // 128 * 128
    assert lib.kda_chunk_fwd_workspace_size(1, 4096, 16, 16, 128, 128, 64, 0) == \
        64 * 16 * rec(128, 128)
    assert lib.kda_chunk_fwd_workspace_size(8, 9849, 16, 32, 128, 64, 64, 1) == \
        (9849 // 64 + 9) * 32 * rec(128, 64)
    assert lib.kda_chunk_fwd_workspace_size(1, 64, 1, 1, 64, 128, 64, 0) == 0
