"""gdn_chunk_fwd_noalloc: the forward for callers that may not allocate device memory.

Some callers cannot call cudaMalloc: a serving loop that must not take an
allocator's locks or risk the device synchronisation an allocation can bring,
or code living inside a runtime that hands out all device memory from its own
pool.  For them the library carries a fixed 32 MiB workspace in static device
memory.  This file is collected last on purpose (a run that stops at the first
failure has run everything else first); it also passes alone in a fresh process.
"""
import ctypes

import pytest
import torch

from linear_attention_prefill_gb300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu


def _noalloc(lib, x, o, hT, N):
    q = x["q"]
    cu = x["cu_seqlens"]
    return lib.gdn_chunk_fwd_noalloc(
        q.data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(), x["g"].data_ptr(),
        x["beta"].data_ptr(), None if x["h0"] is None else x["h0"].data_ptr(), o.data_ptr(),
        hT.data_ptr(), N, q.shape[1], q.shape[2], x["v"].shape[2], q.shape[3], x["v"].shape[3],
        64, ctypes.c_float(x["scale"]), None if cu is None else cu.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("w", [
    Workload("fixed", (1000,), 2, 4, 128, 128, 64, "bf16", h0_std=0.1, seed=41),
    Workload("packed", (300, 0, 650), 2, 4, 128, 128, 64, "bf16", h0_std=0.1, varlen=True, seed=42),
], ids=["fixed", "packed"])
def test_noalloc_matches_workspace_entry_point_twice(cuda_lib, w):
    lib = cuda_lib.load_library()
    for call in range(2):  # two calls in a row share the built-in workspace
        x = make_inputs(w, device="cuda", seed=w.seed + call)
        o_ref, h_ref = cuda_lib.gdn_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                                              cu_seqlens=x["cu_seqlens"])
        o = torch.empty_like(o_ref)
        hT = torch.empty_like(h_ref)
        rc = _noalloc(lib, x, o, hT, w.n_seqs)
        torch.cuda.synchronize()
        assert rc == 0, lib.gdn_last_error()
        # the same kernels on the same inputs: bit for bit
        assert torch.equal(o, o_ref) and torch.equal(hT, h_ref)


def test_noalloc_rejects_sizes_beyond_its_workspace(cuda_lib):
    lib = cuda_lib.load_library()
    w = Workload("big", (4096,), 16, 16, 128, 128, 64, "bf16", seed=43)
    assert cuda_lib.gdn_chunk_fwd_workspace_size(1, 4096, 16, 16, 128, 128) > 32 << 20
    x = make_inputs(w, device="cuda")
    o = torch.empty_like(x["v"])
    hT = torch.empty((1, 16, 128, 128), dtype=torch.float32, device="cuda")
    assert _noalloc(lib, x, o, hT, 1) == 1
    assert b"built-in workspace" in lib.gdn_last_error()
