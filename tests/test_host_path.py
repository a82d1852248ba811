"""The host-memory entry points: gdn_chunk_fwd_host and the two-stream HostPipeline give
the same o and hT as the device call, bit for bit, for several in-flight calls."""
import pytest
import torch

from linear_attention_prefill_gb300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu


def host_copy(x):
    return {k: (None if x[k] is None else x[k].detach().cpu().pin_memory())
            for k in ("q", "k", "v", "g", "beta", "h0", "cu_seqlens")}


@pytest.mark.parametrize("op", ["gdn", "ssd"])
def test_host_pipeline_matches_device_calls(cuda_lib, op):
    fwd = cuda_lib.gdn_chunk_fwd if op == "gdn" else cuda_lib.ssd_chunk_fwd
    pipe = cuda_lib.HostPipeline(chunk=64, device="cuda", op=op, depth=2)
    cases = []
    for seed in range(3):  # three calls in flight over two streams, different inputs
        w = Workload("case", (100, 0, 70), 1, 2, 128, 64, 64, "bf16", h0_std=0.1, varlen=True,
                     seed=70 + seed)
        x = make_inputs(w, device="cuda")
        scale = 128 ** -0.5 if op == "gdn" else 1.0
        o, hT = fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], cu_seqlens=x["cu_seqlens"],
                    scale=scale)
        cases.append((o.cpu(), hT.cpu(), pipe.submit(host_copy(x))))
    for i, (o_ref, h_ref, (o_h, hT_h, done, bi, bo)) in enumerate(cases):
        done.synchronize()
        if i < len(cases) - len(pipe.slots):
            continue  # this slot's pinned outputs were reused by a later call
        assert torch.equal(o_h, o_ref) and torch.equal(hT_h, h_ref)
        assert bi > 0 and bo == o_h.numel() * o_h.element_size() + hT_h.numel() * 4


def test_host_call_matches_device_call(cuda_lib):
    w = Workload("case", (150,), 1, 2, 128, 128, 64, "bf16", h0_std=0.1, seed=73)
    x = make_inputs(w, device="cuda")
    o, hT = cuda_lib.gdn_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    o_h, hT_h, bi, bo = cuda_lib.gdn_chunk_fwd_host(host_copy(x), chunk=64, device="cuda")
    torch.cuda.synchronize()
    assert torch.equal(o_h, o.cpu()) and torch.equal(hT_h, hT.cpu())
