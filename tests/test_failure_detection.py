"""Failure detection without a GPU fault: a bounded device-side wait that runs out is
reported to the host as GDN_ERR_TIMEOUT through gdn_device_status, and the CUDA context
stays usable afterwards.  The wait is made to expire on purpose (an mbarrier that nothing
completes, a limit of ~2^20 cycles); nothing traps, faults or hangs."""
import pytest
import torch

from helpers import check_heads
from linear_attention_prefill_gb300.workloads import Workload, make_inputs


@pytest.mark.gpu
def test_expired_wait_is_reported_and_the_context_survives(cuda_lib):
    cuda_lib.gdn_device_status()  # start from a clean error word
    cuda_lib.gdn_selftest_expired_wait(1 << 20)
    with pytest.raises(cuda_lib.GdnError) as e:
        cuda_lib.gdn_device_status()
    assert e.value.status == 4  # GDN_ERR_TIMEOUT
    cuda_lib.gdn_device_status()  # the word was read and cleared
    # the context still runs the forward correctly
    w = Workload("case", (130,), 1, 2, 128, 128, 64, "bf16", h0_std=0.1, seed=50)
    x = make_inputs(w, device="cuda")
    o, hT = cuda_lib.gdn_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    torch.cuda.synchronize()
    check_heads(x, o, hT, heads=range(2), dtype="bf16")
    cuda_lib.gdn_device_status()  # and no wait of the forward expired


def test_selftest_rejects_a_bad_limit_without_a_device():
    from linear_attention_prefill_gb300 import _build, binding
    _build.build()
    lib = binding.load_library()
    assert lib.gdn_selftest_expired_wait(-1, None) == 1
    assert lib.gdn_selftest_expired_wait(1 << 40, None) == 1
