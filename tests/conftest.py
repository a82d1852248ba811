import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libgdn.so")
    config.addinivalue_line("markers", "slow: long-running case")


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA binding, on a machine with a GPU; skips elsewhere."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_attention_prefill_gb300 as lap
    return lap


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Every parity comparison of the run: raw max-abs/RMS, the error after the bf16
    storage allowance (the one the tolerance applies to) and the NMSE."""
    try:
        from helpers import RECORDS
    except ImportError:
        return
    if not RECORDS:
        return
    tr = terminalreporter
    tr.section("parity against the fp64 oracle")
    tr.write_line(f"{'test':58s} {'qty':3s} {'raw maxabs/RMS':>14s} {'adjusted':>10s} {'NMSE':>10s}")
    for name, qty, raw, adj, e in RECORDS:
        tr.write_line(f"{name[:58]:58s} {qty:3s} {raw:14.3e} {adj:10.3e} {e:10.3e}")
    worst = {}
    for name, qty, raw, adj, e in RECORDS:
        w = worst.setdefault(qty, [0.0, 0.0, 0.0])
        w[0], w[1], w[2] = max(w[0], raw), max(w[1], adj), max(w[2], e)
    for qty, (raw, adj, e) in worst.items():
        tr.write_line(f"worst {qty}: raw {raw:.3e}, adjusted {adj:.3e}, NMSE {e:.3e} "
                      f"over {sum(1 for r in RECORDS if r[1] == qty)} comparisons")
