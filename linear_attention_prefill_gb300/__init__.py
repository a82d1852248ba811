"""GB300-native Gated DeltaNet chunked-prefill forward (sm_103a CUDA behind a C ABI).

The compute lives in libgdn.so (``csrc/``, C ABI in ``include/gdn.h``); this
package holds the Python binding with the ABI's names, the seeded synthetic
workloads and the algorithmic byte/FLOP model.  The same kernels also run the
Mamba-2 SSD scan (the recurrence without the delta rule's erase term), and Kimi
Delta Attention (the delta rule with a per-key-channel gate) shares the chain.
"""
from .binding import (GdnError, HostPipeline, chain_kind, gdn_chunk_fwd, gdn_chunk_fwd_host, gdn_chunk_fwd_prologue,
                      gdn_chunk_fwd_workspace_size, gdn_recurrent_step_prologue,
                      gdn_device_status, gdn_recurrent_step, gdn_selftest_expired_wait,
                      kda_chunk_fwd, kda_chunk_fwd_workspace_size, kda_recurrent_step,
                      load_library, ssd_chunk_fwd, ssd_recurrent_step, status_string)

__all__ = ["GdnError", "HostPipeline", "chain_kind", "gdn_chunk_fwd", "gdn_chunk_fwd_host", "gdn_chunk_fwd_prologue",
           "gdn_chunk_fwd_workspace_size", "gdn_recurrent_step_prologue",
           "gdn_device_status", "gdn_recurrent_step", "gdn_selftest_expired_wait", "load_library",
           "kda_chunk_fwd", "kda_chunk_fwd_workspace_size", "kda_recurrent_step",
           "ssd_chunk_fwd", "ssd_recurrent_step", "status_string"]
