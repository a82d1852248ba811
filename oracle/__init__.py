"""fp64 CPU oracle for the Gated DeltaNet chunked-prefill forward, the Mamba-2
SSD scan and Kimi Delta Attention (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU baseline and
reference arm may import this package.  The product path never does.
"""
from .gdn_oracle import (gdn_dense, gdn_recurrent, gdn_chunked, gdn_step, chains, qk_head,
                         forward_substitution_inverse, recurrent_chain, chunked_chain,
                         prologue)
from .ssd_oracle import (ssd_recurrent, ssd_unrolled, ssd_chunked, ssd_step,
                         ssd_recurrent_chain)
from .kda_oracle import kda_recurrent, kda_transitions, kda_chunked, kda_step

__all__ = ["gdn_dense", "gdn_recurrent", "gdn_chunked", "gdn_step", "chains", "qk_head",
           "forward_substitution_inverse", "recurrent_chain", "chunked_chain", "prologue",
           "ssd_recurrent", "ssd_unrolled", "ssd_chunked", "ssd_step", "ssd_recurrent_chain",
           "kda_recurrent", "kda_transitions", "kda_chunked", "kda_step"]
