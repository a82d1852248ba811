"""fp64 CPU oracle for the Gated DeltaNet chunked-prefill forward (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU baseline and
reference arm may import this package.  The product path never does.
"""
from .gdn_oracle import (gdn_dense, gdn_recurrent, gdn_chunked, gdn_step, chains, qk_head,
                         forward_substitution_inverse, recurrent_chain, chunked_chain)

__all__ = ["gdn_dense", "gdn_recurrent", "gdn_chunked", "gdn_step", "chains", "qk_head",
           "forward_substitution_inverse", "recurrent_chain", "chunked_chain"]
