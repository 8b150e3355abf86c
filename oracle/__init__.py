"""fp64 CPU oracle for tree-verify MLA attention -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never calls it, and it
shares no code with the library: both read inputs drawn by
``speculative_decode_mla_tree_gb300.workloads`` and nothing else.

Every function restates one step of the verify call the pages describe, in
plain numpy (float64 for all floating point), with the passage it follows in
its docstring. Page titles used in citations:

* "Deploying a Custom sm_120 Verify Kernel into Production: The Validate Gate"
* "The Moment of Truth: Flipping the Switch on a Custom CUDA Verify Kernel"
* "The Pivot to Live Cutover: A Decision Point in Custom CUDA Kernel Integration"

Parity pins (tests/test_oracle.py) tie each function to something other than
itself: brute force, library routines, closed forms, invariants and the
shapes the pages print. No function here is "parity unpinned".
"""
from .tree_verify import (  # noqa: F401
    bf16_bits_to_f64,
    draft_kv_scatter,
    kv_indices_build,
    ancestors_or_self,
    tree_mask_pack,
    tree_mask_pack_bits,
    verify_attention,
    verify_attention_split,
    lse_merge,
    split_bounds,
)
