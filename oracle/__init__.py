"""fp64 CPU oracle for packed, document-masked, chunked causal attention.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package; the product path never
does.  It shares no code with the CUDA library.

The arithmetic lives in ``hdp_oracle.c`` (plain loops, fp64); this module only
builds it with gcc and marshals numpy arrays through ctypes.

Parity pins (see ``tests/test_oracle_pins.py``): every function here is pinned
against brute force, closed forms, invariants or the worked example of
Figure 2(b) in the ByteScale research digest; none is "parity unpinned".
"""
from .oracle import (  # noqa: F401
    build,
    plan,
    plan_sizes,
    attention,
    attention_rows,
    attention_f64,
    attention_bwd,
    attention_bwd_dq_rows,
    attention_bwd_dkv_rows,
    attention_bwd_dkv_doc,
    bf16_bits_to_f64,
    merge,
    flops_total,
    flops_per_shard,
    tile_worklist,
    library_path,
    num_threads,
)
