"""CPU oracle for exact scaled-dot-product attention forward (fp64).

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it. It shares
no code with the CUDA library in ``attention_fa2_attn_gb300/`` and imports
nothing from it.

Every function here is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle_pins.py`` against numbers the source pages print, closed
forms, or an independent brute force. No function is "parity unpinned".
"""

from .attention import (  # noqa: F401
    NEG_INF,
    attention_backward,
    attention_backward_rows,
    attention_online,
    attention_online_normalized,
    attention_partials,
    attention_rows,
    attention_three_pass,
    backward_rowsum,
    causal_mask,
    decode_paged,
    kv_head_of,
    lse_merge,
    paged_gather,
    split_ranges,
    visible,
)
