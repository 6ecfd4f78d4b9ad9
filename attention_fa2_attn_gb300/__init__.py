"""GB300 (sm_103a) fused attention forward: prefill, split-KV decode, paged decode.

The computation runs in the CUDA library ``libfa_gb300.so`` (C ABI in
``include/fa_gb300.h``); ``api`` holds thin PyTorch-facing wrappers with the
same names, ``costmodel`` the FLOP and byte accounting used for rooflines.
"""

from .api import (  # noqa: F401
    FAError,
    fa_bwd,
    fa_bwd_workspace_bytes,
    fa_decode_num_splits,
    fa_decode_paged,
    fa_decode_splitkv,
    fa_decode_splitkv_static,
    fa_decode_workspace_bytes,
    fa_fwd,
    fa_fwd_f32,
    fa_fwd_kv_outer,
    fa_fwd_kv_outer_workspace_bytes,
    fa_get_last_device_error,
    fa_get_wait_timeouts,
    fa_lse_merge,
    fa_num_splits_heuristic,
    fa_num_splits_prefill,
    fa_selftest_wait_timeout,
    fa_set_wait_timeout_ns,
)
