"""The allocation-free split-KV decode entry point, fa_decode_splitkv_static.

It exists for callers that cannot allocate device memory around the call
(graph capture, engines that own all device memory, latency-critical loops):
its split partials live in a fixed array inside the library instead of a
caller workspace. Called here through the C ABI on two calls in a row -- the
second with other shapes and split counts, so leftovers of the first call in
the shared array would show. Each call must give the same bits as the
workspace entry point, fa_decode_splitkv (the same kernels with the same split
count), and both must match the fp64 oracle. This file is collected last on
purpose.
"""

import ctypes
import math

import pytest
import torch

import fa_inputs as fi
import oracle
from parity import compare

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _call_static(L, q, k, v, causal, n, scale):
    B, Hq, T, d = q.shape
    Hkv, S = k.shape[1], k.shape[2]
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, T), dtype=torch.float32, device=q.device)
    st = L.fa_decode_splitkv_static(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
        ctypes.c_void_p(o.data_ptr()), ctypes.c_void_p(lse.data_ptr()), B, Hq, Hkv, T, S, d, scale, int(causal), n,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, o, lse


def test_static_scratch_matches_workspace_entry_point_twice():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import attention_fa2_attn_gb300 as fa
    from attention_fa2_attn_gb300 import _lib

    L = _lib.lib()
    w = fi.SPLITKV_DECODE
    problems = [
        (w.B, w.Hq, w.Hkv, w.T, w.S, w.d, True, w.num_splits, w.index),  # the split-KV workload, 16 splits
        (2, 16, 4, 2, 5000, 64, True, 7, 95),  # other shapes and split count
    ]
    for call, (B, Hq, Hkv, T, S, d, causal, n, index) in enumerate(problems):
        qc, kc, vc = fi.qkv(B, Hq, Hkv, T, S, d, index)
        q, k, v = qc.to(DEV), kc.to(DEV), vc.to(DEV)
        scale = 1.0 / math.sqrt(d)
        o_ws, l_ws = fa.fa_decode_splitkv(q, k, v, causal=causal, num_splits=n, scale=scale)
        st, o, l = _call_static(L, q, k, v, causal, n, scale)
        assert st == 0, L.fa_status_string(st)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ws) and torch.equal(l, l_ws), f"call {call}: not bit-identical to fa_decode_splitkv"
        o_ref, l_ref = oracle.attention_three_pass(qc, kc, vc, scale, causal)
        compare(o, l, o_ref, l_ref, what=f"call {call}")
    assert fa.fa_get_last_device_error()[0] == 0
    # partials that would not fit the fixed array are refused up front
    q, k, v = (x.to(DEV) for x in fi.qkv(64, 64, 8, 1, 256, 128, 96))
    st, _, _ = _call_static(L, q, k, v, True, 4, 0.1)
    assert st == 2  # FA_ERR_UNSUPPORTED
