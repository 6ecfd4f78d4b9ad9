"""The C-ABI library builds, loads and exports every declared symbol; host-side
checks reject bad arguments before anything is launched (CPU only: no call
here reaches a CUDA API)."""

import ctypes
import json
import os

import pytest

from attention_fa2_attn_gb300 import _lib

G = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_worked_examples.json")))
P = ctypes.c_void_p(256)  # a fake, aligned, non-null "device pointer": never dereferenced here
MIS = ctypes.c_void_p(258)  # misaligned


@pytest.fixture(scope="module")
def L():
    return _lib.lib(build_if_missing=True)


def test_exports_every_header_symbol(L):
    names = _lib.header_symbols()
    assert len(names) >= 13
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(_lib.SIGNATURES), "binding and header disagree"


def test_version_and_strings(L):
    assert L.fa_version() >= 100
    assert L.fa_status_string(_lib.FA_ERR_TIMEOUT) == b"FA_ERR_TIMEOUT"
    assert L.fa_status_string(99) == b"FA_ERR_UNKNOWN"


def test_split_heuristic_page_example(L):
    g = G["split_count"]
    n = L.fa_num_splits_heuristic(g["batch"], g["kv_heads"], g["context"], g["num_sms"])
    assert n == g["splits"]
    assert g["context"] // n == g["keys_per_split"]
    assert n * g["kv_heads"] == g["split_blocks"]
    assert abs(g["split_blocks"] / g["num_sms"] - g["waves"]) < g["tol"]
    assert abs(g["unsplit_blocks"] / g["num_sms"] - g["unsplit_sm_fraction"]) < g["tol"]
    # no split once batch x KV heads fills the GPU ("not worth it at high batch")
    assert L.fa_num_splits_heuristic(64, 8, 8192, 132) == 1
    assert L.fa_num_splits_heuristic(16, 8, 8192, 132) == 1
    # GB300: 152 SMs
    assert L.fa_num_splits_heuristic(1, 8, 131072, 152) == 19
    # never fewer than 256 keys per split
    assert L.fa_num_splits_heuristic(1, 1, 1000, 152) == 4
    assert L.fa_num_splits_heuristic(0, 8, 100, 152) == 1


def test_prefill_split_heuristic(L):
    # one head of 8192 positions, d any: 64 query tiles -> 32 pairs; 152 SMs -> 4 ranges
    assert L.fa_num_splits_prefill(1, 1, 1, 8192, 8192, 152) == 4
    # one head of 4096: 16 pairs -> 9 ranges (ceil(4096 / 512) = 8 caps it)
    assert L.fa_num_splits_prefill(1, 1, 1, 4096, 4096, 152) == 8
    # the prefill workload already fills the GPU: 4 x 16 heads x 16 pairs
    assert L.fa_num_splits_prefill(4, 16, 16, 4096, 4096, 152) == 1
    # GQA: 8 query heads per KV head stack 16 positions per 128-row tile
    assert L.fa_num_splits_prefill(1, 8, 1, 1024, 65536, 152) == 4  # 64 tiles -> 32 pairs
    assert L.fa_num_splits_prefill(1, 6, 4, 100, 100, 152) == 1  # Hq not a multiple of Hkv
    assert L.fa_num_splits_prefill(1, 1, 1, 128, 100000, 152) == 64  # one pair: capped at 64


def test_workspace_bytes(L):
    assert L.fa_decode_workspace_bytes(1, 32, 1, 128, 1) == 0
    n, rows, d = 16, 32, 128
    ob = ((n * rows * d * 4 + 255) // 256) * 256
    assert L.fa_decode_workspace_bytes(1, 32, 1, 128, 16) == ob + n * rows * 4


def _fwd(L, *, q=P, k=P, v=P, o=P, lse=None, B=1, Hq=2, Hkv=2, T=8, S=8, d=128, scale=0.125, causal=0):
    return L.fa_fwd(q, k, v, o, lse, B, Hq, Hkv, T, S, d, scale, causal, None)


def test_fwd_rejects_bad_arguments(L):
    assert _fwd(L, q=None) == _lib.FA_ERR_INVALID_ARG
    assert _fwd(L, k=MIS) == _lib.FA_ERR_INVALID_ARG
    assert _fwd(L, Hq=3, Hkv=2) == _lib.FA_ERR_INVALID_ARG
    assert _fwd(L, T=0) == _lib.FA_ERR_INVALID_ARG
    assert _fwd(L, S=0) == _lib.FA_ERR_INVALID_ARG
    assert _fwd(L, scale=0.0) == _lib.FA_ERR_INVALID_ARG
    assert _fwd(L, scale=float("nan")) == _lib.FA_ERR_INVALID_ARG
    assert _fwd(L, d=96) == _lib.FA_ERR_UNSUPPORTED
    assert _fwd(L, Hq=6, Hkv=2) == _lib.FA_ERR_UNSUPPORTED  # group of 3
    assert _fwd(L, Hq=32, Hkv=1) == _lib.FA_ERR_UNSUPPORTED  # group of 32
    assert L.fa_fwd_f32(P, P, P, P, None, 1, 1, 1, 4, 4, 200, 0.1, 0, None) == _lib.FA_ERR_UNSUPPORTED


def test_decode_rejects_bad_arguments(L):
    # more than 16 stacked rows (group 8 x T 3 = 24) run on the prefill kernel: its key
    # split needs the workspace like decode's, and it takes only groups of 1, 2, 4, 8, 16
    assert L.fa_decode_splitkv(P, P, P, P, None, 1, 8, 1, 3, 100, 128, 0.1, 1, 2, None, 0, None) == _lib.FA_ERR_INVALID_ARG
    assert L.fa_decode_splitkv(P, P, P, P, None, 1, 6, 2, 9, 100, 128, 0.1, 1, 1, None, 0, None) == _lib.FA_ERR_UNSUPPORTED
    args = [P, P, P, P, P, P, None, 2, 8, 1, 3, 4, 16, 8, 128, 0.1, 1, 4, None, 0, None]
    assert L.fa_decode_paged(*args) == _lib.FA_ERR_UNSUPPORTED
    # the static-scratch entry keeps the 16-row limit
    assert L.fa_decode_splitkv_static(P, P, P, P, None, 1, 8, 1, 3, 100, 128, 0.1, 1, 1, None) == _lib.FA_ERR_UNSUPPORTED
    # a split count above one needs a large enough, 256-byte aligned workspace
    assert L.fa_decode_splitkv(P, P, P, P, None, 1, 8, 2, 1, 100, 128, 0.1, 1, 4, None, 0, None) == _lib.FA_ERR_INVALID_ARG
    need = L.fa_decode_workspace_bytes(1, 8, 1, 128, 4)
    assert L.fa_decode_splitkv(P, P, P, P, None, 1, 8, 2, 1, 100, 128, 0.1, 1, 4, P, need - 1, None) == _lib.FA_ERR_INVALID_ARG
    assert L.fa_decode_splitkv(P, P, P, P, None, 1, 8, 2, 1, 100, 128, 0.1, 1, 4, ctypes.c_void_p(272), need, None) == _lib.FA_ERR_INVALID_ARG
    assert L.fa_decode_splitkv(P, P, P, P, None, 1, 8, 2, 1, 100, 128, 0.1, 1, -1, None, 0, None) == _lib.FA_ERR_INVALID_ARG
    # paged: only 16-token pages
    args = [P, P, P, P, P, P, None, 2, 8, 2, 1, 4, 32, 8, 128, 0.1, 1, 1, None, 0, None]
    assert L.fa_decode_paged(*args) == _lib.FA_ERR_UNSUPPORTED
    args[12] = 16
    args[3] = None  # no block table
    assert L.fa_decode_paged(*args) == _lib.FA_ERR_INVALID_ARG
    assert L.fa_lse_merge(P, P, P, None, 0, 4, 128, None) == _lib.FA_ERR_INVALID_ARG
    assert L.fa_lse_merge(P, P, P, None, 2, 4, 512, None) == _lib.FA_ERR_UNSUPPORTED


def test_kv_outer_workspace_and_rejections(L):
    rows, d = 2 * 4 * 100, 128
    need = ((rows * d * 4 + 255) // 256) * 256 + 2 * rows * 4
    assert L.fa_fwd_kv_outer_workspace_bytes(2, 4, 100, d) == need
    assert L.fa_fwd_kv_outer_workspace_bytes(0, 4, 100, d) == 0

    def ko(*, q=P, ws=P, ws_bytes=need, B=2, Hq=4, Hkv=2, T=100, S=300, d=128, scale=0.1, bands=1):
        return L.fa_fwd_kv_outer(q, P, P, P, None, B, Hq, Hkv, T, S, d, scale, 1, bands, ws, ws_bytes, None)

    assert ko(q=None) == _lib.FA_ERR_INVALID_ARG
    assert ko(bands=0) == _lib.FA_ERR_INVALID_ARG
    assert ko(ws=None) == _lib.FA_ERR_INVALID_ARG
    assert ko(ws_bytes=need - 1) == _lib.FA_ERR_INVALID_ARG
    assert ko(ws=MIS) == _lib.FA_ERR_INVALID_ARG
    assert ko(scale=-1.0) == _lib.FA_ERR_INVALID_ARG
    assert ko(Hq=3) == _lib.FA_ERR_INVALID_ARG
    assert ko(d=96, ws_bytes=1 << 30) == _lib.FA_ERR_UNSUPPORTED
    assert ko(Hq=12, Hkv=4, ws_bytes=1 << 30) == _lib.FA_ERR_UNSUPPORTED  # group of 3


def test_bwd_workspace_and_rejections(L):
    # two fp32 values per query row, rows padded to a multiple of 4 (16 bytes)
    assert L.fa_bwd_workspace_bytes(2, 4, 301) == 2 * 2 * 4 * 304 * 4
    assert L.fa_bwd_workspace_bytes(1, 1, 8) == 2 * 8 * 4
    assert L.fa_bwd_workspace_bytes(0, 4, 8) == 0
    need = L.fa_bwd_workspace_bytes(1, 2, 8)

    def bwd(*, ws=P, ws_bytes=need, Hq=2, Hkv=2, d=128, lse=P):
        return L.fa_bwd(P, P, P, P, lse, P, P, P, P, 1, Hq, Hkv, 8, 8, d, 0.1, 1, ws, ws_bytes, None)

    assert bwd(ws_bytes=need - 1) == _lib.FA_ERR_INVALID_ARG
    assert bwd(ws=None) == _lib.FA_ERR_INVALID_ARG
    assert bwd(lse=None) == _lib.FA_ERR_INVALID_ARG
    assert bwd(Hq=3) == _lib.FA_ERR_INVALID_ARG
    assert bwd(d=96) == _lib.FA_ERR_UNSUPPORTED


def test_workspace_size_counts_bytes_of_any_dtype():
    import torch

    from attention_fa2_attn_gb300.api import _ws_bytes

    assert _ws_bytes(torch.empty(10, dtype=torch.float32), 40, "cpu") == 40
    assert _ws_bytes(torch.empty(40, dtype=torch.uint8), 40, "cpu") == 40
    with pytest.raises(ValueError):
        _ws_bytes(torch.empty(9, dtype=torch.float32), 40, "cpu")
    with pytest.raises(ValueError):
        _ws_bytes(torch.empty(20, dtype=torch.float32)[::2], 40, "cpu")


def test_wait_timeout_clamp_and_unwind_floor(L):
    """The settable wait bound has a 1 ms floor; the waits a CTA makes before it
    exits (its copies landing, its MMAs draining) are bounded by at least 1 s,
    whatever is set."""
    w, u = ctypes.c_ulonglong(0), ctypes.c_ulonglong(0)
    L.fa_get_wait_timeouts(ctypes.byref(w), ctypes.byref(u))
    default = w.value
    assert (default, u.value) == (4_000_000_000, 4_000_000_000)
    try:
        for set_ns, want_wait, want_unwind in (
            (0, 10**6, 10**9),
            (1, 10**6, 10**9),
            (999_999, 10**6, 10**9),
            (10**6, 10**6, 10**9),
            (5 * 10**8, 5 * 10**8, 10**9),
            (10**9, 10**9, 10**9),
            (7 * 10**9, 7 * 10**9, 7 * 10**9),
        ):
            L.fa_set_wait_timeout_ns(set_ns)
            L.fa_get_wait_timeouts(ctypes.byref(w), ctypes.byref(u))
            assert (w.value, u.value) == (want_wait, want_unwind), set_ns
        L.fa_get_wait_timeouts(None, None)  # either pointer may be NULL
    finally:
        L.fa_set_wait_timeout_ns(default)


def test_decode_split_choice_is_made_in_one_place(L):
    """fa_decode_num_splits is the choice num_splits = 0 makes: the decode rule for
    at most 16 stacked rows per KV head, the prefill rule above that (contiguous
    K/V), no split for paged K/V with many rows."""
    ds = L.fa_decode_num_splits
    assert ds(1, 32, 8, 1, 131072, 0, 152) == L.fa_num_splits_heuristic(1, 8, 131072, 152) == 19
    assert ds(64, 64, 8, 1, 8192, 1, 152) == L.fa_num_splits_heuristic(64, 8, 8192, 152) == 1
    assert ds(1, 8, 2, 4, 5000, 1, 152) == L.fa_num_splits_heuristic(1, 2, 5000, 152)  # 16 rows: decode kernel
    assert ds(1, 8, 2, 5, 5000, 0, 152) == L.fa_num_splits_prefill(1, 8, 2, 5, 5000, 152)  # 20 rows: prefill kernel
    assert ds(1, 1, 1, 8192, 8192, 0, 152) == L.fa_num_splits_prefill(1, 1, 1, 8192, 8192, 152) == 4
    assert ds(1, 1, 1, 8192, 8192, 1, 152) == 1
    assert ds(0, 1, 1, 1, 100, 0, 152) == 1
    assert ds(1, 6, 4, 1, 100, 0, 152) == 1  # Hq not a multiple of Hkv
    # the binding sizes its workspace from the library's answer; it holds no rule of its own
    from attention_fa2_attn_gb300 import api

    for args in ((1, 32, 8, 1, 131072, False), (1, 1, 1, 8192, 8192, False), (3, 16, 4, 2, 9000, True),
                 (1, 16, 2, 40, 2304, True), (2, 4, 4, 300, 2200, False)):
        assert api.fa_decode_num_splits(*args, num_sms=152) == ds(*args[:5], int(args[5]), 152), args
