"""Parity of split-KV decode, the LSE merge and paged decode with the fp64 oracle."""

import math

import numpy as np
import pytest
import torch

import fa_inputs as fi
import oracle
from parity import compare

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _fa():
    import attention_fa2_attn_gb300 as fa

    return fa


SPLIT_CASES = [
    # B, Hq, Hkv, T, S, d, causal, splits
    (2, 8, 2, 1, 1000, 128, True, 1),
    (2, 8, 2, 1, 1000, 128, True, 3),
    (2, 8, 2, 1, 1000, 128, True, 16),
    (1, 32, 8, 1, 4097, 128, True, 0),
    (1, 8, 1, 2, 777, 64, True, 5),  # two new queries per head: 16 stacked rows
    (3, 4, 4, 1, 130, 64, False, 2),
    (1, 16, 2, 2, 300, 128, True, 64),  # more splits than 64-key tiles: empty splits
    (1, 4, 1, 3, 2, 128, True, 2),  # T > S: the first row sees no key
    (1, 32, 8, 1, 4097, 128, True, 16),
    (1, 32, 8, 1, 4097, 128, True, 17),
    (2, 16, 1, 1, 3000, 64, False, 8),
    (1, 16, 2, 1, 200, 128, True, 16),  # most splits empty
]


@pytest.mark.parametrize("case", SPLIT_CASES, ids=lambda c: "B{}_Hq{}_Hkv{}_T{}_S{}_d{}_{}_n{}".format(*c[:6], "causal" if c[6] else "full", c[7]))
def test_splitkv_small(case):
    B, Hq, Hkv, T, S, d, causal, n = case
    q, k, v = fi.qkv(B, Hq, Hkv, T, S, d, 60 + S % 11)
    scale = 1.0 / math.sqrt(d)
    o_ref, l_ref = oracle.attention_three_pass(q, k, v, scale, causal)
    o, l = _fa().fa_decode_splitkv(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, num_splits=n, scale=scale)
    compare(o, l, o_ref, l_ref, what=str(case))


def test_splitkv_full_size():
    w = fi.SPLITKV_DECODE
    q, k, v = fi.qkv(w.B, w.Hq, w.Hkv, w.T, w.S, w.d, w.index)
    o_ref, l_ref = oracle.attention_three_pass(q, k, v, w.scale, w.causal)
    o, l = _fa().fa_decode_splitkv(q.to(DEV), k.to(DEV), v.to(DEV), causal=w.causal, num_splits=w.num_splits, scale=w.scale)
    compare(o, l, o_ref, l_ref, what=w.name)
    # the split count does not change the result beyond rounding ("any split is exact")
    o1, l1 = _fa().fa_decode_splitkv(q.to(DEV), k.to(DEV), v.to(DEV), causal=w.causal, num_splits=1, scale=w.scale)
    compare(o1, l1, o_ref, l_ref, what=w.name + " unsplit")


@pytest.mark.parametrize("n", [2, 11, 12, 16, 17, 40])
def test_split_counts_on_both_merge_load_groups(n):
    """One (batch, KV head) split 2 to 40 ways: the merge takes its narrow load group
    below 12 splits and its wide one from 12, and more than 32 splits take two lse
    chunks. A NaN-filled workspace shows that every partial the merge reads was written."""
    B, Hq, Hkv, T, S, d = 1, 4, 1, 1, 3000, 128
    q, k, v = fi.qkv(B, Hq, Hkv, T, S, d, 91)
    o_ref, l_ref = oracle.attention_three_pass(q, k, v, 1.0 / math.sqrt(d), True)
    fa = _fa()
    ws = torch.full((fa.fa_decode_workspace_bytes(B, Hq, T, d, n) // 4,), float("nan"), device=DEV)
    o, l = fa.fa_decode_splitkv(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, num_splits=n, workspace=ws)
    compare(o, l, o_ref, l_ref, what=f"n={n}")


def test_merge_worked_example():
    """Partials of the scores [1, 2] | [3] with V = identity rows merge to the
    page's numbers: lse 3.408, weights 0.335 and 0.665."""
    q, k, vv = np.zeros((1, 1, 1, 3)), np.zeros((1, 1, 3, 3)), np.eye(3).reshape(1, 1, 3, 3)
    q[0, 0, 0, 0] = 1.0
    k[0, 0, :, 0] = [1.0, 2.0, 3.0]
    op, lp = oracle.attention_partials(q, k, vv, 1.0, False, 2)
    o_part = torch.tensor(op.reshape(2, 1, 3), dtype=torch.float32, device=DEV)
    lse_part = torch.tensor(lp.reshape(2, 1), dtype=torch.float32, device=DEV)
    o, l = _fa().fa_lse_merge(o_part, lse_part)
    assert abs(float(l[0]) - 3.408) < 5e-4
    got = o[0].float().cpu().numpy()
    assert abs(got[0] + got[1] - 0.335) < 5e-3 and abs(got[2] - 0.665) < 5e-3


@pytest.mark.parametrize("n,rows,d", [(7, 50, 128), (1, 3, 64), (5, 9, 1), (32, 17, 33), (33, 6, 100), (70, 5, 256)])
def test_merge_random_with_empty_splits(n, rows, d):
    """Any split count (more than one warp's worth included), row count and width."""
    g = torch.Generator().manual_seed(3 + n + d)
    # partials are averages of V rows: keep them in that range, where the bf16 output's own
    # rounding stays well inside the output tolerance
    o_part = torch.randn(n, rows, d, generator=g) * 0.25
    lse_part = torch.randn(n, rows, generator=g) * 5
    lse_part[min(2, n - 1)] = -math.inf if n > 1 else lse_part[0]  # an empty split
    lse_part[:, min(7, rows - 1)] = -math.inf  # a row that saw no key at all
    o_ref, l_ref = oracle.lse_merge(o_part.numpy(), lse_part.numpy())
    o, l = _fa().fa_lse_merge(o_part.to(DEV), lse_part.to(DEV))
    compare(o, l, o_ref, l_ref, what="merge")


def _paged_problem(B, Hq, Hkv, T, d, seqlens, max_pages, index):
    k_pages, v_pages, table, _ = fi.paged_kv(B, Hkv, max_pages * 16, d, 16, index)
    q = fi.decode_q(B, Hq, T, d, index)
    sl = torch.tensor(seqlens, dtype=torch.int32)
    return q, k_pages, v_pages, table, sl


PAGED_CASES = [
    # B, Hq, Hkv, T, d, seqlens, max_pages, splits
    (3, 8, 2, 1, 128, [40, 16, 1], 3, 1),
    (3, 8, 2, 1, 128, [40, 16, 1], 3, 2),
    (4, 16, 2, 1, 64, [1000, 333, 64, 0], 64, 3),
    (2, 8, 1, 2, 128, [517, 260], 40, 1),
    (2, 64, 8, 1, 128, [2048, 1500], 128, 4),
    (2, 64, 8, 1, 128, [2048, 9], 128, 16),  # one sequence with mostly empty splits
]


@pytest.mark.parametrize("case", PAGED_CASES, ids=lambda c: "B{}_Hq{}_Hkv{}_T{}_d{}_n{}".format(*c[:5], c[7]))
def test_paged_small(case):
    B, Hq, Hkv, T, d, seqlens, max_pages, n = case
    q, kp, vp, table, sl = _paged_problem(B, Hq, Hkv, T, d, seqlens, max_pages, 70 + B)
    scale = 1.0 / math.sqrt(d)
    o_ref, l_ref = oracle.decode_paged(q, kp, vp, table, sl, 16, scale, True)
    o, l = _fa().fa_decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV), sl.to(DEV), causal=True,
                                 num_splits=n, scale=scale)
    compare(o, l, o_ref, l_ref, what=str(case))


def test_paged_equals_contiguous_bit_exact():
    """Gathering the pages into contiguous K/V and running the split-KV path on
    them gives the same bits: the block-table gather is exact."""
    B, Hq, Hkv, T, d, S = 3, 32, 8, 1, 128, 1024
    q, kp, vp, table, _ = _paged_problem(B, Hq, Hkv, T, d, [S] * B, S // 16, 81)
    sl = torch.full((B,), S, dtype=torch.int32)
    kc = torch.stack([torch.from_numpy(oracle.paged_gather(kp.float(), table[b], S, 16)) for b in range(B)]).bfloat16()
    vc = torch.stack([torch.from_numpy(oracle.paged_gather(vp.float(), table[b], S, 16)) for b in range(B)]).bfloat16()
    for n in (1, 3):
        o1, l1 = _fa().fa_decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV), sl.to(DEV), num_splits=n)
        o2, l2 = _fa().fa_decode_splitkv(q.to(DEV), kc.to(DEV), vc.to(DEV), num_splits=n)
        assert torch.equal(o1, o2) and torch.equal(l1, l2), n


def test_paged_full_size():
    w = fi.PAGED_DECODE
    kp, vp, table, sl = fi.paged_kv(w.B, w.Hkv, w.S, w.d, w.page_size, w.index)
    q = fi.decode_q(w.B, w.Hq, w.T, w.d, w.index)
    o, l = _fa().fa_decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV), sl.to(DEV), causal=True,
                                 num_splits=1, scale=w.scale)
    o_ref, l_ref = oracle.decode_paged(q, kp, vp, table, sl, 16, w.scale, True)
    compare(o, l, o_ref, l_ref, what=w.name)


def test_paged_bad_table_entry_is_reported():
    """A block-table entry outside the pool is never dereferenced: the kernel's
    bounds check records FA_ERR_BOUNDS and the call returns normally."""
    fa = _fa()
    B, Hq, Hkv, T, d = 2, 8, 2, 1, 128
    q, kp, vp, table, sl = _paged_problem(B, Hq, Hkv, T, d, [64, 64], 4, 83)
    bad = table.clone()
    bad[1, 2] = kp.shape[0] + 5
    assert fa.fa_get_last_device_error()[0] == 0
    fa.fa_decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), bad.to(DEV), sl.to(DEV), num_splits=1)
    st, word = fa.fa_get_last_device_error()
    assert st == 5 and (word & 0xFF) == 5
    # sequence 0 did not touch the bad entry and is still exact
    o, l = fa.fa_decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV), sl.to(DEV), num_splits=1)
    o_ref, l_ref = oracle.decode_paged(q, kp, vp, table, sl, 16, 1 / math.sqrt(d), True)
    compare(o, l, o_ref, l_ref, what="after bounds error")
    assert fa.fa_get_last_device_error()[0] == 0


def test_zero_splits_same_choice_through_python_and_c():
    """num_splits = 0 is resolved by the library alone: the Python call (which only
    sizes the workspace from fa_decode_num_splits), a direct C call with an ample
    workspace, and an explicit call with that count give the same bits."""
    import ctypes

    fa = _fa()
    from attention_fa2_attn_gb300 import _lib

    L = _lib.lib()
    for B, Hq, Hkv, T, S, d in ((1, 32, 8, 1, 16384, 128), (1, 2, 2, 600, 3000, 64)):
        q, k, v = (t.to(DEV) for t in fi.qkv(B, Hq, Hkv, T, S, d, 130 + d))
        n = fa.fa_decode_num_splits(B, Hq, Hkv, T, S)
        assert n > 1
        o_py, l_py = fa.fa_decode_splitkv(q, k, v, causal=True, num_splits=0)
        o_n, l_n = fa.fa_decode_splitkv(q, k, v, causal=True, num_splits=n)
        ws = torch.empty(fa.fa_decode_workspace_bytes(B, Hq, T, d, 64), dtype=torch.uint8, device=DEV)
        o_c, l_c = torch.empty_like(q), torch.empty((B, Hq, T), dtype=torch.float32, device=DEV)
        st = L.fa_decode_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o_c.data_ptr(), l_c.data_ptr(), B, Hq,
                                 Hkv, T, S, d, 1.0 / math.sqrt(d), 1, 0, ws.data_ptr(), ws.numel(),
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == 0
        torch.cuda.synchronize()
        assert torch.equal(o_py, o_n) and torch.equal(l_py, l_n)
        assert torch.equal(o_c, o_n) and torch.equal(l_c, l_n)
