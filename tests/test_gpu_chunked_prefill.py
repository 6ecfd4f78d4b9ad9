"""Chunked prefill / multi-token steps over the K/V cache: more than 16 query rows
per KV head, run by the tensor-core prefill kernel through the decode entry
points (paged: each 128-key tile gathered from eight 16-token pages).

The oracle is the same one as for decode: each sequence's keys and values are
gathered through its block-table row and the three-pass definition runs on
them, with the bottom-right mask (the T new tokens sit at positions
seqlens[b] - T .. seqlens[b] - 1).
"""

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


def _paged_problem(B, Hq, Hkv, T, d, seqlens, max_pages, index):
    k_pages, v_pages, table, _ = fi.paged_kv(B, Hkv, max_pages * 16, d, 16, index)
    q = fi.decode_q(B, Hq, T, d, index)
    return q, k_pages, v_pages, table, torch.tensor(seqlens, dtype=torch.int32)


CASES = [
    # B, Hq, Hkv, T, d, seqlens, max_pages, causal
    (3, 8, 2, 100, 128, [100, 357, 1000], 64, True),  # g = 4: 400 stacked rows per KV head
    (2, 4, 4, 300, 64, [300, 2049], 129, True),  # MHA, ragged last tile and last page
    (2, 16, 2, 33, 128, [20, 700], 44, True),  # T > seqlen: the first rows of sequence 0 see no key
    (1, 8, 8, 130, 128, [517], 33, False),
    (2, 8, 1, 17, 64, [0, 64], 4, True),  # an empty sequence: O = 0, lse = -inf
    (2, 32, 2, 9, 128, [4000, 128], 250, True),  # g = 16: 144 rows
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}_Hq{}_Hkv{}_T{}_d{}_{}".format(*c[:5], "causal" if c[7] else "full"))
def test_paged_chunked_prefill(case):
    B, Hq, Hkv, T, d, seqlens, max_pages, causal = case
    q, kp, vp, table, sl = _paged_problem(B, Hq, Hkv, T, d, seqlens, max_pages, 90 + T % 13)
    scale = 1.0 / math.sqrt(d)
    o_ref, l_ref = oracle.decode_paged(q, kp, vp, table, sl, 16, scale, causal)
    o, l = _fa().fa_decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV), sl.to(DEV), causal=causal,
                                 num_splits=0, scale=scale)
    compare(o, l, o_ref, l_ref, what=str(case))


def _poison_unused(pages, table, seqlens):
    """NaN in every pool row that no sequence's valid token occupies."""
    pages = pages.clone()
    used = torch.zeros(pages.shape[:2], dtype=torch.bool)
    for b, S in enumerate(seqlens.tolist()):
        for t in range(S):
            used[int(table[b, t // 16]), t % 16] = True
    pages[~used] = float("nan")
    return pages


def test_pool_rows_past_the_end_are_never_used():
    """Tail slots of each sequence's last page and the pages after it hold NaN:
    a masked key must contribute exactly nothing (no 0 * NaN)."""
    B, Hq, Hkv, T, d = 3, 16, 4, 70, 128
    seqlens = [70, 1001, 333]
    q, kp, vp, table, sl = _paged_problem(B, Hq, Hkv, T, d, seqlens, 70, 97)
    kp, vp = _poison_unused(kp, table, sl), _poison_unused(vp, table, sl)
    scale = 1.0 / math.sqrt(d)
    o_ref, l_ref = oracle.decode_paged(q, kp, vp, table, sl, 16, scale, True)
    o, l = _fa().fa_decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV), sl.to(DEV), causal=True,
                                 scale=scale)
    assert torch.isfinite(o.float()).all()
    compare(o, l, o_ref, l_ref, what="poisoned pool")


def test_paged_chunked_equals_contiguous_bit_exact():
    """The page gather is exact: the same problem on the gathered contiguous K/V
    through fa_fwd gives the same bits."""
    B, Hq, Hkv, T, d, S = 2, 16, 4, 200, 128, 1000
    q, kp, vp, table, _ = _paged_problem(B, Hq, Hkv, T, d, [S] * B, 63, 98)
    sl = torch.full((B,), S, dtype=torch.int32)
    kc = torch.stack([torch.from_numpy(oracle.paged_gather(kp.float(), table[b], S, 16)) for b in range(B)]).bfloat16()
    vc = torch.stack([torch.from_numpy(oracle.paged_gather(vp.float(), table[b], S, 16)) for b in range(B)]).bfloat16()
    for causal in (True, False):
        o1, l1 = _fa().fa_decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV), sl.to(DEV), causal=causal)
        o2, l2 = _fa().fa_fwd(q.to(DEV), kc.to(DEV), vc.to(DEV), causal=causal)
        assert torch.equal(o1, o2) and torch.equal(l1, l2), causal


def test_contiguous_many_rows():
    """fa_decode_splitkv with 256 stacked rows runs the prefill kernel, unsplit or
    with its keys cut into ranges; a key split over the paged cache is refused
    rather than silently ignored."""
    fa = _fa()
    B, Hq, Hkv, T, S, d = 1, 8, 2, 64, 3000, 128
    q, k, v = fi.qkv(B, Hq, Hkv, T, S, d, 99)
    scale = 1.0 / math.sqrt(d)
    o_ref, l_ref = oracle.attention_three_pass(q, k, v, scale, True)
    for n in (1, 3):
        o, l = fa.fa_decode_splitkv(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, num_splits=n, scale=scale)
        compare(o, l, o_ref, l_ref, what=f"contiguous many rows, {n} ranges")
    qp, kp, vp, table, sl = _paged_problem(1, 8, 2, 64, 128, [3000], 188, 99)
    with pytest.raises(fa.FAError):
        fa.fa_decode_paged(qp.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV), sl.to(DEV), num_splits=3)


def test_chunked_bad_table_entry_is_reported():
    fa = _fa()
    B, Hq, Hkv, T, d = 2, 8, 2, 40, 128
    q, kp, vp, table, sl = _paged_problem(B, Hq, Hkv, T, d, [300, 300], 19, 100)
    bad = table.clone()
    bad[1, 5] = -3
    assert fa.fa_get_last_device_error()[0] == 0
    fa.fa_decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), bad.to(DEV), sl.to(DEV))
    st, word = fa.fa_get_last_device_error()
    assert st == 5 and (word & 0xFF) == 5 and (word >> 8) == 8
    o, l = fa.fa_decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV), sl.to(DEV))
    o_ref, l_ref = oracle.decode_paged(q, kp, vp, table, sl, 16, 1 / math.sqrt(d), True)
    compare(o, l, o_ref, l_ref, what="after bounds error")
    assert fa.fa_get_last_device_error()[0] == 0


def test_chunked_prefill_large_sampled():
    """A serving-sized chunk: 8 sequences of up to 8192 cached tokens, 512 new
    tokens each, GQA 32/8; sampled rows against the oracle."""
    w = fi.CHUNKED_PREFILL
    q, kp, vp, table, sl = fi.chunked_prefill_problem(w)
    o, l = _fa().fa_decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV), sl.to(DEV), causal=True,
                                 scale=w.scale)
    o, l = o.cpu(), l.cpu()
    rows = fi.sample_rows(w.B, w.Hq, w.T, 512, 11)
    og, lg, orf, lrf = [], [], [], []
    for b in range(w.B):
        mine = [(0, h, i) for (bb, h, i) in rows if bb == b]
        if not mine:
            continue
        S = int(sl[b])
        kb = torch.from_numpy(oracle.paged_gather(kp.float(), table[b], S, 16))[None]
        vb = torch.from_numpy(oracle.paged_gather(vp.float(), table[b], S, 16))[None]
        o_ref, l_ref = oracle.attention_rows(q[b : b + 1], kb, vb, mine, w.scale, True)
        idx = torch.tensor(mine)
        og.append(o[b][idx[:, 1], idx[:, 2]])
        lg.append(l[b][idx[:, 1], idx[:, 2]])
        orf.append(o_ref)
        lrf.append(l_ref)
    compare(torch.cat(og), torch.cat(lg), np.concatenate(orf), np.concatenate(lrf), what=w.name)
