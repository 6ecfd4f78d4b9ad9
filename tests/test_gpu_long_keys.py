"""Parity at key counts far past the workloads': 2^20 + 37 keys per sequence, so
each K and V tensor (and each paged pool) is over 2 GiB and byte offsets into it
pass 2^31. This exercises the 64-bit address arithmetic of every path, the ring
counters and barrier phases over 8193 key tiles per item, split ranges of over
65536 keys, and the backward's 98316 dK/dV CTAs and 8193-step dQ loops.

Inputs are drawn on the device from the seeded generators. The oracle checks a
sample of query rows: each row is independent, so it is exact against the whole
K/V plane of its KV head ("Kernel visualization: Flash Attention 1", "The tiled
version"). The standard bf16 bounds apply.
"""

import math

import pytest
import torch

import fa_inputs as fi
import oracle
from parity import compare
from test_gpu_backward import _grad_compare  # the backward's bounds, relative to each gradient's largest entry

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
S_LONG = (1 << 20) + 37


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    yield
    torch.cuda.empty_cache()


def _fa():
    import attention_fa2_attn_gb300 as fa

    return fa


def _check_rows(o, l, q, k, v, rows, scale, causal, what):
    o_ref, l_ref = oracle.attention_rows(q, k, v, rows, scale, causal)
    idx = torch.tensor(rows)
    og = o.cpu()[idx[:, 0], idx[:, 1], idx[:, 2]]
    lg = l.cpu()[idx[:, 0], idx[:, 1], idx[:, 2]]
    compare(og, lg, o_ref, l_ref, what=what)


@pytest.mark.parametrize("num_splits", [0, 16])
def test_decode_long_keys(num_splits):
    """Split-KV decode, GQA 32/8, one new token over 2^20 + 37 cached keys."""
    B, Hq, Hkv, T, S, d = 1, 32, 8, 1, S_LONG, 128
    q, k, v = fi.qkv(B, Hq, Hkv, T, S, d, 900, device=DEV)
    scale = 1.0 / math.sqrt(d)
    o, l = _fa().fa_decode_splitkv(q, k, v, causal=True, num_splits=num_splits, scale=scale)
    rows = [(0, h, 0) for h in (0, 5, 13, 22, 31)]  # query heads over KV heads 0, 1, 3, 5, 7
    _check_rows(o, l, q, k, v, rows, scale, True, f"decode n{num_splits}")
    del q, k, v


@pytest.mark.parametrize("causal", [False, True])
def test_prefill_long_keys(causal):
    """The prefill kernel: 200 query rows per head over 2^20 + 37 keys, 8 heads, so
    each CTA's item streams 8193 key tiles; then the same through the key split."""
    B, Hq, Hkv, T, S, d = 1, 8, 8, 200, S_LONG, 128
    q, k, v = fi.qkv(B, Hq, Hkv, T, S, d, 910 + int(causal), device=DEV)
    scale = 1.0 / math.sqrt(d)
    rows = sorted({(0, h, i) for h in (0, 7) for i in (0, 1, 63, 64, 127, 128, 199)} |
                  {(0, 3, i) for i in (17, 150)})
    fa = _fa()
    o, l = fa.fa_fwd(q, k, v, causal=causal, scale=scale)
    _check_rows(o, l, q, k, v, rows, scale, causal, f"prefill causal={causal}")
    o2, l2 = fa.fa_decode_splitkv(q, k, v, causal=causal, num_splits=7, scale=scale)
    _check_rows(o2, l2, q, k, v, rows, scale, causal, f"key split causal={causal}")
    del q, k, v


def _scatter_pages(x, table, page_size):
    """Contiguous [B][Hkv][S][d] (S a multiple of page_size) laid out as a pool
    [B * max_pages][page_size][Hkv][d] through ``table`` [B][max_pages]."""
    B, Hkv, S, d = x.shape
    mp = S // page_size
    pages = x.view(B, Hkv, mp, page_size, d).permute(0, 2, 3, 1, 4).reshape(B * mp, page_size, Hkv, d)
    pool = torch.empty_like(pages)
    pool[table.reshape(-1).long()] = pages
    return pool


def test_paged_long_pool():
    """Paged decode over a 2.15 GB pool per operand (65536 16-token pages, 8 KV
    heads): bit-identical to the contiguous path when every sequence is full, and
    against the oracle with ragged sequence lengths."""
    B, Hq, Hkv, T, S, d = 2, 16, 8, 1, 1 << 19, 128
    q, k, v = fi.qkv(B, Hq, Hkv, T, S, d, 920, device=DEV)
    mp = S // 16
    perm = torch.randperm(B * mp, generator=fi._gen(4000 + 920))
    table = perm.view(B, mp).to(torch.int32).to(DEV)
    kp, vp = _scatter_pages(k, table, 16), _scatter_pages(v, table, 16)
    scale = 1.0 / math.sqrt(d)
    fa = _fa()
    full = torch.full((B,), S, dtype=torch.int32, device=DEV)
    o_p, l_p = fa.fa_decode_paged(q, kp, vp, table, full, causal=True, num_splits=5, scale=scale)
    o_c, l_c = fa.fa_decode_splitkv(q, k, v, causal=True, num_splits=5, scale=scale)
    assert torch.equal(o_p, o_c) and torch.equal(l_p, l_c)
    ragged = [S - 1000 + 5, 70001]
    o_r, l_r = fa.fa_decode_paged(q, kp, vp, table, torch.tensor(ragged, dtype=torch.int32, device=DEV),
                                  causal=True, scale=scale)
    for b, sb in enumerate(ragged):
        rows = [(0, h, 0) for h in (0, 9, 15)]
        _check_rows(o_r[b : b + 1], l_r[b : b + 1], q[b : b + 1], k[b : b + 1, :, :sb], v[b : b + 1, :, :sb], rows,
                    scale, True, f"paged ragged b{b}")
    del q, k, v, kp, vp


@pytest.mark.parametrize("causal", [False, True])
def test_backward_long_keys(causal):
    """fa_fwd then fa_bwd with 256 query rows per head over 2^20 + 37 keys, 12
    heads: K, V, dK and dV are 3.2 GB each, and head 10 lies wholly past 2^31
    bytes. dQ rows (each over every key) and dK/dV rows (each over every query row)
    of heads 1 and 10 are checked against the oracle, given those heads' planes."""
    B, H, T, S, d = 1, 12, 256, S_LONG, 128
    q, k, v = fi.qkv(B, H, H, T, S, d, 930 + int(causal), device=DEV)
    do = fi.randn((B, H, T, d), 5930 + int(causal), device=DEV)
    scale = 1.0 / math.sqrt(d)
    fa = _fa()
    o, lse = fa.fa_fwd(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = fa.fa_bwd(q, k, v, o, lse, do, causal=causal, scale=scale)
    for h in (1, 10):
        sl = slice(h, h + 1)
        q_rows = [(0, 0, i) for i in (0, 77, 128, 255)]
        k_rows = [(0, 0, j) for j in (0, 12345, S - T - 1, S - T, S - 100, S - 1)]
        rq, rk, rv = oracle.attention_backward_rows(q[:, sl], k[:, sl], v[:, sl], do[:, sl], o[:, sl].float(),
                                                    lse[:, sl], q_rows, k_rows, scale, causal)
        iq = torch.tensor([i for _, _, i in q_rows])
        ik = torch.tensor([j for _, _, j in k_rows])
        _grad_compare(dq[0, h].cpu()[iq], rq, f"dq head {h} causal={causal}")
        _grad_compare(dk[0, h].cpu()[ik], rk, f"dk head {h} causal={causal}")
        _grad_compare(dv[0, h].cpu()[ik], rv, f"dv head {h} causal={causal}")
    del q, k, v, do, o, dq, dk, dv
