"""Parity of the FlashAttention-1-order forward (key tiles outer, the running
O', m, l of every query row through HBM) with the fp64 oracle.

Small cases go against the oracle's own FlashAttention-1 recurrence
(normalised o', running denominator, "The tiled version"), which the oracle
pins tie to the three-pass definition. The serving-sized cases are compared on
sampled rows, each computed exactly by the oracle. Tolerances are those of the
bf16 forward.
"""

import math

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


CASES = [
    # B, Hq, Hkv, T, S, d, causal, row_bands
    (1, 1, 1, 128, 128, 64, False, 1),  # one step: first and last key tile at once
    (1, 2, 2, 300, 517, 128, True, 1),  # ragged query and key tails
    (2, 4, 2, 130, 257, 64, True, 2),  # GQA 2, two bands
    (1, 4, 4, 257, 129, 128, True, 3),  # T > S: the first tile sees no key at all
    (1, 8, 1, 200, 700, 128, False, 1),  # GQA 8
    (2, 2, 2, 384, 384, 128, False, 5),  # more bands than query tiles: clamped
    (1, 16, 1, 100, 1000, 64, True, 1),  # GQA 16, one query tile, eight key tiles
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}_Hq{}_Hkv{}_T{}_S{}_d{}_{}_r{}".format(
    *c[:6], "causal" if c[6] else "full", c[7]))
def test_kv_outer_small(case):
    B, Hq, Hkv, T, S, d, causal, bands = case
    q, k, v = fi.qkv(B, Hq, Hkv, T, S, d, 200 + T % 23)
    scale = 1.0 / math.sqrt(d)
    o_ref, l_ref = oracle.attention_online_normalized(q, k, v, scale, causal, block=128)
    o, l = _fa().fa_fwd_kv_outer(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, scale=scale, row_bands=bands)
    compare(o, l, o_ref, l_ref, what=str(case))


def test_bands_do_not_change_the_bits():
    """A query tile's recurrence runs over the same key tiles in the same order
    whatever band holds it, so the band count leaves every bit unchanged."""
    B, Hq, Hkv, T, S, d = 2, 4, 2, 700, 900, 128
    q, k, v = (t.to(DEV) for t in fi.qkv(B, Hq, Hkv, T, S, d, 211))
    for causal in (False, True):
        o1, l1 = _fa().fa_fwd_kv_outer(q, k, v, causal=causal, row_bands=1)
        for bands in (2, 6):
            o2, l2 = _fa().fa_fwd_kv_outer(q, k, v, causal=causal, row_bands=bands)
            assert torch.equal(o1, o2) and torch.equal(l1, l2), (causal, bands)


def test_workspace_needs_no_initialisation():
    """The first key tile of every query tile starts from an empty state, so a
    workspace full of NaN gives the same result as a zeroed one."""
    fa = _fa()
    B, Hq, Hkv, T, S, d = 1, 4, 4, 300, 400, 128
    q, k, v = (t.to(DEV) for t in fi.qkv(B, Hq, Hkv, T, S, d, 212))
    n = fa.fa_fwd_kv_outer_workspace_bytes(B, Hq, T, d)
    ws_nan = torch.full((n // 4,), float("nan"), dtype=torch.float32, device=DEV)
    ws_zero = torch.zeros(n // 4, dtype=torch.float32, device=DEV)
    o1, l1 = fa.fa_fwd_kv_outer(q, k, v, causal=True, workspace=ws_nan.view(torch.uint8))
    o2, l2 = fa.fa_fwd_kv_outer(q, k, v, causal=True, workspace=ws_zero.view(torch.uint8))
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.isfinite(o1.float()).all()


def _sampled(w, bands, nrows, seed):
    q, k, v = fi.qkv(w.B, w.Hq, w.Hkv, w.T, w.S, w.d, w.index)
    o, l = _fa().fa_fwd_kv_outer(q.to(DEV), k.to(DEV), v.to(DEV), causal=w.causal, scale=w.scale, row_bands=bands)
    rows = fi.sample_rows(w.B, w.Hq, w.T, nrows, seed)
    o_ref, l_ref = oracle.attention_rows(q, k, v, rows, w.scale, w.causal)
    idx = torch.tensor(rows)
    o, l = o.cpu(), l.cpu()
    compare(o[idx[:, 0], idx[:, 1], idx[:, 2]], l[idx[:, 0], idx[:, 1], idx[:, 2]], o_ref, l_ref, what=w.name)


def test_kv_outer_prefill_mha_sampled():
    """The prefill workload (B=4, H=16, N=4096, d=128) with the pages' grid, one
    CTA per (batch, head): 32 key tiles x 32 query tiles per CTA."""
    _sampled(fi.PREFILL_MHA, 1, 256, 31)


def test_kv_outer_causal_gqa_sampled():
    """The causal GQA workload (B=1, Hq=64, Hkv=8, N=8192, d=128) in two bands per head."""
    _sampled(fi.CAUSAL_GQA, 2, 128, 32)
