"""Seeded random shapes for every entry point, against the fp64 oracle at the standard
bounds: batch, heads, GQA group (1..16), head dimension (64, 128), query and key
counts (ragged, T < S and T > S), causal or not, split counts, page tables and
sequence lengths are drawn from one generator per test, so each run checks the
same shapes. Sizes stay small enough for the oracle to finish each case in well
under a second.
"""

import math
import random

import pytest
import torch

import fa_inputs as fi
import oracle
from parity import compare
from test_gpu_backward import _grad_compare  # the backward's bounds, relative to each gradient's largest entry

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
GROUPS = (1, 2, 4, 8, 16)


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _fa():
    import attention_fa2_attn_gb300 as fa

    return fa


def _shapes(seed, n, t_max, s_max, budget=2.0e8):
    """n shapes (B, Hq, Hkv, T, S, d, causal) with B*Hq*T*S*d below budget."""
    rng = random.Random(seed)
    out = []
    while len(out) < n:
        B = rng.randint(1, 3)
        Hkv = rng.randint(1, 3)
        g = rng.choice(GROUPS)
        d = rng.choice((64, 128))
        T = rng.randint(1, t_max)
        S = rng.randint(1, s_max)
        if B * Hkv * g * T * S * d > budget:
            continue
        out.append((B, g * Hkv, Hkv, T, S, d, rng.random() < 0.5))
    return out


def _ids(c):
    return "B{}_Hq{}_Hkv{}_T{}_S{}_d{}_{}".format(*c[:6], "causal" if c[6] else "full")


@pytest.mark.parametrize("case", _shapes(1234, 24, 400, 1200), ids=_ids)
def test_random_prefill(case):
    B, Hq, Hkv, T, S, d, causal = case
    q, k, v = fi.qkv(B, Hq, Hkv, T, S, d, 300 + (T * 7 + S) % 97)
    scale = 1.0 / math.sqrt(d)
    o_ref, l_ref = oracle.attention_three_pass(q, k, v, scale, causal)
    o, l = _fa().fa_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, scale=scale)
    compare(o, l, o_ref, l_ref, what=_ids(case))


def _decode_cases(seed, n):
    """Decode-shaped problems: at most 16 stacked query rows per KV head, a split count."""
    rng = random.Random(seed)
    out = []
    while len(out) < n:
        B = rng.randint(1, 4)
        Hkv = rng.randint(1, 4)
        g = rng.choice(GROUPS)
        T = rng.randint(1, max(1, 16 // g))
        S = rng.randint(1, 6000)
        d = rng.choice((64, 128))
        splits = rng.choice((0, 1, 2, 3, 5, 8, 16))
        if B * Hkv * g * T * S * d > 2.0e8:
            continue
        out.append((B, g * Hkv, Hkv, T, S, d, splits))
    return out


@pytest.mark.parametrize("case", _decode_cases(5678, 20),
                         ids=lambda c: "B{}_Hq{}_Hkv{}_T{}_S{}_d{}_n{}".format(*c))
def test_random_decode(case):
    """The decode kernel (split ranges and the LSE merge), bottom-right causal."""
    B, Hq, Hkv, T, S, d, n = case
    q, k, v = fi.qkv(B, Hq, Hkv, T, S, d, 400 + S % 89)
    scale = 1.0 / math.sqrt(d)
    o_ref, l_ref = oracle.attention_three_pass(q, k, v, scale, True)
    o, l = _fa().fa_decode_splitkv(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, num_splits=n, scale=scale)
    compare(o, l, o_ref, l_ref, what=str(case))


@pytest.mark.parametrize("case", _shapes(9012, 12, 600, 2500), ids=_ids)
def test_random_key_split(case):
    """Prefill-shaped problems through the key split (more than 16 rows per KV head
    where the shape has them; the decode kernel otherwise), 2-7 ranges."""
    B, Hq, Hkv, T, S, d, causal = case
    n = 2 + (T + S) % 6
    q, k, v = fi.qkv(B, Hq, Hkv, T, S, d, 500 + (T + 3 * S) % 83)
    scale = 1.0 / math.sqrt(d)
    o_ref, l_ref = oracle.attention_three_pass(q, k, v, scale, causal)
    o, l = _fa().fa_decode_splitkv(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, num_splits=n, scale=scale)
    compare(o, l, o_ref, l_ref, what=_ids(case) + f"_n{n}")


def _paged_cases(seed, n):
    rng = random.Random(seed)
    out = []
    while len(out) < n:
        B = rng.randint(1, 4)
        Hkv = rng.randint(1, 3)
        g = rng.choice(GROUPS)
        T = rng.choice((1, 1, 2, rng.randint(3, 200)))  # decode steps and chunked prefills
        max_pages = rng.randint(1, 160)
        d = rng.choice((64, 128))
        seqlens = [rng.randint(0, max_pages * 16) for _ in range(B)]
        if B * Hkv * g * T * max_pages * 16 * d > 2.0e8:
            continue
        out.append((B, g * Hkv, Hkv, T, d, max_pages, tuple(seqlens)))
    return out


@pytest.mark.parametrize("case", _paged_cases(3456, 16),
                         ids=lambda c: "B{}_Hq{}_Hkv{}_T{}_d{}_pages{}".format(*c[:6]))
def test_random_paged(case):
    """Paged K/V through a random-permutation block table: the decode kernel for at
    most 16 stacked rows, the chunked prefill otherwise; sequences of any length up to
    the table's reach, empty ones included."""
    B, Hq, Hkv, T, d, max_pages, seqlens = case
    k_pages, v_pages, table, _ = fi.paged_kv(B, Hkv, max_pages * 16, d, 16, 600 + max_pages % 71)
    q = fi.decode_q(B, Hq, T, d, 600 + T % 53)
    sl = torch.tensor(seqlens, dtype=torch.int32)
    scale = 1.0 / math.sqrt(d)
    o_ref, l_ref = oracle.decode_paged(q, k_pages, v_pages, table, sl, 16, scale, True)
    o, l = _fa().fa_decode_paged(q.to(DEV), k_pages.to(DEV), v_pages.to(DEV), table.to(DEV), sl.to(DEV),
                                 causal=True, scale=scale)
    compare(o, l, o_ref, l_ref, what=str(case[:6]))


@pytest.mark.parametrize("case", _shapes(7890, 8, 300, 400, budget=4.0e7), ids=_ids)
def test_random_backward(case):
    B, Hq, Hkv, T, S, d, causal = case
    q, k, v = fi.qkv(B, Hq, Hkv, T, S, d, 700 + (T + S) % 61)
    do = fi.randn((B, Hq, T, d), 800 + T % 59)
    scale = 1.0 / math.sqrt(d)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    fa = _fa()
    o, lse = fa.fa_fwd(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = fa.fa_bwd(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    rq, rk, rv = oracle.attention_backward(q, k, v, do, scale, causal, o=o.float().cpu(), lse=lse.cpu())
    _grad_compare(dq, rq, _ids(case) + " dq")
    _grad_compare(dk, rk, _ids(case) + " dk")
    _grad_compare(dv, rv, _ids(case) + " dv")
