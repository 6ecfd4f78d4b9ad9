"""Prefill-shaped problems whose query tiles do not fill the GPU, with the keys cut
into ranges ("How many splits for decode", applied to the prefill kernel's work
items) and the partials merged ("The log-sum-exp merge"): parity with the fp64
oracle, including empty ranges and the one-head sweep of the prefill workload.
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


CASES = [
    # B, Hq, Hkv, T, S, d, causal, splits
    (1, 1, 1, 300, 1000, 64, False, 3),
    (1, 2, 1, 300, 1000, 128, True, 3),
    (2, 4, 4, 200, 700, 128, False, 5),
    (1, 4, 2, 257, 129, 128, True, 4),  # 2 key tiles, 4 ranges: empty ranges; T > S: rows with no key
    (1, 8, 1, 64, 2000, 64, True, 7),  # GQA group 8
    (1, 1, 1, 1000, 1000, 128, True, 0),  # the heuristic picks the count
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}_Hq{}_Hkv{}_T{}_S{}_d{}_{}_n{}".format(*c[:6], "causal" if c[6] else "full", c[7]))
def test_split_prefill_small(case):
    B, Hq, Hkv, T, S, d, causal, n = case
    q, k, v = fi.qkv(B, Hq, Hkv, T, S, d, 110 + T % 9)
    scale = 1.0 / math.sqrt(d)
    o_ref, l_ref = oracle.attention_three_pass(q, k, v, scale, causal)
    o, l = _fa().fa_decode_splitkv(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, num_splits=n, scale=scale)
    compare(o, l, o_ref, l_ref, what=str(case))


def test_split_matches_unsplit():
    """Cutting the keys into ranges changes only rounding ("any split is exact")."""
    fa = _fa()
    B, Hq, Hkv, T, S, d = 1, 2, 2, 2048, 2048, 128
    q, k, v = (t.to(DEV) for t in fi.qkv(B, Hq, Hkv, T, S, d, 120))
    o1, l1 = fa.fa_fwd(q, k, v, causal=True)
    o8, l8 = fa.fa_decode_splitkv(q, k, v, causal=True, num_splits=8)
    assert float((o1.float() - o8.float()).abs().max()) < 1e-2
    assert float((l1 - l8).abs().max()) < 1e-3
    assert torch.equal(torch.isinf(l1), torch.isinf(l8))


@pytest.mark.parametrize("N,d", fi.PREFILL_MHA.sweep)
def test_one_head_sweep_split(N, d):
    """The prefill workload's one-head sweep, keys split by the heuristic; sampled rows."""
    fa = _fa()
    q, k, v = fi.qkv(1, 1, 1, N, N, d, 10 + d // 64)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n = fa.fa_num_splits_prefill(1, 1, 1, N, N, sms)
    assert n > 1
    scale = 1.0 / math.sqrt(d)
    o, l = fa.fa_decode_splitkv(q.to(DEV), k.to(DEV), v.to(DEV), causal=False, num_splits=0, scale=scale)
    rows = fi.sample_rows(1, 1, N, 512, 7)
    o_ref, l_ref = oracle.attention_rows(q, k, v, rows, scale, False)
    idx = torch.tensor(rows)
    compare(o.cpu()[idx[:, 0], idx[:, 1], idx[:, 2]], l.cpu()[idx[:, 0], idx[:, 1], idx[:, 2]], o_ref, l_ref,
            what=f"sweep {N} x {d}, {n} ranges")
