"""Every entry point at softmax scales other than 1/sqrt(d).

The scale multiplies the scores before the softmax ("Softmax and FlashAttention",
"Concept": S = Q K^T scaled); the kernels fold scale * log2(e) into one constant
of the base-2 exponent. With N(0, 1) inputs at d = 128, scale 0.02 makes every row
nearly uniform, and 1.7 spreads a row's scores over about +-20, so nearly every row
is close to one-hot and the running max climbs often. Each case is compared with
the fp64 oracle at the standard bounds.

V is drawn at 0.25 * N(0, 1) (exact in bf16). With nearly one-hot rows O is close to
a single V row, and at |O| >= 4 half a bf16 ulp of O (0.0156) alone exceeds the 1e-2
bound on O; at a quarter of the size O stays below about 1.2, where that rounding
is at most 0.0039 and the bound measures the computation.
"""

import pytest
import torch

import fa_inputs as fi
import oracle
from parity import compare
from test_gpu_backward import _grad_compare  # the backward's bounds, relative to each gradient's largest entry

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
SCALES = (0.02, 0.5, 1.7)
V_SCALE = 0.25


def _qkv(B, Hq, Hkv, T, S, d, seed):
    q, k, v = fi.qkv(B, Hq, Hkv, T, S, d, seed)
    return q, k, (v.float() * V_SCALE).bfloat16()


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _fa():
    import attention_fa2_attn_gb300 as fa

    return fa


@pytest.mark.parametrize("scale", SCALES)
@pytest.mark.parametrize("d,causal", [(128, False), (64, True)])
def test_prefill_scales(scale, d, causal):
    B, Hq, Hkv, T, S = 1, 4, 2, 300, 700
    q, k, v = _qkv(B, Hq, Hkv, T, S, d, 950 + d)
    o_ref, l_ref = oracle.attention_three_pass(q, k, v, scale, causal)
    o, l = _fa().fa_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, scale=scale)
    compare(o, l, o_ref, l_ref, what=f"prefill scale {scale}")


@pytest.mark.parametrize("scale", SCALES)
def test_decode_and_key_split_scales(scale):
    """The decode kernel (one token, 5 ranges) and the prefill kernel's key split
    (40 stacked rows per KV head, 3 ranges)."""
    fa = _fa()
    q, k, v = _qkv(2, 8, 2, 1, 3000, 128, 960)
    o_ref, l_ref = oracle.attention_three_pass(q, k, v, scale, True)
    o, l = fa.fa_decode_splitkv(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, num_splits=5, scale=scale)
    compare(o, l, o_ref, l_ref, what=f"decode scale {scale}")
    q, k, v = _qkv(1, 8, 2, 10, 1500, 64, 961)
    o_ref, l_ref = oracle.attention_three_pass(q, k, v, scale, True)
    o, l = fa.fa_decode_splitkv(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, num_splits=3, scale=scale)
    compare(o, l, o_ref, l_ref, what=f"key split scale {scale}")


@pytest.mark.parametrize("scale", SCALES)
@pytest.mark.parametrize("T", [1, 50])
def test_paged_scales(scale, T):
    """Paged decode (T = 1) and the chunked prefill over the cache (T = 50, 100 rows
    per KV head), ragged sequence lengths."""
    B, Hq, Hkv, S, d = 3, 4, 2, 1100, 128
    k_pages, v_pages, table, _ = fi.paged_kv(B, Hkv, S, d, 16, 970)
    v_pages = (v_pages.float() * V_SCALE).bfloat16()
    q = fi.decode_q(B, Hq, T, d, 971 + T)
    sl = torch.tensor([S, 517, 64], dtype=torch.int32)
    o_ref, l_ref = oracle.decode_paged(q, k_pages, v_pages, table, sl, 16, scale, True)
    o, l = _fa().fa_decode_paged(q.to(DEV), k_pages.to(DEV), v_pages.to(DEV), table.to(DEV), sl.to(DEV),
                                 causal=True, scale=scale)
    compare(o, l, o_ref, l_ref, what=f"paged T{T} scale {scale}")


@pytest.mark.parametrize("scale", SCALES)
def test_kv_outer_scales(scale):
    B, Hq, Hkv, T, S, d = 1, 2, 2, 260, 400, 128
    q, k, v = _qkv(B, Hq, Hkv, T, S, d, 980)
    o_ref, l_ref = oracle.attention_online_normalized(q, k, v, scale, True, block=128)
    o, l = _fa().fa_fwd_kv_outer(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, scale=scale)
    compare(o, l, o_ref, l_ref, what=f"kv_outer scale {scale}")


@pytest.mark.parametrize("scale", SCALES)
def test_backward_scales(scale):
    B, Hq, Hkv, T, S, d = 1, 4, 2, 200, 330, 128
    q, k, v = _qkv(B, Hq, Hkv, T, S, d, 990)
    do = fi.randn((B, Hq, T, d), 991)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    fa = _fa()
    o, lse = fa.fa_fwd(qd, kd, vd, causal=True, scale=scale)
    dq, dk, dv = fa.fa_bwd(qd, kd, vd, o, lse, dod, causal=True, scale=scale)
    rq, rk, rv = oracle.attention_backward(q, k, v, do, scale, True, o=o.float().cpu(), lse=lse.cpu())
    _grad_compare(dq, rq, f"dq scale {scale}")
    _grad_compare(dk, rk, f"dk scale {scale}")
    _grad_compare(dv, rv, f"dv scale {scale}")
