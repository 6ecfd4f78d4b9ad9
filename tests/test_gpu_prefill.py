"""Parity of the prefill kernels (tcgen05 bf16 and fp32 SIMT) with the fp64 oracle."""

import math

import numpy as np
import pytest
import torch

import fa_inputs as fi
import oracle
from parity import compare, compare_f32

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import attention_fa2_attn_gb300 as fa

    return fa


def _fa():
    import attention_fa2_attn_gb300 as fa

    return fa


def test_smoke_fp32_and_bf16():
    w = fi.SMOKE
    q, k, v = fi.qkv(w.B, w.Hq, w.Hkv, w.T, w.S, w.d, w.index, dtype=torch.float32)
    o_ref, l_ref = oracle.attention_three_pass(q, k, v, w.scale, w.causal)
    o, l = _fa().fa_fwd_f32(q.to(DEV), k.to(DEV), v.to(DEV), causal=w.causal, scale=w.scale)
    compare_f32(o, l, o_ref, l_ref, what="smoke fp32")
    qb, kb, vb = q.bfloat16(), k.bfloat16(), v.bfloat16()
    o_ref, l_ref = oracle.attention_three_pass(qb, kb, vb, w.scale, w.causal)
    o, l = _fa().fa_fwd(qb.to(DEV), kb.to(DEV), vb.to(DEV), causal=w.causal, scale=w.scale)
    compare(o, l, o_ref, l_ref, what="smoke bf16")


CASES = [
    # B, Hq, Hkv, T, S, d, causal
    (1, 2, 2, 300, 300, 128, False),
    (1, 2, 2, 300, 300, 128, True),
    (2, 4, 1, 200, 333, 64, True),
    (1, 8, 1, 130, 517, 128, True),
    (1, 4, 2, 257, 129, 128, True),  # T > S: the first rows see no key
    (1, 16, 1, 64, 64, 64, False),
    (1, 2, 2, 1, 700, 128, True),
    (1, 1, 1, 5, 3, 64, False),
    (2, 4, 2, 384, 256, 64, False),
    (1, 8, 4, 512, 512, 128, True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}_Hq{}_Hkv{}_T{}_S{}_d{}_{}".format(*c[:6], "causal" if c[6] else "full"))
def test_prefill_small(case):
    B, Hq, Hkv, T, S, d, causal = case
    q, k, v = fi.qkv(B, Hq, Hkv, T, S, d, 50 + T % 7)
    scale = 1.0 / math.sqrt(d)
    o_ref, l_ref = oracle.attention_three_pass(q, k, v, scale, causal)
    o, l = _fa().fa_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, scale=scale)
    compare(o, l, o_ref, l_ref, what=str(case))
    # the fp32 path on the same values (upcast), to 1e-5
    o32, l32 = _fa().fa_fwd_f32(q.float().to(DEV), k.float().to(DEV), v.float().to(DEV), causal=causal, scale=scale)
    compare_f32(o32, l32, o_ref, l_ref, what=str(case) + " fp32")


@pytest.mark.parametrize("case", [(1, 4, 4, 700, 700, 128, True), (2, 8, 2, 333, 1000, 64, True), (1, 2, 2, 900, 300, 64, True)])
def test_visible_key_count_is_exact(case):
    """q = 0 makes every visible score equal, so lse = ln(#visible keys): the
    count recovered from the GPU's lse must equal the mask's, bit for bit."""
    B, Hq, Hkv, T, S, d, causal = case
    q = torch.zeros(B, Hq, T, d, dtype=torch.bfloat16)
    _, k, v = fi.qkv(B, Hq, Hkv, T, S, d, 77)
    _, l = _fa().fa_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, scale=0.1)
    l = l.cpu().double().numpy()
    vis = oracle.causal_mask(T, S, causal).sum(axis=1)
    cnt = np.where(np.isfinite(l), np.rint(np.exp(l)), 0).astype(np.int64)
    for b in range(B):
        for h in range(Hq):
            assert np.array_equal(cnt[b, h], vis), (b, h)


def test_worked_softmax_123_on_gpu():
    """Scores 1, 2, 3 (exact in bf16) and V = identity rows: O is the softmax itself."""
    d = 64
    q = torch.zeros(1, 1, 1, d)
    q[0, 0, 0, 0] = 1.0
    k = torch.zeros(1, 1, 3, d)
    k[0, 0, :, 0] = torch.tensor([1.0, 2.0, 3.0])
    v = torch.zeros(1, 1, 3, d)
    v[0, 0, 0, 0] = v[0, 0, 1, 1] = v[0, 0, 2, 2] = 1.0
    o, l = _fa().fa_fwd(q.bfloat16().to(DEV), k.bfloat16().to(DEV), v.bfloat16().to(DEV), scale=1.0)
    got = o[0, 0, 0, :3].float().cpu().numpy()
    assert np.allclose(got, [0.090, 0.245, 0.665], atol=1e-2)
    assert abs(float(l[0, 0, 0]) - math.log(math.e + math.e**2 + math.e**3)) < 1e-3


def test_large_scores_stay_finite():
    """Scores near +-1000 overflow a softmax without the max subtracted."""
    B, Hq, Hkv, T, S, d = 1, 2, 2, 128, 256, 64
    q, k, v = fi.qkv(B, Hq, Hkv, T, S, d, 91)
    q = (q.float() * 120).bfloat16()  # |score| up to ~1000 at scale 1/8
    scale = 0.125
    o_ref, l_ref = oracle.attention_three_pass(q, k, v, scale, True)
    o, l = _fa().fa_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, scale=scale)
    assert float(np.abs(l_ref[np.isfinite(l_ref)]).max()) > 300
    # Scores this large make P nearly one-hot, so O is close to single V rows
    # (|v| up to ~4): a mismatch between the rounded P of the P V product and the
    # sum that normalises O would show here at the standard bounds.
    compare(o, l, o_ref, l_ref, what="large scores")


def _sampled_check(w, n_rows, seed):
    q, k, v = fi.qkv(w.B, w.Hq, w.Hkv, w.T, w.S, w.d, w.index)
    o, l = _fa().fa_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=w.causal, scale=w.scale)
    rows = fi.sample_rows(w.B, w.Hq, w.T, n_rows, seed)
    o_ref, l_ref = oracle.attention_rows(q, k, v, rows, w.scale, w.causal)
    idx = torch.tensor(rows)
    og = o.cpu()[idx[:, 0], idx[:, 1], idx[:, 2]]
    lg = l.cpu()[idx[:, 0], idx[:, 1], idx[:, 2]]
    return compare(og, lg, o_ref, l_ref, what=w.name)


def test_prefill_mha_full_size_sampled():
    _sampled_check(fi.PREFILL_MHA, 2048, 5)


def test_causal_gqa_full_size_sampled():
    _sampled_check(fi.CAUSAL_GQA, 2048, 6)


def test_prefill_mha_d64_full_size_sampled():
    """The prefill workload's shapes at head dimension 64 (B=4, H=16, N=4096,
    non-causal), the d = 64 instantiation in the launch configuration it is timed in."""
    w = fi.PREFILL_MHA
    _sampled_check(fi.Workload(w.name.replace("d128", "d64"), w.index, w.B, w.Hq, w.Hkv, w.T, w.S, 64, False),
                   2048, 8)


@pytest.mark.parametrize("N,d", fi.PREFILL_MHA.sweep)
def test_one_head_sweep_sampled(N, d):
    w = fi.Workload(f"sweep_{N}_{d}", 10 + d // 64, 1, 1, 1, N, N, d, False)
    _sampled_check(w, 512, 7)


def test_failure_detection_wait_times_out():
    """A bounded wait on a barrier nothing arrives on must report FA_ERR_TIMEOUT
    and leave the context usable."""
    fa = _fa()
    assert fa.fa_get_last_device_error()[0] == 0
    fa.fa_selftest_wait_timeout(20_000_000)  # 20 ms
    st, word = fa.fa_get_last_device_error()
    assert st == 4 and (word & 0xFF) == 4 and (word >> 8) == 1
    assert fa.fa_get_last_device_error()[0] == 0  # cleared
    # the context still works
    test_smoke_fp32_and_bf16()


def test_api_errors_raise():
    fa = _fa()
    q = torch.zeros(1, 3, 8, 128, dtype=torch.bfloat16, device=DEV)
    k = torch.zeros(1, 2, 8, 128, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(fa.FAError):
        fa.fa_fwd(q, k, k)
    q = torch.zeros(1, 2, 8, 96, dtype=torch.bfloat16, device=DEV)
    k = torch.zeros(1, 2, 8, 96, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(fa.FAError):
        fa.fa_fwd(q, k, k)


def test_binding_rejects_mismatched_tensors():
    """The library takes every size from q and k and writes outputs through bare
    pointers, so the binding refuses, before any launch, tensors whose shapes would
    let it read or write past an allocation."""
    fa = _fa()
    bf = dict(dtype=torch.bfloat16, device=DEV)
    q = torch.zeros(2, 4, 64, 64, **bf)
    k = torch.zeros(2, 2, 96, 64, **bf)
    bad = [
        lambda: fa.fa_fwd(q, k, torch.zeros(2, 2, 48, 64, **bf)),                     # v shorter than k
        lambda: fa.fa_fwd(torch.zeros(1, 4, 64, 64, **bf), k, k),                       # batch differs
        lambda: fa.fa_fwd(q, k, k, out=torch.zeros(2, 4, 32, 64, **bf)),               # out too small
        lambda: fa.fa_fwd(q, k, k, out=torch.zeros(2, 4, 64, 64, dtype=torch.float32, device=DEV)),
        lambda: fa.fa_fwd(q, k, k, lse=torch.zeros(2, 4, 63, device=DEV)),              # lse too small
        lambda: fa.fa_fwd(q, k, k, out=torch.zeros(2, 4, 64, 128, **bf)[..., ::2]),     # strided out
        lambda: fa.fa_decode_splitkv(q[:, :, :1], k, k, out=torch.zeros(2, 4, 2, 64, **bf)),
        lambda: fa.fa_fwd_kv_outer(q, k, torch.zeros(2, 2, 96, 32, **bf)),
        lambda: fa.fa_bwd(q, k, k, q, torch.zeros(2, 4, 64, device=DEV), torch.zeros(2, 4, 32, 64, **bf)),
        lambda: fa.fa_bwd(q, k, k, q, torch.zeros(2, 4, 64, device=DEV), q, dk=torch.zeros(2, 2, 95, 64, **bf)),
        lambda: fa.fa_decode_paged(q[:, :, :1], torch.zeros(10, 16, 2, 64, **bf), torch.zeros(10, 16, 2, 64, **bf),
                                   torch.zeros(3, 5, dtype=torch.int32, device=DEV),
                                   torch.zeros(2, dtype=torch.int32, device=DEV)),        # table rows != batch
    ]
    for i, call in enumerate(bad):
        with pytest.raises(ValueError):
            call()
    st, word = fa.fa_get_last_device_error()
    assert st == 0, hex(word)
