"""Parity of the backward kernels (dQ, dK, dV) with the fp64 oracle.

The backward's inputs are q, k, v, dO and the forward's saved O and LSE; the
oracle gets the same saved O (bf16) and LSE (fp32) the kernels read, so the
comparison measures the backward alone. Tolerances (per gradient tensor G,
relative to its largest magnitude): max |err| <= 2e-2 * max|G_ref|, mean
|err| <= 2e-3 * max|G_ref|. The kernels round P and dS to bf16 before the
tensor-core products (relative 2^-9 each) and the results to bf16 (another
2^-9); with fp32 accumulation the error stays a small multiple of 2^-9 of the
largest entry.
"""

import math

import numpy as np
import pytest
import torch

import fa_inputs as fi
import oracle

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
MAX_REL = 2e-2
MEAN_REL = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _fa():
    import attention_fa2_attn_gb300 as fa

    return fa


def _grad_compare(got, ref, what):
    got = got.detach().float().cpu().double().numpy()
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite"
    scale = max(float(np.abs(ref).max()), 1e-30)
    err = np.abs(got - ref)
    assert err.max() <= MAX_REL * scale, f"{what}: max |err| {err.max():.3e} > {MAX_REL} * {scale:.3e}"
    assert err.mean() <= MEAN_REL * scale, f"{what}: mean |err| {err.mean():.3e} > {MEAN_REL} * {scale:.3e}"
    return float(err.max() / scale)


def _problem(B, Hq, Hkv, T, S, d, causal, seed):
    q, k, v = fi.qkv(B, Hq, Hkv, T, S, d, seed)
    do = fi.randn((B, Hq, T, d), 5000 + seed)
    scale = 1.0 / math.sqrt(d)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = _fa().fa_fwd(qd, kd, vd, causal=causal, scale=scale)
    return q, k, v, do, scale, qd, kd, vd, dod, o, lse


CASES = [
    # B, Hq, Hkv, T, S, d, causal
    (1, 1, 1, 128, 128, 64, False),
    (1, 2, 2, 200, 300, 128, True),
    (2, 4, 2, 130, 257, 64, True),  # GQA 2, ragged tiles
    (1, 8, 1, 64, 512, 128, True),  # GQA 8: 16 positions x 8 heads per tile
    (1, 4, 4, 257, 129, 128, True),  # T > S: rows with no visible key
    (1, 16, 1, 100, 100, 64, False),  # GQA 16
    (2, 2, 2, 384, 384, 128, False),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}_Hq{}_Hkv{}_T{}_S{}_d{}_{}".format(*c[:6], "causal" if c[6] else "full"))
def test_backward_small(case):
    B, Hq, Hkv, T, S, d, causal = case
    q, k, v, do, scale, qd, kd, vd, dod, o, lse = _problem(B, Hq, Hkv, T, S, d, causal, 130 + T % 17)
    dq, dk, dv = _fa().fa_bwd(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    rq, rk, rv = oracle.attention_backward(q, k, v, do, scale, causal, o=o.float().cpu(), lse=lse.cpu())
    _grad_compare(dq, rq, f"{case} dq")
    _grad_compare(dk, rk, f"{case} dk")
    _grad_compare(dv, rv, f"{case} dv")


def test_backward_full_size_sampled():
    """The prefill workload's shapes (B=4, H=16, N=4096, d=128, non-causal): dQ rows
    and dK/dV rows sampled, each computed exactly by the oracle over all keys or
    all queries of its head."""
    w = fi.PREFILL_MHA
    q, k, v = fi.qkv(w.B, w.Hq, w.Hkv, w.T, w.S, w.d, w.index)
    do = fi.randn((w.B, w.Hq, w.T, w.d), 5000 + w.index)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = _fa().fa_fwd(qd, kd, vd, causal=w.causal, scale=w.scale)
    dq, dk, dv = _fa().fa_bwd(qd, kd, vd, o, lse, dod, causal=w.causal, scale=w.scale)
    qrows = fi.sample_rows(w.B, w.Hq, w.T, 256, 21)
    krows = fi.sample_rows(w.B, w.Hkv, w.S, 256, 22)
    rq, rk, rv = oracle.attention_backward_rows(q, k, v, do, o.float().cpu(), lse.cpu(), qrows, krows, w.scale,
                                                w.causal)
    iq, ik = torch.tensor(qrows), torch.tensor(krows)
    _grad_compare(dq.cpu()[iq[:, 0], iq[:, 1], iq[:, 2]], rq, "dq rows")
    _grad_compare(dk.cpu()[ik[:, 0], ik[:, 1], ik[:, 2]], rk, "dk rows")
    _grad_compare(dv.cpu()[ik[:, 0], ik[:, 1], ik[:, 2]], rv, "dv rows")


def test_backward_causal_gqa_sampled():
    """The causal GQA workload's shapes (B=1, Hq=64, Hkv=8, N=8192, d=128), sampled rows."""
    w = fi.CAUSAL_GQA
    q, k, v = fi.qkv(w.B, w.Hq, w.Hkv, w.T, w.S, w.d, w.index)
    do = fi.randn((w.B, w.Hq, w.T, w.d), 5000 + w.index)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = _fa().fa_fwd(qd, kd, vd, causal=True, scale=w.scale)
    dq, dk, dv = _fa().fa_bwd(qd, kd, vd, o, lse, dod, causal=True, scale=w.scale)
    qrows = fi.sample_rows(w.B, w.Hq, w.T, 128, 23)
    krows = fi.sample_rows(w.B, w.Hkv, w.S, 128, 24)
    rq, rk, rv = oracle.attention_backward_rows(q, k, v, do, o.float().cpu(), lse.cpu(), qrows, krows, w.scale, True)
    iq, ik = torch.tensor(qrows), torch.tensor(krows)
    _grad_compare(dq.cpu()[iq[:, 0], iq[:, 1], iq[:, 2]], rq, "dq rows")
    _grad_compare(dk.cpu()[ik[:, 0], ik[:, 1], ik[:, 2]], rk, "dk rows")
    _grad_compare(dv.cpu()[ik[:, 0], ik[:, 1], ik[:, 2]], rv, "dv rows")


def test_backward_api_errors():
    fa = _fa()
    q = torch.zeros(1, 2, 8, 128, dtype=torch.bfloat16, device=DEV)
    lse = torch.zeros(1, 2, 8, device=DEV)
    with pytest.raises(ValueError):
        fa.fa_bwd(q, q, q, q, lse, q, workspace=torch.empty(4, dtype=torch.uint8, device=DEV))
    q96 = torch.zeros(1, 2, 8, 96, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(fa.FAError):
        fa.fa_bwd(q96, q96, q96, q96, lse, q96)


def test_backward_workspace_needs_no_initialisation_and_is_deterministic():
    """The row pass writes every value the two passes read (positions past T come in
    as zeros from the tensor map's bounds), so a NaN-filled workspace changes nothing;
    no atomics are involved, so a repeat gives the same bits."""
    fa = _fa()
    B, Hq, Hkv, T, S, d = 2, 8, 2, 301, 450, 128  # T not a multiple of 4: padded rows
    q, k, v, do, scale, qd, kd, vd, dod, o, lse = _problem(B, Hq, Hkv, T, S, d, True, 141)
    n = fa.fa_bwd_workspace_bytes(B, Hq, T)
    ws_nan = torch.full((n // 4,), float("nan"), dtype=torch.float32, device=DEV)
    g1 = fa.fa_bwd(qd, kd, vd, o, lse, dod, causal=True, scale=scale, workspace=ws_nan.view(torch.uint8))
    g2 = fa.fa_bwd(qd, kd, vd, o, lse, dod, causal=True, scale=scale)
    for a, b_ in zip(g1, g2):
        assert torch.equal(a, b_)
    rq, rk, rv = oracle.attention_backward(q, k, v, do, scale, True, o=o.float().cpu(), lse=lse.cpu())
    _grad_compare(g1[0], rq, "dq")
    _grad_compare(g1[1], rk, "dk")
    _grad_compare(g1[2], rv, "dv")
