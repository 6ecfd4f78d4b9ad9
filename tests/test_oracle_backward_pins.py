"""Pins of the fp64 backward oracle (CPU only).

The oracle writes the gradients of O = softmax(scale * Q K^T) V out by the chain
rule with P rebuilt from the saved log-sum-exp and D = rowsum(dO * O)
("Attention kernel chains", "What the backward pass saves"). These checks pin it
to things other than its own formulas:
  * central finite differences of L = sum(dO * O), O from the (separately pinned)
    three-pass forward;
  * torch autograd of the plain forward definition, in fp64;
  * closed forms: one key (softmax constant: dQ = dK = 0, dV = sum of dO),
    identical value rows (O independent of the weights: dQ = dK = 0);
and ``test_planted_backward_mistakes_are_caught`` plants plausible mistakes in the
oracle and asserts some pin fails for each.
"""

import numpy as np
import pytest

import oracle
import oracle.attention as oa


def _problem(B, Hq, Hkv, T, S, d, seed):
    r = np.random.default_rng(seed)
    return (r.standard_normal((B, Hq, T, d)), r.standard_normal((B, Hkv, S, d)), r.standard_normal((B, Hkv, S, d)),
            r.standard_normal((B, Hq, T, d)))


def _loss(q, k, v, do, scale, causal):
    o, _ = oracle.attention_three_pass(q, k, v, scale, causal)
    return float((o * do).sum())


def check_backward_finite_differences():
    # GQA group 2, bottom-right causal with T < S, and T > S (rows that see no key)
    for (B, Hq, Hkv, T, S, d, causal, seed) in ((1, 2, 1, 3, 5, 3, True, 1), (1, 2, 2, 4, 2, 2, True, 2),
                                                 (2, 1, 1, 2, 3, 2, False, 3)):
        q, k, v, do = _problem(B, Hq, Hkv, T, S, d, seed)
        scale = 0.7
        dq, dk, dv = oracle.attention_backward(q, k, v, do, scale, causal)
        eps = 1e-6
        for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            for idx in np.ndindex(x.shape):
                old = x[idx]
                x[idx] = old + eps
                lp = _loss(q, k, v, do, scale, causal)
                x[idx] = old - eps
                lm = _loss(q, k, v, do, scale, causal)
                x[idx] = old
                fd = (lp - lm) / (2 * eps)
                assert abs(fd - g[idx]) < 1e-7 * max(1.0, abs(fd)), (name, idx, fd, g[idx])


def check_backward_autograd():
    torch = pytest.importorskip("torch")
    B, Hq, Hkv, T, S, d = 2, 4, 2, 5, 7, 6
    q, k, v, do = _problem(B, Hq, Hkv, T, S, d, 4)
    scale = 0.4
    for causal in (False, True):
        tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
        g = Hq // Hkv
        kr, vr = tk.repeat_interleave(g, dim=1), tv.repeat_interleave(g, dim=1)
        x = scale * tq @ kr.transpose(-1, -2)
        if causal:
            i = torch.arange(T)[:, None]
            j = torch.arange(S)[None, :]
            x = x.masked_fill(j > i + (S - T), float("-inf"))
        o = torch.softmax(x, dim=-1) @ vr
        (o * torch.tensor(do)).sum().backward()
        dq, dk, dv = oracle.attention_backward(q, k, v, do, scale, causal)
        for got, ref in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
            assert np.allclose(got, ref.numpy(), atol=1e-12, rtol=1e-12)


def check_backward_closed_forms():
    # one key: P = 1 whatever the scores, so dQ = dK = 0 and dV = sum over the group's rows of dO
    q, k, v, do = _problem(1, 2, 1, 4, 1, 3, 5)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.9, False)
    assert np.abs(dq).max() < 1e-14 and np.abs(dk).max() < 1e-14
    assert np.allclose(dv[0, 0, 0], do[0].sum(axis=(0, 1)), atol=1e-13)
    # identical value rows: O = v whatever P is, so dQ = dK = 0
    q, k, v, do = _problem(1, 1, 1, 3, 6, 4, 6)
    v[:] = v[:, :, :1, :]
    dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.5, True)
    assert np.abs(dq).max() < 1e-13 and np.abs(dk).max() < 1e-13
    # a row with no visible key (causal, T > S) takes no gradient
    q, k, v, do = _problem(1, 1, 1, 4, 2, 3, 7)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.5, True)
    assert np.all(dq[0, 0, :2] == 0.0)


BACKWARD_CHECKS = [check_backward_finite_differences, check_backward_autograd, check_backward_closed_forms]


@pytest.mark.parametrize("check", BACKWARD_CHECKS, ids=lambda c: c.__name__)
def test_backward_pin(check):
    check()


def test_backward_rowsum():
    r = np.random.default_rng(8)
    do, o = r.standard_normal((2, 3, 4, 5)), r.standard_normal((2, 3, 4, 5))
    d = oracle.backward_rowsum(do, o)
    assert d.shape == (2, 3, 4)
    assert abs(d[1, 2, 3] - sum(do[1, 2, 3, c] * o[1, 2, 3, c] for c in range(5))) < 1e-14


def test_planted_backward_mistakes_are_caught(monkeypatch):
    """Each plausible mistake, planted in the backward oracle, makes a pin fail."""
    mistakes = {
        "D left out": lambda mp: mp.setattr(oa, "_softmax_grad", lambda p, dp, dsum: p * dp),
        "P not normalised": lambda mp: mp.setattr(
            oa, "_bwd_probs", lambda x, lse, vis: np.where(vis, np.exp(x - np.max(np.where(vis, x, -np.inf), axis=1, keepdims=True)), 0.0)),
        "dK without the scale": lambda mp: mp.setattr(oa, "_score_grads", lambda ds, q, k, scale: (scale * (ds @ k), ds.T @ q)),
        "dQ and dK swapped roles": lambda mp: mp.setattr(oa, "_score_grads", lambda ds, q, k, scale: (scale * (ds @ k), scale * (ds.T @ k))),
        "gqa h % Hkv": lambda mp: mp.setattr(oa, "kv_head_of", lambda h, Hq, Hkv: h % Hkv),
    }
    for name, plant in mistakes.items():
        with monkeypatch.context() as mp:
            plant(mp)
            failed = False
            for c in BACKWARD_CHECKS:
                try:
                    c()
                except (AssertionError, ValueError, IndexError):
                    failed = True
                    break
            assert failed, f"planted mistake not caught: {name}"


def test_backward_rows_match_full():
    """The sampled-row backward equals the full one on the rows it computes."""
    for causal in (False, True):
        q, k, v, do = _problem(2, 4, 2, 9, 7, 5, 9)
        o, lse = oracle.attention_three_pass(q, k, v, 0.6, causal)
        dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.6, causal, o=o, lse=lse)
        qrows = [(0, 0, 0), (1, 3, 8), (0, 2, 4), (1, 1, 1)]
        krows = [(0, 0, 0), (1, 1, 6), (0, 1, 3)]
        rq, rk, rv = oracle.attention_backward_rows(q, k, v, do, o, lse, qrows, krows, 0.6, causal)
        for n, (b, h, i) in enumerate(qrows):
            assert np.allclose(rq[n], dq[b, h, i], atol=1e-13)
        for n, (b, hk, j) in enumerate(krows):
            assert np.allclose(rk[n], dk[b, hk, j], atol=1e-13)
            assert np.allclose(rv[n], dv[b, hk, j], atol=1e-13)
