"""Pins of the fp64 oracle to what the pages and the mathematics fix (CPU only).

Each ``check_*`` function raises AssertionError on a mismatch. The tests call
them on the oracle as written, and ``test_planted_mistakes_are_caught`` plants
plausible mistakes in the oracle (a wrong GQA map, a top-left mask, a dropped
scale, swapped K/V) and asserts that some pin fails for each.
"""

import json
import math
import os
from decimal import Decimal, getcontext

import numpy as np
import pytest

import oracle
import oracle.attention as oa

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_worked_examples.json")))


def _scores_123_problem():
    """q, k, v whose scaled scores are 1, 2, 3 and whose V is the identity,
    so the output row is the softmax weights themselves."""
    q = np.zeros((1, 1, 1, 3))
    q[0, 0, 0, 0] = 1.0
    k = np.zeros((1, 1, 3, 3))
    k[0, 0, :, 0] = [1.0, 2.0, 3.0]
    v = np.eye(3).reshape(1, 1, 3, 3)
    return q, k, v


# --------------------------------------------------------------------------- #
# Worked numbers printed on the pages
# --------------------------------------------------------------------------- #
def check_softmax_123():
    g = GOLDEN["softmax_123"]
    q, k, v = _scores_123_problem()
    for fn in (oracle.attention_three_pass, oracle.attention_online, oracle.attention_online_normalized):
        o, lse = fn(q, k, v, 1.0, False) if fn is oracle.attention_three_pass else fn(q, k, v, 1.0, False, 2)
        assert np.allclose(o[0, 0, 0], g["weights"], atol=g["tol"]), (fn.__name__, o[0, 0, 0])


def check_online_trace():
    g = GOLDEN["online_trace"]
    q, k, v = _scores_123_problem()
    seen = []
    o, _ = oracle.attention_online(q, k, v, 1.0, False, block=2, trace=lambda bh, i, m, l, a: seen.append((m[0], l[0], a[0])))
    assert len(seen) == 2
    (m1, l1, _), (m2, l2, a2) = seen
    t = g["tol"]
    assert abs(m1 - g["after_block_1"]["m"]) < t and abs(l1 - g["after_block_1"]["l"]) < t, seen
    assert abs(m2 - g["after_block_2"]["m"]) < t, seen
    assert abs(a2 - g["after_block_2"]["alpha"]) < t, seen
    assert abs(l2 - g["after_block_2"]["l"]) < t, seen
    assert abs(o[0, 0, 0, 2] - g["weight_of_3"]) < t


def check_lse_merge_worked():
    g = GOLDEN["lse_merge"]
    q, k, v = _scores_123_problem()
    op, lp = oracle.attention_partials(q, k, v, 1.0, False, num_splits=2)  # keys [1,2] | [3]
    t = g["tol"]
    assert np.allclose(lp[:, 0, 0, 0], g["lse_parts"], atol=t), lp[:, 0, 0, 0]
    o, lse = oracle.lse_merge(op, lp)
    assert abs(lse[0, 0, 0] - g["lse"]) < t, lse
    # V is the identity: the first worker's share is O[0] + O[1], the second's is O[2]
    w1 = o[0, 0, 0, 0] + o[0, 0, 0, 1]
    w2 = o[0, 0, 0, 2]
    assert abs(w1 - g["weights"][0]) < t and abs(w2 - g["weights"][1]) < t, (w1, w2)
    sm = GOLDEN["softmax_123"]["weights"]
    assert abs(w1 - (sm[0] + sm[1])) < 2 * t  # "0.335 is 0.090 + 0.245"


def check_causal_decode():
    g = GOLDEN["causal_decode"]
    T, S = g["T"], g["S"]
    m = oracle.causal_mask(T, S, True)
    vis = np.nonzero(m[0])[0]
    assert vis[0] == g["visible_first"] and vis[-1] == g["visible_last"] and len(vis) == S
    # the top-left alignment the page warns against sees key 0 only
    top_left = np.tril(np.ones((T, S), dtype=bool))
    assert top_left[0].sum() == g["top_left_visible_count"]
    assert not np.array_equal(m, top_left)


# --------------------------------------------------------------------------- #
# Mask rule by enumeration, for every small (T, S)
# --------------------------------------------------------------------------- #
def check_mask_enumeration():
    for T in range(1, 7):
        for S in range(1, 7):
            m = oracle.causal_mask(T, S, True)
            # query i is the (S - T + i)-th position of the sequence; it sees its own
            # position and every earlier one, and nothing before position 0 exists.
            for i in range(T):
                pos = S - T + i
                want = [0 <= j <= pos for j in range(S)]
                assert list(m[i]) == want, (T, S, i)
                assert oracle.visible(i, S - 1, T, S, True) == (i == T - 1 or pos >= S - 1)
            if T == S:  # square case: the textbook lower triangle
                assert np.array_equal(m, np.tril(np.ones((T, S), dtype=bool)))
            assert oracle.causal_mask(T, S, False).all()


# --------------------------------------------------------------------------- #
# Exactness of the online forms and of any split
# --------------------------------------------------------------------------- #
def _rand_problem(seed, B, Hq, Hkv, T, S, d, scale_q=1.0):
    r = np.random.default_rng(seed)
    q = r.standard_normal((B, Hq, T, d)) * scale_q
    k = r.standard_normal((B, Hkv, S, d))
    v = r.standard_normal((B, Hkv, S, d))
    return q, k, v


def check_online_equals_three_pass():
    tol = GOLDEN["online_exactness"]["assert_rel"]
    for seed, (B, Hq, Hkv, T, S, d) in enumerate([(1, 2, 1, 37, 200, 16), (2, 4, 2, 64, 64, 8), (1, 1, 1, 5, 300, 3)]):
        q, k, v = _rand_problem(seed, B, Hq, Hkv, T, S, d)
        for causal in (False, True):
            o3, l3 = oracle.attention_three_pass(q, k, v, 0.3, causal)
            for block in (1, 7, 64, 1000):
                o1, l1 = oracle.attention_online(q, k, v, 0.3, causal, block)
                o2, l2 = oracle.attention_online_normalized(q, k, v, 0.3, causal, block)
                for o, l in ((o1, l1), (o2, l2)):
                    assert np.all(np.abs(o - o3) <= tol * (1 + np.abs(o3))), (causal, block)
                    fin = np.isfinite(l3)
                    assert np.array_equal(fin, np.isfinite(l))
                    assert np.all(np.abs(l[fin] - l3[fin]) <= tol * (1 + np.abs(l3[fin])))


def check_split_invariance():
    for seed, (T, S) in enumerate([(3, 50), (1, 17), (8, 8), (10, 4)]):
        q, k, v = _rand_problem(100 + seed, 1, 4, 2, T, S, 8)
        for causal in (False, True):
            o3, l3 = oracle.attention_three_pass(q, k, v, 0.5, causal)
            for n in (1, 2, 3, 5, 16, 64):  # n > S leaves trailing splits empty
                op, lp = oracle.attention_partials(q, k, v, 0.5, causal, n)
                om, lm = oracle.lse_merge(op, lp)
                assert np.allclose(om, o3, atol=1e-12, rtol=0), (T, S, n, causal)
                fin = np.isfinite(l3)
                assert np.array_equal(fin, np.isfinite(lm))
                assert np.allclose(lm[fin], l3[fin], atol=1e-12, rtol=0)


# --------------------------------------------------------------------------- #
# Closed forms and special cases
# --------------------------------------------------------------------------- #
def check_closed_forms():
    scale = 0.37
    r = np.random.default_rng(7)
    for fn in (oracle.attention_three_pass, oracle.attention_online):
        # one key: O = v0, lse = x0
        q, k, v = _rand_problem(1, 1, 2, 2, 4, 1, 5)
        o, lse = fn(q, k, v, scale, False)
        assert np.allclose(o, np.broadcast_to(v[:, :, :1], o.shape), atol=1e-14)
        assert np.allclose(lse, scale * np.einsum("bhtd,bhd->bht", q, k[:, :, 0]), atol=1e-14)
        # identical keys: O = mean of the visible values, lse = x + ln |J|
        S = 9
        key = r.standard_normal(6)
        k = np.broadcast_to(key, (1, 1, S, 6)).copy()
        v = r.standard_normal((1, 1, S, 6))
        q = r.standard_normal((1, 1, 4, 6))
        for causal in (False, True):
            o, lse = fn(q, k, v, scale, causal)
            for i in range(4):
                n_vis = S - 4 + i + 1 if causal else S
                assert np.allclose(o[0, 0, i], v[0, 0, :n_vis].mean(axis=0), atol=1e-13)
                assert abs(lse[0, 0, i] - (scale * q[0, 0, i] @ key + math.log(n_vis))) < 1e-13
        # q = 0: the uniform average, lse = ln S
        q = np.zeros((1, 1, 3, 6))
        v = r.standard_normal((1, 1, S, 6))
        k = r.standard_normal((1, 1, S, 6))
        o, lse = fn(q, k, v, scale, False)
        assert np.allclose(o[0, 0], v[0, 0].mean(axis=0), atol=1e-14)
        assert np.allclose(lse, math.log(S), atol=1e-14)
        # every value row the same: O is that row whatever the scores
        row = r.standard_normal(6)
        v = np.broadcast_to(row, (1, 1, S, 6)).copy()
        q = r.standard_normal((1, 1, 3, 6)) * 5
        o, _ = fn(q, k, v, scale, True)
        assert np.allclose(o[0, 0], row, atol=1e-13)
        # no visible key (causal, T > S): O = 0, lse = -inf for the first T - S rows
        q, k, v = _rand_problem(3, 1, 1, 1, 6, 2, 4)
        o, lse = fn(q, k, v, scale, True)
        assert np.all(o[0, 0, :4] == 0) and np.all(np.isneginf(lse[0, 0, :4]))
        assert np.all(np.isfinite(lse[0, 0, 4:]))
        # rows are convex combinations of the visible value rows
        q, k, v = _rand_problem(4, 1, 1, 1, 5, 12, 3, scale_q=3.0)
        o, _ = fn(q, k, v, scale, False)
        assert np.all(o <= v.max(axis=2, keepdims=True) + 1e-14) and np.all(o >= v.min(axis=2, keepdims=True) - 1e-14)


def check_gqa():
    q, k, v = _rand_problem(11, 2, 8, 2, 5, 13, 4)
    g = 8 // 2
    # textbook grouped-query attention: KV head repeated g times consecutively
    k_rep = np.repeat(k, g, axis=1)
    v_rep = np.repeat(v, g, axis=1)
    for causal in (False, True):
        o, lse = oracle.attention_three_pass(q, k, v, 0.4, causal)
        o2, lse2 = oracle.attention_three_pass(q, k_rep, v_rep, 0.4, causal)
        assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
    assert [oracle.kv_head_of(h, 64, 8) for h in (0, 7, 8, 63)] == [0, 0, 1, 7]


def check_key_permutation_invariance():
    q, k, v = _rand_problem(12, 1, 2, 2, 4, 20, 5)
    perm = np.random.default_rng(1).permutation(20)
    o, lse = oracle.attention_three_pass(q, k, v, 0.6, False)
    o2, lse2 = oracle.attention_three_pass(q, k[:, :, perm], v[:, :, perm], 0.6, False)
    assert np.allclose(o, o2, atol=1e-14) and np.allclose(lse, lse2, atol=1e-14)


def check_paged_equals_contiguous():
    r = np.random.default_rng(5)
    B, Hq, Hkv, d, ps = 3, 4, 2, 8, 16
    seqlens = np.array([40, 16, 1])
    max_pages = 3
    n_pool = B * max_pages
    table = r.permutation(n_pool).reshape(B, max_pages).astype(np.int32)
    kc = r.standard_normal((B, Hkv, max_pages * ps, d))
    vc = r.standard_normal((B, Hkv, max_pages * ps, d))
    k_pages = np.zeros((n_pool, ps, Hkv, d))
    v_pages = np.zeros((n_pool, ps, Hkv, d))
    for b in range(B):  # scatter the contiguous cache into the pool by the table
        for p in range(max_pages):
            for t in range(ps):
                k_pages[table[b, p], t] = kc[b, :, p * ps + t]
                v_pages[table[b, p], t] = vc[b, :, p * ps + t]
    for b in range(B):
        got = oracle.paged_gather(k_pages, table[b], int(seqlens[b]), ps)
        assert np.array_equal(got, kc[b, :, : seqlens[b]])  # bit-exact
    q = r.standard_normal((B, Hq, 2, d))
    o, lse = oracle.decode_paged(q, k_pages, v_pages, table, seqlens, ps, 0.3, True)
    for b in range(B):
        S = int(seqlens[b])
        o2, l2 = oracle.attention_three_pass(q[b : b + 1], kc[b : b + 1, :, :S], vc[b : b + 1, :, :S], 0.3, True)
        assert np.array_equal(o[b], o2[0]) and np.array_equal(lse[b], l2[0])
    bad = table.copy()
    bad[0, 0] = n_pool
    with pytest.raises(IndexError):
        oracle.paged_gather(k_pages, bad[0], 16, ps)


def check_overflow_safe():
    # scores near +-1000: e^1000 overflows even in fp64, the max-subtracted form does not
    with np.errstate(over="ignore"):
        assert np.isinf(np.exp(np.float64(1000.0)))
    q = np.zeros((1, 1, 2, 2))
    q[0, 0, 0] = [1000.0, 0.0]
    q[0, 0, 1] = [-1000.0, 0.0]
    k = np.array([[1.0, 0.0], [0.999, 0.0], [-1.0, 0.0]]).reshape(1, 1, 3, 2)
    v = np.array([[1.0, 0.0], [0.0, 1.0], [0.0, 0.0]]).reshape(1, 1, 3, 2)
    for fn in (oracle.attention_three_pass, oracle.attention_online, oracle.attention_online_normalized):
        o, lse = fn(q, k, v, 1.0, False)
        assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
        # row 0: scores 1000, 999, -1000 -> weights 1/(1+e^-1), e^-1/(1+e^-1), ~0
        w0 = 1.0 / (1.0 + math.exp(-1.0))
        assert abs(o[0, 0, 0, 0] - w0) < 1e-14 and abs(o[0, 0, 0, 1] - (1 - w0)) < 1e-14
        assert abs(lse[0, 0, 0] - (1000.0 + math.log1p(math.exp(-1.0)))) < 1e-12
        # row 1: scores -1000, -999, 1000 -> all weight on the third key
        assert abs(o[0, 0, 1]).max() < 1e-300 and abs(lse[0, 0, 1] - 1000.0) < 1e-12


def check_decimal_brute_force():
    """Independent arithmetic: 50-digit decimal exp/ln of the definition on tiny inputs."""
    getcontext().prec = 50
    r = np.random.default_rng(21)
    for trial in range(6):
        T, S, d = 1 + trial % 3, 2 + trial, 1 + trial % 4
        causal = trial % 2 == 1
        q = r.standard_normal((1, 1, T, d)) * 2
        k = r.standard_normal((1, 1, S, d))
        v = r.standard_normal((1, 1, S, d))
        scale = 0.5 + 0.1 * trial
        o3, l3 = oracle.attention_three_pass(q, k, v, scale, causal)
        o1, l1 = oracle.attention_online(q, k, v, scale, causal, block=2)
        for i in range(T):
            keys = [j for j in range(S) if (not causal) or j <= i + S - T]
            if not keys:
                assert np.isneginf(l3[0, 0, i])
                continue
            xs = {j: Decimal(scale) * sum(Decimal(q[0, 0, i, c]) * Decimal(k[0, 0, j, c]) for c in range(d)) for j in keys}
            z = sum(x.exp() for x in xs.values())
            lse = float(z.ln())
            out = [float(sum((xs[j].exp() / z) * Decimal(v[0, 0, j, c]) for j in keys)) for c in range(d)]
            for o, l in ((o3, l3), (o1, l1)):
                assert abs(l[0, 0, i] - lse) < 1e-13
                assert np.allclose(o[0, 0, i], out, atol=1e-14, rtol=0)


ALL_CHECKS = [
    check_softmax_123,
    check_online_trace,
    check_lse_merge_worked,
    check_causal_decode,
    check_mask_enumeration,
    check_online_equals_three_pass,
    check_split_invariance,
    check_closed_forms,
    check_gqa,
    check_key_permutation_invariance,
    check_paged_equals_contiguous,
    check_overflow_safe,
    check_decimal_brute_force,
]


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check()


def _fails_some_pin():
    for c in ALL_CHECKS:
        try:
            c()
        except (AssertionError, IndexError, ValueError):
            return True
    return False


def test_planted_mistakes_are_caught(monkeypatch):
    """Each plausible mistake, planted in the oracle, makes at least one pin fail."""
    orig_three = oa.attention_three_pass
    orig_visible_mask = oa.causal_mask
    mistakes = {
        "gqa h % Hkv": lambda mp: mp.setattr(oa, "kv_head_of", lambda h, Hq, Hkv: h % Hkv),
        "top-left mask": lambda mp: mp.setattr(
            oa, "causal_mask", lambda T, S, causal=True: np.tril(np.ones((T, S), dtype=bool)) if causal else np.ones((T, S), dtype=bool)
        ),
        "strict mask": lambda mp: mp.setattr(
            oa, "causal_mask", lambda T, S, causal=True: (orig_visible_mask(T, S, causal) & ~np.eye(T, S, S - T, dtype=bool)) if causal else np.ones((T, S), dtype=bool)
        ),
        "dropped scale": lambda mp: mp.setattr(oa, "attention_three_pass", lambda q, k, v, scale, causal=False: orig_three(q, k, v, 1.0, causal)),
        "k and v swapped": lambda mp: mp.setattr(oa, "attention_three_pass", lambda q, k, v, scale, causal=False: orig_three(q, v, k, scale, causal)),
    }
    for name, plant in mistakes.items():
        with monkeypatch.context() as mp:
            plant(mp)
            # the package re-exports the functions: patch those names too
            for attr in ("kv_head_of", "causal_mask", "attention_three_pass"):
                mp.setattr(oracle, attr, getattr(oa, attr))
            assert _fails_some_pin(), f"planted mistake not caught: {name}"
