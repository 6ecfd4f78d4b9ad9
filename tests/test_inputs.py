"""The seeded input recipe shared by the oracle and the GPU tests: the same seed gives the
same bits, the block table is a permutation of the pool (every page used exactly once), and
the row sample covers the first, middle and last tiles."""

import numpy as np
import torch

import fa_inputs as fi


def test_same_seed_same_bits():
    a = fi.qkv(1, 4, 2, 33, 65, 64, 7)
    b = fi.qkv(1, 4, 2, 33, 65, 64, 7)
    for x, y in zip(a, b):
        assert x.dtype == torch.bfloat16 and torch.equal(x, y)
    c = fi.qkv(1, 4, 2, 33, 65, 64, 8)
    assert not torch.equal(a[0], c[0])
    q, k, v = a
    assert q.shape == (1, 4, 33, 64) and k.shape == (1, 2, 65, 64) and v.shape == (1, 2, 65, 64)


def test_block_table_is_a_permutation_of_the_pool():
    B, Hkv, S, d, ps = 5, 2, 100, 64, 16
    kp, vp, table, seqlens = fi.paged_kv(B, Hkv, S, d, ps, 3)
    max_pages = -(-S // ps)
    assert table.dtype == torch.int32 and table.shape == (B, max_pages)
    assert kp.shape == (B * max_pages, ps, Hkv, d) and vp.shape == kp.shape
    assert sorted(table.flatten().tolist()) == list(range(B * max_pages))
    assert torch.equal(seqlens, torch.full((B,), S, dtype=torch.int32))
    _, _, table2, _ = fi.paged_kv(B, Hkv, S, d, ps, 3)
    assert torch.equal(table, table2)


def test_row_sample_covers_the_edge_tiles():
    B, Hq, T = 2, 3, 300
    rows = fi.sample_rows(B, Hq, T, 50, 11)
    assert rows == sorted(set(rows))
    assert all(0 <= b < B and 0 <= h < Hq and 0 <= i < T for b, h, i in rows)
    for bb, hh in ((0, 0), (B - 1, Hq - 1)):
        for i in list(range(0, 128)) + list(range(256, 300)) + list(range(128, 256)):
            assert (bb, hh, i) in rows


def test_chunked_problem_shapes():
    w = fi.CHUNKED_PREFILL
    q, kp, vp, table, seqlens = fi.chunked_prefill_problem(w)
    assert q.shape == (w.B, w.Hq, w.T, w.d)
    assert seqlens.tolist() == list(fi.CHUNKED_SEQLENS[: w.B])
    assert all(w.T <= s <= w.S for s in seqlens.tolist())


def test_climbing_inputs_have_the_stated_structure():
    """The rescale-path inputs: same seed, same bits; each tile's first hot key scores
    its level (log2 units) for a query row near u; mixed rows see the reverse."""
    import math

    d, S, scale = 64, 5 * 128, 0.125
    steps = (30.0, 10.0, 3.3, 12.0, 1.0)
    a = fi.climbing_qkv(1, 2, 2, 8, S, d, 7, scale, steps=steps, mixed_rows=True)
    b = fi.climbing_qkv(1, 2, 2, 8, S, d, 7, scale, steps=steps, mixed_rows=True)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    q, k, v = (t.double() for t in a)
    levels = fi.climbing_levels(5, "rise", steps)
    assert levels == [30.0, 40.0, 43.3, 55.3, 56.3]
    for t in range(5):
        x = scale * float(q[0, 0, 0] @ k[0, 0, t * 128]) * math.log2(math.e)  # row 0 climbs
        assert abs(x - levels[t]) < 0.05 * levels[t] + 0.5, (t, x)
        y = scale * float(q[0, 0, 1] @ k[0, 0, t * 128]) * math.log2(math.e)  # row 1 (odd) is reversed
        assert y < -0.9 * levels[t] + 0.5, (t, y)
    # the ordinary keys score like N(0, 1)
    ordinary = scale * (q[0, 0, 0] @ k[0, 0, 1:128].T)
    assert float(ordinary.abs().max()) < 6.0
    # rise then fall
    assert fi.climbing_levels(6, "rise_fall", (0.0, 10.0, 5.0)) == [0.0, 10.0, 15.0, 12.0, 7.0, -3.0]


def test_page_scatter_round_trips_through_the_oracle_gather():
    """pages_from_contiguous lays K/V out by its block table; the oracle's own gather
    rebuilds every sequence exactly (one table for K and V)."""
    import oracle

    k = fi.randn((2, 3, 100, 64), 11)
    v = fi.randn((2, 3, 100, 64), 12)
    kp, vp, table = fi.pages_from_contiguous(k, v, 16, 13)
    assert table.shape == (2, 7) and sorted(table.flatten().tolist()) == list(range(14))
    for bb in range(2):
        kg = oracle.paged_gather(kp.float(), table[bb], 100, 16)
        vg = oracle.paged_gather(vp.float(), table[bb], 100, 16)
        assert np.array_equal(kg, k[bb].float().numpy()) and np.array_equal(vg, v[bb].float().numpy())
