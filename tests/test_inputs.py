"""The seeded input recipe shared by the oracle and the GPU tests: the same seed gives the
same bits, the block table is a permutation of the pool (every page used exactly once), and
the row sample covers the first, middle and last tiles."""

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
