"""Seeded synthetic inputs shared by the oracle tests, the GPU parity tests and the bench.

This module holds shapes and random draws only: none of the attention
arithmetic. Both sides (the fp64 oracle and the CUDA library) receive the
tensors it returns; neither side is imported here.

Recipe: values are i.i.d. N(0, 1) drawn in fp32 by ``torch.randn`` from a
``torch.Generator`` seeded per tensor (Q = 1000 + c, K = 2000 + c,
V = 3000 + c, page permutation = 4000 + c, c = the workload's index), then
cast to bf16 where the workload is bf16. Paged K/V pools are drawn page by
page in pool order and a seeded random permutation of the pool is the block
table, so a sequence's pages are scattered across the pool.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    B: int
    Hq: int
    Hkv: int
    T: int
    S: int
    d: int
    causal: bool
    dtype: str = "bf16"  # "bf16", or "f32" for the fp32 smoke problem
    num_splits: int = 0  # split-KV decode: number of key ranges (0: not a split workload)
    page_size: int = 0  # paged decode: tokens per page (0: contiguous K/V)
    note: str = ""
    sweep: tuple = field(default_factory=tuple)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# The five workloads: names say what each is, with its sizes.
SMOKE = Workload("smoke_b1_h1_n256_d64", 0, 1, 1, 1, 256, 256, 64, False, dtype="f32",
                 note="fp32 inputs plus a bf16 copy; non-causal")
PREFILL_MHA = Workload("prefill_mha_b4_h16_n4096_d128", 1, 4, 16, 16, 4096, 4096, 128, False,
                       note="non-causal MHA", sweep=((4096, 64), (4096, 128), (8192, 64), (8192, 128)))
CAUSAL_GQA = Workload("causal_gqa_b1_hq64_hkv8_n8192_d128", 2, 1, 64, 8, 8192, 8192, 128, True,
                      note="causal, group 8")
SPLITKV_DECODE = Workload("splitkv_decode_b1_hq32_hkv8_s131072_d128", 3, 1, 32, 8, 1, 131072, 128, True,
                          num_splits=16, note="one new query over 131072 cached keys, 16 splits")
PAGED_DECODE = Workload("paged_decode_b64_hq64_hkv8_s8192_d128_p16", 4, 64, 64, 8, 1, 8192, 128, True,
                        page_size=16, note="16-token pages scattered by a random-permutation block table")

WORKLOADS = {w.name: w for w in (SMOKE, PREFILL_MHA, CAUSAL_GQA, SPLITKV_DECODE, PAGED_DECODE)}

# Beyond the five: chunked prefill over the paged cache. Each of 8 sequences
# appends 512 new tokens to a cache of CHUNKED_SEQLENS[b] tokens (the new ones
# included), 16-token pages scattered by the seeded permutation.
CHUNKED_PREFILL = Workload("chunked_prefill_paged_b8_hq32_hkv8_t512_s8192_d128_p16", 5, 8, 32, 8, 512, 8192, 128,
                           True, page_size=16, note="512 new tokens per sequence over a paged cache of up to 8192")
CHUNKED_SEQLENS = (8192, 7000, 6144, 5000, 4096, 3000, 2048, 1024)


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def randn(shape, seed: int, dtype=torch.bfloat16, device="cpu") -> torch.Tensor:
    """i.i.d. N(0,1) in fp32 from ``seed``, cast to ``dtype``."""
    x = torch.randn(*shape, generator=_gen(seed, device), dtype=torch.float32, device=device)
    return x if dtype == torch.float32 else x.to(dtype)


def qkv(B, Hq, Hkv, T, S, d, index: int, dtype=torch.bfloat16, device="cpu"):
    """q [B][Hq][T][d], k, v [B][Hkv][S][d], seeded by the workload index."""
    q = randn((B, Hq, T, d), 1000 + index, dtype, device)
    k = randn((B, Hkv, S, d), 2000 + index, dtype, device)
    v = randn((B, Hkv, S, d), 3000 + index, dtype, device)
    return q, k, v


def paged_kv(B, Hkv, S, d, page_size, index: int, dtype=torch.bfloat16, device="cpu", seqlens=None):
    """A paged K/V cache: pools [P][page_size][Hkv][d] and an int32 block table [B][max_pages].

    Every sequence has ``max_pages = ceil(S / page_size)`` table entries and
    the pool holds exactly B * max_pages pages; the table is a seeded random
    permutation of the pool. ``seqlens`` (int32 [B]) defaults to S for every
    sequence.
    """
    max_pages = -(-S // page_size)
    P = B * max_pages
    k_pages = randn((P, page_size, Hkv, d), 2000 + index, dtype, device)
    v_pages = randn((P, page_size, Hkv, d), 3000 + index, dtype, device)
    perm = torch.randperm(P, generator=_gen(4000 + index))
    table = perm.view(B, max_pages).to(torch.int32).to(device)
    if seqlens is None:
        seqlens = torch.full((B,), S, dtype=torch.int32, device=device)
    return k_pages, v_pages, table, seqlens


def decode_q(B, Hq, T, d, index: int, dtype=torch.bfloat16, device="cpu"):
    return randn((B, Hq, T, d), 1000 + index, dtype, device)


def chunked_prefill_problem(w: Workload = CHUNKED_PREFILL, device="cpu"):
    """q [B][Hq][T][d], the paged pools, block table and seqlens of the chunked-prefill workload."""
    k_pages, v_pages, table, _ = paged_kv(w.B, w.Hkv, w.S, w.d, w.page_size, w.index, device=device)
    q = decode_q(w.B, w.Hq, w.T, w.d, w.index, device=device)
    seqlens = torch.tensor(CHUNKED_SEQLENS[: w.B], dtype=torch.int32, device=device)
    return q, k_pages, v_pages, table, seqlens


def sample_rows(B, Hq, T, n: int, seed: int, tile: int = 128):
    """A seeded sample of (b, h, i) query rows for checking large problems.

    ``n`` random rows plus every row of the first tile, the last tile (ragged
    tail included) and one tile in the middle of (b=0, h=0) and of
    (b=B-1, h=Hq-1).
    """
    g = _gen(seed)
    b = torch.randint(0, B, (n,), generator=g)
    h = torch.randint(0, Hq, (n,), generator=g)
    i = torch.randint(0, T, (n,), generator=g)
    rows = {(int(x), int(y), int(z)) for x, y, z in zip(b, h, i)}
    for bb, hh in ((0, 0), (B - 1, Hq - 1)):
        for start in (0, (T // 2 // tile) * tile, ((T - 1) // tile) * tile):
            for r in range(start, min(T, start + tile)):
                rows.add((bb, hh, r))
    return sorted(rows)


# Score levels, in log2 units, that the hot keys of successive 128-key tiles sit
# at: rises both below and above the kernels' rescale slack of 8, so that a row's
# reference max is sometimes kept (the largest p then exceeds 1) and sometimes
# moved (O and the running sum rescaled by 2^(m_old - m_new)).
CLIMB_STEPS = (0.0, 10.0, 5.0, 12.0, 3.0, 9.0, 7.0, 20.0, 1.0, 11.0, 6.0, 8.5, 2.0, 14.0, 4.0, 10.0, 7.5, 9.5)


def climbing_levels(n_tiles: int, pattern: str = "rise", steps=CLIMB_STEPS) -> list:
    """Per key tile, the level (log2 units) of that tile's hot keys.

    ``rise``: cumulative ``steps``, so the maximum climbs on every tile.
    ``rise_fall``: the same climb for the first half of the tiles, then back down.
    """
    lv, acc = [], 0.0
    for t in range(n_tiles):
        acc += steps[t % len(steps)]
        lv.append(acc)
    if pattern == "rise_fall":
        half = (n_tiles + 1) // 2
        lv = lv[:half] + [lv[2 * half - 1 - t] - 3.0 for t in range(half, n_tiles)]
    elif pattern != "rise":
        raise ValueError(pattern)
    return lv


def climbing_qkv(B, Hq, Hkv, T, S, d, index: int, scale: float, pattern: str = "rise", hot: int = 1,
                 mixed_rows: bool = False, steps=CLIMB_STEPS, v_scale: float = 1.0, v_hot=None, tile: int = 128,
                 dtype=torch.bfloat16):
    """Inputs whose row maximum climbs tile by tile (the online softmax's rescale path).

    Each (batch, KV head) gets a direction u ~ N(0, I_d). Query rows are
    u + 0.05 N(0, I) (with ``mixed_rows``, rows at odd positions use -u instead,
    so that, within a group of adjacent rows, some climb and some do not). In key
    tile t, the first ``hot`` keys are u scaled so that scale * (u . k) equals
    climbing_levels(...)[t] * ln 2 minus 0.7 per further hot key (several keys
    share the weight), plus 0.1 N(0, I) noise; all other keys are N(0, 1).
    Values are v_scale * N(0, 1); with ``v_hot`` set, the hot keys' value rows
    are the constant v_hot instead. Seeds as in ``qkv``; u from 5000 + index.
    """
    g = _gen(2000 + index)
    u = torch.randn(B, Hkv, 1, d, generator=_gen(5000 + index))
    k = torch.randn(B, Hkv, S, d, generator=g)
    v = v_scale * torch.randn(B, Hkv, S, d, generator=_gen(3000 + index))
    n_tiles = -(-S // tile)
    levels = climbing_levels(n_tiles, pattern, steps)
    usq = (u * u).sum(-1, keepdim=True)  # [B][Hkv][1][1]
    for t in range(n_tiles):
        for j in range(min(hot, S - t * tile)):
            r = t * tile + j
            x = levels[t] * math.log(2.0) - 0.7 * j  # target scaled score (natural units)
            k[:, :, r : r + 1, :] = u * (x / scale) / usq + 0.1 * k[:, :, r : r + 1, :]
            if v_hot is not None:
                v[:, :, r, :] = v_hot
    sign = torch.ones(T, 1)
    if mixed_rows:
        sign[1::2] = -1.0
    qn = torch.randn(B, Hq, T, d, generator=_gen(1000 + index))
    q = u.repeat_interleave(Hq // Hkv, dim=1) * sign + 0.05 * qn
    return q.contiguous().to(dtype), k.to(dtype), v.to(dtype)


def pages_from_contiguous(k, v, page_size: int, index: int):
    """Lay contiguous K and V [B][Hkv][S][d] out as pools [P][page_size][Hkv][d]
    scattered by one seeded random-permutation block table [B][ceil(S/page_size)]
    (pool slots past S are zero). Returns (k_pool, v_pool, table)."""
    B, Hkv, S, d = k.shape
    max_pages = -(-S // page_size)
    P = B * max_pages
    perm = torch.randperm(P, generator=_gen(4000 + index))
    table = perm.view(B, max_pages).to(torch.int32)
    pools = []
    for x in (k, v):
        pool = torch.zeros(P, page_size, Hkv, d, dtype=x.dtype)
        for b in range(B):
            for p in range(max_pages):
                rows = x[b, :, p * page_size : min(S, (p + 1) * page_size), :]  # [Hkv][n][d]
                pool[int(table[b, p]), : rows.shape[1]] = rows.transpose(0, 1)
        pools.append(pool)
    return pools[0], pools[1], table
