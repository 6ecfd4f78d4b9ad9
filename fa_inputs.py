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
