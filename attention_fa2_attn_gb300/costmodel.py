"""FLOP and byte accounting for the roofline numbers.

Formulas restated from the pages:
  * "Softmax and FlashAttention", section "Maths" (HBM traffic): standard
    attention moves e(2Nd + 4N^2 + 2Nd) bytes; FlashAttention-2 moves
    e(2Nd + 2N^2 d / Br) with no L2 reuse and 4eNd at the floor, e bytes per
    value.
  * "Attention kernel chains", "What FlashAttention removes from HBM":
    4 N^2 d FLOPs per head (two GEMMs of 2 N^2 d), unchanged by tiling; the
    causal convention halves it.
  * "GQA loads KV once per group" and "The block-table cost of paged
    attention": a decode step reads every K/V byte of its KV heads once;
    the block table costs 4 bytes per page.
"""

from __future__ import annotations


def attention_flops(B: int, Hq: int, T: int, S: int, d: int, causal: bool) -> float:
    """4*T*S*d per query head (QK^T and PV), halved for causal."""
    f = 4.0 * B * Hq * T * S * d
    return f / 2.0 if causal else f


def attention_backward_flops(B: int, Hq: int, T: int, S: int, d: int, causal: bool) -> float:
    """The backward's five products per (query, key) pair and head (S, dP, dV, dK, dQ),
    2*d FLOP each: 2.5 times the forward's 4*T*S*d, halved for causal.
    (The dQ kernel here recomputes S and dP, executing seven; the metric counts five.)"""
    return 2.5 * attention_flops(B, Hq, T, S, d, causal)


def visible_pairs(T: int, S: int, causal: bool) -> int:
    """(query, key) pairs the mask leaves visible for T queries over S keys.

    Bottom-right alignment: query i (0-based) sits at key position i + S - T and
    sees keys 0 .. min(S - 1, i + S - T); rows past the start see none.
    """
    if not causal:
        return T * S
    total = 0
    lo = S - T + 1  # keys row 0 sees (may be <= 0)
    # rows with a positive count form an arithmetic run capped at S
    for i in range(T):
        total += max(0, min(S, lo + i))
    return total


def chunked_attention_flops(Hq: int, T: int, seqlens, d: int, causal: bool = True) -> float:
    """4*d FLOP per visible (query, key) pair and query head, summed over sequences:
    T new queries per sequence over its seqlens[b] keys, bottom-right aligned."""
    return 4.0 * Hq * d * sum(visible_pairs(T, int(S), causal) for S in seqlens)


def standard_attention_bytes(N: int, d: int, e: int = 2) -> float:
    """Three-kernel attention of one head: read Q, K; write+read S; write+read P; read V; write O."""
    return e * (2 * N * d + 4 * N * N + 2 * N * d)


def flash2_bytes(N: int, d: int, e: int = 2, Br: int = 128) -> float:
    """FlashAttention-2, one head, no L2 reuse: Q and O once, K and V once per query block."""
    return e * (2 * N * d + 2 * N * N * d / Br)


def flash2_floor_bytes(N: int, d: int, e: int = 2) -> float:
    """Every value of Q, K, V and O moved once."""
    return 4 * e * N * d


def flash2_tile_bytes(N: int, d: int, e: int = 2, Br: int = 128, Bc: int = 128) -> tuple[float, float]:
    """Per-tile counter over the (query block i, key block j) loop: (moved, once).

    ``moved`` counts a Q block when its row of tiles starts and a K and V
    block at every tile (no L2 reuse); ``once`` counts each K/V block only for
    the first query block (every re-read hits L2). Neither includes the O write.
    """
    moved = once = 0.0
    nq = -(-N // Br)
    nk = -(-N // Bc)
    for i in range(nq):
        for j in range(nk):
            if j == 0:
                moved += e * Br * d
                once += e * Br * d
            moved += 2 * e * Bc * d
            if i == 0:
                once += 2 * e * Bc * d
    return moved, once


def flash1_bytes(N: int, d: int, e: int = 2, Bc: int = 128, e_state: int = 4) -> float:
    """FlashAttention-1 loop order, one head ("Kernel visualization: Flash Attention 1",
    "Counting trips across HBM"): K and V read once; Q and the running O, m, l read
    once per key tile, and O, m, l written back once per key tile (Tc = ceil(N / Bc)
    key tiles). Q, K, V take e bytes a value, the running state e_state."""
    tc = -(-N // Bc)
    state = N * d * e_state + 2 * N * e_state  # O, m, l of every row
    return 2 * N * d * e + tc * (N * d * e + 2 * state)


def kv_outer_bytes(B: int, Hq: int, T: int, S: int, d: int, causal: bool = False, row_bands: int = 1, e: int = 2,
                   Br: int = 128, Bc: int = 128) -> float:
    """Bytes the FlashAttention-1-order kernel (fa_fwd_kv_outer) moves per launch,
    counted over its loop nest with no reuse between CTAs. Each CTA loads every key
    tile its band needs once (K and V). At each (key tile j, query tile i) step it
    reads Q_i. Unless j is the tile's first key tile, it also reads the fp32 state
    O', m, l. Unless j is the tile's last key tile (bottom-right causal mask), it
    writes that state back; the last writes bf16 O and fp32 lse instead. A tile
    that sees no key writes O = 0 and lse once."""
    n_qt = -(-T // Br)
    n_kt = -(-S // Bc)
    R = max(1, min(row_bands, n_qt))
    state = d * 4 + 8  # O', m, l of one row
    final = d * e + 4  # O and lse of one row

    def jmax(i):
        if not causal:
            return n_kt - 1
        last_key = min(T, (i + 1) * Br) - 1 + S - T
        return -1 if last_key < 0 else min(n_kt - 1, last_key // Bc)

    per_head = 0
    for band in range(R):
        lo, hi = band * n_qt // R, (band + 1) * n_qt // R
        band_jmax = -1
        for i in range(lo, hi):
            rows = min(T, (i + 1) * Br) - i * Br
            jm = jmax(i)
            band_jmax = max(band_jmax, jm)
            if jm >= 0:
                steps = jm + 1
                per_head += steps * rows * d * e + 2 * (steps - 1) * rows * state
            per_head += rows * final
        for j in range(band_jmax + 1):
            per_head += 2 * (min(S, (j + 1) * Bc) - j * Bc) * d * e
    return float(per_head) * B * Hq


def prefill_compulsory_bytes(B: int, Hq: int, Hkv: int, T: int, S: int, d: int, e: int = 2) -> float:
    """Q read, O written, K and V read once, fp32 lse written."""
    return e * (2 * B * Hq * T * d + 2 * B * Hkv * S * d) + 4 * B * Hq * T


def decode_kv_bytes(B: int, Hkv: int, S: int, d: int, e: int = 2) -> float:
    """K and V of every KV head read once (grouped query heads share them)."""
    return 2.0 * B * Hkv * S * d * e


def decode_bytes(B: int, Hq: int, Hkv: int, T: int, S: int, d: int, e: int = 2, page_size: int = 0) -> float:
    """Algorithmic bytes of one decode step: K/V once, Q read, O written, fp32 lse
    written, and 4 bytes per block-table entry when paged."""
    b = decode_kv_bytes(B, Hkv, S, d, e) + 2.0 * e * B * Hq * T * d + 4.0 * B * Hq * T
    if page_size:
        b += 4.0 * B * (-(-S // page_size))
    return b


def gqa_kv_read_bytes(batch: int, context: int, kv_bytes_per_token: int, tp: int, group: int, grouped: bool) -> float:
    """KV bytes read per GPU per decode step; without grouping each query head re-reads its KV head."""
    b = batch * context * kv_bytes_per_token / tp
    return b if grouped else b * group


def paged_block_bytes(page_tokens: int, kv_heads: int, d: int, e: int = 2) -> int:
    """K and V bytes of one page across the KV heads of a layer."""
    return page_tokens * kv_heads * d * 2 * e
