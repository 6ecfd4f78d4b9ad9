"""fp64 oracle for fused attention forward: prefill, split-KV partials + merge, paged decode.

TEST INFRASTRUCTURE ONLY (see the package docstring). Plain, slow, obviously
correct: numpy fp64, one (batch, head) plane at a time, no fusion or blocking
beyond what the cited passage states.

Sources (page title, section):
  [FA1]   "Kernel visualization: Flash Attention 1" (linearalgebraforprogrammers.com):
          "Derivation" (the per-key recurrence for m, d', o'), "The tiled version".
  [SFA]   "Softmax and FlashAttention" (gpu-kernels-explained.vercel.app):
          "Concept" (standard three-kernel attention, safe softmax, the online
          softmax), "Maths" (exactness of the online form).
  [CHAIN] "Attention kernel chains: tiling, the online softmax, merges and masks"
          (inferenceinterviews.com): "The online softmax on numbers", "The
          log-sum-exp merge", "The causal mask for a decode step", "What the
          backward pass saves", "GQA loads KV once per group", "The block-table
          cost of paged attention".

Conventions (readings where the pages are silent):
  * Layout: q, o are [B][Hq][T][d]; k, v are [B][Hkv][S][d] (per-(batch, head)
    planes of [rows][d], as the FA1 kernel indexes them).
  * Scores are x_j = scale * (q . k_j); lse is the natural log-sum-exp of the
    scaled scores, lse = m + ln(l) ([CHAIN] "What the backward pass saves"
    saves one such value per query row; "The log-sum-exp merge" uses ln).
  * Causal masking is bottom-right aligned: query row i of T sits at position
    S - T + i and sees key j iff j <= i + (S - T) ([CHAIN] "The causal mask for
    a decode step").
  * A row that sees no key (causal with T > S) has O = 0 and lse = -inf.
  * GQA: query head h reads KV head h // (Hq // Hkv) (contiguous groups).
  * Paged K/V pools are [num_pages][page_size][Hkv][d]; block_table[b][p] is
    the pool page holding tokens p*page_size .. p*page_size + page_size - 1 of
    sequence b; K and V share one table entry per page.
"""

from __future__ import annotations

import math

import numpy as np

NEG_INF = float("-inf")


# --------------------------------------------------------------------------- #
# Masks and head mapping
# --------------------------------------------------------------------------- #
def visible(i: int, j: int, T: int, S: int, causal: bool) -> bool:
    """Whether query row i (of T new queries) may attend to key j (of S keys).

    [CHAIN] "The causal mask for a decode step": the T new queries are the last
    T positions, so row i sits at position S - T + i and sees key j exactly
    when j <= i + (S - T). Without a mask every key is visible.
    """
    if not causal:
        return True
    return j <= i + (S - T)


def causal_mask(T: int, S: int, causal: bool = True) -> np.ndarray:
    """Boolean [T][S] visibility matrix: the rule of :func:`visible` for every (i, j)."""
    if not causal:
        return np.ones((T, S), dtype=bool)
    i = np.arange(T)[:, None]
    j = np.arange(S)[None, :]
    return j <= i + (S - T)


def kv_head_of(h: int, Hq: int, Hkv: int) -> int:
    """KV head read by query head h under GQA ([CHAIN] "GQA loads KV once per group").

    The g = Hq / Hkv query heads of a group are contiguous: heads
    kv*g .. kv*g + g - 1 share KV head kv.
    """
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    return h // (Hq // Hkv)


def _as64(x) -> np.ndarray:
    """fp64 numpy copy of an array-like; torch tensors (any dtype, bf16 included)
    are converted through their own ``double()`` without importing torch here."""
    if hasattr(x, "detach") and hasattr(x, "double"):
        return x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def _check_shapes(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be 4-D [B][H][rows][d]")
    B, Hq, T, d = q.shape
    Bk, Hkv, S, dk = k.shape
    if k.shape != v.shape or Bk != B or dk != d:
        raise ValueError("k, v must be [B][Hkv][S][d] matching q")
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    return B, Hq, Hkv, T, S, d


# --------------------------------------------------------------------------- #
# Three-pass standard attention: the plain definition
# --------------------------------------------------------------------------- #
def _three_pass_plane(q, k, v, scale, causal):
    """One (batch, head) plane by the three-kernel recipe of [SFA] "Concept".

    Pass 1 materialises the scores S = scale * Q K^T; pass 2 is the safe
    softmax along each row, p = e^{x - m} / sum_j e^{x_j - m} with m the row
    max ([SFA] "Concept", second animation); pass 3 is O = P V.
    Returns (O [T][d], lse [T]).
    """
    T, S = q.shape[0], k.shape[0]
    x = scale * (q @ k.T)  # pass 1: [T][S] scores
    if causal:
        vis = causal_mask(T, S, True)
        x = np.where(vis, x, NEG_INF)
    m = x.max(axis=1) if S > 0 else np.full(T, NEG_INF)
    o = np.zeros((T, q.shape[1]), dtype=np.float64)
    lse = np.full(T, NEG_INF, dtype=np.float64)
    live = np.isfinite(m)  # rows with at least one visible key
    if live.any():
        e = np.exp(x[live] - m[live, None])  # masked entries give exp(-inf) = 0
        l = e.sum(axis=1)
        p = e / l[:, None]  # pass 2: the probabilities P
        o[live] = p @ v  # pass 3: O = P V
        lse[live] = m[live] + np.log(l)
    return o, lse


def attention_three_pass(q, k, v, scale: float, causal: bool = False):
    """Exact attention by materialising S and P ([SFA] "Concept"; [FA1] "Derivation").

    q [B][Hq][T][d], k, v [B][Hkv][S][d] -> (o [B][Hq][T][d], lse [B][Hq][T]), fp64.
    """
    q, k, v = _as64(q), _as64(k), _as64(v)
    B, Hq, Hkv, T, S, d = _check_shapes(q, k, v)
    o = np.zeros((B, Hq, T, d))
    lse = np.full((B, Hq, T), NEG_INF)
    for b in range(B):
        for h in range(Hq):
            hk = kv_head_of(h, Hq, Hkv)
            o[b, h], lse[b, h] = _three_pass_plane(q[b, h], k[b, hk], v[b, hk], scale, causal)
    return o, lse


def attention_rows(q, k, v, rows, scale: float, causal: bool = False):
    """The three-pass definition for a sample of query rows only.

    Rows are independent ([FA1] "The tiled version": every query row runs its
    own loop), so each (b, h, i) in ``rows`` is computed exactly against the
    whole K/V plane of its KV head. ``q`` may be any indexable [B][Hq][T][d]
    array (a torch tensor is converted one plane at a time).
    Returns (o [n][d], lse [n]) in the order of ``rows``.
    """
    B, Hq, T, d = q.shape
    Hkv, S = k.shape[1], k.shape[2]
    out_o = np.zeros((len(rows), d))
    out_l = np.full(len(rows), NEG_INF)
    by_plane: dict[tuple[int, int], list[tuple[int, int]]] = {}
    for n, (b, h, i) in enumerate(rows):
        by_plane.setdefault((int(b), int(h)), []).append((n, int(i)))
    for (b, h), items in by_plane.items():
        hk = kv_head_of(h, Hq, Hkv)
        kk = _as64(k[b, hk])
        vv = _as64(v[b, hk])
        qq = _as64(q[b, h])
        for n, i in items:
            x = scale * (kk @ qq[i])  # scores of row i against every key
            if causal:
                x = np.where(np.arange(S) <= i + (S - T), x, NEG_INF)
            m = x.max() if S > 0 else NEG_INF
            if not np.isfinite(m):
                continue
            e = np.exp(x - m)
            l = e.sum()
            out_o[n] = (e / l) @ vv
            out_l[n] = m + math.log(l)
    return out_o, out_l


# --------------------------------------------------------------------------- #
# One-pass online softmax, FlashAttention-2 order (unnormalised u, divide once)
# --------------------------------------------------------------------------- #
def _online_plane(q, k, v, scale, causal, block, trace=None):
    """One plane by streaming key blocks of width ``block``.

    Carries per query row the running max m, the running sum l and the
    unnormalised output u ([CHAIN] "The online softmax on numbers": the state
    per row is the running max, the running sum and the unnormalised output).
    For each block ([FA1] "The tiled version", [SFA] "Maths"):
        m'     = max(m, max_j x_j)
        alpha  = e^{m - m'}
        l      = l * alpha + sum_j e^{x_j - m'}
        u      = u * alpha + sum_j e^{x_j - m'} V[j]
    and after the last block O = u / l, lse = m + ln l (the FlashAttention-2
    division "once at the end").
    ``trace`` (optional) is called as trace(block_index, m, l, alpha) with the
    per-row carries after each block.
    """
    T, S = q.shape[0], k.shape[0]
    d = q.shape[1]
    m = np.full(T, NEG_INF)
    l = np.zeros(T)
    u = np.zeros((T, d))
    vis_all = causal_mask(T, S, True) if causal else None
    for bi, j0 in enumerate(range(0, S, block)):
        j1 = min(S, j0 + block)
        x = scale * (q @ k[j0:j1].T)  # scores of this block only: [T][j1-j0]
        if vis_all is not None:
            x = np.where(vis_all[:, j0:j1], x, NEG_INF)
        m_new = np.maximum(m, x.max(axis=1))
        live = np.isfinite(m_new)  # rows that have seen a visible key so far
        alpha = np.zeros(T)
        # rows whose old max was finite rescale by e^{m - m'}; rows with m = -inf had l = u = 0
        had = live & np.isfinite(m)
        alpha[had] = np.exp(m[had] - m_new[had])
        p = np.zeros_like(x)
        p[live] = np.exp(x[live] - m_new[live, None])
        l = np.where(live, l * alpha + p.sum(axis=1), l)
        u = np.where(live[:, None], u * alpha[:, None] + p @ v[j0:j1], u)
        m = m_new
        if trace is not None:
            trace(bi, m.copy(), l.copy(), alpha.copy())
    o = np.zeros((T, d))
    lse = np.full(T, NEG_INF)
    live = l > 0
    o[live] = u[live] / l[live, None]
    lse[live] = m[live] + np.log(l[live])
    return o, lse


def attention_online(q, k, v, scale: float, causal: bool = False, block: int = 128, trace=None):
    """Exact attention by the one-pass online softmax, FlashAttention-2 loop order.

    Same contract as :func:`attention_three_pass`; ``block`` is the key-block
    width Bc. ``trace`` as in :func:`_online_plane`, called with an extra
    leading (b, h) argument: trace((b, h), block_index, m, l, alpha).
    """
    q, k, v = _as64(q), _as64(k), _as64(v)
    B, Hq, Hkv, T, S, d = _check_shapes(q, k, v)
    if block < 1:
        raise ValueError("block must be >= 1")
    o = np.zeros((B, Hq, T, d))
    lse = np.full((B, Hq, T), NEG_INF)
    for b in range(B):
        for h in range(Hq):
            hk = kv_head_of(h, Hq, Hkv)
            tr = None if trace is None else (lambda *a, _bh=(b, h): trace(_bh, *a))
            o[b, h], lse[b, h] = _online_plane(q[b, h], k[b, hk], v[b, hk], scale, causal, block, tr)
    return o, lse


# --------------------------------------------------------------------------- #
# One-pass, FlashAttention-1 normalised form (o' and d' of [FA1] "Derivation")
# --------------------------------------------------------------------------- #
def _online_normalized_plane(q, k, v, scale, causal, block):
    """The recurrence exactly as [FA1] "The tiled version" writes it.

    Carries the normalised partial output o' (not u), the running max m and
    the partial denominator d':
        m_i  = max(m_{i-1}, local max)
        d'_i = d'_{i-1} e^{m_{i-1} - m_i} + sum_j e^{x_i[j] - m_i}
        o'_i = o'_{i-1} * d'_{i-1} e^{m_{i-1} - m_i} / d'_i + sum_j e^{x_i[j] - m_i} / d'_i * V[j]
    starting from m_0 = -inf, d'_0 = 0, o'_0 = 0.
    """
    T, S = q.shape[0], k.shape[0]
    d = q.shape[1]
    m = np.full(T, NEG_INF)
    dp = np.zeros(T)
    op = np.zeros((T, d))
    vis_all = causal_mask(T, S, True) if causal else None
    for j0 in range(0, S, block):
        j1 = min(S, j0 + block)
        x = scale * (q @ k[j0:j1].T)
        if vis_all is not None:
            x = np.where(vis_all[:, j0:j1], x, NEG_INF)
        m_new = np.maximum(m, x.max(axis=1))
        live = np.isfinite(m_new)
        corr = np.zeros(T)  # e^{m_{i-1} - m_i}; zero while nothing was seen
        had = live & np.isfinite(m)
        corr[had] = np.exp(m[had] - m_new[had])
        w = np.zeros_like(x)
        w[live] = np.exp(x[live] - m_new[live, None])
        d_new = np.where(live, dp * corr + w.sum(axis=1), dp)
        safe = np.where(live, d_new, 1.0)
        op = np.where(
            live[:, None],
            op * (dp * corr / safe)[:, None] + (w / safe[:, None]) @ v[j0:j1],
            op,
        )
        dp, m = d_new, m_new
    lse = np.full(T, NEG_INF)
    live = dp > 0
    lse[live] = m[live] + np.log(dp[live])
    return np.where(live[:, None], op, 0.0), lse


def attention_online_normalized(q, k, v, scale: float, causal: bool = False, block: int = 128):
    """Exact attention by the FlashAttention-1 normalised recurrence (o', d')."""
    q, k, v = _as64(q), _as64(k), _as64(v)
    B, Hq, Hkv, T, S, d = _check_shapes(q, k, v)
    o = np.zeros((B, Hq, T, d))
    lse = np.full((B, Hq, T), NEG_INF)
    for b in range(B):
        for h in range(Hq):
            hk = kv_head_of(h, Hq, Hkv)
            o[b, h], lse[b, h] = _online_normalized_plane(q[b, h], k[b, hk], v[b, hk], scale, causal, block)
    return o, lse


# --------------------------------------------------------------------------- #
# Split-KV partials and the log-sum-exp merge
# --------------------------------------------------------------------------- #
def split_ranges(S: int, num_splits: int) -> list[tuple[int, int]]:
    """Contiguous key ranges: split s covers [s*c, min(S, (s+1)*c)) with c = ceil(S / n).

    Trailing splits may be empty when n does not divide S evenly.
    """
    if num_splits < 1:
        raise ValueError("num_splits must be >= 1")
    c = -(-S // num_splits)
    return [(min(S, s * c), min(S, (s + 1) * c)) for s in range(num_splits)]


def attention_partials(q, k, v, scale: float, causal: bool, num_splits: int):
    """Normalised partial outputs and their lse, one per key range.

    [CHAIN] "The log-sum-exp merge": each worker writes a normalised partial
    output and its lse. Split s is exact attention over its key range alone;
    the mask keeps the global key index (key j of the whole sequence). An
    empty or fully masked split has O_s = 0 and lse_s = -inf.
    Returns (o_parts [n][B][Hq][T][d], lse_parts [n][B][Hq][T]).
    """
    q, k, v = _as64(q), _as64(k), _as64(v)
    B, Hq, Hkv, T, S, d = _check_shapes(q, k, v)
    o_parts = np.zeros((num_splits, B, Hq, T, d))
    lse_parts = np.full((num_splits, B, Hq, T), NEG_INF)
    for s, (j0, j1) in enumerate(split_ranges(S, num_splits)):
        if j1 <= j0:
            continue
        for b in range(B):
            for h in range(Hq):
                hk = kv_head_of(h, Hq, Hkv)
                x = scale * (q[b, h] @ k[b, hk, j0:j1].T)
                if causal:
                    x = np.where(causal_mask(T, S, True)[:, j0:j1], x, NEG_INF)
                m = x.max(axis=1)
                live = np.isfinite(m)
                if not live.any():
                    continue
                e = np.exp(x[live] - m[live, None])
                l = e.sum(axis=1)
                o_parts[s, b, h][live] = (e / l[:, None]) @ v[b, hk, j0:j1]
                lse_parts[s, b, h][live] = m[live] + np.log(l)
    return o_parts, lse_parts


def lse_merge(o_parts, lse_parts):
    """Merge normalised partials ([CHAIN] "The log-sum-exp merge").

    lse = ln sum_s e^{lse_s}; O = sum_s e^{lse_s - lse} O_s. Computed with the
    largest lse_s subtracted first so no exponent overflows. Axis 0 indexes
    the splits; any trailing shape is allowed (o_parts has one more trailing
    axis, d). Splits with lse_s = -inf get weight 0; a row whose splits are
    all -inf merges to O = 0, lse = -inf.
    """
    o_parts = _as64(o_parts)
    lse_parts = _as64(lse_parts)
    mx = lse_parts.max(axis=0)
    live = np.isfinite(mx)
    safe_mx = np.where(live, mx, 0.0)
    w_un = np.where(np.isfinite(lse_parts), np.exp(lse_parts - safe_mx), 0.0)
    tot = w_un.sum(axis=0)
    lse = np.where(live, safe_mx + np.log(np.where(live, tot, 1.0)), NEG_INF)
    w = np.where(np.isfinite(lse_parts), np.exp(lse_parts - np.where(live, lse, 0.0)), 0.0)
    o = (w[..., None] * o_parts).sum(axis=0)
    o = np.where(live[..., None], o, 0.0)
    return o, lse


# --------------------------------------------------------------------------- #
# Paged KV
# --------------------------------------------------------------------------- #
def paged_gather(pages, table_row, seqlen: int, page_size: int) -> np.ndarray:
    """Rebuild one sequence's contiguous [Hkv][seqlen][d] K (or V) from its pages.

    [CHAIN] "The block-table cost of paged attention": token t of the sequence
    lives in slot t % page_size of pool page table_row[t // page_size].
    ``pages`` is [num_pages][page_size][Hkv][d].
    """
    n_pages = -(-seqlen // page_size)
    if n_pages > len(table_row):
        raise ValueError("sequence longer than its block-table row")
    Hkv, d = int(pages.shape[2]), int(pages.shape[3])
    out = np.zeros((Hkv, seqlen, d), dtype=np.float64)
    for p in range(n_pages):
        page = int(table_row[p])
        if not 0 <= page < int(pages.shape[0]):
            raise IndexError(f"block table entry {page} outside the pool")
        t0 = p * page_size
        t1 = min(seqlen, t0 + page_size)
        out[:, t0:t1, :] = np.transpose(_as64(pages[page, : t1 - t0]), (1, 0, 2))
    return out


def decode_paged(q, k_pages, v_pages, block_table, seqlens, page_size: int, scale: float, causal: bool = True):
    """Attention of T new queries per sequence over a paged K/V cache.

    Gathers each sequence's keys and values through its block-table row and
    runs the three-pass definition against them, with the bottom-right mask
    when ``causal``. q [B][Hq][T][d]; pools [P][page_size][Hkv][d];
    block_table [B][max_pages]; seqlens [B]. One sequence at a time, so the
    gathered copy stays small.
    Returns (o [B][Hq][T][d], lse [B][Hq][T]).
    """
    B, Hq, T, d = q.shape
    o = np.zeros((B, Hq, T, d))
    lse = np.full((B, Hq, T), NEG_INF)
    for b in range(B):
        S = int(seqlens[b])
        kb = paged_gather(k_pages, block_table[b], S, page_size)[None]
        vb = paged_gather(v_pages, block_table[b], S, page_size)[None]
        ob, lb = attention_three_pass(_as64(q[b : b + 1]), kb, vb, scale, causal)
        o[b], lse[b] = ob[0], lb[0]
    return o, lse


# --------------------------------------------------------------------------- #
# Backward: gradients of O with respect to Q, K and V
# --------------------------------------------------------------------------- #
def _bwd_probs(x, lse, vis):
    """P = exp(S - LSE) from the saved log-sum-exp ([CHAIN] "What the backward pass
    saves"); masked entries and rows with no visible key (lse = -inf) give 0."""
    p = np.zeros_like(x)
    live = np.isfinite(lse)
    if live.any():
        p[live] = np.where(vis[live], np.exp(x[live] - lse[live, None]), 0.0)
    return p


def _softmax_grad(p, dp, dsum):
    """dS = P * (dP - D): the softmax Jacobian applied to dP, with D = rowsum(dO * O)."""
    return p * (dp - dsum[:, None])


def _score_grads(ds, q, k, scale):
    """Through S = scale * Q K^T: dQ = scale * dS K, dK = scale * dS^T Q."""
    return scale * (ds @ k), scale * (ds.T @ q)


def attention_backward(q, k, v, do, scale: float, causal: bool = False, o=None, lse=None):
    """Gradients of O = softmax(scale * Q K^T) V for an upstream gradient dO.

    [CHAIN] "What the backward pass saves": the forward keeps Q, K, V, O and one
    log-sum-exp per query row; the backward rebuilds each probability as
    P = exp(S - LSE) with S = scale * Q K^T, and the softmax gradient needs the
    one extra vector D = rowsum(dO * O), formed once before the main loop. The
    rest is the chain rule through O = P V and P = softmax(S), written out per
    (batch, query head):
        dV  = P^T dO                 (O = P V)
        dP  = dO V^T
        dS  = P * (dP - D)           (softmax Jacobian: dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik),
                                      and sum_k P_ik dP_ik = dO_i . O_i = D_i)
        dQ  = scale * dS K           (S = scale * Q K^T)
        dK  = scale * dS^T Q
    A KV head's dK and dV sum over the query heads of its group (GQA: head h
    reads KV head h // g). Masked scores have P = 0; a row with no visible key
    contributes nothing.
    o, lse: the saved forward outputs; when omitted they come from the
    three-pass forward. q, do [B][Hq][T][d]; k, v [B][Hkv][S][d].
    Returns (dq, dk, dv) in fp64 with the shapes of q, k, v.
    """
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    B, Hq, Hkv, T, S, d = _check_shapes(q, k, v)
    if o is None or lse is None:
        o, lse = attention_three_pass(q, k, v, scale, causal)
    o, lse = _as64(o), _as64(lse)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    vis = causal_mask(T, S, causal)
    dsum_all = backward_rowsum(do, o)  # D, once before the main loop
    for b in range(B):
        for h in range(Hq):
            hk = kv_head_of(h, Hq, Hkv)
            x = scale * (q[b, h] @ k[b, hk].T)  # S
            p = _bwd_probs(x, lse[b, h], vis)
            dp = do[b, h] @ v[b, hk].T
            ds = _softmax_grad(p, dp, dsum_all[b, h])
            dv[b, hk] += p.T @ do[b, h]
            dqh, dkh = _score_grads(ds, q[b, h], k[b, hk], scale)
            dq[b, h] = dqh
            dk[b, hk] += dkh
    return dq, dk, dv


def backward_rowsum(do, o):
    """D = rowsum(dO * O), one value per query row ([CHAIN] "What the backward pass saves")."""
    return (_as64(do) * _as64(o)).sum(axis=-1)


def attention_backward_rows(q, k, v, do, o, lse, q_rows, k_rows, scale: float, causal: bool = False):
    """The backward of ``attention_backward`` for samples of rows only.

    Rows of dQ are independent of one another: dQ_i = scale * sum_j dS_ij k_j
    needs only query row i against every key. A row of dK or dV needs its key
    against every query row of every head in the group: dV_j = sum P_ij dO_i,
    dK_j = scale * sum dS_ij q_i. Each sampled row is computed exactly in
    O(rows * d) from the same formulas ([CHAIN] "What the backward pass saves").
    q_rows: (b, h, i) query rows; k_rows: (b, hk, j) key rows.
    Returns (dq [len(q_rows)][d], dk [len(k_rows)][d], dv [len(k_rows)][d]).
    """
    q, k, v, do, o, lse = _as64(q), _as64(k), _as64(v), _as64(do), _as64(o), _as64(lse)
    B, Hq, Hkv, T, S, d = _check_shapes(q, k, v)
    g = Hq // Hkv
    dsum = {}

    def dsum_of(b, h):
        if (b, h) not in dsum:
            dsum[(b, h)] = backward_rowsum(do[b, h], o[b, h])
        return dsum[(b, h)]

    dq = np.zeros((len(q_rows), d))
    for n, (b, h, i) in enumerate(q_rows):
        hk = kv_head_of(h, Hq, Hkv)
        vis = np.array([visible(i, j, T, S, causal) for j in range(S)])
        x = scale * (k[b, hk] @ q[b, h, i])
        p = np.where(vis, np.exp(x - lse[b, h, i]), 0.0) if np.isfinite(lse[b, h, i]) else np.zeros(S)
        dp = v[b, hk] @ do[b, h, i]
        ds = p * (dp - dsum_of(b, h)[i])
        dq[n] = scale * (ds @ k[b, hk])
    dk = np.zeros((len(k_rows), d))
    dv = np.zeros((len(k_rows), d))
    for n, (b, hk, j) in enumerate(k_rows):
        vis = np.array([visible(i, j, T, S, causal) for i in range(T)])
        for h in range(hk * g, (hk + 1) * g):
            x = scale * (q[b, h] @ k[b, hk, j])
            live = np.isfinite(lse[b, h]) & vis
            p = np.zeros(T)
            p[live] = np.exp(x[live] - lse[b, h][live])
            dp = do[b, h] @ v[b, hk, j]
            ds = p * (dp - dsum_of(b, h))
            dv[n] += p @ do[b, h]
            dk[n] += scale * (ds @ q[b, h])
    return dq, dk, dv
