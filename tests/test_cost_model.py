"""The FLOP/byte accounting used for the rooflines, pinned to the pages' numbers (CPU only)."""

import json
import math
import os

from attention_fa2_attn_gb300 import costmodel as cm

G = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_worked_examples.json")))
MB = 1e6
MiB = 2**20
GiB = 2**30


def test_byte_table():
    t = G["byte_table"]
    e, br = t["bytes_per_value"], t["block_rows"]
    for row in t["rows"]:
        N, d = row["N"], row["d"]
        assert math.isclose(cm.standard_attention_bytes(N, d, e) / MB, row["standard_MB"], rel_tol=t["rel_tol"])
        assert math.isclose(cm.flash2_bytes(N, d, e, br) / MB, row["flash_MB"], rel_tol=t["rel_tol"])
        # the floor is printed to two or three significant digits
        assert math.isclose(cm.flash2_floor_bytes(N, d, e) / MB, row["floor_MB"], rel_tol=0.03)


def test_tile_counter_matches_closed_form():
    for N, d in ((4096, 64), (1024, 128), (640, 64)):
        moved, once = cm.flash2_tile_bytes(N, d, 2, 128, 128)
        o_write = 2 * N * d
        assert math.isclose(moved + o_write, cm.flash2_bytes(N, d, 2, 128), rel_tol=1e-12)
        assert math.isclose(once + o_write, cm.flash2_floor_bytes(N, d, 2), rel_tol=1e-12)


def test_flash_removes():
    g = G["flash_removes"]
    N, d, e = g["N"], g["d"], g["bytes_per_value"]
    assert N * N * e / MiB == g["scores_MiB"]
    assert cm.flash2_floor_bytes(N, d, e) / MiB == g["compulsory_MiB"]
    fl = cm.attention_flops(1, 1, N, N, d, False)
    assert abs(fl / 1e9 - g["gflop"]) < 0.05
    assert abs(fl / cm.flash2_floor_bytes(N, d, e) - g["flop_per_byte"]) < 1
    assert abs(cm.standard_attention_bytes(N, d, e) / MiB - g["naive_MiB_about"]) < 0.05 * g["naive_MiB_about"]
    assert cm.attention_flops(1, 1, N, N, d, True) == fl / 2


def test_backward_saves():
    g = G["backward_saves"]
    assert g["heads"] * g["N"] * 4 / MiB == g["lse_MiB"]
    assert g["heads"] * g["N"] ** 2 * 2 / GiB == g["p_GiB_bf16"]


def test_gqa_bytes():
    g = G["gqa_bytes"]
    grouped = cm.gqa_kv_read_bytes(g["batch"], g["context"], g["kv_bytes_per_token"], g["tp"], g["group"], True)
    ungrouped = cm.gqa_kv_read_bytes(g["batch"], g["context"], g["kv_bytes_per_token"], g["tp"], g["group"], False)
    assert grouped / GiB == g["grouped_GiB"] and ungrouped / GiB == g["ungrouped_GiB"]


def test_paged_block():
    g = G["paged_block"]
    blk = cm.paged_block_bytes(g["page_tokens"], g["kv_heads"], g["d"], g["bytes_per_value"])
    assert blk == g["block_KiB"] * 1024
    assert abs(100 * 4 / blk - g["table_fraction_pct"]) < 0.0005
    assert g["tile_tokens"] // g["page_tokens"] == g["lookups_per_tile"]


def test_decode_bytes_for_the_workloads():
    # split-KV decode: 2 * 8 heads * 131072 * 128 * 2 B of K/V
    assert cm.decode_kv_bytes(1, 8, 131072, 128) == 536870912
    # paged decode: 64 sequences * 8 heads * 8192 tokens * 128 * 2 B * (K, V)
    assert cm.decode_kv_bytes(64, 8, 8192, 128) == 2147483648
    assert cm.decode_bytes(64, 64, 8, 1, 8192, 128, page_size=16) > cm.decode_kv_bytes(64, 8, 8192, 128)


def test_visible_pairs_brute_force():
    """The closed-loop count equals enumerating the mask (key j visible iff j <= i + S - T)."""
    for T, S in ((1, 7), (5, 5), (9, 4), (512, 8192), (33, 20), (3, 0)):
        brute = sum(1 for i in range(T) for j in range(S) if j <= i + S - T)
        assert cm.visible_pairs(T, S, True) == brute
        assert cm.visible_pairs(T, S, False) == T * S
    # square causal: N(N+1)/2, the exact count behind the "halved" convention
    assert cm.visible_pairs(4096, 4096, True) == 4096 * 4097 // 2
    assert cm.chunked_attention_flops(2, 3, [3, 5], 8) == 4.0 * 2 * 8 * (6 + 12)


def test_flash1_counting_trips():
    """The FlashAttention-1 count with two key tiles ("Counting trips across HBM"):
    K and V once, Q, O, m, l read twice, O, m, l written twice."""
    N, d = 256, 64
    e, es = 2, 4
    state = N * d * es + 2 * N * es
    assert cm.flash1_bytes(N, d, e, Bc=128, e_state=es) == 2 * N * d * e + 2 * N * d * e + 4 * state


def test_kv_outer_bytes_against_the_page_count():
    """Non-causal, one band: the kernel's count is the pages' FlashAttention-1 count
    less the first key tile's state read and the last one's state write, plus the
    final bf16 O and lse."""
    for N, d in ((4096, 128), (1024, 64), (640, 128)):
        state = N * (d * 4 + 8)
        expect = cm.flash1_bytes(N, d, 2, 128, 4) - 2 * state + N * (2 * d + 4)
        assert cm.kv_outer_bytes(1, 1, N, N, d) == expect
        # bands reload K and V once each
        assert cm.kv_outer_bytes(1, 1, N, N, d, row_bands=2) == expect + 2 * N * d * 2
    # causal, T = S = 256: tile 0 needs key tile 0 only, tile 1 both
    d = 64
    got = cm.kv_outer_bytes(1, 1, 256, 256, d, causal=True)
    q_reads = 3 * 128 * d * 2
    state_io = 2 * 128 * (d * 4 + 8)  # tile 1: state out after key tile 0, in before key tile 1
    assert got == q_reads + state_io + 256 * (2 * d + 4) + 2 * 256 * d * 2
    # T > S: a tile no key reaches writes O = 0 and lse only
    assert cm.kv_outer_bytes(1, 1, 256, 100, d, causal=True) == (
        128 * (2 * d + 4) + 128 * d * 2 + 128 * (2 * d + 4) + 2 * 100 * d * 2)
