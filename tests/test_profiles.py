"""The committed DRAM traffic figures against the byte model: every kernel's measured
read + write bytes per launch must be its algorithmic bytes within a few percent (a
kernel that re-read its inputs, or a figure taken on another workload, would fail).
The prefill figure may sit below the compulsory bytes: part of O is still in L2 when
the launch ends, and ncu counts only DRAM writes."""

import os

import pytest

import fa_inputs as fi
from attention_fa2_attn_gb300 import costmodel as cm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _traffic():
    out = {}
    for line in open(os.path.join(ROOT, "profiles", "traffic.txt")):
        if line.startswith("#") or not line.strip():
            continue
        parts = line.split()
        out[parts[0]] = (parts[1], float(parts[3]), parts[4])
    return out


def _expected():
    w, s, pg = fi.PREFILL_MHA, fi.SPLITKV_DECODE, fi.PAGED_DECODE
    return {
        "prefill_tc_kernel": (w.name, cm.prefill_compulsory_bytes(w.B, w.Hq, w.Hkv, w.T, w.S, w.d), 0.80, 1.05),
        "decode_kernel_splitkv": (s.name, cm.decode_bytes(s.B, s.Hq, s.Hkv, s.T, s.S, s.d), 0.99, 1.03),
        "decode_kernel_paged": (pg.name, cm.decode_bytes(pg.B, pg.Hq, pg.Hkv, pg.T, pg.S, pg.d, page_size=pg.page_size),
                                0.99, 1.03),
        "kv_outer_kernel_one_cta_per_head": (w.name, cm.kv_outer_bytes(w.B, w.Hq, w.T, w.S, w.d, w.causal, 1), 0.97,
                                             1.03),
    }


@pytest.mark.parametrize("kernel", sorted(_expected()))
def test_measured_traffic_matches_the_byte_model(kernel):
    t = _traffic()
    assert kernel in t, f"{kernel} has no traffic line"
    src, measured, workload = t[kernel]
    name, algorithmic, lo, hi = _expected()[kernel]
    assert workload == name, (workload, name)
    assert os.path.exists(os.path.join(ROOT, "attention_fa2_attn_gb300", "csrc", src)), src
    ratio = measured / algorithmic
    assert lo <= ratio <= hi, f"{kernel}: measured {measured:.4g} B vs algorithmic {algorithmic:.4g} B ({ratio:.3f})"
