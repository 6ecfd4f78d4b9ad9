"""The entry points under CUDA-graph capture and on concurrent streams.

Every call is asynchronous on the caller's stream and its kernels are
deterministic (no atomics, fixed reduction orders), so a graph replay, or the
same calls spread over several streams at once, must give results bit-identical
to plain calls on the same inputs.
"""

import pytest
import torch

import fa_inputs as fi

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _fa():
    import attention_fa2_attn_gb300 as fa

    return fa


class _Problem:
    """Inputs of four calls: causal GQA prefill, split-KV decode, paged decode over a
    ragged batch, and the backward of the prefill."""

    def __init__(self, seed):
        self.pq, self.pk, self.pv = (x.to(DEV) for x in fi.qkv(1, 8, 2, 300, 520, 128, seed))
        self.dq_, self.dk_, self.dv_ = (x.to(DEV) for x in fi.qkv(2, 16, 4, 1, 3000, 64, seed + 1))
        kp, vp, table, _ = fi.paged_kv(3, 2, 900, 128, 16, seed + 2)
        self.kp, self.vp, self.table = kp.to(DEV), vp.to(DEV), table.to(DEV)
        self.sl = torch.tensor([900, 411, 17], dtype=torch.int32, device=DEV)
        self.tq = fi.decode_q(3, 8, 1, 128, seed + 3).to(DEV)
        self.do = fi.randn((1, 8, 300, 128), seed + 4).to(DEV)

    def copy_from(self, other):
        for name in ("pq", "pk", "pv", "dq_", "dk_", "dv_", "kp", "vp", "table", "sl", "tq", "do"):
            getattr(self, name).copy_(getattr(other, name))


def _run(fa, x):
    """The four calls on the current stream; returns their outputs."""
    o, lse = fa.fa_fwd(x.pq, x.pk, x.pv, causal=True)
    od, ld = fa.fa_decode_splitkv(x.dq_, x.dk_, x.dv_, causal=True, num_splits=6)
    op, lp = fa.fa_decode_paged(x.tq, x.kp, x.vp, x.table, x.sl, causal=True, num_splits=3)
    g = fa.fa_bwd(x.pq, x.pk, x.pv, o, lse, x.do, causal=True)
    return (o, lse, od, ld, op, lp) + tuple(g)


def _assert_same(a, b, what):
    for i, (x, y) in enumerate(zip(a, b)):
        assert torch.equal(x, y), f"{what}: output {i} differs"


def test_graph_replay_matches_plain_calls():
    fa = _fa()
    static = _Problem(1100)
    _run(fa, static)  # first calls outside capture (library state, kernel attributes)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            outs = _run(fa, static)
    torch.cuda.synchronize()
    for seed in (1200, 1300):
        fresh = _Problem(seed)
        static.copy_from(fresh)
        graph.replay()
        torch.cuda.synchronize()
        _assert_same(outs, _run(fa, fresh), f"replay with inputs {seed}")
    st, word = fa.fa_get_last_device_error()
    assert st == 0, hex(word)


def test_concurrent_streams_match_plain_calls():
    """Three problems issued on three streams without waiting for one another."""
    fa = _fa()
    probs = [_Problem(1400 + 100 * i) for i in range(3)]
    ref = [_run(fa, p) for p in probs]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in probs]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    got = []
    for p, s in zip(probs, streams):
        with torch.cuda.stream(s):
            got.append(_run(fa, p))
    torch.cuda.synchronize()
    for i, (a, b) in enumerate(zip(got, ref)):
        _assert_same(a, b, f"stream {i}")
    st, word = fa.fa_get_last_device_error()
    assert st == 0, hex(word)


def test_launch_after_event_wait_sees_the_copied_inputs():
    """A call that follows another call on its stream launches as a programmatic
    dependent of it, but an event wait between them (inputs copied on another
    stream) must still hold it back: the 201 MB host-to-device copy below takes
    about a millisecond, far longer than the short call ahead on the stream, so a
    launch that ignored the event would read the zero-filled buffers."""
    fa = _fa()
    shape_q, shape_kv = (4, 16, 4096, 128), (4, 16, 4096, 128)
    qh, kh, vh = (fi.randn(s, 1500 + i).pin_memory() for i, s in enumerate((shape_q, shape_kv, shape_kv)))
    q1, k1, v1 = (torch.zeros(s, dtype=torch.bfloat16, device=DEV) for s in (shape_q, shape_kv, shape_kv))
    tq, tk, tv = (x.to(DEV) for x in fi.qkv(1, 1, 1, 64, 64, 128, 1503))
    copy_stream, work_stream = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    copied = torch.cuda.Event()
    with torch.cuda.stream(copy_stream):
        for dst, src in ((q1, qh), (k1, kh), (v1, vh)):
            dst.copy_(src, non_blocking=True)
        copied.record(copy_stream)
    with torch.cuda.stream(work_stream):
        fa.fa_fwd(tq, tk, tv)  # a short call ahead on the stream
        work_stream.wait_event(copied)
        o, lse = fa.fa_fwd(q1, k1, v1)
    torch.cuda.synchronize()
    o_ref, lse_ref = fa.fa_fwd(q1, k1, v1)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
