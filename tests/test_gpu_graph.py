"""CUDA-graph capture of the device entry points.

A latency-bound caller (a decode loop, a chain of ring steps) captures the library's
launches once and replays them.  Every device entry point except the host-buffer ring
is capturable: no allocation, no synchronisation and no pageable copy inside.  A
replayed graph must give the same bits as the same calls made eagerly.
"""

import math

import pytest
import torch

import context_ring_attention_cp_gb300 as cpa
from context_ring_attention_cp_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from context_ring_attention_cp_gb300 import _build
    _build.build()
    cpa.load_library()


def _capture(fn, stream):
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=stream):
        fn(torch.cuda.current_stream())
    return g


def _replay(g, stream, times=2):
    with torch.cuda.stream(stream):
        for _ in range(times):
            g.replay()
    torch.cuda.synchronize()


@pytest.mark.parametrize("overlap", [False, True], ids=["plain", "overlapped"])
def test_ring_step_chain_replays_bit_equal(overlap):
    # cp single-step launches: EMIT, then ACCUMULATE, the last one FINALIZE.  The chain
    # rewrites its whole running triple, so replaying it twice gives the same bits.
    # Overlapped, the captured launches after the first are programmatic dependents of
    # the one before (graph edges of that kind); the eager chain they are held to is plain.
    b, S, hq, hkv, d, cp = 1, 4096, 8, 2, 128, 4
    q, k, v = synth.prefill_inputs(b, S, hq, hkv, d, std=0.5, seed=91)
    desc = cpa.make_desc(b, S, hq, hkv, d, cp, 1.0 / math.sqrt(d), 1)

    def buffers():
        o = torch.full((b, S, hq, d), float("nan"), dtype=torch.float32, device="cuda")
        m = torch.full((b, hq, S), float("nan"), dtype=torch.float32, device="cuda")
        return o, m, torch.full_like(m, float("nan"))

    def chain(o, m, l, stream, extra=0):
        for t in range(cp):
            mode = cpa.CP_MODE_EMIT if t == 0 else cpa.CP_MODE_ACCUMULATE
            if t == cp - 1:
                mode |= cpa.CP_MODE_FINALIZE
            cpa.cp_ring_step_partial_attn(desc, t, t + 1, q, k, v, o, m, l, mode | extra, stream)

    eager = buffers()
    chain(*eager, torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert cpa.cp_take_device_status() == 0

    side = torch.cuda.Stream()
    graphed = buffers()
    extra = cpa.CP_MODE_OVERLAP_PREVIOUS if overlap else 0
    g = _capture(lambda st: chain(*graphed, st, extra), side)
    _replay(g, side)
    assert cpa.cp_take_device_status() == 0
    for x, y in zip(eager, graphed):
        assert torch.equal(x, y)


def test_fused_ring_replays_bit_equal():
    b, S, hq, hkv, d, cp = 2, 2048, 4, 4, 64, 2
    q, k, v = synth.prefill_inputs(b, S, hq, hkv, d, std=0.5, seed=92)
    desc = cpa.make_desc(b, S, hq, hkv, d, cp, 1.0 / math.sqrt(d), 1)
    mode = cpa.CP_MODE_EMIT | cpa.CP_MODE_FINALIZE
    outs = []
    for graphed in (False, True):
        o = torch.full((b, S, hq, d), float("nan"), dtype=torch.float32, device="cuda")
        m = torch.full((b, hq, S), float("nan"), dtype=torch.float32, device="cuda")
        l = torch.full_like(m, float("nan"))
        fn = lambda st: cpa.cp_ring_step_partial_attn(desc, 0, cp, q, k, v, o, m, l, mode, st)  # noqa: E731
        if graphed:
            side = torch.cuda.Stream()
            _replay(_capture(fn, side), side)
        else:
            fn(torch.cuda.current_stream())
            torch.cuda.synchronize()
        assert cpa.cp_take_device_status() == 0
        outs.append((o, m, l))
    for x, y in zip(*outs):
        assert torch.equal(x, y)


@pytest.mark.parametrize("shape", [(1, 1024, 4, 4, 64, 2), (1, 1000, 2, 2, 128, 2)], ids=["tiny", "ragged_d128"])
def test_split_ring_replays_bit_equal(shape):
    # Few single query tiles: each tile's key walk is split over a cluster of CTAs (a
    # cluster launch), which replays from a graph with the eager call's bits.
    b, S, hq, hkv, d, cp = shape
    q, k, v = synth.prefill_inputs(b, S, hq, hkv, d, std=1.0, seed=94)
    desc = cpa.make_desc(b, S, hq, hkv, d, cp, 1.0 / math.sqrt(d), 1)
    mode = cpa.CP_MODE_EMIT | cpa.CP_MODE_FINALIZE
    outs = []
    for graphed in (False, True):
        o = torch.full((b, S, hq, d), float("nan"), dtype=torch.float32, device="cuda")
        m = torch.full((b, hq, S), float("nan"), dtype=torch.float32, device="cuda")
        l = torch.full_like(m, float("nan"))
        fn = lambda st: cpa.cp_ring_step_partial_attn(desc, 0, cp, q, k, v, o, m, l, mode, st)  # noqa: E731
        if graphed:
            side = torch.cuda.Stream()
            _replay(_capture(fn, side), side)
        else:
            fn(torch.cuda.current_stream())
            torch.cuda.synchronize()
        assert cpa.cp_take_device_status() == 0
        assert torch.isfinite(o).all()
        outs.append((o, m, l))
    for x, y in zip(*outs):
        assert torch.equal(x, y)


def test_merge_and_tree_replay_bit_equal():
    n, b, rows, heads, d = 8, 1, 300, 3, 128
    gen = torch.Generator(device="cpu").manual_seed(93)
    o = torch.randn((n, b, rows, heads, d), generator=gen).cuda()
    m = torch.randn((n, b, heads, rows), generator=gen).cuda()
    l = torch.rand((n, b, heads, rows), generator=gen).add_(0.5).cuda()
    ws = torch.empty(cpa.cp_merge_tree_workspace_bytes(b, rows, heads, d, n) // 4 + 1, dtype=torch.float32,
                     device="cuda")
    order = [3, 1, 7, 0, 5, 2, 6, 4]

    def run(outs, st):
        cpa.cp_merge_partials(b, rows, heads, d, n, o, m, l, *outs[0], order=order, finalize=True, stream=st)
        cpa.cp_merge_partials_tree(b, rows, heads, d, n, o, m, l, ws, ws.numel() * 4, *outs[1], finalize=True,
                                   stream=st)

    def buffers():
        res = []
        for _ in range(2):
            oo = torch.full((b, rows, heads, d), float("nan"), dtype=torch.float32, device="cuda")
            mo = torch.full((b, heads, rows), float("nan"), dtype=torch.float32, device="cuda")
            res.append((oo, mo, torch.full_like(mo, float("nan"))))
        return res

    eager = buffers()
    run(eager, torch.cuda.current_stream())
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    graphed = buffers()
    _replay(_capture(lambda st: run(graphed, st), side), side)
    for a, c in zip(eager, graphed):
        for x, y in zip(a, c):
            assert torch.equal(x, y)


@pytest.mark.parametrize("case", [(2, 4096, 4, 4, 128, 4), (2, 4096, 16, 1, 256, 4)],
                         ids=["streaming", "shared_kv"])
def test_decode_replays_bit_equal(case):
    b, L, hq, hkv, d, cp = case
    q, k, v = synth.decode_inputs(b, L, hq, hkv, d, seed=94)
    desc = cpa.make_desc(b, L, hq, hkv, d, cp, 1.0 / math.sqrt(d), 0)
    ws_bytes = cpa.cp_passq_workspace_bytes(desc)
    outs = []
    for graphed in (False, True):
        ws = torch.empty(ws_bytes // 4, dtype=torch.float32, device="cuda")
        out = torch.full((b, hq, d), float("nan"), dtype=torch.float32, device="cuda")
        mo = torch.full((b, hq), float("nan"), dtype=torch.float32, device="cuda")
        lo = torch.full_like(mo, float("nan"))
        fn = lambda st: cpa.cp_passq_decode(desc, q, k, v, ws, ws_bytes, out, mo, lo, st)  # noqa: E731
        if graphed:
            side = torch.cuda.Stream()
            _replay(_capture(fn, side), side)
        else:
            fn(torch.cuda.current_stream())
            torch.cuda.synchronize()
        assert cpa.cp_take_device_status() == 0
        outs.append((out, mo, lo))
    for x, y in zip(*outs):
        assert torch.equal(x, y)
