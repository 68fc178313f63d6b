"""Ring-step prefill attention on the GPU against the fp64 oracle (parity tests).

Tolerances (bf16 inputs, fp32 accumulation): output max-abs <= 2e-2 and
mean-abs <= 2e-3; per-step lse = m + ln l within 2e-3; rows that see no key in
a step must be exactly the identity (-inf, 0, 0).
"""

import math

import numpy as np
import pytest
import torch

import context_ring_attention_cp_gb300 as cpa
from context_ring_attention_cp_gb300 import synth
from oracle import attention as OA
from oracle import ring as OR

from gpu_util import (LSE_ABS, assert_out_close, f64, ring_buffers, run_ring)

pytestmark = pytest.mark.gpu

EMIT, ACC, FIN = cpa.CP_MODE_EMIT, cpa.CP_MODE_ACCUMULATE, cpa.CP_MODE_FINALIZE

# (b, S, h_q, h_kv, d, cp, std): several 128-row tiles, ragged chunk tails (C % 128 != 0),
# odd and even GQA groups, cp = 1, a single-token chunk, batch > 1.
SMALL = [
    (1, 1024, 4, 4, 64, 2, 1.0),     # the tiny workload
    (2, 512, 4, 2, 128, 2, 0.5),
    (1, 1000, 2, 1, 128, 2, 1.0),    # C = 250: 128 + 122-row tiles
    (1, 768, 6, 2, 64, 4, 1.0),      # C = 96 < 128, g = 3 (a pair and a single)
    (1, 2048, 8, 2, 128, 8, 0.5),    # C = 128
    (1, 384, 3, 3, 64, 1, 1.0),      # cp = 1
    (1, 8, 2, 2, 64, 4, 1.0),        # C = 1
    (3, 640, 4, 1, 128, 5, 0.5),     # C = 64, g = 4, b = 3
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from context_ring_attention_cp_gb300 import _build
    _build.build()
    cpa.load_library()


@pytest.fixture(scope="module", autouse=True)
def _paired_tiles():
    # Multi-head launches under one wave of single tiles run one tile per CTA; the small
    # parity cases here would take that path.  Force two tiles per CTA (the path of every
    # launch of more than a wave); test_tile_pairing_modes_give_the_same_bits covers the rest.
    cpa.load_library()
    cpa.cp_set_kernel_choice(cpa.CP_KNOB_RING_PAIRING, 1)
    yield
    cpa.cp_set_kernel_choice(cpa.CP_KNOB_RING_PAIRING, -1)


def _inputs(b, S, hq, hkv, d, std, seed):
    return synth.prefill_inputs(b, S, hq, hkv, d, std=std, seed=seed, device="cuda")


@pytest.mark.parametrize("case", SMALL, ids=[str(c) for c in SMALL])
def test_full_ring_equals_causal_attention(case):
    b, S, hq, hkv, d, cp, std = case
    q, k, v = _inputs(b, S, hq, hkv, d, std, seed=hash(case) & 0xFFFF)
    o, m, l = run_ring(q, k, v, cp, 0, cp, EMIT | FIN)
    ref_out, ref_m, ref_l, _ = OA.full_causal_attention(f64(q), f64(k), f64(v), 1.0 / math.sqrt(d))
    assert_out_close(o.cpu().numpy(), ref_out, f"out {case}")
    lse = (m + torch.log(l)).cpu().numpy()
    assert np.abs(lse - (ref_m + np.log(ref_l))).max() <= LSE_ABS
    assert np.abs(m.cpu().numpy() - ref_m).max() <= LSE_ABS


@pytest.mark.parametrize("case", SMALL[:6], ids=[str(c) for c in SMALL[:6]])
def test_each_step_emits_the_oracle_step_triple(case):
    b, S, hq, hkv, d, cp, std = case
    q, k, v = _inputs(b, S, hq, hkv, d, std, seed=7 + (hash(case) & 0xFF))
    qf, kf, vf = f64(q), f64(k), f64(v)
    scale = 1.0 / math.sqrt(d)
    for t in range(cp):
        o, m, l = run_ring(q, k, v, cp, t, t + 1, EMIT)
        o, m, l = o.cpu().numpy(), m.cpu().numpy(), l.cpu().numpy()
        for r in range(cp):
            rows, rm, rl, ro = OR.ring_step_triple(qf, kf, vf, scale, cp, r, t)
            gm, gl = m[:, :, rows], l[:, :, rows]
            go = np.moveaxis(o[:, rows], 1, 2)  # [b, hq, rows, d]
            empty = np.isneginf(rm)
            assert np.all(np.isneginf(gm[empty])) and np.all(gl[empty] == 0) and np.all(go[empty] == 0)
            live = ~empty
            assert np.all(np.isfinite(gm[live])) and np.all(gl[live] > 0)
            assert np.abs((gm + np.log(np.where(live, gl, 1)))[live] - (rm + np.log(np.where(live, rl, 1)))[live]).max() <= LSE_ABS
            assert np.abs(gm[live] - rm[live]).max() <= LSE_ABS
            ref_out = ro[live] / rl[live][:, None]
            assert_out_close(go[live] / gl[live][:, None], ref_out, f"step {t} rank {r}")


@pytest.mark.parametrize("case", [SMALL[1], SMALL[3], SMALL[7], (1, 2048, 8, 2, 128, 4, 0.5)],
                         ids=["b2", "ragged_g3", "cp5", "whole_tiles_gqa4"])
def test_accumulate_steps_then_finalize(case):
    b, S, hq, hkv, d, cp, std = case
    q, k, v = _inputs(b, S, hq, hkv, d, std, seed=99)
    bufs = ring_buffers(b, S, hq, d, identity=True)
    order = list(range(cp))[::-1]  # any step order merges to the same result
    for i, t in enumerate(order):
        mode = ACC | (FIN if i == cp - 1 else 0)
        run_ring(q, k, v, cp, t, t + 1, mode, bufs)
    ref_out, ref_m, ref_l, _ = OA.full_causal_attention(f64(q), f64(k), f64(v), 1.0 / math.sqrt(d))
    assert_out_close(bufs[0].cpu().numpy(), ref_out, "accumulated")
    assert np.abs(bufs[1].cpu().numpy() - ref_m).max() <= LSE_ABS


@pytest.mark.parametrize("case", [SMALL[1], SMALL[2], SMALL[3], SMALL[4]],
                         ids=["b2", "ragged_250", "ragged_g3", "c128"])
def test_accumulate_into_the_identity_triple_equals_emit(case):
    # Against m = -inf, l = 0, O = 0 the merge weights are alpha = 0 and beta = 1, so
    # ACCUMULATE stores fmaf(0, 0, O * f) = O * f: the value EMIT stores, bit for bit.
    # Whole 128-row tiles combine in shared memory, ragged ones row by row; both are held
    # to EMIT here, at every step.
    b, S, hq, hkv, d, cp, std = case
    q, k, v = _inputs(b, S, hq, hkv, d, std, seed=31)
    for t in range(cp):
        acc = run_ring(q, k, v, cp, t, t + 1, ACC, ring_buffers(b, S, hq, d, identity=True))
        emit = run_ring(q, k, v, cp, t, t + 1, EMIT)
        for x, y in zip(acc, emit):
            assert torch.equal(x, y), f"step {t}"


def test_emit_then_merge_kernel_finalize_matches_fused():
    b, S, hq, hkv, d, cp = 1, 1024, 4, 2, 128, 4
    q, k, v = _inputs(b, S, hq, hkv, d, 0.5, seed=5)
    fo, fm, fl = run_ring(q, k, v, cp, 0, cp, EMIT | FIN)
    eo, em, el = run_ring(q, k, v, cp, 0, cp, EMIT)
    out = torch.empty_like(eo); mo = torch.empty_like(em); lo = torch.empty_like(el)
    cpa.cp_merge_partials(b, S, hq, d, 1, eo, em, el, out, mo, lo, finalize=True)
    torch.cuda.synchronize()
    assert torch.equal(mo, fm) and torch.equal(lo, fl)
    assert (out - fo).abs().max().item() <= 1e-6


def test_two_step_ranges_accumulate_to_full():
    b, S, hq, hkv, d, cp = 1, 2048, 4, 4, 64, 8
    q, k, v = _inputs(b, S, hq, hkv, d, 1.0, seed=6)
    bufs = ring_buffers(b, S, hq, d, identity=True)
    run_ring(q, k, v, cp, 0, 3, ACC, bufs)
    run_ring(q, k, v, cp, 3, cp, ACC | FIN, bufs)
    ref = run_ring(q, k, v, cp, 0, cp, EMIT | FIN)
    # P is rounded to bf16 against each launch's own exponent reference, so two
    # launches and one fused launch differ at that rounding level (both are
    # checked against the oracle below).
    assert (bufs[0] - ref[0]).abs().max().item() <= 5e-3
    ref_out, _, _, _ = OA.full_causal_attention(f64(q), f64(k), f64(v), 1.0 / math.sqrt(d))
    assert_out_close(bufs[0].cpu().numpy(), ref_out, "two ranges")


@pytest.mark.parametrize("case", [(1, 1536, 4, 2, 128, 1), (2, 1000, 3, 3, 64, 1), (1, 2048, 8, 2, 128, 4)])
def test_fused_finalize_is_bit_identical_to_emit_then_one_part_merge(case):
    # cp = 1 degeneracy (and any cp): the fused EMIT | FINALIZE launch equals an EMIT
    # launch followed by the merge kernel finalising its single part, bit for bit.
    b, S, hq, hkv, d, cp = case
    q, k, v = _inputs(b, S, hq, hkv, d, 0.5, seed=sum(case))
    fo, fm, fl = run_ring(q, k, v, cp, 0, cp, EMIT | FIN)
    eo, em, el = run_ring(q, k, v, cp, 0, cp, EMIT)
    out = torch.empty_like(eo); mo = torch.empty_like(em); lo = torch.empty_like(el)
    cpa.cp_merge_partials(b, S, hq, d, 1, eo, em, el, out, mo, lo, finalize=True)
    torch.cuda.synchronize()
    assert torch.equal(mo, fm) and torch.equal(lo, fl) and torch.equal(out, fo)


def test_cp1_equals_unsplit_and_any_cp_agrees():
    b, S, hq, hkv, d = 1, 1536, 4, 2, 128
    q, k, v = _inputs(b, S, hq, hkv, d, 0.5, seed=8)
    base = run_ring(q, k, v, 1, 0, 1, EMIT | FIN)[0]
    for cp in (2, 3, 4, 6):
        other = run_ring(q, k, v, cp, 0, cp, EMIT | FIN)[0]
        assert (other - base).abs().max().item() <= 2e-3, cp


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("ramp", ["up", "down"])
@pytest.mark.parametrize("heads", [(2, 2), (4, 2)])
def test_large_logit_growth_forces_exact_rescales(d, ramp, heads):
    # Key magnitudes ramp along the sequence so the running max of many rows grows
    # by far more than the 2^8 threshold between the tiles a query tile visits
    # (the ring visits the diagonal chunk first, then earlier chunks): O is
    # rescaled in TMEM, possibly several times per row.
    hq, hkv = heads
    b, S, cp = 1, 1024, 4
    q, k, v = _inputs(b, S, hq, hkv, d, 1.0, seed=9 + d)
    ramp_t = torch.linspace(0.0, 6.0, S, device="cuda")
    if ramp == "down":
        ramp_t = ramp_t.flip(0)
    k = (k.float() * ramp_t.view(1, S, 1, 1)).to(torch.bfloat16)
    q = (q.float() * 3.0).to(torch.bfloat16)
    o, m, l = run_ring(q, k, v, cp, 0, cp, EMIT | FIN)
    ref_out, ref_m, ref_l, _ = OA.full_causal_attention(f64(q), f64(k), f64(v), 1.0 / math.sqrt(d))
    assert_out_close(o.cpu().numpy(), ref_out, f"rescale d={d} {ramp} {heads}")
    assert np.abs(m.cpu().numpy() - ref_m).max() <= LSE_ABS
    assert np.abs((m + torch.log(l)).cpu().numpy() - (ref_m + np.log(ref_l))).max() <= LSE_ABS


def test_invalid_arguments_launch_nothing():
    q, k, v = _inputs(1, 256, 2, 2, 64, 1.0, seed=1)
    o, m, l = ring_buffers(1, 256, 2, 64)
    desc = cpa.make_desc(1, 256, 2, 2, 64, 3, 0.125, 1)  # 256 % 6 != 0
    with pytest.raises(cpa.CpError):
        cpa.cp_ring_step_partial_attn(desc, 0, 3, q, k, v, o, m, l, EMIT)
    desc = cpa.make_desc(1, 256, 2, 2, 64, 2, 0.125, 1)
    with pytest.raises(cpa.CpError):
        # a raw address skips the binding's tensor checks and reaches the C ABI's alignment check
        cpa.cp_ring_step_partial_attn(desc, 0, 2, q, k, v, o.data_ptr() + 4, m, l, EMIT)
    assert cpa.cp_take_device_status() == 0


SEQ = cpa.CP_LAYOUT_SEQUENTIAL


def _run_ranks(q, k, v, cp, layout, r0, r1, t0, t1, mode, bufs):
    b, S, hq, d = q.shape
    desc = cpa.make_desc(b, S, hq, k.shape[2], d, cp, 1.0 / math.sqrt(d), 1)
    cpa.cp_ring_rank_partial_attn(desc, layout, r0, r1, t0, t1, q, k, v, *bufs, mode)
    assert cpa.cp_take_device_status() == 0


@pytest.mark.parametrize("case", [SMALL[0], SMALL[1], SMALL[3], SMALL[4], SMALL[7]],
                         ids=["tiny", "b2", "ragged_g3", "cp8", "cp5"])
def test_sequential_layout_full_ring_equals_causal_attention(case):
    b, S, hq, hkv, d, cp, std = case
    q, k, v = _inputs(b, S, hq, hkv, d, std, seed=31)
    bufs = ring_buffers(b, S, hq, d)
    _run_ranks(q, k, v, cp, SEQ, 0, cp, 0, cp, EMIT | FIN, bufs)
    ref_out, ref_m, _, _ = OA.full_causal_attention(f64(q), f64(k), f64(v), 1.0 / math.sqrt(d))
    assert_out_close(bufs[0].cpu().numpy(), ref_out, f"sequential {case}")
    assert np.abs(bufs[1].cpu().numpy() - ref_m).max() <= LSE_ABS


def test_sequential_layout_step_triples():
    b, S, hq, hkv, d, cp, std = 1, 1024, 4, 2, 128, 4, 0.5
    q, k, v = _inputs(b, S, hq, hkv, d, std, seed=32)
    qf, kf, vf = f64(q), f64(k), f64(v)
    for t in range(cp):
        bufs = ring_buffers(b, S, hq, d)
        _run_ranks(q, k, v, cp, SEQ, 0, cp, t, t + 1, EMIT, bufs)
        o, m, l = (x.cpu().numpy() for x in bufs)
        for r in range(cp):
            rows, rm, rl, ro = OR.ring_step_triple(qf, kf, vf, 1.0 / math.sqrt(d), cp, r, t, layout="sequential")
            gm, gl, go = m[:, :, rows], l[:, :, rows], np.moveaxis(o[:, rows], 1, 2)
            empty = np.isneginf(rm)
            assert np.all(np.isneginf(gm[empty])) and np.all(gl[empty] == 0) and np.all(go[empty] == 0)
            live = ~empty
            if live.any():
                assert np.abs(gm[live] - rm[live]).max() <= LSE_ABS
                assert_out_close(go[live] / gl[live][:, None], ro[live] / rl[live][:, None], f"seq t{t} r{r}")


@pytest.mark.parametrize("heads", [(4, 2), (3, 3), (6, 2)], ids=["gqa2", "mha", "g3"])
@pytest.mark.parametrize("layout", [cpa.CP_LAYOUT_BALANCED, SEQ])
def test_rank_ranges_touch_only_their_rows_and_compose(layout, heads):
    b, S, d, cp = 1, 2048, 128, 4
    hq, hkv = heads
    q, k, v = _inputs(b, S, hq, hkv, d, 0.5, seed=33)
    full = ring_buffers(b, S, hq, d)
    _run_ranks(q, k, v, cp, layout, 0, cp, 0, cp, EMIT | FIN, full)
    lay = "sequential" if layout == SEQ else "balanced"
    parts = ring_buffers(b, S, hq, d)
    for x in parts:
        x.fill_(float("nan"))
    for r in range(cp):
        _run_ranks(q, k, v, cp, layout, r, r + 1, 0, cp, EMIT | FIN, parts)
        done = np.concatenate([OR.rank_rows(S, cp, rr, lay) for rr in range(r + 1)])
        rest = np.setdiff1d(np.arange(S), done)
        o = parts[0].cpu().numpy()
        assert np.isnan(o[0, rest]).all(), "a rank launch wrote rows it does not own"
        assert np.isfinite(o[0, done]).all()
    # each rank's rows match the all-ranks launch bit for bit (same tiles, same order)
    for x, y in zip(parts, full):
        assert torch.equal(x, y)


def test_bounded_wait_timeout_is_reported_and_recovers():
    """A wait that nothing completes gives up (about 1 s), records CP_ERR_TIMEOUT,
    ring launches skip their work until the status is taken, then work again."""
    import time
    assert cpa.cp_take_device_status() == 0
    b, S, hq, hkv, d, cp = 1, 512, 2, 2, 64, 2
    q, k, v = _inputs(b, S, hq, hkv, d, 1.0, seed=41)
    t0 = time.time()
    cpa.cp_selftest_wait_timeout()
    bufs = ring_buffers(b, S, hq, d)
    for x in bufs:
        x.fill_(float("nan"))
    desc = cpa.make_desc(b, S, hq, hkv, d, cp, 1.0 / math.sqrt(d), 1)
    cpa.cp_ring_step_partial_attn(desc, 0, cp, q, k, v, *bufs, EMIT | FIN)  # queued behind the stalled wait
    torch.cuda.synchronize()
    assert 0.5 < time.time() - t0 < 30.0
    assert all(torch.isnan(x).all() for x in bufs), "a ring launch ran while the status word held an error"
    assert cpa.cp_take_device_status() == cpa.CP_ERR_TIMEOUT
    assert cpa.cp_take_device_status() == 0  # taken: cleared
    o, m, l = run_ring(q, k, v, cp, 0, cp, EMIT | FIN)
    ref_out, _, _, _ = OA.full_causal_attention(f64(q), f64(k), f64(v), 1.0 / math.sqrt(d))
    assert_out_close(o.cpu().numpy(), ref_out, "after recovery")


@pytest.mark.parametrize("name", ["gqa", "long", "mha", "mha64", "gqa-sequential"])
def test_full_size_workload_sampled_rows(name):
    """The benchmark's launch (all steps, one launch, finalised) at full size; rows sampled.
    gqa-sequential: the GQA workload under the sequential chunk layout, one launch per
    virtual rank as the rank-balance measurement runs it."""
    w = synth.WORKLOADS[name.split("-")[0]]
    q, k, v = synth.prefill_inputs(w["b"], w["S"], w["h_q"], w["h_kv"], w["d"], std=w["std"], seed=w["seed"])
    if name.endswith("sequential"):
        o, m, l = ring_buffers(w["b"], w["S"], w["h_q"], w["d"])
        for r in range(w["cp"]):
            _run_ranks(q, k, v, w["cp"], SEQ, r, r + 1, 0, w["cp"], EMIT | FIN, (o, m, l))
    else:
        o, m, l = run_ring(q, k, v, w["cp"], 0, w["cp"], EMIT | FIN)
    rows = synth.sample_rows(w["S"], w["cp"], 64, seed=w["seed"])
    heads = [0, 5, w["h_q"] - 1]
    g = w["h_q"] // w["h_kv"]
    scale = 1.0 / math.sqrt(w["d"])
    for h in heads:
        kh = h // g
        qs = f64(q[0, rows, h:h + 1])                          # [R, 1, d]
        ks = f64(k[0, :, kh:kh + 1])[None]                    # [1, S, 1, d]
        vs = f64(v[0, :, kh:kh + 1])[None]
        qfull = np.zeros((1, w["S"], 1, w["d"]))
        qfull[0, rows] = qs
        ref_out, ref_m, ref_l = OA.causal_attention_rows(qfull, ks, vs, scale, 0, [0], rows)
        got = o[0, rows, h].cpu().numpy()
        assert_out_close(got, ref_out[0], f"{name} head {h}")
        lse = (m[0, h, rows] + torch.log(l[0, h, rows])).cpu().numpy()
        assert np.abs(lse - (ref_m[0] + np.log(ref_l[0]))).max() <= LSE_ABS
    del q, k, v, o, m, l
    torch.cuda.empty_cache()


@pytest.mark.parametrize("S", [16384, 16000], ids=["whole_tiles", "ragged_tiles"])
def test_grouped_item_order_writes_every_row_once(S):
    # 2 sequences x 8 kv heads of about 8 MB of K/V each: the full ring runs its CTAs in
    # four groups of (sequence, kv head) units (S 16000: chunks of 7 whole tiles and one of
    # 104 rows).  Every output row of every head must be written (NaN-filled buffers) and
    # sampled rows of heads in every group match the oracle.
    b, hq, hkv, d, cp = 2, 32, 8, 128, 8
    q, k, v = _inputs(b, S, hq, hkv, d, 0.5, seed=77)
    o = torch.full((b, S, hq, d), float("nan"), dtype=torch.float32, device="cuda")
    m = torch.full((b, hq, S), float("nan"), dtype=torch.float32, device="cuda")
    l = torch.full((b, hq, S), float("nan"), dtype=torch.float32, device="cuda")
    run_ring(q, k, v, cp, 0, cp, EMIT | FIN, (o, m, l))
    assert torch.isfinite(o).all() and torch.isfinite(m).all() and torch.isfinite(l).all()
    assert (l > 0).all()
    rows = synth.sample_rows(S, cp, 8, seed=77)
    g = hq // hkv
    scale = 1.0 / math.sqrt(d)
    for bi in range(b):
        for h in (0, 9, 18, 31):  # kv heads 0, 2, 4, 7
            kh = h // g
            qfull = np.zeros((1, S, 1, d))
            qfull[0, rows] = f64(q[bi, rows, h:h + 1])
            ks = f64(k[bi, :, kh:kh + 1])[None]
            vs = f64(v[bi, :, kh:kh + 1])[None]
            ref_out, ref_m, ref_l = OA.causal_attention_rows(qfull, ks, vs, scale, 0, [0], rows)
            assert_out_close(o[bi, rows, h].cpu().numpy(), ref_out[0], f"seq {bi} head {h}")
            lse = (m[bi, h, rows] + torch.log(l[bi, h, rows])).cpu().numpy()
            assert np.abs(lse - (ref_m[0] + np.log(ref_l[0]))).max() <= LSE_ABS
    # one launch per rank (each grouped the same way over its own items) writes exactly
    # that rank's rows, and together they equal the all-ranks launch bit for bit
    parts = tuple(torch.full_like(x, float("nan")) for x in (o, m, l))
    for r in range(cp):
        _run_ranks(q, k, v, cp, cpa.CP_LAYOUT_BALANCED, r, r + 1, 0, cp, EMIT | FIN, parts)
        mine = OR.rank_rows(S, cp, r, "balanced")
        assert torch.isfinite(parts[0][:, mine]).all(), f"rank {r} left rows unwritten"
    for x, y in zip(parts, (o, m, l)):
        assert torch.equal(x, y)
    del q, k, v, o, m, l, parts
    torch.cuda.empty_cache()


def _random_cases(n, seed):
    # Seeded random problems within what the oracle finishes in about a second each:
    # chunk lengths 1-299 (ragged tiles and single tokens), cp 1-8, GQA groups 1-4,
    # both head dimensions, batch 1-2, the workloads' two input scales (the output
    # tolerance is absolute, and P's bf16 rounding error grows with |V|), a random step
    # range and a random kernel choice (tile pairing and key-walk split automatic or forced).
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < n:
        cp = int(rng.choice([1, 2, 3, 4, 5, 8]))
        C = int(rng.integers(1, 300))
        hkv, g = int(rng.integers(1, 4)), int(rng.choice([1, 2, 3, 4]))
        b = int(rng.choice([1, 2]))
        S = 2 * cp * C
        if S > 1600 or hkv * g > 8 or b * S * hkv * g > 6400:
            continue
        d = int(rng.choice([64, 128]))
        std = float(rng.choice([0.5, 1.0]))
        t0 = int(rng.integers(0, cp))
        t1 = int(rng.integers(t0 + 1, cp + 1))
        pairing, split = int(rng.choice([-1, 0, 1])), int(rng.choice([-1, 0]))
        cases.append((b, S, hkv * g, hkv, d, cp, std, t0, t1, pairing, split))
    return cases


RANDOM = _random_cases(48, 20260101)


@pytest.mark.parametrize("case", RANDOM, ids=[f"r{i}" for i in range(len(RANDOM))])
def test_random_shapes_and_step_ranges_against_the_oracle(case):
    b, S, hq, hkv, d, cp, std, t0, t1, pairing, split = case
    cpa.cp_set_kernel_choice(cpa.CP_KNOB_RING_PAIRING, pairing)
    cpa.cp_set_kernel_choice(cpa.CP_KNOB_RING_KV_SPLIT, split)
    try:
        q, k, v = _inputs(b, S, hq, hkv, d, std, seed=1000 + S + hq + d)
        qf, kf, vf = f64(q), f64(k), f64(v)
        scale = 1.0 / math.sqrt(d)
        # the whole ring, finalised
        o, m, l = run_ring(q, k, v, cp, 0, cp, EMIT | FIN)
        ref_out, ref_m, ref_l, _ = OA.full_causal_attention(qf, kf, vf, scale)
        assert_out_close(o.cpu().numpy(), ref_out, f"out {case}")
        assert np.abs((m + torch.log(l)).cpu().numpy() - (ref_m + np.log(ref_l))).max() <= LSE_ABS
        # the merged triple of the step range [t0, t1)
        o, m, l = run_ring(q, k, v, cp, t0, t1, EMIT)
        rm, rl, ro = OR.ring_attention(qf, kf, vf, scale, cp, steps=range(t0, t1))
        gm, gl, go = m.cpu().numpy(), l.cpu().numpy(), np.moveaxis(o.cpu().numpy(), 1, 2)
        ro = np.moveaxis(ro, 1, 2)
        empty = np.isneginf(rm)
        assert np.all(np.isneginf(gm[empty])) and np.all(gl[empty] == 0) and np.all(go[empty] == 0)
        live = ~empty
        if live.any():
            assert np.abs(gm[live] - rm[live]).max() <= LSE_ABS
            assert np.abs(np.log(gl[live]) + gm[live] - np.log(rl[live]) - rm[live]).max() <= LSE_ABS
            assert_out_close(go[live] / gl[live][:, None], ro[live] / rl[live][:, None], f"steps {t0}-{t1} {case}")
    finally:
        cpa.cp_set_kernel_choice(cpa.CP_KNOB_RING_PAIRING, 1)
        cpa.cp_set_kernel_choice(cpa.CP_KNOB_RING_KV_SPLIT, -1)


@pytest.mark.parametrize("scale", [0.3, 2.0 / math.sqrt(128)])
def test_softmax_scale_is_the_one_passed(scale):
    # The scale is an explicit argument: a kernel that used 1/sqrt(d) regardless would
    # fail here (fused ring and one EMIT step, against the oracle at the same scale).
    b, S, hq, hkv, d, cp = 1, 1024, 4, 2, 128, 4
    q, k, v = _inputs(b, S, hq, hkv, d, 1.0, seed=44)
    desc = cpa.make_desc(b, S, hq, hkv, d, cp, scale, 1)
    o, m, l = ring_buffers(b, S, hq, d)
    cpa.cp_ring_step_partial_attn(desc, 0, cp, q, k, v, o, m, l, EMIT | FIN)
    assert cpa.cp_take_device_status() == 0
    qf, kf, vf = f64(q), f64(k), f64(v)
    ref_out, ref_m, ref_l, _ = OA.full_causal_attention(qf, kf, vf, scale)
    assert_out_close(o.cpu().numpy(), ref_out, f"scale {scale}")
    assert np.abs(m.cpu().numpy() - ref_m).max() <= LSE_ABS
    o1, m1, l1 = ring_buffers(b, S, hq, d)
    cpa.cp_ring_step_partial_attn(desc, 1, 2, q, k, v, o1, m1, l1, EMIT)
    assert cpa.cp_take_device_status() == 0
    m1n, l1n = m1.cpu().numpy(), l1.cpu().numpy()
    for r in range(cp):
        rows, rm, rl, ro = OR.ring_step_triple(qf, kf, vf, scale, cp, r, 1)
        live = ~np.isneginf(rm)
        gm, gl = m1n[:, :, rows], l1n[:, :, rows]
        assert np.abs(gm[live] - rm[live]).max() <= LSE_ABS
        assert np.abs((gm + np.log(np.where(live, gl, 1)))[live] - (rm + np.log(np.where(live, rl, 1)))[live]).max() <= LSE_ABS


def test_per_step_accumulate_chain_at_full_size():
    # How the method runs on cp devices: one launch per ring step, each merged into the
    # running triple, the last one normalising (GQA workload, full size).  P is rounded
    # to bf16 against each launch's own reference, so the chain and the fused ring agree
    # to that rounding; sampled rows are held to the oracle.
    w = synth.WORKLOADS["gqa"]
    b, S, hq, hkv, d, cp = w["b"], w["S"], w["h_q"], w["h_kv"], w["d"], w["cp"]
    q, k, v = synth.prefill_inputs(b, S, hq, hkv, d, std=w["std"], seed=w["seed"])
    chain = ring_buffers(b, S, hq, d, identity=True)
    for t in range(cp):
        run_ring(q, k, v, cp, t, t + 1, ACC | (FIN if t == cp - 1 else 0), chain)
    fused = run_ring(q, k, v, cp, 0, cp, EMIT | FIN)
    assert torch.equal(chain[1], fused[1])  # the max is exact in any grouping
    assert (chain[0] - fused[0]).abs().max().item() <= 5e-3
    rows = synth.sample_rows(S, cp, 16, seed=w["seed"] + 1)
    g = hq // hkv
    scale = 1.0 / math.sqrt(d)
    for h in (3, 30):
        kh = h // g
        qfull = np.zeros((1, S, 1, d))
        qfull[0, rows] = f64(q[0, rows, h:h + 1])
        ref_out, _, _ = OA.causal_attention_rows(qfull, f64(k[0, :, kh:kh + 1])[None], f64(v[0, :, kh:kh + 1])[None],
                                                 scale, 0, [0], rows)
        assert_out_close(chain[0][0, rows, h].cpu().numpy(), ref_out[0], f"chain head {h}")
    del q, k, v, chain, fused
    torch.cuda.empty_cache()


OVL = cpa.CP_MODE_OVERLAP_PREVIOUS


def _launch_chain(desc, q, k, v, bufs, cp, extra):
    # cp single-step launches with no synchronisation between them: EMIT, ACCUMULATE...,
    # the last one FINALIZE
    for t in range(cp):
        md = (EMIT if t == 0 else ACC) | (FIN if t == cp - 1 else 0) | extra
        cpa.cp_ring_step_partial_attn(desc, t, t + 1, q, k, v, *bufs, md)


def _nan_buffers(b, S, hq, d):
    o, m, l = ring_buffers(b, S, hq, d)
    for x in (o, m, l):
        x.fill_(float("nan"))
    return o, m, l


@pytest.mark.parametrize("case", SMALL, ids=[f"S{c[1]}_h{c[2]}x{c[3]}_d{c[4]}_cp{c[5]}_b{c[0]}" for c in SMALL])
def test_overlapped_step_chain_gives_the_same_bits(case):
    # With CP_MODE_OVERLAP_PREVIOUS each launch may start while the one before it runs and
    # waits for it before touching (o, m, l).  The chain is launched twice in a row into
    # the same buffers (the second chain's EMIT rewrites rows the first chain's last launch
    # is finalising) and must give the bits of the same chain with every launch serialised.
    b, S, hq, hkv, d, cp, std = case
    q, k, v = _inputs(b, S, hq, hkv, d, std, seed=S + 7 * hq + d)
    desc = cpa.make_desc(b, S, hq, hkv, d, cp, 1.0 / math.sqrt(d), 1)
    plain = _nan_buffers(b, S, hq, d)
    _launch_chain(desc, q, k, v, plain, cp, 0)
    torch.cuda.synchronize()
    ovl = _nan_buffers(b, S, hq, d)
    _launch_chain(desc, q, k, v, ovl, cp, OVL)
    _launch_chain(desc, q, k, v, ovl, cp, OVL)
    torch.cuda.synchronize()
    assert cpa.cp_take_device_status() == 0
    for x, y in zip(plain, ovl):
        assert torch.equal(x, y)


def test_overlap_flag_on_a_split_launch_changes_nothing():
    # Launches whose key walks are split over clusters run without the dependent-launch
    # attribute; the flag must still be accepted and give the same bits.
    cpa.cp_set_kernel_choice(cpa.CP_KNOB_RING_PAIRING, -1)
    try:
        b, S, hq, hkv, d, cp = 1, 1024, 4, 4, 64, 2
        q, k, v = _inputs(b, S, hq, hkv, d, 1.0, seed=4242)
        desc = cpa.make_desc(b, S, hq, hkv, d, cp, 1.0 / math.sqrt(d), 1)
        ref = _nan_buffers(b, S, hq, d)
        cpa.cp_ring_step_partial_attn(desc, 0, cp, q, k, v, *ref, EMIT | FIN)
        got = _nan_buffers(b, S, hq, d)
        cpa.cp_ring_step_partial_attn(desc, 0, cp, q, k, v, *got, EMIT | FIN | OVL)
        cpa.cp_ring_step_partial_attn(desc, 0, cp, q, k, v, *got, EMIT | FIN | OVL)
        torch.cuda.synchronize()
        assert cpa.cp_take_device_status() == 0
        for x, y in zip(ref, got):
            assert torch.equal(x, y)
    finally:
        cpa.cp_set_kernel_choice(cpa.CP_KNOB_RING_PAIRING, 1)


def test_overlapped_step_chain_at_full_size():
    # The GQA workload's ring as cp overlapped single-step launches: the same bits as the
    # serialised chain, whose agreement with the fused ring and the oracle is checked above.
    w = synth.WORKLOADS["gqa"]
    b, S, hq, hkv, d, cp = w["b"], w["S"], w["h_q"], w["h_kv"], w["d"], w["cp"]
    q, k, v = synth.prefill_inputs(b, S, hq, hkv, d, std=w["std"], seed=w["seed"])
    desc = cpa.make_desc(b, S, hq, hkv, d, cp, 1.0 / math.sqrt(d), 1)
    plain = _nan_buffers(b, S, hq, d)
    _launch_chain(desc, q, k, v, plain, cp, 0)
    torch.cuda.synchronize()
    ovl = _nan_buffers(b, S, hq, d)
    _launch_chain(desc, q, k, v, ovl, cp, OVL)
    torch.cuda.synchronize()
    assert cpa.cp_take_device_status() == 0
    for x, y in zip(plain, ovl):
        assert torch.equal(x, y)
    del q, k, v, plain, ovl
    torch.cuda.empty_cache()


# Odd groups (one query head per K/V head, or three): a CTA takes two consecutive 128-row
# tiles of one head, and the first tile sees one fully masked K/V tile on its chunk's
# diagonal.  Chunks of 250 rows (a 122-row second tile), 384 rows (a pair and a single
# tile) and 320 rows (a pair and a 64-row single).
MHA = [(1, 1000, 2, 2, 128, 2, 1.0), (2, 3072, 2, 2, 128, 4, 0.5), (1, 1280, 3, 3, 64, 2, 1.0),
       (1, 1536, 6, 2, 128, 2, 0.5), (2, 1000, 3, 1, 64, 2, 1.0)]


@pytest.mark.parametrize("case", MHA, ids=["C250", "C384_b2", "C320_d64", "g3_C384", "g3_C250_b2"])
def test_row_paired_tiles_full_ring_and_steps(case):
    b, S, hq, hkv, d, cp, std = case
    q, k, v = _inputs(b, S, hq, hkv, d, std, seed=3 + (hash(case) & 0xFF))
    qf, kf, vf = f64(q), f64(k), f64(v)
    scale = 1.0 / math.sqrt(d)
    o, m, l = run_ring(q, k, v, cp, 0, cp, EMIT | FIN)
    ref_out, ref_m, ref_l, _ = OA.full_causal_attention(qf, kf, vf, scale)
    assert_out_close(o.cpu().numpy(), ref_out, f"out {case}")
    assert np.abs(m.cpu().numpy() - ref_m).max() <= LSE_ABS
    # every ring step's triple, and the steps accumulated in reverse order
    bufs = ring_buffers(b, S, hq, d, identity=True)
    for t in range(cp):
        o, m, l = run_ring(q, k, v, cp, t, t + 1, EMIT)
        o, m, l = o.cpu().numpy(), m.cpu().numpy(), l.cpu().numpy()
        for r in range(cp):
            rows, rm, rl, ro = OR.ring_step_triple(qf, kf, vf, scale, cp, r, t)
            gm, gl = m[:, :, rows], l[:, :, rows]
            go = np.moveaxis(o[:, rows], 1, 2)
            empty = np.isneginf(rm)
            assert np.all(np.isneginf(gm[empty])) and np.all(gl[empty] == 0) and np.all(go[empty] == 0)
            live = ~empty
            assert np.abs(gm[live] - rm[live]).max() <= LSE_ABS
            assert_out_close(go[live] / gl[live][:, None], ro[live] / rl[live][:, None], f"step {t} rank {r}")
    for i, t in enumerate(range(cp - 1, -1, -1)):
        run_ring(q, k, v, cp, t, t + 1, ACC | (FIN if i == cp - 1 else 0), bufs)
    assert_out_close(bufs[0].cpu().numpy(), ref_out, "accumulated")


@pytest.mark.parametrize("case", [SMALL[0], SMALL[5], SMALL[6], MHA[0], MHA[1], MHA[2]],
                         ids=["tiny", "cp1", "C1", "C250", "C384_b2", "C320_d64"])
def test_tile_pairing_modes_give_the_same_bits(case):
    """Multi-head: one tile per CTA, two row tiles per CTA and the automatic choice compute
    every row alike."""
    b, S, hq, hkv, d, cp, std = case
    q, k, v = _inputs(b, S, hq, hkv, d, std, seed=11)
    got = {}
    cpa.cp_set_kernel_choice(cpa.CP_KNOB_RING_KV_SPLIT, 0)  # the split sums in another order
    try:
        for mode in ("single", "pair", "auto"):
            cpa.cp_set_kernel_choice(cpa.CP_KNOB_RING_PAIRING, {"single": 0, "pair": 1, "auto": -1}[mode])
            full = run_ring(q, k, v, cp, 0, cp, EMIT | FIN)
            step = run_ring(q, k, v, cp, cp - 1, cp, EMIT)
            acc = run_ring(q, k, v, cp, 0, 1, EMIT)
            if cp > 1:
                run_ring(q, k, v, cp, 1, 2, ACC | FIN, acc)
            got[mode] = (full, step, acc)
    finally:
        cpa.cp_set_kernel_choice(cpa.CP_KNOB_RING_PAIRING, 1)  # this module's setting
        cpa.cp_set_kernel_choice(cpa.CP_KNOB_RING_KV_SPLIT, -1)
    for mode in ("pair", "auto"):
        for xs, ys in zip(got["single"], got[mode]):
            for x, y in zip(xs, ys):
                assert torch.equal(x, y), f"{mode} {case}"


# Single query tiles filling at most half the GPU split each tile's key walk over a
# cluster of 2, 4 or 8 CTAs and merge the parts' triples on chip.  (b, S, h_q, h_kv, d,
# cp, std): the tiny workload (32 tiles, clusters of 4), ragged 122-row tiles, chunks
# shorter than a tile, cp = 1, one-token chunks (parts that see no key), 64 tiles
# (clusters of 2), b = 2.
SPLIT = [
    (1, 1024, 4, 4, 64, 2, 1.0),
    (1, 1000, 2, 2, 128, 2, 1.0),
    (2, 768, 3, 3, 64, 4, 1.0),
    (1, 384, 3, 3, 64, 1, 1.0),
    (1, 8, 2, 2, 64, 4, 1.0),
    (1, 4096, 2, 2, 128, 4, 0.5),
    (1, 2048, 1, 1, 128, 8, 0.5),
]


@pytest.mark.parametrize("case", SPLIT, ids=[str(c) for c in SPLIT])
def test_key_walk_split_over_a_cluster(case):
    b, S, hq, hkv, d, cp, std = case
    q, k, v = _inputs(b, S, hq, hkv, d, std, seed=500 + (hash(case) & 0xFF))
    qf, kf, vf = f64(q), f64(k), f64(v)
    scale = 1.0 / math.sqrt(d)
    cpa.cp_set_kernel_choice(cpa.CP_KNOB_RING_PAIRING, 0)  # one query tile per CTA: the split's form
    try:
        # the whole ring against the oracle, and against the unsplit launch
        o, m, l = run_ring(q, k, v, cp, 0, cp, EMIT | FIN)
        ref_out, ref_m, ref_l, _ = OA.full_causal_attention(qf, kf, vf, scale)
        assert_out_close(o.cpu().numpy(), ref_out, f"split {case}")
        assert np.abs(m.cpu().numpy() - ref_m).max() <= LSE_ABS
        assert np.abs((m + torch.log(l)).cpu().numpy() - (ref_m + np.log(ref_l))).max() <= LSE_ABS
        cpa.cp_set_kernel_choice(cpa.CP_KNOB_RING_KV_SPLIT, 0)
        uo, um, ul = run_ring(q, k, v, cp, 0, cp, EMIT | FIN)
        cpa.cp_set_kernel_choice(cpa.CP_KNOB_RING_KV_SPLIT, -1)
        assert torch.equal(m, um)  # the max is exact in any grouping
        # P is rounded to bf16 against each part's own exponent reference (as between two
        # step-range launches), so the outputs agree at that rounding level
        assert (o - uo).abs().max().item() <= 5e-3
        assert ((l - ul).abs() <= 1e-5 * ul.abs()).all()
        # every step's triple against the oracle's step triple (identity rows exact)
        for t in range(cp):
            so, sm, sl = run_ring(q, k, v, cp, t, t + 1, EMIT)
            so, sm, sl = so.cpu().numpy(), sm.cpu().numpy(), sl.cpu().numpy()
            for r in range(cp):
                rows, rm, rl, ro = OR.ring_step_triple(qf, kf, vf, scale, cp, r, t)
                gm, gl = sm[:, :, rows], sl[:, :, rows]
                go = np.moveaxis(so[:, rows], 1, 2)
                empty = np.isneginf(rm)
                assert np.all(np.isneginf(gm[empty])) and np.all(gl[empty] == 0) and np.all(go[empty] == 0)
                live = ~empty
                assert np.abs(gm[live] - rm[live]).max(initial=0.0) <= LSE_ABS
                if live.any():
                    assert_out_close(go[live] / gl[live][:, None], ro[live] / rl[live][:, None],
                                     f"split step {t} rank {r}")
        # the steps accumulated in reverse order, then finalised
        bufs = ring_buffers(b, S, hq, d, identity=True)
        for i, t in enumerate(range(cp)[::-1]):
            run_ring(q, k, v, cp, t, t + 1, ACC | (FIN if i == cp - 1 else 0), bufs)
        assert_out_close(bufs[0].cpu().numpy(), ref_out, f"split accumulated {case}")
        # ACCUMULATE into the identity triple stores what EMIT stores, bit for bit
        acc = run_ring(q, k, v, cp, 0, 1, ACC, ring_buffers(b, S, hq, d, identity=True))
        emit = run_ring(q, k, v, cp, 0, 1, EMIT)
        for x, y in zip(acc, emit):
            assert torch.equal(x, y)
    finally:
        cpa.cp_set_kernel_choice(cpa.CP_KNOB_RING_PAIRING, 1)  # this module's setting
        cpa.cp_set_kernel_choice(cpa.CP_KNOB_RING_KV_SPLIT, -1)


def test_split_rank_launches_write_their_rows_and_compose():
    # One launch per virtual rank (balanced layout) has few single tiles, so each splits its
    # key walks over larger clusters than the all-ranks launch: every rank writes exactly
    # its own rows, and together they give the oracle's attention.
    b, S, hq, hkv, d, cp, std = 1, 2048, 2, 2, 64, 4, 1.0
    q, k, v = _inputs(b, S, hq, hkv, d, std, seed=77)
    cpa.cp_set_kernel_choice(cpa.CP_KNOB_RING_PAIRING, 0)
    try:
        bufs = ring_buffers(b, S, hq, d)
        for x in bufs:
            x.fill_(float("nan"))
        C = S // (2 * cp)
        for r in range(cp):
            _run_ranks(q, k, v, cp, cpa.CP_LAYOUT_BALANCED, r, r + 1, 0, cp, EMIT | FIN, bufs)
            o = bufs[0].cpu().numpy()
            own = np.zeros(S, bool)
            for rr in range(r + 1):
                own[rr * C:(rr + 1) * C] = True
                own[(2 * cp - 1 - rr) * C:(2 * cp - rr) * C] = True
            assert np.isfinite(o[0, own]).all() and np.isnan(o[0, ~own]).all(), f"rank {r}"
        ref_out, ref_m, _, _ = OA.full_causal_attention(f64(q), f64(k), f64(v), 1.0 / math.sqrt(d))
        assert_out_close(bufs[0].cpu().numpy(), ref_out, "split rank launches")
        assert np.abs(bufs[1].cpu().numpy() - ref_m).max() <= LSE_ABS
        full = run_ring(q, k, v, cp, 0, cp, EMIT | FIN)
        assert torch.equal(full[1], bufs[1])  # the max is exact in any grouping
        assert (full[0] - bufs[0]).abs().max().item() <= 5e-3
    finally:
        cpa.cp_set_kernel_choice(cpa.CP_KNOB_RING_PAIRING, 1)  # this module's setting


def test_split_launch_skips_while_the_status_holds_an_error():
    """A split launch (clusters of 4) queued behind a wait that gives up writes nothing and
    completes: every CTA of every cluster passes both cluster barriers on the skip path."""
    import time
    assert cpa.cp_take_device_status() == 0
    b, S, hq, hkv, d, cp = 1, 1024, 4, 4, 64, 2  # the tiny workload's shape
    q, k, v = _inputs(b, S, hq, hkv, d, 1.0, seed=42)
    cpa.cp_set_kernel_choice(cpa.CP_KNOB_RING_PAIRING, 0)
    try:
        t0 = time.time()
        cpa.cp_selftest_wait_timeout()
        bufs = ring_buffers(b, S, hq, d)
        for x in bufs:
            x.fill_(float("nan"))
        desc = cpa.make_desc(b, S, hq, hkv, d, cp, 1.0 / math.sqrt(d), 1)
        cpa.cp_ring_step_partial_attn(desc, 0, cp, q, k, v, *bufs, EMIT | FIN)
        torch.cuda.synchronize()
        assert 0.5 < time.time() - t0 < 30.0
        assert all(torch.isnan(x).all() for x in bufs), "a split launch ran while the status word held an error"
        assert cpa.cp_take_device_status() == cpa.CP_ERR_TIMEOUT
        o, m, l = run_ring(q, k, v, cp, 0, cp, EMIT | FIN)
        ref_out, _, _, _ = OA.full_causal_attention(f64(q), f64(k), f64(v), 1.0 / math.sqrt(d))
        assert_out_close(o.cpu().numpy(), ref_out, "split after recovery")
    finally:
        cpa.cp_set_kernel_choice(cpa.CP_KNOB_RING_PAIRING, 1)  # this module's setting
