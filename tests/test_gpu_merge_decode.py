"""LSE merge and pass-Q decode on the GPU against the fp64 oracle (parity tests).

Merge tolerance: per row, max|gpu - ref| / max|ref| <= 1e-5, for the oracle and
between any two merge orders; m is exact (max is order-free).  Decode: output
max-abs <= 2e-2, mean-abs <= 2e-3, lse within 2e-3.
"""

import math

import numpy as np
import pytest
import torch

import context_ring_attention_cp_gb300 as cpa
from context_ring_attention_cp_gb300 import synth
from oracle import attention as OA
from oracle import ring as OR

from gpu_util import LSE_ABS, MERGE_REL, assert_out_close, assert_rowwise_rel, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from context_ring_attention_cp_gb300 import _build
    _build.build()
    cpa.load_library()


def _merge(o, m, l, order=None, finalize=False):
    n, b, rows, heads, d = o.shape
    oo = torch.empty((b, rows, heads, d), dtype=torch.float32, device=o.device)
    mo = torch.empty((b, heads, rows), dtype=torch.float32, device=o.device)
    lo = torch.empty_like(mo)
    cpa.cp_merge_partials(b, rows, heads, d, n, o, m, l, oo, mo, lo, order=order, finalize=finalize)
    return oo, mo, lo


def _oracle_parts(o, m, l, heads_sel):
    """Oracle-layout triples [rows*heads_sel] for each part (fp64)."""
    parts = []
    for p in range(o.shape[0]):
        om = o[p, 0][:, heads_sel].cpu().double().numpy()          # [rows, H, d]
        mm = m[p, 0][heads_sel].cpu().double().numpy().T            # [rows, H]
        ll = l[p, 0][heads_sel].cpu().double().numpy().T
        parts.append((mm, ll, om))
    return parts


@pytest.mark.parametrize("shape", [(4, 1, 37, 3, 8), (32, 1, 96, 5, 128), (7, 2, 33, 2, 64), (3, 1, 5, 2, 512),
                                   (256, 1, 32, 1, 16), (1, 1, 70, 4, 128)])
def test_merge_matches_oracle_small(shape):
    n, b, rows, heads, d = shape
    draws = [synth.merge_parts(n, heads, rows, d, spread=80.0, seed=n * 31 + d + bi) for bi in range(b)]
    o = torch.cat([x[0] for x in draws], dim=1).contiguous()  # [n, b, rows, heads, d]
    m = torch.cat([x[1] for x in draws], dim=1).contiguous()  # [n, b, heads, rows]
    l = torch.cat([x[2] for x in draws], dim=1).contiguous()
    rng = np.random.default_rng(n)
    order = rng.permutation(n)
    for fin in (False, True):
        go, gm, gl = _merge(o, m, l, order=order, finalize=fin)
        torch.cuda.synchronize()
        for bi in range(b):
            parts = [(m[p, bi].T.cpu().double().numpy(), l[p, bi].T.cpu().double().numpy(),
                      o[p, bi].cpu().double().numpy()) for p in range(n)]
            rm, rl, ro = OR.merge_in_order(parts, order)
            assert np.array_equal(gm[bi].T.cpu().double().numpy(), rm)
            assert np.abs(gl[bi].T.cpu().double().numpy() - rl).max() <= MERGE_REL * max(1.0, np.abs(rl).max())
            if fin:
                ref, _ = OR.finalize((rm, rl, ro))
            else:
                ref = ro
            assert_rowwise_rel(go[bi].cpu().numpy(), ref, MERGE_REL, f"merge {shape} fin={fin}")


def test_merge_identity_rows_and_single_part():
    n, rows, heads, d = 3, 40, 2, 32
    o, m, l = synth.merge_parts(n, heads, rows, d, seed=4)
    m[:, :, :, 7] = -math.inf; l[:, :, :, 7] = 0; o[:, :, 7] = 0  # a row that is the identity everywhere
    go, gm, gl = _merge(o, m, l, finalize=True)
    torch.cuda.synchronize()
    assert torch.isneginf(gm[0, :, 7]).all() and (gl[0, :, 7] == 0).all() and (go[0, 7] == 0).all()
    assert not torch.isnan(go).any()
    # one part is returned as is (m, l exact; O exact when not finalised)
    go1, gm1, gl1 = _merge(o[:1], m[:1], l[:1])
    torch.cuda.synchronize()
    assert torch.equal(gm1, m[0]) and torch.equal(gl1, l[0]) and torch.equal(go1, o[0])


def test_merge_stress_workload_orders_and_tree():
    """64 heads x 128 x 4096 rows, 32 parts, spread +-80: 10 seeded orders and one tree order."""
    w = synth.WORKLOADS["merge"]
    n, heads, rows, d = w["parts"], w["heads"], w["rows"], w["d"]
    o, m, l = synth.merge_parts(n, heads, rows, d, spread=w["spread"], seed=w["seed"])
    rng = np.random.default_rng(w["seed"])
    orders = [rng.permutation(n) for _ in range(10)]
    outs = []
    for order in orders:
        go, gm, gl = _merge(o, m, l, order=order)
        outs.append((go, gm, gl))
    torch.cuda.synchronize()
    # tree order: balanced pairwise merges over index order with n_parts = 2 calls
    level = [(o[p:p + 1], m[p:p + 1], l[p:p + 1]) for p in range(n)]
    while len(level) > 1:
        nxt = []
        for i in range(0, len(level), 2):
            a, b = level[i], level[i + 1]
            co, cm, cl = _merge(torch.cat([a[0], b[0]]), torch.cat([a[1], b[1]]), torch.cat([a[2], b[2]]))
            nxt.append((co.unsqueeze(0), cm.unsqueeze(0), cl.unsqueeze(0)))
        level = nxt
    tree = (level[0][0][0], level[0][1][0], level[0][2][0])
    torch.cuda.synchronize()
    ref_o, ref_m, ref_l = outs[0]
    for go, gm, gl in outs[1:] + [tree]:
        assert torch.equal(gm, ref_m)  # max is exact in any order
        assert ((gl - ref_l).abs() <= MERGE_REL * ref_l.abs()).all()
        err = (go - ref_o).abs().amax(dim=-1)
        scale = ref_o.abs().amax(dim=-1)
        assert (err <= MERGE_REL * scale).all()
    # oracle on a head subset (fp64 over all 32 parts, fold in the first order)
    hs = [0, 17, 63]
    parts = _oracle_parts(o, m, l, hs)
    rm, rl, ro = OR.merge_in_order(parts, orders[0])
    assert np.array_equal(ref_m[0][hs].T.cpu().double().numpy(), rm)
    assert_rowwise_rel(ref_o[0][:, hs].cpu().numpy(), ro, MERGE_REL, "merge stress vs oracle")
    assert np.abs(ref_l[0][hs].T.cpu().double().numpy() - rl).max() <= MERGE_REL * np.abs(rl).max()


def _merge_tree(o, m, l, finalize=False):
    n, b, rows, heads, d = o.shape
    nbytes = cpa.cp_merge_tree_workspace_bytes(b, rows, heads, d, n)
    ws = torch.empty(nbytes // 4, dtype=torch.float32, device=o.device)
    oo = torch.empty((b, rows, heads, d), dtype=torch.float32, device=o.device)
    mo = torch.empty((b, heads, rows), dtype=torch.float32, device=o.device)
    lo = torch.empty_like(mo)
    cpa.cp_merge_partials_tree(b, rows, heads, d, n, o, m, l, ws, nbytes, oo, mo, lo, finalize=finalize)
    return oo, mo, lo


@pytest.mark.parametrize("shape", [(2, 1, 37, 3, 8), (4, 2, 33, 2, 64), (8, 1, 96, 5, 128), (32, 1, 64, 4, 128),
                                   (256, 1, 16, 2, 16), (16, 3, 1, 16, 512)])
def test_tree_merge_matches_oracle_and_flat_merge(shape):
    n, b, rows, heads, d = shape
    draws = [synth.merge_parts(n, heads, rows, d, spread=80.0, seed=7 * n + d + bi) for bi in range(b)]
    o = torch.cat([x[0] for x in draws], dim=1).contiguous()
    m = torch.cat([x[1] for x in draws], dim=1).contiguous()
    l = torch.cat([x[2] for x in draws], dim=1).contiguous()
    for fin in (False, True):
        to, tm, tl = _merge_tree(o, m, l, finalize=fin)
        fo, fm, fl = _merge(o, m, l, finalize=fin)
        torch.cuda.synchronize()
        assert torch.equal(tm, fm)  # max is exact in any grouping
        assert ((tl - fl).abs() <= MERGE_REL * fl.abs()).all()
        assert_rowwise_rel(to.cpu().numpy(), fo.cpu().numpy().astype(np.float64), MERGE_REL, f"tree vs flat {shape}")
        for bi in range(b):
            parts = [(m[p, bi].T.cpu().double().numpy(), l[p, bi].T.cpu().double().numpy(),
                      o[p, bi].cpu().double().numpy()) for p in range(n)]
            rm, rl, ro = OR.merge_tree_halves(parts)
            assert np.array_equal(tm[bi].T.cpu().double().numpy(), rm)
            ref = OR.finalize((rm, rl, ro))[0] if fin else ro
            assert_rowwise_rel(to[bi].cpu().numpy(), ref, MERGE_REL, f"tree vs oracle {shape}")


def _random_merge_cases(n, seed):
    # Seeded random merges: 1-64 parts in a random fold order (and, for a power-of-two
    # count, the halving tree), batch 1-2, 1-199 rows, 1-5 heads, d any multiple of 4 up to
    # 512 (so both the register and the TMA-fed kernels run), ~1 % identity entries.
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        parts = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 13, 16, 31, 32, 47, 64]))
        d = int(rng.choice([4, 8, 36, 64, 128, 128, 200, 256, 512]))
        cases.append((parts, int(rng.integers(1, 3)), int(rng.integers(1, 200)), int(rng.integers(1, 6)), d))
    return cases


MERGE_RANDOM = _random_merge_cases(24, 20260103)


@pytest.mark.parametrize("shape", MERGE_RANDOM, ids=[f"r{i}" for i in range(len(MERGE_RANDOM))])
def test_random_merges_against_the_oracle(shape):
    n, b, rows, heads, d = shape
    draws = [synth.merge_parts(n, heads, rows, d, spread=80.0, seed=13 * n + d + rows + bi) for bi in range(b)]
    o = torch.cat([x[0] for x in draws], dim=1).contiguous()
    m = torch.cat([x[1] for x in draws], dim=1).contiguous()
    l = torch.cat([x[2] for x in draws], dim=1).contiguous()
    order = np.random.default_rng(n + rows).permutation(n)
    tree = n >= 2 and (n & (n - 1)) == 0
    for fin in (False, True):
        go, gm, gl = _merge(o, m, l, order=order, finalize=fin)
        if tree:
            to, tm, tl = _merge_tree(o, m, l, finalize=fin)
        torch.cuda.synchronize()
        for bi in range(b):
            parts = [(m[p, bi].T.cpu().double().numpy(), l[p, bi].T.cpu().double().numpy(),
                      o[p, bi].cpu().double().numpy()) for p in range(n)]
            rm, rl, ro = OR.merge_in_order(parts, order)
            assert np.array_equal(gm[bi].T.cpu().double().numpy(), rm)
            assert np.abs(gl[bi].T.cpu().double().numpy() - rl).max() <= MERGE_REL * max(1.0, np.abs(rl).max())
            ref = OR.finalize((rm, rl, ro))[0] if fin else ro
            assert_rowwise_rel(go[bi].cpu().numpy(), ref, MERGE_REL, f"merge {shape} fin={fin}")
            if tree:
                hm, hl, ho = OR.merge_tree_halves(parts)
                assert np.array_equal(tm[bi].T.cpu().double().numpy(), hm)
                href = OR.finalize((hm, hl, ho))[0] if fin else ho
                assert_rowwise_rel(to[bi].cpu().numpy(), href, MERGE_REL, f"tree {shape} fin={fin}")


def test_tree_merge_rejects_bad_part_counts():
    o, m, l = synth.merge_parts(3, 2, 8, 8, seed=1)
    with pytest.raises(cpa.CpError):
        cpa.cp_merge_tree_workspace_bytes(1, 8, 2, 8, 3)
    ws = torch.empty(1 << 16, dtype=torch.float32, device="cuda")
    out = torch.empty((1, 8, 2, 8), dtype=torch.float32, device="cuda")
    ml = torch.empty((1, 2, 8), dtype=torch.float32, device="cuda")
    with pytest.raises(cpa.CpError):
        cpa.cp_merge_partials_tree(1, 8, 2, 8, 3, o, m, l, ws, ws.numel() * 4, out, ml, ml.clone())


TREE_LEVEL_SHAPES = [(2, 2, 33, 3, 64), (8, 2, 33, 3, 64), (32, 1, 64, 4, 128), (64, 2, 20, 3, 32),
                     (128, 1, 24, 2, 64), (256, 1, 16, 2, 16),
                     # d = 128 with up to 64 parts: the TMA-fed kernels (ragged 16-row blocks, b > 1)
                     (2, 2, 33, 3, 128), (4, 1, 16, 1, 128), (8, 3, 40, 2, 128), (16, 1, 7, 5, 128),
                     (64, 2, 20, 3, 128)]


@pytest.mark.parametrize("kernel", [-1, 0], ids=["auto", "plain-load"])
@pytest.mark.parametrize("shape", TREE_LEVEL_SHAPES)
def test_tree_merge_equals_level_by_level_two_part_merges(shape, kernel):
    # The one-pass tree does at every node what a two-part merge does, so it must
    # equal the halving tree run level by level through cp_merge_partials bit for bit,
    # with the TMA-fed kernels (d = 128, up to 64 parts) and with the plain-load ones.
    if kernel == 0 and shape[-1] != 128:
        pytest.skip("only d = 128 has a second kernel")
    cpa.cp_set_kernel_choice(cpa.CP_KNOB_MERGE_KERNEL, kernel)
    try:
        _tree_vs_levels(shape)
    finally:
        cpa.cp_set_kernel_choice(cpa.CP_KNOB_MERGE_KERNEL, -1)


def _tree_vs_levels(shape):
    n, b, rows, heads, d = shape
    draws = [synth.merge_parts(n, heads, rows, d, spread=80.0, seed=11 * n + bi) for bi in range(b)]
    o = torch.cat([x[0] for x in draws], dim=1).contiguous()
    m = torch.cat([x[1] for x in draws], dim=1).contiguous()
    l = torch.cat([x[2] for x in draws], dim=1).contiguous()
    for fin in (False, True):
        to, tm, tl = _merge_tree(o, m, l, finalize=fin)
        lo, lm, ll = o, m, l
        k = n
        while k >= 2:
            # level: part i with part i + k/2, as one two-part merge over (i, batch)
            last = k == 2
            oo = torch.empty((k // 2 * b, rows, heads, d), dtype=torch.float32, device="cuda")
            mo = torch.empty((k // 2 * b, heads, rows), dtype=torch.float32, device="cuda")
            lo2 = torch.empty_like(mo)
            cpa.cp_merge_partials(k // 2 * b, rows, heads, d, 2, lo, lm, ll, oo, mo, lo2, finalize=fin and last)
            lo = oo.view(k // 2, b, rows, heads, d)
            lm = mo.view(k // 2, b, heads, rows)
            ll = lo2.view(k // 2, b, heads, rows)
            k //= 2
        torch.cuda.synchronize()
        assert torch.equal(tm, lm[0]) and torch.equal(tl, ll[0]) and torch.equal(to, lo[0]), f"{shape} fin={fin}"


# ------------------------------------------------------------------ decode

def _decode(q, k, v, cp):
    b, hq, d = q.shape
    L, hkv = k.shape[1], k.shape[2]
    desc = cpa.make_desc(b, L, hq, hkv, d, cp, 1.0 / math.sqrt(d), 0)
    ws_bytes = cpa.cp_passq_workspace_bytes(desc)
    ws = torch.empty(ws_bytes // 4, dtype=torch.float32, device="cuda")
    out = torch.empty((b, hq, d), dtype=torch.float32, device="cuda")
    mo = torch.empty((b, hq), dtype=torch.float32, device="cuda")
    lo = torch.empty_like(mo)
    cpa.cp_passq_decode(desc, q, k, v, ws, ws_bytes, out, mo, lo)
    assert cpa.cp_take_device_status() == 0
    return out, mo, lo


DECODE_SMALL = [(2, 4096, 4, 4, 128, 4), (3, 2048, 8, 2, 64, 2), (1, 1024, 2, 1, 256, 1),
                (2, 8192, 16, 16, 512, 8), (1, 3000, 4, 2, 512, 3), (2, 96, 4, 4, 128, 8),
                (1, 12, 2, 2, 64, 4), (2, 8, 4, 2, 128, 8)]  # the last: one key per shard


@pytest.mark.parametrize("case", DECODE_SMALL, ids=[str(c) for c in DECODE_SMALL])
def test_decode_matches_oracle(case):
    b, L, hq, hkv, d, cp = case
    q, k, v = synth.decode_inputs(b, L, hq, hkv, d, seed=L + d)
    out, mo, lo = _decode(q, k, v, cp)
    ref_out, ref_m, ref_l = OA.decode_attention(f64(q), f64(k), f64(v), 1.0 / math.sqrt(d))
    assert_out_close(out.cpu().numpy(), ref_out, f"decode {case}")
    lse = (mo + torch.log(lo)).cpu().numpy()
    assert np.abs(lse - (ref_m + np.log(ref_l))).max() <= LSE_ABS
    assert np.abs(mo.cpu().numpy() - ref_m).max() <= LSE_ABS


def _random_decode_cases(n, seed):
    # Seeded random pass-Q decode problems: the SIMT kernel (groups 1, 2, 4; d up to 512
    # with g * d <= 1024) and the shared-K/V tensor-core kernel (groups 16, 32; d 128-512),
    # shard lengths 1-1499 (ragged key tiles and single keys), cp 1-8, batch 1-3.
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < n:
        cp = int(rng.choice([1, 2, 3, 4, 5, 8]))
        shard = int(rng.integers(1, 1500))
        b = int(rng.integers(1, 4))
        if rng.random() < 0.5:
            d = int(rng.choice([64, 128, 256, 512]))
            g = int(rng.choice([g for g in (1, 2, 4) if g * d <= 1024]))
            hkv = int(rng.integers(1, 5))
        else:
            d = int(rng.choice([128, 256, 512]))
            g = int(rng.choice([16, 32]))
            hkv = int(rng.integers(1, 3))
        cases.append((b, cp * shard, hkv * g, hkv, d, cp))
    return cases


DECODE_RANDOM = _random_decode_cases(24, 20260102)


@pytest.mark.parametrize("case", DECODE_RANDOM, ids=[f"r{i}" for i in range(len(DECODE_RANDOM))])
def test_random_decode_problems_against_the_oracle(case):
    b, L, hq, hkv, d, cp = case
    q, k, v = synth.decode_inputs(b, L, hq, hkv, d, seed=7 * L + d + hq)
    out, mo, lo = _decode(q, k, v, cp)
    ref_out, ref_m, ref_l = OA.decode_attention(f64(q), f64(k), f64(v), 1.0 / math.sqrt(d))
    assert_out_close(out.cpu().numpy(), ref_out, f"decode {case}")
    assert np.abs(mo.cpu().numpy() - ref_m).max() <= LSE_ABS
    lse = (mo + torch.log(lo)).cpu().numpy()
    assert np.abs(lse - (ref_m + np.log(ref_l))).max() <= LSE_ABS


# Query heads sharing one K/V head (MQA / MLA-style): the tensor-core decode kernel.
# Shapes 7 and 8 split each shard into unequal key ranges (5 and 4 tiles), the second
# ending on a ragged tile; the last two hold one key per shard.
MQA_SMALL = [(2, 4096, 16, 1, 512, 4), (1, 2048, 32, 1, 128, 2), (1, 3000, 16, 1, 256, 3),
             (2, 384, 32, 2, 128, 1), (1, 200, 16, 1, 512, 2), (3, 8192, 16, 1, 128, 8),
             (1, 2100, 16, 1, 256, 2), (1, 4200, 32, 1, 128, 4),
             (1, 8, 16, 1, 128, 8), (2, 2, 32, 1, 256, 2)]  # one key per shard


@pytest.mark.parametrize("case", MQA_SMALL, ids=[str(c) for c in MQA_SMALL])
def test_shared_kv_decode_matches_oracle(case):
    b, L, hq, hkv, d, cp = case
    q, k, v = synth.decode_inputs(b, L, hq, hkv, d, seed=L + 3 * d)
    out, mo, lo = _decode(q, k, v, cp)
    ref_out, ref_m, ref_l = OA.decode_attention(f64(q), f64(k), f64(v), 1.0 / math.sqrt(d))
    assert_out_close(out.cpu().numpy(), ref_out, f"mqa decode {case}")
    assert np.abs(mo.cpu().numpy() - ref_m).max() <= LSE_ABS
    lse = (mo + torch.log(lo)).cpu().numpy()
    assert np.abs(lse - (ref_m + np.log(ref_l))).max() <= LSE_ABS


def test_shared_kv_decode_with_k_equal_v():
    # MLA-style: one latent per token serves as key and value (the same buffer twice)
    b, L, hq, d, cp = 2, 4096, 16, 512, 4
    q, k, _ = synth.decode_inputs(b, L, hq, 1, d, seed=77)
    out, _, _ = _decode(q, k, k, cp)
    ref_out, _, _ = OA.decode_attention(f64(q), f64(k), f64(k), 1.0 / math.sqrt(d))
    assert_out_close(out.cpu().numpy(), ref_out, "mla-style")


def test_shared_kv_decode_forced_rescales():
    b, L, hq, d, cp = 1, 8192, 16, 256, 2
    q, k, v = synth.decode_inputs(b, L, hq, 1, d, seed=78)
    ramp = torch.linspace(0.0, 6.0, L, device="cuda").view(1, L, 1, 1)
    k = (k.float() * ramp).to(torch.bfloat16)
    q = (q.float() * 3.0).to(torch.bfloat16)
    out, mo, lo = _decode(q, k, v, cp)
    ref_out, ref_m, ref_l = OA.decode_attention(f64(q), f64(k), f64(v), 1.0 / math.sqrt(d))
    assert_out_close(out.cpu().numpy(), ref_out, "mqa rescale")
    assert np.abs(mo.cpu().numpy() - ref_m).max() <= LSE_ABS


def test_shared_kv_decode_workload_sampled():
    """b8, 16 query heads on one 512-wide K/V head, L131072, cp8, at full size; sampled sequences."""
    b, L, hq, d, cp = 8, 131072, 16, 512, 8
    q, k, v = synth.decode_inputs(b, L, hq, 1, d, seed=20260006)
    out, mo, lo = _decode(q, k, v, cp)
    scale = 1.0 / math.sqrt(d)
    for bi in (0, 5):
        ref_out, ref_m, ref_l = OA.decode_attention(f64(q[bi:bi + 1]), f64(k[bi:bi + 1]), f64(v[bi:bi + 1]), scale)
        assert_out_close(out[bi:bi + 1].cpu().numpy(), ref_out, f"mqa workload seq {bi}")
        assert np.abs(mo[bi].cpu().numpy() - ref_m[0]).max() <= LSE_ABS
    del q, k, v
    torch.cuda.empty_cache()


def test_decode_shards_do_not_change_the_answer():
    b, L, hq, hkv, d = 2, 4096, 4, 4, 128
    q, k, v = synth.decode_inputs(b, L, hq, hkv, d, seed=3)
    base = _decode(q, k, v, 1)[0]
    for cp in (2, 4, 8, 16):
        assert (_decode(q, k, v, cp)[0] - base).abs().max().item() <= 1e-4


def test_decode_workload_sampled_heads():
    """b8, 16 heads, d512, L131072, cp8 at full size; oracle on sampled (sequence, head) pairs."""
    w = synth.WORKLOADS["decode"]
    q, k, v = synth.decode_inputs(w["b"], w["S"], w["h_q"], w["h_kv"], w["d"], seed=w["seed"])
    out, mo, lo = _decode(q, k, v, w["cp"])
    scale = 1.0 / math.sqrt(w["d"])
    for bi, h in [(0, 0), (3, 7), (7, 15), (5, 2)]:
        ref_out, ref_m, ref_l = OA.decode_attention(f64(q[bi:bi + 1, h:h + 1]), f64(k[bi:bi + 1, :, h:h + 1]),
                                                    f64(v[bi:bi + 1, :, h:h + 1]), scale)
        assert_out_close(out[bi, h].cpu().numpy(), ref_out[0, 0], f"decode workload ({bi},{h})")
        assert abs(float(mo[bi, h] + torch.log(lo[bi, h])) - float(ref_m[0, 0] + np.log(ref_l[0, 0]))) <= LSE_ABS
    del q, k, v
    torch.cuda.empty_cache()


def test_decode_rejects_small_workspace():
    q, k, v = synth.decode_inputs(1, 256, 2, 2, 128, seed=1)
    desc = cpa.make_desc(1, 256, 2, 2, 128, 2, 0.1, 0)
    need = cpa.cp_passq_workspace_bytes(desc)
    ws = torch.empty(need // 4, dtype=torch.float32, device="cuda")
    out = torch.empty((1, 2, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(cpa.CpError):
        cpa.cp_passq_decode(desc, q, k, v, ws, need - 4, out)


@pytest.mark.parametrize("case", [(2, 4096, 4, 4, 128, 4), (2, 4096, 16, 1, 256, 4)], ids=["streaming", "shared_kv"])
def test_decode_scale_is_the_one_passed(case):
    # Both decode kernels against the oracle at a scale other than 1/sqrt(d).
    b, L, hq, hkv, d, cp = case
    scale = 0.7 / math.sqrt(d)
    q, k, v = synth.decode_inputs(b, L, hq, hkv, d, seed=55)
    desc = cpa.make_desc(b, L, hq, hkv, d, cp, scale, 0)
    ws_bytes = cpa.cp_passq_workspace_bytes(desc)
    ws = torch.empty(ws_bytes // 4, dtype=torch.float32, device="cuda")
    out = torch.empty((b, hq, d), dtype=torch.float32, device="cuda")
    mo = torch.empty((b, hq), dtype=torch.float32, device="cuda")
    lo = torch.empty_like(mo)
    cpa.cp_passq_decode(desc, q, k, v, ws, ws_bytes, out, mo, lo)
    assert cpa.cp_take_device_status() == 0
    ref_out, ref_m, ref_l = OA.decode_attention(f64(q), f64(k), f64(v), scale)
    assert_out_close(out.cpu().numpy(), ref_out, f"decode scale {case}")
    assert np.abs(mo.cpu().numpy() - ref_m).max() <= LSE_ABS


@pytest.mark.parametrize("shape", [(2, 1, 37, 3, 128), (8, 2, 300, 5, 128), (32, 1, 96, 4, 128),
                                   (64, 3, 17, 2, 128), (13, 1, 16, 1, 128)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("finalize", [False, True])
def test_tma_merge_gives_the_register_merges_bits(shape, finalize):
    """d = 128 and up to 64 parts take the TMA-fed merge; it folds the same parts in the same
    order with the same arithmetic as the register-pipelined merge (merge-kernel knob 0)."""
    n, b, rows, heads, d = shape
    gen = torch.Generator(device="cpu").manual_seed(1000 + n + rows)
    o = torch.randn((n, b, rows, heads, d), generator=gen).cuda()
    m = (torch.randn((n, b, heads, rows), generator=gen) * 20).cuda()
    m[0, 0, 0, :3] = -math.inf  # some identity parts
    l = torch.rand((n, b, heads, rows), generator=gen).add_(0.5).cuda()
    l[0, 0, 0, :3] = 0.0
    order = list(np.random.default_rng(n).permutation(n))
    got = {}
    try:
        for tma in ("1", "0"):
            cpa.cp_set_kernel_choice(cpa.CP_KNOB_MERGE_KERNEL, int(tma))
            got[tma] = _merge(o, m, l, order=order, finalize=finalize)
            assert cpa.cp_take_device_status() == 0
    finally:
        cpa.cp_set_kernel_choice(cpa.CP_KNOB_MERGE_KERNEL, -1)
    for x, y in zip(got["1"], got["0"]):
        assert torch.equal(x, y)
