"""Pins of the CPU oracle to facts outside itself (CPU only).

Each pin is a ``check_*`` function taking the implementation under test, so the
same checks run against the oracle (must pass) and against planted mutants of
it (must fail) — see ``test_pins_catch_planted_mistakes``.  Sources:
"G5 上下文并行建模设计规格" (G5 CP modelling spec): Terms table (名词定义),
Algorithm / formulas (算法 / 公式), Use case (用例说明), Acceptance table (验收标准).
"""

import itertools
import json
import math
import os

import mpmath
import numpy as np
import pytest

import oracle
from oracle import attention as OA
from oracle import comm as OC
from oracle import ring as OR

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_integers.json")


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# ---------------------------------------------------------------------------
# attention: arbitrary-precision brute force and closed forms
# ---------------------------------------------------------------------------

def _brute_force_causal(q, k, v, scale):
    """Direct exp without any max shift, 40 significant digits, pure loops."""
    mpmath.mp.dps = 40
    b, S, hq, d = q.shape
    hkv = k.shape[2]
    g = hq // hkv
    out = np.empty(q.shape)
    lse = np.empty((b, hq, S))
    for bi, h, i in itertools.product(range(b), range(hq), range(S)):
        kh = h // g
        den = mpmath.mpf(0)
        num = [mpmath.mpf(0)] * d
        for j in range(i + 1):
            x = mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(q[bi, i, h, c]) * mpmath.mpf(k[bi, j, kh, c])
                                                for c in range(d))
            e = mpmath.exp(x)
            den += e
            for c in range(d):
                num[c] += e * mpmath.mpf(v[bi, j, kh, c])
        for c in range(d):
            out[bi, i, h, c] = float(num[c] / den)
        lse[bi, h, i] = float(mpmath.log(den))
    return out, lse


def check_brute_force(attn):
    for (b, S, hq, hkv, d, seed) in [(1, 7, 2, 1, 3, 1), (2, 12, 4, 2, 4, 2), (1, 9, 3, 3, 2, 3)]:
        q, k, v = _rand((b, S, hq, d), seed), _rand((b, S, hkv, d), seed + 10), _rand((b, S, hkv, d), seed + 20)
        scale = 1.0 / math.sqrt(d)
        out, m, l, _ = attn(q, k, v, scale)
        ref, lse = _brute_force_causal(q, k, v, scale)
        np.testing.assert_allclose(out, ref, rtol=0, atol=1e-13)
        np.testing.assert_allclose(m + np.log(l), lse, rtol=0, atol=1e-13)


def check_closed_forms(attn):
    b, S, hq, hkv, d = 1, 16, 2, 2, 5
    v = _rand((b, S, hkv, d), 5)
    k = _rand((b, S, hkv, d), 6)
    # q = 0: every visible logit is 0, so row i is the mean of v_0..v_i
    out, _, l, _ = attn(np.zeros((b, S, hq, d)), k, v, 0.3)
    prefix_mean = np.cumsum(v, axis=1) / np.arange(1, S + 1)[None, :, None, None]
    np.testing.assert_allclose(out, prefix_mean, rtol=0, atol=1e-14)
    np.testing.assert_array_equal(l[0, 0], np.arange(1, S + 1, dtype=np.float64))
    # constant value rows: the output is that row whatever the weights
    q = _rand((b, S, hq, d), 7)
    vc = np.broadcast_to(np.array([1.5, -2.0, 0.25, 3.0, -0.5]), (b, S, hkv, d)).copy()
    out, _, _, _ = attn(q, k, vc, 0.7)
    np.testing.assert_allclose(out, vc, rtol=0, atol=1e-14)
    # row 0 sees only key 0: exactly v_0, with l = 1
    out, m, l, _ = attn(q, k, v, 0.7)
    np.testing.assert_array_equal(out[0, 0, :, :], v[0, 0, :, :])
    np.testing.assert_array_equal(l[0, :, 0], np.ones(hq))
    np.testing.assert_allclose(m[0, 0, 0], 0.7 * q[0, 0, 0] @ k[0, 0, 0], rtol=1e-15)
    # a spike: key 5 is 50 logits above every other visible key -> out ~ v_5 for rows >= 5
    q1 = np.zeros((1, S, 1, 3)); q1[..., 0] = 1.0
    k1 = np.zeros((1, S, 1, 3)); k1[0, 5, 0, 0] = 50.0
    v1 = _rand((1, S, 1, 3), 8)
    out, _, _, _ = attn(q1, k1, v1, 1.0)
    for i in range(5, S):
        np.testing.assert_allclose(out[0, i, 0], v1[0, 5, 0], rtol=0, atol=S * math.exp(-50) * 10)


def check_gqa_mapping(attn):
    # h_q = 6 over h_kv = 2: heads 0..2 use kv head 0, heads 3..5 kv head 1
    b, S, hq, hkv, d = 1, 10, 6, 2, 4
    q, k, v = _rand((b, S, hq, d), 11), _rand((b, S, hkv, d), 12), _rand((b, S, hkv, d), 13)
    out, _, _, _ = attn(q, k, v, 0.5)
    for h in range(hq):
        kh = h // 3
        single, _, _, _ = attn(q[:, :, h:h + 1], k[:, :, kh:kh + 1], v[:, :, kh:kh + 1], 0.5)
        np.testing.assert_allclose(out[:, :, h:h + 1], single, rtol=0, atol=1e-15)
    # the grouping is observable: a different kv head per group changes the answer
    k2 = k.copy(); k2[:, :, 1] *= 3.0  # not a uniform logit shift, so softmax sees it
    out2, _, _, _ = attn(q, k2, v, 0.5)
    assert np.abs(out2[:, :, :3] - out[:, :, :3]).max() == 0.0
    assert np.abs(out2[:, 1:, 3:] - out[:, 1:, 3:]).max() > 1e-3


def test_brute_force_pins_full_attention():
    check_brute_force(OA.full_causal_attention)


def test_closed_forms_pin_full_attention():
    check_closed_forms(OA.full_causal_attention)


def test_gqa_mapping():
    check_gqa_mapping(OA.full_causal_attention)


def test_sampled_rows_equal_full_rows():
    b, S, hq, hkv, d = 2, 40, 4, 2, 8
    q, k, v = _rand((b, S, hq, d), 21), _rand((b, S, hkv, d), 22), _rand((b, S, hkv, d), 23)
    out, m, l, _ = OA.full_causal_attention(q, k, v, 0.35)
    rows, heads = [0, 1, 17, 39], [0, 3]
    so, sm, sl = OA.causal_attention_rows(q, k, v, 0.35, 1, heads, rows)
    np.testing.assert_allclose(so, out[1][np.ix_(rows, heads)].transpose(1, 0, 2), rtol=0, atol=1e-14)
    np.testing.assert_allclose(sm, m[1][np.ix_(heads, rows)], rtol=0, atol=1e-14)
    np.testing.assert_allclose(sl, l[1][np.ix_(heads, rows)], rtol=1e-14)


def test_bf16_decode_matches_library_conversion():
    import torch
    bits = np.array([0x3F80, 0xC000, 0x7F80, 0xFF80, 0x0001, 0x8000, 0x3EAA, 0x4049, 0x7F7F], dtype=np.uint16)
    got = oracle.bf16_bits_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(got, ref)
    assert got[0] == 1.0 and got[1] == -2.0 and got[4] == 2.0 ** -133
    rnd = np.random.default_rng(0).integers(0, 1 << 16, size=4096, dtype=np.uint16)
    rnd = rnd[(rnd & 0x7F80) != 0x7F80]  # drop NaN patterns (NaN != NaN)
    ref = torch.from_numpy(rnd.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.bf16_bits_to_f64(rnd), ref)


# ---------------------------------------------------------------------------
# decode
# ---------------------------------------------------------------------------

def check_decode(dec):
    # the decode query scores every key: equal to the last row of causal attention
    b, L, hq, hkv, d = 2, 23, 4, 2, 6
    qs, k, v = _rand((b, L, hq, d), 31), _rand((b, L, hkv, d), 32), _rand((b, L, hkv, d), 33)
    full_out, full_m, full_l, _ = OA.full_causal_attention(qs, k, v, 0.4)
    out, m, l = dec(qs[:, L - 1], k, v, 0.4)
    np.testing.assert_allclose(out, full_out[:, L - 1], rtol=0, atol=1e-14)
    np.testing.assert_allclose(m, full_m[:, :, L - 1], rtol=0, atol=1e-15)
    np.testing.assert_allclose(l, full_l[:, :, L - 1], rtol=1e-14)


def test_decode_equals_last_causal_row():
    check_decode(OA.decode_attention)


@pytest.mark.parametrize("cp", [1, 2, 4, 8])
def test_decode_shards_merge_to_unsplit(cp):
    b, L, hq, hkv, d = 2, 64, 4, 4, 8
    q, k, v = _rand((b, hq, d), 41), _rand((b, L, hkv, d), 42), _rand((b, L, hkv, d), 43)
    out, m, l = OA.decode_attention(q, k, v, 0.3)
    sm, sl, so = OA.decode_shard_triples(q, k, v, 0.3, cp)
    parts = [(sm[s], sl[s], so[s]) for s in range(cp)]
    mm, ll, oo = OR.merge_in_order(parts)
    np.testing.assert_array_equal(mm, m)  # max is exact in any grouping
    np.testing.assert_allclose(ll, l, rtol=1e-13)
    np.testing.assert_allclose(oo / ll[..., None], out, rtol=0, atol=1e-13)


# ---------------------------------------------------------------------------
# merge algebra
# ---------------------------------------------------------------------------

def _random_triples(n, rows, d, seed, spread=80.0, identity_frac=0.0):
    rng = np.random.default_rng(seed)
    parts = []
    for _ in range(n):
        m = rng.uniform(-spread, spread, rows)
        l = rng.uniform(1, 64, rows)
        o = l[:, None] * np.clip(rng.standard_normal((rows, d)), -4, 4)
        ident = rng.random(rows) < identity_frac
        m[ident], l[ident], o[ident] = -np.inf, 0.0, 0.0
        parts.append((m, l, o))
    return parts


def check_merge(merge):
    a, b, c = _random_triples(3, 200, 7, 51, spread=20.0)
    ab_c = merge(merge(a, b), c)
    a_bc = merge(a, merge(b, c))
    ba = merge(b, a)
    ab = merge(a, b)
    for x, y in zip(ab_c, a_bc):
        np.testing.assert_allclose(x, y, rtol=1e-13, atol=0)
    for x, y in zip(ab, ba):
        np.testing.assert_allclose(x, y, rtol=1e-13, atol=0)
    np.testing.assert_array_equal(ab_c[0], a_bc[0])
    # identity is an exact no-op on both sides, and identity with identity stays identity
    ident = OR.identity_triple((200,), 7)
    for left in (merge(a, ident), merge(ident, a)):
        for x, y in zip(left, a):
            np.testing.assert_array_equal(x, y)
    im, il, io = merge(ident, ident)
    assert np.all(np.isneginf(im)) and np.all(il == 0) and np.all(io == 0) and not np.isnan(io).any()
    # splitting a softmax's keys anywhere and merging gives the unsplit triple
    rng = np.random.default_rng(52)
    x = rng.standard_normal((30, 50)) * 3
    v = rng.standard_normal((50, 4))
    whole = OA._triple_from_logits(x, v)
    cut = [0, 3, 17, 18, 50]
    pieces = [OA._triple_from_logits(x[:, s:e], v[s:e]) for s, e in zip(cut[:-1], cut[1:])]
    acc = pieces[0]
    for p in pieces[1:]:
        acc = merge(acc, p)
    np.testing.assert_array_equal(acc[0], whole[0])
    np.testing.assert_allclose(acc[1], whole[1], rtol=1e-13)
    np.testing.assert_allclose(acc[2], whole[2], rtol=1e-12, atol=1e-13)


def test_merge_algebra():
    check_merge(OR.merge)


def test_merge_orders_and_tree_agree():
    parts = _random_triples(32, 300, 5, 61, spread=80.0, identity_frac=0.01)
    # never all parts identity in one row
    parts[0][0][:] = np.where(np.isneginf(parts[0][0]), 0.0, parts[0][0])
    parts[0][1][:] = np.where(parts[0][1] == 0, 1.0, parts[0][1])
    ref = OR.merge_in_order(parts)
    rng = np.random.default_rng(62)
    for _ in range(5):
        order = rng.permutation(32)
        got = OR.merge_in_order(parts, order)
        np.testing.assert_array_equal(got[0], ref[0])
        np.testing.assert_allclose(got[1], ref[1], rtol=1e-13)
        np.testing.assert_allclose(got[2], ref[2], rtol=1e-12, atol=1e-300)
    tree = OR.merge_tree(parts)
    np.testing.assert_array_equal(tree[0], ref[0])
    np.testing.assert_allclose(tree[1], ref[1], rtol=1e-13)


def test_finalize():
    m = np.array([0.0, -np.inf, 2.0])
    l = np.array([2.0, 0.0, 4.0])
    o = np.array([[2.0, 4.0], [0.0, 0.0], [4.0, -8.0]])
    out, lse = OR.finalize((m, l, o))
    np.testing.assert_array_equal(out, [[1.0, 2.0], [0.0, 0.0], [1.0, -2.0]])
    np.testing.assert_allclose(lse, [math.log(2.0), -np.inf, 2.0 + math.log(4.0)])


# ---------------------------------------------------------------------------
# plan, ring restatement, CP = 1
# ---------------------------------------------------------------------------

def check_ring_equals_full(ring_attention):
    b, S, hq, hkv, d = 2, 64, 4, 2, 8
    q, k, v = _rand((b, S, hq, d), 71), _rand((b, S, hkv, d), 72), _rand((b, S, hkv, d), 73)
    out, m, l, onum = OA.full_causal_attention(q, k, v, 0.3)
    for cp in (1, 2, 4, 8):
        rm, rl, ro = ring_attention(q, k, v, 0.3, cp)
        np.testing.assert_array_equal(rm, m)
        np.testing.assert_allclose(rl, l, rtol=1e-13)
        np.testing.assert_allclose(ro, onum, rtol=1e-12, atol=1e-13)


def test_ring_restatement_equals_full_attention():
    check_ring_equals_full(OR.ring_attention)


def test_step_triples_cover_keys_exactly_once():
    # over the cp steps of a rank the visible key sets are disjoint and their union is {j <= i}
    S, cp = 48, 4
    src = OR.step_source(cp)
    for r in range(cp):
        rows = OR.rank_rows(S, cp, r)
        seen = np.zeros((rows.size, S), dtype=int)
        for t in range(cp):
            keys = OR.rank_rows(S, cp, src[r][t])
            seen[:, keys] += (keys[None, :] <= rows[:, None])
        np.testing.assert_array_equal(seen, (np.arange(S)[None, :] <= rows[:, None]).astype(int))


def test_step_identity_rows_where_no_key_visible():
    # source rank above r: the head chunk of r sees nothing at that step
    b, S, hq, hkv, d = 1, 32, 2, 1, 4
    q, k, v = _rand((b, S, hq, d), 81), _rand((b, S, hkv, d), 82), _rand((b, S, hkv, d), 83)
    cp, r, t = 4, 1, 3  # s = (1 - 3) mod 4 = 2 > r
    rows, m, l, o = OR.ring_step_triple(q, k, v, 0.5, cp, r, t)
    C = S // (2 * cp)
    assert np.all(np.isneginf(m[:, :, :C])) and np.all(l[:, :, :C] == 0) and np.all(o[:, :, :C] == 0)
    assert np.all(np.isfinite(m[:, :, C:])) and np.all(l[:, :, C:] > 0)


def test_cp1_degeneracy():
    # Terms table row "CP=1 退化": no split, no communication, same result as the unsplit path
    S = 40
    assert OR.chunk_begin(S, 1) == [0, 20, 40]
    assert OR.rank_chunks(1) == [[0, 1]]
    assert OR.step_source(1) == [[0]]
    assert OC.passkv_bytes(S, 1, 4096) == (0, 40 * 4096)
    assert OR.step_pairs_closed_form(S, 1) == [[S * (S + 1) // 2]]
    b, hq, hkv, d = 1, 2, 2, 4
    q, k, v = _rand((b, S, hq, d), 91), _rand((b, S, hkv, d), 92), _rand((b, S, hkv, d), 93)
    _, m, l, onum = OA.full_causal_attention(q, k, v, 0.5)
    rm, rl, ro = OR.ring_attention(q, k, v, 0.5, 1)
    np.testing.assert_array_equal(rm, m)
    np.testing.assert_allclose(rl, l, rtol=1e-14)
    np.testing.assert_allclose(ro, onum, rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("S,cp", [(8, 1), (8, 2), (16, 4), (24, 3), (64, 8), (96, 6), (128, 16)])
def test_pair_counts_enumeration_equals_closed_form(S, cp):
    enum = OR.step_pairs_enumerated(S, cp)
    closed = OR.step_pairs_closed_form(S, cp)
    assert enum == closed
    totals = [sum(row) for row in enum]
    assert len(set(totals)) == 1  # equal work per rank
    assert sum(totals) == S * (S + 1) // 2  # every causal pair exactly once
    C = S // (2 * cp)
    # eq. g5cp-step-flops: off step 0, a step is exactly 1/cp^2 of the S^2/2 full-square count
    for r in range(cp):
        for t in range(1, cp):
            assert enum[r][t] * cp * cp * 2 == S * S
    assert totals[0] == C * (2 * cp * C + 1)


@pytest.mark.parametrize("S,cp", [(8, 1), (16, 2), (24, 3), (64, 4), (96, 8)])
def test_sequential_layout_pairs_and_totals(S, cp):
    enum = OR.step_pairs_enumerated(S, cp, "sequential")
    assert enum == OR.step_pairs_sequential_closed_form(S, cp)
    assert [sum(row) for row in enum] == OR.sequential_split_pairs(S, cp)
    assert sum(sum(row) for row in enum) == S * (S + 1) // 2
    assert OR.rank_chunks(cp, "sequential") == [[2 * r, 2 * r + 1] for r in range(cp)]


def test_sequential_layout_ring_equals_full_attention():
    b, S, hq, hkv, d = 1, 48, 4, 2, 8
    q, k, v = _rand((b, S, hq, d), 171), _rand((b, S, hkv, d), 172), _rand((b, S, hkv, d), 173)
    _, m, l, onum = OA.full_causal_attention(q, k, v, 0.3)
    for cp in (1, 2, 3, 4):
        rm, rl, ro = OR.ring_attention(q, k, v, 0.3, cp, layout="sequential")
        np.testing.assert_array_equal(rm, m)
        np.testing.assert_allclose(rl, l, rtol=1e-13)
        np.testing.assert_allclose(ro, onum, rtol=1e-12, atol=1e-13)


def test_sequential_split_is_unbalanced():
    # the comparison the Terms table draws: a plain split loads the last rank far more
    S, cp = 4096, 8
    seq = OR.sequential_split_pairs(S, cp)
    assert sum(seq) == S * (S + 1) // 2
    assert seq[-1] / seq[0] > 2 * cp - 2  # ratio ~ 2cp-1, far from balanced
    assert len(set(sum(r) for r in OR.step_pairs_closed_form(S, cp))) == 1


def test_plan_rejects_bad_arguments():
    for S, cp in [(10, 0), (10, -1), (10, 3), (0, 1), (7, 1)]:
        with pytest.raises(ValueError):
            OR.chunk_begin(S, cp)


# ---------------------------------------------------------------------------
# communication volumes
# ---------------------------------------------------------------------------

def _simulate_ring_bytes(S, cp, c_kv):
    """Move real per-token KV byte buffers round a ring of cp ranks; count bytes sent."""
    n = S // cp
    held = [np.zeros(n * c_kv, dtype=np.uint8) + r for r in range(cp)]
    sent_per_step = []
    for _ in range(cp - 1):
        sent = sum(h.nbytes for h in held)  # every rank sends the block it holds
        held = [held[(r - 1) % cp] for r in range(cp)]
        sent_per_step.append(sent // cp)  # per rank
    # after cp-1 rotations, rank r has seen every block exactly once (block r+1 last)
    assert [int(h[0]) for h in held] == [(r + 1) % cp for r in range(cp)]
    return sum(sent_per_step), (sent_per_step[0] if sent_per_step else n * c_kv)


@pytest.mark.parametrize("S,cp,c_kv", [(64, 1, 8), (64, 2, 8), (96, 4, 3), (320, 8, 20), (512, 16, 16)])
def test_passkv_bytes_equal_simulated_ring(S, cp, c_kv):
    assert OC.passkv_bytes(S, cp, c_kv) == _simulate_ring_bytes(S, cp, c_kv)


def test_passq_reduce_is_the_size_of_the_triples():
    # the reduce message of one rank is its partial output plus a max and a denominator per head
    for b, n_h, d_head, itemsize in [(8, 16, 512, 2), (8, 16, 512, 4), (3, 5, 7, 4)]:
        dtype = {2: np.float16, 4: np.float32}[itemsize]
        o = np.zeros((b, n_h, d_head), dtype)
        m = np.zeros((b, n_h), dtype)
        l = np.zeros((b, n_h), dtype)
        q = np.zeros((b, n_h * d_head), dtype)
        d = n_h * d_head  # hidden size
        dispatch, reduce_ = OC.passq_bytes(b, d, n_h, itemsize)
        assert dispatch == q.nbytes
        assert reduce_ == o.nbytes + m.nbytes + l.nbytes


def _simulate_kv_footprint(b, S, cp, c_kv, layers_local, layout="balanced"):
    """Allocate the KV cache every rank holds under the chunk plan and count its bytes.

    Rank r keeps, for each of its L_local layers and each of the b sequences, c_kv
    bytes (K and V together) for every token of its two chunks.  Returns the bytes
    held by each rank, counted from real arrays."""
    C = S // (2 * cp)
    held = []
    for r in range(cp):
        tokens = sum(C for _ in OR.rank_chunks(cp, layout)[r])
        caches = [np.zeros((b, tokens, c_kv), dtype=np.uint8) for _ in range(layers_local)]
        held.append(sum(a.nbytes for a in caches))
    return held


FOOTPRINT_CASES = [(1, 64, 1, 8, 1), (2, 96, 4, 3, 5), (3, 128, 8, 20, 2), (1, 256, 16, 16, 3), (4, 48, 2, 7, 4)]


def check_kv_footprint(fn):
    for b, S, cp, c_kv, L in FOOTPRINT_CASES:
        held = _simulate_kv_footprint(b, S, cp, c_kv, L)
        assert len(set(held)) == 1  # the balanced split gives every rank the same KV
        assert fn(b, S, c_kv, L, cp) == held[0], (b, S, cp, c_kv, L)
        seq = _simulate_kv_footprint(b, S, cp, c_kv, L, layout="sequential")
        assert seq == held  # the layout moves tokens between chunks, never the per-rank count


def test_kv_footprint_equals_allocated_cache():
    # memory paragraph of the Algorithm / formulas section: b * S * c_kv * L_local / cp per rank
    check_kv_footprint(OC.kv_bytes_per_rank)


@pytest.mark.parametrize("kind", ["drop_b", "drop_layers", "drop_cp", "c_kv_per_k_only"])
def test_footprint_pin_catches_planted_mistakes(kind):
    def mutant(b, S, c_kv, L, cp):
        if kind == "drop_b":
            return S * c_kv * L // cp
        if kind == "drop_layers":
            return b * S * c_kv // cp
        if kind == "drop_cp":
            return b * S * c_kv * L
        return b * S * (c_kv // 2) * L // cp
    assert _fails(check_kv_footprint, mutant), f"planted footprint mistake {kind!r} slipped through"


def _per_token_kv_bytes(h_kv, d_head, itemsize):
    """c_kv counted from the K and V rows one token appends to the cache of one layer."""
    dtype = {2: np.float16, 4: np.float32}[itemsize]
    k_row = np.zeros((h_kv, d_head), dtype)
    v_row = np.zeros((h_kv, d_head), dtype)
    return k_row.nbytes + v_row.nbytes


def test_c_kv_of_grouped_heads_equals_one_token_of_cache():
    for h_kv, d_head, s in [(4, 64, 2), (8, 128, 2), (1, 512, 2), (8, 128, 4), (3, 5, 2)]:
        assert OC.c_kv_gqa(h_kv, d_head, s) == _per_token_kv_bytes(h_kv, d_head, s)


def test_workload_byte_counts_written_out():
    # c_kv and eq. g5cp-passkv-bytes at the three prefill workloads, multiplied out by hand:
    #   tiny  h_kv 4, d 64:   c_kv = 2*4*64*2  = 1024 B; M = 1 * 512 * 1024      = 524,288
    #   gqa   h_kv 8, d 128:  c_kv = 2*8*128*2 = 4096 B; M = 7 * 4096 * 4096     = 117,440,512
    #   long  h_kv 8, d 128:  c_kv = 4096 B;            M = 15 * 8192 * 4096     = 503,316,480
    # and the 1M use case with the MLA c_kv of Appendix B: M = 7 * 131072 * 320 = 293,601,280.
    assert OC.c_kv_gqa(4, 64, 2) == 1024
    assert OC.c_kv_gqa(8, 128, 2) == 4096
    assert OC.passkv_bytes(1024, 2, 1024) == (524_288, 524_288)
    assert OC.passkv_bytes(32768, 8, 4096) == (117_440_512, 16_777_216)
    assert OC.passkv_bytes(131072, 16, 4096) == (503_316_480, 33_554_432)
    assert OC.passkv_bytes(1 << 20, 8, 320) == (293_601_280, 41_943_040)
    # pass-Q at the decode workload (b 8, n_h 16, d = 16 * 512 = 8192):
    #   dispatch 8*8192*2 = 131,072; reduce 8*(8192+32)*2 = 131,584 (s = 2), 263,168 (s = 4)
    assert OC.passq_bytes(8, 8192, 16, 2) == (131_072, 131_584)
    assert OC.passq_bytes(8, 8192, 16, 4) == (262_144, 263_168)


def test_page_integers():
    g = json.load(open(GOLDEN))
    uc = g["use_case_prefill"]
    S, cp = uc["S"], uc["cp"]
    begins = OR.chunk_begin(S, cp)
    tokens = [begins[a + 1] - begins[a] + begins[b + 1] - begins[b] for a, b in OR.rank_chunks(cp)]
    assert tokens == [uc["tokens_per_rank"]] * cp
    src = OR.step_source(cp)
    assert len(src[0]) == uc["ring_step_compute_ops"]
    assert sum(1 for t in range(cp) if src[0][t] != 0) == uc["p2p_ops"]
    c16 = g["use_case_cp16"]
    before = OC.kv_bytes_per_rank(1, S, 320, 61, c16["cp_before"])
    after = OC.kv_bytes_per_rank(1, S, 320, 61, c16["cp_after"])
    assert after / before == c16["kv_ratio_after_over_before"]
    dec = g["use_case_decode"]
    assert dec["L"] // dec["cp"] == dec["shard_len"]
    for cpv in g["dag_structure"]["cp_values"]:
        s = OR.step_source(cpv)
        assert all(len(row) == cpv for row in s)
        # each rank receives cp-1 foreign blocks, every one exactly once
        assert all(sorted(row) == list(range(cpv)) for row in s)
        assert all(sum(1 for x in row if x != r) == cpv - 1 for r, row in enumerate(s))
    c_kv = g["mla_c_kv"]["c_kv"]
    for cpv in (1, 2, 8, 64, 1024):
        total, per = OC.passkv_bytes(S, cpv, c_kv)
        assert total <= S * c_kv  # the asymptotic upper bound M ~ S*c_kv
        assert total + per == S * c_kv
    assert OC.passkv_bytes(S, 1024, c_kv)[0] / (S * c_kv) > 0.999


def test_u64_bounds():
    assert OC.fits_u64(OC.U64_MAX) and not OC.fits_u64(OC.U64_MAX + 1)
    total, _ = OC.passkv_bytes(1 << 40, 2, 1 << 30)
    assert not OC.fits_u64(total)


# ---------------------------------------------------------------------------
# planted mistakes: each mutant of the oracle must fail at least one pin
# ---------------------------------------------------------------------------

def _mutant_full_attention(kind):
    def attn(q, k, v, scale):
        q, k, v = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
        b, S, hq, d = q.shape
        hkv = k.shape[2]
        g = hq // hkv
        i = np.arange(S)[:, None]
        j = np.arange(S)[None, :]
        invisible = (j >= i) if kind == "strict_diagonal" else (j > i)
        out = np.empty(q.shape); onum = np.empty(q.shape)
        m = np.empty((b, hq, S)); l = np.empty((b, hq, S))
        for bi in range(b):
            for h in range(hq):
                kh = (h % hkv) if kind == "gqa_modulo" else h // g
                kk = k[bi, :, kh, :]
                x = scale * (q[bi, :, h, :] @ kk.T)
                if kind == "transposed":
                    x = x.T.copy()
                x[invisible] = -np.inf
                if kind == "no_scale":
                    x = x / scale
                mm, ll, oo = OA._triple_from_logits(x, v[bi, :, kh, :])
                if kind == "normalise_by_count":
                    ll = (~invisible).sum(1).astype(float)
                m[bi, h], l[bi, h], onum[bi, :, h] = mm, ll, oo
                with np.errstate(all="ignore"):
                    out[bi, :, h] = oo / ll[:, None]
        return out, m, l, onum
    return attn


def _mutant_merge(kind):
    def merge(a, b):
        ma, la, oa = a
        mb, lb, ob = b
        m = np.maximum(ma, mb)
        shift = np.where(np.isfinite(m), m, 0.0)
        wa = np.exp(ma - shift)
        wb = np.exp(shift - mb) if kind == "sign" else np.exp(mb - shift)
        if kind == "drop_b_in_l":
            return m, wa * la + lb, wa[..., None] * oa + wb[..., None] * ob
        if kind == "no_guard":
            wa = np.exp(ma - m); wb = np.exp(mb - m)
        return m, wa * la + wb * lb, wa[..., None] * oa + wb[..., None] * ob
    return merge


def _fails(fn, *args):
    try:
        with np.errstate(all="ignore"):
            fn(*args)
    except (AssertionError, ValueError, FloatingPointError, IndexError):
        return True
    return False


@pytest.mark.parametrize("kind", ["strict_diagonal", "gqa_modulo", "transposed", "no_scale", "normalise_by_count"])
def test_pins_catch_planted_attention_mistakes(kind):
    mut = _mutant_full_attention(kind)
    assert OA.full_causal_attention  # the real oracle passes the same checks (tests above)
    caught = (_fails(check_closed_forms, mut) or _fails(check_gqa_mapping, mut)
              or _fails(check_brute_force, mut))
    assert caught, f"planted mistake {kind!r} slipped through every pin"


@pytest.mark.parametrize("kind", ["sign", "drop_b_in_l", "no_guard"])
def test_pins_catch_planted_merge_mistakes(kind):
    assert _fails(check_merge, _mutant_merge(kind)), f"planted merge mistake {kind!r} slipped through"


def test_halving_tree_equals_fold_and_pairwise_tree():
    parts = _random_triples(16, 120, 6, 181, spread=40.0, identity_frac=0.02)
    parts[0][0][:] = np.where(np.isneginf(parts[0][0]), 0.0, parts[0][0])
    parts[0][1][:] = np.where(parts[0][1] == 0, 1.0, parts[0][1])
    fold = OR.merge_in_order(parts)
    for tree in (OR.merge_tree_halves(parts), OR.merge_tree(parts)):
        np.testing.assert_array_equal(tree[0], fold[0])
        np.testing.assert_allclose(tree[1], fold[1], rtol=1e-13)
        np.testing.assert_allclose(tree[2], fold[2], rtol=1e-12, atol=1e-300)
    with pytest.raises(ValueError):
        OR.merge_tree_halves(parts[:3])
