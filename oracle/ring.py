"""Balanced ring plan, per-step partial triples and the LSE merge (test infrastructure only).

Source: "G5 上下文并行建模设计规格" (G5 CP modelling spec).

* Terms table (名词定义), row "Balanced chunk split": the sequence is cut into
  2*cp chunks and each rank holds a head/tail pair, so every rank does the same
  work in every step.  Reading taken: rank r holds chunk r (head) and chunk
  2*cp-1-r (tail); its local rows are the head chunk followed by the tail chunk.
* Terms table, rows "Pass-KV" and "Ring step": K/V blocks travel round the
  ring for cp-1 steps; in each step a rank computes partial attention on the
  block it holds.  Reading taken for the (unstated) direction: at step t rank r
  holds the block that started on rank s = (r - t) mod cp, so step 0 is the
  local block.
* Algorithm / formulas section (算法 / 公式), eq. g5cp-step-flops: per rank
  per step the balanced split gives F_attn / cp^2.  Here the work is counted
  exactly as visible (query, key) pairs.
* Terms table, row "Partial attention": the triple (max / numerator /
  denominator) merges associatively and in any order.
* Terms table, row "CP=1 退化": with cp = 1 nothing is split or sent, and the
  result equals the path without CP.
"""

from __future__ import annotations

import numpy as np

from .attention import _check_shapes, _triple_from_logits

NEG_INF = -np.inf


# ---------------------------------------------------------------------------
# plan
# ---------------------------------------------------------------------------

def _check_plan_args(S, cp):
    if not isinstance(cp, (int, np.integer)) or cp < 1:
        raise ValueError("cp must be an explicit positive integer")
    if S < 1 or S % (2 * cp) != 0:
        raise ValueError("S must be a positive multiple of 2*cp")


def chunk_begin(S, cp):
    """Start token of each of the 2*cp chunks, plus S at the end (length 2cp+1)."""
    _check_plan_args(S, cp)
    C = S // (2 * cp)
    return [k * C for k in range(2 * cp + 1)]


LAYOUTS = ("balanced", "sequential")


def rank_chunks(cp, layout="balanced"):
    """The two chunks of every rank.

    balanced:   [r, 2cp-1-r]  (head/tail pairing, Terms table "Balanced chunk split")
    sequential: [2r, 2r+1]    (the plain split the Terms table contrasts it with:
                               rank r holds tokens [r*S/cp, (r+1)*S/cp))
    """
    if layout == "balanced":
        return [[r, 2 * cp - 1 - r] for r in range(cp)]
    if layout == "sequential":
        return [[2 * r, 2 * r + 1] for r in range(cp)]
    raise ValueError(f"unknown layout {layout!r}")


def step_source(cp):
    """step_src[r][t]: the rank whose K/V block rank r holds at ring step t."""
    return [[(r - t) % cp for t in range(cp)] for r in range(cp)]


def rank_rows(S, cp, r, layout="balanced"):
    """Global row indices owned by rank r: its first chunk then its second chunk."""
    C = S // (2 * cp)
    first, second = rank_chunks(cp, layout)[r]
    return np.concatenate([np.arange(first * C, (first + 1) * C),
                           np.arange(second * C, (second + 1) * C)])


def step_pairs_enumerated(S, cp, layout="balanced"):
    """Visible (query, key) pairs per (rank, step) for one head, counted one by one."""
    _check_plan_args(S, cp)
    src = step_source(cp)
    out = [[0] * cp for _ in range(cp)]
    for r in range(cp):
        rows = rank_rows(S, cp, r, layout)
        for t in range(cp):
            keys = rank_rows(S, cp, src[r][t], layout)
            out[r][t] = int((keys[None, :] <= rows[:, None]).sum())
    return out


def step_pairs_closed_form(S, cp):
    """Visible pairs per (rank, step): 2*C^2, plus C at step 0 (the two causal diagonals).

    Derivation: for source s < r both query chunks see all of chunk s and none
    of the tail of s; for s > r only the tail query chunk sees both chunks of s;
    at t = 0 the two diagonal blocks give C(C+1)/2 each and the (tail, head)
    block C^2.
    """
    _check_plan_args(S, cp)
    C = S // (2 * cp)
    return [[2 * C * C + (C if t == 0 else 0) for t in range(cp)] for _ in range(cp)]


def step_pairs_sequential_closed_form(S, cp):
    """Visible pairs per (rank, step) under the sequential layout (n = S/cp rows per rank).

    Source s < r: the whole n x n block is visible; s = r (step 0): the causal
    triangle n(n+1)/2; s > r: nothing.
    """
    _check_plan_args(S, cp)
    n = S // cp
    src = step_source(cp)
    return [[(n * n if src[r][t] < r else (n * (n + 1) // 2 if src[r][t] == r else 0)) for t in range(cp)]
            for r in range(cp)]


def sequential_split_pairs(S, cp):
    """Visible pairs per rank under a plain sequential split (chunk S/cp per rank), for comparison."""
    if cp < 1 or S % cp != 0:
        raise ValueError("S must be a multiple of cp")
    n = S // cp
    return [n * r * n + n * (n + 1) // 2 for r in range(cp)]


# ---------------------------------------------------------------------------
# merge
# ---------------------------------------------------------------------------

def identity_triple(shape_rows, d):
    """The merge identity (-inf, 0, 0) for ``shape_rows`` rows of width d."""
    return (np.full(shape_rows, NEG_INF), np.zeros(shape_rows), np.zeros(tuple(shape_rows) + (d,)))


def merge(a, b):
    """LSE combine of two triples (m, l, O); O carries a trailing d axis.

    m = max(m_a, m_b); each side is weighted by exp(m_side - m); a side whose
    max is -inf weighs 0 (the shift is taken as 0 when both are -inf, so the
    identity merges to the identity and never to NaN).
    """
    ma, la, oa = a
    mb, lb, ob = b
    m = np.maximum(ma, mb)
    shift = np.where(np.isfinite(m), m, 0.0)
    wa = np.exp(ma - shift)
    wb = np.exp(mb - shift)
    return m, wa * la + wb * lb, wa[..., None] * oa + wb[..., None] * ob


def merge_in_order(parts, order=None):
    """Fold a list of triples left to right in ``order`` (default: index order)."""
    if order is None:
        order = range(len(parts))
    order = list(order)
    acc = parts[order[0]]
    for p in order[1:]:
        acc = merge(acc, parts[p])
    return acc


def merge_tree(parts):
    """Balanced binary-tree merge over index order (pairs, then pairs of pairs, ...)."""
    level = list(parts)
    while len(level) > 1:
        nxt = [merge(level[i], level[i + 1]) for i in range(0, len(level) - 1, 2)]
        if len(level) % 2:
            nxt.append(level[-1])
        level = nxt
    return level[0]


def merge_tree_halves(parts):
    """Log-depth tree where each level merges part i with part i + n/2 (n a power of two)."""
    level = list(parts)
    if len(level) & (len(level) - 1):
        raise ValueError("the halving tree needs a power-of-two number of parts")
    while len(level) > 1:
        half = len(level) // 2
        level = [merge(level[i], level[i + half]) for i in range(half)]
    return level[0]


def finalize(triple):
    """Normalised output O / l (0 where l = 0) and lse = m + ln l."""
    m, l, o = triple
    safe = np.where(l > 0, l, 1.0)
    out = np.where((l > 0)[..., None], o / safe[..., None], 0.0)
    with np.errstate(divide="ignore"):
        lse = m + np.log(l)
    return out, lse


# ---------------------------------------------------------------------------
# ring steps
# ---------------------------------------------------------------------------

def ring_step_triple(q, k, v, scale, cp, r, t, layout="balanced"):
    """Partial triple of virtual rank r at ring step t, over its local rows.

    Rows: rank r's head chunk then tail chunk (global positions in
    ``rank_rows``).  Keys: the two chunks of source rank s = (r - t) mod cp.
    Query i sees key j when j <= i (global positions).  Rows with no visible
    key are the identity.

    Returns ``(rows, m [b, h_q, 2C], l [b, h_q, 2C], O [b, h_q, 2C, d])``.
    """
    q, k, v = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
    b, S, hq, hkv, d = _check_shapes(q, k, v)
    _check_plan_args(S, cp)
    g = hq // hkv
    s = (r - t) % cp
    rows = rank_rows(S, cp, r, layout)
    keys = rank_rows(S, cp, s, layout)
    invisible = keys[None, :] > rows[:, None]
    n = rows.size
    m = np.empty((b, hq, n))
    l = np.empty((b, hq, n))
    o = np.empty((b, hq, n, d))
    for bi in range(b):
        for h in range(hq):
            kh = h // g
            x = scale * (q[bi, rows, h, :] @ k[bi, keys, kh, :].T)
            x[invisible] = NEG_INF
            mm, ll, oo = _triple_from_logits(x, v[bi, keys, kh, :])
            m[bi, h], l[bi, h], o[bi, h] = mm, ll, oo
    return rows, m, l, o


def ring_attention(q, k, v, scale, cp, steps=None, layout="balanced"):
    """Ring restatement: every rank merges its per-step triples in step order.

    ``steps`` (default all of 0..cp-1) selects which ring steps are merged.
    Returns the merged triple in global row layout:
    ``(m [b, h_q, S], l [b, h_q, S], O [b, S, h_q, d])``; rows that saw no key
    in the selected steps hold the identity.
    """
    q = np.asarray(q, dtype=np.float64)
    b, S, hq, d = q.shape
    if steps is None:
        steps = range(cp)
    m = np.full((b, hq, S), NEG_INF)
    l = np.zeros((b, hq, S))
    o = np.zeros((b, S, hq, d))
    for r in range(cp):
        rows = rank_rows(S, cp, r, layout)
        acc = (m[:, :, rows], l[:, :, rows], np.moveaxis(o[:, rows], 1, 2))
        for t in steps:
            _, sm, sl, so = ring_step_triple(q, k, v, scale, cp, r, t, layout)
            acc = merge(acc, (sm, sl, so))
        m[:, :, rows] = acc[0]
        l[:, :, rows] = acc[1]
        o[:, rows] = np.moveaxis(acc[2], 2, 1)
    return m, l, o
