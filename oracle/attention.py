"""Plain float64 softmax attention (test infrastructure only).

Source: "G5 上下文并行建模设计规格" (G5 CP modelling spec).

* Terms table (名词定义), row "Partial attention": attention over a subset of
  keys carries the online-softmax triple (max / numerator / denominator) so
  that blocks can be merged.  Here the triple of a query row over a key set J
  is, with x_j = scale * <q, k_j>:

      m = max_{j in J} x_j
      l = sum_{j in J} exp(x_j - m)                       (denominator)
      O = sum_{j in J} exp(x_j - m) * v_j                 (numerator, unnormalised)

  and the attention output is O / l.  The page does not print the scale;
  the reading taken is 1/sqrt(head_dim), passed in explicitly.
* Terms table, row "Balanced chunk split", says the split is made "under the
  causal mask"; the reading taken is the inclusive diagonal: query at global
  position i sees keys j <= i.
* Use case section (用例说明), decode paragraph: one query per sequence is
  scored against the KV held by the ranks; the query comes after every cached
  key, so every key is visible.

Layouts (token-major, as in the per-card shape table of the pypto-lib
TP->EP issue page): q ``[b, S, h_q, d]``, k/v ``[b, S, h_kv, d]``; m/l
``[b, h_q, S]``.  Grouped-query heads map as kv_head = h // (h_q // h_kv).
"""

from __future__ import annotations

import numpy as np

NEG_INF = -np.inf


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Decode raw bfloat16 bit patterns (uint16) to float64 exactly.

    A bfloat16 is the upper half of an IEEE float32, so shifting the 16 bits
    into the top of a 32-bit word gives the float32 with the same value.
    """
    bits = np.asarray(bits)
    if bits.dtype != np.uint16:
        raise TypeError("bf16 inputs must be given as uint16 bit patterns")
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def _triple_from_logits(x: np.ndarray, v: np.ndarray):
    """Triple (m, l, O) of logit rows ``x [..., n]`` (-inf = invisible) with values ``v [n, d]``.

    Rows with no visible key give the identity (-inf, 0, 0): the shift used
    for the exponent is 0 there, and exp(-inf) = 0.
    """
    m = x.max(axis=-1)
    shift = np.where(np.isfinite(m), m, 0.0)
    p = np.exp(x - shift[..., None])
    l = p.sum(axis=-1)
    o = p @ v
    return m, l, o


def _check_shapes(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [b, S, h, d]")
    b, s, hq, d = q.shape
    if k.shape != v.shape or k.shape[0] != b or k.shape[3] != d:
        raise ValueError("k and v must be [b, S_kv, h_kv, d] matching q")
    hkv = k.shape[2]
    if hq % hkv != 0:
        raise ValueError("h_q must be a multiple of h_kv")
    return b, s, hq, hkv, d


def full_causal_attention(q, k, v, scale):
    """Full causal softmax attention, the unsplit (cp = 1) computation.

    Returns ``(out, m, l, o)``: out = O / l ``[b, S, h_q, d]``; m, l
    ``[b, h_q, S]``; o the unnormalised numerator ``[b, S, h_q, d]``.
    """
    q, k, v = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
    b, s, hq, hkv, d = _check_shapes(q, k, v)
    g = hq // hkv
    i = np.arange(s)[:, None]
    j = np.arange(k.shape[1])[None, :]
    invisible = j > i
    out = np.empty((b, s, hq, d))
    onum = np.empty((b, s, hq, d))
    m = np.empty((b, hq, s))
    l = np.empty((b, hq, s))
    for bi in range(b):
        for h in range(hq):
            kh = h // g
            x = scale * (q[bi, :, h, :] @ k[bi, :, kh, :].T)
            x[invisible] = NEG_INF
            mh, lh, oh = _triple_from_logits(x, v[bi, :, kh, :])
            m[bi, h] = mh
            l[bi, h] = lh
            onum[bi, :, h] = oh
            out[bi, :, h] = oh / lh[:, None]
    return out, m, l, onum


def causal_attention_rows(q, k, v, scale, b_index, heads, rows):
    """Causal attention for selected query rows, one row at a time.

    For each (head, row) pair in the cross product of ``heads`` x ``rows`` of
    batch ``b_index``: logits against keys 0..row inclusive.  Used where the
    full S x S computation is too large (long sequences): each sampled output
    is computed from its own definition.

    Returns ``(out [len(heads), len(rows), d], m [H, R], l [H, R])``.
    """
    q = np.asarray(q)
    k = np.asarray(k)
    v = np.asarray(v)
    hq, hkv = q.shape[2], k.shape[2]
    g = hq // hkv
    d = q.shape[3]
    out = np.empty((len(heads), len(rows), d))
    m = np.empty((len(heads), len(rows)))
    l = np.empty((len(heads), len(rows)))
    for a, h in enumerate(heads):
        kh = h // g
        for c, i in enumerate(rows):
            kk = np.asarray(k[b_index, : i + 1, kh, :], dtype=np.float64)
            vv = np.asarray(v[b_index, : i + 1, kh, :], dtype=np.float64)
            qq = np.asarray(q[b_index, i, h, :], dtype=np.float64)
            x = scale * (kk @ qq)
            mm, ll, oo = _triple_from_logits(x[None, :], vv)
            m[a, c] = mm[0]
            l[a, c] = ll[0]
            out[a, c] = oo[0] / ll[0]
    return out, m, l


def decode_attention(q, k, v, scale):
    """Pass-Q decode attention: one query per sequence, every key visible.

    q ``[b, h_q, d]``; k/v ``[b, L, h_kv, d]``.  Returns ``(out, m, l)`` with
    out ``[b, h_q, d]`` and m, l ``[b, h_q]``.
    """
    q = np.asarray(q, dtype=np.float64)
    b, hq, d = q.shape
    hkv = k.shape[2]
    g = hq // hkv
    out = np.empty((b, hq, d))
    m = np.empty((b, hq))
    l = np.empty((b, hq))
    for bi in range(b):
        for h in range(hq):
            kh = h // g
            kk = np.asarray(k[bi, :, kh, :], dtype=np.float64)
            vv = np.asarray(v[bi, :, kh, :], dtype=np.float64)
            x = scale * (kk @ q[bi, h])
            mm, ll, oo = _triple_from_logits(x[None, :], vv)
            m[bi, h] = mm[0]
            l[bi, h] = ll[0]
            out[bi, h] = oo[0] / ll[0]
    return out, m, l


def decode_shard_triples(q, k, v, scale, cp):
    """Per-shard partial triples of pass-Q decode.

    Shard ``s`` holds keys ``[s*L/cp, (s+1)*L/cp)`` (contiguous ranges, the
    reading taken of "each rank holds its local KV shard", use case section).
    Returns ``(m [cp, b, h_q], l [cp, b, h_q], O [cp, b, h_q, d])``,
    O unnormalised.
    """
    q = np.asarray(q, dtype=np.float64)
    b, hq, d = q.shape
    L, hkv = k.shape[1], k.shape[2]
    if cp < 1 or L % cp != 0:
        raise ValueError("KV length must be a multiple of cp")
    g = hq // hkv
    n = L // cp
    m = np.empty((cp, b, hq))
    l = np.empty((cp, b, hq))
    o = np.empty((cp, b, hq, d))
    for s in range(cp):
        for bi in range(b):
            for h in range(hq):
                kh = h // g
                kk = np.asarray(k[bi, s * n:(s + 1) * n, kh, :], dtype=np.float64)
                vv = np.asarray(v[bi, s * n:(s + 1) * n, kh, :], dtype=np.float64)
                x = scale * (kk @ q[bi, h])
                mm, ll, oo = _triple_from_logits(x[None, :], vv)
                m[s, bi, h] = mm[0]
                l[s, bi, h] = ll[0]
                o[s, bi, h] = oo[0]
    return m, l, o
