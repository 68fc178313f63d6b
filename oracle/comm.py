"""Closed-form CP communication volumes as exact integers (test infrastructure only).

Source: "G5 上下文并行建模设计规格" (G5 CP modelling spec),
Algorithm / formulas section (算法 / 公式):

* eq. g5cp-passkv-bytes: per rank and layer the pass-KV ring moves
  M_passkv = (cp - 1) * (S / cp) * c_kv bytes; each ring step moves
  (S / cp) * c_kv.  c_kv (Terms table) is the K+V bytes per token per layer,
  already counting both K and V.
* Pass-Q paragraph: the query dispatch is b * d * s_dtype bytes and the reduce
  message b * (d + 2 * n_h) * s_dtype bytes (d = the partial output vector,
  2 * n_h = the per-head max and denominator), both independent of S.
* Memory paragraph: per-rank KV footprint b * S * c_kv * L_local / cp.

Readings taken: S must divide by cp (no padding: the design-rationale
section forbids silent fallbacks); the pass-KV formula carries no batch factor,
exactly as printed.  Python integers never overflow; ``U64_MAX`` marks what
fits the library's uint64 results.
"""

from __future__ import annotations

U64_MAX = (1 << 64) - 1


def passkv_bytes(S, cp, c_kv):
    """(total over the cp-1 rotations, per ring step) in bytes."""
    if cp < 1 or S < 0 or c_kv < 0 or S % cp != 0:
        raise ValueError("need cp >= 1, S >= 0, c_kv >= 0 and S divisible by cp")
    per_step = (S // cp) * c_kv
    return (cp - 1) * per_step, per_step


def passq_bytes(b, d, n_h, s_dtype):
    """(dispatch, reduce) message sizes of pass-Q in bytes."""
    if min(b, d, n_h, s_dtype) < 0:
        raise ValueError("sizes must be non-negative")
    return b * d * s_dtype, b * (d + 2 * n_h) * s_dtype


def kv_bytes_per_rank(b, S, c_kv, layers_local, cp):
    """Per-rank KV cache footprint b * S * c_kv * L_local / cp (requires exact division)."""
    num = b * S * c_kv * layers_local
    if cp < 1 or num % cp != 0:
        raise ValueError("footprint must divide evenly by cp")
    return num // cp


def c_kv_gqa(h_kv, d_head, s_kv):
    """K+V bytes per token for grouped-query attention: 2 * h_kv * d_head * s_kv."""
    return 2 * h_kv * d_head * s_kv


def fits_u64(*values):
    return all(0 <= x <= U64_MAX for x in values)
