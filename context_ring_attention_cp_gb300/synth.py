"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke run.

This module draws random numbers and nothing else: it holds none of the
attention, merge or planning arithmetic.  Both the CUDA path and the CPU oracle
read the same bf16 bits (``bf16_bits`` hands them to the oracle as uint16).

Workloads (head shapes from the pypto-lib TP->EP issue page — 16 heads of
width 512 per card — and from the xserv pipeline-parallel page — Qwen3-8B's
32 query / 8 kv heads of width 128):

=====  ==========================================================  ==========
name   shape                                                       values
=====  ==========================================================  ==========
tiny   prefill b1, 4 heads (MHA), d64, S1024, cp2                   N(0,1)
gqa    prefill b1, 32 q / 8 kv heads, d128, S32768, cp8             N(0,1)*0.5
decode pass-Q b8, 16 heads (MHA), d512, L131072, cp8                N(0,1)
long   prefill b1, 32 q / 8 kv heads, d128, S131072, cp16           N(0,1)*0.5
merge  64 heads x 128 x 4096 rows, 32 partial triples               see below
=====  ==========================================================  ==========

Seeds are 20260000 + the workload's index (1..5).
"""

from __future__ import annotations

import math

import numpy as np
import torch

WORKLOADS = {
    "tiny": dict(kind="prefill", b=1, S=1024, h_q=4, h_kv=4, d=64, cp=2, std=1.0, seed=20260001),
    "gqa": dict(kind="prefill", b=1, S=32768, h_q=32, h_kv=8, d=128, cp=8, std=0.5, seed=20260002),
    "decode": dict(kind="decode", b=8, S=131072, h_q=16, h_kv=16, d=512, cp=8, std=1.0, seed=20260003),
    "long": dict(kind="prefill", b=1, S=131072, h_q=32, h_kv=8, d=128, cp=16, std=0.5, seed=20260004),
    "merge": dict(kind="merge", heads=64, d=128, rows=4096, parts=32, spread=80.0, seed=20260005),
    # multi-head (one query head per K/V head) at the GQA workload's size
    "mha": dict(kind="prefill", b=1, S=32768, h_q=32, h_kv=32, d=128, cp=8, std=0.5, seed=20260006),
    # head dimension 64 at scale: multi-head, 16 heads, the GQA workload's length and cp
    "mha64": dict(kind="prefill", b=1, S=32768, h_q=16, h_kv=16, d=64, cp=8, std=0.5, seed=20260007),
}

_CHUNK = 1 << 26  # elements drawn per randn call (bounds the fp32 staging buffer)


def _randn_bf16(shape, std, gen, device):
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        x = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        flat[s:e].copy_(x)  # round to nearest even
    return out


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def prefill_inputs(b, S, h_q, h_kv, d, std=1.0, seed=0, device="cuda"):
    """Q [b,S,h_q,d], K, V [b,S,h_kv,d] in bf16, values N(0, std^2) rounded to bf16."""
    g = _gen(seed, device)
    q = _randn_bf16((b, S, h_q, d), std, g, device)
    k = _randn_bf16((b, S, h_kv, d), std, g, device)
    v = _randn_bf16((b, S, h_kv, d), std, g, device)
    return q, k, v


def decode_inputs(b, L, h_q, h_kv, d, std=1.0, seed=0, device="cuda"):
    """q [b,h_q,d], K, V [b,L,h_kv,d] in bf16."""
    g = _gen(seed, device)
    q = _randn_bf16((b, h_q, d), std, g, device)
    k = _randn_bf16((b, L, h_kv, d), std, g, device)
    v = _randn_bf16((b, L, h_kv, d), std, g, device)
    return q, k, v


def merge_parts(parts, heads, rows, d, spread=80.0, seed=0, device="cuda", identity_frac=0.01):
    """Synthetic partial triples in the merge layout (batch 1).

    Per (part, head, row): m ~ U(-spread, spread); l ~ U(1, 64) (a real block of
    n keys has 1 <= l <= n); O = l * u with u ~ N(0,1)^d clipped to |u| <= 4 (so
    O / l lies in the range of value vectors).  About ``identity_frac`` of the
    entries are the identity (-inf, 0, 0), never all parts of one (head, row).
    Returns o [parts, 1, rows, heads, d], m and l [parts, 1, heads, rows], fp32.
    """
    g = _gen(seed, device)
    m = (torch.rand((parts, 1, heads, rows), generator=g, device=device) * 2 - 1) * spread
    l = 1 + torch.rand((parts, 1, heads, rows), generator=g, device=device) * 63
    u = torch.randn((parts, 1, rows, heads, d), generator=g, device=device).clamp_(-4, 4)
    o = u * l.permute(0, 1, 3, 2).unsqueeze(-1)
    ident = torch.rand((parts, 1, heads, rows), generator=g, device=device) < identity_frac
    ident[0] &= ~ident.all(dim=0)[0]  # keep part 0 where every part drew the identity
    m[ident] = -math.inf
    l[ident] = 0.0
    o.masked_fill_(ident.permute(0, 1, 3, 2).unsqueeze(-1), 0.0)
    return o.contiguous(), m.contiguous(), l.contiguous()


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns as a numpy uint16 array (host copy)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def sample_rows(S, cp, n_random, seed):
    """Rows for sampled checks: first/last row of every one of the 2cp chunks,
    rows 0 and S-1, plus ``n_random`` seeded random rows; sorted, unique."""
    C = S // (2 * cp)
    rows = {0, S - 1}
    for c in range(2 * cp):
        rows.add(c * C)
        rows.add((c + 1) * C - 1)
    rng = np.random.default_rng(seed)
    rows.update(int(x) for x in rng.integers(0, S, size=n_random))
    return sorted(rows)
