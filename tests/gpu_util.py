"""Helpers shared by the GPU parity tests (calls go through the C-ABI binding)."""

import math

import numpy as np
import torch

import context_ring_attention_cp_gb300 as cpa
import oracle

# Tolerances for bf16 inputs with fp32 accumulation against the fp64 oracle.
OUT_MAX_ABS = 2e-2
OUT_MEAN_ABS = 2e-3
LSE_ABS = 2e-3
MERGE_REL = 1e-5  # per row: max|a - b| / max|b|


def f64(t):
    """bf16 device tensor -> exact float64 numpy array via the oracle's bit decoding."""
    return oracle.bf16_bits_to_f64(t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def ring_buffers(b, S, hq, d, device="cuda", identity=False):
    o = torch.empty((b, S, hq, d), dtype=torch.float32, device=device)
    m = torch.empty((b, hq, S), dtype=torch.float32, device=device)
    l = torch.empty((b, hq, S), dtype=torch.float32, device=device)
    if identity:
        o.zero_(); m.fill_(-math.inf); l.zero_()
    return o, m, l


def run_ring(q, k, v, cp, t0, t1, mode, bufs=None):
    b, S, hq, d = q.shape
    hkv = k.shape[2]
    desc = cpa.make_desc(b, S, hq, hkv, d, cp, 1.0 / math.sqrt(d), 1)
    o, m, l = bufs if bufs is not None else ring_buffers(b, S, hq, d)
    cpa.cp_ring_step_partial_attn(desc, t0, t1, q, k, v, o, m, l, mode)
    assert cpa.cp_take_device_status() == 0
    return o, m, l


def assert_out_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    assert err.max() <= OUT_MAX_ABS, f"{what}: max abs err {err.max():.3e} > {OUT_MAX_ABS}"
    assert err.mean() <= OUT_MEAN_ABS, f"{what}: mean abs err {err.mean():.3e} > {OUT_MEAN_ABS}"
    return float(err.max()), float(err.mean())


def assert_rowwise_rel(got, ref, tol, what=""):
    got = np.asarray(got, dtype=np.float64).reshape(-1, got.shape[-1])
    ref = np.asarray(ref, dtype=np.float64).reshape(-1, ref.shape[-1])
    scale = np.abs(ref).max(axis=1)
    err = np.abs(got - ref).max(axis=1)
    live = scale > 0
    assert np.all(err[~live] == 0), f"{what}: identity rows not exactly zero"
    rel = (err[live] / scale[live]).max() if live.any() else 0.0
    assert rel <= tol, f"{what}: row-relative err {rel:.3e} > {tol}"
    return float(rel)
