"""The full ring on host buffers (cp_ring_attn_host) against the device-buffer call and the oracle.

cp_ring_attn_host runs the same kernel over groups of virtual ranks, with the
copies in and out overlapped, so its outputs must equal cp_ring_step_partial_attn
over all steps in EMIT | FINALIZE mode bit for bit (each CTA computes the same
rows from the same data in either launch).  Its partial launches never split a
query tile's key walk over a CTA cluster, so the device launch it is compared
with runs with that split turned off.  One case is also held to the fp64
oracle at the suite's prefill tolerances (output max-abs <= 2e-2, mean-abs <=
2e-3; lse within 2e-3).
"""

import math

import numpy as np
import pytest
import torch

import context_ring_attention_cp_gb300 as cpa
from context_ring_attention_cp_gb300 import synth
from oracle import attention as OA

from gpu_util import LSE_ABS, assert_out_close, f64, run_ring

pytestmark = pytest.mark.gpu

EMIT, FIN = cpa.CP_MODE_EMIT, cpa.CP_MODE_FINALIZE

# (b, S, h_q, h_kv, d, cp): cp = 1, odd cp, cp > 8 (groups of two ranks), batch > 1
# (strided copies), ragged chunks (C % 128 != 0), d = 64.
CASES = [
    (1, 1024, 4, 4, 64, 2),
    (2, 1536, 4, 2, 128, 3),
    (1, 384, 3, 3, 64, 1),
    (1, 4096, 8, 2, 128, 16),
    (3, 640, 4, 1, 128, 5),
    (1, 4096, 32, 8, 128, 8),
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from context_ring_attention_cp_gb300 import _build
    _build.build()
    cpa.load_library()
    cpa.cp_set_kernel_choice(cpa.CP_KNOB_RING_KV_SPLIT, 0)
    yield
    cpa.cp_set_kernel_choice(cpa.CP_KNOB_RING_KV_SPLIT, -1)


def _host_call(desc, q, k, v, pinned=True):
    b, S, hq, d = q.shape
    hq_, hk_, hv_ = (x.cpu() for x in (q, k, v))
    o = torch.full((b, S, hq, d), float("nan"), dtype=torch.float32)
    m = torch.full((b, hq, S), float("nan"), dtype=torch.float32)
    l = torch.full((b, hq, S), float("nan"), dtype=torch.float32)
    if pinned:
        hq_, hk_, hv_, o, m, l = (x.pin_memory() for x in (hq_, hk_, hv_, o, m, l))
    nbytes = cpa.cp_ring_attn_host_workspace_bytes(desc)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    cpa.cp_ring_attn_host(desc, hq_, hk_, hv_, o, m, l, ws, nbytes)
    torch.cuda.synchronize()
    assert cpa.cp_take_device_status() == 0
    return o, m, l


@pytest.mark.parametrize("case", CASES, ids=[str(c) for c in CASES])
def test_host_ring_equals_device_ring(case):
    b, S, hq, hkv, d, cp = case
    q, k, v = synth.prefill_inputs(b, S, hq, hkv, d, std=0.5, seed=sum(case))
    desc = cpa.make_desc(b, S, hq, hkv, d, cp, 1.0 / math.sqrt(d), 1)
    o, m, l = _host_call(desc, q, k, v)
    od, md, ld = run_ring(q, k, v, cp, 0, cp, EMIT | FIN)
    assert torch.equal(o, od.cpu())
    assert torch.equal(m, md.cpu())
    assert torch.equal(l, ld.cpu())


def test_host_ring_against_the_oracle_and_with_pageable_memory():
    b, S, hq, hkv, d, cp = 2, 1024, 4, 2, 128, 4
    q, k, v = synth.prefill_inputs(b, S, hq, hkv, d, std=1.0, seed=7)
    desc = cpa.make_desc(b, S, hq, hkv, d, cp, 1.0 / math.sqrt(d), 1)
    o, m, l = _host_call(desc, q, k, v, pinned=False)
    ref_out, ref_m, ref_l, _ = OA.full_causal_attention(f64(q), f64(k), f64(v), 1.0 / math.sqrt(d))
    assert_out_close(o.numpy(), ref_out, "host ring out")
    lse = (m + torch.log(l)).numpy()
    assert np.abs(lse - (ref_m + np.log(ref_l))).max() <= LSE_ABS
    o2, m2, l2 = _host_call(desc, q, k, v, pinned=True)
    assert torch.equal(o, o2) and torch.equal(m, m2) and torch.equal(l, l2)


def test_two_calls_in_a_row_on_one_stream_reuse_the_workspace():
    # The second call's copies into the workspace must wait for the first call's
    # kernels and copies out: both results must match their own device-buffer run.
    b, S, hq, hkv, d, cp = 1, 2048, 8, 2, 128, 8
    desc = cpa.make_desc(b, S, hq, hkv, d, cp, 1.0 / math.sqrt(d), 1)
    nbytes = cpa.cp_ring_attn_host_workspace_bytes(desc)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    runs = []
    for seed in (11, 12):
        q, k, v = synth.prefill_inputs(b, S, hq, hkv, d, std=0.5, seed=seed)
        hq_, hk_, hv_ = (x.cpu().pin_memory() for x in (q, k, v))
        outs = [torch.empty(shape, dtype=torch.float32).pin_memory()
                for shape in ((b, S, hq, d), (b, hq, S), (b, hq, S))]
        cpa.cp_ring_attn_host(desc, hq_, hk_, hv_, *outs, ws, nbytes)
        runs.append((q, k, v, outs, (hq_, hk_, hv_)))
    torch.cuda.synchronize()
    for q, k, v, (o, m, l), _ in runs:
        od, md, ld = run_ring(q, k, v, cp, 0, cp, EMIT | FIN)
        assert torch.equal(o, od.cpu()) and torch.equal(m, md.cpu()) and torch.equal(l, ld.cpu())


def test_host_ring_at_full_size_equals_the_device_ring():
    # The end-to-end call the benchmark times (GQA workload, pinned host buffers) gives
    # the device-buffer launch's outputs bit for bit; that launch is held to the oracle
    # on sampled rows at the same size in test_gpu_prefill.
    w = synth.WORKLOADS["gqa"]
    q, k, v = synth.prefill_inputs(w["b"], w["S"], w["h_q"], w["h_kv"], w["d"], std=w["std"], seed=w["seed"])
    desc = cpa.make_desc(w["b"], w["S"], w["h_q"], w["h_kv"], w["d"], w["cp"], 1.0 / math.sqrt(w["d"]), 1)
    o, m, l = _host_call(desc, q, k, v)
    od, md, ld = run_ring(q, k, v, w["cp"], 0, w["cp"], EMIT | FIN)
    assert torch.equal(m, md.cpu()) and torch.equal(l, ld.cpu())
    assert torch.equal(o, od.cpu())
    del q, k, v, od, md, ld
    torch.cuda.empty_cache()
