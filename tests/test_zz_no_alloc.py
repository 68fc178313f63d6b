"""Pass-Q decode through the entry point that allocates nothing.

cp_passq_decode_noalloc serves callers that cannot allocate device memory where
they decode: a plug-in whose host runtime owns all of HBM and passes it only
input and output buffers, or a token loop that must not call cudaMalloc because
it may synchronise the device.  Its partials go to a fixed 8 MiB scratch array
inside the library instead of a caller workspace.

These tests call it through the C-ABI and check that it returns what the
workspace entry point (cp_passq_decode) returns for the same inputs, and what the
fp64 oracle's decode attention gives, within the decode tolerances used everywhere
in the suite (output max-abs <= 2e-2, mean-abs <= 2e-3; lse within 2e-3), on two
calls in a row with different inputs: the shared scratch keeps the previous call's
contents, and that must not leak into the next result.  One case is large enough
that the scratch holds fewer key ranges per shard than the workspace entry point
uses; it too is held to the oracle.  This file is collected last so that a run
stopping at the first failure has run every other test before it.
"""

import math

import numpy as np
import pytest
import torch

import context_ring_attention_cp_gb300 as cpa
import oracle
from context_ring_attention_cp_gb300 import synth
from oracle import attention as OA

pytestmark = pytest.mark.gpu

OUT_MAX_ABS = 2e-2
OUT_MEAN_ABS = 2e-3
LSE_ABS = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from context_ring_attention_cp_gb300 import _build
    _build.build()
    cpa.load_library()


def _with_workspace(desc, q, k, v):
    nbytes = cpa.cp_passq_workspace_bytes(desc)
    ws = torch.empty(nbytes // 4, dtype=torch.float32, device="cuda")
    out = torch.empty((desc.b, desc.h_q, desc.d), dtype=torch.float32, device="cuda")
    m = torch.empty((desc.b, desc.h_q), dtype=torch.float32, device="cuda")
    l = torch.empty_like(m)
    cpa.cp_passq_decode(desc, q, k, v, ws, nbytes, out, m, l)
    torch.cuda.synchronize()
    return out, m, l


def _without_workspace(desc, q, k, v):
    out = torch.empty((desc.b, desc.h_q, desc.d), dtype=torch.float32, device="cuda")
    m = torch.empty((desc.b, desc.h_q), dtype=torch.float32, device="cuda")
    l = torch.empty_like(m)
    cpa.cp_passq_decode_noalloc(desc, q, k, v, out, m, l)
    torch.cuda.synchronize()
    return out, m, l


def _f64(t):
    return oracle.bf16_bits_to_f64(synth.bf16_bits(t))


def _close_to_oracle(got, q, k, v, d, seqs=None):
    """The decode output and lse of the sequences ``seqs`` against the fp64 oracle."""
    seqs = range(q.shape[0]) if seqs is None else seqs
    for bi in seqs:
        ref_out, ref_m, ref_l = OA.decode_attention(_f64(q[bi:bi + 1]), _f64(k[bi:bi + 1]), _f64(v[bi:bi + 1]),
                                                    1.0 / math.sqrt(d))
        err = np.abs(got[0][bi:bi + 1].cpu().numpy() - ref_out)
        assert err.max() <= OUT_MAX_ABS and err.mean() <= OUT_MEAN_ABS, (bi, err.max(), err.mean())
        lse = (got[1][bi] + torch.log(got[2][bi])).cpu().numpy()
        assert np.abs(lse - (ref_m[0] + np.log(ref_l[0]))).max() <= LSE_ABS, bi


def _close(got, ref):
    err = (got[0] - ref[0]).abs()
    assert torch.isfinite(got[0]).all()
    assert err.max().item() <= OUT_MAX_ABS and err.mean().item() <= OUT_MEAN_ABS
    lse_got = got[1] + torch.log(got[2])
    lse_ref = ref[1] + torch.log(ref[2])
    assert (lse_got - lse_ref).abs().max().item() <= LSE_ABS


def test_noalloc_matches_workspace_decode_on_two_calls_in_a_row():
    # two different problems back to back: the second runs over the first one's leftovers
    cases = [(8, 16384, 16, 16, 512, 8, 101), (3, 6144, 8, 2, 128, 3, 202), (4, 8192, 16, 1, 512, 4, 303)]
    results = []
    for b, L, hq, hkv, d, cp, seed in cases:
        q, k, v = synth.decode_inputs(b, L, hq, hkv, d, seed=seed)
        desc = cpa.make_desc(b, L, hq, hkv, d, cp, 1.0 / math.sqrt(d), 0)
        ref = _with_workspace(desc, q, k, v)
        got = _without_workspace(desc, q, k, v)
        _close(got, ref)
        _close_to_oracle(got, q, k, v, d)
        results.append((desc, q, k, v, ref))
    # and the first problem again, after the second one overwrote the scratch
    desc, q, k, v, ref = results[0]
    _close(_without_workspace(desc, q, k, v), ref)
    assert cpa.cp_take_device_status() == 0


def test_noalloc_with_fewer_key_ranges_than_the_workspace_path_matches_the_oracle():
    # 16 query heads on one 512-wide K/V head, b8, L131072, cp8: the workspace entry point
    # cuts each shard into more key ranges than the scratch can hold partials for, so the
    # no-alloc call runs with fewer, longer ranges.  Twice in a row, then against the
    # oracle on two full sequences and against the workspace path on all of them.
    b, L, hq, hkv, d, cp = 8, 131072, 16, 1, 512, 8
    desc = cpa.make_desc(b, L, hq, hkv, d, cp, 1.0 / math.sqrt(d), 0)
    assert cpa.cp_passq_workspace_bytes(desc) > cpa.CP_PASSQ_NOALLOC_SCRATCH_BYTES
    q, k, v = synth.decode_inputs(b, L, hq, hkv, d, seed=404)
    first = _without_workspace(desc, q, k, v)
    got = _without_workspace(desc, q, k, v)
    assert torch.equal(first[0], got[0]) and torch.equal(first[1], got[1]) and torch.equal(first[2], got[2])
    _close(got, _with_workspace(desc, q, k, v))
    _close_to_oracle(got, q, k, v, d, seqs=(0, 6))
    assert cpa.cp_take_device_status() == 0
    del q, k, v
    torch.cuda.empty_cache()


def test_noalloc_rejects_problems_larger_than_its_scratch():
    # 8 shards x 64 sequences x 64 heads x (512 + 2) floats = 67 MB of partials > 8 MiB
    desc = cpa.make_desc(64, 4096, 64, 64, 512, 8, 1.0 / math.sqrt(512), 0)
    q = torch.zeros(16, dtype=torch.bfloat16, device="cuda")  # never read: rejected before any launch
    out = torch.zeros(16, dtype=torch.float32, device="cuda")
    with pytest.raises(cpa.CpError) as e:  # raw addresses: the C ABI's own check, not the binding's
        cpa.cp_passq_decode_noalloc(desc, q.data_ptr(), q.data_ptr(), q.data_ptr(), out.data_ptr())
    assert e.value.status == 2 and "scratch" in str(e.value)
    assert cpa.CP_PASSQ_NOALLOC_SCRATCH_BYTES == 8 << 20
    assert np.all(out.cpu().numpy() == 0)
