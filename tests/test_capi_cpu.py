"""C-ABI checks that need no GPU: symbols, host planner, byte counts, argument errors.

No test here launches a kernel: every device-side call below carries an
argument the library rejects before touching CUDA.
"""

import ctypes
import os
import re

import numpy as np
import pytest
import torch

from oracle import comm as OC
from oracle import ring as OR

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cpattn.h")


@pytest.fixture(scope="module")
def cpa():
    from context_ring_attention_cp_gb300 import _build
    _build.build()
    import context_ring_attention_cp_gb300 as cpa
    cpa.load_library()
    return cpa


def _declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"CPATTN_API\s+[\w\s\*]+?\b(cp_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    syms = _declared_symbols()
    for name in ["cp_plan_balanced_chunks", "cp_plan_chunks", "cp_ring_step_partial_attn",
                 "cp_ring_rank_partial_attn", "cp_merge_partials", "cp_merge_partials_tree",
                 "cp_merge_tree_workspace_bytes", "cp_passq_decode", "cp_comm_bytes",
                 "cp_passq_workspace_bytes", "cp_status_string", "cp_take_device_status"]:
        assert name in syms, name


def test_library_exports_every_declared_symbol(cpa):
    lib = ctypes.CDLL(cpa.library_path())
    for name in _declared_symbols():
        assert hasattr(lib, name), f"{name} declared in cpattn.h but not exported"


def test_status_strings(cpa):
    assert cpa.cp_status_string(0) == "CP_OK"
    assert cpa.cp_status_string(5) == "CP_ERR_TIMEOUT"
    assert cpa.cp_status_string(99) == "CP_ERR_UNKNOWN"


@pytest.mark.parametrize("S,cp", [(2, 1), (8, 2), (24, 3), (64, 8), (96, 6), (1024, 2), (32768, 8),
                                  (131072, 16), (1 << 20, 8), (4096, 32)])
def test_plan_bit_exact_against_oracle(cpa, S, cp):
    plan = cpa.cp_plan_balanced_chunks(S, cp)
    assert plan["chunk_begin"].tolist() == OR.chunk_begin(S, cp)
    assert plan["rank_chunks"].tolist() == OR.rank_chunks(cp)
    assert plan["step_src"].tolist() == OR.step_source(cp)
    assert plan["step_pairs"].tolist() == OR.step_pairs_closed_form(S, cp)
    if S <= 128:
        assert plan["step_pairs"].tolist() == OR.step_pairs_enumerated(S, cp)


@pytest.mark.parametrize("S,cp", [(2, 1), (16, 2), (24, 3), (64, 4), (96, 8), (32768, 8), (131072, 16)])
def test_sequential_plan_bit_exact_against_oracle(cpa, S, cp):
    plan = cpa.cp_plan_chunks(S, cp, cpa.CP_LAYOUT_SEQUENTIAL)
    assert plan["chunk_begin"].tolist() == OR.chunk_begin(S, cp)
    assert plan["rank_chunks"].tolist() == OR.rank_chunks(cp, "sequential")
    assert plan["step_src"].tolist() == OR.step_source(cp)
    assert plan["step_pairs"].tolist() == OR.step_pairs_sequential_closed_form(S, cp)
    assert plan["step_pairs"].sum(axis=1).tolist() == OR.sequential_split_pairs(S, cp)
    if S <= 128:
        assert plan["step_pairs"].tolist() == OR.step_pairs_enumerated(S, cp, "sequential")
    balanced = cpa.cp_plan_chunks(S, cp, cpa.CP_LAYOUT_BALANCED)
    assert balanced["step_pairs"].tolist() == cpa.cp_plan_balanced_chunks(S, cp)["step_pairs"].tolist()


def test_plan_rejects_unknown_layout(cpa):
    with pytest.raises(cpa.CpError) as e:
        cpa.cp_plan_chunks(16, 2, 2)
    assert e.value.status == 1


@pytest.mark.parametrize("layout,r0,r1", [(2, 0, 1), (-1, 0, 1), (0, -1, 1), (0, 1, 1), (0, 0, 3), (1, 2, 1)])
def test_rank_range_rejects(cpa, layout, r0, r1):
    desc = cpa.make_desc(1, 1024, 4, 4, 64, 2, 0.125, 1)
    with pytest.raises(cpa.CpError) as e:
        cpa.cp_ring_rank_partial_attn(desc, layout, r0, r1, 0, 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, stream=0)
    assert e.value.status == 1


@pytest.mark.parametrize("S,cp", [(0, 1), (10, 0), (10, -2), (10, 3), (7, 1), (12, 4)])
def test_plan_rejects(cpa, S, cp):
    with pytest.raises(cpa.CpError) as e:
        cpa.cp_plan_balanced_chunks(S, cp)
    assert e.value.status == 1


COMM_CASES = [
    # (S, cp, c_kv, b, d, n_h, s)
    (1024, 2, 2 * 4 * 64 * 2, 0, 0, 0, 0),
    (32768, 8, 2 * 8 * 128 * 2, 0, 0, 0, 0),
    (131072, 16, 2 * 8 * 128 * 2, 0, 0, 0, 0),
    (131072, 8, 0, 8, 16 * 512, 16, 2),
    (131072, 8, 0, 8, 16 * 512, 16, 4),
    (1 << 20, 8, 320, 1, 7168, 128, 2),
    (1 << 20, 1, 320, 1, 1, 1, 1),
    (0, 4, 100, 0, 0, 0, 0),
]


@pytest.mark.parametrize("case", COMM_CASES)
def test_comm_bytes_bit_exact_against_oracle(cpa, case):
    S, cp, c_kv, b, d, n_h, s = case
    got = cpa.cp_comm_bytes(S, cp, c_kv, b, d, n_h, s)
    total, per = OC.passkv_bytes(S, cp, c_kv)
    disp, red = OC.passq_bytes(b, d, n_h, s)
    assert (got["passkv_total"], got["passkv_per_step"]) == (total, per)
    assert (got["passq_dispatch"], got["passq_reduce"]) == (disp, red)


@pytest.mark.parametrize("b,S,cp,c_kv,L", [(1, 1 << 20, 8, 320, 61), (1, 1 << 20, 16, 320, 61), (8, 131072, 8, 16384, 1),
                                             (2, 96, 4, 3, 5), (1, 64, 1, 8, 0)])
def test_kv_bytes_per_rank_bit_exact(cpa, b, S, cp, c_kv, L):
    got = cpa.cp_comm_bytes(S, cp, c_kv, b=b, layers_local=L)["kv_bytes_per_rank"]
    assert got == OC.kv_bytes_per_rank(b, S, c_kv, L, cp)


def test_kv_per_rank_halves_from_cp8_to_cp16(cpa):
    # use case section: raising cp from 8 to 16 halves the KV each card holds
    a = cpa.cp_comm_bytes(1 << 20, 8, 320, b=1, layers_local=61)["kv_bytes_per_rank"]
    c = cpa.cp_comm_bytes(1 << 20, 16, 320, b=1, layers_local=61)["kv_bytes_per_rank"]
    assert 2 * c == a


def test_comm_bytes_at_the_workloads(cpa):
    # c_kv = K and V, h_kv heads of d_head bf16 values: 2*4*64*2 = 1024 B (tiny) and
    # 2*8*128*2 = 4096 B (gqa, long); eq. g5cp-passkv-bytes multiplied out by hand
    for S, cp, c_kv, total, per_step in [(1024, 2, 1024, 524_288, 524_288),
                                         (32768, 8, 4096, 117_440_512, 16_777_216),
                                         (131072, 16, 4096, 503_316_480, 33_554_432)]:
        got = cpa.cp_comm_bytes(S, cp, c_kv)
        assert (got["passkv_total"], got["passkv_per_step"]) == (total, per_step)
    # pass-Q at the decode workload: b 8, n_h 16, d = 16 * 512
    got = cpa.cp_comm_bytes(131072, 8, 0, b=8, d=8192, n_h=16, s_dtype=2)
    assert (got["passq_dispatch"], got["passq_reduce"]) == (131_072, 131_584)
    # per-rank KV of the gqa workload over 36 layers: 1 * 32768 * 4096 * 36 / 8
    got = cpa.cp_comm_bytes(32768, 8, 4096, b=1, layers_local=36)
    assert got["kv_bytes_per_rank"] == 603_979_776


def test_comm_bytes_overflow_and_errors(cpa):
    big = (1 << 62)
    with pytest.raises(cpa.CpError) as e:
        cpa.cp_comm_bytes(big, 2, 1 << 10)
    assert e.value.status == 3
    assert not OC.fits_u64(OC.passkv_bytes(big, 2, 1 << 10)[0])
    # the largest values that still fit must come back exact
    S = (1 << 63) - 2  # even, divisible by cp = 2
    got = cpa.cp_comm_bytes(S, 2, 2)
    assert got["passkv_per_step"] == OC.passkv_bytes(S, 2, 2)[1] <= OC.U64_MAX
    with pytest.raises(cpa.CpError) as e:
        cpa.cp_comm_bytes(10, 3, 1)  # S not divisible by cp
    assert e.value.status == 1
    with pytest.raises(cpa.CpError) as e:
        cpa.cp_comm_bytes(10, 0, 1)
    assert e.value.status == 1
    with pytest.raises(cpa.CpError) as e:
        cpa.cp_comm_bytes(10, 1, 1, b=-1)
    assert e.value.status == 1
    with pytest.raises(cpa.CpError) as e:
        cpa.cp_comm_bytes(10, 1, 1, layers_local=-1)
    assert e.value.status == 1
    with pytest.raises(cpa.CpError) as e:  # footprint overflows even though the ring bytes fit
        cpa.cp_comm_bytes(1 << 40, 1, 1 << 10, b=1 << 20, layers_local=1)
    assert e.value.status == 3


# --- device entry points: argument errors only (rejected before any CUDA call) ---

FAKE = 1 << 20  # a 16-byte aligned stand-in address; never dereferenced (rejected first)


def _desc(cpa, **kw):
    base = dict(b=1, S=1024, h_q=4, h_kv=4, d=64, cp=2, scale=0.125, causal=1)
    base.update(kw)
    return cpa.make_desc(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(cp=0), 1), (dict(cp=-1), 1), (dict(S=1000, cp=8), 1), (dict(S=0), 1), (dict(b=0), 1),
    (dict(h_q=6, h_kv=4), 1), (dict(scale=0.0), 1), (dict(scale=-1.0), 1), (dict(scale=float("inf")), 1),
    (dict(scale=float("nan")), 1), (dict(d=96), 2), (dict(d=256), 2), (dict(causal=0), 2),
    # beyond the kernel's 32-bit row, batch and head indexing
    (dict(S=1 << 30, cp=1), 2), (dict(b=65536, S=2, cp=1), 2), (dict(h_q=65536, h_kv=65536, S=2, cp=1), 2),
])
def test_ring_rejects_descriptors(cpa, kw, status):
    with pytest.raises(cpa.CpError) as e:
        cpa.cp_ring_step_partial_attn(_desc(cpa, **kw), 0, 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, stream=0)
    assert e.value.status == status


@pytest.mark.parametrize("t0,t1,mode", [(-1, 1, 0), (1, 1, 0), (0, 3, 0), (2, 1, 0), (0, 2, 8), (0, 2, -1)])
def test_ring_rejects_steps_and_modes(cpa, t0, t1, mode):
    with pytest.raises(cpa.CpError) as e:
        cpa.cp_ring_step_partial_attn(_desc(cpa), t0, t1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, mode, stream=0)
    assert e.value.status == 1


@pytest.mark.parametrize("bad", [0, 1, 2, 3, 4, 5])
def test_ring_rejects_null_or_misaligned(cpa, bad):
    ptrs = [FAKE] * 6
    for p in (0, FAKE + 8):
        ptrs[bad] = p
        with pytest.raises(cpa.CpError) as e:
            cpa.cp_ring_step_partial_attn(_desc(cpa), 0, 2, *ptrs, 0, stream=0)
        assert e.value.status == 1


@pytest.mark.parametrize("args,status", [
    (dict(batch=0), 1), (dict(rows=0), 1), (dict(n_parts=0), 1), (dict(n_parts=257), 1), (dict(d=6), 1),
    (dict(d=516), 2), (dict(order=[0, 0]), 1), (dict(order=[0, 2]), 1), (dict(order=[1]), 1),
    (dict(o_parts=FAKE + 4), 1), (dict(m_out=0), 1),
])
def test_merge_rejects(cpa, args, status):
    kw = dict(batch=1, rows=8, heads=2, d=8, n_parts=2, o_parts=FAKE, m_parts=FAKE, l_parts=FAKE,
              o_out=FAKE, m_out=FAKE, l_out=FAKE, order=None)
    kw.update(args)
    with pytest.raises(cpa.CpError) as e:
        cpa.cp_merge_partials(kw["batch"], kw["rows"], kw["heads"], kw["d"], kw["n_parts"], kw["o_parts"],
                              kw["m_parts"], kw["l_parts"], kw["o_out"], kw["m_out"], kw["l_out"],
                              order=kw["order"], stream=0)
    assert e.value.status == status


@pytest.mark.parametrize("kw,status", [
    (dict(S=1000, cp=3), 1), (dict(cp=0), 1), (dict(d=96), 2), (dict(d=1024), 2), (dict(h_q=16, h_kv=2), 2),
    (dict(h_q=8, h_kv=2, d=512), 2), (dict(causal=1), 2), (dict(h_q=3, h_kv=2), 1),
])
def test_decode_rejects(cpa, kw, status):
    base = dict(b=2, S=1024, h_q=4, h_kv=4, d=128, cp=2, scale=0.1, causal=0)
    base.update(kw)
    desc = cpa.make_desc(**base)
    with pytest.raises(cpa.CpError) as e:
        cpa.cp_passq_decode(desc, FAKE, FAKE, FAKE, FAKE, 1 << 30, FAKE, stream=0)
    assert e.value.status == status
    with pytest.raises(cpa.CpError) as e:
        cpa.cp_passq_workspace_bytes(desc)
    assert e.value.status == status


def test_binding_has_no_fallback(tmp_path, monkeypatch):
    import context_ring_attention_cp_gb300 as cpa
    monkeypatch.setattr(cpa, "_LIB", None)
    monkeypatch.setattr(cpa, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        cpa.cp_comm_bytes(8, 2, 1)


@pytest.mark.parametrize("n", [0, 1, 3, 6, 12])
def test_tree_merge_needs_a_power_of_two(cpa, n):
    with pytest.raises(cpa.CpError) as e:
        cpa.cp_merge_tree_workspace_bytes(1, 8, 2, 8, n)
    assert e.value.status == 1


def test_tree_merge_needs_no_workspace_and_at_most_256_parts(cpa):
    # the tree is computed in one pass: no intermediate levels in memory
    assert cpa.cp_merge_tree_workspace_bytes(1, 4096, 64, 128, 32) == 0
    assert cpa.cp_merge_tree_workspace_bytes(1, 8, 2, 8, 256) == 0
    with pytest.raises(cpa.CpError) as e:
        cpa.cp_merge_tree_workspace_bytes(1, 8, 2, 8, 512)
    assert e.value.status == 1


def _round256(x):
    return (x + 255) // 256 * 256


def test_host_ring_workspace_size(cpa):
    # device copies of q, k, v (bf16), o (fp32) and m, l (fp32), each rounded up to 256 bytes
    b, S, hq, hkv, d = 2, 1000, 6, 2, 128
    want = (_round256(b * S * hq * d * 2) + 2 * _round256(b * S * hkv * d * 2) + _round256(b * S * hq * d * 4)
            + 2 * _round256(b * hq * S * 4))
    assert cpa.cp_ring_attn_host_workspace_bytes(_desc(cpa, b=b, S=S, h_q=hq, h_kv=hkv, d=d)) == want


@pytest.mark.parametrize("kw,status", [(dict(cp=0), 1), (dict(S=1000, cp=8), 1), (dict(h_q=6, h_kv=4), 1),
                                       (dict(d=96), 2), (dict(causal=0), 2)])
def test_host_ring_rejects_descriptors(cpa, kw, status):
    with pytest.raises(cpa.CpError) as e:
        cpa.cp_ring_attn_host_workspace_bytes(_desc(cpa, **kw))
    assert e.value.status == status
    with pytest.raises(cpa.CpError) as e:
        cpa.cp_ring_attn_host(_desc(cpa, **kw), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4096, 1 << 40, stream=0)
    assert e.value.status == status


@pytest.mark.parametrize("bad", range(7))
def test_host_ring_rejects_null_pointers_and_small_or_misaligned_workspace(cpa, bad):
    desc = _desc(cpa)
    need = cpa.cp_ring_attn_host_workspace_bytes(desc)
    ptrs = [FAKE] * 6 + [4096]
    ptrs[bad] = 0
    with pytest.raises(cpa.CpError) as e:
        cpa.cp_ring_attn_host(desc, *ptrs, need, stream=0)
    assert e.value.status == 1
    with pytest.raises(cpa.CpError) as e:  # workspace one byte short
        cpa.cp_ring_attn_host(desc, *([FAKE] * 6), 4096, need - 1, stream=0)
    assert e.value.status == 1
    with pytest.raises(cpa.CpError) as e:  # workspace not 256-byte aligned
        cpa.cp_ring_attn_host(desc, *([FAKE] * 6), 4096 + 16, need, stream=0)
    assert e.value.status == 1


def _ring_tensors(b=1, S=1024, hq=4, hkv=2, d=64):
    q = torch.zeros((b, S, hq, d), dtype=torch.bfloat16)
    k = torch.zeros((b, S, hkv, d), dtype=torch.bfloat16)
    v = torch.zeros_like(k)
    o = torch.zeros((b, S, hq, d), dtype=torch.float32)
    m = torch.zeros((b, hq, S), dtype=torch.float32)
    return [q, k, v, o, m, torch.zeros_like(m)]


@pytest.mark.parametrize("bad", ["dtype", "layout", "size", "device"])
def test_binding_checks_tensor_arguments(cpa, bad):
    """The binding rejects a tensor the kernels would read or write out of bounds, before any call."""
    desc = _desc(cpa, h_q=4, h_kv=2)
    args = _ring_tensors()
    if bad == "dtype":
        args[0] = args[0].float()
    elif bad == "layout":
        args[3] = torch.zeros((1, 1024, 4, 128), dtype=torch.float32)[..., ::2]
    elif bad == "size":
        args[4] = args[4][:, :, :512]
    # "device": host tensors passed to a device entry point
    with pytest.raises(ValueError):
        cpa.cp_ring_step_partial_attn(desc, 0, 2, *args, 0, stream=0)


def test_binding_checks_merge_decode_and_host_ring_arguments(cpa):
    o = torch.zeros((2, 1, 8, 2, 8), dtype=torch.float32)
    ml = torch.zeros((2, 1, 2, 8), dtype=torch.float32)
    oo = torch.zeros((1, 8, 2, 8), dtype=torch.float32)
    mo = torch.zeros((1, 2, 8), dtype=torch.float32)
    with pytest.raises(ValueError):  # too few parts in o_parts
        cpa.cp_merge_partials(1, 8, 2, 8, 3, o, ml, ml, oo, mo, mo, stream=0)
    with pytest.raises(ValueError):  # workspace smaller than the bytes passed
        cpa.cp_merge_partials_tree(1, 8, 2, 8, 2, o, ml, ml, torch.zeros(4), 64, oo, mo, mo, stream=0)
    ddesc = cpa.make_desc(1, 256, 2, 2, 128, 2, 0.1, 0)
    q = torch.zeros((1, 2, 128), dtype=torch.bfloat16)
    kv = torch.zeros((1, 256, 2, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError):  # out must be fp32
        cpa.cp_passq_decode(ddesc, q, kv, kv, FAKE, 1 << 20, torch.zeros((1, 2, 128), dtype=torch.bfloat16), stream=0)
    with pytest.raises(ValueError):  # the host-buffer ring wants host tensors and a device workspace
        cpa.cp_ring_attn_host(_desc(cpa, h_q=4, h_kv=2), *_ring_tensors(), torch.zeros(1 << 10, dtype=torch.uint8),
                              1 << 10, stream=0)


class _FakeCudaTensor:
    """Stands in for a CUDA tensor on a chosen device (no GPU is needed to test the check)."""

    def __init__(self, index, dtype=torch.float32, numel=64):
        self.dtype, self.is_cuda, self._n = dtype, True, numel
        self.device = torch.device("cuda", index)

    def is_contiguous(self):
        return True

    def numel(self):
        return self._n

    def element_size(self):
        return 4

    def data_ptr(self):
        return 4096

    def get_device(self):
        return self.device.index


def test_binding_rejects_a_tensor_on_another_device(cpa, monkeypatch):
    # kernels run on the current device: a tensor of another GPU must never reach them
    monkeypatch.setattr(cpa, "_current_device", lambda: 0)
    assert cpa._arg(_FakeCudaTensor(0), "o", "test", torch.float32, 64) == 4096
    with pytest.raises(ValueError, match="cuda:1"):
        cpa._arg(_FakeCudaTensor(1), "o", "test", torch.float32, 64)
    desc = _desc(cpa, S=8, h_q=1, h_kv=1, d=8)
    args = [_FakeCudaTensor(0, torch.bfloat16)] * 3 + [_FakeCudaTensor(0)] * 3
    args[4] = _FakeCudaTensor(1)
    with pytest.raises(ValueError, match="m is on cuda:1"):
        cpa.cp_ring_step_partial_attn(desc, 0, 2, *args, 0, stream=0)


def test_kernel_choice_settings(cpa):
    lib = cpa.load_library()
    for knob in (cpa.CP_KNOB_RING_PAIRING, cpa.CP_KNOB_MERGE_KERNEL, cpa.CP_KNOB_RING_KV_SPLIT):
        for value in (-1, 0, 1, -1):
            cpa.cp_set_kernel_choice(knob, value)
        for bad in (-2, 2):
            assert lib.cp_set_kernel_choice(knob, bad) == 1
    for bad_knob in (-1, 3, 99):
        with pytest.raises(cpa.CpError) as e:
            cpa.cp_set_kernel_choice(bad_knob, 0)
        assert e.value.status == 1


def test_library_reads_no_environment_variable():
    # kernel choices are explicit settings, never read from the caller's environment
    import glob
    for path in glob.glob(os.path.join(os.path.dirname(__file__), "..", "context_ring_attention_cp_gb300", "csrc", "*")):
        assert "getenv" not in open(path).read(), path
