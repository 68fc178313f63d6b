"""Thin Python binding of ``libcpattn.so`` — argument marshalling only.

Every function here has the name of the C-ABI entry point it calls
(``include/cpattn.h``) and does nothing but turn tensors into pointers and
sizes, pick the current CUDA stream, and raise :class:`CpError` on a non-OK
status.  All computation happens in the library's CUDA kernels (or, for the
planner and byte counts, in its host C++).  There is no fallback: if the
library is missing this module raises on first use.

PyTorch is used only for device memory and streams.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

__all__ = [
    "CpError", "AttnDesc", "CP_MODE_EMIT", "CP_MODE_ACCUMULATE", "CP_MODE_FINALIZE", "CP_MODE_OVERLAP_PREVIOUS",
    "CP_MAX_MERGE_PARTS", "library_path", "load_library", "cp_status_string",
    "cp_ring_attn_host", "cp_ring_attn_host_workspace_bytes",
    "cp_plan_balanced_chunks", "cp_plan_chunks", "cp_comm_bytes", "cp_ring_step_partial_attn",
    "cp_ring_rank_partial_attn", "cp_merge_partials", "CP_LAYOUT_BALANCED", "CP_LAYOUT_SEQUENTIAL",
    "cp_passq_workspace_bytes", "cp_passq_decode", "cp_passq_decode_noalloc", "cp_take_device_status",
    "cp_merge_tree_workspace_bytes", "cp_merge_partials_tree", "cp_selftest_wait_timeout",
    "cp_set_kernel_choice", "CP_KNOB_RING_PAIRING", "CP_KNOB_MERGE_KERNEL", "CP_KNOB_RING_KV_SPLIT",
]

CP_OK = 0
CP_ERR_INVALID_ARGUMENT = 1
CP_ERR_UNSUPPORTED = 2
CP_ERR_OVERFLOW = 3
CP_ERR_CUDA = 4
CP_ERR_TIMEOUT = 5
CP_MODE_EMIT = 0
CP_MODE_ACCUMULATE = 1
CP_MODE_FINALIZE = 2
CP_MODE_OVERLAP_PREVIOUS = 4
CP_LAYOUT_BALANCED = 0
CP_LAYOUT_SEQUENTIAL = 1
CP_MAX_MERGE_PARTS = 256
CP_PASSQ_NOALLOC_SCRATCH_BYTES = 8 << 20
CP_KNOB_RING_PAIRING = 0
CP_KNOB_MERGE_KERNEL = 1
CP_KNOB_RING_KV_SPLIT = 2

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB = None


def library_path() -> str:
    return os.path.join(_PKG, "libcpattn.so")


class CpError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {cp_status_string(status)} ({status})")


class AttnDesc(ctypes.Structure):
    """Mirror of ``cp_attn_desc``."""
    _fields_ = [("b", ctypes.c_int64), ("S", ctypes.c_int64), ("h_q", ctypes.c_int64),
                ("h_kv", ctypes.c_int64), ("d", ctypes.c_int64), ("cp", ctypes.c_int64),
                ("scale", ctypes.c_float), ("causal", ctypes.c_int32)]


class _CommQuery(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("S", "cp", "c_kv", "b", "d", "n_h", "s_dtype", "layers_local")]


class _CommResult(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in ("passkv_total", "passkv_per_step", "passq_dispatch",
                                               "passq_reduce", "kv_bytes_per_rank")]


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32


def load_library():
    """Load ``libcpattn.so`` (it must have been built); raises if it is absent."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built: run __graft_entry__.build() (or "
                           "python -m context_ring_attention_cp_gb300._build) first")
    lib = ctypes.CDLL(path)
    sig = {
        "cp_status_string": (ctypes.c_char_p, [_I32]),
        "cp_plan_balanced_chunks": (_I32, [_I64, _I32, _P, _P, _P, _P]),
        "cp_plan_chunks": (_I32, [_I64, _I32, _I32, _P, _P, _P, _P]),
        "cp_ring_rank_partial_attn": (_I32, [ctypes.POINTER(AttnDesc), _I32, _I32, _I32, _I32, _I32, _P, _P, _P, _P,
                                             _P, _P, _I32, _P]),
        "cp_comm_bytes": (_I32, [ctypes.POINTER(_CommQuery), ctypes.POINTER(_CommResult)]),
        "cp_ring_step_partial_attn": (_I32, [ctypes.POINTER(AttnDesc), _I32, _I32, _P, _P, _P, _P, _P, _P,
                                             _I32, _P]),
        "cp_merge_partials": (_I32, [_I64, _I64, _I64, _I64, _I32, _P, _P, _P, _P, _P, _P, _P, _I32, _P]),
        "cp_passq_workspace_bytes": (_I32, [ctypes.POINTER(AttnDesc), ctypes.POINTER(ctypes.c_size_t)]),
        "cp_passq_decode": (_I32, [ctypes.POINTER(AttnDesc), _P, _P, _P, _P, ctypes.c_size_t, _P, _P, _P, _P]),
        "cp_take_device_status": (_I32, [_P, ctypes.POINTER(_I32)]),
        "cp_merge_tree_workspace_bytes": (_I32, [_I64, _I64, _I64, _I64, _I32, ctypes.POINTER(ctypes.c_size_t)]),
        "cp_merge_partials_tree": (_I32, [_I64, _I64, _I64, _I64, _I32, _P, _P, _P, _P, ctypes.c_size_t, _P, _P, _P,
                                          _I32, _P]),
        "cp_passq_decode_noalloc": (_I32, [ctypes.POINTER(AttnDesc), _P, _P, _P, _P, _P, _P, _P]),
        "cp_selftest_wait_timeout": (_I32, [_P]),
        "cp_set_kernel_choice": (_I32, [_I32, _I32]),
        "cp_ring_attn_host_workspace_bytes": (_I32, [ctypes.POINTER(AttnDesc), ctypes.POINTER(ctypes.c_size_t)]),
        "cp_ring_attn_host": (_I32, [ctypes.POINTER(AttnDesc), _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def _ptr(x) -> Optional[int]:
    """Device address of a tensor (or an int address, or None)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _current_device() -> int:
    import torch
    return torch.cuda.current_device()


def _arg(x, name: str, where: str, dtype=None, numel: int = 0, nbytes: int = 0, cuda: bool = True,
         dev: Optional[list] = None) -> Optional[int]:
    """Address of a tensor argument, after the checks the C ABI cannot make through a plain
    pointer: dtype, contiguity, size against the descriptor, and device (CUDA tensors must
    be on the current device, where the kernels run).  A wrong buffer would otherwise be
    read or written out of bounds by the kernels.  None and raw int addresses pass
    through unchecked.  ``dev`` is a one-element list that caches the current device
    across the arguments of one call."""
    if x is None or isinstance(x, int):
        return x
    if dtype is not None and x.dtype != dtype:
        raise ValueError(f"{where}: {name} must be {dtype}, got {x.dtype}")
    if not x.is_contiguous():
        raise ValueError(f"{where}: {name} must be contiguous")
    n = x.numel()
    if n < numel:
        raise ValueError(f"{where}: {name} holds {n} elements, the descriptor needs {numel}")
    if nbytes and n * x.element_size() < nbytes:
        raise ValueError(f"{where}: {name} holds {n * x.element_size()} bytes, {nbytes} were passed")
    index = x.get_device()  # -1 for a host tensor
    if (index >= 0) != cuda:
        raise ValueError(f"{where}: {name} must be a {'CUDA' if cuda else 'host (CPU)'} tensor")
    if cuda:
        cur = dev[0] if dev is not None else None
        if cur is None:
            cur = _current_device()
            if dev is not None:
                dev[0] = cur
        if index != cur:
            raise ValueError(f"{where}: {name} is on cuda:{index}, but the current device "
                             f"(where the kernels run) is cuda:{cur}")
    return x.data_ptr()


def _ring_args(desc, q, k, v, o, m, l, where: str, cuda: bool = True, dev: Optional[list] = None):
    import torch
    b, S, hq, hkv, d = desc.b, desc.S, desc.h_q, desc.h_kv, desc.d  # ctypes fields read as ints
    n_q, n_kv, n_ml = b * S * hq * d, b * S * hkv * d, b * hq * S
    dev = [None] if dev is None else dev
    bf16, f32 = torch.bfloat16, torch.float32
    # positional arguments: this runs on every launch, and a latency-bound caller feels it
    return (_arg(q, "q", where, bf16, n_q, 0, cuda, dev), _arg(k, "k", where, bf16, n_kv, 0, cuda, dev),
            _arg(v, "v", where, bf16, n_kv, 0, cuda, dev), _arg(o, "o", where, f32, n_q, 0, cuda, dev),
            _arg(m, "m", where, f32, n_ml, 0, cuda, dev), _arg(l, "l", where, f32, n_ml, 0, cuda, dev))


def _merge_args(batch, rows, heads, d, n_parts, o_parts, m_parts, l_parts, o_out, m_out, l_out, where: str):
    import torch
    n, b, r, h, d = int(n_parts), int(batch), int(rows), int(heads), int(d)
    dev = [None]
    return (_arg(o_parts, "o_parts", where, torch.float32, n * b * r * h * d, dev=dev),
            _arg(m_parts, "m_parts", where, torch.float32, n * b * h * r, dev=dev),
            _arg(l_parts, "l_parts", where, torch.float32, n * b * h * r, dev=dev),
            _arg(o_out, "o_out", where, torch.float32, b * r * h * d, dev=dev),
            _arg(m_out, "m_out", where, torch.float32, b * h * r, dev=dev),
            _arg(l_out, "l_out", where, torch.float32, b * h * r, dev=dev))


def _decode_args(desc, q, k, v, out, m_out, l_out, where: str):
    import torch
    b, L, hq, hkv, d = int(desc.b), int(desc.S), int(desc.h_q), int(desc.h_kv), int(desc.d)
    dev = [None]
    return (_arg(q, "q", where, torch.bfloat16, b * hq * d, dev=dev),
            _arg(k, "k", where, torch.bfloat16, b * L * hkv * d, dev=dev),
            _arg(v, "v", where, torch.bfloat16, b * L * hkv * d, dev=dev),
            _arg(out, "out", where, torch.float32, b * hq * d, dev=dev),
            _arg(m_out, "m_out", where, torch.float32, b * hq, dev=dev),
            _arg(l_out, "l_out", where, torch.float32, b * hq, dev=dev))


def _stream(stream, dev: Optional[list] = None) -> Optional[int]:
    """The cudaStream_t to launch on: the given stream, or the current stream of the current
    device (``dev`` may hold that device, looked up by the argument checks)."""
    if stream is None:
        import torch
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is None:
            return torch.cuda.current_stream().cuda_stream
        d = dev[0] if dev is not None and dev[0] is not None else torch.cuda.current_device()
        return raw(d)
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str) -> None:
    if status != CP_OK:
        raise CpError(status, where)


def cp_status_string(status: int) -> str:
    return load_library().cp_status_string(int(status)).decode()


def make_desc(b, S, h_q, h_kv, d, cp, scale, causal) -> AttnDesc:
    return AttnDesc(int(b), int(S), int(h_q), int(h_kv), int(d), int(cp), float(scale), int(causal))


def cp_plan_balanced_chunks(S: int, cp: int) -> dict:
    """Host planner (balanced layout); returns the four plan arrays as numpy arrays."""
    return cp_plan_chunks(S, cp, CP_LAYOUT_BALANCED, _name="cp_plan_balanced_chunks")


def cp_plan_chunks(S: int, cp: int, layout: int = CP_LAYOUT_BALANCED, _name: str = "cp_plan_chunks") -> dict:
    """Host planner for either chunk layout; returns the four plan arrays as numpy arrays."""
    lib = load_library()
    if not isinstance(cp, (int, np.integer)) or cp < 1 or cp > (1 << 20):
        # the arrays below are sized by cp: reject before allocating (the library checks again)
        raise CpError(CP_ERR_INVALID_ARGUMENT, "cp_plan_balanced_chunks")
    chunk_begin = np.zeros(2 * cp + 1, np.int64)
    rank_chunks = np.zeros((cp, 2), np.int32)
    step_src = np.zeros((cp, cp), np.int32)
    step_pairs = np.zeros((cp, cp), np.int64)
    if _name == "cp_plan_balanced_chunks":
        st = lib.cp_plan_balanced_chunks(int(S), int(cp), chunk_begin.ctypes.data, rank_chunks.ctypes.data,
                                         step_src.ctypes.data, step_pairs.ctypes.data)
    else:
        st = lib.cp_plan_chunks(int(S), int(cp), int(layout), chunk_begin.ctypes.data, rank_chunks.ctypes.data,
                                step_src.ctypes.data, step_pairs.ctypes.data)
    _check(st, _name)
    return {"chunk_begin": chunk_begin, "rank_chunks": rank_chunks, "step_src": step_src,
            "step_pairs": step_pairs}


def cp_comm_bytes(S, cp, c_kv, b=0, d=0, n_h=0, s_dtype=0, layers_local=0) -> dict:
    """Closed-form pass-KV / pass-Q byte counts and per-rank KV footprint (host, exact uint64)."""
    lib = load_library()
    q = _CommQuery(int(S), int(cp), int(c_kv), int(b), int(d), int(n_h), int(s_dtype), int(layers_local))
    r = _CommResult()
    _check(lib.cp_comm_bytes(ctypes.byref(q), ctypes.byref(r)), "cp_comm_bytes")
    return {"passkv_total": int(r.passkv_total), "passkv_per_step": int(r.passkv_per_step),
            "passq_dispatch": int(r.passq_dispatch), "passq_reduce": int(r.passq_reduce),
            "kv_bytes_per_rank": int(r.kv_bytes_per_rank)}


def cp_ring_step_partial_attn(desc: AttnDesc, step_begin: int, step_end: int, q, k, v, o, m, l,
                              mode: int = CP_MODE_EMIT, stream=None) -> None:
    """Ring steps [step_begin, step_end) for all virtual ranks (see include/cpattn.h)."""
    lib = load_library()
    dev = [None]
    ptrs = _ring_args(desc, q, k, v, o, m, l, "cp_ring_step_partial_attn", dev=dev)
    st = lib.cp_ring_step_partial_attn(ctypes.byref(desc), int(step_begin), int(step_end), *ptrs, int(mode),
                                       _stream(stream, dev))
    _check(st, "cp_ring_step_partial_attn")


def cp_ring_rank_partial_attn(desc: AttnDesc, layout: int, rank_begin: int, rank_end: int, step_begin: int,
                              step_end: int, q, k, v, o, m, l, mode: int = CP_MODE_EMIT, stream=None) -> None:
    """Ring steps [step_begin, step_end) for the virtual ranks [rank_begin, rank_end) under a layout."""
    lib = load_library()
    st = lib.cp_ring_rank_partial_attn(ctypes.byref(desc), int(layout), int(rank_begin), int(rank_end),
                                       int(step_begin), int(step_end),
                                       *_ring_args(desc, q, k, v, o, m, l, "cp_ring_rank_partial_attn"), int(mode),
                                       _stream(stream))
    _check(st, "cp_ring_rank_partial_attn")


def cp_ring_attn_host_workspace_bytes(desc: AttnDesc) -> int:
    """Bytes of device workspace cp_ring_attn_host needs for ``desc``."""
    n = ctypes.c_size_t(0)
    _check(load_library().cp_ring_attn_host_workspace_bytes(ctypes.byref(desc), ctypes.byref(n)),
           "cp_ring_attn_host_workspace_bytes")
    return int(n.value)


def cp_ring_attn_host(desc: AttnDesc, q_host, k_host, v_host, o_host, m_host, l_host, workspace,
                      workspace_bytes: int, stream=None) -> None:
    """The full balanced ring (EMIT | FINALIZE) on host tensors, copies overlapped with compute.

    The host tensors are CPU tensors (pinned for overlap); ``workspace`` is a device buffer of at
    least cp_ring_attn_host_workspace_bytes(desc) bytes.  Asynchronous on ``stream``.
    """
    lib = load_library()
    where = "cp_ring_attn_host"
    ptrs = _ring_args(desc, q_host, k_host, v_host, o_host, m_host, l_host, where, cuda=False)
    ws = _arg(workspace, "workspace", where, nbytes=int(workspace_bytes))
    st = lib.cp_ring_attn_host(ctypes.byref(desc), *ptrs, ws, int(workspace_bytes), _stream(stream))
    _check(st, "cp_ring_attn_host")


def cp_merge_partials(batch, rows, heads, d, n_parts, o_parts, m_parts, l_parts, o_out, m_out, l_out,
                      order=None, finalize=False, stream=None) -> None:
    """LSE merge of n_parts triples in ``order`` (a host sequence, or None for index order)."""
    lib = load_library()
    order_arr = None
    order_ptr = None
    if order is not None:
        order_arr = np.ascontiguousarray(np.asarray(order, dtype=np.int32))
        if order_arr.size != int(n_parts):
            raise CpError(CP_ERR_INVALID_ARGUMENT, "cp_merge_partials")
        order_ptr = order_arr.ctypes.data
    po, pm, pl, oo, om, ol = _merge_args(batch, rows, heads, d, n_parts, o_parts, m_parts, l_parts, o_out, m_out,
                                         l_out, "cp_merge_partials")
    st = lib.cp_merge_partials(int(batch), int(rows), int(heads), int(d), int(n_parts), po, pm, pl, order_ptr, oo, om,
                               ol, int(bool(finalize)), _stream(stream))
    _check(st, "cp_merge_partials")


def cp_merge_tree_workspace_bytes(batch, rows, heads, d, n_parts) -> int:
    lib = load_library()
    n = ctypes.c_size_t(0)
    _check(lib.cp_merge_tree_workspace_bytes(int(batch), int(rows), int(heads), int(d), int(n_parts),
                                             ctypes.byref(n)), "cp_merge_tree_workspace_bytes")
    return int(n.value)


def cp_merge_partials_tree(batch, rows, heads, d, n_parts, o_parts, m_parts, l_parts, workspace, workspace_bytes,
                           o_out, m_out, l_out, finalize=False, stream=None) -> None:
    """Log-depth tree reduction of n_parts (a power of two) triples; part i merges with part i + n/2."""
    lib = load_library()
    where = "cp_merge_partials_tree"
    po, pm, pl, oo, om, ol = _merge_args(batch, rows, heads, d, n_parts, o_parts, m_parts, l_parts, o_out, m_out,
                                         l_out, where)
    ws = _arg(workspace, "workspace", where, nbytes=int(workspace_bytes))
    st = lib.cp_merge_partials_tree(int(batch), int(rows), int(heads), int(d), int(n_parts), po, pm, pl, ws,
                                    int(workspace_bytes), oo, om, ol, int(bool(finalize)), _stream(stream))
    _check(st, "cp_merge_partials_tree")


def cp_passq_workspace_bytes(desc: AttnDesc) -> int:
    lib = load_library()
    n = ctypes.c_size_t(0)
    _check(lib.cp_passq_workspace_bytes(ctypes.byref(desc), ctypes.byref(n)), "cp_passq_workspace_bytes")
    return int(n.value)


def cp_passq_decode(desc: AttnDesc, q, k, v, workspace, workspace_bytes: int, out, m_out=None, l_out=None,
                    stream=None) -> None:
    """Pass-Q decode: partials over cp shards, then the LSE reduce into ``out``."""
    lib = load_library()
    pq, pk, pv, po, pm, pl = _decode_args(desc, q, k, v, out, m_out, l_out, "cp_passq_decode")
    ws = _arg(workspace, "workspace", "cp_passq_decode", nbytes=int(workspace_bytes))
    st = lib.cp_passq_decode(ctypes.byref(desc), pq, pk, pv, ws, int(workspace_bytes), po, pm, pl, _stream(stream))
    _check(st, "cp_passq_decode")


def cp_passq_decode_noalloc(desc: AttnDesc, q, k, v, out, m_out=None, l_out=None, stream=None) -> None:
    """Pass-Q decode without a workspace, for callers that cannot allocate device memory.

    The partials go to the library's fixed scratch of CP_PASSQ_NOALLOC_SCRATCH_BYTES
    (8 MiB per GPU, held until exit).  Calls share that scratch: do not let two of
    them overlap on the GPU.  A problem too large for it raises CpError with
    CP_ERR_UNSUPPORTED before anything is launched.
    """
    lib = load_library()
    st = lib.cp_passq_decode_noalloc(ctypes.byref(desc),
                                     *_decode_args(desc, q, k, v, out, m_out, l_out, "cp_passq_decode_noalloc"),
                                     _stream(stream))
    if st == CP_ERR_UNSUPPORTED:
        raise CpError(st, "cp_passq_decode_noalloc (unsupported shape, or partials larger than the "
                          f"{CP_PASSQ_NOALLOC_SCRATCH_BYTES >> 20} MiB fixed scratch)")
    _check(st, "cp_passq_decode_noalloc")


def cp_set_kernel_choice(knob: int, value: int) -> None:
    """Process-wide kernel choice for tests and diagnostics (-1 = automatic); every choice
    computes the same bits."""
    _check(load_library().cp_set_kernel_choice(int(knob), int(value)), "cp_set_kernel_choice")


def cp_selftest_wait_timeout(stream=None) -> None:
    """Launch the bounded-wait self-test (records CP_ERR_TIMEOUT after about a second)."""
    _check(load_library().cp_selftest_wait_timeout(_stream(stream)), "cp_selftest_wait_timeout")


def cp_take_device_status(stream=None) -> int:
    """Synchronise the stream; return and clear the device status word."""
    lib = load_library()
    s = _I32(0)
    _check(lib.cp_take_device_status(_stream(stream), ctypes.byref(s)), "cp_take_device_status")
    return int(s.value)
