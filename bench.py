"""Benchmark of the ring-step prefill (and pass-Q decode / merge) on one node.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one pass of the hot path over the GQA prefill workload (b1,
32 q / 8 kv heads, d128, S32768, cp8): the host chunk plan, the ring-step
attention of all cp virtual ranks over all cp steps in one launch (the
between-step merge fused, output finalised), and the closed-form byte counts.
Inputs (402 MB of bf16 Q/K/V) exceed the 129 MB L2, so no flush is needed.

Rank 0 prints one JSON line.  ``value`` is prefill TFLOP/s over all ranks
(algorithmic FLOPs 4*b*h_q*d*S(S+1)/2 per step).  Under torchrun every rank runs
an independent replica (weak scaling, no collective on the data path).
The line also carries the dominant kernel's roofline, an end-to-end number
through the C-ABI with host buffers, the CPU oracle baseline, SM clocks sampled
during the timed region, and secondary lines for pass-Q decode (GB/s) and the
LSE merge (GB/s).

``--impl reference`` times the CPU oracle (fp64, test infrastructure) on a
bounded row sample of the same workload on the host cores.  The headline line and
the tiny, long, decode and merge secondary lines each carry the oracle timed on the
same inputs (the whole tiny workload; bounded samples of the others, with the
full-workload time extrapolated from them) on a spawn pool of one single-threaded
worker per host core (unless --skip-cpu).
"""

from __future__ import annotations

import os

if os.environ.get("CPATTN_ORACLE_WORKER") == "1":
    # spawned oracle workers: one BLAS thread each, so `cores` is the pool size
    for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[_v] = "1"

import argparse
import json
import math
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
WORKLOAD = "gqa"
# Seeded random rows per head in the long workload's cpu_baseline sample (one head per kv
# head): about 10 s of fp64 work on 16 cores.
LONG_BASELINE_ROWS = 1536
METRIC = "ring-step prefill TFLOP/s (% bf16 peak); pass-Q decode GB/s (% HBM peak)"


# ---------------------------------------------------------------------------
# workload arithmetic (algorithmic work, not what the kernels happen to move)
# ---------------------------------------------------------------------------

def prefill_flops(w):
    pairs = w["S"] * (w["S"] + 1) // 2
    return 4 * w["b"] * w["h_q"] * w["d"] * pairs


def decode_bytes(w):
    b, L, hq, hkv, d, cp = w["b"], w["S"], w["h_q"], w["h_kv"], w["d"], w["cp"]
    kv = 2 * b * L * hkv * d * 2
    q = b * hq * d * 2
    partials = 2 * cp * b * hq * (d + 2) * 4  # written once, read once by the reduce
    out = b * hq * d * 4
    return kv + q + partials + out


def merge_bytes(w):
    n, h, r, d = w["parts"], w["heads"], w["rows"], w["d"]
    return n * h * r * (d + 2) * 4 + h * r * (d + 2) * 4


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the
# ring kernel on this workload, from the ncu capture of that kernel.  It is reported
# only while ring_attn.cu is the source that was captured (sha256 prefix below);
# otherwise traffic is null.
RING_TRAFFIC = {"sha256_prefix": "00629399275168dc", "bytes": 891984640}


def headline_config(world):
    """The headline workload's config, the same object on both arms of the benchmark."""
    from context_ring_attention_cp_gb300 import synth
    w = synth.WORKLOADS[WORKLOAD]
    return {"workload": "prefill ring attention, GQA: b1, 32 q / 8 kv heads, d128, S32768, cp8",
            "b": w["b"], "S": w["S"], "h_q": w["h_q"], "h_kv": w["h_kv"], "d": w["d"], "cp": w["cp"],
            "l2": "inputs (402 MB) larger than L2; no flush",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def ring_traffic():
    import hashlib
    path = os.path.join(ROOT, "context_ring_attention_cp_gb300", "csrc", "ring_attn.cu")
    with open(path, "rb") as f:
        digest = hashlib.sha256(f.read()).hexdigest()
    return RING_TRAFFIC["bytes"] if digest.startswith(RING_TRAFFIC["sha256_prefix"]) else None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.15)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.strip() for r in self.file.read().splitlines() if r.strip()]
        self.file.close()
        os.unlink(self.file.name)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle (test infrastructure) on bounded samples, on all of the host's cores
# ---------------------------------------------------------------------------

def _oracle_warm(_):
    sys.path.insert(0, ROOT)
    import oracle  # noqa: F401
    return 0


def _load(path):
    return np.load(path, mmap_mode="r")


def _oracle_prefill_rows_task(args):
    """One task: causal attention of some sampled rows of one query head (fp64 oracle).
    The inputs are bf16 bit files: the sampled Q rows [R, h_q, d] and K, V [S, h_kv, d]."""
    qpath, kpath, vpath, h, kh, rows, sel, scale = args
    sys.path.insert(0, ROOT)
    import oracle
    from oracle import attention as OA
    t0 = time.perf_counter()
    k = oracle.bf16_bits_to_f64(np.ascontiguousarray(_load(kpath)[:, kh, :]))
    v = oracle.bf16_bits_to_f64(np.ascontiguousarray(_load(vpath)[:, kh, :]))
    S, d = k.shape
    qfull = np.zeros((1, S, 1, d))
    qfull[0, rows, 0] = oracle.bf16_bits_to_f64(np.ascontiguousarray(_load(qpath)[sel, h, :]))
    OA.causal_attention_rows(qfull, k[None, :, None], v[None, :, None], scale, 0, [0], rows)
    return sum(4 * d * (i + 1) for i in rows), len(rows), time.perf_counter() - t0


def _oracle_decode_shard_task(args):
    """One task: the pass-Q partial triple of one (sequence, head) over one KV shard (fp64
    oracle).  The inputs are bf16 bit files: q [d], and the shard's K, V rows [n, d]."""
    qpath, kpath, vpath, scale = args
    sys.path.insert(0, ROOT)
    import oracle
    from oracle import attention as OA
    t0 = time.perf_counter()
    q = oracle.bf16_bits_to_f64(np.ascontiguousarray(_load(qpath)))
    k = oracle.bf16_bits_to_f64(np.ascontiguousarray(_load(kpath)))
    v = oracle.bf16_bits_to_f64(np.ascontiguousarray(_load(vpath)))
    OA.decode_shard_triples(q[None, None], k[None, :, None], v[None, :, None], scale, 1)
    return 2 * k.size * 2, 1, time.perf_counter() - t0  # the bf16 K and V bytes this shard reads


def _oracle_merge_task(args):
    """One task: the fold of n parts over a block of rows of one head (fp64 oracle).
    The inputs are fp32 files: m, l [n, R] and O [n, R, d] of that head."""
    mpath, lpath, opath, r0, r1 = args
    sys.path.insert(0, ROOT)
    from oracle import ring as OR
    t0 = time.perf_counter()
    m, l, o = _load(mpath), _load(lpath), _load(opath)
    n, _, d = o.shape
    parts = [(np.asarray(m[p, r0:r1], np.float64), np.asarray(l[p, r0:r1], np.float64),
              np.asarray(o[p, r0:r1], np.float64)) for p in range(n)]
    OR.merge_in_order(parts)
    return (n + 1) * (r1 - r0) * (d + 2) * 4, r1 - r0, time.perf_counter() - t0  # fp32 parts read + triple written


class OraclePool:
    """A spawn pool of single-threaded oracle workers, one per host core, created once and
    shared by every CPU leg.  Inputs reach the workers as memory-mapped .npy files in a
    temporary directory (removed on close), so nothing large is pickled."""

    def __init__(self, workers):
        import multiprocessing as mp
        self.workers = int(workers)
        self.dir = tempfile.TemporaryDirectory(prefix="cpattn_oracle_")
        self._n = 0
        os.environ["CPATTN_ORACLE_WORKER"] = "1"
        try:
            self.pool = mp.get_context("spawn").Pool(self.workers)
        finally:
            os.environ.pop("CPATTN_ORACLE_WORKER", None)
        self.pool.map(_oracle_warm, range(self.workers))  # imports happen before any timing

    def save(self, arr):
        self._n += 1
        path = os.path.join(self.dir.name, f"a{self._n}.npy")
        np.save(path, np.ascontiguousarray(arr))
        return path

    def run(self, fn, tasks):
        """All tasks at once over the pool: (total work, total rows or units, wall seconds)."""
        t0 = time.perf_counter()
        res = self.pool.map(fn, tasks, chunksize=1)
        wall = time.perf_counter() - t0
        return sum(r[0] for r in res), sum(r[1] for r in res), wall

    def close(self):
        self.pool.close()
        self.pool.join()
        self.dir.cleanup()

    def describe(self):
        return {"cores": self.workers, "host_cpus": os.cpu_count()}


def oracle_prefill_leg(pool, w, q, k, v, heads, n_random, seed, full_rows=False, run=True):
    """The oracle on sampled rows (or every row) of a prefill workload; b = 1.

    Sample (per head in ``heads``): the first and last row of each of the 2cp chunks, rows 0
    and S-1, and ``n_random`` seeded random rows; ``full_rows`` takes every row instead.
    Returns the cpu_baseline object: fp64 TFLOP/s, rows/s and the full-config time.  With
    ``run=False`` the inputs are written out now and a callable that runs the oracle and
    returns that object is returned instead."""
    from context_ring_attention_cp_gb300 import synth
    S, d, g = w["S"], w["d"], w["h_q"] // w["h_kv"]
    rows = list(range(S)) if full_rows else synth.sample_rows(S, w["cp"], n_random, seed)
    qpath = pool.save(synth.bf16_bits(q[0, rows]))
    kpath = pool.save(synth.bf16_bits(k[0]))
    vpath = pool.save(synth.bf16_bits(v[0]))
    # split each head's rows so that every worker gets work of about the same size
    per_head = max(1, (2 * pool.workers + len(heads) - 1) // len(heads))
    tasks = []
    for h in heads:
        for part in range(per_head):
            sel = list(range(part, len(rows), per_head))
            if sel:
                tasks.append((qpath, kpath, vpath, h, h // g, [rows[i] for i in sel], sel, 1.0 / math.sqrt(d)))
    job = lambda: _prefill_leg_result(pool, w, heads, rows, n_random, full_rows, tasks,  # noqa: E731
                                      *pool.run(_oracle_prefill_rows_task, tasks))
    return job() if run else job


def _prefill_leg_result(pool, w, heads, rows, n_random, full_rows, tasks, flops, nrows, wall):
    S = w["S"]
    rate = flops / wall
    full_flops = prefill_flops(w)
    out = {"value": round(rate / 1e12, 6), "unit": "TFLOP/s", "kind": "oracle", **pool.describe(),
           "rows_per_s": round(nrows / wall, 1), "seconds": round(wall, 3)}
    if full_rows and len(heads) == w["h_q"]:
        out["full_config_s"] = {"value": round(wall, 3), "how": "measured (every row of every head)"}
        out["sample"] = (f"the whole workload: {len(heads)} heads x {S} causal rows (fp64 numpy), "
                         f"{len(tasks)} tasks on {pool.workers} single-threaded spawn workers")
    else:
        out["full_config_s"] = {"value": round(full_flops / rate, 1),
                                "how": "extrapolated: the workload's FLOPs / the sample's fp64 FLOP rate"}
        out["sample"] = (f"{len(heads)} heads x {len(rows)} rows (first and last row of each chunk, rows 0 and "
                         f"S-1, {n_random} seeded random rows; causal, fp64 numpy), {len(tasks)} tasks on "
                         f"{pool.workers} single-threaded spawn workers")
    return out


def oracle_decode_leg(pool, w, q, k, v, pairs, run=True):
    """The oracle's pass-Q shard triples for the sampled (sequence, head) pairs, every shard
    of each pair a task; GB/s of bf16 K/V read, and the full-config time extrapolated.
    ``run=False``: as for the prefill leg."""
    from context_ring_attention_cp_gb300 import synth
    L, cp, d, g = w["S"], w["cp"], w["d"], w["h_q"] // w["h_kv"]
    n = L // cp
    tasks = []
    for bi, h in pairs:
        qpath = pool.save(synth.bf16_bits(q[bi, h]))
        for s in range(cp):
            kpath = pool.save(synth.bf16_bits(k[bi, s * n:(s + 1) * n, h // g]))
            vpath = pool.save(synth.bf16_bits(v[bi, s * n:(s + 1) * n, h // g]))
            tasks.append((qpath, kpath, vpath, 1.0 / math.sqrt(d)))
    job = lambda: _decode_leg_result(pool, w, pairs, tasks, *pool.run(_oracle_decode_shard_task, tasks))  # noqa
    return job() if run else job


def _decode_leg_result(pool, w, pairs, tasks, nbytes, _, wall):
    L, cp, d = w["S"], w["cp"], w["d"]
    n = L // cp
    rate = nbytes / wall
    full = 2 * w["b"] * L * w["h_q"] * d * 2
    return {"value": round(rate / 1e9, 4), "unit": "GB/s", "kind": "oracle", **pool.describe(),
            "seconds": round(wall, 3),
            "full_config_s": {"value": round(full / rate, 2),
                              "how": "extrapolated: all (sequence, head) pairs' K/V bytes / the sample's rate"},
            "sample": f"{len(pairs)} (sequence, head) pairs x {cp} shards of {n} keys (fp64 numpy shard triples), "
                      f"{len(tasks)} tasks on {pool.workers} single-threaded spawn workers"}


def oracle_merge_leg(pool, w, po, pm, pl, heads, run=True):
    """The oracle's left fold over all parts for every row of the sampled heads, in row
    blocks; GB/s of fp32 triples read and written, and the full-config time extrapolated.
    ``run=False``: as for the prefill leg."""
    R = w["rows"]
    blocks = max(1, (2 * pool.workers + len(heads) - 1) // len(heads))
    step = (R + blocks - 1) // blocks
    tasks = []
    for h in heads:
        mpath = pool.save(pm[:, 0, h, :].cpu().numpy())
        lpath = pool.save(pl[:, 0, h, :].cpu().numpy())
        opath = pool.save(po[:, 0, :, h].cpu().numpy())
        tasks += [(mpath, lpath, opath, r0, min(R, r0 + step)) for r0 in range(0, R, step)]
    job = lambda: _merge_leg_result(pool, w, heads, tasks, *pool.run(_oracle_merge_task, tasks))  # noqa: E731
    return job() if run else job


def _merge_leg_result(pool, w, heads, tasks, nbytes, _, wall):
    R = w["rows"]
    rate = nbytes / wall
    return {"value": round(rate / 1e9, 4), "unit": "GB/s", "kind": "oracle", **pool.describe(),
            "seconds": round(wall, 3),
            "full_config_s": {"value": round(merge_bytes(w) / rate, 2),
                              "how": "extrapolated: the workload's bytes / the sample's rate"},
            "sample": f"{len(heads)} heads x {R} rows x {w['parts']} parts (fp64 numpy fold), {len(tasks)} tasks on "
                      f"{pool.workers} single-threaded spawn workers"}


# ---------------------------------------------------------------------------
# GPU arms
# ---------------------------------------------------------------------------

def max_over_ranks(x: float, dist) -> float:
    """The largest value of ``x`` over all ranks (the slowest rank's time)."""
    if dist is None:
        return float(x)
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank_step: int, world: int, steps: int, total_ms: float) -> float:
    """Aggregate throughput: the work of every rank over the slowest rank's time."""
    return flops_per_rank_step * world * steps / (total_ms * 1e-3) / 1e12


def _events_time(fn, iters, stream):
    import torch
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(iters):
        fn()
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / iters


def bench_ours(args, rank, world, dist):
    import torch

    import context_ring_attention_cp_gb300 as cpa
    from context_ring_attention_cp_gb300 import _build, synth

    # the oracle's worker pool (spawned, one single-threaded worker per host core) is made
    # before the first GPU call and shared by every CPU leg
    pool = OraclePool(args.cpu_workers) if (rank == 0 and not args.skip_cpu) else None
    if rank == 0 or world == 1:
        _build.build()
    if dist is not None:
        dist.barrier()
    cpa.load_library()
    dev = torch.cuda.current_device()
    stream = torch.cuda.current_stream()
    peaks = load_peaks()
    w = synth.WORKLOADS[WORKLOAD]
    b, S, hq, hkv, d, cp = w["b"], w["S"], w["h_q"], w["h_kv"], w["d"], w["cp"]
    q, k, v = synth.prefill_inputs(b, S, hq, hkv, d, std=w["std"], seed=w["seed"] + rank)
    o = torch.empty((b, S, hq, d), dtype=torch.float32, device="cuda")
    m = torch.empty((b, hq, S), dtype=torch.float32, device="cuda")
    l = torch.empty((b, hq, S), dtype=torch.float32, device="cuda")
    desc = cpa.make_desc(b, S, hq, hkv, d, cp, 1.0 / math.sqrt(d), 1)
    mode = cpa.CP_MODE_EMIT | cpa.CP_MODE_FINALIZE
    c_kv = 2 * hkv * d * 2
    flops = prefill_flops(w)
    kernel_ms = []
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * args.steps)]

    def step(i=None):
        plan = cpa.cp_plan_balanced_chunks(S, cp)              # a1: chunk plan (host)
        if i is not None:
            ev[2 * i].record(stream)
        cpa.cp_ring_step_partial_attn(desc, 0, cp, q, k, v, o, m, l, mode, stream)  # a2-a4 (one launch)
        if i is not None:
            ev[2 * i + 1].record(stream)
        cpa.cp_comm_bytes(S, cp, c_kv)                         # a6: byte accounting (host)
        return plan

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if cpa.cp_take_device_status() != 0:
        raise RuntimeError("device status error during warm-up")
    sampler = ClockSampler(dev)
    sampler.start()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        step(i)
    t_end.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clocks = sampler.stop()
    total_ms = t_start.elapsed_time(t_end)
    kernel_ms = [ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(args.steps)]
    if cpa.cp_take_device_status() != 0:
        raise RuntimeError("device status error in the timed region")
    total_ms = max_over_ranks(total_ms, dist)
    ms_per_step = total_ms / args.steps
    value = whole_job_tflops(flops, world, args.steps, total_ms)

    kern_ms = statistics.mean(kernel_ms)
    achieved = flops / (kern_ms * 1e-3) / 1e12
    # The step is this one kernel, timed alone in a sub-second loop (the clocks record
    # shows whether the power cap engaged): the burst GEMM peak is the denominator,
    # the sustained one is reported beside it.
    peak = peaks["bf16_tflops"]
    roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "traffic": ring_traffic(),
                "algorithmic_bytes": int(q.numel() * 2 + k.numel() * 2 + v.numel() * 2 + (o.numel() + 2 * m.numel()) * 4),
                "kernel": "ring_attn_kernel<128, balanced>", "kernel_ms": round(kern_ms, 4),
                "peak_kind": f"bf16 burst ({peaks['source']})",
                "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4)}

    # ---- end to end through the C-ABI with host buffers (pinned), copies inside the timed region
    e2e = None
    if not args.skip_e2e:
        # The host-buffer entry point: Q, K, V in pinned host memory, O, m, l back into
        # pinned host memory, copies overlapped with the ring launches inside the call.
        hq_, hk_, hv_ = (x.cpu().pin_memory() for x in (q, k, v))
        ho = torch.empty(o.shape, dtype=torch.float32).pin_memory()
        hm = torch.empty(m.shape, dtype=torch.float32).pin_memory()
        hl = torch.empty(l.shape, dtype=torch.float32).pin_memory()
        ws_bytes = cpa.cp_ring_attn_host_workspace_bytes(desc)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")

        def e2e_step():
            cpa.cp_plan_balanced_chunks(S, cp)
            cpa.cp_ring_attn_host(desc, hq_, hk_, hv_, ho, hm, hl, ws, ws_bytes, stream)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        n_e2e = max(3, min(args.steps, 20))
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            e2e_step()
        torch.cuda.synchronize()
        e2e_ms = (time.perf_counter() - t0) * 1e3 / n_e2e
        e2e = {"value": round(flops * world / (e2e_ms * 1e-3) / 1e12, 1), "unit": "TFLOP/s",
               "ms_per_step": round(e2e_ms, 3), "api": "cp_ring_attn_host (pinned host buffers)",
               "h2d_bytes_per_step": int(q.numel() * 2 + k.numel() * 2 + v.numel() * 2),
               "d2h_bytes_per_step": int((o.numel() + m.numel() + l.numel()) * 4)}
        del hq_, hk_, hv_, ho, hm, hl, ws

    secondary = {}
    if not args.skip_secondary and rank == 0:
        secondary = secondary_lines(cpa, synth, peaks, stream, pool=pool)

    cpu = None
    if pool is not None:
        # every head x the sampled rows of this workload (the inputs timed above)
        cpu = oracle_prefill_leg(pool, w, q, k, v, list(range(hq)), args.cpu_baseline_rows, seed=w["seed"])
        pool.close()

    line = {"metric": METRIC, "value": round(value, 1), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1)*0.5 bf16 Q/K/V)",
            "config": headline_config(world),
            "step": "plan + one ring launch over all cp steps (merge fused, finalised) + byte counts",
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": args.steps,
            "clocks": clocks, "secondary": secondary}
    return line


def secondary_lines(cpa, synth, peaks, stream, pool=None):
    import torch
    out = {}
    # The oracle legs' inputs are written out beside each GPU line, but the legs run after
    # the last GPU line: right after the long workload's leg (about 8 s on every host core)
    # the next two GPU lines measured 5-6 % lower than in a run without it.
    cpu_jobs = []
    # one ring step (t = 1) of all cp virtual ranks on the GQA workload, EMIT: the spec's
    # per-step unit of work, cp * 2C^2 visible pairs per head (F_attn / cp per step in all)
    w = synth.WORKLOADS[WORKLOAD]
    q, k, v = synth.prefill_inputs(w["b"], w["S"], w["h_q"], w["h_kv"], w["d"], std=w["std"], seed=w["seed"])
    o = torch.empty((w["b"], w["S"], w["h_q"], w["d"]), dtype=torch.float32, device="cuda")
    m = torch.empty((w["b"], w["h_q"], w["S"]), dtype=torch.float32, device="cuda")
    l = torch.empty_like(m)
    desc = cpa.make_desc(w["b"], w["S"], w["h_q"], w["h_kv"], w["d"], w["cp"], 1.0 / math.sqrt(w["d"]), 1)
    ovl = cpa.CP_MODE_OVERLAP_PREVIOUS
    C = w["S"] // (2 * w["cp"])
    step_flops = 4 * w["b"] * w["h_q"] * w["d"] * w["cp"] * 2 * C * C

    def one_step(mode):
        # the step launched 20 times in a row; and the same with every launch a programmatic
        # dependent of the one before (CP_MODE_OVERLAP_PREVIOUS), as a rank's stream of steps
        fn = lambda: cpa.cp_ring_step_partial_attn(desc, 1, 2, q, k, v, o, m, l, mode, stream)  # noqa
        fo = lambda: cpa.cp_ring_step_partial_attn(desc, 1, 2, q, k, v, o, m, l, mode | ovl, stream)  # noqa
        for _ in range(3):
            fn()
            fo()
        ms = _events_time(fn, 20, stream)
        ms_o = _events_time(fo, 20, stream)
        return ms, {"ms": round(ms_o, 4), "value": round(step_flops / (ms_o * 1e-3) / 1e12, 1)}

    ms, overlapped = one_step(cpa.CP_MODE_EMIT)
    tf = step_flops / (ms * 1e-3) / 1e12
    out["prefill_one_step_emit"] = {
        "workload": "one ring step (t=1, all 8 virtual ranks, EMIT) of the GQA prefill workload",
        "value": round(tf, 1), "unit": "TFLOP/s", "ms": round(ms, 4), "flops": step_flops,
        "peak": peaks["bf16_tflops"], "frac": round(tf / peaks["bf16_tflops"], 4), "overlapped": overlapped}
    # the same step merged into a running triple (what every step after the first does
    # when each rank launches per step): O, m and l are read as well as written
    cpa.cp_ring_step_partial_attn(desc, 0, 1, q, k, v, o, m, l, cpa.CP_MODE_EMIT, stream)
    ms, overlapped = one_step(cpa.CP_MODE_ACCUMULATE)
    tf = step_flops / (ms * 1e-3) / 1e12
    out["prefill_one_step_accumulate"] = {
        "workload": "one ring step (t=1, all 8 virtual ranks, ACCUMULATE into the step-0 triple) "
                    "of the GQA prefill workload",
        "value": round(tf, 1), "unit": "TFLOP/s", "ms": round(ms, 4), "flops": step_flops,
        "peak": peaks["bf16_tflops"], "frac": round(tf / peaks["bf16_tflops"], 4), "overlapped": overlapped}
    # the whole ring as cp launches of one step each (the first EMIT, then ACCUMULATE, the
    # last normalising), as the steps run when each rank launches per step; each launch a
    # programmatic dependent of the one before (its CTAs start in the previous launch's
    # tail), and for comparison the same launches fully serialised
    def chain(extra):
        for t in range(w["cp"]):
            md = cpa.CP_MODE_EMIT if t == 0 else cpa.CP_MODE_ACCUMULATE
            if t == w["cp"] - 1:
                md |= cpa.CP_MODE_FINALIZE
            cpa.cp_ring_step_partial_attn(desc, t, t + 1, q, k, v, o, m, l, md | extra, stream)
    ovl = cpa.CP_MODE_OVERLAP_PREVIOUS
    for _ in range(3):
        chain(ovl)
        chain(0)
    ms_serial = _events_time(lambda: chain(0), 10, stream)
    ms = _events_time(lambda: chain(ovl), 10, stream)
    tf = prefill_flops(w) / (ms * 1e-3) / 1e12
    out["prefill_per_step_chain"] = {
        "workload": "the GQA prefill ring as 8 single-step launches (EMIT, ACCUMULATE..., the last "
                    "FINALIZE) instead of one fused launch, each overlapping the previous one's tail "
                    "(CP_MODE_OVERLAP_PREVIOUS)",
        "value": round(tf, 1), "unit": "TFLOP/s", "ms": round(ms, 4), "flops": prefill_flops(w),
        "launches": w["cp"], "peak": peaks["bf16_tflops"], "frac": round(tf / peaks["bf16_tflops"], 4),
        "serialised": {"ms": round(ms_serial, 4),
                       "value": round(prefill_flops(w) / (ms_serial * 1e-3) / 1e12, 1)}}
    del q, k, v, o, m, l
    torch.cuda.empty_cache()
    # per-virtual-rank work under the balanced (method) and sequential (plain) layouts:
    # one launch per rank covering all its ring steps
    w = synth.WORKLOADS[WORKLOAD]
    q, k, v = synth.prefill_inputs(w["b"], w["S"], w["h_q"], w["h_kv"], w["d"], std=w["std"], seed=w["seed"])
    o = torch.empty((w["b"], w["S"], w["h_q"], w["d"]), dtype=torch.float32, device="cuda")
    m = torch.empty((w["b"], w["h_q"], w["S"]), dtype=torch.float32, device="cuda")
    l = torch.empty_like(m)
    desc = cpa.make_desc(w["b"], w["S"], w["h_q"], w["h_kv"], w["d"], w["cp"], 1.0 / math.sqrt(w["d"]), 1)
    balance = {}
    for name, layout in (("balanced", cpa.CP_LAYOUT_BALANCED), ("sequential", cpa.CP_LAYOUT_SEQUENTIAL)):
        pairs = cpa.cp_plan_chunks(w["S"], w["cp"], layout)["step_pairs"].sum(axis=1)
        times = []
        for r in range(w["cp"]):
            fn = lambda: cpa.cp_ring_rank_partial_attn(desc, layout, r, r + 1, 0, w["cp"], q, k, v, o, m, l,  # noqa
                                                       cpa.CP_MODE_EMIT | cpa.CP_MODE_FINALIZE, stream)
            fn()
            times.append(_events_time(fn, 3, stream))
        balance[name] = {"rank_ms": [round(x, 4) for x in times],
                         "max_over_min_ms": round(max(times) / min(times), 3),
                         "rank_pairs_per_head": [int(x) for x in pairs],
                         "max_over_min_pairs": round(float(pairs.max() / pairs.min()), 3)}
    out["rank_balance"] = {"workload": "GQA prefill, one launch per virtual rank (all its ring steps)", **balance}
    del q, k, v, o, m, l
    torch.cuda.empty_cache()
    # long prefill: b1, 32/8 heads, d128, S131072, cp16 (one fused ring launch, 140.7 TFLOP)
    w = synth.WORKLOADS["long"]
    q, k, v = synth.prefill_inputs(w["b"], w["S"], w["h_q"], w["h_kv"], w["d"], std=w["std"], seed=w["seed"])
    o = torch.empty((w["b"], w["S"], w["h_q"], w["d"]), dtype=torch.float32, device="cuda")
    m = torch.empty((w["b"], w["h_q"], w["S"]), dtype=torch.float32, device="cuda")
    l = torch.empty_like(m)
    desc = cpa.make_desc(w["b"], w["S"], w["h_q"], w["h_kv"], w["d"], w["cp"], 1.0 / math.sqrt(w["d"]), 1)
    mode = cpa.CP_MODE_EMIT | cpa.CP_MODE_FINALIZE
    fn = lambda: cpa.cp_ring_step_partial_attn(desc, 0, w["cp"], q, k, v, o, m, l, mode, stream)  # noqa: E731
    fn()
    ms = _events_time(fn, 3, stream)
    tf = prefill_flops(w) / (ms * 1e-3) / 1e12
    out["prefill_long"] = {"workload": "prefill ring attention, long: b1, 32/8 heads, d128, S131072, cp16",
                           "value": round(tf, 1), "unit": "TFLOP/s", "ms": round(ms, 3), "flops": prefill_flops(w),
                           "peak": peaks["bf16_tflops"], "frac": round(tf / peaks["bf16_tflops"], 4)}
    if pool is not None:  # one query head per kv head x the sampled rows
        g = w["h_q"] // w["h_kv"]
        cpu_jobs.append(("prefill_long", oracle_prefill_leg(pool, w, q, k, v, list(range(0, w["h_q"], g)),
                                                            LONG_BASELINE_ROWS, seed=w["seed"], run=False)))
    del q, k, v, o, m, l
    torch.cuda.empty_cache()
    # multi-head prefill: b1, 32/32 heads, d128, S32768, cp8 (the GQA workload's FLOPs with
    # four times its K/V); a CTA pairs two row tiles of one head
    w = synth.WORKLOADS["mha"]
    q, k, v = synth.prefill_inputs(w["b"], w["S"], w["h_q"], w["h_kv"], w["d"], std=w["std"], seed=w["seed"])
    o = torch.empty((w["b"], w["S"], w["h_q"], w["d"]), dtype=torch.float32, device="cuda")
    m = torch.empty((w["b"], w["h_q"], w["S"]), dtype=torch.float32, device="cuda")
    l = torch.empty_like(m)
    desc = cpa.make_desc(w["b"], w["S"], w["h_q"], w["h_kv"], w["d"], w["cp"], 1.0 / math.sqrt(w["d"]), 1)
    fn = lambda: cpa.cp_ring_step_partial_attn(desc, 0, w["cp"], q, k, v, o, m, l, mode, stream)  # noqa: E731
    for _ in range(2):
        fn()
    ms = _events_time(fn, 5, stream)
    tf = prefill_flops(w) / (ms * 1e-3) / 1e12
    out["prefill_mha"] = {"workload": "prefill ring attention, multi-head: b1, 32/32 heads, d128, S32768, cp8",
                          "value": round(tf, 1), "unit": "TFLOP/s", "ms": round(ms, 3), "flops": prefill_flops(w),
                          "peak": peaks["bf16_tflops"], "frac": round(tf / peaks["bf16_tflops"], 4)}
    del q, k, v, o, m, l
    torch.cuda.empty_cache()
    # head dimension 64 at scale: b1, 16/16 heads, d64, S32768, cp8 (half the MMA cycles of
    # d128 for the same softmax work)
    w = synth.WORKLOADS["mha64"]
    q, k, v = synth.prefill_inputs(w["b"], w["S"], w["h_q"], w["h_kv"], w["d"], std=w["std"], seed=w["seed"])
    o = torch.empty((w["b"], w["S"], w["h_q"], w["d"]), dtype=torch.float32, device="cuda")
    m = torch.empty((w["b"], w["h_q"], w["S"]), dtype=torch.float32, device="cuda")
    l = torch.empty_like(m)
    desc = cpa.make_desc(w["b"], w["S"], w["h_q"], w["h_kv"], w["d"], w["cp"], 1.0 / math.sqrt(w["d"]), 1)
    fn = lambda: cpa.cp_ring_step_partial_attn(desc, 0, w["cp"], q, k, v, o, m, l, mode, stream)  # noqa: E731
    for _ in range(3):
        fn()
    ms = _events_time(fn, 10, stream)
    tf = prefill_flops(w) / (ms * 1e-3) / 1e12
    out["prefill_d64"] = {"workload": "prefill ring attention, head dimension 64: b1, 16/16 heads, d64, S32768, cp8",
                          "value": round(tf, 1), "unit": "TFLOP/s", "ms": round(ms, 3), "flops": prefill_flops(w),
                          "peak": peaks["bf16_tflops"], "frac": round(tf / peaks["bf16_tflops"], 4)}
    del q, k, v, o, m, l
    torch.cuda.empty_cache()
    # tiny prefill: b1, 4/4 heads, d64, S1024, cp2 (0.54 GFLOP).  A few CTAs per head and
    # 1 MB of inputs that stay in L2: launch- and latency-bound, reported as measured.
    w = synth.WORKLOADS["tiny"]
    q, k, v = synth.prefill_inputs(w["b"], w["S"], w["h_q"], w["h_kv"], w["d"], std=w["std"], seed=w["seed"])
    o = torch.empty((w["b"], w["S"], w["h_q"], w["d"]), dtype=torch.float32, device="cuda")
    m = torch.empty((w["b"], w["h_q"], w["S"]), dtype=torch.float32, device="cuda")
    l = torch.empty_like(m)
    desc = cpa.make_desc(w["b"], w["S"], w["h_q"], w["h_kv"], w["d"], w["cp"], 1.0 / math.sqrt(w["d"]), 1)
    mode = cpa.CP_MODE_EMIT | cpa.CP_MODE_FINALIZE
    fn = lambda: cpa.cp_ring_step_partial_attn(desc, 0, w["cp"], q, k, v, o, m, l, mode, stream)  # noqa: E731
    for _ in range(10):
        fn()
    ms = _events_time(fn, 200, stream)
    tf = prefill_flops(w) / (ms * 1e-3) / 1e12
    # the same launches replayed from a CUDA graph (20 per graph): no host launch cost
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=torch.cuda.Stream()):  # captured off the default stream
        for _ in range(20):
            cpa.cp_ring_step_partial_attn(desc, 0, w["cp"], q, k, v, o, m, l, mode, torch.cuda.current_stream())
    for _ in range(3):
        graph.replay()
    ms_graph = _events_time(graph.replay, 10, stream) / 20
    out["prefill_tiny"] = {"workload": "prefill ring attention, tiny: b1, 4/4 heads, d64, S1024, cp2 "
                                       "(inputs in L2; launch- and latency-bound)",
                           "value": round(tf, 2), "unit": "TFLOP/s", "us": round(ms * 1e3, 2),
                           "us_in_cuda_graph": round(ms_graph * 1e3, 2),
                           "flops": prefill_flops(w), "peak": peaks["bf16_tflops"],
                           "frac": round(tf / peaks["bf16_tflops"], 4)}
    if pool is not None:  # the whole workload: every row of every head
        cpu_jobs.append(("prefill_tiny", oracle_prefill_leg(pool, w, q, k, v, list(range(w["h_q"])), 0,
                                                            seed=w["seed"], full_rows=True, run=False)))
    del q, k, v, o, m, l
    torch.cuda.empty_cache()
    # pass-Q decode: b8, 16 heads, d512, L131072, cp8 (34.4 GB of K/V)
    w = synth.WORKLOADS["decode"]
    q, k, v = synth.decode_inputs(w["b"], w["S"], w["h_q"], w["h_kv"], w["d"], seed=w["seed"])
    desc = cpa.make_desc(w["b"], w["S"], w["h_q"], w["h_kv"], w["d"], w["cp"], 1.0 / math.sqrt(w["d"]), 0)
    nbytes = cpa.cp_passq_workspace_bytes(desc)
    ws = torch.empty(nbytes // 4, dtype=torch.float32, device="cuda")
    res = torch.empty((w["b"], w["h_q"], w["d"]), dtype=torch.float32, device="cuda")
    fn = lambda: cpa.cp_passq_decode(desc, q, k, v, ws, nbytes, res, None, None, stream)  # noqa: E731
    for _ in range(3):
        fn()
    ms = _events_time(fn, 10, stream)
    gbs = decode_bytes(w) / (ms * 1e-3) / 1e9
    out["decode"] = {"workload": "pass-Q decode: b8, 16 heads, d512, L131072, cp8", "value": round(gbs, 1),
                     "unit": "GB/s", "ms": round(ms, 4), "bytes": decode_bytes(w), "peak": peaks["hbm_gbs"],
                     "frac": round(gbs / peaks["hbm_gbs"], 4), "launches_per_call": 2}
    if pool is not None:  # 16 (sequence, head) pairs, two per sequence, every shard of each
        pairs = [(bi, h) for bi in range(w["b"]) for h in (bi % w["h_q"], (bi + 8) % w["h_q"])]
        cpu_jobs.append(("decode", oracle_decode_leg(pool, w, q, k, v, pairs, run=False)))
    del q, k, v, ws
    torch.cuda.empty_cache()
    # pass-Q decode with 16 query heads sharing one 512-wide K/V head (MQA / MLA-style), tensor cores
    b, L, hq, hkv, d, cp = 8, 131072, 16, 1, 512, 8
    q, k, v = synth.decode_inputs(b, L, hq, hkv, d, seed=20260006)
    desc = cpa.make_desc(b, L, hq, hkv, d, cp, 1.0 / math.sqrt(d), 0)
    nbytes = cpa.cp_passq_workspace_bytes(desc)
    ws = torch.empty(nbytes // 4, dtype=torch.float32, device="cuda")
    res = torch.empty((b, hq, d), dtype=torch.float32, device="cuda")
    fn = lambda: cpa.cp_passq_decode(desc, q, k, v, ws, nbytes, res, None, None, stream)  # noqa: E731
    for _ in range(3):
        fn()
    ms = _events_time(fn, 20, stream)
    wd = dict(b=b, S=L, h_q=hq, h_kv=hkv, d=d, cp=cp)
    gbs = decode_bytes(wd) / (ms * 1e-3) / 1e9
    out["decode_shared_kv"] = {"workload": "pass-Q decode, 16 q heads on one 512-wide K/V head: b8, L131072, cp8",
                               "value": round(gbs, 1), "unit": "GB/s", "ms": round(ms, 4), "bytes": decode_bytes(wd),
                               "tflops": round(4 * b * hq * d * L / (ms * 1e-3) / 1e12, 1),
                               "peak": peaks["hbm_gbs"], "frac": round(gbs / peaks["hbm_gbs"], 4),
                               "kernel": "mqa_decode_kernel<512,16> (tcgen05) + lse merge"}
    del q, k, v, ws
    torch.cuda.empty_cache()
    # LSE merge: 32 parts x 64 heads x 4096 rows x 128
    w = synth.WORKLOADS["merge"]
    po, pm, pl = synth.merge_parts(w["parts"], w["heads"], w["rows"], w["d"], spread=w["spread"], seed=w["seed"])
    mo = torch.empty((1, w["rows"], w["heads"], w["d"]), dtype=torch.float32, device="cuda")
    mm = torch.empty((1, w["heads"], w["rows"]), dtype=torch.float32, device="cuda")
    ml = torch.empty_like(mm)
    order = np.random.default_rng(w["seed"]).permutation(w["parts"])
    fn = lambda: cpa.cp_merge_partials(1, w["rows"], w["heads"], w["d"], w["parts"], po, pm, pl, mo, mm, ml,  # noqa
                                       order=order, stream=stream)
    for _ in range(3):
        fn()
    ms = _events_time(fn, 20, stream)
    gbs = merge_bytes(w) / (ms * 1e-3) / 1e9
    out["merge"] = {"workload": "LSE merge: 32 parts x 64 heads x 4096 rows x 128", "value": round(gbs, 1),
                    "unit": "GB/s", "ms": round(ms, 4), "bytes": merge_bytes(w), "peak": peaks["hbm_gbs"],
                    "frac": round(gbs / peaks["hbm_gbs"], 4)}
    if pool is not None:  # every row of 16 of the 64 heads
        cpu_jobs.append(("merge", oracle_merge_leg(pool, w, po, pm, pl, list(range(0, w["heads"], 4)), run=False)))
    # the same 32 parts reduced as the log-depth halving tree (5 levels of pairwise
    # merges), computed in one pass
    nbytes = cpa.cp_merge_tree_workspace_bytes(1, w["rows"], w["heads"], w["d"], w["parts"])
    fn = lambda: cpa.cp_merge_partials_tree(1, w["rows"], w["heads"], w["d"], w["parts"], po, pm, pl, None,  # noqa
                                            nbytes, mo, mm, ml, stream=stream)
    for _ in range(3):
        fn()
    tms = _events_time(fn, 20, stream)
    gbs_tree = merge_bytes(w) / (tms * 1e-3) / 1e9
    out["merge_tree"] = {"workload": "LSE merge of the same 32 parts as a 5-level tree (part i with i + n/2), one pass",
                         "value": round(gbs_tree, 1), "unit": "GB/s", "ms": round(tms, 4), "bytes": merge_bytes(w),
                         "peak": peaks["hbm_gbs"], "frac": round(gbs_tree / peaks["hbm_gbs"], 4), "launches": 1}
    del po, pm, pl, mo
    torch.cuda.empty_cache()
    for key, job in cpu_jobs:
        out[key]["cpu_baseline"] = job()
    return out


def bench_reference(args, rank, world):
    """The CPU oracle as the reference arm: each step is the oracle over a bounded row sample
    of the same workload (every head x the first and last row of each chunk, rows 0 and
    S-1 and seeded random rows, a new draw each step) on a spawn pool of one
    single-threaded worker per host core."""
    if rank != 0:
        return None
    from context_ring_attention_cp_gb300 import synth
    w = synth.WORKLOADS[WORKLOAD]
    pool = OraclePool(args.cpu_workers)
    try:
        q, k, v = synth.prefill_inputs(w["b"], w["S"], w["h_q"], w["h_kv"], w["d"], std=w["std"], seed=w["seed"],
                                       device="cpu")
        heads = list(range(w["h_q"]))
        for i in range(args.warmup):
            oracle_prefill_leg(pool, w, q, k, v, heads, args.cpu_random_rows, seed=i)
        legs = [oracle_prefill_leg(pool, w, q, k, v, heads, args.cpu_random_rows, seed=1000 + i)
                for i in range(args.steps)]
    finally:
        pool.close()
    tot_s = sum(x["seconds"] for x in legs)
    tot_flops = sum(x["value"] * 1e12 * x["seconds"] for x in legs)
    value = tot_flops / tot_s / 1e12
    cpu = dict(legs[-1])
    cpu["value"] = round(value, 6)
    cpu["seconds"] = round(tot_s, 3)
    cpu["full_config_s"] = {"value": round(prefill_flops(w) / (value * 1e12), 1),
                            "how": "extrapolated: the workload's FLOPs / the samples' fp64 FLOP rate"}
    cpu["sample"] = f"per step: {legs[-1]['sample']}"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tot_s * 1e3 / args.steps, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1)*0.5 bf16 Q/K/V)",
            "config": headline_config(world),
            "cpu_baseline": cpu,
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def profile_case(name, steps):
    """One kernel on a capture-sized case (a few GB on the device) for ncu; prints its time."""
    import torch
    import context_ring_attention_cp_gb300 as cpa
    from context_ring_attention_cp_gb300 import _build, synth
    _build.build()
    cpa.load_library()
    stream = torch.cuda.current_stream()
    unit = "GB/s"
    if name in ("ring-step", "ring-step-accumulate"):  # one ring step (t = 1) of the GQA workload
        w = synth.WORKLOADS[WORKLOAD]
        q, k, v = synth.prefill_inputs(w["b"], w["S"], w["h_q"], w["h_kv"], w["d"], std=w["std"], seed=w["seed"])
        o = torch.empty((w["b"], w["S"], w["h_q"], w["d"]), dtype=torch.float32, device="cuda")
        m = torch.empty((w["b"], w["h_q"], w["S"]), dtype=torch.float32, device="cuda")
        l = torch.empty_like(m)
        desc = cpa.make_desc(w["b"], w["S"], w["h_q"], w["h_kv"], w["d"], w["cp"], 1.0 / math.sqrt(w["d"]), 1)
        mode = cpa.CP_MODE_EMIT
        if name == "ring-step-accumulate":  # into the step-0 triple
            cpa.cp_ring_step_partial_attn(desc, 0, 1, q, k, v, o, m, l, cpa.CP_MODE_EMIT, stream)
            mode = cpa.CP_MODE_ACCUMULATE
        fn = lambda: cpa.cp_ring_step_partial_attn(desc, 1, 2, q, k, v, o, m, l, mode, stream)  # noqa: E731
        C = w["S"] // (2 * w["cp"])
        work = 4 * w["b"] * w["h_q"] * w["d"] * w["cp"] * 2 * C * C / 1e3  # so that work / s / 1e9 is TFLOP/s
        unit = "TFLOP/s"
    elif name == "ring-mha":  # the multi-head workload's fused ring (32/32 heads, row-paired tiles)
        w = synth.WORKLOADS["mha"]
        q, k, v = synth.prefill_inputs(w["b"], w["S"], w["h_q"], w["h_kv"], w["d"], std=w["std"], seed=w["seed"])
        o = torch.empty((w["b"], w["S"], w["h_q"], w["d"]), dtype=torch.float32, device="cuda")
        m = torch.empty((w["b"], w["h_q"], w["S"]), dtype=torch.float32, device="cuda")
        l = torch.empty_like(m)
        desc = cpa.make_desc(w["b"], w["S"], w["h_q"], w["h_kv"], w["d"], w["cp"], 1.0 / math.sqrt(w["d"]), 1)
        mode = cpa.CP_MODE_EMIT | cpa.CP_MODE_FINALIZE
        fn = lambda: cpa.cp_ring_step_partial_attn(desc, 0, w["cp"], q, k, v, o, m, l, mode, stream)  # noqa: E731
        work = prefill_flops(w) / 1e3
        unit = "TFLOP/s"
    elif name in ("ring-tiny", "ring-d64"):  # the tiny workload (key walks split over clusters) / d64 at scale
        w = synth.WORKLOADS["tiny" if name == "ring-tiny" else "mha64"]
        q, k, v = synth.prefill_inputs(w["b"], w["S"], w["h_q"], w["h_kv"], w["d"], std=w["std"], seed=w["seed"])
        o = torch.empty((w["b"], w["S"], w["h_q"], w["d"]), dtype=torch.float32, device="cuda")
        m = torch.empty((w["b"], w["h_q"], w["S"]), dtype=torch.float32, device="cuda")
        l = torch.empty_like(m)
        desc = cpa.make_desc(w["b"], w["S"], w["h_q"], w["h_kv"], w["d"], w["cp"], 1.0 / math.sqrt(w["d"]), 1)
        mode = cpa.CP_MODE_EMIT | cpa.CP_MODE_FINALIZE
        fn = lambda: cpa.cp_ring_step_partial_attn(desc, 0, w["cp"], q, k, v, o, m, l, mode, stream)  # noqa: E731
        work = prefill_flops(w) / 1e3
        unit = "TFLOP/s"
    elif name == "decode-small":  # b8, 16 heads, d512, L8192, cp8: 2.1 GB of K/V
        b, L, h, d, cp = 8, 8192, 16, 512, 8
        q, k, v = synth.decode_inputs(b, L, h, h, d, seed=7)
        desc = cpa.make_desc(b, L, h, h, d, cp, 1.0 / math.sqrt(d), 0)
        nbytes = cpa.cp_passq_workspace_bytes(desc)
        ws = torch.empty(nbytes // 4, dtype=torch.float32, device="cuda")
        out = torch.empty((b, h, d), dtype=torch.float32, device="cuda")
        fn = lambda: cpa.cp_passq_decode(desc, q, k, v, ws, nbytes, out, None, None, stream)  # noqa: E731
        work = 2 * b * L * h * d * 2
    elif name == "decode-shared-kv":  # b8, 16 q heads on one 512-wide K/V head, L131072, cp8: 2.1 GB
        b, L, hq, hkv, d, cp = 8, 131072, 16, 1, 512, 8
        q, k, v = synth.decode_inputs(b, L, hq, hkv, d, seed=7)
        desc = cpa.make_desc(b, L, hq, hkv, d, cp, 1.0 / math.sqrt(d), 0)
        nbytes = cpa.cp_passq_workspace_bytes(desc)
        ws = torch.empty(nbytes // 4, dtype=torch.float32, device="cuda")
        out = torch.empty((b, hq, d), dtype=torch.float32, device="cuda")
        fn = lambda: cpa.cp_passq_decode(desc, q, k, v, ws, nbytes, out, None, None, stream)  # noqa: E731
        work = 2 * b * L * hkv * d * 2
    elif name == "merge":  # the merge-stress workload itself: 4.5 GB
        w = synth.WORKLOADS["merge"]
        po, pm, pl = synth.merge_parts(w["parts"], w["heads"], w["rows"], w["d"], spread=w["spread"], seed=w["seed"])
        mo = torch.empty((1, w["rows"], w["heads"], w["d"]), dtype=torch.float32, device="cuda")
        mm = torch.empty((1, w["heads"], w["rows"]), dtype=torch.float32, device="cuda")
        ml = torch.empty_like(mm)
        fn = lambda: cpa.cp_merge_partials(1, w["rows"], w["heads"], w["d"], w["parts"], po, pm, pl, mo, mm, ml,  # noqa
                                           stream=stream)
        work = merge_bytes(w)
    elif name == "merge-tree":  # the merge-stress parts reduced as the halving tree, one pass
        w = synth.WORKLOADS["merge"]
        po, pm, pl = synth.merge_parts(w["parts"], w["heads"], w["rows"], w["d"], spread=w["spread"], seed=w["seed"])
        mo = torch.empty((1, w["rows"], w["heads"], w["d"]), dtype=torch.float32, device="cuda")
        mm = torch.empty((1, w["heads"], w["rows"]), dtype=torch.float32, device="cuda")
        ml = torch.empty_like(mm)
        fn = lambda: cpa.cp_merge_partials_tree(1, w["rows"], w["heads"], w["d"], w["parts"], po, pm, pl, None, 0,  # noqa
                                                mo, mm, ml, stream=stream)
        work = merge_bytes(w)
    else:
        raise SystemExit(f"unknown --case {name}")
    for _ in range(3):
        fn()
    ms = _events_time(fn, steps, stream)
    print(json.dumps({"case": name, "ms": round(ms, 4), unit: round(work / (ms * 1e-3) / 1e9, 1)}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-workers", type=int, default=os.cpu_count() or 1,
                    help="oracle worker processes (default: every host core)")
    ap.add_argument("--cpu-random-rows", type=int, default=64,
                    help="seeded random rows per head in each step's sample of the reference arm")
    ap.add_argument("--cpu-baseline-rows", type=int, default=2048,
                    help="seeded random rows per head in the headline's cpu_baseline sample "
                         "(about 10 s of fp64 work on 16 cores)")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-secondary", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--case", choices=["ring-step", "ring-step-accumulate", "ring-mha", "ring-tiny", "ring-d64",
                                       "decode-small",
                                       "decode-shared-kv", "merge", "merge-tree"], default=None,
                    help="time one kernel on a capture-sized case (for ncu) instead of the benchmark")
    args = ap.parse_args()
    if args.case is not None:
        sys.path.insert(0, ROOT)
        profile_case(args.case, args.steps)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    sys.path.insert(0, ROOT)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if args.impl == "reference":
        line = bench_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    import torch
    if world > 1:
        import torch.distributed as tdist
        local = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl")
        dist = tdist
    line = bench_ours(args, rank, world, dist)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
