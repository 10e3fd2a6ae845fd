#!/usr/bin/env python3
"""Benchmark of the fused DiT QK-RMSNorm + RoPE on the Wan-A14B shape.

One step = one qknr_forward over the full Wan workload: a packed bf16 QKV
activation [32760, 3*40*128] (a 21x30x52 latent grid), per-head RMSNorm of
the 40 Q and 40 K heads (head_dim 128) with fp32 gains, then interleaved
RoPE from a shared fp32 cos/sin row per token (3-axis 44/42/42 split),
in place, V untouched.

Prints one JSON line: microseconds per call (whole job), achieved HBM
bandwidth against the measured copy peak, the CPU oracle's time on a
bounded sample, an end-to-end number from pinned host buffers (one
qknr_forward_host call per step), the SM clocks seen during the timed
region, the launch count, and (with the default workload) every other
workload and variant timed the same way (``configs``).  ``--impl
reference`` times the fp64 CPU oracle instead.

Multi-GPU: one process per GPU (torchrun); every rank runs its own full
workload (replicas, weak scaling), timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from diffusion_transformer_qk_gb300 import inputs as I  # noqa: E402

METRIC = "fused QK-RMSNorm+RoPE µs/call and achieved HBM GB/s (% of peak), Wan 40x128"
UNIT = "us/call"
DEFAULT_WORKLOAD = "wan_32760x40x128"
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ("qknr_kernel.cuh", "qknr_ptx.cuh", "qknr_api.cu", "qknr_internal.h")


# ---------------------------------------------------------------------------
# distributed plumbing (replicas: barrier and max over ranks only)

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def dist_init(backend: str):
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        os.environ.setdefault("MASTER_PORT", "29511")
        dist.init_process_group(backend, rank=rank, world_size=world)
    return rank, world, local


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    """Largest value of x over all ranks (x itself when not distributed)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_us_per_call(max_elapsed_s: float, steps: int, world: int) -> float:
    """Microseconds per call over the whole job: every rank made `steps`
    calls inside the slowest rank's elapsed time."""
    return max_elapsed_s * 1e6 / (steps * world)


# ---------------------------------------------------------------------------
# measured peaks, clocks, traffic record

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(sources=KERNEL_SOURCES) -> str:
    """sha256 over the given kernel source files (in order)."""
    h = hashlib.sha256()
    for name in sources:
        with open(os.path.join(ROOT, "diffusion_transformer_qk_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu record, if it was taken
    on the current sources of that kernel; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(workload)
        if not rec or rec.get("kernel_src_sha256") != kernel_source_hash(rec.get("sources", KERNEL_SOURCES)):
            return None
    except Exception:
        return None
    return rec.get("dram_bytes_per_launch")


class NvmlClockSampler:
    """SM clock and clock-event reasons read through NVML (libnvidia-ml, by
    ctypes; read-only queries) every millisecond on a thread, so that even a
    timed region of a few milliseconds has samples.  Raises if NVML or the
    device cannot be opened; ClockSampler then falls back to nvidia-smi."""

    # nvmlClocksEventReasons bits
    REASONS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40,
               "hw_power_brake_slowdown": 0x80}

    def __init__(self, uuid: str, period_s: float = 0.001):
        import ctypes

        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.lib = lib
        self.dev = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.dev)) != 0:
            raise RuntimeError("nvmlDeviceGetHandleByUUID failed")
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint(0)
        lib.nvmlDeviceGetMaxClockInfo(self.dev, 1, ctypes.byref(mx))       # NVML_CLOCK_SM
        self.max_mhz = float(mx.value) or None
        self.samples = []
        self.period = period_s
        self.running = True
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        import ctypes

        mhz, reasons = ctypes.c_uint(0), ctypes.c_ulonglong(0)
        while self.running:
            ok = self.lib.nvmlDeviceGetClockInfo(self.dev, 1, ctypes.byref(mhz)) == 0
            ok = ok and self.reasons_fn(self.dev, ctypes.byref(reasons)) == 0
            if ok:
                self.samples.append((time.perf_counter(), float(mhz.value), int(reasons.value)))
            time.sleep(self.period)

    def stop(self):
        self.running = False
        self.thread.join(timeout=5)
        self.lib.nvmlShutdown()

    def summary(self, t0: float, t1: float):
        inside = [(m, r) for t, m, r in self.samples if t0 <= t <= t1]
        note = "NVML, sampled every 1 ms during the timed region"
        if not inside:
            inside = [(m, r) for _, m, r in self.samples]
            note = "NVML; no sample fell inside the timed region: samples span warm-up and timed steps"
        reasons = sorted({n for _, r in inside for n, bit in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(m for m, _ in inside) if inside else None, "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(inside), "note": note}


def clock_sampler(uuid_or_index: str):
    """The NVML sampler when NVML is there, else nvidia-smi's."""
    if uuid_or_index.startswith("GPU-"):
        try:
            return NvmlClockSampler(uuid_or_index)
        except Exception:
            pass
    return ClockSampler(uuid_or_index)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str):
        self.samples = []
        self.error = None
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", gpu_id, "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception as e:  # no nvidia-smi
            self.error = str(e)
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == len(self.FIELDS):
                self.samples.append((time.perf_counter(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        if self.error:
            return {"error": self.error}
        inside = [s for t, s in self.samples if t0 <= t <= t1]
        note = "sampled during the timed region"
        if not inside:
            inside = [s for _, s in self.samples]
            note = "timed region shorter than the 100 ms sampling period: samples span warm-up and timed steps"
        mhz = []
        reasons = set()
        max_mhz = None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in inside:
            try:
                mhz.append(float(s[0]))
                max_mhz = float(s[1])
            except ValueError:
                pass
            for n, v in zip(names, s[3:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": max_mhz,
                "reasons": sorted(reasons), "samples": len(inside), "note": note}


# ---------------------------------------------------------------------------
# CPU oracle timing

def oracle_rows(w, inp, rows):
    """The oracle over the given token rows of one workload instance."""
    from oracle import qknr_oracle as O

    if w.packed:
        return O.forward_packed(inp["qkv"], w.dtype, w.n_heads_q, w.n_heads_k, w.n_heads_v, w.head_dim,
                                inp["gamma_q"], inp["gamma_k"], w.eps, inp["cos"], inp["sin"], w.cos_dtype,
                                w.rope_style, "shared_row", rows=rows)
    return [O.forward_separate(inp[n], w.dtype, h, w.head_dim, inp[g], w.eps, inp["cos"], inp["sin"],
                               w.cos_dtype, w.rope_style, "shared_row", rows=rows)
            for n, h, g in (("q", w.n_heads_q, "gamma_q"), ("k", w.n_heads_k, "gamma_k"))]


def time_oracle_workload(w, inp, target_s: float, tokens: int):
    """Time the oracle on the first token rows, as many as take about
    target_s seconds; returns (us per full call, rows, seconds).  The
    expanded-layout workloads hold equal values in every head's table row,
    so the oracle runs them from the shared rows (the same numbers)."""
    rows_avail = (inp["qkv"] if w.packed else inp["q"]).shape[0]
    probe = np.arange(min(256, rows_avail))
    t0 = time.perf_counter()
    oracle_rows(w, inp, probe)
    per_tok = (time.perf_counter() - t0) / len(probe)
    n = int(min(rows_avail, max(len(probe), target_s / max(per_tok, 1e-9))))
    t0 = time.perf_counter()
    oracle_rows(w, inp, np.arange(n))
    dt = time.perf_counter() - t0
    return dt / n * tokens * 1e6, n, dt


# The oracle on every host core: a process pool (spawn, so it is safe after
# the GPU has been used).  Each worker makes its own seeded rows of the
# workload once, outside the timing; the oracle's cost does not depend on
# the values, so no activation data crosses processes.

_pool_w = None
_pool_inp = None


def _oracle_worker_init(w, rows):
    global _pool_w, _pool_inp
    _pool_w = w
    _pool_inp = I.make_inputs(w, tokens=rows)
    oracle_rows(w, _pool_inp, np.arange(min(8, rows)))       # first-call costs


def _oracle_worker_task(_):
    n = (_pool_inp["qkv"] if _pool_w.packed else _pool_inp["q"]).shape[0]
    oracle_rows(_pool_w, _pool_inp, np.arange(n))
    return n


class OraclePool:
    """The unchanged oracle over ``rows`` token rows per task, on
    ``processes`` worker processes (default: every core this process may
    run on)."""

    def __init__(self, w, rows: int, processes: int = 0):
        import multiprocessing as mp

        self.processes = processes or len(os.sched_getaffinity(0))
        self.rows = rows
        self.pool = mp.get_context("spawn").Pool(self.processes, initializer=_oracle_worker_init,
                                                 initargs=(w, rows))
        # every worker has finished its initializer once it has run a task
        self.run_round(2)

    def run_round(self, tasks_per_worker: int = 1) -> tuple:
        """Run tasks_per_worker tasks on every worker; (seconds, rows)."""
        t0 = time.perf_counter()
        done = self.pool.map(_oracle_worker_task, range(self.processes * tasks_per_worker), chunksize=1)
        return time.perf_counter() - t0, sum(done)

    def close(self):
        self.pool.close()
        self.pool.join()


def time_oracle_all_cores(w, tokens: int, per_row_s: float, target_s: float, processes: int = 0):
    """us per full call of `tokens` rows with the oracle on every core, from
    about target_s seconds of work; returns (us, cores, rows, seconds)."""
    rows = int(max(32, min(4096, 0.25 / max(per_row_s, 1e-9))))       # about 0.25 s per task
    pool = OraclePool(w, rows, processes)
    try:
        per_round = rows * per_row_s
        k = int(max(1, round(target_s / max(per_round, 1e-9))))
        dt, n = pool.run_round(k)
    finally:
        pool.close()
    return dt / n * tokens * 1e6, pool.processes, n, dt, rows


# ---------------------------------------------------------------------------
# the reference arm: the CPU oracle as it stands, on every host core

def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    # one task of `rows` rows per core and step; steps sized so the warm-up
    # and timed steps end in about two minutes
    probe_inp = I.make_inputs(w, tokens=64)
    t0 = time.perf_counter()
    oracle_rows(w, probe_inp, np.arange(64))
    per_row = (time.perf_counter() - t0) / 64
    per_step = 120.0 / (args.steps + args.warmup)
    rows = int(max(1, min(4096, per_step / max(per_row, 1e-9))))
    pool = OraclePool(w, rows, args.oracle_processes)
    times = []
    try:
        for i in range(args.warmup + args.steps):
            dt, n = pool.run_round(1)
            if i >= args.warmup:
                times.append(dt / n)
    finally:
        pool.close()
    us = statistics.fmean(times) * w.tokens * 1e6
    sample = (f"{rows} token rows per core per step ({pool.processes} processes, one task each) of the "
              f"{w.tokens}-token workload, scaled to a full call by tokens; fp64 numpy")
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, world),
        "cpu_baseline": {"value": us, "unit": UNIT, "cores": pool.processes, "kind": "oracle", "sample": sample},
        "e2e": {"value": us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w, world, tokens=None):
    if isinstance(w, I.GroupNormWorkload):
        return {"workload": w.name, "shape_nchw": [w.n, w.c, w.h, w.w], "groups": w.groups, "in_place": True,
                "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas x{world}"}
    if isinstance(w, I.AdaLNWorkload):
        return {"workload": w.name, "tokens": w.tokens if tokens is None else tokens, "hidden": w.hidden,
                "rows_per_batch": w.seq, "mod_dtype": w.mod_dtype, "in_place": True,
                "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas x{world}"}
    return {
        "workload": w.name, "tokens": w.tokens if tokens is None else tokens, "n_heads_q": w.n_heads_q, "n_heads_k": w.n_heads_k,
        "n_heads_v": w.n_heads_v, "head_dim": w.head_dim, "layout": "packed_qkv" if w.packed else "separate",
        "rope": w.rope_style, "cos_layout": w.cos_layout, "cos_dtype": w.cos_dtype,
        "rope_axes": list(w.axes_dim), "in_place": not w.out_of_place,
        "launch_form": ("packed" if w.packed else ("q+k in one launch" if w.single_launch else "one launch per tensor")),
        "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas x{world}",
    }


# ---------------------------------------------------------------------------
# our arm

class Runner:
    """Device buffers and launch arguments of one workload.  A step is the
    list of launches that processes the whole workload once: one launch for
    a packed QKV activation, one per tensor (Q, then K) for FLUX.2's
    separate tensors."""

    def __init__(self, w, dev, tune, status, tokens=None, inp=None):
        import torch

        from diffusion_transformer_qk_gb300 import qknr as Q

        self.Q, self.w, self.dev = Q, w, dev
        self.tokens = w.tokens if tokens is None else tokens
        if inp is None:
            inp = I.make_inputs(w, tokens=self.tokens)
        self.inp = inp
        D = w.head_dim

        def dev_bits(a):
            return torch.from_numpy(a.view(np.int16)).view(
                torch.bfloat16 if w.dtype == "bf16" else torch.float16)

        def dev_tab(a):
            t = torch.from_numpy(a) if w.cos_dtype == "fp32" else torch.from_numpy(a.view(np.int16)).view(
                torch.bfloat16)
            return t

        self.host = {}
        if w.packed:
            self.host["qkv"] = dev_bits(inp["qkv"])
        else:
            for n in ("q", "k", "v"):
                self.host[n] = dev_bits(inp[n])
        self.host["gamma_q"] = torch.from_numpy(inp["gamma_q"])
        self.host["gamma_k"] = torch.from_numpy(inp["gamma_k"])
        cos, sin = dev_tab(inp["cos"]), dev_tab(inp["sin"])
        if w.cos_layout == "per_head_expanded":
            H = w.n_heads_q
            cos = cos[:, None, :].expand(cos.shape[0], H, D).contiguous()
            sin = sin[:, None, :].expand(sin.shape[0], H, D).contiguous()
        self.host["cos"], self.host["sin"] = cos, sin
        self.d = {k: v.to(dev) for k, v in self.host.items()}
        self.tune = tune
        kw = dict(rope_style=w.rope_style, cos_layout=w.cos_layout, eps=w.eps, dev_status=status, **tune)
        d = self.d
        if w.packed:
            out = None
            if w.out_of_place:
                self.d["out"] = torch.empty_like(d["qkv"])
                self.host["out"] = torch.empty_like(self.host["qkv"])
                out = self.d["out"]
            self.args = [Q.packed_args(d["qkv"], w.n_heads_q, w.n_heads_k, w.n_heads_v, D, d["gamma_q"],
                                       d["gamma_k"], d["cos"], d["sin"], out=out, **kw)]
            self.bytes_per_launch = I.algorithmic_bytes(w, tokens=self.tokens)
            self.outputs = ["out" if w.out_of_place else "qkv"]
        elif w.single_launch:
            self.args = [Q.make_args(q=d["q"], k=d["k"], n_heads_q=w.n_heads_q, n_heads_k=w.n_heads_k, head_dim=D,
                                     gamma_q=d["gamma_q"], gamma_k=d["gamma_k"], cos=d["cos"], sin=d["sin"], **kw)]
            self.bytes_per_launch = I.algorithmic_bytes(w, tokens=self.tokens)
            self.outputs = ["q", "k"]
        else:
            self.args = [Q.make_args(q=d["q"], n_heads_q=w.n_heads_q, head_dim=D, gamma_q=d["gamma_q"],
                                     cos=d["cos"], sin=d["sin"], **kw),
                         Q.make_args(k=d["k"], n_heads_k=w.n_heads_k, head_dim=D, gamma_k=d["gamma_k"],
                                     cos=d["cos"], sin=d["sin"], **kw)]
            self.bytes_per_launch = I.algorithmic_bytes(w, launches="q", tokens=self.tokens)
            self.outputs = ["q", "k"]
        self.info = Q.query(self.args[0])
        self.launch = Q.launch

    def step(self, stream):
        for a in self.args:
            self.Q.launch(a, stream)

    def e2e_buffers(self, chunk_rows):
        """Pinned host copies of every input and output.  Packed workloads go
        through qknr_forward_host (the binding's HostPipeline: copies in,
        kernel and copies out overlapped on three streams inside the
        library); separate tensors are copied in, processed and copied out
        on one stream."""
        self.pinned = {k: v.pin_memory() for k, v in self.host.items() if k not in self.outputs or k in
                       ("qkv", "q", "k")}
        self.pinned_out = {k: torch_empty_pinned_like(self.host[k]) for k in self.outputs}
        h2d = sum(t.numel() * t.element_size() for t in self.pinned.values())
        d2h = sum(t.numel() * t.element_size() for t in self.pinned_out.values())
        self.pipe = None
        if self.w.packed and not self.w.out_of_place:
            # in place on the pinned host activation: the Q|K columns of each
            # row go to the device and back; V is never read or written
            qkv = self.pinned["qkv"]
            self.pipe = self.Q.HostPipeline(qkv.shape[1], qkv.dtype, chunk_rows=chunk_rows, device=self.dev)
            es = qkv.element_size()
            qk = (self.w.n_heads_q + self.w.n_heads_k) * self.w.head_dim
            tables = sum(self.pinned[k].numel() * self.pinned[k].element_size()
                         for k in ("gamma_q", "gamma_k", "cos", "sin") if k in self.pinned)
            h2d = qkv.shape[0] * qk * es + tables
            d2h = qkv.shape[0] * qk * es
        return h2d, d2h

    def e2e_result(self):
        """The pinned host tensor holding the e2e result."""
        return self.pinned["qkv"] if self.pipe is not None else self.pinned_out[self.outputs[0]]

    def e2e_step(self, stream):
        if self.pipe is not None:
            w, p = self.w, self.pinned
            self.pipe(p["qkv"], w.n_heads_q, w.n_heads_k, w.n_heads_v, w.head_dim, p["gamma_q"], p["gamma_k"],
                      p["cos"], p["sin"], rope_style=w.rope_style, cos_layout=w.cos_layout, eps=w.eps, **self.tune)
            return
        for k, t in self.pinned.items():
            self.d[k].copy_(t, non_blocking=True)
        self.step(stream)
        for k, t in self.pinned_out.items():
            t.copy_(self.d[k], non_blocking=True)


class AdaLNRunner:
    """Device buffers and launch arguments of an AdaLN scale/shift workload
    (one launch per step, in place)."""

    def __init__(self, w, dev, tune, status, tokens=None, inp=None):
        import torch

        from diffusion_transformer_qk_gb300 import qknr as Q

        self.Q, self.w, self.dev, self.tune = Q, w, dev, tune
        self.tokens = w.tokens if tokens is None else tokens
        self.inp = I.make_adaln_inputs(w, tokens=self.tokens) if inp is None else inp
        act = torch.bfloat16 if w.dtype == "bf16" else torch.float16

        def bits(a, dt):
            return torch.from_numpy(a.view(np.int16)).view(dt)

        self.host = {"x": bits(self.inp["x"], act)}
        for k in ("scale", "shift"):
            m = self.inp[k]
            self.host[k] = torch.from_numpy(m) if w.mod_dtype == "fp32" else bits(m, act)
        self.d = {k: v.to(dev) for k, v in self.host.items()}
        self.args = [Q.adaln_args(self.d["x"], self.d["scale"], self.d["shift"], rows_per_batch=w.seq, eps=w.eps,
                                  dev_status=status, **tune)]
        self.launch = Q.adaln_launch
        self.bytes_per_launch = I.adaln_algorithmic_bytes(w, tokens=self.tokens)
        self.outputs = ["x"]
        self.info = Q.adaln_query(self.args[0])
        self.pipe = None

    def step(self, stream):
        for a in self.args:
            self.launch(a, stream)

    def e2e_buffers(self, chunk_rows):
        self.pinned = {k: v.pin_memory() for k, v in self.host.items()}
        self.pinned_out = {"x": torch_empty_pinned_like(self.host["x"])}
        h2d = sum(t.numel() * t.element_size() for t in self.pinned.values())
        d2h = self.pinned_out["x"].numel() * self.pinned_out["x"].element_size()
        return h2d, d2h

    def e2e_step(self, stream):
        for k, t in self.pinned.items():
            self.d[k].copy_(t, non_blocking=True)
        self.step(stream)
        self.pinned_out["x"].copy_(self.d["x"], non_blocking=True)


class GroupNormRunner:
    """Device buffers and arguments of a VAE group-norm + SiLU workload.  One
    step is one call: one launch on the fused or the cluster path, two
    launches (statistics, apply) per batch of groups on the two-pass path.
    The caller-owned workspace is allocated once here."""

    def __init__(self, w, dev, tune, status, tokens=None):
        import re

        import torch

        from diffusion_transformer_qk_gb300 import qknr as Q

        self.Q, self.w, self.dev, self.tune = Q, w, dev, tune
        self.tokens = w.elements
        self.inp = I.make_gn_inputs(w)
        act = torch.bfloat16 if w.dtype == "bf16" else torch.float16
        self.host = {"x": torch.from_numpy(self.inp["x"].view(np.int16)).view(act),
                     "gamma": torch.from_numpy(self.inp["gamma"]), "beta": torch.from_numpy(self.inp["beta"])}
        self.d = {k: v.to(dev) for k, v in self.host.items()}
        a = Q.gn_args(self.d["x"], w.groups, self.d["gamma"], self.d["beta"], eps=w.eps, dev_status=status,
                      mode=tune.get("gn_mode", "auto"))
        self.workspace = torch.empty(Q.gn_workspace_bytes(a), dtype=torch.uint8, device=dev)
        a.workspace, a.workspace_bytes = self.workspace.data_ptr(), self.workspace.numel()
        self.args = [a]
        self.launch = Q.gn_launch
        self.bytes_per_launch = I.gn_algorithmic_bytes(w)
        self.outputs = ["x"]
        self.pipe = None
        self.info = Q.gn_query(a)
        if self.info["kernel"].startswith(("gn_fused", "gn_cluster")):
            self.launches_per_call = 1
        else:
            m = re.search(r" x(\d+),", self.info["kernel"])
            self.launches_per_call = 2 * (int(m.group(1)) if m else 1)

    def step(self, stream):
        for a in self.args:
            self.launch(a, stream)

    def e2e_buffers(self, chunk_rows):
        self.pinned = {k: v.pin_memory() for k, v in self.host.items()}
        self.pinned_out = {"x": torch_empty_pinned_like(self.host["x"])}
        h2d = sum(t.numel() * t.element_size() for t in self.pinned.values())
        return h2d, self.pinned_out["x"].numel() * self.pinned_out["x"].element_size()

    def e2e_step(self, stream):
        for k, t in self.pinned.items():
            self.d[k].copy_(t, non_blocking=True)
        self.step(stream)
        self.pinned_out["x"].copy_(self.d["x"], non_blocking=True)


def torch_empty_pinned_like(t):
    import torch

    return torch.empty(t.shape, dtype=t.dtype, pin_memory=True)


def run_ours(args, w):
    import torch

    from diffusion_transformer_qk_gb300 import build as B
    from diffusion_transformer_qk_gb300 import qknr as Q

    rank, world, local = dist_init("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B.ensure_built()
    Q.load()

    status = torch.zeros(1, dtype=torch.int32, device=dev)
    if isinstance(w, I.GroupNormWorkload):
        tune = dict(gn_mode=args.gn_mode)
    else:
        tune = dict(ctas_per_sm=args.ctas_per_sm, stages=args.stages, consumer_warps=args.consumer_warps,
                    group_warps=args.group_warps, flags=Q.FLAG_NO_OVERLAP if args.no_overlap else 0)
    runner = {I.AdaLNWorkload: AdaLNRunner, I.GroupNormWorkload: GroupNormRunner}.get(type(w), Runner)
    run = runner(w, dev, tune, status, args.tokens)
    stream = torch.cuda.current_stream(dev)
    L = len(run.args)

    for _ in range(args.warmup):
        run.step(stream)
    torch.cuda.synchronize(dev)

    props = torch.cuda.get_device_properties(dev)
    gpu_id = ("GPU-" + str(props.uuid)) if getattr(props, "uuid", None) else str(local)
    sampler = clock_sampler(gpu_id)
    time.sleep(0.3)                       # let the sampler start
    for _ in range(args.warmup):
        run.step(stream)
    K = args.steps
    # Inputs smaller than twice the L2 would be partly served from L2 on the
    # next step: write a buffer of twice the L2 between steps and time only
    # the launches (per-launch events) in that case.
    l2 = getattr(props, "L2_cache_size", 0) or 129 * 2 ** 20
    flush = None
    if args.l2_flush == "on" or (args.l2_flush == "auto" and run.bytes_per_launch * L < 2 * l2):
        flush = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)
    # A step of one launch with no flush runs back to back: the launch's
    # average duration over the timed region is the region's time / K, and
    # no event sits between launches (an event there makes each launch wait
    # for the previous one to drain).  Otherwise every launch is bracketed
    # by its own pair of events.
    per_launch = L > 1 or flush is not None
    n_ev = K * L if per_launch else 0
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    barrier()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    e0.record(stream)
    j = 0
    for _ in range(K):
        if flush is not None:
            flush.fill_(1.0)
        for a in run.args:
            if per_launch:
                starts[j].record(stream)
            run.launch(a, stream)
            if per_launch:
                ends[j].record(stream)
            j += 1
    e1.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.perf_counter()
    barrier()
    sampler.stop()
    clocks = sampler.summary(t0, t1)

    if per_launch:
        kernel_ms = statistics.fmean(s.elapsed_time(e) for s, e in zip(starts, ends))
    else:
        kernel_ms = e0.elapsed_time(e1) / K
    if flush is None:
        elapsed = e0.elapsed_time(e1) / 1e3
    else:
        # the step time is the launches' own time; the flushes are excluded
        elapsed = kernel_ms * L * K / 1e3
    st = int(status.item())
    if st != 0:
        raise RuntimeError(f"kernel reported status {st} ({Q.STATUS.get(st)})")
    max_elapsed = max_over_ranks(elapsed, dev)
    max_kernel_ms = max_over_ranks(kernel_ms, dev)

    # end to end through the public API: pinned host inputs -> device -> calls -> host
    e2e = None
    if not args.no_e2e:
        n_e2e = min(K, args.e2e_steps)
        h2d, d2h = run.e2e_buffers(args.e2e_chunk_rows)
        for _ in range(3):
            run.e2e_step(stream)
        torch.cuda.synchronize(dev)
        barrier()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(n_e2e):
            run.e2e_step(stream)
        s1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_s = max_over_ranks(s0.elapsed_time(s1) / 1e3, dev)
        e2e = {"value": whole_job_us_per_call(e2e_s, n_e2e, world), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "path": ("one qknr_forward_host call per step (C ABI, through the binding's HostPipeline), in "
                        "place on the pinned host activation: the library copies the Q|K columns of rows in "
                        "chunks of %d host->device, runs qknr_forward on each and copies them back, overlapped "
                        "on three streams; the gains and tables are copied host->device each step (V is neither "
                        "read nor written by the operation, so it never leaves the host)"
                        % args.e2e_chunk_rows) if run.pipe else
                       "pinned host -> device copies, qknr_forward via the Python binding, device -> pinned host, "
                       "one stream"}
        if getattr(w, "packed", False):
            # each e2e step starts from the host input, so V comes back unchanged
            D3 = (w.n_heads_q + w.n_heads_k) * w.head_dim
            back = run.e2e_result().view(torch.int16).numpy().view(np.uint16)
            if not np.array_equal(back[:, D3:], run.inp["qkv"][:, D3:]):
                raise RuntimeError("e2e: V slice changed")
        if int(status.item()) != 0 or (run.pipe is not None and run.pipe.read_status() != 0):
            raise RuntimeError("kernel reported a timeout during the e2e loop")

    if rank != 0:
        return 0

    value = whole_job_us_per_call(max_elapsed, K, world)
    achieved = run.bytes_per_launch / (max_kernel_ms / 1e3) / 1e9
    peak, peak_kind = hbm_peak()
    # the record is of the named workload as it stands (not of an override)
    named = I.WORKLOADS.get(w.name) or I.ADALN_WORKLOADS.get(w.name) or I.GN_WORKLOADS.get(w.name)
    traffic = recorded_traffic(w.name) if named == w else None
    info = run.info
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": max_elapsed * 1e3 / K, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": dict(workload_config(w, world, run.tokens),
                       l2=("L2 flushed between steps (write of 2x L2); launches timed by per-launch events"
                           if flush is not None else
                           ("inputs larger than L2 (no flush)" if run.bytes_per_launch * L >= 2 * l2 else
                            "not flushed (--l2-flush off): a hot number, inputs partly served from L2"))),
        "gbs": run.bytes_per_launch * L * K * world / max_elapsed / 1e9,
        "pct_of_hbm_peak": 100.0 * achieved / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "peak_source": f"{peak_kind} copy bandwidth (hbm_gbs)",
                     "algorithmic_bytes_per_launch": run.bytes_per_launch, "kernel_us": max_kernel_ms * 1e3,
                     "launches_per_step": L, "kernel": info["kernel"],
                     "kernel_timing": ("per-launch CUDA events" if per_launch else
                                       "CUDA events around the back-to-back timed region / steps")},
        "gpu_launches": K * L * getattr(run, "launches_per_call", 1),
        "clocks": clocks,
        "launch": {k: info[k] for k in ("grid", "block", "dyn_smem", "stages", "ctas_per_sm", "consumer_warps",
                                        "stage_bytes", "registers", "num_sms", "prefetch_rows") if k in info},
    }
    if e2e:
        line["e2e"] = e2e
    if world == 1 and not args.no_cpu_baseline and isinstance(w, I.Workload):
        us1, n1, dt1 = time_oracle_workload(w, run.inp, args.cpu_seconds, run.tokens)
        single = {"value": us1, "unit": UNIT, "cores": 1,
                  "sample": f"first {n1} of {w.tokens} token rows, {dt1:.1f} s, fp64 numpy, 1 thread, "
                            f"scaled to a full call of {run.tokens} rows by tokens"}
        usn, cores, nn, dtn, rows = time_oracle_all_cores(w, run.tokens, dt1 / n1, args.cpu_seconds,
                                                          args.oracle_processes)
        line["cpu_baseline"] = {"value": usn, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": f"{nn} token rows in tasks of {rows} on {cores} processes, {dtn:.1f} s, "
                                          f"fp64 numpy, scaled to a full call of {run.tokens} rows by tokens",
                                "single_thread": single}
    if world == 1 and args.configs == "all" and w == I.WORKLOADS[DEFAULT_WORKLOAD] and args.tokens is None:
        line["configs"] = run_config_sweep(dev, status, args.config_steps, 5, peak)
        line["configs_note"] = ("every workload and variant at its full size, default launch shapes, "
                                f"{args.config_steps} calls each after 5 warm-up calls; frac = achieved / "
                                f"{peak_kind} hbm_gbs {peak:.1f} GB/s; kernel sources sha256 "
                                f"{kernel_source_hash()[:16]}")
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# every workload and variant, timed in the same run as the headline

# (workload, overrides): the five configurations the pages' kernels are
# quoted on and their table, pairing, dtype and launch-form variants, then
# the next rows (AdaLN scale/shift, VAE group norm + SiLU).  Consecutive
# entries with the same activation shape, dtype and seed share one drawn
# activation.
CONFIG_SWEEP = (
    ("tiny_256x24x64", {}),
    ("dense_4096x24x128", {}),
    ("dense_4096x24x128", {"dtype": "fp16"}),
    ("wan_32760x40x128", {}),
    ("wan_32760x40x128", {"rope_style": "rotate_half"}),
    ("wan_32760x40x128_bf16cos", {}),
    ("wan_32760x40x128_expanded", {}),
    ("wan_32760x40x128_expanded", {"rope_style": "rotate_half"}),
    ("wan_32760x40x128_expanded_bf16cos", {}),
    ("wan_32760x40x128_expanded_bf16cos", {"rope_style": "rotate_half"}),
    ("wan_32760x40x128_out_of_place", {}),
    ("flux2_2x4608x48x128", {}),
    ("flux2_2x4608x48x128_single_launch", {}),
    ("flux2_2x4608x48x128", {"dtype": "fp16"}),
    ("flux2_2x4608x48x128_single_launch", {"dtype": "fp16"}),
    ("adaln_flux2_2x4608x6144", {}),
    ("adaln_wan_32760x5120", {}),
    ("gn_vae_1x128x1024x1024", {}),
    ("gn_vae_1x256x512x512", {}),
    ("gn_vae_1x512x256x256", {}),
    ("gn_vae_1x512x128x128", {}),
)


# workloads also timed with plain launches (no programmatic dependent
# launch), beside the default entry
SWEEP_PLAIN_LAUNCH = ("dense_4096x24x128", "flux2_2x4608x48x128")


def sweep_entry_name(name: str, over: dict) -> str:
    return name + "".join(f"[{v}]" for v in over.values())


def _activation_key(w):
    if not isinstance(w, I.Workload):
        return None
    return (w.batch, w.seq, w.n_heads_q, w.n_heads_k, w.n_heads_v, w.head_dim, w.dtype, w.packed, w.scale,
            w.seed)


def time_steps(step, stream, steps: int, flush, dev) -> float:
    """Seconds per step: with `flush` (a buffer of twice the L2) each step
    follows a write of it and is timed by its own pair of CUDA events;
    without, the steps run back to back between one pair of events."""
    import torch

    if flush is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / 1e3 / steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush.fill_(1.0)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    return statistics.fmean(a.elapsed_time(b) for a, b in zip(starts, ends)) / 1e3


def copy_rate(bytes_moved: int, flush, stream, dev, steps: int) -> float:
    """GB/s of a device copy (torch copy_) that reads and writes
    `bytes_moved` in all, timed like the kernel it is set against."""
    import torch

    n = max(8, bytes_moved // 4)
    a = torch.ones(n, dtype=torch.bfloat16, device=dev)
    b = torch.empty_like(a)
    for _ in range(5):
        b.copy_(a)
    t = time_steps(lambda: b.copy_(a), stream, steps, flush, dev)
    moved = 2 * a.numel() * a.element_size()
    del a, b
    return moved / t / 1e9


def run_config_sweep(dev, status, steps: int, warmup: int, peak: float):
    """Time every entry of CONFIG_SWEEP once (default launch shapes).  An
    entry's step is one call of the workload: one launch, or for FLUX.2's
    separate tensors one launch per tensor (Q, then K) back to back.  Calls
    whose launches move under twice the L2 are flushed between calls and
    timed per call; larger ones run back to back."""
    import torch

    stream = torch.cuda.current_stream(dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 0) or 129 * 2 ** 20
    flush_buf = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)
    out = {}
    cache_key, cache_inp = None, None
    plan = []
    for name, over in CONFIG_SWEEP:
        plan.append((name, over, False))
        if not over and name in SWEEP_PLAIN_LAUNCH:
            plan.append((name, over, True))
    for name, over, plain in plan:
        base = I.WORKLOADS.get(name) or I.ADALN_WORKLOADS.get(name) or I.GN_WORKLOADS[name]
        w = base.with_(**over) if over else base
        inp = None
        key = _activation_key(w)
        if key is not None:
            if key != cache_key:
                cache_key, cache_inp = None, None
                cache_key, cache_inp = key, I.make_inputs(w)
            inp = dict(cache_inp)
            inp["cos"], inp["sin"] = I.rope_table(w)
        from diffusion_transformer_qk_gb300 import qknr as Q

        flags = dict(flags=Q.FLAG_NO_OVERLAP) if plain else {}
        if isinstance(w, I.GroupNormWorkload):
            run = GroupNormRunner(w, dev, dict(gn_mode="auto"), status)
        elif isinstance(w, I.AdaLNWorkload):
            run = AdaLNRunner(w, dev, flags, status)
        else:
            run = Runner(w, dev, flags, status, inp=inp)
        L = len(run.args)
        step_bytes = run.bytes_per_launch * L
        flush = flush_buf if run.bytes_per_launch < 2 * l2 else None
        for _ in range(warmup):
            run.step(stream)
        torch.cuda.synchronize(dev)
        t = time_steps(lambda: run.step(stream), stream, steps, flush, dev)
        achieved = step_bytes / t / 1e9
        copy = copy_rate(step_bytes, flush, stream, dev, min(steps, 100))
        info = run.info
        entry = {
            "us_per_call": t * 1e6, "launches_per_call": L * getattr(run, "launches_per_call", 1),
            "algorithmic_bytes": step_bytes, "achieved_gbs": achieved, "frac": achieved / peak,
            "same_size_copy_gbs": copy, "frac_of_same_size_copy": achieved / copy,
            "l2": ("flushed between calls (write of 2x L2), each call timed by its own pair of CUDA events"
                   if flush is not None else
                   "launches move more than 2x L2: calls back to back between one pair of CUDA events"),
            "dtype": w.dtype, "kernel": info["kernel"],
            "launch": {k: info[k] for k in ("grid", "block", "dyn_smem", "stages", "consumer_warps", "group_warps",
                                            "prefetch_rows", "registers") if k in info},
        }
        if isinstance(w, I.Workload):
            entry.update(cos_dtype=w.cos_dtype, cos_layout=w.cos_layout, rope=w.rope_style,
                         launch_form=(("packed, out of place (V copied)" if w.out_of_place else "packed, in place")
                                      if w.packed else ("q+k in one launch" if w.single_launch
                                                        else "one launch per tensor (Q, then K)")))
        if L > 1:
            entry["us_per_launch"] = t * 1e6 / L
        if flush is not None:
            # the same calls back to back without the flush: inputs partly
            # served from L2 across calls (the hot number; frac of the HBM
            # peak then overstates DRAM work and is not reported)
            t_hot = time_steps(lambda: run.step(stream), stream, steps, None, dev)
            entry["hot"] = {"us_per_call": t_hot * 1e6, "achieved_gbs": step_bytes / t_hot / 1e9,
                            "l2": "calls back to back, no flush"}
        if not over and not plain:
            # ncu DRAM bytes per launch, when the committed record is of these sources
            entry["traffic_per_launch"] = recorded_traffic(name)
        if not isinstance(w, I.GroupNormWorkload):
            entry["launch_mode"] = ("plain stream order" if plain else
                                    "programmatic dependent launch (the default)")
        st = int(status.item())
        if st != 0:
            raise RuntimeError(f"{name}: kernel reported status {st}")
        out[sweep_entry_name(name, over) + ("[plain launch]" if plain else "")] = entry
        del run
        torch.cuda.empty_cache()
    del flush_buf, cache_inp
    torch.cuda.empty_cache()
    return out


def run_copy_calibration(args):
    """A device copy (torch ``copy_``) of the same bytes as each workload
    size, timed the way the kernels are: per-launch CUDA events after an L2
    flush, and back to back.  The copy rate grows with size well past L2,
    so a kernel's fraction of a same-size copy separates its own overhead
    from the ramp-up and tail that any launch of that size pays."""
    import torch

    dev = torch.device("cuda", 0)
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 129 * 2 ** 20
    flush = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for mb in (25, 50, 113, 134, 268, 671, 1024):
        n = int(mb * 1e6) // 2
        a = torch.ones(n, dtype=torch.bfloat16, device=dev)
        b = torch.empty_like(a)
        for _ in range(5):
            b.copy_(a)
        times = []
        for _ in range(50):
            flush.fill_(1.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            b.copy_(a)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            times.append(e0.elapsed_time(e1) / 1e3)
        k = 200
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(k):
            b.copy_(a)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        moved = 2 * a.numel() * a.element_size()
        t_flush, t_b2b = statistics.median(times), e0.elapsed_time(e1) / 1e3 / k
        print(json.dumps({"copy_mb": mb, "bytes_moved": moved, "flushed_us": t_flush * 1e6,
                          "flushed_gbs": moved / t_flush / 1e9, "back_to_back_us": t_b2b * 1e6,
                          "back_to_back_gbs": moved / t_b2b / 1e9}), flush=True)
    return 0


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=5000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD,
                   choices=sorted(I.WORKLOADS) + sorted(I.ADALN_WORKLOADS) + sorted(I.GN_WORKLOADS))
    p.add_argument("--tokens", type=int, default=None,
                   help="run the first N token rows of the workload (small profiling cases)")
    p.add_argument("--ctas-per-sm", type=int, default=0)
    p.add_argument("--stages", type=int, default=0)
    p.add_argument("--consumer-warps", type=int, default=0)
    p.add_argument("--group-warps", type=int, default=0)
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--e2e-chunk-rows", type=int, default=2048)
    p.add_argument("--l2-flush", choices=["auto", "on", "off"], default="auto")
    p.add_argument("--dtype", choices=["bf16", "fp16"], default=None,
                   help="activation dtype of the workload (default: the workload's own, bf16)")
    p.add_argument("--no-overlap", action="store_true",
                   help="launch without programmatic dependent launch (plain stream order)")
    p.add_argument("--rope-style", choices=["interleaved", "rotate_half"], default=None,
                   help="QK workloads: pairing (default: the workload's own)")
    p.add_argument("--gn-mode", choices=["auto", "fused", "two_pass", "cluster"], default="auto",
                   help="group-norm workloads: which path to time")
    p.add_argument("--copy-calibration", action="store_true",
                   help="print the device copy rate at the workloads' sizes (one JSON line each) and exit")
    p.add_argument("--configs", choices=["all", "none"], default="all",
                   help="with the default workload on one GPU: also time every workload and variant "
                        "(the line's 'configs' object)")
    p.add_argument("--config-steps", type=int, default=300)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--oracle-processes", type=int, default=0,
                   help="worker processes of the all-core oracle timing (0 = every available core)")
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be >= 3")
    if args.copy_calibration:
        return run_copy_calibration(args)
    w = I.WORKLOADS.get(args.workload) or I.ADALN_WORKLOADS.get(args.workload) or I.GN_WORKLOADS[args.workload]
    if args.dtype and args.dtype != w.dtype:
        kw = {"dtype": args.dtype}
        if isinstance(w, I.AdaLNWorkload) and w.mod_dtype != "fp32":
            kw["mod_dtype"] = args.dtype                  # modulation rows in the activation dtype
        w = w.with_(**kw)
    if args.rope_style and isinstance(w, I.Workload) and args.rope_style != w.rope_style:
        w = w.with_(rope_style=args.rope_style)
    if args.impl == "reference":
        if not isinstance(w, I.Workload):
            p.error("--impl reference times the QK-norm + RoPE oracle; pick a QK workload")
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
