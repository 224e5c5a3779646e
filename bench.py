#!/usr/bin/env python
"""Throughput benchmark of one full error-feedback step on GB300.

Workload (default ``slab_2p31``): a flat fp32 slab of n = 2**31 gradient
elements per worker, W = 4 simulated workers on one GPU, Student-t(3) x 1e-3
gradients.  One step runs the whole hot path three times over the same
gradients, as the configuration asks:
  1. top-0.1 % error feedback with int32 indices for each worker, then the
     receive side (sum of the 4 packets into a dense G, SGD eta = 0.1);
  2. the same with bitmap-indexed packets (own residuals, own weights);
  3. 1-bit error feedback (beta1 = 0.9) for each worker, then the sign sum
     and SGD.
Units per step: 3 variants x W x n gradient elements.  ``value`` is in
G elements / s over all ranks.  Inputs (134 GB of state) are far larger than
the 129 MB L2, so no flush is needed between steps.

``--impl reference`` times the CPU oracle (numpy, one host core) on a bounded
sample of the same workload and prints the same line with
``"impl": "reference"``.  Under torchrun each rank runs its own replica
(the path needs no cross-GPU exchange); rank 0 prints.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "G grad elements/s per EF compress+apply step; HBM GB/s vs GB300 peak (1 GPU)"
UNIT = "G grad elements/s"

# DRAM traffic of one topk_fused launch from one ncu capture (--set full of
# the second launch of `bench.py --case topk --n 139460608`, the 32768-element
# tile form the slab uses; see profiles/): 1115.82 MB read + 510.79 MB
# written = 11.663 bytes per element.  Reported, scaled by n, only while the
# captured code still hashes to what was captured (the kernel's region of
# ef_topk.cu, from its staging struct to the end of the kernel, and the
# shared device header); otherwise null.  (Reads scale with n exactly; the
# writes fall short of 4 B per element by the dirty lines still in L2 when
# the captured launch ends, about 47 MB at this size, so the scaled figure
# slightly understates a full-size launch.)
FUSED_TRAFFIC_PER_ELEMENT = 11.663
FUSED_TRAFFIC_SOURCES = {
    # (file, first marker, end marker or None for the whole file): sha256
    ("error_feedback_gradient_gb300/csrc/ef_topk.cu", "struct FusedStage {",
     "// A segment's select list:"):
        "3753e85d6aa015f49e35a1dce9c4e04aa1c455146fca744b6913da4b58621f94",
    ("error_feedback_gradient_gb300/csrc/ef_common.cuh", None, None):
        "47c54bef91d740610d7262dd7a0102c11fdd086020fe4996e0643bfb02242e40",
}


def fused_traffic(n: int):
    import hashlib
    for (rel, first, end), digest in FUSED_TRAFFIC_SOURCES.items():
        try:
            with open(os.path.join(ROOT, rel), "rb") as f:
                src = f.read()
        except OSError:
            return None
        if first is not None:
            a, b = src.find(first.encode()), src.find(end.encode())
            if a < 0 or b < a:
                return None
            src = src[a:b]
        if hashlib.sha256(src).hexdigest() != digest:
            return None
    return FUSED_TRAFFIC_PER_ELEMENT * n


# ---------------------------------------------------------------------------
# distributed plumbing (replicas; barrier + max over ranks)
# ---------------------------------------------------------------------------


def dist_setup():
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not dist.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# the workload
# ---------------------------------------------------------------------------


class SlabStep:
    """State and launches of one full step of the slab workload."""

    def __init__(self, n: int, workers: int, dev):
        import torch
        from error_feedback_gradient_gb300 import workloads as wl
        import error_feedback_gradient_gb300 as efg
        self.efg, self.torch = efg, torch
        self.wl = wl.workload("slab_2p31", n)
        self.n, self.W, self.dev = n, workers, dev
        self.k = self.wl.total_k
        self.offs, self.ks = list(self.wl.seg_offsets), list(self.wl.seg_k)
        f32 = torch.float32
        nw = (n + 31) // 32
        self.g = [self.wl.gradient(w, 1, dev) for w in range(workers)]
        z = lambda: torch.zeros(n, dtype=f32, device=dev)   # noqa: E731
        self.e_int = [z() for _ in range(workers)]
        self.e_bm = [z() for _ in range(workers)]
        self.eps = [z() for _ in range(workers)]
        w0 = self.wl.weights(dev)
        self.w_int, self.w_bm, self.w_sign = w0, w0.clone(), w0.clone()
        self.G = torch.empty(n, dtype=f32, device=dev)
        self.vals_int = [torch.empty(self.k, dtype=f32, device=dev) for _ in range(workers)]
        self.idx_int = [torch.empty(self.k, dtype=torch.int32, device=dev) for _ in range(workers)]
        self.vals_bm = [torch.empty(self.k, dtype=f32, device=dev) for _ in range(workers)]
        self.bm = [torch.empty(nw, dtype=torch.int32, device=dev) for _ in range(workers)]
        self.bits = [torch.empty(nw, dtype=torch.int32, device=dev) for _ in range(workers)]
        u8 = torch.uint8
        self.ws_int = torch.empty(efg.topk_workspace_size(n, self.offs, self.ks, efg.IDX_INT32),
                                  dtype=u8, device=dev)
        self.ws_bm = torch.empty(efg.topk_workspace_size(n, self.offs, self.ks, efg.IDX_BITMAP),
                                 dtype=u8, device=dev)
        self.ws_ai = torch.empty(efg.aggregate_workspace_size(workers, efg.IDX_INT32, n),
                                 dtype=u8, device=dev)
        self.ws_ab = torch.empty(efg.aggregate_workspace_size(workers, efg.IDX_BITMAP, n),
                                 dtype=u8, device=dev)
        self.prof = None   # list of (kernel_id, start_event, stop_event) filled per launch
        self.streams = None

    def use_worker_streams(self):
        """Run each worker's three compress calls on a stream of its own, so
        that one worker's short selection and packing kernels overlap the
        other workers' streaming passes; the three aggregates stay on the
        caller's stream, each after the packets it reads.  Each worker gets
        its own top-k workspaces."""
        torch, efg = self.torch, self.efg
        u8 = torch.uint8
        self.streams = [torch.cuda.Stream() for _ in range(self.W)]
        self.ws_int_w = [self.ws_int] + [torch.empty_like(self.ws_int) for _ in range(self.W - 1)]
        self.ws_bm_w = [self.ws_bm] + [torch.empty_like(self.ws_bm) for _ in range(self.W - 1)]
        ev = lambda: [torch.cuda.Event() for _ in range(self.W)]   # noqa: E731
        self.ev_fork = torch.cuda.Event()
        self.ev_int, self.ev_bm, self.ev_sign = ev(), ev(), ev()
        del u8, efg

    # units and algorithmic bytes --------------------------------------------
    @property
    def units(self) -> int:
        return 3 * self.W * self.n

    def algorithmic_bytes(self) -> dict:
        n, W, k = self.n, self.W, self.k
        return {
            # read g_raw + e, write e (the fused pass) + packet write by the emit
            "topk_int32": W * (12 * n + 8 * k),
            "topk_bitmap": W * (12 * n + n / 8 + 4 * k),
            "sign": W * (12 * n + n / 8),
            # dense G write + packet reads + w read-modify-write where touched
            "aggregate_int32": 4 * n + 8 * W * k + 8 * W * k,
            "aggregate_bitmap": 4 * n + W * n / 8 + 4 * W * k + 8 * W * k,
            # w read + write, G write, W bit vectors
            "sign_apply": 12 * n + W * n / 8,
        }

    def _hook(self, kernel_id):
        if self.prof is None:
            return
        torch = self.torch
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        b.record()     # creates the events; the library re-records them
        self.efg.binding.profile_events(kernel_id, a, b)
        self.prof.append((kernel_id, a, b))

    def step(self):
        if self.streams is not None and self.prof is None:
            return self._step_streams()
        efg = self.efg
        for w in range(self.W):
            self._hook(efg.binding.KERNEL_TOPK_FUSED)
            efg.topk_compress(self.g[w], self.e_int[w], self.offs, self.ks, self.vals_int[w],
                              self.idx_int[w], None, self.ws_int, efg.IDX_INT32)
        self._hook(efg.binding.KERNEL_SPARSE_APPLY)
        efg.sparse_aggregate_apply(self.vals_int, self.idx_int, None, [self.k] * self.W, self.n,
                                   self.wl.eta, self.G, self.w_int, self.ws_ai, efg.IDX_INT32)
        for w in range(self.W):
            self._hook(efg.binding.KERNEL_TOPK_FUSED)
            efg.topk_compress(self.g[w], self.e_bm[w], self.offs, self.ks, self.vals_bm[w],
                              None, self.bm[w], self.ws_bm, efg.IDX_BITMAP)
        self._hook(efg.binding.KERNEL_SPARSE_APPLY)
        efg.sparse_aggregate_apply(self.vals_bm, None, self.bm, [self.k] * self.W, self.n,
                                   self.wl.eta, self.G, self.w_bm, self.ws_ab, efg.IDX_BITMAP)
        for w in range(self.W):
            self._hook(efg.binding.KERNEL_SIGN)
            efg.sign_compress(self.g[w], self.eps[w], self.wl.beta1, self.bits[w])
        self._hook(efg.binding.KERNEL_SIGN_APPLY)
        efg.sign_aggregate_apply(self.bits, self.n, efg.APPLY_SGD, self.wl.eta, self.wl.beta1,
                                 self.G, self.w_sign)

    def _step_streams(self):
        torch, efg = self.torch, self.efg
        main = torch.cuda.current_stream()
        self.ev_fork.record(main)
        for w, st in enumerate(self.streams):
            st.wait_event(self.ev_fork)
            with torch.cuda.stream(st):
                efg.topk_compress(self.g[w], self.e_int[w], self.offs, self.ks,
                                  self.vals_int[w], self.idx_int[w], None, self.ws_int_w[w],
                                  efg.IDX_INT32)
                self.ev_int[w].record(st)
                efg.topk_compress(self.g[w], self.e_bm[w], self.offs, self.ks, self.vals_bm[w],
                                  None, self.bm[w], self.ws_bm_w[w], efg.IDX_BITMAP)
                self.ev_bm[w].record(st)
                efg.sign_compress(self.g[w], self.eps[w], self.wl.beta1, self.bits[w])
                self.ev_sign[w].record(st)
        for ev in self.ev_int:
            main.wait_event(ev)
        efg.sparse_aggregate_apply(self.vals_int, self.idx_int, None, [self.k] * self.W, self.n,
                                   self.wl.eta, self.G, self.w_int, self.ws_ai, efg.IDX_INT32)
        for ev in self.ev_bm:
            main.wait_event(ev)
        efg.sparse_aggregate_apply(self.vals_bm, None, self.bm, [self.k] * self.W, self.n,
                                   self.wl.eta, self.G, self.w_bm, self.ws_ab, efg.IDX_BITMAP)
        for ev in self.ev_sign:
            main.wait_event(ev)
        efg.sign_aggregate_apply(self.bits, self.n, efg.APPLY_SGD, self.wl.eta, self.wl.beta1,
                                 self.G, self.w_sign)

    def clear_hooks(self):
        for kid in (1, 2, 3, 4):
            self.efg.binding.profile_events(kid, None, None)

    def check_status(self):
        extra = (self.ws_int_w[1:] + self.ws_bm_w[1:]) if self.streams is not None else []
        for ws in [self.ws_int, self.ws_bm, self.ws_ai, self.ws_ab] + extra:
            st = self.efg.workspace_status(ws)
            if st != 0:
                raise RuntimeError(f"device status {st}")


def oracle_step(g_list, n, k, eta, beta1, w0):
    """One full step of the slab workload by the CPU oracle (numpy) on
    host arrays; same three variants as SlabStep.step."""
    import numpy as np
    import oracle
    W = len(g_list)
    offs, ks = [0, n], [k]
    z = np.zeros(n, np.float32)
    pk = [oracle.topk_ef_step(g, z, offs, ks, "int32") for g in g_list]
    G = oracle.sparse_aggregate(pk, n)
    oracle.sgd_apply(w0, G, eta)
    pb = [oracle.topk_ef_step(g, z, offs, ks, "bitmap") for g in g_list]
    G = oracle.sparse_aggregate(pb, n)
    oracle.sgd_apply(w0, G, eta)
    bits = [oracle.sign_ef_step(g, z, beta1)[0] for g in g_list]
    G = oracle.sign_aggregate(bits, n)
    oracle.sgd_apply(w0, G, eta)
    return 3 * W * n


def oracle_sample_inputs(sample_n: int, workers: int, device="cpu"):
    from error_feedback_gradient_gb300 import workloads as wl
    w = wl.workload("slab_2p31", sample_n)
    g = [w.gradient(i, 1, device).cpu().numpy() for i in range(workers)]
    return g, w.total_k, w.eta, w.beta1, w.weights(device).cpu().numpy()


def time_oracle(sample_n: int, workers: int, repeats: int = 1):
    g, k, eta, beta1, w0 = oracle_sample_inputs(sample_n, workers)
    units = 0
    t0 = time.perf_counter()
    for _ in range(repeats):
        units += oracle_step(g, sample_n, k, eta, beta1, w0)
    dt = time.perf_counter() - t0
    return units, dt, k


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------


def run_reference(args, rank, world):
    """CPU oracle as the reference arm: each step is one oracle step on a
    bounded sample of the workload (sample_n elements per worker)."""
    if rank != 0:
        return
    sample_n = args.ref_sample
    g, k, eta, beta1, w0 = oracle_sample_inputs(sample_n, args.workers)
    for _ in range(args.warmup):
        oracle_step(g, sample_n, k, eta, beta1, w0)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(g, sample_n, k, eta, beta1, w0)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    units = 3 * args.workers * sample_n * args.steps
    value = units / total / 1e9
    sample = (f"{args.workers} workers x {sample_n} elements (k = {k}, 0.1 %) per step, "
              "all three variants, numpy on one host core")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload_desc, "n": args.n, "workers": args.workers,
                   "reference_sample_elements_per_worker": sample_n},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample, "host_cpus": os.cpu_count()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def run_ours(args, rank, world, local):
    import torch
    import error_feedback_gradient_gb300 as efg

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    efg.library()
    s = SlabStep(args.n, args.workers, dev)
    if args.worker_streams == "on":
        s.use_worker_streams()
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        s.step()
    torch.cuda.synchronize()
    s.check_status()

    # timed region: K steps between barriers + synchronize, CUDA events
    clocks = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    launches0 = efg.kernel_launches()
    barrier()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record()
    for _ in range(args.steps):
        s.step()
    ev1.record()
    torch.cuda.synchronize()
    barrier()
    launches = efg.kernel_launches() - launches0
    clk = clocks.stop() if clocks else None
    ms = ev0.elapsed_time(ev1) / args.steps
    ms_max = max_over_ranks(ms)
    value = world * s.units / (ms_max * 1e-3) / 1e9

    # per-kernel times from the profiling hook (same stream, same work)
    s.prof = []
    for _ in range(args.prof_steps):
        s.step()
    torch.cuda.synchronize()
    per = {}
    for kid, a, b in s.prof:
        per.setdefault(kid, []).append(a.elapsed_time(b))
    s.prof = None
    s.clear_hooks()
    s.check_status()
    ab = s.algorithmic_bytes()
    peak, peak_kind = load_peaks()
    n = s.n
    kernels = {}
    names = {1: "topk_fused", 2: "sign_compress", 4: "sign_aggregate_apply"}
    kb = {1: 12 * n, 2: 12.125 * n, 4: ab["sign_apply"]}
    # the step calls sparse_aggregate_apply twice, int32 packets then bitmap
    # packets; the hook records them in that order
    if 3 in per:
        ts = per.pop(3)
        for i, fmt in enumerate(("int32", "bitmap")):
            names[30 + i] = f"sparse_aggregate_apply_{fmt}"
            kb[30 + i] = ab[f"aggregate_{fmt}"]
            per[30 + i] = ts[i::2]
    for kid, ts in per.items():
        avg = statistics.mean(ts)
        d = {"launches_per_step": len(ts) // max(1, args.prof_steps), "avg_ms": avg}
        if kb.get(kid):
            d["algorithmic_bytes"] = kb[kid]
            d["achieved_gbs"] = kb[kid] / (avg * 1e-3) / 1e9
            d["frac_of_peak"] = d["achieved_gbs"] / load_peaks()[0]
        if kid in (30, 31):
            d["note"] = "the apply kernel alone; the run-boundary pass before it is not timed"
        kernels[names[kid]] = d
    top = kernels["topk_fused"]
    roofline = {"bound": "hbm", "kernel": "topk_fused",
                "achieved": top["achieved_gbs"], "peak": peak, "unit": "GB/s",
                "frac": top["achieved_gbs"] / peak, "peak_source": peak_kind,
                "traffic": (args.traffic_per_launch if args.traffic_per_launch is not None
                            else fused_traffic(n)),
                "algorithmic_bytes_per_launch": 12 * n}
    step_bytes = sum(ab.values())

    # end to end through the public API with host buffers
    e2e = run_e2e(args, s) if args.e2e_steps > 0 else None

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload_desc, "n": args.n, "workers": args.workers,
                   "k": s.k, "variants": ["topk_int32", "topk_bitmap", "sign_1bit"],
                   "units_per_step": s.units, "parallelism": "replicas",
                   "schedule": ("compress calls on one stream per worker, aggregates on the "
                                "caller's stream; per-kernel times from a serial step"
                                if args.worker_streams == "on" else "one stream"),
                   "l2": "inputs larger than L2 (no flush)"},
        "step_hbm": {"algorithmic_bytes": step_bytes,
                     "gbs": step_bytes / (ms_max * 1e-3) / 1e9,
                     "frac_of_peak": step_bytes / (ms_max * 1e-3) / 1e9 / peak},
        "roofline": roofline, "kernels": kernels,
        "cpu_baseline": None, "e2e": e2e, "clocks": clk,
        "gpu_launches": launches,
    }
    del s
    torch.cuda.empty_cache()
    if args.extras and rank == 0:
        line["per_config"] = run_extras(args, dev)
        line["next_rows"] = run_next(args, dev)
    # the CPU oracle baseline last (rank 0, N = 1 only), after the GPU legs,
    # so its host allocations cannot disturb the pinned-memory uploads
    if rank == 0 and world == 1 and args.baseline_sample > 0:
        units, dt, k = time_oracle(args.baseline_sample, args.workers)
        line["cpu_baseline"] = {
            "value": units / dt / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": (f"one oracle step on {args.workers} workers x {args.baseline_sample} "
                       f"elements (k = {k}), all three variants, {dt:.1f} s"),
            "host_cpus": os.cpu_count()}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_e2e(args, s):
    """Same metric through the public API with host buffers.  Every step
    copies each worker's gradient from pinned host memory, runs the step and
    reads the step's compressed packets back (int32 packets, bitmap packets,
    sign bits).  The copies run on their own streams and are double
    buffered, as a user overlapping input upload with compute would do: the
    gradients of step t+1 upload while step t computes, and step t's packets
    download while step t+1's gradients upload.  Each worker's gradient
    uploads on a stream of its own: on some hosts one stream's host-to-device
    copy reaches only a third of what concurrent copies reach.  The timed
    region spans the first upload to the last download (CUDA events)."""
    import torch
    host_g = []
    for t in s.g:
        h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        h.copy_(t)
        host_g.append(h)
    sets = [s.g, [torch.empty_like(t) for t in s.g]]
    outs = s.vals_int + s.idx_int + s.vals_bm + s.bm + s.bits
    host_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs]
    h2d = sum(t.numel() * t.element_size() for t in host_g)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    ups = [torch.cuda.Stream() for _ in host_g]
    down = torch.cuda.Stream()
    main = torch.cuda.current_stream()
    K = args.e2e_steps

    def run(steps):
        copied = [[torch.cuda.Event() for _ in host_g] for _ in range(2)]
        computed = [torch.cuda.Event() for _ in range(2)]
        downloaded = torch.cuda.Event()

        def upload(b):
            for up, dst, src, ev in zip(ups, sets[b], host_g, copied[b]):
                with torch.cuda.stream(up):
                    up.wait_event(computed[b])   # the set's previous reader is done
                    dst.copy_(src, non_blocking=True)
                    ev.record(up)

        for b in range(2):
            computed[b].record(main)
        upload(0)
        for t in range(steps):
            b = t % 2
            if t + 1 < steps:
                upload(1 - b)
            for ev in copied[b]:
                main.wait_event(ev)
            if t > 0:
                main.wait_event(downloaded)      # packets of step t-1 are read back
            s.g = sets[b]
            s.step()
            computed[b].record(main)
            with torch.cuda.stream(down):
                down.wait_event(computed[b])
                for dst, src in zip(host_out, outs):
                    dst.copy_(src, non_blocking=True)
                downloaded.record(down)
        main.wait_event(downloaded)

    def run_serial(steps):
        for t in range(steps):
            for dst, src in zip(sets[0], host_g):
                dst.copy_(src, non_blocking=True)
            s.g = sets[0]
            s.step()
            for dst, src in zip(host_out, outs):
                dst.copy_(src, non_blocking=True)

    if args.e2e_mode == "serial":
        run = run_serial        # noqa: F811
    run(2)
    torch.cuda.synchronize()
    barrier()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    run(K)
    b.record()
    torch.cuda.synchronize()
    barrier()
    s.g = sets[0]
    ms = max_over_ranks(a.elapsed_time(b) / K)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    return {"value": world * s.units / (ms * 1e-3) / 1e9, "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "mode": args.e2e_mode}


def run_extras(args, dev):
    """The other configurations, timed briefly with CUDA events (context for
    the main line; each is also a parity test case), each with one step of
    the CPU oracle timed on one host core beside it (``cpu_oracle``)."""
    import numpy as np
    import torch
    import error_feedback_gradient_gb300 as efg
    from error_feedback_gradient_gb300 import workloads as wl
    import oracle   # the CPU-baseline leg of each configuration only
    out = {}

    def oracle_time(fn):
        t0 = time.perf_counter()
        fn()
        return time.perf_counter() - t0

    def cpu_line(units, dt, sample):
        return {"g_elems_per_s": units / dt / 1e9, "seconds": dt, "cores": 1,
                "kind": "oracle", "sample": sample}

    def timed(fn, reps):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    # top-k single tensor 2^20 (W = 1, + aggregate + SGD)
    w = wl.workload("topk_2p20")
    g = w.gradient(0, 1, dev)
    e = torch.zeros_like(g)
    v = torch.empty(w.total_k, device=dev)
    i = torch.empty(w.total_k, dtype=torch.int32, device=dev)
    ws = torch.empty(efg.topk_workspace_size(w.n, w.seg_offsets, w.seg_k), dtype=torch.uint8,
                     device=dev)
    wa = torch.empty(efg.aggregate_workspace_size(1, 0, w.n), dtype=torch.uint8, device=dev)
    G = torch.empty_like(g)
    wt = w.weights(dev)

    def c1():
        efg.topk_compress(g, e, w.seg_offsets, w.seg_k, v, i, None, ws)
        efg.sparse_aggregate_apply([v], [i], None, [w.total_k], w.n, w.eta, G, wt, wa)
    ms = timed(c1, 50)
    # the same step replayed from a CUDA graph (launch overhead removed)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        c1()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        c1()
    ms_graph = timed(graph.replay, 50)
    g_np, w_np = g.cpu().numpy(), wt.cpu().numpy()

    def o1():
        pk = oracle.topk_ef_step(g_np, np.zeros(w.n, np.float32), w.seg_offsets, w.seg_k)
        oracle.sgd_apply(w_np, oracle.sparse_aggregate([pk], w.n), w.eta)
    dt = oracle_time(o1)
    out["topk_2p20"] = {"ms_per_step": ms, "g_elems_per_s": w.n / ms / 1e6,
                        "ms_per_step_cuda_graph": ms_graph,
                        "note": "L2-resident and launch-bound",
                        "cpu_oracle": cpu_line(w.n, dt, "one whole step (compress, receive "
                                               "side, SGD)")}
    del g, e, v, i, ws, wa, G, wt, g_np, w_np

    # 1-bit on 2^24 with the momentum
    w = wl.workload("sign_2p24")
    g = w.gradient(0, 1, dev)
    eps = torch.zeros_like(g)
    m = torch.zeros_like(g)
    bits = torch.empty((w.n + 31) // 32, dtype=torch.int32, device=dev)

    def c2():
        efg.sign_compress(g, eps, w.beta1, bits)
        efg.sign_aggregate_apply([bits], w.n, efg.APPLY_MOMENTUM, 0.0, w.beta1, None, m)
    ms = timed(c2, 50)
    g_np = g.cpu().numpy()

    def o2():
        z = np.zeros(w.n, np.float32)
        b, _ = oracle.sign_ef_step(g_np, z, w.beta1)
        oracle.onebit_momentum(z, oracle.decode_signs(b, w.n), w.beta1)
    dt = oracle_time(o2)
    out["sign_2p24"] = {"ms_per_step": ms, "g_elems_per_s": w.n / ms / 1e6,
                        "gbs": (12.125 + 8.125) * w.n / ms / 1e6,
                        "cpu_oracle": cpu_line(w.n, dt, "one whole step (1-bit compress, "
                                               "momentum)")}
    del g, eps, m, bits, g_np

    # layerwise ResNet-50
    w = wl.workload("resnet50")
    g = w.gradient(0, 1, dev)
    e = torch.zeros_like(g)
    v = torch.empty(w.total_k, device=dev)
    i = torch.empty(w.total_k, dtype=torch.int32, device=dev)
    ws = torch.empty(efg.topk_workspace_size(w.n, w.seg_offsets, w.seg_k), dtype=torch.uint8,
                     device=dev)

    def c3():
        efg.topk_compress(g, e, w.seg_offsets, w.seg_k, v, i, None, ws)
    ms = timed(c3, 30)
    g_np = g.cpu().numpy()
    dt = oracle_time(lambda: oracle.topk_ef_step(g_np, np.zeros(w.n, np.float32),
                                                 w.seg_offsets, w.seg_k))
    out["resnet50"] = {"ms_per_step": ms, "g_elems_per_s": w.n / ms / 1e6,
                       "gbs": (12 * w.n + 8 * w.total_k) / ms / 1e6,
                       "cpu_oracle": cpu_line(w.n, dt, "one whole layerwise step (161 "
                                              "tensors)")}
    del g, e, v, i, ws, g_np

    # BERT-large flat, 8 workers + aggregate
    w = wl.workload("bert_large")
    gs = [w.gradient(k, 1, dev) for k in range(w.workers)]
    es = [torch.zeros_like(gs[0]) for _ in range(w.workers)]
    vs = [torch.empty(w.total_k, device=dev) for _ in range(w.workers)]
    idx = [torch.empty(w.total_k, dtype=torch.int32, device=dev) for _ in range(w.workers)]
    wss = [torch.empty(efg.topk_workspace_size(w.n, w.seg_offsets, w.seg_k),
                       dtype=torch.uint8, device=dev) for _ in range(w.workers)]
    wa = torch.empty(efg.aggregate_workspace_size(w.workers, 0, w.n), dtype=torch.uint8,
                     device=dev)
    G = torch.empty_like(gs[0])
    wt = w.weights(dev)
    # as the main step: each worker's compress on a stream of its own when
    # --worker-streams is on, the aggregate after all of them
    streams = ([torch.cuda.Stream() for _ in range(w.workers)]
               if args.worker_streams == "on" else None)
    fork = torch.cuda.Event()
    done = [torch.cuda.Event() for _ in range(w.workers)]

    def c4():
        main = torch.cuda.current_stream()
        fork.record(main)
        for k in range(w.workers):
            st = streams[k] if streams else main
            st.wait_event(fork)
            with torch.cuda.stream(st):
                efg.topk_compress(gs[k], es[k], w.seg_offsets, w.seg_k, vs[k], idx[k], None,
                                  wss[k])
                done[k].record(st)
        for ev in done:
            main.wait_event(ev)
        efg.sparse_aggregate_apply(vs, idx, None, [w.total_k] * w.workers, w.n, w.eta, G, wt, wa)
    ms = timed(c4, 10)
    bytes_ = w.workers * (12 * w.n + 8 * w.total_k) + 4 * w.n + 16 * w.workers * w.total_k
    # oracle: one worker's compress in full, then the receive side of the
    # eight packets the GPU produced (the oracle's apply takes them as input)
    g_np = gs[0].cpu().numpy()
    packets = [{"indices": t.cpu().numpy(), "values": u.cpu().numpy()} for t, u in zip(idx, vs)]
    w_np = wt.cpu().numpy()
    t_c = oracle_time(lambda: oracle.topk_ef_step(g_np, np.zeros(w.n, np.float32),
                                                  w.seg_offsets, w.seg_k))
    t_a = oracle_time(lambda: oracle.sgd_apply(w_np, oracle.sparse_aggregate(packets, w.n),
                                               w.eta))
    dt = w.workers * t_c + t_a
    out["bert_large"] = {"ms_per_step": ms, "g_elems_per_s": w.workers * w.n / ms / 1e6,
                         "gbs": bytes_ / ms / 1e6,
                         "schedule": "stream per worker" if streams else "one stream",
                         "cpu_oracle": dict(cpu_line(w.workers * w.n, dt,
                                                     f"one worker's compress timed ({t_c:.1f} s) "
                                                     f"and counted {w.workers} times, plus the "
                                                     f"receive side of {w.workers} packets "
                                                     f"({t_a:.1f} s)"))}
    return out


def run_next(args, dev):
    """The widened rows beyond the step, each timed at the slab size (one
    worker, 2^31 elements, top-0.1 %) with CUDA events, with the oracle timed
    beside it on a sample."""
    import numpy as np
    import torch
    import error_feedback_gradient_gb300 as efg
    from error_feedback_gradient_gb300 import workloads as wl
    import oracle   # the CPU-baseline leg of each row only
    out = {}

    def timed(fn, reps):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    n = args.n
    k = wl.k_from_ratio(n, 1, 1000)
    offs, ks = [0, n], [k]
    g = wl.student_t3(n, 1e-3, wl.seed(5, 0, 1), dev)
    e = torch.zeros_like(g)
    v = torch.empty(k, device=dev)
    idx = torch.empty(k, dtype=torch.int32, device=dev)
    ws = torch.empty(efg.topk_workspace_size(n, offs, ks), dtype=torch.uint8, device=dev)
    ms_plain = timed(lambda: efg.topk_compress(g, e, offs, ks, v, idx, None, ws), 5)
    del ws

    # 8-bit packet values
    q = torch.empty(k, dtype=torch.int8, device=dev)
    sc = torch.empty(1, device=dev)
    wsq = torch.empty(efg.topk_q8_workspace_size(n, offs, ks), dtype=torch.uint8, device=dev)
    ms_q8 = timed(lambda: efg.topk_compress_q8(g, e, offs, ks, q, sc, idx, None, wsq), 5)
    ms_dq = timed(lambda: efg.q8_dequantize(q, sc, ks, v), 20)
    del wsq
    sample = 1 << 22
    rng = np.random.default_rng(3)
    gs = (rng.standard_t(3, sample) * 1e-3).astype(np.float32)
    es = np.zeros(sample, np.float32)
    ksm = wl.k_from_ratio(sample, 1, 1000)
    t0 = time.perf_counter()
    oracle.topk_q8_ef_step(gs, es, [0, sample], [ksm])
    dt = time.perf_counter() - t0
    q_bytes = 17 * k   # max pass 4 B, quantise pass 4 + 4 + 1 + 4 B per entry
    out["topk_q8"] = {
        "workload": f"one tensor of {n} elements, k = {k} (top-0.1 %), int32 indices",
        "ms_topk_compress": ms_plain, "ms_topk_compress_q8": ms_q8,
        "ms_q8_passes": ms_q8 - ms_plain,
        "q8_pass_algorithmic_bytes": q_bytes,
        "q8_pass_gbs": q_bytes / ((ms_q8 - ms_plain) * 1e-3) / 1e9 if ms_q8 > ms_plain else None,
        "note": "the quantiser's residual write is one scattered 4-byte store per entry",
        "ms_q8_dequantize": ms_dq, "dequantize_gbs": 5 * k / (ms_dq * 1e-3) / 1e9,
        "g_elems_per_s": n / ms_q8 / 1e6,
        "cpu_baseline": {"g_elems_per_s": sample / dt / 1e9, "cores": 1, "kind": "oracle",
                         "sample": f"one oracle step on {sample} elements, k = {ksm}"}}
    del g, e, v, q, sc

    # index codecs on the packet of the last top-k call (k ascending indices)
    codecs = {"local16": efg.CODEC_LOCAL16, "runvarint": efg.CODEC_RUNVARINT,
              "block256": efg.CODEC_BLOCK256}
    enc_o = {"local16": oracle.encode_local16, "runvarint": oracle.encode_runvarint,
             "block256": oracle.encode_block256}
    idx_sample = np.sort(rng.choice(sample, ksm, replace=False)).astype(np.int64)
    rows = {}
    for name, codec in codecs.items():
        mb, wb = efg.index_codec_sizes(codec, k, n)
        buf = torch.empty((mb + 3) // 4, dtype=torch.int32, device=dev)
        ob = torch.zeros(1, dtype=torch.int64, device=dev)
        wsc = torch.empty(wb, dtype=torch.uint8, device=dev)
        back = torch.empty(k, dtype=torch.int32, device=dev)
        ms_enc = timed(lambda: efg.index_encode(codec, idx, n, buf, ob, wsc), 10)
        nbytes = int(ob.item())
        ms_dec = timed(lambda: efg.index_decode(codec, buf, nbytes, k, n, back, wsc), 10)
        ok = bool(torch.equal(back, idx)) and efg.workspace_status(wsc) == 0
        t0 = time.perf_counter()
        enc_o[name](idx_sample, sample)
        dt = time.perf_counter() - t0
        rows[name] = {
            "stream_bytes": nbytes, "bytes_per_index": nbytes / k,
            "ms_encode": ms_enc, "ms_decode": ms_dec,
            "encode_gbs": (4 * k + nbytes) / (ms_enc * 1e-3) / 1e9,
            "decode_gbs": (4 * k + nbytes) / (ms_dec * 1e-3) / 1e9,
            "round_trip_exact": ok,
            "cpu_baseline": {"indices_per_s": ksm / dt, "cores": 1, "kind": "oracle",
                             "sample": f"oracle encode of {ksm} indices from {sample}"}}
        del buf, ob, wsc, back
    out["index_codecs"] = {"workload": f"the int32 packet of one tensor of {n} elements, "
                                       f"k = {k} (4 bytes per index as int32)",
                           "codecs": rows}
    del idx
    torch.cuda.empty_cache()

    # random magnitude-proportional sparsification (expected k)
    g = wl.student_t3(n, 1e-3, wl.seed(5, 0, 1), dev)
    e = torch.zeros_like(g)
    cap = 2 * k
    v = torch.empty(cap, device=dev)
    ix = torch.empty(cap, dtype=torch.int32, device=dev)
    cnt = torch.empty(2, dtype=torch.int64, device=dev)
    wsr = torch.empty(efg.randk_workspace_size(n, offs, ks), dtype=torch.uint8, device=dev)
    stepno = [0]

    def rk():
        stepno[0] += 1
        efg.randk_compress(g, e, offs, ks, 2024, stepno[0], v, ix, cnt, wsr)
    ms_rk = timed(rk, 5)
    kept = int(cnt[-1].item())
    rk_bytes = 12 * n + 8 * kept
    gs2 = (rng.standard_t(3, sample) * 1e-3).astype(np.float32)
    t0 = time.perf_counter()
    oracle.randk_ef_step(gs2, np.zeros(sample, np.float32), [0, sample], [ksm], 1, 1, 2 * ksm)
    dt = time.perf_counter() - t0
    out["random_sparsification"] = {
        "workload": f"one tensor of {n} elements, expected k = {k}",
        "ms_per_call": ms_rk, "kept_last_call": kept,
        "algorithmic_bytes": rk_bytes,
        "note": "algorithmic: 12 B/element (read g_raw and e, write e) + 8 B per kept "
                "element; the draws ride on the one pass over g at a sampled upper bound of "
                "the coefficient, and the candidate and keep bits add 1/4 B/element",
        "gbs": rk_bytes / (ms_rk * 1e-3) / 1e9,
        "g_elems_per_s": n / ms_rk / 1e6,
        "cpu_baseline": {"g_elems_per_s": sample / dt / 1e9, "cores": 1, "kind": "oracle",
                         "sample": f"one oracle step on {sample} elements, k = {ksm}"}}
    del g, e, v, ix, cnt, wsr
    torch.cuda.empty_cache()
    return out


def run_exchange(args, rank, world, local):
    """The exchanged step (--exchange): one worker per rank, each with its own
    gradient of n elements; per step a top-0.1 % int32 compress, then the
    packet exchange across the ranks (all-gather of the packets, or the
    index-range reduce-scatter) and the receive side with SGD.  Units per
    step: world x n gradient elements.  With one process a world-size-1
    group is created, so the collectives still run."""
    import socket
    import torch
    import torch.distributed as dist
    import error_feedback_gradient_gb300 as efg
    from error_feedback_gradient_gb300 import exchange as ex
    from error_feedback_gradient_gb300 import workloads as wl

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if not dist.is_initialized():
        with socket.socket() as sk:
            sk.bind(("127.0.0.1", 0))
            port = sk.getsockname()[1]
        dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0,
                                world_size=1)
    n = args.n
    wk = wl.workload("slab_2p31", n)
    k = wk.total_k
    offs, ks = list(wk.seg_offsets), list(wk.seg_k)
    g = wk.gradient(rank, 1, dev)
    e = torch.zeros_like(g)
    vals = torch.empty(k, device=dev)
    idx = torch.empty(k, dtype=torch.int32, device=dev)
    ws = torch.empty(efg.topk_workspace_size(n, offs, ks), dtype=torch.uint8, device=dev)
    x = ex.Exchange(n, k, efg.IDX_INT32)
    w = torch.empty(ex.padded_length(n, world), device=dev)
    w[:n].copy_(wk.weights(dev))
    G = torch.empty(n if args.exchange == "allgather" else x.s, device=dev)

    def step():
        efg.topk_compress(g, e, offs, ks, vals, idx, None, ws)
        if args.exchange == "allgather":
            x.allgather_apply(vals, idx, wk.eta, G, w[:n])
        else:
            x.range_apply(vals, idx, wk.eta, w, G)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    dist.barrier()
    launches0 = efg.kernel_launches()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        step()
    b.record()
    torch.cuda.synchronize()
    dist.barrier()
    ms = max_over_ranks(a.elapsed_time(b) / args.steps)
    if efg.workspace_status(ws) != 0:
        raise RuntimeError("top-k device status")
    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": world * n / (ms * 1e-3) / 1e9, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": (f"exchanged step: one worker per rank, n={n} "
                                    f"Student-t(3)x1e-3, top-0.1% int32 (k={k}), "
                                    f"{args.exchange} exchange, receive side + SGD eta="
                                    f"{wk.eta}"),
                       "exchange": args.exchange, "parallelism": f"dp{world}",
                       "l2": "inputs larger than L2 (no flush)"},
            "gpu_launches": efg.kernel_launches() - launches0}), flush=True)


def run_case(args):
    """One entry point alone, three calls, for profiling its kernels in
    isolation (--case): 'topk' (one tensor of n elements, top-0.1 %),
    'aggregate' (4 workers' int32 packets of 0.1 % over n, with G and SGD),
    'randk' (random sparsification of one tensor, expected 0.1 %), 'resnet50'
    (the layerwise top-k step over the 161 ResNet-50 gradient tensors),
    'topk_2p20' (the 2^20-element top-1 % step with its receive side), 'sign'
    (1-bit compression of 4 workers' gradients of n elements, then their
    sign aggregate with G and SGD), 'q8' (top-0.1 % with 8-bit values, then
    the receiver's dequantisation) or 'codec' (a top-0.1 % packet of n
    elements encoded and decoded with each index codec)."""
    import torch
    import error_feedback_gradient_gb300 as efg
    from error_feedback_gradient_gb300 import workloads as wl
    dev = torch.device("cuda", 0)
    n = args.n
    k = wl.k_from_ratio(n, 1, 1000)
    if args.case == "topk":
        g = wl.student_t3(n, 1e-3, 1, dev)
        e = wl.normal(n, 1e-4, 2, dev)
        v = torch.empty(k, device=dev)
        ix = torch.empty(k, dtype=torch.int32, device=dev)
        ws = torch.empty(efg.topk_workspace_size(n, [0, n], [k]), dtype=torch.uint8, device=dev)
        for _ in range(3):
            efg.topk_compress(g, e, [0, n], [k], v, ix, None, ws)
    elif args.case == "aggregate":
        W = 4
        gen = torch.Generator(device=dev)
        gen.manual_seed(1)
        stride = n // k
        base = torch.arange(k, device=dev, dtype=torch.int64) * stride
        ix = [torch.sort(base + torch.randint(0, stride, (k,), device=dev, generator=gen))
              .values.to(torch.int32) for _ in range(W)]
        vals = [torch.randn(k, device=dev, generator=gen) * 1e-3 for _ in range(W)]
        G = torch.empty(n, device=dev)
        w = torch.zeros(n, device=dev)
        ws = torch.empty(efg.aggregate_workspace_size(W, efg.IDX_INT32, n), dtype=torch.uint8,
                         device=dev)
        for _ in range(3):
            efg.sparse_aggregate_apply(vals, ix, None, [k] * W, n, 0.1, G, w, ws)
    elif args.case == "topk_2p20":
        w = wl.workload("topk_2p20")
        n, k = w.n, w.total_k
        g = w.gradient(0, 1, dev)
        e = torch.zeros_like(g)
        v = torch.empty(k, device=dev)
        ix = torch.empty(k, dtype=torch.int32, device=dev)
        ws = torch.empty(efg.topk_workspace_size(n, w.seg_offsets, w.seg_k), dtype=torch.uint8,
                         device=dev)
        wa = torch.empty(efg.aggregate_workspace_size(1, efg.IDX_INT32, n), dtype=torch.uint8,
                         device=dev)
        G = torch.empty_like(g)
        wt = w.weights(dev)
        for _ in range(3):
            efg.topk_compress(g, e, w.seg_offsets, w.seg_k, v, ix, None, ws)
            efg.sparse_aggregate_apply([v], [ix], None, [k], n, w.eta, G, wt, wa)
    elif args.case == "resnet50":
        w = wl.workload("resnet50")
        n, k = w.n, w.total_k
        g = w.gradient(0, 1, dev)
        e = torch.zeros_like(g)
        v = torch.empty(k, device=dev)
        ix = torch.empty(k, dtype=torch.int32, device=dev)
        ws = torch.empty(efg.topk_workspace_size(n, w.seg_offsets, w.seg_k), dtype=torch.uint8,
                         device=dev)
        for _ in range(3):
            efg.topk_compress(g, e, w.seg_offsets, w.seg_k, v, ix, None, ws)
    elif args.case == "randk":
        g = wl.student_t3(n, 1e-3, 1, dev)
        e = torch.zeros_like(g)
        v = torch.empty(2 * k, device=dev)
        ix = torch.empty(2 * k, dtype=torch.int32, device=dev)
        cnt = torch.empty(2, dtype=torch.int64, device=dev)
        ws = torch.empty(efg.randk_workspace_size(n, [0, n], [k]), dtype=torch.uint8, device=dev)
        for step in range(3):
            efg.randk_compress(g, e, [0, n], [k], 7, step, v, ix, cnt, ws)
    elif args.case == "sign":
        W = 4
        g = wl.student_t3(n, 1e-3, 1, dev)
        eps = torch.zeros_like(g)
        bits = [torch.empty((n + 31) // 32, dtype=torch.int32, device=dev) for _ in range(W)]
        G = torch.empty(n, device=dev)
        w = torch.zeros(n, device=dev)
        for _ in range(3):
            for b in bits:
                efg.sign_compress(g, eps, 0.9, b)
            efg.sign_aggregate_apply(bits, n, efg.APPLY_SGD, 0.1, 0.9, G, w)
    elif args.case == "q8":
        g = wl.student_t3(n, 1e-3, 1, dev)
        e = wl.normal(n, 1e-4, 2, dev)
        q = torch.empty(k, dtype=torch.int8, device=dev)
        sc = torch.empty(1, device=dev)
        ix = torch.empty(k, dtype=torch.int32, device=dev)
        v = torch.empty(k, device=dev)
        ws = torch.empty(efg.topk_q8_workspace_size(n, [0, n], [k]), dtype=torch.uint8,
                         device=dev)
        for _ in range(3):
            efg.topk_compress_q8(g, e, [0, n], [k], q, sc, ix, None, ws)
            efg.q8_dequantize(q, sc, [k], v)
    else:
        g = wl.student_t3(n, 1e-3, 1, dev)
        e = torch.zeros_like(g)
        v = torch.empty(k, device=dev)
        ix = torch.empty(k, dtype=torch.int32, device=dev)
        ws = torch.empty(efg.topk_workspace_size(n, [0, n], [k]), dtype=torch.uint8, device=dev)
        efg.topk_compress(g, e, [0, n], [k], v, ix, None, ws)
        back = torch.empty(k, dtype=torch.int32, device=dev)
        for _ in range(3):
            for codec in (efg.CODEC_LOCAL16, efg.CODEC_RUNVARINT, efg.CODEC_BLOCK256):
                mb, wb = efg.index_codec_sizes(codec, k, n)
                out = torch.empty((mb + 3) // 4, dtype=torch.int32, device=dev)
                ob = torch.zeros(1, dtype=torch.int64, device=dev)
                cws = torch.empty(wb, dtype=torch.uint8, device=dev)
                efg.index_encode(codec, ix, n, out, ob, cws)
                efg.index_decode(codec, out, int(ob.item()), k, n, back, cws)
                if not torch.equal(back, ix):
                    raise SystemExit(f"codec {codec}: round trip differs")
    torch.cuda.synchronize()
    status = 0 if args.case == "sign" else efg.workspace_status(ws)
    print(json.dumps({"case": args.case, "n": n, "k": k, "status": status}))


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--n", type=int, default=1 << 31, help="elements per worker")
    p.add_argument("--workers", type=int, default=4)
    p.add_argument("--prof-steps", type=int, default=2)
    p.add_argument("--e2e-steps", type=int, default=8)
    p.add_argument("--worker-streams", choices=["on", "off"], default="on",
                   help="on: each worker's compress calls on a stream of its own; "
                        "off: the whole step on one stream")
    p.add_argument("--e2e-mode", choices=["pipelined", "serial"], default="pipelined",
                   help="pipelined: uploads double-buffered against compute on their own "
                        "streams; serial: upload, step, download in turn")
    p.add_argument("--baseline-sample", type=int, default=1 << 27,
                   help="elements per worker in the timed oracle sample (0: skip)")
    p.add_argument("--ref-sample", type=int, default=1 << 21,
                   help="elements per worker in one reference-arm step")
    p.add_argument("--traffic-per-launch", type=float, default=None,
                   help="DRAM bytes of one topk_fused launch at this size, from ncu")
    p.add_argument("--no-extras", dest="extras", action="store_false")
    p.add_argument("--exchange", choices=["allgather", "range"], default=None,
                   help="time the exchanged step instead: one worker per rank, top-k, "
                        "packet exchange across the ranks, receive side")
    p.add_argument("--case", choices=["topk", "aggregate", "randk", "resnet50", "topk_2p20",
                                       "sign", "q8", "codec"],
                   default=None,
                   help="run one entry point alone (three calls at --n) for profiling")
    args = p.parse_args(argv)
    if args.case:
        run_case(args)
        return
    args.workload_desc = (f"slab_2p31: flat fp32 slab n={args.n} per worker, W={args.workers}, "
                          "Student-t(3)x1e-3; top-0.1% int32 + bitmap EF and 1-bit EF "
                          "(beta1=0.9), each aggregated locally with SGD eta=0.1")
    rank, world, local = dist_setup()
    if args.exchange and args.impl == "ours":
        run_exchange(args, rank, world, local)
    elif args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
