#!/usr/bin/env python
"""Benchmark of the FP4 indexer scorer (libfp4idx.so) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step is one pass of the scorer over one batch of synthetic input, through
the C ABI.  The default workload is the 4-row x 32-head verify decode over
16,384 MXFP4 keys on shuffled 64-key pages (SGLang PR 42861's benchmark
shape): per step the full logits [4, 16384] and the top-2048 of every row.
Other workloads: ``long_decode`` (16 requests x 4 rows over 100k/400k keys,
fused top-2048), ``tiny`` (4 rows x 8 heads over 1,024 keys).

Prints one JSON line.  ``value`` is query x key scores per second over all
ranks (a score is one (row, visible key) pair of the step), timed on the
device with CUDA events over K graph-replayed steps with the inputs already
in HBM; ``e2e`` repeats the measurement with the per-step inputs copied from
pinned host memory and the results read back inside the timed region.
``--impl reference`` times the CPU oracle on a bounded sample of the same
workload instead.  Multi-GPU runs (torchrun) are independent replicas.
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
sys.path.insert(0, ROOT)

METRIC = ("query×key scores/sec and µs/call; % of HBM BW (decode) / FP4 TC peak (prefill)")
UNIT = "scores/s"
L2_BYTES = 129 * 1024 * 1024

# DRAM bytes per launch from ncu captures, valid only for the kernel sources
# they were taken on (sha256 of the csrc/ files, first 16 hex digits).
RECORDED_TRAFFIC: dict = {
    # ncu --set full, one launch of the long-decode top-k scorer: read 282,581,248 B
    # + write 22,283,776 B.
    ("long_decode", "scorer_topk"): {"sha": "556025c8954f9223", "bytes": 304865024},
}


def source_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fp4_sparse_attention_gb300", "csrc")
    for fn in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self) -> dict:
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower() in ("active", "1", "yes"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
WORKLOADS = {
    "verify16k": dict(maker="verify_decode_16k", k=2048, logits=True),
    "long_decode": dict(maker="long_batched_decode", k=2048, logits=False),
    "tiny": dict(maker="tiny_mx_decode", k=64, logits=True),
}


def kv_bytes_per_key(fmt: int) -> int:
    return 64 + (4 if fmt == 0 else 8)


def visible_pairs(p) -> int:
    import oracle

    return int(oracle.visible_all(p).sum())


def make_host_problem(name: str):
    from fp4_sparse_attention_gb300 import workloads as wl

    return getattr(wl, WORKLOADS[name]["maker"])()


_CUDART = None


def cudart():
    """The CUDA runtime torch loaded into this process (for event-record nodes)."""
    global _CUDART
    if _CUDART is None:
        import ctypes

        import torch

        torch.cuda.init()
        path = None
        with open("/proc/self/maps") as f:
            for line in f:
                if "libcudart.so" in line:
                    path = line.split()[-1]
                    break
        _CUDART = ctypes.CDLL(path) if path else False
    return _CUDART or None


def record_external(event, stream) -> bool:
    """Record `event` on `stream` as an event-record node when the stream is
    being captured (cudaEventRecordExternal), so it can be timed per replay."""
    import ctypes

    rt = cudart()
    if rt is None:
        return False
    rt.cudaEventRecordWithFlags.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]
    rt.cudaEventRecordWithFlags.restype = ctypes.c_int
    return rt.cudaEventRecordWithFlags(ctypes.c_void_p(event.cuda_event), ctypes.c_void_p(stream.cuda_stream),
                                       1) == 0


class OursBench:
    """Device-resident decode step: [logits] + top-k score + top-k merge, graph captured."""

    def __init__(self, host, spec, device):
        import torch

        from fp4_sparse_attention_gb300 import binding as B

        self.B, self.torch = B, torch
        self.host, self.spec, self.device = host, spec, device
        self.k = spec["k"]
        base = B.DeviceProblem.from_host(host, device=device)
        key_bytes = host.k.nbytes + host.k_scale.nbytes
        # Enough K-cache copies that a step never finds its keys in L2.
        self.copies = 1 if key_bytes >= 2 * L2_BYTES else int(min(512, -(-2 * L2_BYTES // key_bytes)))
        self.problems = [base]
        for _ in range(self.copies - 1):
            self.problems.append(B.DeviceProblem(
                format=base.format, num_heads=base.num_heads, num_kv_heads=base.num_kv_heads,
                page_size=base.page_size, q=base.q, q_scale=base.q_scale, k=base.k.clone(),
                k_scale=base.k_scale.clone(), cu_seqlens_q=base.cu_seqlens_q, cu_seqlens_k=base.cu_seqlens_k,
                block_table=base.block_table, page_offsets=base.page_offsets, visible_len=base.visible_len,
                causal=base.causal, qo_offset=base.qo_offset, max_seqlen_q=base.max_seqlen_q,
                max_seqlen_k=base.max_seqlen_k))
        T = base.num_rows
        self.w = torch.as_tensor(host.w).to(device)
        self.ld = (host.max_seqlen_k + 3) // 4 * 4
        self.logits = torch.empty((T, self.ld), dtype=torch.float32, device=device) if spec["logits"] else None
        self.idx = torch.empty((T, self.k), dtype=torch.int32, device=device)
        self.val = torch.empty((T, self.k), dtype=torch.float32, device=device)
        self.cnt = torch.empty((T,), dtype=torch.int32, device=device)
        self.ws = torch.empty((B.fp4idx_topk_workspace_bytes(base, self.k),), dtype=torch.uint8, device=device)
        self.kernels = (["scorer_logits"] if spec["logits"] else []) + ["scorer_topk", "topk_merge"]
        self.launches_per_step = len(self.kernels)
        self.graphs = []
        self.events = []

    def _calls(self, prob):
        B = self.B
        calls = []
        if self.logits is not None:
            calls.append(lambda: B.fp4idx_logits(prob, self.w, out=self.logits))
        calls.append(lambda: B.fp4idx_topk_score(prob, self.w, self.k, self.ws))
        calls.append(lambda: B.fp4idx_topk_merge(prob, self.k, self.idx, self.val, self.cnt, self.ws))
        return calls

    def _step(self, prob, evs=None):
        stream = self.torch.cuda.current_stream(self.device)
        ok = True
        if evs is not None:
            ok &= record_external(evs[0], stream)
        for i, call in enumerate(self._calls(prob)):
            call()
            if evs is not None:
                ok &= record_external(evs[i + 1], stream)
        return ok

    def capture(self):
        torch = self.torch
        s = torch.cuda.Stream(device=self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(s):
            for prob in self.problems[:2]:
                self._step(prob)
        torch.cuda.current_stream(self.device).wait_stream(s)
        torch.cuda.synchronize(self.device)
        self.timed_nodes = True
        for prob in self.problems:
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(self.launches_per_step + 1)]
            for e in evs:  # torch creates the CUDA event lazily, on its first record
                e.record(s)
            torch.cuda.synchronize(self.device)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self.timed_nodes &= self._step(prob, evs)
            self.graphs.append(g)
            self.events.append(evs)

    def run(self, j: int):
        self.graphs[j % len(self.graphs)].replay()

    def kernel_times_ms(self, used: int) -> dict:
        """Mean device time of each kernel of the step over the timed replays,
        from the event-record nodes inside the step graphs."""
        out = {name: [] for name in self.kernels}
        for evs in self.events[:used]:
            for n, name in enumerate(self.kernels):
                out[name].append(evs[n].elapsed_time(evs[n + 1]))
        return {name: float(np.mean(v)) for name, v in out.items() if v}

    def kernel_times_isolated_ms(self, reps: int = 64) -> dict:
        """Fallback when event nodes cannot be timed: each kernel of the step
        replayed back to back in single-kernel graphs over the input copies."""
        torch = self.torch
        res = {}
        for n, name in enumerate(self.kernels):
            graphs = []
            for prob in self.problems[:reps]:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    self._calls(prob)[n]()
                graphs.append(g)
            for g in graphs[:3]:
                g.replay()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(self.device)
            a.record()
            for j in range(reps):
                graphs[j % len(graphs)].replay()
            b.record()
            torch.cuda.synchronize(self.device)
            res[name] = a.elapsed_time(b) / reps
        return res

    # -- end to end: per-step inputs from pinned host memory, results read back
    def e2e(self, steps: int) -> dict:
        torch = self.torch
        B = self.B
        prob = self.problems[0]
        pin = lambda t: t.cpu().pin_memory()
        h_in = [pin(prob.q), pin(prob.q_scale), pin(self.w), pin(prob.block_table)]
        if prob.visible_len is not None:
            h_in.append(pin(prob.visible_len))
        d_in = [prob.q, prob.q_scale, self.w, prob.block_table] + (
            [prob.visible_len] if prob.visible_len is not None else [])
        d_out = [self.idx, self.val, self.cnt] + ([self.logits] if self.logits is not None else [])
        h_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in d_out]
        bi = sum(t.numel() * t.element_size() for t in h_in)
        bo = sum(t.numel() * t.element_size() for t in h_out)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(self.device)
        t0 = time.perf_counter()
        start.record()
        for _ in range(steps):
            for h, d in zip(h_in, d_in):
                d.copy_(h, non_blocking=True)
            if self.logits is not None:
                B.fp4idx_logits(prob, self.w, out=self.logits)
            B.fp4idx_topk(prob, self.w, self.k, indices=self.idx, values=self.val, valid_count=self.cnt,
                          workspace=self.ws)
            for h, d in zip(h_out, d_out):
                h.copy_(d, non_blocking=True)
        end.record()
        torch.cuda.synchronize(self.device)
        wall = time.perf_counter() - t0
        return {"ms": start.elapsed_time(end), "wall_s": wall, "h2d": bi, "d2h": bo}


def kernel_algorithmic_bytes(host, name: str, k: int) -> int:
    """Algorithmic HBM bytes of one launch: K codes + scales of every key a
    request can see (each read once), Q codes + scales, w, and the outputs."""
    import oracle

    vis = oracle.visible_all(host)
    keys = 0
    for b in range(host.num_seqs):
        r0, r1 = int(host.cu_seqlens_q[b]), int(host.cu_seqlens_q[b + 1])
        keys += int(vis[r0:r1].max()) if r1 > r0 else 0
    kv = keys * kv_bytes_per_key(host.format)
    T, H = host.q.shape[0], host.num_heads
    qb = host.q.nbytes + host.q_scale.nbytes + T * H * 4
    if name == "scorer_logits":
        return kv + qb + T * ((host.max_seqlen_k + 3) // 4 * 4) * 4
    if name == "scorer_topk":
        return kv + qb
    if name == "topk_merge":
        return T * k * 8 + T * 4
    raise KeyError(name)


def cpu_baseline(host, spec, budget_s: float = 10.0) -> dict:
    """The oracle on the host cores over a bounded sample: the last row of
    the first request, its full logits and its top-k, repeated for ~budget_s."""
    import oracle

    row = int(host.cu_seqlens_q[1]) - 1
    vis = oracle.visible(host, row)
    op = oracle.OracleProblem(host)
    reps, t0 = 0, time.perf_counter()
    while True:
        if spec["logits"]:
            oracle.logits_rows(op, vis, rows=[row])
        oracle.topk(op, spec["k"], rows=[row])
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    return {"value": reps * vis / el, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"row {row} ({vis} visible keys): full logits and top-{spec['k']}" if spec["logits"]
            else f"row {row} ({vis} visible keys): top-{spec['k']}", "seconds": round(el, 2), "reps": reps}


# ---------------------------------------------------------------------------
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def reduce_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def run_reference(args, world, rank):
    if rank != 0:
        return
    spec = WORKLOADS[args.workload]
    host = make_host_problem(args.workload)
    import oracle

    oracle.build()
    row = int(host.cu_seqlens_q[1]) - 1
    vis = oracle.visible(host, row)
    op = oracle.OracleProblem(host)

    def step():
        if spec["logits"]:
            oracle.logits_rows(op, vis, rows=[row])
        oracle.topk(op, spec["k"], rows=[row])

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    value = args.steps * vis / el
    sample = f"row {row} ({vis} visible keys) per step: " + ("full logits and " if spec["logits"] else "") + \
        f"top-{spec['k']}"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {**host.summary(), "sample": sample},
        "cpu_baseline": {"value": value, "unit": UNIT, "kind": "oracle", "cores": oracle.num_threads(),
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, world, rank, local):
    import torch

    from fp4_sparse_attention_gb300 import build as fbuild

    if not os.path.exists(os.path.join(ROOT, "fp4_sparse_attention_gb300", "libfp4idx.so")):
        fbuild.build()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    spec = WORKLOADS[args.workload]
    host = make_host_problem(args.workload)
    bench = OursBench(host, spec, device)
    bench.capture()
    pairs = visible_pairs(host)
    for j in range(args.warmup):
        bench.run(j)
    torch.cuda.synchronize(device)
    # ~1 s of untimed load so the clock sampler sees the GPU busy
    t0 = time.perf_counter()
    j = 0
    with ClockSampler(local) as clocks:
        while time.perf_counter() - t0 < 1.0:
            bench.run(j)
            j += 1
            if j % 64 == 0:
                torch.cuda.synchronize(device)
        torch.cuda.synchronize(device)
        barrier(world)
        torch.cuda.synchronize(device)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record()
        for j in range(args.steps):
            bench.run(j)
        end.record()
        torch.cuda.synchronize(device)
        barrier(world)
    ms = start.elapsed_time(end)
    ms_max = reduce_max(ms, world)
    kt_method = "event-record nodes inside the timed step graphs"
    try:
        if not bench.timed_nodes:
            raise RuntimeError("event-record nodes unavailable")
        kt = bench.kernel_times_ms(min(args.steps, len(bench.graphs)))
    except RuntimeError:
        kt = bench.kernel_times_isolated_ms()
        kt_method = "each kernel back to back in single-kernel graphs"
    value = world * args.steps * pairs / (ms_max * 1e-3)

    # e2e through the public call with host buffers
    e2e_steps = max(3, min(args.steps, 50))
    e2e = bench.e2e(e2e_steps)
    e2e_ms = reduce_max(e2e["ms"], world)

    peaks = measured_peaks()
    dominant = max(kt, key=lambda n: kt[n])
    alg = kernel_algorithmic_bytes(host, dominant, spec["k"])
    achieved = alg / (kt[dominant] * 1e-3) / 1e9
    sha = source_sha()
    rec = RECORDED_TRAFFIC.get((args.workload, dominant))
    traffic = rec["bytes"] if rec and rec["sha"] == sha else None
    line = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_max / args.steps,
        "us_per_call": 1e3 * ms_max / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp4-e2m1 x fp4-e2m1 -> fp32",
        "data": "synthetic",
        "config": {**host.summary(),
                   "step": ("logits + " if spec["logits"] else "") + f"top-{spec['k']} (score + merge)",
                   "scores_per_step": pairs,
                   "l2": (f"inputs rotated over {bench.copies} K-cache copies "
                          f"({bench.copies * (host.k.nbytes + host.k_scale.nbytes) / 2**20:.0f} MiB > 2x L2)"
                          if bench.copies > 1 else "K cache larger than 2x L2"),
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                     "algorithmic_bytes": alg, "launch_us": kt[dominant] * 1e3,
                     "peak_source": peaks["source"]},
        "kernels_us": {n: round(v * 1e3, 3) for n, v in kt.items()},
        "kernels_timing": kt_method,
        "e2e": {"value": world * e2e_steps * pairs / (e2e_ms * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "ms_per_step": e2e_ms / e2e_steps},
        "gpu_launches": args.steps * bench.launches_per_step,
        "clocks": clocks.summary(),
        "source_sha": sha,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle

        oracle.build()
        line["cpu_baseline"] = cpu_baseline(host, spec)
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="verify16k")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
