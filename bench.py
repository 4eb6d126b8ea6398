#!/usr/bin/env python
"""Benchmark of the FP4 indexer scorer (libfp4idx.so) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step is one pass of the scorer over one batch of synthetic input, through
the C ABI.  The default workload is the causal prefill: 32,768 query rows
over 32,768 MXFP4 keys, 64 heads, the top-2048 of every row with full logits
never materialised (the largest single-GPU shape; its roofline is the FP4
tensor pipe).  Other workloads: ``verify16k`` (SGLang PR 42861's benchmark
shape: 4 rows x 32 heads over 16,384 keys, full logits + top-2048),
``long_decode`` (16 requests x 4 rows over 100k/400k keys, fused top-2048),
``block_scores`` (4 x 4,096 causal rows over 8,192 keys, Hq=32 / Hkv=4,
NVFP4: the [Hq, 64, T] block maxima), ``tiny`` (4 rows x 8 heads over 1,024
keys) and the ones listed in WORKLOADS.

Prints one JSON line.  ``value`` is query x key scores per second over all
ranks (a score is one (row, visible key) pair of the step, over all heads),
timed on the device with CUDA events over K graph-replayed steps with the
inputs already in HBM; ``e2e`` repeats the measurement with the per-step
inputs copied from pinned host memory and the results read back inside the
timed region.  ``--impl reference`` times the CPU oracle on a bounded sample
of the same workload instead.  Multi-GPU runs (torchrun) are independent
replicas.
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


def unit_of(spec) -> str:
    """The K-cache writer counts keys written; every other workload scores."""
    return "keys/s" if spec["kind"] == "store" else UNIT
L2_BYTES = 129 * 1024 * 1024

# DRAM bytes per launch from ncu captures, valid only for the kernel sources
# they were taken on (sha256 of the csrc/ files, first 16 hex digits).
RECORDED_TRAFFIC: dict = {
    # ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum (one pass), one launch of
    # the GQA NVFP4 block-score kernel: read 52,000,256 B + write 84,906,240 B (the
    # [32, 64, 16,384] fp32 scores).
    ("block_scores", "block_scores"): {"sha": "27c1a344977f94ff", "bytes": 136906496},
    ("block_topk", "block_scores"): {"sha": "27c1a344977f94ff", "bytes": 136906496},
    # ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum (one pass), one launch on
    # the full workload: read 157,189,376 B (inputs: q 142.6 MB, w 8.4 MB, K 2.2 MB) +
    # write 504,214,528 B (every CTA's candidates at or above its k-th bucket, for the merge).
    ("prefill", "scorer_topk"): {"sha": "27c1a344977f94ff", "bytes": 661403904},
    # the same for the long batched decode: read 290,656,256 B (272.1 MB of K) + write
    # 23,139,584 B (partial lists).
    ("long_decode", "scorer_topk"): {"sha": "27c1a344977f94ff", "bytes": 313795840},
    # the same, prefill 8k: read 39,348,736 B + write 64,539,136 B.
    ("prefill_8k", "scorer_topk"): {"sha": "27c1a344977f94ff", "bytes": 103887872},
}


def source_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fp4_sparse_attention_gb300", "csrc")
    for fn in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


# Dense FP4 : bf16 tensor throughput of the part's nominal figures (13.5 : 2.25
# PFLOP/s); the FP4 peak is the measured bf16 peak times this ratio.
FP4_PER_BF16 = 6.0


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


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
# kind "topk": [logits +] top-k score + merge; kind "block": block maxima;
# kind "logits": the full logits alone (the pages' own per-call measurement).
# bound: the roofline of the workload's scorer kernel.
WORKLOADS = {
    "verify16k": dict(maker="verify_decode_16k", kind="topk", k=2048, logits=True, fused=True, bound="hbm"),
    "long_decode": dict(maker="long_batched_decode", kind="topk", k=2048, logits=False, bound="hbm"),
    "long_decode_slots": dict(maker="long_batched_decode", kind="topk", k=2048, logits=False, bound="hbm",
                              slots=True),
    "block_scores": dict(maker="nvfp4_gqa_block_scores", kind="block", k=0, logits=False, bound="tensor"),
    "block_topk": dict(maker="nvfp4_gqa_block_scores", kind="block", k=0, block_k=16, logits=False,
                       bound="tensor"),
    "prefill": dict(maker="prefill_32k", kind="topk", k=2048, logits=False, bound="tensor"),
    "prefill_8k": dict(maker="prefill_8k", kind="topk", k=2048, logits=False, bound="tensor"),
    "tiny": dict(maker="tiny_mx_decode", kind="topk", k=64, logits=True, bound="hbm"),
    "store_k": dict(maker="kcache_write_1m", kind="store", k=0, logits=False, bound="hbm", tokens=1 << 20),
    "logits16k": dict(maker="verify_decode_16k", kind="logits", k=0, logits=True, bound="hbm"),
    "logits100k": dict(maker="verify_decode_100k", kind="logits", k=0, logits=True, bound="hbm"),
    "logits400k": dict(maker="verify_decode_400k", kind="logits", k=0, logits=True, bound="hbm"),
    # SGLang PR 42861's full call: bf16 queries quantised, the per-token slot
    # table turned into request metadata, fused-table logits
    "p1_paged16k": dict(maker="p1_paged_16k", kind="paged", k=0, logits=True, bound="hbm"),
    "p1_paged100k": dict(maker="p1_paged_100k", kind="paged", k=0, logits=True, bound="hbm"),
    "p1_paged400k": dict(maker="p1_paged_400k", kind="paged", k=0, logits=True, bound="hbm"),
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
    """Device-resident step, graph captured: [logits +] top-k score + merge, or
    the block maxima."""

    def __init__(self, host, spec, device):
        import torch

        from fp4_sparse_attention_gb300 import binding as B

        self.B, self.torch = B, torch
        self.host, self.spec, self.device = host, spec, device
        self.k = spec["k"]
        self.block = spec["kind"] == "block"
        self.store = spec["kind"] == "store"
        if spec["kind"] == "paged":
            self._init_paged()
            return
        base = B.DeviceProblem.from_host(host, device=device)
        T = base.num_rows
        self.w = None if host.w is None else torch.as_tensor(host.w).to(device)
        in_bytes = sum(t.numel() * t.element_size() for t in (base.q, base.q_scale, base.k, base.k_scale))
        if self.w is not None:
            in_bytes += self.w.numel() * 4
        self.input_bytes = in_bytes
        # Enough input copies (queries, keys, weights) that a step never finds them in L2.
        self.copies = 1 if in_bytes >= 2 * L2_BYTES else int(min(512, -(-2 * L2_BYTES // in_bytes)))
        self.problems, self.ws_list = [base], [self.w]
        for _ in range(self.copies - 1):
            self.problems.append(B.DeviceProblem(
                format=base.format, num_heads=base.num_heads, num_kv_heads=base.num_kv_heads,
                page_size=base.page_size, q=base.q.clone(), q_scale=base.q_scale.clone(), k=base.k.clone(),
                k_scale=base.k_scale.clone(), cu_seqlens_q=base.cu_seqlens_q, cu_seqlens_k=base.cu_seqlens_k,
                block_table=base.block_table, page_offsets=base.page_offsets, visible_len=base.visible_len,
                causal=base.causal, qo_offset=base.qo_offset, max_seqlen_q=base.max_seqlen_q,
                max_seqlen_k=base.max_seqlen_k))
            self.ws_list.append(None if self.w is None else self.w.clone())
        if self.store:
            # 2^20 tokens of bf16 keys (256 MB, larger than 2x L2) to distinct random slots
            g = torch.Generator(device="cpu").manual_seed(7)
            self.tokens = spec["tokens"]
            self.keys = (torch.randn((self.tokens, base.num_kv_heads, 128), generator=g) * 4).to(torch.bfloat16).to(device)
            cap = base.k.shape[0] * base.page_size
            self.slots = torch.randperm(cap, generator=g)[: self.tokens].to(torch.int32).to(device)
            self.kernels = ["store_k"]
        elif self.block:
            self.scores = torch.empty((base.num_heads, base.ktiles, T), dtype=torch.float32, device=device)
            self.kernels = ["block_scores"]
            self.block_k = spec.get("block_k", 0)
            if self.block_k:
                self.bidx = torch.empty((base.num_heads, T, self.block_k), dtype=torch.int32, device=device)
                self.bval = torch.empty((base.num_heads, T, self.block_k), dtype=torch.float32, device=device)
                self.bcnt = torch.empty((base.num_heads, T), dtype=torch.int32, device=device)
                self.kernels.append("block_topk")
        else:
            self.ld = (host.max_seqlen_k + 3) // 4 * 4
            self.logits = torch.empty((T, self.ld), dtype=torch.float32, device=device) if spec["logits"] else None
            self.idx = torch.empty((T, self.k), dtype=torch.int32, device=device)
            self.val = torch.empty((T, self.k), dtype=torch.float32, device=device)
            self.cnt = torch.empty((T,), dtype=torch.int32, device=device)
            self.ws = torch.empty((B.fp4idx_topk_workspace_bytes(base, self.k) if self.k > 0 else 0,),
                                  dtype=torch.uint8, device=device)
            if spec["kind"] == "logits":
                self.kernels = ["scorer_logits"]
            elif spec.get("fused"):
                # one call: scorer logits + per-row selection from them (two kernels)
                self.kernels = ["logits_topk"]
            else:
                self.kernels = (["scorer_logits"] if spec["logits"] else []) + ["scorer_topk", "topk_merge"]
            if spec.get("slots"):
                self.slots = torch.empty((T, self.k), dtype=torch.int32, device=device)
                self.kernels.append("topk_slots")
            self.launch_count = 2 if spec.get("fused") else len(self.kernels)
        self.launches_per_step = getattr(self, "launch_count", len(self.kernels))
        self.graphs = []
        self.events = []

    def _init_paged(self):
        """Per copy: bf16 queries, the fused table, req / req_table / lens and
        w as inputs; the quantised queries and the request metadata as the
        step's own intermediate buffers."""
        torch, B, host, device = self.torch, self.B, self.host, self.device
        T, H = host.num_rows, host.num_heads
        nb, cap = host.req_table.shape
        npg = (cap + host.page_size - 1) // host.page_size
        dev = lambda a: torch.as_tensor(a).to(device).contiguous()
        src = dict(qb=dev(host.q.view(np.int16)).view(torch.bfloat16), table=dev(host.k), req=dev(host.req),
                   rt=dev(host.req_table), lens=dev(host.visible_len), w=dev(host.w))
        self.input_bytes = sum(t.numel() * t.element_size() for t in src.values())
        self.copies = 1 if self.input_bytes >= 2 * L2_BYTES else int(min(512, -(-2 * L2_BYTES // self.input_bytes)))
        self.sets, self.problems = [], []
        for c in range(self.copies):
            st = dict(src) if c == 0 else {n: t.clone() for n, t in src.items()}
            st["codes"] = torch.empty((T, H, 64), dtype=torch.uint8, device=device)
            st["scales"] = torch.empty((T, H, 4), dtype=torch.uint8, device=device)
            st["cu_q"] = torch.empty((nb + 1,), dtype=torch.int32, device=device)
            st["cu_k"] = torch.empty((nb + 1,), dtype=torch.int32, device=device)
            st["bt"] = torch.empty((nb, npg), dtype=torch.int32, device=device)
            st["prob"] = B.DeviceProblem(
                format=host.format, num_heads=H, num_kv_heads=host.num_kv_heads, page_size=host.page_size,
                q=st["codes"], q_scale=st["scales"], k=st["table"], k_scale=None, kv_layout=B.KV_FUSED,
                cu_seqlens_q=st["cu_q"], cu_seqlens_k=st["cu_k"], block_table=st["bt"], visible_len=st["lens"],
                max_seqlen_q=T, max_seqlen_k=cap)
            self.sets.append(st)
            self.problems.append(st["prob"])
        self.ld = cap
        self.logits = torch.empty((T, cap), dtype=torch.float32, device=device)
        self.kernels = ["quantize_q", "token_table", "scorer_logits"]
        self.launches_per_step = 5  # the token table takes three kernels
        self.graphs, self.events = [], []

    def _paged_calls(self, st):
        B, host = self.B, self.host
        return [lambda: B.fp4idx_quantize_q(st["qb"], st["codes"], st["scales"]),
                lambda: B.fp4idx_pages_from_token_table(st["req"], st["rt"], host.page_size, host.k.shape[0],
                                                        out=(st["cu_q"], st["cu_k"], st["bt"])),
                lambda: B.fp4idx_logits(st["prob"], st["w"], out=self.logits)]

    def _calls(self, n):
        B = self.B
        if self.spec["kind"] == "paged":
            return self._paged_calls(self.sets[n])
        prob, w = self.problems[n], self.ws_list[n]
        if self.store:
            return [lambda: B.fp4idx_store_k(self.keys, self.slots, prob.page_size, prob.k, prob.k_scale)]
        if self.block:
            calls = [lambda: B.fp4idx_block_scores(prob, out=self.scores)]
            if self.block_k:
                calls.append(lambda: B.fp4idx_block_topk(self.scores, self.block_k, self.bidx, self.bval, self.bcnt))
            return calls
        if self.spec["kind"] == "logits":
            return [lambda: B.fp4idx_logits(prob, w, out=self.logits)]
        if self.spec.get("fused"):
            return [lambda: B.fp4idx_logits_topk(prob, w, self.k, logits=self.logits, indices=self.idx,
                                                 values=self.val, valid_count=self.cnt)]
        calls = []
        if self.logits is not None:
            calls.append(lambda: B.fp4idx_logits(prob, w, out=self.logits))
        calls.append(lambda: B.fp4idx_topk_score(prob, w, self.k, self.ws))
        calls.append(lambda: B.fp4idx_topk_merge(prob, self.k, self.idx, self.val, self.cnt, self.ws))
        if self.spec.get("slots"):
            calls.append(lambda: B.fp4idx_topk_slots(prob, self.idx, slots=self.slots))
        return calls

    def _step(self, n, evs=None):
        stream = self.torch.cuda.current_stream(self.device)
        ok = True
        if evs is not None:
            ok &= record_external(evs[0], stream)
        for i, call in enumerate(self._calls(n)):
            call()
            if evs is not None:
                ok &= record_external(evs[i + 1], stream)
        return ok

    def capture(self):
        torch = self.torch
        s = torch.cuda.Stream(device=self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(s):
            for n in range(min(2, len(self.problems))):
                self._step(n)
        torch.cuda.current_stream(self.device).wait_stream(s)
        torch.cuda.synchronize(self.device)
        # the timed graphs hold the step's kernels alone (event-record nodes
        # between them would break the programmatic-launch overlap of
        # consecutive kernels); a second set, with an event-record node after
        # every call, gives the per-kernel times
        self.timed_nodes = True
        for n in range(len(self.problems)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self._step(n)
            self.graphs.append(g)
        self.probe_graphs = []
        for n in range(min(len(self.problems), 64)):
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(self.kernels) + 1)]
            for e in evs:  # torch creates the CUDA event lazily, on its first record
                e.record(s)
            torch.cuda.synchronize(self.device)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self.timed_nodes &= self._step(n, evs)
            self.probe_graphs.append(g)
            self.events.append(evs)

    def run(self, j: int):
        self.graphs[j % len(self.graphs)].replay()

    def run_probes(self, steps: int) -> int:
        """Replay the instrumented graphs (inputs rotated as in the timed
        region); returns how many replays the event times cover."""
        used = min(steps, len(self.probe_graphs))
        for j in range(used):
            self.probe_graphs[j].replay()
        self.torch.cuda.synchronize(self.device)
        return used

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
            for c in range(min(reps, len(self.problems))):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    self._calls(c)[n]()
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
        if self.spec["kind"] == "paged":
            return self._e2e_paged(steps)
        prob = self.problems[0]
        d_in = [prob.q, prob.q_scale, prob.block_table] + ([self.w] if self.w is not None else []) + (
            [prob.visible_len] if prob.visible_len is not None else [])
        if self.store:
            d_in = [self.keys, self.slots]
        h_in = [t.cpu().pin_memory() for t in d_in]
        if self.store:
            d_out = [self.slots[:1]]  # completion marker (the cache is resident state)
        elif self.block:
            d_out = [self.scores] + ([self.bidx, self.bval, self.bcnt] if self.block_k else [])
        elif self.spec["kind"] == "logits":
            d_out = [self.logits]
        else:
            d_out = [self.idx, self.val, self.cnt] + ([self.logits] if self.logits is not None else []) + (
                [self.slots] if self.spec.get("slots") else [])
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
            if self.store:
                B.fp4idx_store_k(self.keys, self.slots, prob.page_size, prob.k, prob.k_scale)
            elif self.block:
                B.fp4idx_block_scores(prob, out=self.scores)
                if self.block_k:
                    B.fp4idx_block_topk(self.scores, self.block_k, self.bidx, self.bval, self.bcnt)
            elif self.spec["kind"] == "logits":
                B.fp4idx_logits(prob, self.w, out=self.logits)
            elif self.spec.get("fused"):
                B.fp4idx_logits_topk(prob, self.w, self.k, logits=self.logits, indices=self.idx, values=self.val,
                                     valid_count=self.cnt)
            else:
                if self.logits is not None:
                    B.fp4idx_logits(prob, self.w, out=self.logits)
                B.fp4idx_topk(prob, self.w, self.k, indices=self.idx, values=self.val, valid_count=self.cnt,
                              workspace=self.ws)
                if self.spec.get("slots"):
                    B.fp4idx_topk_slots(prob, self.idx, slots=self.slots)
            for h, d in zip(h_out, d_out):
                h.copy_(d, non_blocking=True)
        end.record()
        torch.cuda.synchronize(self.device)
        wall = time.perf_counter() - t0
        return {"ms": start.elapsed_time(end), "wall_s": wall, "h2d": bi, "d2h": bo}


    def _e2e_paged(self, steps: int) -> dict:
        """The PR's call from pinned host buffers: bf16 queries, req,
        req_table, lens and w copied in every step (the fused table is
        resident cache state), the logits read back."""
        torch = self.torch
        st = self.sets[0]
        d_in = [st["qb"], st["req"], st["rt"], st["lens"], st["w"]]
        h_in = [t.cpu().pin_memory() for t in d_in]
        h_out = torch.empty(self.logits.shape, dtype=self.logits.dtype, pin_memory=True)
        bi = sum(t.numel() * t.element_size() for t in h_in)
        bo = h_out.numel() * h_out.element_size()
        calls = self._paged_calls(st)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(self.device)
        t0 = time.perf_counter()
        start.record()
        for _ in range(steps):
            for h, d in zip(h_in, d_in):
                d.copy_(h, non_blocking=True)
            for call in calls:
                call()
            h_out.copy_(self.logits, non_blocking=True)
        end.record()
        torch.cuda.synchronize(self.device)
        return {"ms": start.elapsed_time(end), "wall_s": time.perf_counter() - t0, "h2d": bi, "d2h": bo}


def kernel_algorithmic_bytes(host, name: str, k: int) -> int:
    """Algorithmic HBM bytes of one launch.  Scorer kernels: the K codes +
    scales of every key a request can see (each read once per request), Q
    codes + scales and w -- the inputs only; what they write is reported
    apart (kernel_output_bytes).  Other kernels: what they read and write."""
    import oracle

    vis = oracle.visible_all(host)
    keys = 0
    for b in range(host.num_seqs):
        r0, r1 = int(host.cu_seqlens_q[b]), int(host.cu_seqlens_q[b + 1])
        keys += int(vis[r0:r1].max()) if r1 > r0 else 0
    kv = keys * kv_bytes_per_key(host.format) * host.num_kv_heads
    T, H = host.q.shape[0], host.num_heads
    # the scorer reads FP4 query codes and scales (bf16 queries: after quantisation)
    qcodes = T * H * (64 + (4 if host.format == 0 else 8))
    qb = qcodes + (T * H * 4 if host.w is not None else 0)
    if name in ("scorer_logits", "scorer_topk", "logits_topk", "block_scores"):
        return kv + qb
    if name == "quantize_q":  # bf16 queries read, codes + scales written
        return T * H * (256 + 68)
    if name == "token_table":  # req and the slot table read, metadata written
        nb, cap = host.req_table.shape
        return T * 4 + nb * cap * 4 + 2 * (nb + 1) * 4 + nb * ((cap + host.page_size - 1) // host.page_size) * 4
    if name == "topk_merge":
        return T * k * 8 + T * 4
    if name == "store_k":  # bf16 keys read, codes + scales written, per token and K head
        return k * host.num_kv_heads * (256 + 68) + k * 4
    if name == "topk_slots":  # positions read, one table entry gathered per position, slots written
        return T * k * 12
    if name == "block_topk":  # scores read once; indices, values, counts written
        bk = k or 16
        return H * ((host.max_seqlen_k + 127) // 128) * T * 4 + H * T * (bk * 8 + 4)
    raise KeyError(name)


def kernel_output_bytes(host, name: str, k: int) -> int:
    """Bytes a scorer launch writes (not part of its roofline bytes): full
    logits, the top-k (indices + values + counts) or the block maxima."""
    T, H = host.q.shape[0], host.num_heads
    ld = (host.max_seqlen_k + 3) // 4 * 4
    if name == "scorer_logits":
        return T * ld * 4
    if name == "logits_topk":
        return T * ld * 4 + T * k * 8 + T * 4
    if name == "block_scores":
        return H * ((host.max_seqlen_k + 127) // 128) * T * 4
    return 0


def kernel_algorithmic_flops(host) -> int:
    """FP4 tensor FLOPs of the visible part of the QK contraction:
    2 * 128 per (row, head, visible key)."""
    import oracle

    return int(oracle.visible_all(host).astype(np.int64).sum()) * host.num_heads * 2 * 128


def roofline(host, spec, name: str, launch_ms: float, step_ms: float, peaks: dict) -> dict:
    """Roofline of one kernel: the scorer kernels against the workload's bound
    (HBM bytes for decode, FP4 tensor FLOPs for prefill / block scores), the
    merge against HBM."""
    tensor = spec["bound"] == "tensor" and name in ("scorer_topk", "scorer_logits", "block_scores")
    if tensor:
        flops = kernel_algorithmic_flops(host)
        sustained = step_ms > 1.0  # a long step runs the tensor pipe at its power-capped rate
        bf16 = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
        peak = bf16 * FP4_PER_BF16
        achieved = flops / (launch_ms * 1e-3) / 1e12
        return {"bound": "tensor", "kernel": name, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": None, "algorithmic_flops": flops,
                "launch_us": launch_ms * 1e3,
                "peak_source": f"{peaks['source']} bf16 {'sustained' if sustained else 'burst'} "
                               f"{bf16:.1f} TFLOP/s x {FP4_PER_BF16:g} (nominal FP4/bf16 ratio)"}
    kk = spec.get("block_k", 0) if name == "block_topk" else (spec.get("tokens", 0) if name == "store_k" else spec["k"])
    alg = kernel_algorithmic_bytes(host, name, kk)
    achieved = alg / (launch_ms * 1e-3) / 1e9
    out = {"bound": "hbm", "kernel": name, "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
           "frac": achieved / peaks["hbm_gbs"], "traffic": None, "algorithmic_bytes": alg,
           "launch_us": launch_ms * 1e3, "peak_source": peaks["source"]}
    ob = kernel_output_bytes(host, name, kk)
    if ob:
        out["output_bytes"] = ob  # written by the launch, outside algorithmic_bytes and frac
    return out


def oracle_sample(host, spec):
    """One bounded unit of oracle work on the workload: the last row of the
    first request -- its full logits and top-k, or all its block maxima."""
    import oracle

    row = int(host.cu_seqlens_q[1]) - 1
    vis = oracle.visible(host, row)
    op = oracle.OracleProblem(host)
    if spec["kind"] == "store":
        n = 8192
        rng = np.random.default_rng(0)
        keys = (rng.standard_normal((n, host.num_kv_heads, 128)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        slots = rng.permutation(host.k.shape[0] * host.page_size)[:n].astype(np.int32)
        k, ks = host.k.copy(), host.k_scale.copy()

        def step():
            oracle.store_k(keys, slots, host.page_size, k, ks)
        return step, n, f"{n} keys quantized and written"
    if spec["kind"] == "block":
        bk = spec.get("block_k", 0)

        def step():
            sc, _, _ = oracle.block_scores(op, host.ktiles, rows=[row])
            if bk:
                oracle.block_topk(sc, bk)
        what = f"row {row} ({vis} visible keys): its block maxima for all {host.num_heads} heads" + \
            (f" and their top-{bk} blocks" if bk else "")
    elif spec["kind"] in ("logits", "paged"):
        def step():
            oracle.logits_rows(op, vis, rows=[row])
        what = f"row {row} ({vis} visible keys): its full logits" + (
            " (bf16 queries, per-token slot table, fused table)" if spec["kind"] == "paged" else "")
    else:
        def step():
            if spec["logits"]:
                oracle.logits_rows(op, vis, rows=[row])
            oracle.topk(op, spec["k"], rows=[row])
        what = f"row {row} ({vis} visible keys): " + ("full logits and " if spec["logits"] else "") + \
            f"top-{spec['k']}"
    return step, vis, what


def cpu_baseline(host, spec, budget_s: float = 10.0) -> dict:
    """The oracle on the host cores over a bounded sample (oracle_sample),
    repeated for ~budget_s."""
    import oracle

    step, vis, what = oracle_sample(host, spec)
    reps, t0 = 0, time.perf_counter()
    while True:
        step()
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    return {"value": reps * vis / el, "unit": unit_of(spec), "cores": oracle.num_threads(), "kind": "oracle",
            "sample": what, "seconds": round(el, 2), "reps": reps}


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
    step, vis, what = oracle_sample(host, spec)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    value = args.steps * vis / el
    sample = what + " per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit_of(spec), "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {**host.summary(), "sample": sample},
        "cpu_baseline": {"value": value, "unit": unit_of(spec), "kind": "oracle", "cores": oracle.num_threads(),
                         "sample": sample},
        "e2e": {"value": value, "unit": unit_of(spec), "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
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
    pairs = spec["tokens"] if spec["kind"] == "store" else visible_pairs(host)
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
    kt_method = "event-record nodes after every call, in copies of the step graphs replayed after the timed region"
    try:
        if not bench.timed_nodes:
            raise RuntimeError("event-record nodes unavailable")
        kt = bench.kernel_times_ms(bench.run_probes(max(args.steps, 16)))
    except RuntimeError:
        kt = bench.kernel_times_isolated_ms()
        kt_method = "each kernel back to back in single-kernel graphs"
    value = world * args.steps * pairs / (ms_max * 1e-3)

    # e2e through the public call with host buffers
    e2e_steps = max(3, min(args.steps, 50))
    e2e = bench.e2e(e2e_steps)
    e2e_ms = reduce_max(e2e["ms"], world)

    peaks = measured_peaks()
    step_ms = ms_max / args.steps
    dominant = max(kt, key=lambda n: kt[n])
    roof = roofline(host, spec, dominant, kt[dominant], step_ms, peaks)
    sha = source_sha()
    rec = RECORDED_TRAFFIC.get((args.workload, dominant))
    roof["traffic"] = rec["bytes"] if rec and rec["sha"] == sha else None
    if spec["kind"] == "store":
        step_desc = f"MXFP4 K-cache write of {spec['tokens']} bf16 keys to random slots"
    elif spec["kind"] == "block":
        step_desc = f"block maxima [{host.num_heads}, {host.ktiles}, {host.q.shape[0]}]" + \
            (f" + top-{spec['block_k']} blocks per (head, row)" if spec.get("block_k") else "")
    elif spec["kind"] == "logits":
        step_desc = f"full logits [{host.q.shape[0]}, {(host.max_seqlen_k + 3) // 4 * 4}] (no top-k)"
    elif spec["kind"] == "paged":
        step_desc = (f"bf16 queries quantised + per-token slot table to request metadata + full logits "
                     f"[{host.q.shape[0]}, {host.req_table.shape[1]}] from the fused table")
    elif spec.get("fused"):
        step_desc = f"logits + top-{spec['k']} in one call (scorer logits, per-row selection from them)"
    else:
        step_desc = ("logits + " if spec["logits"] else "") + f"top-{spec['k']} (score + merge)" + (
            " + physical slots" if spec.get("slots") else "")
    line = {
        "metric": METRIC,
        "value": value,
        "unit": unit_of(spec),
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": step_ms,
        "us_per_call": 1e3 * step_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp4-e2m1 x fp4-e2m1 -> fp32",
        "data": "synthetic",
        "config": {**host.summary(),
                   "topk": spec["k"],
                   **({"block_topk": spec["block_k"]} if spec.get("block_k") else {}),
                   "step": step_desc,
                   "scores_per_step": pairs,
                   "l2": (f"inputs (q, k, scales, w) rotated over {bench.copies} copies "
                          f"({bench.copies * bench.input_bytes / 2**20:.0f} MiB > 2x L2)"
                          if bench.copies > 1 else
                          f"inputs ({bench.input_bytes / 2**20:.0f} MiB) larger than 2x L2"),
                   "parallelism": f"replicas x{world}"},
        "roofline": roof,
        "kernels_roofline": {n: {"bound": r["bound"], "frac": round(r["frac"], 4), "achieved": round(r["achieved"], 1),
                                 "unit": r["unit"]}
                             for n in kt for r in [roofline(host, spec, n, kt[n], step_ms, peaks)]},
        "kernels_us": {n: round(v * 1e3, 3) for n, v in kt.items()},
        "kernels_timing": kt_method,
        "e2e": {"value": world * e2e_steps * pairs / (e2e_ms * 1e-3), "unit": unit_of(spec),
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
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="prefill")
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
