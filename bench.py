"""Benchmark: one decode step of a llama.cpp-style serving engine over a
quantized KV cache -- quantize-on-append of the new token(s) into the cache,
then split-K decode attention over the whole packed cache (den_llama.cpp:
Q4_G64 KV cache, 32K..196K context).

Default workload: 1 sequence, 24 query heads / 4 kv heads, head_dim 256,
Q4_G64 K and V, 32,767 cached tokens + 1 appended (attention over 32,768),
fp16 inputs (the "gqa32k" workload of workloads/).  ``--config`` selects
another workload by index.

Metric: decode-attention KV-read GB/s = packed K+V bytes of all attended
tokens per step / step time, plus microseconds per generated token.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl ours|reference]

The same JSON line carries, under ``also``, the attention measurements of the
other long-context workloads (196,608 keys, the 16-sequence MTP verify batch,
the mixed q8_0-K pair at 65,536 keys), taken the same way in the same run.

``--impl reference`` times the CPU oracle (fp64 attention over the dequantized
cache) on the host cores, on the same workload.  Under torchrun each rank runs
an independent replica (the work is data-parallel across sequences; there is
no data exchange), the step time is the max over ranks and ``value`` is the
sum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "decode-attention KV GB/s (fraction of HBM peak) and us/token at 32K/196K ctx"
L2_BYTES = 129 * 1024 * 1024


def _dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError, TypeError):      # no file, not JSON, no or bad entry
        return 6800.0, "fallback"


def _bf16_peak():
    """The measured dense bf16 burst rate (TFLOP/s): the peak of an fp16 tensor
    contraction timed alone (fp16 and bf16 run at the same nominal rate)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, ValueError, KeyError, TypeError):
        return 1900.0, "fallback"


# The sources of the kernels the committed captures profile (the decode
# kernels and the merge) and of their launch (split policy, tensor maps).
_PROFILED_SOURCES = ("kvq_api.cu", "kvq_decode_common.cuh", "kvq_decode_tc.cu", "kvq_decode_tc.cuh",
                     "kvq_decode_warp.cu", "kvq_internal.cuh", "kvq_merge.cu", "kvq_ptx.cuh", "kvq_tensor_map.cu")


def _kernel_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "quantized_kv_cache_q4_gb300", "csrc")
    for name in _PROFILED_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def _traffic(config_name: str):
    """DRAM bytes per launch of the attention call from the committed ncu
    summary, if it was taken on the kernel sources as they are now."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
        e = t.get(config_name)
        if e and e.get("kernel_hash") == _kernel_hash():
            return e["dram_bytes_per_launch"]
    except (OSError, ValueError, KeyError):                  # no capture recorded for these sources
        pass
    return None


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            self.path = os.path.join("/tmp", f"kvq_clocks_{os.getpid()}.csv")
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:                                       # no nvidia-smi: no clock record
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.out.close()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def reduce_max(x: float, dist, device) -> float:
    """Max of a per-rank scalar over all ranks (identity without a process group)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_rank: int, ms_max: float, world: int) -> float:
    """Whole-job throughput: every rank moves bytes_per_rank per step; the job's
    step time is the slowest rank's."""
    return world * bytes_per_rank / (ms_max * 1e-3) / 1e9


def oracle_step_time(wl, k_or, v_or, n_threads):
    """One step of the oracle: quantize-append the new tokens, then fp64
    attention over the whole cache.  Returns seconds."""
    import oracle
    t0 = time.perf_counter()
    oracle.quantize_append(k_or, wl.k_new, wl.cached_len)
    oracle.quantize_append(v_or, wl.v_new, wl.cached_len)
    oracle.decode_attention(k_or, v_or, wl.q, wl.kv_len, wl.spec.scale, n_threads=n_threads)
    return time.perf_counter() - t0


def oracle_caches(wl, append=False):
    import oracle
    sp = wl.spec
    k = oracle.Cache(sp.k_codec, sp.n_seq, sp.n_kv_heads, sp.head_dim, wl.capacity)
    v = oracle.Cache(sp.v_codec, sp.n_seq, sp.n_kv_heads, sp.head_dim, wl.capacity)
    for s in range(sp.n_seq):
        L = int(wl.cached_len[s])
        for c, src in ((k, wl.k_prefill), (v, wl.v_prefill)):
            qs, sc = oracle.quantize(c.codec, np.ascontiguousarray(src[s].transpose(1, 0, 2)))
            c.qs[s, :, :L] = qs
            c.scales[s, :, :L] = sc
    return k, v


def cpu_threads() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):                        # not available on this platform
        return os.cpu_count() or 1


def oracle_threads() -> int:
    """Threads the oracle runs with on all host cores: one per core, spread over
    (sequence, kv head, query row) items."""
    return cpu_threads()


def time_oracle(wl, k, v, threads, budget_s, max_steps):
    """Mean seconds of whole oracle steps, repeated until about budget_s."""
    n, total = 0, 0.0
    while (n == 0 or total < budget_s) and n < max_steps:
        total += oracle_step_time(wl, k, v, threads)
        n += 1
    return total / n, n, total


def cpu_baseline(wl, kv_bytes, budget_s=10.0, max_steps=1000):
    """The oracle timed on the host cores, single-threaded and on all cores."""
    import oracle
    oracle.build()
    k, v = oracle_caches(wl)
    host = cpu_threads()
    threads = oracle_threads()
    t1, n1, tot1 = time_oracle(wl, k, v, 1, budget_s, max_steps)
    tn, nn, totn = time_oracle(wl, k, v, threads, budget_s, max_steps)
    step = f"full {wl.spec.name} steps (append + fp64 attention over {int(wl.kv_len.sum())} tokens)"
    return {"value": round(kv_bytes / tn / 1e9, 4), "unit": "GB/s", "cores": threads, "host_cores": host,
            "threads": threads, "kind": "oracle",
            "sample": f"{nn} {step} on {threads} threads, {totn:.1f} s",
            "single_thread": {"value": round(kv_bytes / t1 / 1e9, 4), "unit": "GB/s", "threads": 1,
                              "sample": f"{n1} {step} on 1 thread, {tot1:.1f} s"},
            "all_cores": {"value": round(kv_bytes / tn / 1e9, 4), "unit": "GB/s", "threads": threads}}


def run_reference(args, wl, kv_bytes):
    """The oracle timed on the host cores: each step is the full workload step."""
    import oracle
    oracle.build()
    k, v = oracle_caches(wl)
    threads = oracle_threads()
    for _ in range(args.warmup):
        oracle_step_time(wl, k, v, threads)
    times = [oracle_step_time(wl, k, v, threads) for _ in range(args.steps)]
    t = sum(times) / len(times)
    val = kv_bytes / t / 1e9
    sample = f"full {wl.spec.name} step (append + fp64 attention over {int(wl.kv_len.sum())} tokens) x {args.steps}"
    return {"impl": "reference", "metric": METRIC, "value": round(val, 4), "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded numpy Gaussian K/V/Q; no dataset or weights)",
            "config": _config(wl, args),
            "cpu_baseline": {"value": round(val, 4), "unit": "GB/s", "cores": threads, "host_cores": cpu_threads(),
                             "threads": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": round(val, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


_CODEC_NAME = {workloads.Q4_G64: "q4_g64", workloads.Q8_0: "q8_0", workloads.Q4_G32: "q4_g32",
               workloads.NVFP4: "nvfp4"}


def _config(wl, args, extra=None):
    sp = wl.spec
    c = {"workload": sp.name, "n_seq": sp.n_seq, "n_heads": sp.n_heads, "n_kv_heads": sp.n_kv_heads,
         "head_dim": sp.head_dim, "kv_len": int(wl.kv_len.max()) if sp.n_seq == 1 else "ragged",
         "total_kv_tokens": int(wl.kv_len.sum()), "n_q": sp.n_q,
         "k_codec": _CODEC_NAME[sp.k_codec], "v_codec": _CODEC_NAME[sp.v_codec]}
    if extra:
        c.update(extra)
    return c


class Session:
    """One workload resident on the GPU: its caches (rotating copies, so that
    every step reads its cache from HBM), the step's inputs and outputs, and
    CUDA graphs of its decode steps."""

    def __init__(self, wl, kv_bytes, args, dev, dist):
        import torch
        import quantized_kv_cache_q4_gb300 as kvq
        self.torch, self.kvq, self.wl, self.kv_bytes, self.args, self.dev, self.dist = (
            torch, kvq, wl, kv_bytes, args, dev, dist)
        sp = wl.spec
        S, Hk, D, H, nq = sp.n_seq, sp.n_kv_heads, sp.head_dim, sp.n_heads, sp.n_q
        self.S, self.D, self.H, self.nq = S, D, H, nq

        def to_dev(a):
            return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

        # resident cache: prefill through the library's own quantizer
        k0 = kvq.KVCache(sp.k_codec, S, Hk, D, wl.capacity, device=dev)
        v0 = kvq.KVCache(sp.v_codec, S, Hk, D, wl.capacity, device=dev)
        zero = torch.zeros(1, dtype=torch.int32, device=dev)
        for s in range(S):
            L = int(wl.cached_len[s])
            kvq.kvq_quantize_append(k0.seq_view(s), v0.seq_view(s), to_dev(wl.k_prefill[s][None]),
                                    to_dev(wl.v_prefill[s][None]), L, zero)
        torch.cuda.synchronize()
        self.cache_bytes = k0.nbytes() + v0.nbytes()
        # rotating copies so that every step reads its cache from HBM, not L2
        self.n_copies = max(1, min(64, math.ceil(4 * L2_BYTES / max(1, kv_bytes))))
        self.caches = [(k0, v0)] + [(k0.clone(), v0.clone()) for _ in range(self.n_copies - 1)]

        # the step's inputs (new K/V rows, q) are views of one device buffer and
        # its results (out, lse) of another, so that the end-to-end legs move
        # each direction with one copy; every view starts on a 256-byte boundary
        def layout(arrays):
            offs, o = [], 0
            for a in arrays:
                offs.append(o)
                o += -(-a.nbytes // 256) * 256
            return offs, o
        in_arrays = [np.ascontiguousarray(a) for a in (wl.k_new, wl.v_new, wl.q)]
        in_offs, in_bytes = layout(in_arrays)
        self.stage_in = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
        self.h_in = torch.zeros(in_bytes, dtype=torch.uint8).pin_memory()
        views = []
        for a, o in zip(in_arrays, in_offs):
            t = torch.from_numpy(a)
            self.h_in[o:o + a.nbytes].copy_(t.reshape(-1).view(torch.uint8))
            views.append(self.stage_in[o:o + a.nbytes].view(t.dtype).view(t.shape))
        self.stage_in.copy_(self.h_in)
        self.k_new, self.v_new, self.q = views
        self.pos0, self.kv_len = to_dev(wl.cached_len), to_dev(wl.kv_len)
        self.max_kv = int(wl.kv_len.max())
        self.n_splits = args.splits if args.splits is not None else 0
        self.n_splits_eff = self.n_splits or kvq.kvq_decode_default_splits(k0, v0, H, nq, self.max_kv)
        self.ws = kvq.alloc_workspace(kvq.kvq_decode_workspace_bytes(k0, v0, H, nq, self.max_kv, self.n_splits), dev)
        self.n_out, n_lse = S * nq * H * D, S * nq * H
        self.lse_off = -(-self.n_out // 64) * 64
        self.stage_out = torch.empty(self.lse_off + n_lse, dtype=torch.float32, device=dev)
        self.out = self.stage_out[:self.n_out].view(S, nq, H, D)
        self.lse = self.stage_out[self.lse_off:self.lse_off + n_lse].view(S, nq, H)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.stream = torch.cuda.Stream(device=dev)

        # CUDA graphs, so that the host is not on the timed path: one per cache
        # copy (one step) and one for a round of n_copies consecutive steps, one
        # per copy, as an engine captures a whole decode step of many layers
        with torch.cuda.stream(self.stream):
            for i in range(self.n_copies):      # warm the launch path before capture
                self.step(i)
        self.stream.synchronize()
        self.graphs = []
        for i in range(self.n_copies):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                self.step(i)
            self.graphs.append(g)
        self.round_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.round_graph, stream=self.stream):
            for i in range(self.n_copies):
                self.step(i)
        torch.cuda.synchronize()
        assert int(self.err.item()) == 0, "device error bits set during set-up"

    def step(self, i, ev=None, res=None):
        """One decode step on cache copy i: append the new rows, then attention."""
        kvq, sp = self.kvq, self.wl.spec
        kc, vc = self.caches[i % self.n_copies]
        o_, l_ = res if res is not None else (self.out, self.lse)
        kvq.kvq_quantize_append(kc, vc, self.k_new, self.v_new, self.nq, self.pos0, self.err, stream=self.stream)
        if ev is not None:
            ev[0].record(self.stream)
        kvq.kvq_decode_attention(kc, vc, self.q, self.nq, self.H, sp.scale, self.kv_len, self.max_kv, self.n_splits,
                                 o_, l_, self.ws, d_err=self.err, stream=self.stream)
        if ev is not None:
            ev[1].record(self.stream)

    def replay_steps(self, n):
        """Exactly n steps: whole rounds, then single steps."""
        for _ in range(n // self.n_copies):
            self.round_graph.replay()
        for i in range(n % self.n_copies):
            self.graphs[i].replay()

    def barrier(self):
        self.torch.cuda.synchronize()
        if self.dist is not None:
            self.dist.barrier()

    def timed_steps(self, steps, soak_s, local):
        """Milliseconds per step over exactly `steps` graph-replayed steps
        (max over ranks), with the clocks sampled from a soak of the same
        replays through the timed region."""
        torch = self.torch
        t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(local) as clocks:
            t_soak = time.perf_counter()
            with torch.cuda.stream(self.stream):
                while time.perf_counter() - t_soak < soak_s:
                    self.replay_steps(64)
                    self.stream.synchronize()
            self.barrier()
            with torch.cuda.stream(self.stream):
                t_start.record(self.stream)
                self.replay_steps(steps)
                t_end.record(self.stream)
            self.barrier()
        ms = reduce_max(t_start.elapsed_time(t_end) / steps, self.dist, self.dev)
        return ms, clocks.summary()

    def attention_eager_ms(self):
        """The attention call alone, eager, with events around each call on its
        stream; a sleep kernel holds the stream while the host enqueues a batch
        of eager steps, so host launch time never shows up between the events."""
        torch = self.torch
        attn_ms = []
        reps = max(1, min(20, self.args.steps // self.n_copies))
        for _ in range(reps):
            evs = []
            with torch.cuda.stream(self.stream):
                torch.cuda._sleep(int(4e6))
                for i in range(self.n_copies):
                    e = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                    self.step(i, e)
                    evs.append(e)
            self.stream.synchronize()
            attn_ms += [a.elapsed_time(b) for a, b in evs]
        return statistics.median(attn_ms)

    def attention_eager_back_to_back_ms(self):
        """The attention call eager (no graph) and back to back, as an engine
        that keeps its stream fed issues it: a sleep kernel holds the stream
        while the host enqueues four calls per cache copy, with events around
        the whole batch only (so each call's start overlaps the previous
        merge, as in the graph); per call = batch time / calls, median of
        three batches."""
        torch, kvq, sp = self.torch, self.kvq, self.wl.spec

        def call(i):
            kc, vc = self.caches[i % self.n_copies]
            kvq.kvq_decode_attention(kc, vc, self.q, self.nq, self.H, sp.scale, self.kv_len, self.max_kv,
                                     self.n_splits, self.out, self.lse, self.ws, d_err=self.err, stream=self.stream)
        n_calls = 4 * self.n_copies
        with torch.cuda.stream(self.stream):
            for i in range(self.n_copies):
                call(i)
        self.stream.synchronize()
        per_call = []
        for _ in range(3):
            a_start, a_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(self.stream):
                torch.cuda._sleep(int(2e7))
                a_start.record(self.stream)
                for j in range(n_calls):
                    call(j)
                a_end.record(self.stream)
            self.stream.synchronize()
            per_call.append(a_start.elapsed_time(a_end) / n_calls)
        return reduce_max(statistics.median(per_call), self.dist, self.dev)

    def attention_graph_ms(self):
        """The attention kernels as a pipelined engine runs them: a graph of one
        attention call per cache copy, back to back (each merge chains into the
        next decode), timed with events around whole replays; per call =
        total / (replays * copies).  Returns (ms, replays)."""
        torch, kvq, sp = self.torch, self.kvq, self.wl.spec
        attn_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(attn_graph, stream=self.stream):
            for i in range(self.n_copies):
                kc, vc = self.caches[i]
                kvq.kvq_decode_attention(kc, vc, self.q, self.nq, self.H, sp.scale, self.kv_len, self.max_kv,
                                         self.n_splits, self.out, self.lse, self.ws, d_err=self.err,
                                         stream=self.stream)
        a_start, a_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_reps = max(3, self.args.steps // self.n_copies)
        with torch.cuda.stream(self.stream):
            for _ in range(2):
                attn_graph.replay()
            a_start.record(self.stream)
            for _ in range(a_reps):
                attn_graph.replay()
            a_end.record(self.stream)
        self.stream.synchronize()
        return reduce_max(a_start.elapsed_time(a_end) / (a_reps * self.n_copies), self.dist, self.dev), a_reps

    def e2e_graph_ms(self, steps, warmup):
        """End to end through the public API, steps replayed from graphs: new
        K/V rows and q from pinned host memory (one copy of the staging buffer);
        the results written by the kernels straight into pinned, device-mapped
        host memory (out and lse are host pointers there); one synchronisation
        a step.  Returns (ms, h2d bytes, d2h bytes, host results)."""
        torch = self.torch
        h_res = torch.zeros(self.stage_out.shape, dtype=self.stage_out.dtype).pin_memory()
        h_out = h_res[:self.n_out].view(self.out.shape)
        h_lse = h_res[self.lse_off:self.lse_off + self.lse.numel()].view(self.lse.shape)
        e2e_graphs = []
        for i in range(self.n_copies):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                self.stage_in.copy_(self.h_in, non_blocking=True)
                self.step(i, res=(h_out, h_lse))
            e2e_graphs.append(g)
        # each replay is launched on the stream and waited for before the next one
        with torch.cuda.stream(self.stream):
            for i in range(warmup):
                e2e_graphs[i % self.n_copies].replay()
                self.stream.synchronize()
        self.barrier()
        t0 = time.perf_counter()
        with torch.cuda.stream(self.stream):
            for i in range(steps):
                e2e_graphs[i % self.n_copies].replay()
                self.stream.synchronize()
        ms = reduce_max((time.perf_counter() - t0) * 1e3 / steps, self.dist, self.dev)
        return ms, self.h_in.numel(), h_res.numel() * h_res.element_size(), (h_out, h_lse)

    def e2e_eager_ms(self, steps, warmup):
        """End to end through the public API with no graph: every step copies the
        new K/V rows and q from pinned host memory, calls kvq_quantize_append and
        kvq_decode_attention (argument checks, split choice and launches on the
        host each time), copies out and lse back to pinned host memory and
        synchronises once.  Returns (ms, host results)."""
        torch = self.torch
        h_res = torch.zeros(self.stage_out.shape, dtype=self.stage_out.dtype).pin_memory()

        def one(i):
            self.stage_in.copy_(self.h_in, non_blocking=True)
            self.step(i)
            h_res.copy_(self.stage_out, non_blocking=True)
            self.stream.synchronize()
        with torch.cuda.stream(self.stream):
            for i in range(warmup):
                one(i)
        self.barrier()
        t0 = time.perf_counter()
        with torch.cuda.stream(self.stream):
            for i in range(steps):
                one(i)
        ms = reduce_max((time.perf_counter() - t0) * 1e3 / steps, self.dist, self.dev)
        h_out = h_res[:self.n_out].view(self.out.shape)
        h_lse = h_res[self.lse_off:self.lse_off + self.lse.numel()].view(self.lse.shape)
        return ms, (h_out, h_lse)


def attention_summary(sess, attn_ms, attn_eager_ms, step_ms, clocks, peak):
    """The attention measurements of one workload (for the ``also`` entries)."""
    sp = sess.wl.spec
    kv = sess.kv_bytes
    gbs = kv / (attn_ms * 1e-3) / 1e9
    return {"workload": sp.name, "kv_bytes_per_step": kv, "total_kv_tokens": int(sess.wl.kv_len.sum()),
            "n_splits": sess.n_splits_eff, "attention_us": round(attn_ms * 1e3, 3),
            "attention_us_eager_call": round(attn_eager_ms * 1e3, 3), "attention_gbs": round(gbs, 2),
            "frac": round(gbs / peak, 4), "traffic": _traffic(sp.name), "step_us": round(step_ms * 1e3, 3),
            "step_gbs": round(kv / (step_ms * 1e-3) / 1e9, 2),
            "us_per_token": round(step_ms * 1e3 / (sp.n_seq * sp.n_q), 4), "clocks": clocks,
            "l2": f"{sess.n_copies} rotating cache copies, steps replayed from CUDA graphs"}


def run_ours(args, wl, kv_bytes, world, rank, local):
    import torch

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sp = wl.spec
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist = dist_mod
    sess = Session(wl, kv_bytes, args, dev, dist)
    with torch.cuda.stream(sess.stream):
        sess.replay_steps(args.warmup)
    sess.barrier()

    # timed region: exactly K steps.  The clock sampler runs from a ~1 s soak of
    # the same replays (part of the warm-up) through the timed region, so the
    # samples are taken under this load with the clocks it settles at.
    ms, clock_summary = sess.timed_steps(args.steps, args.soak, local)
    attn_eager = sess.attention_eager_ms()
    attn_b2b = sess.attention_eager_back_to_back_ms()
    attn, a_reps = sess.attention_graph_ms()
    e2e_ms, h2d, d2h, (h_out, h_lse) = sess.e2e_graph_ms(args.steps, args.warmup)
    # the host copy holds what the device-resident path computes
    assert torch.equal(h_out, sess.out.cpu()) and torch.equal(h_lse, sess.lse.cpu()), "end-to-end results differ"
    eager_ms, (e_out, e_lse) = sess.e2e_eager_ms(args.steps, args.warmup)
    assert torch.equal(e_out, sess.out.cpu()) and torch.equal(e_lse, sess.lse.cpu()), "eager results differ"
    assert int(sess.err.item()) == 0, "device error bits set during the run"

    peak, peak_kind = _peaks()
    achieved = kv_bytes / (attn * 1e-3) / 1e9
    value = job_gbs(kv_bytes, ms, world)
    # kernels launched per step: append + decode (+ merge when the range is split)
    per_step = 2 + (1 if sess.n_splits_eff > 1 else 0)
    launches = args.steps * per_step
    tokens_per_step = sp.n_seq * sp.n_q
    res = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded numpy Gaussian K/V/Q; no dataset or weights)",
        "config": _config(wl, args, {"n_splits": sess.n_splits_eff, "kv_bytes_per_step": kv_bytes,
                                     "cache_bytes": sess.cache_bytes,
                                     "l2": f"{sess.n_copies} rotating cache copies "
                                           f"({sess.n_copies * sess.cache_bytes / 1e6:.0f} MB, >= 4x the 129 MB "
                                           f"L2); steps replayed from CUDA graphs of {sess.n_copies} consecutive "
                                           f"steps, one per copy",
                                     "parallelism": f"replicas x{world}",
                                     "arithmetic": "int4/int8 codes as exact fp16 MMA operands, fp32 accumulate, "
                                                   "fp32 softmax"}),
        "us_per_token": round(ms * 1e3 / tokens_per_step, 4),
        "fraction_of_hbm_peak": round(kv_bytes / (ms * 1e-3) / 1e9 / peak, 4),
        "roofline": {"bound": "hbm", "kernel": "kvq_decode_attention (decode + merge kernels)",
                     "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "traffic": _traffic(sp.name), "attention_us": round(attn * 1e3, 3),
                     "attention_timing": f"graph of {sess.n_copies} back-to-back calls, events around {a_reps} "
                                         f"replays",
                     "attention_us_eager_call": round(attn_eager * 1e3, 3),
                     "attention_us_eager_back_to_back": round(attn_b2b * 1e3, 3)},
        "e2e": {"value": round(job_gbs(kv_bytes, e2e_ms, world), 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 6),
                "path": "steps replayed from CUDA graphs of the public calls; one synchronisation a step"},
        "e2e_eager": {"value": round(job_gbs(kv_bytes, eager_ms, world), 2), "unit": "GB/s",
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(eager_ms, 6),
                      "path": "kvq_quantize_append + kvq_decode_attention called eagerly every step, host copies "
                              "in and out, one synchronisation a step"},
        "gpu_launches": launches,
        "clocks": clock_summary,
    }
    del sess
    torch.cuda.empty_cache()

    # the other long-context workloads, measured the same way in the same run
    if not args.no_also:
        also = {}
        for cfg in ALSO_CONFIGS:
            if cfg == args.config:
                continue
            wl2 = workloads.make(workloads.spec(cfg))
            kv2 = workloads.kv_bytes_per_token(wl2.spec) * int(wl2.kv_len.sum())
            s2 = Session(wl2, kv2, args, dev, dist)
            with torch.cuda.stream(s2.stream):
                s2.replay_steps(args.warmup)
            s2.barrier()
            ms2, clocks2 = s2.timed_steps(args.steps, min(args.soak, 0.5), local)
            eager2 = s2.attention_eager_ms()
            attn2, _ = s2.attention_graph_ms()
            assert int(s2.err.item()) == 0, "device error bits set during the run"
            also[wl2.spec.name] = attention_summary(s2, attn2, eager2, ms2, clocks2, peak)
            del s2
            torch.cuda.empty_cache()
        also["long196k_host_tier"] = host_tier_summary(args, dev, peak)
        torch.cuda.empty_cache()
        also["prefill512_32k"] = prefill_summary(args, dev)
        torch.cuda.empty_cache()
        res["also"] = also
    return res


# workloads measured beside the main one: 196,608 keys, the 16-sequence MTP
# verify batch, the mixed q8_0-K / Q4_G64-V pair at 65,536 keys
ALSO_CONFIGS = (3, 4, 2)


def host_tier_summary(args, dev, peak, resident_frac=0.5, page_tokens=8192, n_slots=4):
    """The 196,608-key workload with its cache in pinned host memory: the first
    half resident on the device, the rest streamed through a ring of n_slots
    pages (kvq_decode_attention_tiered).  Timed with CUDA events around calls on
    the caller's stream (the page copies run on the library's copy stream,
    joined to it)."""
    import torch
    import quantized_kv_cache_q4_gb300 as kvq
    wl = workloads.make(workloads.spec(3))
    sp = wl.spec
    S, Hk, D, H, nq = sp.n_seq, sp.n_kv_heads, sp.head_dim, sp.n_heads, sp.n_q
    kv_len = int(wl.kv_len[0])
    k = kvq.KVCache(sp.k_codec, S, Hk, D, wl.capacity, device=dev)
    v = kvq.KVCache(sp.v_codec, S, Hk, D, wl.capacity, device=dev)
    zero = torch.zeros(1, dtype=torch.int32, device=dev)
    src = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)   # noqa: E731
    kvq.kvq_quantize_append(k, v, src(wl.k_prefill[0][None]), src(wl.v_prefill[0][None]), int(wl.cached_len[0]), zero)
    kvq.kvq_quantize_append(k, v, src(wl.k_new), src(wl.v_new), nq, src(wl.cached_len))
    torch.cuda.synchronize()
    kh, vh = k.to_host(), v.to_host()
    n_res = int(kv_len * resident_frac) // 64 * 64
    ring = kvq.alloc_workspace(kvq.kvq_tiered_ring_bytes(kh, vh, page_tokens, n_slots), dev)
    ws = kvq.alloc_workspace(kvq.kvq_tiered_workspace_bytes(kh, vh, k, v, H, nq, kv_len, n_res, page_tokens), dev)
    q = src(wl.q)
    out = torch.empty((S, nq, H, D), dtype=torch.float32, device=dev)
    lse = torch.empty((S, nq, H), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def call():
        kvq.kvq_decode_attention_tiered(kh, vh, k, v, n_res, q, nq, H, sp.scale, kv_len, page_tokens, n_slots, ring,
                                        out, lse, ws, stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            call()
    stream.synchronize()
    reps = max(5, args.steps // 4)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(reps):
            call()
        b.record(stream)
    stream.synchronize()
    ms = a.elapsed_time(b) / reps
    kv = workloads.kv_bytes_per_token(sp) * kv_len
    streamed = workloads.kv_bytes_per_token(sp) * (kv_len - n_res)
    return {"workload": "long196k, cache in pinned host memory", "resident_tokens": n_res,
            "streamed_tokens": kv_len - n_res, "page_tokens": page_tokens, "ring_slots": n_slots,
            "attention_us": round(ms * 1e3, 3), "attention_gbs": round(kv / (ms * 1e-3) / 1e9, 2),
            "frac": round(kv / (ms * 1e-3) / 1e9 / peak, 4),
            "host_to_device_gbs": round(streamed / (ms * 1e-3) / 1e9, 2),
            "timing": f"events around {reps} eager calls on the caller's stream"}


def prefill_summary(args, dev, n_new=512, total=32768):
    """A prompt chunk through kvq_decode_attention: n_new new tokens of 24 query
    heads over 4 kv heads (head_dim 256, Q4_G64 K/V, fp16 queries) attending
    causally to the total - n_new cached keys and to each other (the
    tensor-core prompt-chunk kernel, default splits).  Graph of back-to-back
    calls, events around replays; FLOPs = 4 * head_dim * (visible keys summed
    over query rows)."""
    import torch
    import quantized_kv_cache_q4_gb300 as kvq
    H, Hk, D = 24, 4, 256
    sp = workloads.Spec("prefill512_32k", 1, H, Hk, D, (total - n_new,), n_new, workloads.Q4_G64,
                        workloads.Q4_G64, "f16", "f16", "normal", workloads.BASE_SEED + 900)
    wl = workloads.make(sp)
    k = kvq.KVCache(sp.k_codec, 1, Hk, D, wl.capacity, device=dev)
    v = kvq.KVCache(sp.v_codec, 1, Hk, D, wl.capacity, device=dev)
    zero = torch.zeros(1, dtype=torch.int32, device=dev)
    src = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)   # noqa: E731
    kvq.kvq_quantize_append(k, v, src(wl.k_prefill[0][None]), src(wl.v_prefill[0][None]), int(wl.cached_len[0]), zero)
    kvq.kvq_quantize_append(k, v, src(wl.k_new), src(wl.v_new), n_new, src(wl.cached_len))
    torch.cuda.synchronize()
    q, kv_len = src(wl.q), src(wl.kv_len)
    out = torch.empty((1, n_new, H, D), dtype=torch.float32, device=dev)
    lse = torch.empty((1, n_new, H), dtype=torch.float32, device=dev)
    n_splits = kvq.kvq_decode_default_splits(k, v, H, n_new, total)
    ws = kvq.alloc_workspace(kvq.kvq_decode_workspace_bytes(k, v, H, n_new, total, 0), dev)
    stream = torch.cuda.Stream(device=dev)

    def call():
        kvq.kvq_decode_attention(k, v, q, n_new, H, sp.scale, kv_len, total, 0, out, lse, ws, stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            call()
    stream.synchronize()
    reps = 10
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(reps):
            call()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = float("inf")
    with torch.cuda.stream(stream):
        g.replay()
        for _ in range(5):
            a.record(stream)
            g.replay()
            b.record(stream)
            b.synchronize()
            best = min(best, a.elapsed_time(b) / reps)
    visible = sum(total - n_new + i + 1 for i in range(n_new)) * H
    tflops = 4.0 * D * visible / (best * 1e-3) / 1e12
    peak, kind = _bf16_peak()
    return {"workload": f"prompt chunk of {n_new} tokens x 24 query heads over {total} keys (4 kv heads, head_dim "
                        f"256, Q4_G64 K/V, fp16 queries)", "n_splits": n_splits,
            "attention_us": round(best * 1e3, 3),
            "roofline": {"bound": "tensor", "achieved": round(tflops, 2), "peak": peak, "unit": "TFLOP/s",
                         "frac": round(tflops / peak, 4), "peak_kind": f"{kind} bf16 dense burst (fp16 runs at the "
                                                                      "same nominal rate)"},
            "timing": f"graph of {reps} back-to-back calls, best of 5 replays"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", type=int, default=1)
    ap.add_argument("--splits", type=int, default=None)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--ref-steps", type=int, default=None, help="oracle steps for the cpu_baseline leg")
    ap.add_argument("--soak", type=float, default=1.0, help="seconds of untimed replays before the timed region")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-also", action="store_true", help="measure the selected workload only")
    ap.add_argument("--prefill", type=int, default=None, metavar="KEYS",
                    help="measure only a 512-token prompt chunk over KEYS keys and print its summary")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    world, rank, local = _dist_env()

    wl = workloads.make(workloads.spec(args.config))
    kv_bytes = workloads.kv_bytes_per_token(wl.spec) * int(wl.kv_len.sum())

    if args.impl == "reference":
        if rank != 0:
            return
        res = run_reference(args, wl, kv_bytes)
        print(json.dumps(res), flush=True)
        return

    if args.prefill is not None:
        if rank == 0:
            print(json.dumps(prefill_summary(args, f"cuda:{local}", total=args.prefill)), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    res = run_ours(args, wl, kv_bytes, world, rank, local)
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(wl, kv_bytes, max_steps=args.ref_steps or 1000)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
