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


# The sources of the kernels the committed captures profile (the Q4_G64 decode
# and the merge) and of their launch (split policy, tensor maps).
_PROFILED_SOURCES = ("kvq_api.cu", "kvq_decode_tc.cu", "kvq_decode_tc.cuh", "kvq_internal.cuh", "kvq_merge.cu",
                     "kvq_ptx.cuh", "kvq_tensor_map.cu")


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
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):                        # not available on this platform
        return os.cpu_count() or 1


def run_reference(args, wl, kv_bytes):
    """The oracle timed on the host cores: each step is the full workload step."""
    import oracle
    oracle.build()
    k, v = oracle_caches(wl)
    units = wl.spec.n_seq * wl.spec.n_kv_heads
    threads = max(1, min(cpu_threads(), units))
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
            "cpu_baseline": {"value": round(val, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
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


def run_ours(args, wl, kv_bytes, world, rank, local):
    import torch
    import quantized_kv_cache_q4_gb300 as kvq

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sp = wl.spec
    S, Hk, D, H, nq = sp.n_seq, sp.n_kv_heads, sp.head_dim, sp.n_heads, sp.n_q

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
    cache_bytes = k0.nbytes() + v0.nbytes()
    # rotating copies so that every step reads its cache from HBM, not L2
    n_copies = max(1, min(64, math.ceil(4 * L2_BYTES / max(1, kv_bytes))))
    caches = [(k0, v0)] + [(k0.clone(), v0.clone()) for _ in range(n_copies - 1)]

    # the step's inputs (new K/V rows, q) are views of one device buffer and its
    # results (out, lse) of another, so that the end-to-end leg below moves each
    # direction with one copy; every view starts on a 256-byte boundary
    def layout(arrays):
        offs, o = [], 0
        for a in arrays:
            offs.append(o)
            o += -(-a.nbytes // 256) * 256
        return offs, o
    in_arrays = [np.ascontiguousarray(a) for a in (wl.k_new, wl.v_new, wl.q)]
    in_offs, in_bytes = layout(in_arrays)
    stage_in = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
    h_in = torch.zeros(in_bytes, dtype=torch.uint8).pin_memory()
    views = []
    for a, o in zip(in_arrays, in_offs):
        t = torch.from_numpy(a)
        h_in[o:o + a.nbytes].copy_(t.reshape(-1).view(torch.uint8))
        views.append(stage_in[o:o + a.nbytes].view(t.dtype).view(t.shape))
    stage_in.copy_(h_in)
    k_new, v_new, q = views
    pos0, kv_len = to_dev(wl.cached_len), to_dev(wl.kv_len)
    max_kv = int(wl.kv_len.max())
    n_splits = args.splits if args.splits is not None else 0
    n_splits_eff = n_splits or kvq.kvq_decode_default_splits(k0, v0, H, nq, max_kv)
    ws = kvq.alloc_workspace(kvq.kvq_decode_workspace_bytes(k0, v0, H, nq, max_kv, n_splits), dev)
    n_out, n_lse = S * nq * H * D, S * nq * H
    lse_off = -(-n_out // 64) * 64
    stage_out = torch.empty(lse_off + n_lse, dtype=torch.float32, device=dev)
    out = stage_out[:n_out].view(S, nq, H, D)
    lse = stage_out[lse_off:lse_off + n_lse].view(S, nq, H)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step(i, ev=None, res=None):
        kc, vc = caches[i % n_copies]
        o_, l_ = res if res is not None else (out, lse)
        kvq.kvq_quantize_append(kc, vc, k_new, v_new, nq, pos0, err, stream=stream)
        if ev is not None:
            ev[0].record(stream)
        kvq.kvq_decode_attention(kc, vc, q, nq, H, sp.scale, kv_len, max_kv, n_splits, o_, l_, ws, d_err=err,
                                 stream=stream)
        if ev is not None:
            ev[1].record(stream)

    # CUDA graphs, so that the host is not on the timed path: one per cache copy
    # (one step) and one for a round of n_copies consecutive steps, one per copy,
    # as an engine captures a whole decode step of many layers in one graph
    graphs = []
    with torch.cuda.stream(stream):
        for i in range(n_copies):      # warm the launch path before capture
            step(i)
    stream.synchronize()
    for i in range(n_copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(i)
        graphs.append(g)
    round_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(round_graph, stream=stream):
        for i in range(n_copies):
            step(i)
    torch.cuda.synchronize()

    def replay_steps(n):
        """Exactly n steps: whole rounds, then single steps."""
        for _ in range(n // n_copies):
            round_graph.replay()
        for i in range(n % n_copies):
            graphs[i].replay()
    assert int(err.item()) == 0, "device error bits set during set-up"

    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist = dist_mod

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()

    with torch.cuda.stream(stream):
        replay_steps(args.warmup)
    barrier()

    # timed region: exactly K steps.  The clock sampler runs from a ~1 s soak of
    # the same replays (part of the warm-up) through the timed region, so the
    # samples are taken under this load with the clocks it settles at.
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        t_soak = time.perf_counter()
        with torch.cuda.stream(stream):
            while time.perf_counter() - t_soak < args.soak:
                replay_steps(64)
                stream.synchronize()
        barrier()
        with torch.cuda.stream(stream):
            t_start.record(stream)
            replay_steps(args.steps)
            t_end.record(stream)
        barrier()
    ms = reduce_max(t_start.elapsed_time(t_end) / args.steps, dist, dev)
    clock_summary = clocks.summary()

    # the attention call alone (its kernels), timed with events on its stream.
    # A sleep kernel holds the stream while the host enqueues a batch of eager
    # steps, so host launch time never shows up between the two events.
    attn_ms = []
    reps = max(1, min(20, args.steps // n_copies))
    for rep in range(reps):
        evs = []
        with torch.cuda.stream(stream):
            torch.cuda._sleep(int(4e6))
            for i in range(n_copies):
                e = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                step(i, e)
                evs.append(e)
        stream.synchronize()
        attn_ms += [a.elapsed_time(b) for a, b in evs]
    attn_eager = statistics.median(attn_ms)

    # the attention kernels as a pipelined engine runs them: a graph of one
    # attention call per cache copy, back to back (each merge chains into the
    # next decode), timed with events around whole replays; per call = / copies
    attn_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(attn_graph, stream=stream):
        for i in range(n_copies):
            kc, vc = caches[i]
            kvq.kvq_decode_attention(kc, vc, q, nq, H, sp.scale, kv_len, max_kv, n_splits, out, lse, ws,
                                     d_err=err, stream=stream)
    a_start, a_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a_reps = max(3, args.steps // n_copies)
    with torch.cuda.stream(stream):
        for _ in range(2):
            attn_graph.replay()
        a_start.record(stream)
        for _ in range(a_reps):
            attn_graph.replay()
        a_end.record(stream)
    stream.synchronize()
    attn = reduce_max(a_start.elapsed_time(a_end) / (a_reps * n_copies), dist, dev)

    # end to end through the public API: new K/V rows and q from pinned host
    # memory (one copy of the staging buffer); the results written by the
    # kernels straight into pinned, device-mapped host memory (out and lse are
    # host pointers there); one synchronisation a step
    h_res = torch.zeros(stage_out.shape, dtype=stage_out.dtype).pin_memory()
    h_out = h_res[:n_out].view(S, nq, H, D)
    h_lse = h_res[lse_off:lse_off + n_lse].view(S, nq, H)
    e2e_graphs = []
    for i in range(n_copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            stage_in.copy_(h_in, non_blocking=True)
            step(i, res=(h_out, h_lse))
        e2e_graphs.append(g)
    # each replay is launched on `stream` and waited for before the next one
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            e2e_graphs[i % n_copies].replay()
            stream.synchronize()
    barrier()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            e2e_graphs[i % n_copies].replay()
            stream.synchronize()
    e2e_ms = reduce_max((time.perf_counter() - t0) * 1e3 / args.steps, dist, dev)
    # the host copy holds what the device-resident path computes
    assert torch.equal(h_out, out.cpu()) and torch.equal(h_lse, lse.cpu()), "end-to-end results differ"
    h2d = h_in.numel() * h_in.element_size()
    d2h = h_res.numel() * h_res.element_size()
    assert int(err.item()) == 0, "device error bits set during the run"

    peak, peak_kind = _peaks()
    achieved = kv_bytes / (attn * 1e-3) / 1e9
    value = job_gbs(kv_bytes, ms, world)
    # kernels launched per step: append + decode (+ merge when the range is split)
    launches = args.steps * (2 + (1 if n_splits_eff > 1 else 0))
    tokens_per_step = sp.n_seq * sp.n_q
    res = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded numpy Gaussian K/V/Q; no dataset or weights)",
        "config": _config(wl, args, {"n_splits": n_splits_eff, "kv_bytes_per_step": kv_bytes,
                                     "cache_bytes": cache_bytes,
                                     "l2": f"{n_copies} rotating cache copies ({n_copies * cache_bytes / 1e6:.0f} MB, "
                                           f">= 4x the 129 MB L2); steps replayed from CUDA graphs of {n_copies} "
                                           f"consecutive steps, one per copy",
                                     "parallelism": f"replicas x{world}",
                                     "arithmetic": "int4/int8 codes as exact fp16 MMA operands, fp32 accumulate, "
                                                   "fp32 softmax"}),
        "us_per_token": round(ms * 1e3 / tokens_per_step, 4),
        "fraction_of_hbm_peak": round(kv_bytes / (ms * 1e-3) / 1e9 / peak, 4),
        "roofline": {"bound": "hbm", "kernel": "kvq_decode_attention (decode + merge kernels)",
                     "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "traffic": _traffic(sp.name), "attention_us": round(attn * 1e3, 3),
                     "attention_timing": f"graph of {n_copies} back-to-back calls, events around {a_reps} replays",
                     "attention_us_eager_call": round(attn_eager * 1e3, 3)},
        "e2e": {"value": round(job_gbs(kv_bytes, e2e_ms, world), 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 6)},
        "gpu_launches": launches,
        "clocks": clock_summary,
    }
    return res


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

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    res = run_ours(args, wl, kv_bytes, world, rank, local)
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        k, v = oracle_caches(wl)
        units = wl.spec.n_seq * wl.spec.n_kv_heads
        threads = max(1, min(cpu_threads(), units))
        n, total = 0, 0.0
        budget = 10.0
        while total < budget and n < (args.ref_steps or 1000):
            total += oracle_step_time(wl, k, v, threads)
            n += 1
        t = total / n
        res["cpu_baseline"] = {"value": round(kv_bytes / t / 1e9, 4), "unit": "GB/s", "cores": threads,
                               "kind": "oracle",
                               "sample": f"{n} full {wl.spec.name} steps (append + fp64 attention over "
                                         f"{int(wl.kv_len.sum())} tokens), {total:.1f} s"}
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
