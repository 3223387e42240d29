"""Benchmark of the tree-verify step on GB300.

One step = one verify round over one batch of synthetic input: tree mask,
split-KV tree attention + merge, per-node argmax, acceptance walk and the
accept(k) commit (five launches of this library's kernels).  Every step
verifies the same workload: each step of a timed graph has its own copy of
prefix_len, all reset by one copy at the graph's start.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 1..5] [--impl ours|reference]

Prints one JSON line.  `value` = verified query rows (tree nodes) per second
over the whole job, inputs resident in HBM, measured with CUDA events around
K CUDA-graph replays; between steps the inputs rotate over enough copies that
each step reads them from HBM, not L2.  `e2e` = the same metric through the
public Python API with pinned host inputs copied in and the results copied
out every step.  `roofline` = the split-KV attention kernel's algorithmic
bytes per launch over its CUDA-event duration, against the measured HBM
copy bandwidth.  `cpu_baseline` = the float64 oracle on the host cores.
With --impl reference the oracle itself is timed as the reference arm.
"""
from __future__ import annotations

import os
import sys

_CORES = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(_CORES))

import argparse
import hashlib
import json
import math
import statistics
import subprocess
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from speculative_decoding_tree_gb300 import workloads as wl  # noqa: E402

METRIC = "tree-verify attention: query rows/s and HBM GB/s vs peak; accept+commit µs"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", type=int, default=4, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    return ap.parse_args()


# ---------------------------------------------------------------- helpers

def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return ws, rank


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws):
    if ws == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(ws, units_per_rank, steps, elapsed_ms_max):
    """Whole-job throughput: every rank's units over the slowest rank's time."""
    return ws * units_per_rank * steps / (elapsed_ms_max / 1e3)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# sources the split kernels are built from: the recorded DRAM traffic holds
# only while none of them has changed
SPLIT_SOURCES = ("tc_ptx.cuh", "tv_internal.cuh", "tv_attn_tc.cu", "tv_attn_tc2.cu", "tv_attn_tcp.cu", "tv_attn_simt.cu")


def kernel_source_hash():
    csrc = os.path.join(ROOT, "speculative_decoding_tree_gb300", "csrc")
    h = hashlib.sha256()
    for f in SPLIT_SOURCES:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload_name):
    """dram bytes per launch of the split kernel from the committed ncu summary,
    only while the kernel sources are unchanged since the capture."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d.get(workload_name)
        if e and e.get("source_hash") == kernel_source_hash():
            return e.get("bytes_per_launch")
    except Exception:
        pass
    return None


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- workloads

def make_sets(spec, device):
    """Enough independent copies of the workload that a step's inputs are not
    in L2 when it starts (rotating over them)."""
    from speculative_decoding_tree_gb300.runner import DeviceStep

    def argmax_cpu(x):          # only to plant draft matches in the synthetic input
        return torch.argmax(x.float(), dim=1)

    # room in the cache for the commits of the back-to-back accept timing
    # (each call advances its own prefix length, up to 6 times)
    spec = spec.replace(cache_margin=max(spec.cache_margin, 64))
    sets = []
    w0 = wl.make_workload(spec, canary=0.0, argmax_fn=argmax_cpu)
    per_set, nsets, _ = set_layout(w0)
    for i in range(nsets):
        w = w0 if i == 0 else wl.make_workload(spec.replace(seed=spec.seed + 7919 * i), canary=0.0,
                                               argmax_fn=argmax_cpu)
        st = DeviceStep(w, device=device)
        st.p0 = st.prefix_len.clone()
        sets.append(st)
    return sets, per_set


def algorithmic_bytes(w):
    """Per verify step, from the workload itself: attention = every K/V
    element of prefix and tree once + Q + O; split kernel = K/V + Q; accept
    = the logits once + 2x the committed K/V rows."""
    sp = w.spec
    es = 4 if sp.dtype == "f32" else 2
    les = 4 if sp.logit_dtype == "f32" else 2
    kv = q = o = 0
    for b in range(sp.batch):
        P = int(w.prefix_len[b])
        n = len(w.parents[b])
        kv += (P + n) * sp.hkv * sp.d * 2 * es
        q += n * sp.hq * sp.d * es
        o += n * sp.hq * sp.d * es
    logits = w.total_rows * sp.vocab * les
    return dict(kv=kv, q=q, o=o, attn=kv + q + o, split=kv + q, logits=logits)


# ---------------------------------------------------------------- our arm

def expansion_timing(cap_stream, reps=5, trees_per_graph=8):
    """Dynamic draft-tree expansion: every step of one whole expansion
    (two launches per step), `trees_per_graph` expansions back to back in one
    CUDA graph, events around the graph; per tree = total / trees.  The
    drafter's rows of every step are resident (a real drafter writes each
    step's rows just before the step, so they would be in L2 as well)."""
    from speculative_decoding_tree_gb300.runner import DeviceExpand
    out = {}
    for key in ("eagle2", "batched"):
        spec = wl.EXPAND_CONFIGS[key]
        dx = DeviceExpand(spec)
        dx.run()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap_stream):
            for _ in range(trees_per_graph):
                dx.run()
        g.replay()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(2_000_000)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3 / trees_per_graph)
        tree_us = statistics.median(ts)
        logit_bytes = sum(r.numel() * r.element_size() for r in dx.rows)
        out[key] = {"workload": spec.name, "batch": spec.batch, "vocab": spec.vocab, "top_k": spec.top_k,
                    "width": spec.width, "max_nodes": spec.max_nodes, "steps": dx.steps,
                    "expansion_us": round(tree_us, 2), "step_us": round(tree_us / dx.steps, 2),
                    "launches": 2 * dx.steps, "draft_logit_bytes": logit_bytes,
                    "gbs": round(logit_bytes / (tree_us * 1e-6) / 1e9, 1),
                    "nodes": int(dx.n_nodes.sum().item()), "device_status": int(dx.status[0].item())}
        del dx, g
    return out


def bf16_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def rope_timing(sets, cap_stream, b2b_us):
    """Tree-position RoPE + K/V scatter for the workload's rows: back-to-back
    calls over the input sets (queries in place); algorithmic bytes = every
    Q, K and V element read once and written once, plus the row metadata."""
    import speculative_decoding_tree_gb300 as tv
    calls = []
    nbytes = 0
    for st_ in sets:
        R, sp = st_.w.total_rows, st_.w.spec
        k_in = torch.randn(R, sp.hkv, sp.d, device=st_.q.device).to(st_.q.dtype)
        v_in = torch.randn(R, sp.hkv, sp.d, device=st_.q.device).to(st_.q.dtype)
        kt = torch.empty_like(st_.k_tree)
        vt = torch.empty_like(st_.v_tree)
        st_.mask()

        def call(st_=st_, k_in=k_in, v_in=v_in, kt=kt, vt=vt):
            tv.tv_tree_rope_scatter(st_.desc, 1e6, st_.q, k_in, v_in, st_.prefix_len, st_.node_offsets, st_.depth,
                                    st_.q, kt, vt, st_.status)
        calls.append(call)
        es = st_.q.element_size()
        nbytes = 2 * R * (sp.hq + 2 * sp.hkv) * sp.d * es + R * 4 * 2
    torch.cuda.synchronize()
    us = b2b_us([calls[i % len(calls)] for i in range(max(24, 8 * len(calls)))])
    return us, nbytes


def lm_head_timing(cap_stream, peak, reps=5, calls=6):
    """Fused lm_head + argmax: `calls` back-to-back calls in one CUDA graph,
    CUDA events; per call = total / calls.  The weights (1 to 1.6 GB) are far
    larger than L2, so every call streams them from HBM.  Algorithmic bytes
    per call: the weights, the hidden rows and the argmax / max-logit
    outputs."""
    from speculative_decoding_tree_gb300.runner import DeviceLmHead
    out = {}
    for key in ("qwen", "batched"):
        spec = wl.LMHEAD_CONFIGS[key]
        lm = DeviceLmHead(spec)
        lm.run()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap_stream):
            for _ in range(calls):
                lm.run()
        g.replay()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(2_000_000)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3 / calls)
        us = statistics.median(ts)
        wbytes = spec.vocab * spec.hidden * 2
        algo = wbytes + spec.rows * spec.hidden * 2 + spec.rows * 8
        flops = 2.0 * spec.rows * spec.vocab * spec.hidden
        gbs = algo / (us * 1e-6) / 1e9
        tflops = flops / (us * 1e-6) / 1e12
        tpeak, tkind = bf16_peak()
        # the bound: weight streaming below the ridge (peak flop/s over peak
        # bytes/s), the tensor cores above it
        tensor = flops / algo > tpeak * 1e12 / (peak * 1e9)
        out[key] = {"workload": spec.name, "rows": spec.rows, "hidden": spec.hidden, "vocab": spec.vocab,
                    "us": round(us, 2), "algorithmic_bytes": algo, "flops": flops, "gbs": round(gbs, 1),
                    "tflops": round(tflops, 1),
                    "roofline": {"bound": "tensor" if tensor else "hbm",
                                 "achieved": round(tflops if tensor else gbs, 1),
                                 "peak": tpeak if tensor else peak, "unit": "TFLOP/s" if tensor else "GB/s",
                                 "frac": round(tflops / tpeak if tensor else gbs / peak, 4),
                                 "peak_source": tkind if tensor else "measured"},
                    "launches": 2, "device_status": int(lm.status[0].item())}
        del lm, g
        torch.cuda.empty_cache()
    return out


def bench_config(spec, w, nsets, per_set, per_big, ws):
    """The workload description both arms print (the reference arm times the
    oracle on the same workload and prints the same dict)."""
    return {
        "workload": spec.name, "batch": spec.batch, "q_heads": spec.hq, "kv_heads": spec.hkv,
        "head_dim": spec.d, "prefix": list(spec.prefix), "tree_rows": int(w.total_rows), "vocab": spec.vocab,
        "paged": spec.paged, "parallelism": "replicas" if ws > 1 else "single",
        "l2": f"inputs rotate over {nsets} copies ({nsets * per_set / 1e6:.0f} MB > 129 MB L2)",
        "timing": (f"CUDA-graph replays of {per_big} whole steps per graph (the remainder one per graph), "
                   "CUDA events; each step of a graph has its own prefix_len, reset once at the graph's start"),
    }


def set_layout(w):
    """Bytes of one input set and how many sets the rotation needs so that a
    step's inputs are not in L2 when it starts."""
    per_set = (w.k_cache.numel() * w.k_cache.element_size() * 2 + w.logits.numel() * w.logits.element_size()
               + w.q.numel() * w.q.element_size() * 2)
    nsets = max(2, math.ceil(3 * L2_BYTES / per_set))
    return per_set, nsets, nsets * max(1, math.ceil(8 / nsets))


class Harness:
    """One workload's rotating device input sets, the step graphs and the
    back-to-back per-call timing."""

    def __init__(self, spec, device, cap_stream, warmup):
        self.spec = spec
        self.cap_stream = cap_stream
        self.sets, self.per_set = make_sets(spec, device)
        self.nsets = len(self.sets)
        self.w = self.sets[0].w
        self.rows = self.w.total_rows
        for i in range(max(warmup, 3)):
            self.step(self.sets[i % self.nsets])
        torch.cuda.synchronize()
        self.graphs = []
        for st in self.sets:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap_stream):
                self.step(st)
            self.graphs.append(g)
        # whole rotations over the input sets in one graph (at least 8 steps),
        # so that graph launches do not sit between every two steps; every
        # step in it does all of its work
        self.per_big = self.nsets * max(1, math.ceil(8 / self.nsets))
        # Each step of the big graph verifies with its own copy of prefix_len
        # (a 16-byte aligned row of pl_big); one copy at the graph's start
        # resets them all to the sets' starting lengths, so the commits of
        # one replay never change the next replay's workload and no reset
        # sits between two steps.
        p0 = self.sets[0].p0
        row = max(4, (p0.numel() + 3) // 4 * 4)
        self.pl_big = torch.zeros((self.per_big, row), dtype=p0.dtype, device=p0.device)
        self.p0_big = self.pl_big.clone()
        for i in range(self.per_big):
            self.p0_big[i, :p0.numel()] = self.sets[i % self.nsets].p0
        self.big = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.big, stream=cap_stream):
            self.pl_big.copy_(self.p0_big, non_blocking=True)
            for i in range(self.per_big):
                st = self.sets[i % self.nsets]
                saved = st.prefix_len
                st.prefix_len = self.pl_big[i, :p0.numel()]
                st.step()
                st.prefix_len = saved
        for i in range(max(warmup, 3)):
            self.graphs[i % self.nsets].replay()
        self.big.replay()
        torch.cuda.synchronize()
        for st in self.sets:
            st.status.zero_()

    @staticmethod
    def step(st):
        st.prefix_len.copy_(st.p0, non_blocking=True)
        st.step()

    def run_steps(self, k):
        """exactly k steps: whole big graphs, then single-step graphs"""
        for _ in range(k // self.per_big):
            self.big.replay()
        for i in range(k % self.per_big):
            self.graphs[i % self.nsets].replay()

    def time_steps(self, k):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(10_000_000)        # let the queue run ahead of the GPU
        e0.record()
        self.run_steps(k)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    def b2b_us(self, calls, reps=5):
        """K back-to-back launches of one call in one CUDA graph, bracketed by
        two events; the per-launch time is the total over K (gaps between
        launches included)."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.cap_stream):
            for c in calls:
                c()
        g.replay()
        torch.cuda.synchronize()
        out = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(2_000_000)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            out.append(e0.elapsed_time(e1) * 1e3 / len(calls))
        del g
        return statistics.median(out)

    def reset_prefix(self):
        for st_ in self.sets:
            st_.prefix_len.copy_(st_.p0)
        torch.cuda.synchronize()

    def accept_pool(self):
        """(set, logits) pairs whose logits total more than 3x L2, so that each
        accept+commit call reads its logits from HBM (sets keep logits of
        their own shape: sets differ in their row count)."""
        own = [st_.logits for st_ in self.sets]
        pool = [(st_, st_.logits) for st_ in self.sets]
        pool_bytes = sum(t.numel() * t.element_size() for t in own)
        while pool_bytes < 3 * L2_BYTES:
            st_ = self.sets[len(pool) % self.nsets]
            pool.append((st_, st_.logits.clone()))
            pool_bytes += st_.logits.numel() * st_.logits.element_size()
        return own, pool

    def breakdown(self, sampled=False):
        """Per-call durations (us): mask, split pass, merge, the whole
        tree_verify_attn call, accept + commit (and its sampled form)."""
        self.reset_prefix()
        n_b2b = max(24, 8 * self.nsets)
        pick = [self.sets[i % self.nsets] for i in range(n_b2b)]
        out = {"split": self.b2b_us([st_.partials for st_ in pick]),
               "attn": self.b2b_us([st_.attn for st_ in pick]),
               "mask": self.b2b_us([st_.mask for st_ in pick]),
               "merge": self.b2b_us([st_.merge for st_ in pick])}
        # accept + commit: each call of the chain has its own prefix_len
        # (preset to the set's prefix) and advances it, so no reset sits
        # between two calls; the cache has room for the six graph replays
        own, pool = self.accept_pool()

        def chain(kind):
            calls = []
            for i in range(max(len(pool), n_b2b)):
                st_, lg = pool[i % len(pool)]
                pl = st_.p0.clone()

                def call(st_=st_, lg=lg, pl=pl, i=i):
                    saved = st_.prefix_len
                    st_.logits, st_.prefix_len = lg, pl
                    if kind == "greedy":
                        st_.accept_commit()
                    else:
                        st_.accept_commit_sampled(1.0, 20240601, i)   # temperature 1, fresh noise per call
                    st_.prefix_len = saved
                calls.append(call)
            return calls
        out["accept"] = self.b2b_us(chain("greedy"))
        if sampled:
            out["accept_sampled"] = self.b2b_us(chain("sampled"))
        for st_, lg in zip(self.sets, own):
            st_.logits = lg
        del pool
        self.reset_prefix()
        return out

    def status(self):
        s = 0
        for st_ in self.sets:
            s |= int(st_.status[0].item())
        return s


def attn_summary(tv, h, bd, peak, peak_kind):
    """The split kernel's roofline and the whole call's fraction for one workload."""
    ab = algorithmic_bytes(h.w)
    plan = tv.tv_attn_plan(h.sets[0].desc)
    achieved = ab["split"] / (bd["split"] * 1e-6) / 1e9
    roof = {
        "kernel": {0: "attn_simt_kernel", 1: "tv_attn_tc_kernel", 2: "tv_attn_tc2_kernel",
                   3: "tv_attn_tcp_kernel"}[plan["kernel"]],
        "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
        "frac": round(achieved / peak, 4), "peak_source": peak_kind,
        "traffic": profiled_traffic(h.spec.name),
        "algorithmic_bytes_per_launch": ab["split"],
    }
    call = {"us": round(bd["attn"], 2), "gbs": round(ab["attn"] / (bd["attn"] * 1e-6) / 1e9, 1),
            "frac": round(ab["attn"] / (bd["attn"] * 1e-6) / 1e9 / peak, 4),
            "algorithmic_bytes": ab["attn"]}
    return roof, call, plan


def run_ours(args, ws, rank):
    import numpy as np  # noqa: F401
    from speculative_decoding_tree_gb300 import _build
    _build.build()
    import speculative_decoding_tree_gb300 as tv

    device = torch.device("cuda", torch.cuda.current_device())
    spec = wl.CONFIGS[args.config]
    cap_stream = torch.cuda.Stream()
    peak, peak_kind = measured_peaks()
    h = Harness(spec, device, cap_stream, args.warmup)
    w, rows, nsets = h.w, h.rows, h.nsets

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    # settle the clocks under load (untimed), then the timed region
    t_end = time.time() + 1.0
    while time.time() < t_end:
        h.run_steps(8 * h.per_big)
        torch.cuda.synchronize()
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    elapsed_ms = h.time_steps(args.steps)
    barrier(ws)
    torch.cuda.synchronize()
    elapsed_ms = max_over_ranks(elapsed_ms, ws)

    bd = h.breakdown(sampled=True)
    roof, call, plan = attn_summary(tv, h, bd, peak, peak_kind)

    # the other single-GPU workloads of the target, measured in the same
    # process the same way (their own rotating input sets, step graphs and
    # back-to-back call timings); the headline workload's entry repeats its
    # own numbers
    per_config = {}
    for c in (3, 4, 5):
        if c == args.config:
            hc, bdc, rc, cc, pc, step_ms, k = h, bd, roof, call, plan, elapsed_ms, args.steps
        else:
            hc = Harness(wl.CONFIGS[c], device, cap_stream, 3)
            k = 64
            step_ms = hc.time_steps(k)
            bdc = hc.breakdown()
            rc, cc, pc = attn_summary(tv, hc, bdc, peak, peak_kind)
        per_config[c] = {
            "workload": hc.spec.name, "tree_rows": hc.rows, "rows_per_s": round(hc.rows * k / (step_ms / 1e3), 1),
            "step_us": round(step_ms * 1e3 / k, 2), "split_us": round(bdc["split"], 2),
            "merge_us": round(bdc["merge"], 2), "mask_us": round(bdc["mask"], 2),
            "accept_commit_us": round(bdc["accept"], 2), "attn_call": cc, "roofline": rc,
            "plan": {key: pc[key] for key in ("kernel", "num_splits", "chunk", "row_tiles", "grid_ctas")},
            "device_status": hc.status(),
        }
        if hc is not h:
            del hc
            torch.cuda.empty_cache()

    expansion = expansion_timing(cap_stream)
    rope_us, rope_bytes = rope_timing(h.sets, cap_stream, h.b2b_us)
    lm_heads = lm_head_timing(cap_stream, peak)
    timing_mode = ("back-to-back launches of each call in one CUDA graph over the rotating input sets, "
                   "programmatic dependent launch between them; per launch = events around the graph / launches")
    clocks = sampler.stop() if sampler else None
    status = h.status()

    # e2e through the public API with host buffers: per step copy the step's
    # inputs in from pinned memory, run the step, copy the results out
    # (rotating over the same input sets as above)
    sets = h.sets
    names_in = ("q", "k_tree", "v_tree", "logits", "draft", "parents", "node_offsets")
    names_out = ("accept_len", "tokens", "path")
    host_in = [{k: getattr(s_, k).cpu().pin_memory() for k in names_in} for s_ in sets]
    host_out = [{k: torch.empty_like(getattr(s_, k), device="cpu").pin_memory() for k in names_out} for s_ in sets]
    h2d = sum(t.numel() * t.element_size() for t in host_in[0].values())
    d2h = sum(t.numel() * t.element_size() for t in host_out[0].values())
    n_e2e = min(args.steps, 50)
    for rep in range(2):
        torch.cuda.synchronize()
        barrier(ws)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(n_e2e):
            j = i % nsets
            s_ = sets[j]
            for k, t in host_in[j].items():
                getattr(s_, k).copy_(t, non_blocking=True)
            s_.prefix_len.copy_(s_.p0, non_blocking=True)
            s_.step()
            for k, t in host_out[j].items():
                t.copy_(getattr(s_, k), non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), ws)

    ms_per_step = elapsed_ms / args.steps
    value = aggregate(ws, rows, args.steps, elapsed_ms)
    config = bench_config(spec, w, nsets, h.per_set, h.per_big, ws)
    res = {
        "metric": METRIC, "value": round(value, 1), "unit": "rows/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": spec.dtype, "data": "synthetic",
        "config": config,
        "rows_timed_per_step": rows,
        "kernel_timing": timing_mode,
        "roofline": roof,
        "e2e": {"value": round(ws * rows * n_e2e / (e2e_ms / 1e3), 1), "unit": "rows/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": h.sets[0].kernels_per_step() * args.steps,
        "clocks": clocks,
        "breakdown_us": {"mask": round(bd["mask"], 2), "attn_split": round(bd["split"], 2),
                         "attn_merge": round(bd["merge"], 2), "accept_commit": round(bd["accept"], 2)},
        "attn_call": call,
        "accept_commit_us": round(bd["accept"], 2),
        "accept_commit_sampled_us": round(bd["accept_sampled"], 2),
        "per_config": {str(c): v for c, v in per_config.items()},
        "rope_scatter": {"us": round(rope_us, 2), "algorithmic_bytes": rope_bytes,
                         "gbs": round(rope_bytes / (rope_us * 1e-6) / 1e9, 1), "launches": 1},
        "expansion": expansion,
        "lm_head_argmax": lm_heads,
        "plan": plan,
        "device_status": status | max(e["device_status"] for e in list(expansion.values()) + list(lm_heads.values()))
                         | max(e["device_status"] for e in per_config.values()),
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(spec, args.cpu_seconds)
    return res


# ---------------------------------------------------------------- oracle arms

def oracle_sample_step(w, rows):
    """The oracle on a bounded sample: attention for the first `rows` tree
    rows (all heads), their argmax, and acceptance + commit of every sequence."""
    import oracle
    import numpy as np
    samples = [(r, h) for r in range(rows) for h in range(w.spec.hq)]
    oracle.tree_attention(w, samples)
    am = np.zeros(w.total_rows, dtype=np.int64)
    am[:rows] = oracle.argmax_rows(w.logits[:rows])
    acc = []
    for b in range(w.batch):
        o0, o1 = w.seq_rows(b)
        acc.append(oracle.accept(w.parents[b], w.draft_tokens[o0:o1].tolist(), am[o0:o1].tolist()))
    oracle.commit(w, acc)


def _oracle_workload(spec):
    import oracle
    return wl.make_workload(spec, canary=0.0, argmax_fn=oracle.argmax_rows)


def cpu_baseline(spec, seconds):
    w = _oracle_workload(spec)
    t = time.perf_counter()
    oracle_sample_step(w, 1)
    one = max(time.perf_counter() - t, 1e-4)
    rows = max(1, min(w.total_rows, int(seconds / one)))
    t = time.perf_counter()
    oracle_sample_step(w, rows)
    dt = time.perf_counter() - t
    return {"value": round(rows / dt, 3), "unit": "rows/s", "cores": _CORES, "kind": "oracle",
            "sample": f"{rows} of {w.total_rows} tree rows (all {spec.hq} heads, float64 attention), their "
                      f"argmax, acceptance and commit; {dt:.1f} s; cores = BLAS/OpenMP thread cap"}


def run_reference(args, ws, rank):
    if rank != 0:
        return None
    spec = wl.CONFIGS[args.config]
    w = _oracle_workload(spec)
    t = time.perf_counter()
    oracle_sample_step(w, 1)
    one = max(time.perf_counter() - t, 1e-4)
    # every tree row per step when the whole run fits about four minutes of
    # host time, else the same bounded sample of rows in every step
    steps_all = args.steps + args.warmup
    budget = 240.0 / max(1, steps_all)
    rows = max(1, min(w.total_rows, int(budget / one)))
    for _ in range(args.warmup):
        oracle_sample_step(w, rows)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle_sample_step(w, rows)
    dt = time.perf_counter() - t
    value = rows * args.steps / dt
    sample = (f"each step: {rows} of {w.total_rows} tree rows (all heads) through the float64 oracle, "
              f"their argmax, acceptance and commit")
    per_set, nsets, per_big = set_layout(w)
    config = bench_config(spec, w, nsets, per_set, per_big, ws)
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "rows/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config,
        "rows_timed_per_step": rows,
        "cpu_baseline": {"value": round(value, 3), "unit": "rows/s", "cores": _CORES, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    if args.impl == "reference":
        ws = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        res = run_reference(args, ws, rank)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    ws, rank = dist_setup()
    res = run_ours(args, ws, rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
