#!/usr/bin/env python
"""Benchmark of the IceCache hot path on GB300.

The contract line is the decode step (selection + GQA union, gather, masked
sparse attention; metric "decode-step µs & HBM GB/s") of the
Qwen3-32B-shaped batch: 16 sequences x 8 KV heads (64 query heads), 100k
tokens per unit, budget 256 tokens, bf16 -- the largest single-GPU
configuration.  One step = one ice_decode_step over the whole batch (one
CUDA graph replay), the selected pages gathered into shared memory (the
contiguous buffer is the variant in "buffer").  value = HBM GB/s on the
step's minimum bytes (parent tables + selected K/V pages once + Q/O), summed
over ranks and divided by the slowest rank's time; ms_per_step is the step
time.  The index build (keys/s), the parent-assignment contraction at 100k,
the other shapes and the pinned-host page pool are reported in "extra".

Each rank runs its own batch (weak scaling; the only collectives are the
barrier and the max of the timings).

Usage: python bench.py [--gpus N --steps K --warmup W --impl ours|reference]
"""
from __future__ import annotations

import argparse
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

METRIC = "decode-step µs & HBM GB/s (select+gather+sparse attn); index-build keys/s"
L2_BYTES = 129 * 2 ** 20
D, S = 128, 16
REFERENCE_RUN_S = 150.0  # wall time the oracle (reference) arm aims for over all its steps


def graph_kernel_nodes(graph):
    """Kernel nodes of a captured CUDA graph (driver API), or None."""
    import ctypes
    try:
        h = graph.raw_cuda_graph()
        cu = ctypes.CDLL("libcuda.so.1")
        n = ctypes.c_size_t(0)
        if cu.cuGraphGetNodes(ctypes.c_void_p(h), None, ctypes.byref(n)) != 0:
            return None
        nodes = (ctypes.c_void_p * n.value)()
        if cu.cuGraphGetNodes(ctypes.c_void_p(h), nodes, ctypes.byref(n)) != 0:
            return None
        count = 0
        for i in range(n.value):
            t = ctypes.c_int(-1)
            if cu.cuGraphNodeGetType(ctypes.c_void_p(nodes[i]), ctypes.byref(t)) != 0:
                return None
            count += t.value == 0  # CU_GRAPH_NODE_TYPE_KERNEL
        return count
    except Exception:
        return None


# DRAM bytes per launch of a kernel from one ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum) on the named workload, with the SHA-256 of the source files
# the kernels and their launcher are built from; reported only while they are unchanged.
# The decode step's entry: the two kernels of ICE_PLAN_SCORE_SELECT captured at batch 4 (32 units) and scaled by the
# units to the 16-sequence batch (per-unit traffic does not depend on the batch).
TRAFFIC = {
    "decode": {"workload": "qwen3_32b_100k", "bytes": 354_081_792, "sha256": {
        "decode_select_tc.cu": "e1bb3c659f0a7ca618e4e526d2725e7008a7810019a25cc7f8f535f55bfebc75",
        "decode_attn_mma.cu": "116f2293b02f8bb342959191b40588d25efecaecdb78946e473417cbc5b66442",
        "select_unit.cuh": "e9fb950a3869e70bb5b99941bbe3a5caa9f6d8414d43b7dc983ecc0ce5e5c767",
        "attn_page.cuh": "85d342159d9748393e05de4c7a6239fd0aff82ae1638b53295ee21aa72426620",
        "tc_common.cuh": "bcc9600b9d3aaad4c363c2b9ce954eb63042c1c048f1de44ffffcd2b99354924",
        "topk_common.cuh": "4da63ede6240bc05d3653a5c8f9b1b7b8ca4df33f012a5fa405d4abde6d9cff4",
        "common.cuh": "53dc15cf41d59e44bc74139d9b0186fadd82c77de4300f0bf51cdbad59c77fd7",
        "internal.h": "d219025c74377dd8f9e11d923f0e86f66ce2550c253f84a76b8d32364939ab7f",
        "abi.cu": "b59a4af786ba69638338aeab3e17defe18d08e634665209de73565912c09a6db",
    }},
}


def measured_traffic(kernel: str, workload: str):
    import hashlib
    t = TRAFFIC.get(kernel)
    if not t or t["workload"] != workload:
        return None
    for name, want in t["sha256"].items():
        src = os.path.join(ROOT, "semantic_paged_kv_gb300", "csrc", name)
        try:
            sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
        except OSError:
            return None
        if sha != want:
            return None
    return t["bytes"]


EXTRAS = ("build", "separate", "longchat", "longchat_b8", "qwen_levels3", "mistral_insert", "host_pool", "llama16k")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qwen3_32b_100k")
    ap.add_argument("--batch", type=int, default=None, help="sequences per rank (default: the workload's)")
    ap.add_argument("--budget", type=int, default=None)
    ap.add_argument("--layers", type=int, default=2, help="distinct layers rotated between timed steps")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-e2e", action="store_true", help="skip the pinned-host pool end-to-end part (profiling runs)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-units", type=int, default=None, help="units in the CPU-baseline sample")
    ap.add_argument("--extras", default=",".join(EXTRAS), help="comma list of " + ", ".join(EXTRAS) + " (or none)")
    ap.add_argument("--reps", type=int, default=30, help="graph replays per extra timing")
    ap.add_argument("--detail", default=None, help="also write every measured number as JSON to this file")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, src="fallback")


def rank_info():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


# ------------------------------------------------------------- clocks ------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
        if self.gpu_id is not None:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons, n = [], None, set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            n += 1
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": n}


def gpu_id_for(dev) -> str | None:
    import torch
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        if dev < len(ids):
            return ids[dev]
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        return str(dev)


# ------------------------------------------------------- CPU oracle leg ---
def host_cpu() -> str:
    """The host's CPU model and logical CPU count, for the CPU-baseline record."""
    name = ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            k, _, v = line.partition(":")
            if k.strip() == "Model name" and v.strip():
                name = v.strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not name:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    k, _, v = line.partition(":")
                    if k.strip().lower() == "model name" and v.strip():
                        name = v.strip()
                        break
        except OSError:
            pass
    import platform
    return f"{name or 'unknown model'} ({platform.machine()}, {os.cpu_count()} logical CPUs)"




def decode_min_bytes(n_parents: int, n_selected: int, batch: int, n_q_heads: int, esz: int = 2) -> int:
    """Algorithmic minimum bytes of one decode step: every parent row once
    (the selection scan), every selected page's K and V rows once, Q in and
    O (fp32) out."""
    return n_parents * D * esz + n_selected * S * D * esz * 2 + batch * n_q_heads * D * (esz + 4)


class OracleDecodeSample:
    """The oracle (as it stands) on a bounded sample of the workload: `units`
    units, each the first n_tokens tokens of the workload's unit (same
    mixture), built by the oracle once (not timed); step() runs the oracle's
    decode step (a6-a10) of every unit, one unit per host thread, and returns
    its wall time."""

    def __init__(self, w: workloads.Workload, budget: int, units: int, n_tokens: int):
        import oracle
        self.oracle, self.w, self.budget, self.units, self.n_tokens = oracle, w, budget, units, n_tokens
        th = oracle.promote_threshold(w.promote_p)
        self.items = [(u // w.n_kv_heads, u % w.n_kv_heads) for u in range(units)]
        self.threads_wanted = min(units, os.cpu_count() or 1)
        oracle.build()
        self.idx = {}

        def build(it):
            K, V = workloads.unit_kv(w, 0, *it, n_tokens=n_tokens)
            self.idx[it] = oracle.build_unit(K, V, seed=w.seed, layer=0, seq=it[0], head=it[1], thresh=th,
                                             S=w.page_size)

        t0 = time.perf_counter()
        oracle.run_units(build, self.items, threads=self.threads_wanted)
        self.build_s = time.perf_counter() - t0
        self.q = {it: workloads.unit_queries(w, 0, *it) for it in self.items}
        self.sel = {}
        self.threads = 1

    def step(self) -> float:
        def dec(it):
            self.sel[it] = len(self.oracle.decode_unit(self.idx[it], self.q[it], self.budget)["sel_pages"])

        t0 = time.perf_counter()
        _, self.threads = self.oracle.run_units(dec, self.items, threads=self.threads_wanted)
        return time.perf_counter() - t0

    @property
    def bytes(self) -> int:
        """Minimum bytes of one step (the same count as the device's)."""
        g = self.w.n_q_heads // self.w.n_kv_heads
        return sum(decode_min_bytes(len(self.idx[it]["parent_tok"]), self.sel[it], 1, g) for it in self.items)

    def describe(self, passes: int, seconds: float) -> str:
        w = self.w
        return (f"{self.units} of {w.units} units (KV heads) of {w.name}, each the first {self.n_tokens} of its "
                f"N={w.n_tokens} tokens (same mixture), index built by the oracle beforehand ({self.build_s:.1f} s, "
                f"not timed); timed: the oracle's decode step (select, union, gather, attention) at budget "
                f"{self.budget}, one unit per host thread, {passes} passes ({seconds:.1f} s); GB/s on the same "
                f"minimum-bytes count as the device")


def cpu_baseline_sample(w, budget, units=None, min_seconds=10.0, max_seconds=30.0):
    units = units or min(w.units, os.cpu_count() or 1, 16)
    smp = OracleDecodeSample(w, budget, units, min(w.n_tokens, 25000))
    t, passes = 0.0, 0
    while passes < 1 or (t < min_seconds and t * (passes + 1) / passes <= max_seconds):
        t += smp.step()
        passes += 1
    value = smp.bytes * passes / t / 1e9
    return {"value": value, "unit": "GB/s", "cores": smp.threads, "kind": "oracle", "cpu": host_cpu(),
            "sample": smp.describe(passes, t),
            "short": f"{units}/{w.units} units, first {smp.n_tokens} tokens each, oracle-built index (untimed); "
                     f"oracle decode, 1 unit/thread, {passes} passes in {t:.0f} s",
            "build_keys_per_s": units * smp.n_tokens / smp.build_s}


def run_reference(args):
    rank, _, world = rank_info()
    if rank != 0:
        return  # the oracle arm runs on rank 0 only
    w = workloads.WORKLOADS[args.workload]
    if args.batch:
        w = w.scaled(batch=args.batch)
    budget = args.budget or max(w.budgets)
    units = args.cpu_units or min(w.units, os.cpu_count() or 1, 16)
    smp = OracleDecodeSample(w, budget, units, min(w.n_tokens, 25000))
    times = [smp.step() for _ in range(args.warmup + args.steps)][args.warmup:]
    total = sum(times)
    value = smp.bytes * len(times) / total / 1e9
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * total / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": compact_config(config_of(w, budget, args.gpus, args.layers)),  # the GPU arm's config
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": smp.threads, "kind": "oracle",
                         "sample": smp.describe(len(times), total), "cpu": host_cpu()},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def config_of(w, budget, gpus, layers):
    return {"workload": w.name, "batch_per_gpu": w.batch, "n_q_heads": w.n_q_heads, "n_kv_heads": w.n_kv_heads,
            "n_tokens": w.n_tokens, "head_dim": w.head_dim, "page_size": w.page_size, "promote_p": w.promote_p,
            "levels": 2, "budget_tokens": budget, "parallelism": f"dp{gpus}",
            "gather": "selected pages into shared memory (contiguous buffer: extra.buffer)",
            "l2": f"{layers} layers rotated (distinct K/V, index, queries), each step reads > 2.5x L2",
            "graph": f"one CUDA graph per pass over the {layers} layers (one decode step each)",
            "workspace": "one decode workspace and output set for all layers, as one stream reuses them"}


# ------------------------------------------------- multi-rank host logic ---
def rank_workload(name: str, rank: int, batch: int | None = None) -> workloads.Workload:
    """Each rank owns its own batch of the workload: same shapes, its own
    seed, so the ranks' units are disjoint and need no exchange."""
    base = workloads.WORKLOADS[name]
    if batch:
        base = base.scaled(batch=batch)
    return base.scaled(seed=base.seed + 1000 * rank)


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest of a host scalar over all ranks (the only collective)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(per_rank_work: float, steps: int, world: int, max_ms: float) -> float:
    """Work of all ranks over the slowest rank's time (weak scaling)."""
    return world * per_rank_work * steps / (max_ms * 1e-3)


# --------------------------------------------------------- device helpers --
class Replay:
    """Times a callable as one CUDA-graph replay after an L2 flush (a 2x L2
    write, then a 2x L2 read of another buffer, so the flush leaves no dirty
    lines to write back inside the timed region); median over reps, with p10
    and p90; CUDA events on the replaying stream."""

    def __init__(self, reps: int):
        import torch
        self.torch, self.reps = torch, reps
        self.flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda")
        self.evict = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
        self.sink = torch.empty((), dtype=torch.float32, device="cuda")
        self.cap = torch.cuda.Stream()

    def graph(self, fn):
        torch = self.torch
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        self.cap.wait_stream(torch.cuda.current_stream())
        try:
            g, kept = torch.cuda.CUDAGraph(keep_graph=True), True  # kept for counting its kernel nodes
        except TypeError:
            g, kept = torch.cuda.CUDAGraph(), False
        with torch.cuda.graph(g, stream=self.cap):
            fn()
        if kept:
            g.instantiate()
        torch.cuda.current_stream().wait_stream(self.cap)
        torch.cuda.synchronize()
        return g

    def __call__(self, fn) -> dict:
        torch = self.torch
        g = self.graph(fn)
        ts = []
        for _ in range(self.reps):
            self.flush.zero_()
            torch.sum(self.evict, dim=0, out=self.sink)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            g.replay()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) * 1000.0)
        return {"us": statistics.median(ts), "p10": float(np.percentile(ts, 10)), "p90": float(np.percentile(ts, 90)),
                "kernels": graph_kernel_nodes(g)}


def build_layer(ice, w, layer: int = 0, n_levels: int = 2, host_pool=None, n_cap=None, keep_kv=False):
    """One layer of the workload on the device: inputs drawn there (the
    host generator's mixture recipe), index built with ice_build_index, the
    build timed with CUDA events."""
    import torch
    cfg = ice.Config(batch=w.batch, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads, n_tokens=w.n_tokens,
                     dtype=ice.ICE_BF16 if w.dtype == "bf16" else ice.ICE_FP32, promote_p=w.promote_p, seed=w.seed,
                     layer=layer, n_levels=n_levels, n_cap=n_cap)
    K, V, C = workloads.batch_kv_device(w, layer)
    Q = workloads.batch_queries_device(w, C, layer)
    p = cfg.params()
    idx = ice.Index(cfg, host_pool=host_pool)
    ws = ice.workspace(ice.ice_build_workspace_bytes(p))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ice.ice_build_index(p, K, V, idx, ws, err)  # first build: lazy set-up out of the timing
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    ice.ice_build_index(p, K, V, idx, ws, err)
    b.record()
    torch.cuda.synchronize()
    st = ice.ice_check(err)
    if st != ice.ICE_OK:
        raise RuntimeError(f"build of {w.name}: device status {ice.ice_status_string(st)}")
    out = dict(cfg=cfg, p=p, idx=idx, Q=Q, err=err, build_ms=a.elapsed_time(b), C=C)
    if keep_kv:
        out.update(K=K, V=V, ws=ws)
    return out


def decode_call(ice, L, budget, buf, with_buffer: bool):
    scale = 1.0 / math.sqrt(D)
    kb, vb, bl = (buf.kbuf, buf.vbuf, buf.buf_len) if with_buffer else (None, None, None)
    return lambda: ice.ice_decode_step(L["p"], L["idx"], L["Q"], budget, buf.sel_pages, buf.sel_count, kb, vb, bl,
                                       scale, buf.O, buf.ws, L["err"])


def decode_bytes(L, buf, w) -> tuple[int, int]:
    """(minimum bytes, bytes of the contiguous buffer's write) of one step."""
    npar, nsel = int(L["idx"].n_parents.sum()), int(buf.sel_count.sum())
    return decode_min_bytes(npar, nsel, w.batch, w.n_q_heads), nsel * S * D * 2 * 2


def separate_calls(ice, pk, rp, L, buf, budget, w):
    """Steps a6-a8, a9 and a10 as the three separate calls on one layer, each
    timed as one replay after an L2 flush: the selection (parent rows read
    once), the gather (the selected pages read from the pool and written to
    the contiguous buffer) and the attention over the buffer (read once), with
    HBM GB/s on each call's algorithmic bytes against the measured copy peak."""
    scale = 1.0 / math.sqrt(D)
    p, idx, Q = L["p"], L["idx"], L["Q"]
    sel = rp(lambda: ice.ice_select_pages(p, idx, Q, budget, buf.sel_pages, buf.sel_count, buf.ws, L["err"]))
    nsel, npar = int(buf.sel_count.sum()), int(idx.n_parents.sum())
    gat = rp(lambda: ice.ice_gather_pages(p, idx, buf.sel_pages, buf.sel_count, buf.kbuf, buf.vbuf, buf.buf_len))
    att = rp(lambda: ice.ice_sparse_attn_decode(p, Q, buf.kbuf, buf.vbuf, buf.buf_len, buf.sel_count, scale, buf.O,
                                                buf.ws))
    page = S * D * 2 * 2  # K and V of one page, bf16
    qo = w.batch * w.n_q_heads * D * (2 + 4)
    b_sel, b_gat, b_att = npar * D * 2 + w.batch * w.n_q_heads * D * 2, 2 * nsel * page, nsel * page + qo
    rate = lambda b, t: b / (t["us"] * 1e-6) / 1e9
    return {"select_us": r3(sel["us"]), "select_gbs": r3(rate(b_sel, sel)),
            "gather_us": r3(gat["us"]), "gather_gbs": r3(rate(b_gat, gat)), "gather_frac": r3(rate(b_gat, gat) / pk["hbm"]),
            "attn_us": r3(att["us"]), "attn_gbs": r3(rate(b_att, att)), "attn_frac": r3(rate(b_att, att) / pk["hbm"]),
            "bytes": {"select": b_sel, "gather": b_gat, "attn": b_att}}


def r3(x):
    """Three significant digits (compact JSON)."""
    if x is None or isinstance(x, (int, str)) or not math.isfinite(x):
        return x
    return float(f"{x:.3g}")


# ------------------------------------------------------------ extra parts --
def steady_decode(ice, pk, rp, w, budget: int, n_layers: int, steps: int = 2000) -> dict:
    """Decode steps timed the way the contract line times them: n_layers
    layers with distinct K/V, index and queries (together well above L2, so
    that a layer's data has left L2 by its next step), one decode workspace
    and one set of outputs, one CUDA graph per pass over the layers, the
    passes back to back; HBM GB/s on the minimum bytes against the measured
    copy peak."""
    import torch
    layers = []
    for layer in range(n_layers):
        layers.append(build_layer(ice, w, layer=layer))
        torch.cuda.empty_cache()
    buf = ice.DecodeBuffers(layers[0]["cfg"], budget)
    for L in layers:
        decode_call(ice, L, budget, buf, False)()
        torch.cuda.synchronize()
        L["bytes"] = decode_bytes(L, buf, w)[0]
    g_all = rp.graph(lambda: [decode_call(ice, L, budget, buf, False)() for L in layers])
    passes = max(1, steps // n_layers)
    for _ in range(3):
        g_all.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(passes):
        g_all.replay()
    b.record()
    torch.cuda.synchronize()
    us = 1000.0 * a.elapsed_time(b) / (passes * n_layers)
    bmin = float(np.mean([L["bytes"] for L in layers]))
    st = [ice.ice_check(L["err"]) for L in layers]
    out = {"us": r3(us), "frac": r3(bmin / (us * 1e-6) / 1e9 / pk["hbm"]), "MB": r3(bmin / 1e6), "layers": n_layers,
           "steps": passes * n_layers}
    if any(x != ice.ICE_OK for x in st):
        out["status"] = ice.ice_status_string(max(st))
    del layers, buf, g_all
    torch.cuda.empty_cache()
    return out


def extra_longchat(ice, pk, rp, batch: int):
    """LongChat-7B shape (32/32 heads, MHA, 100k tokens, log-normal key
    norms): at batch 1 the parent-assignment contraction at 100k (tensor
    peak fraction) and the decode step at budgets 64 and 256; at batch 8 the
    decode step at 256.  Each decode step once after an L2 flush, and at 256
    also steadily as the contract line runs (6 layers at batch 1, about 55 MB
    of minimum bytes each; 2 at batch 8, about 443 MB each)."""
    import torch
    w = workloads.WORKLOADS["longchat_7b_100k"].scaled(batch=batch)
    L = build_layer(ice, w, keep_kv=batch == 1)
    out = {"build_ms": r3(L["build_ms"])}
    if batch == 1:
        t = rp(lambda: ice.ice_build_assign(L["p"], L["K"], L["idx"], L["ws"], L["err"]))
        flops = 2.0 * w.n_tokens * int(L["idx"].n_parents.sum()) * D
        tf = flops / (t["us"] * 1e-6) / 1e12
        out["assign"] = {"us": r3(t["us"]), "tflops": r3(tf), "frac": r3(tf / pk["bf16"])}
        del L["K"], L["V"], L["ws"]
    for budget in ((64, 256) if batch == 1 else (256,)):
        buf = ice.DecodeBuffers(L["cfg"], budget)
        t = rp(decode_call(ice, L, budget, buf, False))
        tb = rp(decode_call(ice, L, budget, buf, True))
        bmin, bbuf = decode_bytes(L, buf, w)
        out[f"d{budget}"] = {"us": r3(t["us"]), "frac": r3(bmin / (t["us"] * 1e-6) / 1e9 / pk["hbm"]),
                             "buf_us": r3(tb["us"]), "buf_frac": r3(bmin / (tb["us"] * 1e-6) / 1e9 / pk["hbm"]),
                             "MB": r3(bmin / 1e6), "kernels": t["kernels"]}
        del buf
    st = ice.ice_check(L["err"])
    del L
    torch.cuda.empty_cache()
    if st != ice.ICE_OK:
        out["status"] = ice.ice_status_string(st)
    out["steady256"] = steady_decode(ice, pk, rp, w, 256, 6 if batch == 1 else 2)
    return out


def extra_levels3(ice, pk, rp, w, budget):
    """The same batch as the contract line with a third index level: the
    descent selection instead of the parent-table scan."""
    import torch
    L = build_layer(ice, w, n_levels=3)
    buf = ice.DecodeBuffers(L["cfg"], budget)
    t = rp(decode_call(ice, L, budget, buf, False))
    tb = rp(decode_call(ice, L, budget, buf, True))
    ts = rp(lambda: ice.ice_select_pages(L["p"], L["idx"], L["Q"], budget, buf.sel_pages, buf.sel_count, buf.ws,
                                         L["err"]))
    out = {"build_ms": r3(L["build_ms"]), "us": r3(t["us"]), "buf_us": r3(tb["us"]), "select_us": r3(ts["us"]),
           "level2_nodes": int(L["idx"].n_nodes2.sum())}
    del L, buf
    torch.cuda.empty_cache()
    return out


def extra_mistral_insert(ice, pk):
    """Mistral-7B shape (32/8 heads, 36,864 tokens): 128 decode steps, each
    preceded by one inserted token per unit (step a11), the index growing.
    The 128 steps are one CUDA graph replayed once (an eager loop would time
    the host's launches once the GPU outruns them), on a freshly built index;
    the inserts alone are a second graph, replayed on another fresh build."""
    import torch
    w = workloads.WORKLOADS["mistral_7b_36k"]
    steps = 128
    L = build_layer(ice, w, n_cap=w.n_tokens + steps, keep_kv=True)
    U = L["cfg"].units
    gen = torch.Generator(device="cuda")
    gen.manual_seed(w.seed * 7919 + 11)
    lab = torch.randint(0, w.centres, (steps, U), generator=gen, device="cuda")
    kn = (L["C"][torch.arange(U, device="cuda")[None, :], lab]
          + w.spread * torch.randn((steps, U, D), generator=gen, device="cuda")).to(torch.bfloat16)
    vn = torch.randn((steps, U, D), generator=gen, device="cuda").to(torch.bfloat16)
    budget = max(w.budgets)
    buf = ice.DecodeBuffers(L["cfg"], budget)
    wsi = ice.workspace(ice.ice_insert_workspace_bytes(L["p"]))
    step = decode_call(ice, L, budget, buf, True)

    def rebuild():
        ice.ice_build_index(L["p"], L["K"], L["V"], L["idx"], L["ws"], L["err"])

    def capture(fn):
        rebuild()
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            fn()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        return g

    def timed(g):
        rebuild()  # the graph's inserts start from the built index again
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        return 1000.0 * a.elapsed_time(b) / steps

    def both():
        for st in range(steps):
            ice.ice_insert_tokens(L["p"], L["idx"], kn[st], vn[st], wsi, L["err"])
            step()

    def inserts():
        for st in range(steps):
            ice.ice_insert_tokens(L["p"], L["idx"], kn[st], vn[st], wsi, L["err"])

    both()  # once eagerly: lazy set-up out of the captures
    torch.cuda.synchronize()
    g_both, g_ins = capture(both), capture(inserts)
    step_us = min(timed(g_both) for _ in range(3))
    insert_us = min(timed(g_ins) for _ in range(3))
    timed(g_both)  # the full sequence last, for the final index size and status
    out = {"insert_us": r3(insert_us), "decode_us": r3(step_us - insert_us), "step_us": r3(step_us),
           "tokens_after": int(L["idx"].n_indexed.sum()), "status": ice.ice_status_string(ice.ice_check(L["err"]))}
    del L, buf, kn, vn, wsi, g_both, g_ins
    torch.cuda.empty_cache()
    return out


def extra_llama16k(ice, pk, rp):
    """Llama-3.1-8B shape at 16k tokens (32/8 heads, needle): the index build
    (its three stages) and the decode step, each a graph replay."""
    import torch
    w = workloads.WORKLOADS["llama31_8b_16k"]
    L = build_layer(ice, w, keep_kv=True)
    p, K, V, idx, ws, err = L["p"], L["K"], L["V"], L["idx"], L["ws"], L["err"]
    tl = rp(lambda: ice.ice_build_lift_promote(p, K, idx, ws, err))
    ta = rp(lambda: ice.ice_build_assign(p, K, idx, ws, err))
    tp = rp(lambda: ice.ice_build_pack(p, K, V, idx, ws, err))
    tb = rp(lambda: ice.ice_build_index(p, K, V, idx, ws, err))
    buf = ice.DecodeBuffers(L["cfg"], 256)
    td = rp(decode_call(ice, L, 256, buf, True))
    keys = w.units * w.n_tokens
    flops = 2.0 * w.n_tokens * int(idx.n_parents.sum()) * D
    out = {"build_us": r3(tb["us"]), "keys_s": r3(keys / (tb["us"] * 1e-6)), "lift_us": r3(tl["us"]),
           "assign_us": r3(ta["us"]), "assign_frac": r3(flops / (ta["us"] * 1e-6) / 1e12 / pk["bf16"]),
           "pack_us": r3(tp["us"]), "decode_us": r3(td["us"])}
    del L, buf
    torch.cuda.empty_cache()
    return out


def host_pool_part(ice, pk, rp, w, budget, e2e_steps):
    """The batch with its page pool in pinned host memory (step a12).
    Returns (e2e, extra): e2e is the decode step through the public API
    with host buffers, every step: Q host -> device (pinned), selection on
    the device, page ids device -> host, host threads gather the selected
    pages into pinned staging, ONE cudaMemcpyAsync to the device, attention,
    O device -> host.  extra: the direct mode (kernels read the pool over
    the CPU-GPU link, Q in and O out per step), the bulk copy alone, and a
    plain 1 GiB pinned host -> device copy as the link's measured peak."""
    import torch
    cfg0 = ice.Config(batch=w.batch, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads, n_tokens=w.n_tokens,
                      promote_p=w.promote_p, seed=w.seed)
    max_sel = ice.max_selected(cfg0, budget)
    hp = ice.HostPool(cfg0, max_sel, n_threads=min(16, os.cpu_count() or 1))
    E = lambda: torch.cuda.Event(enable_timing=True)
    try:
        L = build_layer(ice, w, host_pool=hp)
        cfg, p, idx, Qd, err = L["cfg"], L["p"], L["idx"], L["Q"], L["err"]
        U = cfg.units
        buf = ice.DecodeBuffers(cfg, budget)
        scale = 1.0 / math.sqrt(D)
        Qh = Qd.cpu().pin_memory()
        Oh = torch.empty_like(buf.O, device="cpu").pin_memory()
        selh = torch.empty_like(buf.sel_pages, device="cpu").pin_memory()
        cnth = torch.empty_like(buf.sel_count, device="cpu").pin_memory()
        plen_h = idx.page_len.cpu()  # index metadata, host-resident with the pool
        dst = torch.zeros(hp.staging_bytes, dtype=torch.uint8, device="cuda")
        nb = U * max_sel * S * D * 2
        kbuf = dst[:nb].view(torch.bfloat16).view(U, max_sel, S, D)
        vbuf = dst[nb:2 * nb].view(torch.bfloat16).view(U, max_sel, S, D)
        blen = dst[2 * nb:2 * nb + U * max_sel * 4].view(torch.int32).view(U, max_sel)
        wsa = ice.workspace(ice.ice_decode_workspace_bytes(p, budget, max_sel))

        def staged():
            Qd.copy_(Qh, non_blocking=True)
            ice.ice_select_pages(p, idx, Qd, budget, buf.sel_pages, buf.sel_count, buf.ws, err)
            selh.copy_(buf.sel_pages, non_blocking=True)
            cnth.copy_(buf.sel_count, non_blocking=True)
            torch.cuda.current_stream().synchronize()
            ice.ice_host_pool_gather_h2d(hp, p, selh, cnth, plen_h, max_sel, dst)
            ice.ice_sparse_attn_decode(p, Qd, kbuf, vbuf, blen, buf.sel_count, scale, buf.O, wsa)
            Oh.copy_(buf.O, non_blocking=True)

        def direct():
            Qd.copy_(Qh, non_blocking=True)
            ice.ice_decode_step(p, idx, Qd, budget, buf.sel_pages, buf.sel_count, None, None, None, scale, buf.O,
                                buf.ws, err)
            Oh.copy_(buf.O, non_blocking=True)

        def run(fn, n):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            a, b = E(), E()
            a.record()
            for _ in range(n):
                fn()
            b.record()
            torch.cuda.synchronize()
            return a.elapsed_time(b) / n  # ms per step

        ms_staged = run(staged, e2e_steps)
        ms_direct = run(direct, e2e_steps)
        bmin, _ = decode_bytes(L, buf, w)
        page_bytes = int(buf.sel_count.sum()) * S * D * 2 * 2
        # the bulk copy alone (the staging buffer's bytes) and a plain 1 GiB pinned copy (the link's peak)
        src = torch.empty(hp.staging_bytes, dtype=torch.uint8).pin_memory()
        big_h = torch.empty(1 << 30, dtype=torch.uint8).pin_memory()
        big_d = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")

        def copy_ms(d_, s_):
            best = float("inf")
            for _ in range(5):
                a, b = E(), E()
                a.record()
                d_.copy_(s_, non_blocking=True)
                b.record()
                torch.cuda.synchronize()
                best = min(best, a.elapsed_time(b))
            return best

        bulk_ms = copy_ms(dst, src)
        peak_gbs = (1 << 30) / (copy_ms(big_d, big_h) * 1e-3) / 1e9
        st = ice.ice_check(err)
        h2d = Qh.numel() * Qh.element_size() + hp.staging_bytes
        d2h = selh.numel() * 4 + cnth.numel() * 4 + Oh.numel() * 4
        e2e = {"value": None, "unit": "GB/s", "h2d_bytes_per_step": h2d, "bytes_per_step": bmin,
               "d2h_bytes_per_step": d2h, "steps": e2e_steps, "ms_per_step": ms_staged,
               "how": "pool in pinned host memory; per step: Q H2D, select, ids D2H, host gather, one bulk H2D, "
                      "attention, O D2H",
               "direct": {"value": r3(bmin / (ms_direct * 1e-3) / 1e9), "ms_per_step": r3(ms_direct),
                          "h2d_bytes_per_step": Qh.numel() * Qh.element_size(), "d2h_bytes_per_step": Oh.numel() * 4,
                          "how": "kernels read the selected pages from the host pool over the CPU-GPU link"}}
        extra = {"link_peak_gbs": r3(peak_gbs), "bulk_h2d_gbs": r3(hp.staging_bytes / (bulk_ms * 1e-3) / 1e9),
                 "bulk_frac": r3(hp.staging_bytes / (bulk_ms * 1e-3) / 1e9 / peak_gbs),
                 "direct_page_gbs": r3(page_bytes / (ms_direct * 1e-3) / 1e9),
                 "direct_frac": r3(page_bytes / (ms_direct * 1e-3) / 1e9 / peak_gbs),
                 "staged_ms": r3(ms_staged), "direct_ms": r3(ms_direct), "pool_GB": r3(2 * hp.pool_bytes / 1e9)}
        if st != ice.ICE_OK:
            extra["status"] = ice.ice_status_string(st)
        del L, buf, dst, src, big_h, big_d, kbuf, vbuf, blen
    finally:
        hp.close()
        torch.cuda.empty_cache()
    return e2e, extra


# ------------------------------------------------------------- our arm ----
def run_ours(args):
    import torch
    import torch.distributed as dist

    import semantic_paged_kv_gb300 as ice

    rank, local, world = rank_info()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group(backend="nccl", device_id=torch.device("cuda", local))

    def barrier():
        if world > 1:
            dist.barrier()

    pk = peaks()
    w = rank_workload(args.workload, rank, args.batch)
    budget = args.budget or max(w.budgets)
    E = lambda: torch.cuda.Event(enable_timing=True)
    # ---- the layers: distinct K/V, index and queries per layer, one decode
    # workspace and one set of outputs for all of them (one stream runs the
    # layers one after another, as a serving engine does); one CUDA graph
    # holds one decode step of every layer
    layers = []
    for layer in range(max(1, args.layers)):
        layers.append(build_layer(ice, w, layer=layer))
        torch.cuda.empty_cache()
    buf = ice.DecodeBuffers(layers[0]["cfg"], budget)
    nl = len(layers)
    for L in layers:  # each layer's step once: its selection gives its bytes
        decode_call(ice, L, budget, buf, False)()
        torch.cuda.synchronize()
        L["bytes"] = decode_bytes(L, buf, w)
        L["n_sel"] = int(buf.sel_count.sum())
    rp = Replay(args.reps)
    steps_of = lambda with_buffer: lambda: [decode_call(ice, L, budget, buf, with_buffer)() for L in layers]
    g_all, g_all_buf = rp.graph(steps_of(False)), rp.graph(steps_of(True))
    for L in layers:  # single-layer graphs for a step count that is not a multiple of the layers
        L["g"] = rp.graph(decode_call(ice, L, budget, buf, False))
        L["g_buf"] = rp.graph(decode_call(ice, L, budget, buf, True))
    full, rest = divmod(args.steps, nl)

    def run_steps(with_buffer: bool):
        g = g_all_buf if with_buffer else g_all
        for _ in range(full):
            g.replay()
        for i in range(rest):
            layers[i]["g_buf" if with_buffer else "g"].replay()

    for i in range(max(args.warmup, 3)):
        g_all.replay()
    torch.cuda.synchronize()
    for L in layers:
        st = ice.ice_check(L["err"])
        if st != ice.ICE_OK:
            raise SystemExit(f"device reported status {st}: {ice.ice_status_string(st)}")

    # ---- timed region: exactly `steps` decode steps (full passes over the layers, then the rest)
    sampler = ClockSampler(gpu_id_for(local))
    barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.15)
    t0, t1 = E(), E()
    t0.record()
    run_steps(False)
    t1.record()
    torch.cuda.synchronize()
    # the same steps writing the contiguous buffer (kbuf / vbuf / buf_len) as well
    t2, t3 = E(), E()
    t2.record()
    run_steps(True)
    t3.record()
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop()
    elapsed_ms = max_over_ranks(t0.elapsed_time(t1), world, "cuda")
    buf_ms = max_over_ranks(t2.elapsed_time(t3), world, "cuda")
    ms_step = elapsed_ms / args.steps
    # bytes of the timed steps: layer i % nl at step i
    per_step = [layers[i % nl]["bytes"] for i in range(nl)]
    bmin = float(np.mean([b[0] for b in per_step]))
    bbuf = float(np.mean([b[1] for b in per_step]))
    value = whole_job_rate(bmin, args.steps, world, elapsed_ms) / 1e9  # GB/s
    kernels = graph_kernel_nodes(layers[0]["g"])  # kernels of one step
    k_all = graph_kernel_nodes(g_all)
    launches = (k_all * full + (kernels or 0) * rest) if k_all is not None else None
    # per-step spread (median, p10, p90) with an L2 flush before each replay
    spread = rp(decode_call(ice, layers[0], budget, buf, False)) if rank == 0 else None
    sel_only = rp(lambda: ice.ice_select_pages(layers[0]["p"], layers[0]["idx"], layers[0]["Q"], budget,
                                               buf.sel_pages, buf.sel_count, buf.ws, layers[0]["err"])) if rank == 0 else None
    wanted = set(x for x in args.extras.split(",") if x) if args.extras != "none" else set()
    separate = separate_calls(ice, pk, rp, layers[0], buf, budget, w) if rank == 0 and "separate" in wanted else None
    build_ms = float(np.mean([L["build_ms"] for L in layers]))
    n_par = int(layers[0]["idx"].n_parents.sum())
    n_sel = layers[0]["n_sel"]
    status = ice.ice_status_string(ice.ice_check(layers[0]["err"]))
    del layers, L, buf, g_all, g_all_buf
    torch.cuda.empty_cache()

    # ---- end to end through the public API with host buffers (pinned host page pool)
    e2e, hp_extra = None, None
    try:
        if args.no_e2e:
            raise RuntimeError("skipped (--no-e2e)")
        e2e, hp_extra = host_pool_part(ice, pk, rp, w, budget, args.e2e_steps)
        slowest = max_over_ranks(e2e["ms_per_step"], world, "cuda")
        e2e["value"] = whole_job_rate(e2e.pop("bytes_per_step"), 1, world, slowest) / 1e9
        e2e["ms_per_step"] = r3(slowest)
    except Exception as e:  # reported; the contract line stands
        e2e = {"value": None, "unit": "GB/s", "error": f"{type(e).__name__}: {e}"[:200]}

    extra = {"buffer": {"us": r3(1000 * buf_ms / args.steps),
                        "frac_min": r3(bmin / (buf_ms / args.steps * 1e-3) / 1e9 / pk["hbm"]),
                        "frac_pipe": r3((bmin + bbuf) / (buf_ms / args.steps * 1e-3) / 1e9 / pk["hbm"])},
             "build": {"ms": r3(build_ms), "keys_s": r3(w.units * w.n_tokens / (build_ms * 1e-3))},
             "host_pool": hp_extra}
    if spread:
        extra["step"] = {"p10_us": r3(spread["p10"]), "med_us": r3(spread["us"]), "p90_us": r3(spread["p90"]),
                         "select_us": r3(sel_only["us"])}
    if separate:
        extra["separate"] = separate
    if rank == 0:
        parts = [("longchat", lambda: extra_longchat(ice, pk, rp, 1)),
                 ("longchat_b8", lambda: extra_longchat(ice, pk, rp, 8)),
                 ("qwen_levels3", lambda: extra_levels3(ice, pk, rp, w, budget)),
                 ("mistral_insert", lambda: extra_mistral_insert(ice, pk)),
                 ("llama16k", lambda: extra_llama16k(ice, pk, rp))]
        for name, fn in parts:
            if name not in wanted:
                continue
            try:
                extra[name] = fn()
            except Exception as e:  # reported under its name; the others still run
                extra[name] = {"error": f"{type(e).__name__}: {e}"[:200]}
            torch.cuda.empty_cache()
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        try:
            cpu = cpu_baseline_sample(w, budget, args.cpu_units)
        except Exception as e:
            cpu = {"error": f"{type(e).__name__}: {e}"[:200]}
    barrier()

    if rank == 0:
        ach = bmin / (ms_step * 1e-3) / 1e9
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded Gaussian-mixture KV drawn on the device)",
            "config": config_of(w, budget, world, args.layers),
            "decode_step_us": 1000 * ms_step,
            "roofline": {"kernel": "ice_decode_step" + (" (1 kernel)" if kernels == 1 else f" ({kernels} kernels)"),
                         "bound": "hbm", "achieved": ach, "peak": pk["hbm"], "unit": "GB/s", "frac": ach / pk["hbm"],
                         "peak_source": pk["src"], "bytes_per_launch": int(bmin),
                         "traffic": measured_traffic("decode", w.name) if w.batch == 16 else None},
            "index_build_keys_per_s": w.units * w.n_tokens / (build_ms * 1e-3),
            "e2e": e2e,
            "cpu_baseline": cpu,
            "gpu_launches": launches,
            "clocks": clocks,
            "device_status": status,
            "extra": extra,
        }
        if args.detail:
            with open(args.detail, "w") as f:
                json.dump(line, f, indent=1)
        print(json.dumps(line, indent=1), file=sys.stderr)  # every number, readable
        print(json.dumps(compact(line), separators=(",", ":")))
    if world > 1:
        dist.destroy_process_group()


def compact_config(c: dict) -> dict:
    """The workload config of the contract line in short form (both arms print it)."""
    return {"workload": c["workload"], "batch_per_gpu": c["batch_per_gpu"],
            "heads": f"{c['n_q_heads']}/{c['n_kv_heads']}", "n_tokens": c["n_tokens"],
            "budget_tokens": c["budget_tokens"], "levels": 2, "parallelism": c["parallelism"],
            "gather": "smem", "l2": c["l2"].split(" (")[0] + ", > 2.5x L2 per step",
            "graph": "one per pass over the layers", "workspace": "shared by the layers"}


def compact(d: dict) -> dict:
    """The contract line with every headline number and short keys (the
    full record goes to stderr and --detail)."""
    x = d["extra"]
    c = d["config"]
    g = lambda *ks: _get(x, ks)
    out = {k: d[k] for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                             "higher_is_better", "scaling", "vs_baseline", "dtype")}
    out["value"] = r3(d["value"])
    out["data"] = "synthetic"
    out["config"] = compact_config(c)
    out["decode_step_us"] = r3(d["decode_step_us"])
    rf = d["roofline"]
    out["roofline"] = {"kernel": rf["kernel"], "bound": "hbm", "achieved": r3(rf["achieved"]), "peak": rf["peak"],
                       "unit": "GB/s", "frac": r3(rf["frac"]), "traffic": rf["traffic"]}
    out["index_build_keys_per_s"] = r3(d["index_build_keys_per_s"])
    e = d["e2e"] or {}
    out["e2e"] = {"value": r3(e.get("value")), "unit": "GB/s", "h2d_bytes_per_step": e.get("h2d_bytes_per_step"),
                  "d2h_bytes_per_step": e.get("d2h_bytes_per_step"), "ms": e.get("ms_per_step"),
                  "direct": _get(e, ("direct", "value"))}
    cb = d["cpu_baseline"] or {}
    out["cpu_baseline"] = {"value": r3(cb.get("value")), "unit": cb.get("unit"), "cores": cb.get("cores"),
                           "kind": "oracle", "sample": cb.get("short", cb.get("error"))}
    out["gpu_launches"] = d["gpu_launches"]
    ck = d["clocks"]
    out["clocks"] = {"sm_mhz": ck["sm_mhz"], "sm_max_mhz": ck["sm_max_mhz"], "reasons": ck["reasons"]}
    out["status"] = d["device_status"]
    out["x"] = {"buf_us": g("buffer", "us"), "buf_frac": g("buffer", "frac_min"),
                "p10_p90": [g("step", "p10_us"), g("step", "p90_us")], "sel_us": g("step", "select_us"),
                "build_ms": g("build", "ms"),
                "lc1": [g("longchat", "d256", "us"), g("longchat", "d256", "frac"), g("longchat", "d64", "us")],
                "lc_assign_frac": g("longchat", "assign", "frac"),
                "lc8": [g("longchat_b8", "d256", "us"), g("longchat_b8", "d256", "frac")],
                "lc_steady": [g("longchat", "steady256", "us"), g("longchat", "steady256", "frac"),
                              g("longchat_b8", "steady256", "us"), g("longchat_b8", "steady256", "frac")],
                "lv3_us": g("qwen_levels3", "us"), "ins_us": g("mistral_insert", "insert_us"),
                "sep": [g("separate", "gather_us"), g("separate", "gather_frac"), g("separate", "attn_us"),
                        g("separate", "attn_frac")],
                "l16k": [g("llama16k", "build_us"), g("llama16k", "decode_us"), g("llama16k", "assign_frac")],
                "link": [g("host_pool", "link_peak_gbs"), g("host_pool", "bulk_frac"), g("host_pool", "direct_frac")]}
    return out


def _get(d, keys):
    for k in keys:
        if not isinstance(d, dict) or k not in d:
            return None
        d = d[k]
    return d


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
