#!/usr/bin/env python
"""Benchmark of the IceCache hot path on GB300.

One step = the whole hot path over one layer's batch: index build (lift and
promotion, nearest-parent assignment, page packing and pool scatter) and one
decode step (selection + GQA union, gather, masked sparse attention) at the
workload's largest budget.  value = keys indexed and decoded per second over
all ranks.  Each rank processes its own batch (weak scaling, no collective on
the data path; torch.distributed only carries the barrier and the max of the
timings).

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
REFERENCE_RUN_S = 150.0  # wall time the oracle (reference) arm aims for over all its steps
# kernels of one step when the captured graphs cannot be inspected: lift_count,
# promote_write, assign_tc, pack_cluster, pack_copy, and the decode (the
# per-unit cluster kernel, or score_tc + select_topk + attention)
def static_kernels_per_step(units: int, n_sm: int) -> int:
    return 5 + (1 if units * 8 <= n_sm else 3)


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

# CUDA-core fp32 peak from unit counts and clock: 152 SMs x 128 FMA/clk x 2 x 2.07 GHz
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12
# DRAM bytes per launch of a kernel from one ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum) on the named workload, with the SHA-256 of the kernel's
# source file at capture time; reported only while the source is unchanged.
TRAFFIC = {
    # profiles/assign_tc_llama31_8b_16k.md
    "assign": {"workload": "llama31_8b_16k", "source": "build_assign_tc.cu", "bytes": 40956672,
               "sha256": "e01fe4ae62b7ec7e6b47084d7878e058fb8969145da1313ee833a5079d099c20"},
}


def measured_traffic(kernel: str, workload: str):
    import hashlib
    t = TRAFFIC.get(kernel)
    if not t or t["workload"] != workload:
        return None
    src = os.path.join(ROOT, "semantic_paged_kv_gb300", "csrc", t["source"])
    try:
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
    except OSError:
        return None
    return t["bytes"] if sha == t["sha256"] else None


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama31_8b_16k")
    ap.add_argument("--budget", type=int, default=None)
    ap.add_argument("--sets", type=int, default=4, help="input sets rotated between steps (L2 stays cold)")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-units", type=int, default=None, help="units in the CPU-baseline sample")
    ap.add_argument("--no-at-scale", action="store_true",
                    help="skip the full-size decode and assignment timings (100k-token contexts)")
    ap.add_argument("--at-scale-only", action="store_true",
                    help="run only the full-size timings and print them as one JSON line (profiling runs)")
    ap.add_argument("--at-scale-parts",
                    default="qwen_decode,qwen_decode3,mistral_insert,qwen_host_pool,longchat_assign,longchat_decode",
                    help="comma list of qwen_decode, qwen_decode3, mistral_insert, qwen_host_pool, longchat_assign, "
                         "longchat_decode")
    ap.add_argument("--at-scale-batch", type=int, default=None, help="sequences of the Qwen3-shaped batch (16)")
    ap.add_argument("--at-scale-reps", type=int, default=30)
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


def oracle_sample(w: workloads.Workload, budget: int, units: int, n_tokens: int | None = None, passes: int = 1,
                  min_seconds: float = 0.0, max_seconds: float = float("inf")):
    """Time the oracle (as it stands) on `units` units of the workload: build
    (a1-a5) and one decode step (a6-a10), one unit per host thread.  With
    n_tokens, each unit is the first n_tokens tokens of the workload's unit
    (same mixture).  The pass over the units repeats `passes` times, and more
    while under min_seconds (never starting one past max_seconds).  Returns
    (seconds, passes run, threads)."""
    import oracle
    th = oracle.promote_threshold(w.promote_p)
    items = [(u // w.n_kv_heads, u % w.n_kv_heads) for u in range(units)]
    data = {it: (workloads.unit_kv(w, 0, *it, n_tokens=n_tokens), workloads.unit_queries(w, 0, *it))
            for it in items}

    def one(it):
        (K, V), q = data[it]
        idx = oracle.build_unit(K, V, seed=w.seed, layer=0, seq=it[0], head=it[1], thresh=th, S=w.page_size)
        oracle.decode_unit(idx, q, budget)

    oracle.build()
    t0 = time.perf_counter()
    done, threads = 0, 1
    while True:
        _, threads = oracle.run_units(one, items, threads=min(units, os.cpu_count() or 1))
        done += 1
        dt = time.perf_counter() - t0
        if done >= passes and (dt >= min_seconds or dt * (done + 1) / done > max_seconds):
            break
    return dt, done, threads


def run_reference(args):
    rank, _, world = rank_info()
    if rank != 0:
        return  # the oracle arm runs on rank 0 only
    w = workloads.WORKLOADS[args.workload]
    budget = args.budget or max(w.budgets)
    units = args.cpu_units or min(w.units, os.cpu_count() or 1)
    # each step is a bounded sample: the whole run stays near REFERENCE_RUN_S.
    # A full-N pass over the units is timed once; if K + W such passes would
    # take longer, every step builds the first n' tokens of the same units
    # instead (the oracle's cost grows about as N^2, so n' = N sqrt(share)).
    probe, _, threads = oracle_sample(w, budget, units)
    per_step = REFERENCE_RUN_S / (args.steps + args.warmup)
    n_tok = w.n_tokens
    if probe > per_step:
        n_tok = max(256, int(w.n_tokens * math.sqrt(per_step / probe)))
    times = []
    for i in range(args.warmup + args.steps):
        dt, _, threads = oracle_sample(w, budget, units, n_tokens=n_tok)
        if i >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = units * n_tok * len(times) / total
    sample = (f"{units} of {w.units} units (KV heads) per step, one per host thread, "
              + (f"full N={w.n_tokens}" if n_tok == w.n_tokens else
                 f"first {n_tok} of the N={w.n_tokens} tokens of each unit (a full-N pass took {probe:.1f} s; "
                 f"the oracle's cost per key grows with N, so this rate is above its full-N rate)")
              + f", index build + one decode step at budget {budget}")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "keys/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * total / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, budget, args.gpus, args.sets),
        "cpu_baseline": {"value": value, "unit": "keys/s", "cores": threads, "kind": "oracle", "sample": sample,
                         "cpu": host_cpu()},
        "e2e": {"value": value, "unit": "keys/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def config_of(w, budget, gpus, sets):
    return {"workload": w.name, "batch_per_gpu": w.batch, "n_q_heads": w.n_q_heads, "n_kv_heads": w.n_kv_heads,
            "n_tokens": w.n_tokens, "head_dim": w.head_dim, "page_size": w.page_size, "promote_p": w.promote_p,
            "levels": 2, "budget_tokens": budget, "layers_per_step": 1, "parallelism": f"dp{gpus}",
            "l2": f"inputs rotated over {sets} sets between steps (each set larger than half of L2; "
                  f"{sets} sets > 4x L2 combined)"}


# ------------------------------------------------- multi-rank host logic ---
def rank_workload(name: str, rank: int) -> workloads.Workload:
    """Each rank owns its own batch of the workload: same shapes, its own
    seed, so the ranks' units are disjoint and need no exchange."""
    base = workloads.WORKLOADS[name]
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


def whole_job_rate(units_per_rank: int, per_unit: int, steps: int, world: int, max_ms: float) -> float:
    """Work of all ranks over the slowest rank's time (weak scaling)."""
    return world * units_per_rank * per_unit * steps / (max_ms * 1e-3)


# ------------------------------------------------------------- our arm ----
def at_scale(pk, reps: int = 30, parts=("qwen_decode", "qwen_decode3", "mistral_insert", "qwen_host_pool",
                                        "longchat_assign", "longchat_decode"), qwen_batch=None):
    """Full-size timings of the two parts the roofline targets are quoted on:
    the decode step (select + gather + sparse attention) of the Qwen3-32B-
    shaped batch (16 sequences x 8 KV heads, 100k tokens, budget 256) and of
    the LongChat-7B-shaped one (batch 1, 32 KV heads, 100k tokens), and the
    parent-assignment contraction at 100k tokens (LongChat shape).  Inputs are
    drawn on the device (same mixture recipe as the host generator); each
    timed launch is one CUDA graph replay after an L2 flush, median of
    `reps`, CUDA events on the launching stream."""
    import torch

    import semantic_paged_kv_gb300 as ice

    E = lambda: torch.cuda.Event(enable_timing=True)
    # L2 flush before each timed replay: write a buffer of 2x L2, then read
    # another one of 2x L2, so that the flush's own dirty lines are written
    # back before the timed region instead of inside it
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda")
    evict = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
    sink = torch.empty((), dtype=torch.float32, device="cuda")
    cap = torch.cuda.Stream()

    spread = {}  # p10 and p90 (ms) of the replays of the last timed call

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        cap.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            fn()
        torch.cuda.current_stream().wait_stream(cap)
        ts = []
        for _ in range(reps):
            flush.zero_()
            torch.sum(evict, dim=0, out=sink)
            a, b = E(), E()
            a.record()
            g.replay()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        spread["p10"], spread["p90"] = float(np.percentile(ts, 10)), float(np.percentile(ts, 90))
        return statistics.median(ts)  # ms

    def build(w, n_levels=2):
        cfg = ice.Config(batch=w.batch, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads, n_tokens=w.n_tokens,
                         dtype=ice.ICE_BF16, promote_p=w.promote_p, seed=w.seed, n_levels=n_levels)
        K, V, C = workloads.batch_kv_device(w)
        Q = workloads.batch_queries_device(w, C)
        del C
        p = cfg.params()
        idx = ice.Index(cfg)
        ws = ice.workspace(ice.ice_build_workspace_bytes(p))
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        ice.ice_build_index(p, K, V, idx, ws, err)
        torch.cuda.synchronize()
        return cfg, p, K, V, Q, idx, ws, err

    def decode(cfg, p, Q, idx, err, budget):
        buf = ice.DecodeBuffers(cfg, budget)
        scale = 1.0 / math.sqrt(cfg.head_dim)
        ms = timed(lambda: ice.ice_decode_step(p, idx, Q, budget, buf.sel_pages, buf.sel_count, buf.kbuf, buf.vbuf,
                                               buf.buf_len, scale, buf.O, buf.ws, err))
        us_p10, us_p90 = 1000 * spread["p10"], 1000 * spread["p90"]
        # the selection alone (score table + per-unit top-k and union), same flush
        ms_sel = timed(lambda: ice.ice_select_pages(p, idx, Q, budget, buf.sel_pages, buf.sel_count, buf.ws, err))
        # the same step without the contiguous buffer (pages gathered on chip only)
        ms_nb = timed(lambda: ice.ice_decode_step(p, idx, Q, budget, buf.sel_pages, buf.sel_count, None, None, None,
                                                  scale, buf.O, buf.ws, err))
        d, S = 128, 16
        np_tot = int(idx.n_parents.sum())
        sel_tot = int(buf.sel_count.sum())
        qo = cfg.batch * cfg.n_q_heads * d * (2 + 4)
        b_min = np_tot * d * 2 + sel_tot * S * d * 2 * 2 + qo
        b_pipe = b_min + sel_tot * S * d * 2 * 2
        gbs_min, gbs_pipe = b_min / (ms * 1e-3) / 1e9, b_pipe / (ms * 1e-3) / 1e9
        return {"us": 1000 * ms, "us_p10": us_p10, "us_p90": us_p90, "select_only_us": 1000 * ms_sel,
                "budget_tokens": budget, "parents": np_tot, "selected_pages": sel_tot,
                "bytes_min": b_min, "hbm_gbs_min_bytes": gbs_min, "frac_min_bytes": gbs_min / pk["hbm"],
                "bytes_pipeline": b_pipe, "hbm_gbs_pipeline_bytes": gbs_pipe, "frac_pipeline_bytes": gbs_pipe / pk["hbm"],
                "no_buffer": {"us": 1000 * ms_nb, "bytes": b_min,
                              "hbm_gbs": b_min / (ms_nb * 1e-3) / 1e9,
                              "frac": b_min / (ms_nb * 1e-3) / 1e9 / pk["hbm"],
                              "what": "ice_decode_step with kbuf = vbuf = buf_len = NULL: selected pages gathered "
                                      "into shared memory only; bytes = the minimum (parent tables + selected pages "
                                      "once + Q/O)"}}

    out = {"inputs": "drawn on the device with torch's generator (same mixture recipe as the host draws)",
           "timing": f"median of {reps} CUDA-graph replays, CUDA events; before each, L2 flushed by a 2x L2 write "
                     f"and then a 2x L2 read of another buffer (no dirty flush lines left for the timed region)",
           "peak_source": pk["src"]}
    # Qwen3-32B shape: decode step
    def part_qwen_decode():
        w = workloads.WORKLOADS["qwen3_32b_100k"]
        if qwen_batch:
            w = w.scaled(batch=qwen_batch)
        cfg, p, K, V, Q, idx, ws, err = build(w)
        a, b = E(), E()  # a second build of the same layer, timed
        a.record()
        ice.ice_build_index(p, K, V, idx, ws, err)
        b.record()
        torch.cuda.synchronize()
        build_ms = a.elapsed_time(b)
        del K, V, ws
        key = f"decode_qwen3_32b_100k_b{w.batch}"
        out[key] = decode(cfg, p, Q, idx, err, max(w.budgets))
        out[key]["build_ms"] = build_ms
        out[key]["build_keys_per_s"] = w.batch * w.n_kv_heads * w.n_tokens / (build_ms * 1e-3)
        out[key]["status"] = ice.ice_status_string(ice.ice_check(err))
        del cfg, p, Q, idx, err
        torch.cuda.empty_cache()
    # Qwen3-32B shape with a third index level: the descent reads the level-2
    # table and the chosen nodes' children instead of the whole parent table
    def part_qwen_decode3():
        w = workloads.WORKLOADS["qwen3_32b_100k"]
        if qwen_batch:
            w = w.scaled(batch=qwen_batch)
        cfg, p, K, V, Q, idx, ws, err = build(w, n_levels=3)
        a, b = E(), E()  # a second build of the same layer, timed (two and three levels differ by level 2)
        a.record()
        ice.ice_build_index(p, K, V, idx, ws, err)
        b.record()
        torch.cuda.synchronize()
        build3_ms = a.elapsed_time(b)
        del K, V, ws
        budget = max(w.budgets)
        buf = ice.DecodeBuffers(cfg, budget)
        scale = 1.0 / math.sqrt(cfg.head_dim)
        ms = timed(lambda: ice.ice_decode_step(p, idx, Q, budget, buf.sel_pages, buf.sel_count, buf.kbuf, buf.vbuf,
                                               buf.buf_len, scale, buf.O, buf.ws, err))
        ms_nb = timed(lambda: ice.ice_decode_step(p, idx, Q, budget, buf.sel_pages, buf.sel_count, None, None, None,
                                                  scale, buf.O, buf.ws, err))
        ms_sel = timed(lambda: ice.ice_select_pages(p, idx, Q, budget, buf.sel_pages, buf.sel_count, buf.ws, err))
        n2 = int(idx.n_nodes2.sum())
        sel_tot = int(buf.sel_count.sum())
        out[f"decode3_qwen3_32b_100k_b{w.batch}"] = {
            "us": 1000 * ms, "no_buffer_us": 1000 * ms_nb, "select_only_us": 1000 * ms_sel, "budget_tokens": budget,
            "build_ms": build3_ms,
            "level2_nodes": n2, "parents": int(idx.n_parents.sum()), "selected_pages": sel_tot,
            "what": "n_levels = 3: per head the best k level-2 nodes, then their children; the level-2 table "
                    f"({n2 * 256 / 1e6:.1f} MB) replaces the parent-table scan",
            "status": ice.ice_status_string(ice.ice_check(err))}
        del cfg, p, Q, idx, err, buf
        torch.cuda.empty_cache()
    # Mistral-7B shape: 128 decode steps, each inserting one token per unit
    # first (step a11), the index growing from the 36,864-token build
    def part_mistral_insert():
        w = workloads.WORKLOADS["mistral_7b_36k"]
        steps = 128
        cfg = ice.Config(batch=w.batch, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads, n_tokens=w.n_tokens,
                         dtype=ice.ICE_BF16, promote_p=w.promote_p, seed=w.seed, n_cap=w.n_tokens + steps)
        K, V, C = workloads.batch_kv_device(w)
        Q = workloads.batch_queries_device(w, C)
        p = cfg.params()
        idx = ice.Index(cfg)
        ws = ice.workspace(ice.ice_build_workspace_bytes(p))
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        ice.ice_build_index(p, K, V, idx, ws, err)
        U = cfg.units
        gen = torch.Generator(device="cuda")
        gen.manual_seed(w.seed * 7919 + 11)
        lab = torch.randint(0, w.centres, (steps, U), generator=gen, device="cuda")
        kn = (C[torch.arange(U, device="cuda")[None, :], lab]
              + w.spread * torch.randn((steps, U, 128), generator=gen, device="cuda")).to(torch.bfloat16)
        vn = torch.randn((steps, U, 128), generator=gen, device="cuda").to(torch.bfloat16)
        del K, V, C, ws
        budget = max(w.budgets)
        buf = ice.DecodeBuffers(cfg, budget)
        wsi = ice.workspace(ice.ice_insert_workspace_bytes(p))
        scale = 1.0 / math.sqrt(cfg.head_dim)
        np0 = int(idx.n_parents.sum())
        torch.cuda.synchronize()
        evs = [(E(), E(), E()) for _ in range(steps)]
        for st, (a, b, c) in enumerate(evs):
            a.record()
            ice.ice_insert_tokens(p, idx, kn[st], vn[st], wsi, err)
            b.record()
            ice.ice_decode_step(p, idx, Q, budget, buf.sel_pages, buf.sel_count, buf.kbuf, buf.vbuf, buf.buf_len,
                                scale, buf.O, buf.ws, err)
            c.record()
        torch.cuda.synchronize()
        t_ins = [a.elapsed_time(b) for a, b, _ in evs]
        t_dec = [b.elapsed_time(c) for _, b, c in evs]
        np_avg = (np0 + int(idx.n_parents.sum())) / 2
        ins_bytes = np_avg * 128 * 2 + U * 128 * 2 * 2 * 2  # the parent scan, the new K/V rows in and into the pool
        ins_us = 1000 * statistics.median(t_ins)
        out["insert_mistral_7b_36k"] = {
            "steps": steps, "units": U, "insert_us": ins_us, "decode_step_us": 1000 * statistics.median(t_dec),
            "insert_bytes": ins_bytes, "insert_hbm_gbs": ins_bytes / (ins_us * 1e-6) / 1e9,
            "tokens_after": int(idx.n_indexed.sum()), "parents_after": int(idx.n_parents.sum()),
            "pages_after": int(idx.n_pages.sum()),
            "timing": "median over the 128 steps of eager launches, CUDA events around each call, index warm "
                      "(no L2 flush: the decode loop reuses it)",
            "status": ice.ice_status_string(ice.ice_check(err))}
        del cfg, p, Q, idx, err, buf, kn, vn, wsi
        torch.cuda.empty_cache()
    # Qwen3-32B shape with the page pool in pinned host memory (step a12)
    def part_qwen_host_pool():
        w = workloads.WORKLOADS["qwen3_32b_100k"]
        if qwen_batch:
            w = w.scaled(batch=qwen_batch)
        cfg = ice.Config(batch=w.batch, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads, n_tokens=w.n_tokens,
                         dtype=ice.ICE_BF16, promote_p=w.promote_p, seed=w.seed)
        budget = max(w.budgets)
        max_sel = ice.max_selected(cfg, budget)
        hp = ice.HostPool(cfg, max_sel, n_threads=min(16, os.cpu_count() or 1))
        try:
            K, V, C = workloads.batch_kv_device(w)
            Q = workloads.batch_queries_device(w, C)
            p = cfg.params()
            idx = ice.Index(cfg, host_pool=hp)
            ws = ice.workspace(ice.ice_build_workspace_bytes(p))
            err = torch.zeros(1, dtype=torch.int32, device="cuda")
            ice.ice_build_index(p, K, V, idx, ws, err)
            torch.cuda.synchronize()
            del K, V, C, ws
            buf = ice.DecodeBuffers(cfg, budget)
            scale = 1.0 / math.sqrt(cfg.head_dim)
            # direct: the fused decode reads the selected pages from host memory over the CPU-GPU link
            ms_direct = timed(lambda: ice.ice_decode_step(p, idx, Q, budget, buf.sel_pages, buf.sel_count, buf.kbuf,
                                                          buf.vbuf, buf.buf_len, scale, buf.O, buf.ws, err))
            sel_tot = int(buf.sel_count.sum())
            page_bytes = sel_tot * 16 * 128 * 2 * 2
            # staged: selection on the device, ids to the host, host threads gather the pages into pinned
            # staging, one bulk cudaMemcpyAsync, attention over the copy
            dst = torch.empty(hp.staging_bytes, dtype=torch.uint8, device="cuda")
            plen_h = idx.page_len.cpu()
            U, S, d = cfg.units, cfg.page_size, cfg.head_dim
            nb = U * max_sel * S * d * 2
            kbuf = dst[:nb].view(torch.bfloat16).view(U, max_sel, S, d)
            vbuf = dst[nb:2 * nb].view(torch.bfloat16).view(U, max_sel, S, d)
            blen = dst[2 * nb:2 * nb + U * max_sel * 4].view(torch.int32).view(U, max_sel)
            wall = []
            for r in range(5):
                torch.cuda.synchronize()
                t0 = time.perf_counter()
                ice.ice_select_pages(p, idx, Q, budget, buf.sel_pages, buf.sel_count, buf.ws, err)
                sel_h, cnt_h = buf.sel_pages.cpu(), buf.sel_count.cpu()
                ice.ice_host_pool_gather_h2d(hp, p, sel_h, cnt_h, plen_h, max_sel, dst)
                ice.ice_sparse_attn_decode(p, Q, kbuf, vbuf, blen, buf.sel_count, scale, buf.O, buf.ws)
                torch.cuda.synchronize()
                wall.append(time.perf_counter() - t0)
            # the bulk copy alone: the same bytes, pinned host to device, one cudaMemcpyAsync
            src = torch.empty(hp.staging_bytes, dtype=torch.uint8).pin_memory()
            a, b = E(), E()
            a.record()
            dst.copy_(src, non_blocking=True)
            b.record()
            torch.cuda.synchronize()
            h2d_ms = a.elapsed_time(b)
            out[f"host_pool_qwen3_32b_100k_b{w.batch}"] = {
                "direct_decode_us": 1000 * ms_direct, "direct_page_bytes": page_bytes,
                "direct_link_gbs": page_bytes / (ms_direct * 1e-3) / 1e9,
                "staged_step_ms": 1000 * statistics.median(wall), "staging_bytes": hp.staging_bytes,
                "bulk_h2d_ms": h2d_ms, "bulk_h2d_gbs": hp.staging_bytes / (h2d_ms * 1e-3) / 1e9,
                "host_pool_bytes": 2 * hp.pool_bytes, "host_threads": min(16, os.cpu_count() or 1),
                "timing": "direct: CUDA-graph replays as above; staged: wall clock of select + ids to host + host "
                          "gather + one H2D + attention, median of 5",
                "status": ice.ice_status_string(ice.ice_check(err))}
            del idx, buf, dst, src, kbuf, vbuf, blen
        finally:
            hp.close()
        torch.cuda.empty_cache()
    # LongChat-7B shape: the assignment contraction at 100k tokens, then decode
    def part_longchat():
        w = workloads.WORKLOADS["longchat_7b_100k"]
        cfg, p, K, V, Q, idx, ws, err = build(w)
        if "longchat_assign" in parts:
            ms = timed(lambda: ice.ice_build_assign(p, K, idx, ws, err))
            np_tot = int(idx.n_parents.sum())
            flops = 2.0 * w.n_tokens * np_tot * 128
            tf = flops / (ms * 1e-3) / 1e12
            out["assign_longchat_7b_100k"] = {"us": 1000 * ms, "units": cfg.units, "tokens_per_unit": w.n_tokens,
                                              "parents": np_tot, "flops": flops, "tflops": tf,
                                              "peak_tflops": pk["bf16"], "frac": tf / pk["bf16"],
                                              "peak": "bf16 dense, measured burst"}
        del K, V, ws
        if "longchat_decode" in parts:
            out["decode_longchat_7b_100k_b1"] = decode(cfg, p, Q, idx, err, max(w.budgets))
        out["status"] = ice.ice_status_string(ice.ice_check(err))
        del cfg, p, Q, idx, err
    # each part on its own: a failure is reported under the part's name and the others still run
    for name, fn, wanted in (("qwen_decode", part_qwen_decode, "qwen_decode" in parts),
                             ("qwen_decode3", part_qwen_decode3, "qwen_decode3" in parts),
                             ("mistral_insert", part_mistral_insert, "mistral_insert" in parts),
                             ("qwen_host_pool", part_qwen_host_pool, "qwen_host_pool" in parts),
                             ("longchat", part_longchat, "longchat_assign" in parts or "longchat_decode" in parts)):
        if not wanted:
            continue
        try:
            fn()
        except Exception as e:  # reported, the other parts stand
            out[f"{name}_error"] = f"{type(e).__name__}: {e}"
        torch.cuda.empty_cache()
    del flush, evict, sink
    torch.cuda.empty_cache()
    return out


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

    w = rank_workload(args.workload, rank)
    budget = args.budget or max(w.budgets)
    cfg = ice.Config(batch=w.batch, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads, n_tokens=w.n_tokens,
                     dtype=ice.ICE_BF16 if w.dtype == "bf16" else ice.ICE_FP32, promote_p=w.promote_p, seed=w.seed)
    dt = cfg.torch_dtype
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(w.head_dim)
    sets = []
    for s in range(args.sets):
        K, V = workloads.batch_kv(w, layer=s)
        Q = workloads.batch_queries(w, layer=s)
        c = ice.Config(**{**cfg.__dict__, "layer": s})
        p = c.params()
        st = dict(cfg=c, params=p, Kh=torch.from_numpy(K).to(dt).pin_memory(), Vh=torch.from_numpy(V).to(dt).pin_memory(),
                  Qh=torch.from_numpy(Q).to(dt).pin_memory())
        st["K"], st["V"], st["Q"] = st["Kh"].cuda(), st["Vh"].cuda(), st["Qh"].cuda()
        st["idx"] = ice.Index(c)
        st["ws"] = ice.workspace(ice.ice_build_workspace_bytes(p))
        st["buf"] = ice.DecodeBuffers(c, budget)
        st["idx_reuse"] = ice.Index(c)  # this layer built on the previous set's node structure
        st["Oh"] = torch.empty_like(st["buf"].O, device="cpu").pin_memory()
        sets.append(st)
    set_bytes = sum(x.numel() * x.element_size() for x in (sets[0]["K"], sets[0]["V"], sets[0]["idx"].pool_k,
                                                           sets[0]["idx"].pool_v))

    # the four stages of a step, each a call into the C ABI
    def stages(st):
        p, idx, buf = st["params"], st["idx"], st["buf"]
        return [
            lambda: ice.ice_build_lift_promote(p, st["K"], idx, st["ws"], err),
            lambda: ice.ice_build_assign(p, st["K"], idx, st["ws"], err),
            lambda: ice.ice_build_pack(p, st["K"], st["V"], idx, st["ws"], err),
            lambda: ice.ice_decode_step(p, idx, st["Q"], budget, buf.sel_pages, buf.sel_count, buf.kbuf, buf.vbuf,
                                        buf.buf_len, scale, buf.O, buf.ws, err),
        ]

    for i in range(max(args.warmup, 3)):
        for f in stages(sets[i % len(sets)]):
            f()
    torch.cuda.synchronize()
    status = ice.ice_check(err)
    if status != ice.ICE_OK:
        raise SystemExit(f"device reported status {status}: {ice.ice_status_string(status)}")
    # capture each stage of each input set in a CUDA graph (launch overhead off the host)
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    for st in sets:
        st["graphs"] = []
        for f in stages(st):
            try:
                g, kept = torch.cuda.CUDAGraph(keep_graph=True), True  # keeps the graph for node inspection
            except TypeError:
                g, kept = torch.cuda.CUDAGraph(), False
            with torch.cuda.graph(g, stream=cap):
                f()
            if kept:
                g.instantiate()
            st["graphs"].append(g)
        # the whole step (build + decode of the layer) as one graph: the timed loop
        st["step_graph"] = torch.cuda.CUDAGraph()
        with torch.cuda.graph(st["step_graph"], stream=cap):
            for f in stages(st):
                f()
    # the inter-layer reuse build of each set on the previous set's index
    for i, st in enumerate(sets):
        prev = sets[(i - 1) % len(sets)]["idx"]
        st["reuse"] = (lambda st=st, prev=prev: ice.ice_build_index_reuse(st["params"], st["K"], st["V"], prev,
                                                                          st["idx_reuse"], st["ws"], err))
        st["reuse_graph"] = torch.cuda.CUDAGraph()
        with torch.cuda.graph(st["reuse_graph"], stream=cap):
            st["reuse"]()
    torch.cuda.current_stream().wait_stream(cap)
    torch.cuda.synchronize()

    def step(st, evs=None):
        if evs is None:
            st["step_graph"].replay()
            return
        for k, g in enumerate(st["graphs"]):
            evs[k].record()
            g.replay()
        evs[4].record()

    E = lambda: torch.cuda.Event(enable_timing=True)
    for i in range(2 * len(sets)):  # warm the graphs
        step(sets[i % len(sets)])
        step(sets[i % len(sets)], [E() for _ in range(5)])
    for st in sets:  # every set's index is built now
        st["reuse_graph"].replay()

    # ---- timed region: exactly `steps` steps, each one whole-step graph
    evs = [[E() for _ in range(5)] for _ in range(args.steps)]
    sampler = ClockSampler(gpu_id_for(local))
    barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.15)
    t0, t1 = E(), E()
    t0.record()
    for i in range(args.steps):
        step(sets[i % len(sets)])
    t1.record()
    torch.cuda.synchronize()
    # the same steps again with one graph per stage and events between them:
    # the per-kernel durations of the phases and the roofline
    for i in range(args.steps):
        step(sets[i % len(sets)], evs[i])
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop()
    elapsed_ms = max_over_ranks(t0.elapsed_time(t1), world, "cuda")
    stage = np.array([[e[k].elapsed_time(e[k + 1]) for k in range(4)] for e in evs])  # ms
    lift_ms, assign_ms, pack_ms, decode_ms = stage.mean(0)
    # the reuse build, timed the same way (sets rotated, one graph per build)
    rev = [(E(), E()) for _ in range(args.steps)]
    for i in range(args.steps):
        rev[i][0].record()
        sets[i % len(sets)]["reuse_graph"].replay()
        rev[i][1].record()
    torch.cuda.synchronize()
    reuse_ms = float(np.mean([a.elapsed_time(b) for a, b in rev]))

    # ---- algorithmic work of a step (averaged over the sets)
    d, S, U, N = w.head_dim, w.page_size, cfg.units, w.n_tokens
    esz = 2 if w.dtype == "bf16" else 4
    np_tot = np.mean([int(s["idx"].n_parents.sum()) for s in sets])
    pages_tot = np.mean([int(s["idx"].n_pages.sum()) for s in sets])
    sel_tot = np.mean([int(s["buf"].sel_count.sum()) for s in sets])
    flops_assign = 2.0 * N * np_tot * d
    qo_bytes = cfg.batch * cfg.n_q_heads * d * (esz + 4)
    decode_min_bytes = np_tot * d * esz + sel_tot * S * d * esz * 2 + qo_bytes
    decode_pipe_bytes = decode_min_bytes + sel_tot * S * d * esz * 2  # + the contiguous-buffer write
    pack_bytes = 2 * U * N * d * esz + 2 * pages_tot * S * d * esz
    lift_bytes = U * N * d * esz + np_tot * d * esz
    pk = peaks()
    n_sm = torch.cuda.get_device_properties(local).multi_processor_count
    cands = {
        "assign": (assign_ms, "tensor", flops_assign / (assign_ms * 1e-3) / 1e12, pk["bf16"], "TFLOP/s", flops_assign),
        "pack": (pack_ms, "hbm", pack_bytes / (pack_ms * 1e-3) / 1e9, pk["hbm"], "GB/s", pack_bytes),
        "lift_promote": (lift_ms, "hbm", lift_bytes / (lift_ms * 1e-3) / 1e9, pk["hbm"], "GB/s", lift_bytes),
        "decode": (decode_ms, "hbm", decode_min_bytes / (decode_ms * 1e-3) / 1e9, pk["hbm"], "GB/s", decode_min_bytes),
    }
    if w.dtype != "bf16":
        cands["assign"] = (assign_ms, "alu", flops_assign / (assign_ms * 1e-3) / 1e12, FP32_ALU_TFLOPS, "TFLOP/s",
                           flops_assign)
    # the roofline is reported for the dominant KERNEL: the stages that are one
    # kernel each (parent assignment; decode when it runs as the per-unit
    # cluster kernel); the other stages are reported in "phases"
    single = ["assign"] + (["decode"] if cfg.units * 8 <= n_sm else [])
    dom = max(single, key=lambda k: cands[k][0])
    ms_, bound, ach, peak, unit, work = cands[dom]
    per_step = [graph_kernel_nodes(g) for g in sets[0]["graphs"]]
    kernels_per_step = sum(per_step) if all(x is not None for x in per_step) else static_kernels_per_step(
        cfg.units, n_sm)
    value = whole_job_rate(U, N, args.steps, world, elapsed_ms)

    # ---- end to end with host buffers: H2D of the inputs, the step, D2H of O
    e2e_steps = args.e2e_steps or min(args.steps, 100)
    h2d_bytes = sum(sets[0][k].numel() * sets[0][k].element_size() for k in ("Kh", "Vh", "Qh"))
    d2h = sets[0]["Oh"].numel() * 4
    barrier()
    torch.cuda.synchronize()
    a, b_ = E(), E()
    a.record()
    for i in range(e2e_steps):
        st = sets[i % len(sets)]
        st["K"].copy_(st["Kh"], non_blocking=True)
        st["V"].copy_(st["Vh"], non_blocking=True)
        st["Q"].copy_(st["Qh"], non_blocking=True)
        step(st)
        st["Oh"].copy_(st["buf"].O, non_blocking=True)
    b_.record()
    torch.cuda.synchronize()
    e2e_serial_ms = max_over_ranks(a.elapsed_time(b_), world, "cuda")
    # the same with the next layer's host-to-device copy on a second stream
    # while this layer is built and decoded (the on-device form of the pages'
    # copy / index / compute pipeline): copies of step i + 1 overlap step i
    cs, xs = torch.cuda.Stream(), torch.cuda.current_stream()
    copied = [torch.cuda.Event() for _ in range(e2e_steps)]
    done = [torch.cuda.Event() for _ in range(e2e_steps)]

    def h2d(i):
        st = sets[i % len(sets)]
        with torch.cuda.stream(cs):
            if i >= len(sets):
                cs.wait_event(done[i - len(sets)])  # the set's buffers are free again
            st["K"].copy_(st["Kh"], non_blocking=True)
            st["V"].copy_(st["Vh"], non_blocking=True)
            st["Q"].copy_(st["Qh"], non_blocking=True)
            copied[i].record(cs)

    barrier()
    torch.cuda.synchronize()
    a, b_ = E(), E()
    a.record()
    cs.wait_stream(xs)
    h2d(0)
    for i in range(e2e_steps):
        if i + 1 < e2e_steps:
            h2d(i + 1)
        st = sets[i % len(sets)]
        xs.wait_event(copied[i])
        step(st)
        st["Oh"].copy_(st["buf"].O, non_blocking=True)
        done[i].record(xs)
    b_.record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(a.elapsed_time(b_), world, "cuda")
    e2e_value = whole_job_rate(U, N, e2e_steps, world, e2e_ms)
    compute_ms = elapsed_ms / args.steps * e2e_steps
    copy_ms = max(e2e_serial_ms - compute_ms, 1e-9)
    hidden = min(1.0, max(0.0, (e2e_serial_ms - e2e_ms) / min(copy_ms, compute_ms)))
    status = ice.ice_check(err)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        units = args.cpu_units or min(U, os.cpu_count() or 1)
        cdt, passes, threads = oracle_sample(w, budget, units, min_seconds=10.0, max_seconds=30.0)
        cpu = {"value": passes * units * N / cdt, "unit": "keys/s", "cores": threads, "kind": "oracle",
               "cpu": host_cpu(),
               "sample": f"{units} of {U} units (KV heads) of this workload, full N={N}: index build + one decode "
                         f"step at budget {budget}, one unit per host thread, {passes} passes ({cdt:.1f} s)"}

    scale_res = None
    if rank == 0 and not args.no_at_scale:
        try:
            scale_res = at_scale(pk, args.at_scale_reps, args.at_scale_parts.split(","), args.at_scale_batch)
        except Exception as e:  # reported, the main line stands
            scale_res = {"error": f"{type(e).__name__}: {e}"}
    barrier()

    if rank == 0:
        tr = measured_traffic(dom, w.name)
        line = {
            "metric": METRIC, "value": value, "unit": "keys/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": config_of(w, budget, world, args.sets),
            "phases": {
                "decode_step_us": 1000 * decode_ms,
                "decode_hbm_gbs_min_bytes": decode_min_bytes / (decode_ms * 1e-3) / 1e9,
                "decode_hbm_gbs_pipeline_bytes": decode_pipe_bytes / (decode_ms * 1e-3) / 1e9,
                "index_build_keys_per_s": U * N / ((lift_ms + assign_ms + pack_ms) * 1e-3),
                "build_us": {"lift_promote": 1000 * lift_ms, "assign": 1000 * assign_ms, "pack": 1000 * pack_ms},
                "assign_tflops": flops_assign / (assign_ms * 1e-3) / 1e12,
                "build_reuse_us": 1000 * reuse_ms,
                "index_build_reuse_keys_per_s": U * N / (reuse_ms * 1e-3),
                "build_reuse_as": "ice_build_index_reuse of each input set on the previous set's index (inter-layer "
                                  "reuse: lift, parent keys, table copies, pool; no assignment, no ranking)",
                "parents_per_step": np_tot, "pages_per_step": pages_tot, "selected_pages_per_step": sel_tot,
                "set_bytes": set_bytes,
                "stages_as": "a second timed pass of the same steps: one CUDA graph per stage, events between them "
                             "(the step value replays one graph per step)",
                "stage_gbs": {k: cands[k][2] for k in ("lift_promote", "pack", "decode")},
            },
            "roofline": {"kernel": dom, "bound": bound, "achieved": ach, "peak": peak, "unit": unit,
                         "frac": ach / peak, "peak_source": pk["src"] + (" burst" if bound == "tensor" else ""),
                         "work_per_launch": work, "traffic": tr},
            "at_scale": scale_res,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "keys/s", "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h,
                    "steps": e2e_steps,
                    "how": "every step: H2D of its K, V, Q from pinned host memory, the step (index build + decode, "
                           "one CUDA graph), D2H of O; the next step's H2D runs on a second stream during this step",
                    "serial_value": whole_job_rate(U, N, e2e_steps, world, e2e_serial_ms),
                    "hidden_fraction": hidden,
                    "hidden_fraction_is": "(serial - overlapped time) / min(copy time, compute time), at most 1; "
                                          "copy time = serial time - device-only step time"},
            "gpu_launches": kernels_per_step * args.steps,
            "gpu_launches_counted_from": "captured graph kernel nodes" if all(x is not None for x in per_step)
            else "static plan",
            "clocks": clocks,
            "device_status": ice.ice_status_string(status),
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.at_scale_only:
        import torch
        torch.cuda.set_device(rank_info()[1])
        print(json.dumps({"at_scale": at_scale(peaks(), args.at_scale_reps, args.at_scale_parts.split(","),
                                                args.at_scale_batch)}))
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
