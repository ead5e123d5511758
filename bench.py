#!/usr/bin/env python
"""Benchmark of MLA paged decode on one GB300.

One step = one full layer call of the library (plan -> W_uk absorb -> split-KV
decode -> combine + W_uv) on the DeepSeek-V3-shaped bf16 workload: batch 64,
one query token each, 128 heads, nope 128, rope 64, latent 512, v 128,
64-token pages over a 40k-page pool, cache lengths U[1024, 8192], causal.
Inputs are synthetic and seeded; they are resident in HBM before timing.

Prints one JSON line (rank 0).  The metric is microseconds per layer call
(lower is better); HBM GB/s and TFLOP/s of the same call, the roofline
fraction of the decode kernel and of the whole call, the oracle's CPU time on
a sample of the workload, and an end-to-end figure through host buffers ride
along.

--impl reference times the fp64 CPU oracle (test infrastructure, never tuned)
on the same workload, one whole layer call per step.

Only one GPU is used.  The decode kernel multicasts cache tiles between the two
CTAs of a cluster, and that code is kept to single-GPU processes: with
--gpus > 1 (or WORLD_SIZE > 1) the GPU arm prints a refusal line and exits
without touching a device.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA decode µs/layer, HBM GB/s and tensor TFLOP/s vs roofline (B=64,H=128,4k)"
UNIT = "us/layer"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
LAUNCHES_PER_CALL = 3       # absorb (+ plan), decode (+ split merge), W_uv
CPU_REPEATS = 3             # oracle runs of the whole call for the CPU baseline (median)
SINGLE_THREAD_LIMIT_S = 10  # a 1-thread oracle run longer than this is not repeated
KERNEL_SOURCES = {"decode_splitkv": "mla_decode_attention_06_gb300/csrc/mla_decode_tc.cu"}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["dsv3", "dsv3_mtp", "long", "long_swc", "fp8", "sparse",
                                           "sparse_mtp", "indexer", "prologue"],
                    default="dsv3",
                    help="dsv3 is the headline; indexer and prologue time those entry points on "
                         "the dsv3 batch shape")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--num-splits", type=int, default=0)
    walk = ap.add_mutually_exclusive_group()
    walk.add_argument("--fold-pairs", action="store_true",
                      help="walk consecutive query tokens of a request in pairs (one tile load for both)")
    walk.add_argument("--per-token", action="store_true",
                      help="walk every query token on its own")
    ap.add_argument("--profile-case", action="store_true",
                    help="a smaller case of the workload for ncu captures (dsv3: batch 32 over an "
                         "8192-page pool, 170 MB of attended cache, above the L2 size)")
    return ap.parse_args()


def make_workload(name, profile_case=False):
    from workloads import mla as W
    if profile_case:
        # smaller cases of the same shapes for ncu captures (inputs still above the L2 size)
        return {"dsv3": lambda: W.config_dsv3(B=32, num_pages=8192),
                "dsv3_mtp": lambda: W.config_dsv3_mtp(B=16),
                "fp8": lambda: W.config_fp8(B=32),
                "sparse": lambda: W.config_sparse(B=48)}[name]()
    return {"dsv3": W.config_dsv3, "dsv3_mtp": W.config_dsv3_mtp, "long": W.config_long,
            "long_swc": lambda: W.config_long(window=4096), "fp8": W.config_fp8,
            "sparse": W.config_sparse, "sparse_mtp": W.config_sparse_mtp}[name]()


def workload_desc(p):
    return (f"{p.name}: B={p.B}, T={p.T}, H={p.H}, nope={p.N}, rope={p.R}, latent={p.L}, "
            f"v={p.V}, page={p.ps}, pool pages={p.num_pages}, kv={p.kv_fmt}, w={p.w_fmt}, "
            f"mask={['null', 'causal', 'sliding_window_causal'][p.mask]}"
            + (f", window={p.window}" if p.window else ""))


def key_counts(p):
    """Attended keys per query token (the units of the decode's arithmetic)."""
    import numpy as np
    if p.sparse:
        cnt = np.minimum(p.topk_lengths if p.topk_lengths is not None
                         else np.full(p.B, p.indices.shape[1]), p.indices.shape[1])
        per_req = np.array([int((p.indices[b, :cnt[b]] >= 0).sum()) for b in range(p.B)])
        req = np.repeat(np.arange(p.B), np.diff(p.row_offsets.astype(np.int64)))
        return per_req[req]
    req, pos = p.query_positions()
    lens = p.cache_lens[req].astype(np.int64)
    if p.mask == 0:
        return lens
    hi = pos + 1
    lo = np.maximum(0, hi - p.window) if p.mask == 2 else np.zeros_like(hi)
    return hi - lo


def rows_read(p):
    """Cache rows the method must read: per request, the union of its tokens' key sets
    (a request's query tokens share its cached rows)."""
    import numpy as np
    if p.sparse:
        cnt = np.minimum(p.topk_lengths if p.topk_lengths is not None
                         else np.full(p.B, p.indices.shape[1]), p.indices.shape[1])
        return int(sum(int((p.indices[b, :cnt[b]] >= 0).sum()) for b in range(p.B))), 0
    req, pos = p.query_positions()
    hi = pos + 1 if p.mask != 0 else p.cache_lens[req].astype(np.int64)
    lo = np.maximum(0, pos + 1 - p.window) if p.mask == 2 else np.zeros_like(hi)
    rows, pages = 0, 0
    for b in range(p.B):
        sel = req == b
        if not sel.any():
            continue
        a, e = int(lo[sel].min()), int(hi[sel].max())
        if e > a:
            rows += e - a
            pages += (e - 1) // p.ps - a // p.ps + 1
    return rows, pages


def algorithmic(p):
    """Bytes and FLOPs the call must move / compute (workspace excluded)."""
    keys = int(key_counts(p).sum())
    rows, pages = rows_read(p)
    row = p.row_bytes + (4 if p.kv_fmt == "fp8" else 0)
    kv_bytes = rows * row
    idx_bytes = (rows * 4) if p.sparse else pages * 4
    wb = 1 if p.w_fmt == "fp8" else 2
    w_bytes = p.H * p.L * p.N * wb + p.H * p.V * p.L * wb
    if p.w_fmt == "fp8":
        w_bytes += (p.w_uk_scale.size + p.w_uv_scale.size) * 4
    q_bytes = p.T * p.H * (p.N + p.R) * 2
    out_bytes = p.T * p.H * p.V * 2
    flops_attn = 2 * p.H * keys * (p.L + p.R) + 2 * p.H * keys * p.L
    flops_proj = 2 * p.T * p.H * p.L * p.N + 2 * p.T * p.H * p.V * p.L
    return dict(keys=keys, kv_bytes=kv_bytes, decode_bytes=kv_bytes + idx_bytes,
                total_bytes=kv_bytes + idx_bytes + w_bytes + q_bytes + out_bytes,
                flops=flops_attn + flops_proj, flops_attn=flops_attn)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def kernel_traffic(name):
    """ncu DRAM bytes per launch recorded under profiles/, if the kernel source still matches."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    src = os.path.join(ROOT, KERNEL_SOURCES[name])
    if not os.path.exists(path) or not os.path.exists(src):
        return None
    with open(path) as fh:
        rec = json.load(fh).get(name)
    if not rec:
        return None
    with open(src, "rb") as fh:
        sha = hashlib.sha256(fh.read()).hexdigest()
    return rec.get("bytes_per_launch") if rec.get("source_sha256") == sha else None


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons, n = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            n += 1
            for name, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": n}


def world_size():
    return int(os.environ.get("WORLD_SIZE", "1"))


def rank():
    return int(os.environ.get("RANK", "0"))


def walk_arg(args):
    """The binding's fold_pairs argument: None leaves the query walk to the library."""
    if getattr(args, "fold_pairs", False):
        return True
    if getattr(args, "per_token", False):
        return False
    return None


def folds(p, args) -> bool:
    """Whether the library walks this call's query tokens in pairs (the rule of
    MLA_FLAG_FOLD_PAIRS / MLA_FLAG_PER_TOKEN in include/mla_decode.h)."""
    if p.T < 2 * p.B or p.kv_fmt != "bf16" or p.L != 512 or p.R != 64:
        return False
    w = walk_arg(args)
    return p.sparse if w is None else w


def config_of(p, args):
    """The workload description both arms print (identical keys and values)."""
    return {"workload": workload_desc(p), "global_batch": p.B, "query_tokens": p.T,
            "parallelism": "single GPU",
            "l2": "GPU arm: a 2 x L2-size buffer is written before every timed step",
            "num_splits": args.num_splits or "auto",
            "query_walk": "folded pairs" if folds(p, args) else "one token at a time"}


def oracle_call_seconds(p):
    """Wall time of one whole layer call of the oracle (all query tokens, all heads)."""
    import oracle
    oracle.build()
    t0 = time.perf_counter()
    oracle.decode(p)
    return time.perf_counter() - t0


def single_thread_run(workload, repeats):
    """The oracle on one core (a child process with OMP_NUM_THREADS=1): wall seconds of
    `repeats` whole layer calls, each timed separately.  Stops repeating once one run
    takes longer than SINGLE_THREAD_LIMIT_S."""
    code = ("import json, sys, time; sys.path.insert(0, %r); import bench, oracle; "
            "from workloads import mla as W; "
            "p = W.config_tiny() if %r == 'tiny' else bench.make_workload(%r); "
            "ts = []\n"
            "for i in range(%d):\n"
            "    ts.append(bench.oracle_call_seconds(p))\n"
            "    if ts[-1] > %d: break\n"
            "print(json.dumps({'seconds': ts, 'threads': oracle.num_threads()}))"
            % (ROOT, workload, workload, repeats, SINGLE_THREAD_LIMIT_S))
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env)
    if r.returncode != 0:
        return {"error": (r.stderr or r.stdout)[-300:]}
    d = json.loads(r.stdout.strip().splitlines()[-1])
    return {"us_per_call": statistics.median(d["seconds"]) * 1e6, "runs": len(d["seconds"]),
            "threads": d["threads"]}


def cpu_baseline(p):
    """The oracle as it stands on the host cores: whole layer calls, median of CPU_REPEATS
    on all cores, plus 1-thread runs of the tiny workload and of this one."""
    import oracle
    oracle.build()
    secs = [oracle_call_seconds(p) for _ in range(CPU_REPEATS)]
    us = statistics.median(secs) * 1e6
    return {"value": us, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"the whole layer call ({p.T} query tokens x {p.H} heads), "
                      f"median of {CPU_REPEATS} runs: " + ", ".join(f"{s:.2f} s" for s in secs),
            "single_thread": {"tiny": single_thread_run("tiny", CPU_REPEATS),
                              p.name: single_thread_run(WORKLOAD_OF.get(p.name, "dsv3"), CPU_REPEATS)},
            "cpu_model": cpu_model()}


WORKLOAD_OF = {"dsv3_bf16": "dsv3", "dsv3_mtp": "dsv3_mtp", "long": "long", "long_swc": "long_swc",
               "fp8": "fp8", "sparse": "sparse", "sparse_mtp": "sparse_mtp"}


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


def run_reference(args, p):
    """The oracle timed as the reference arm: one whole layer call per step."""
    if rank() != 0:
        return
    import oracle
    oracle.build()
    secs = []
    w0 = time.perf_counter()
    for i in range(args.warmup + args.steps):
        s = oracle_call_seconds(p)
        if i >= args.warmup:
            secs.append(s)
    wall = time.perf_counter() - w0
    ms = statistics.mean(secs) * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": ms * 1e3, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "config": config_of(p, args),
        "cpu_baseline": {"value": ms * 1e3, "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": f"each step is the whole layer call ({p.T} query tokens x "
                                   f"{p.H} heads); no scaling"},
        "e2e": {"value": ms * 1e3, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s_all_steps": wall,
    }
    print(json.dumps(line), flush=True)


def indexer_workload():
    """The FP8 indexer on the dsv3 decode batch: 64 requests, lengths U[1024, 8192], 64 index
    heads of depth 128 (DeepSeek-style lightning indexer), top 2048, causal."""
    from workloads import mla as W
    from workloads.indexer import make_indexer
    lens = W.Stream(1001, "dsv3-lens").integers(1024, 8192, 64)
    return make_indexer("indexer_dsv3", 1005, H=64, D=128, ps=64, cache_lens=lens, num_pages=6000,
                        top_k=2048)


def prologue_workload():
    """The fused branch prologue on the dsv3 batch (the bf16 cache of config dsv3)."""
    return make_workload("dsv3")


# INT32 lane operations a second on this part (152 SMs x 128 lanes x max SM clock) and the
# lane operations one exact e4m3 multiply-accumulate takes in the indexer's inner loop, as
# written in the source (four byte loads, the significand product, the exponent sum, the
# power of two and a 64-bit multiply-add)
INT_LANE_OPS_PER_S = 152 * 128 * 2.07e9
INDEXER_OPS_PER_MAC = 8


def time_events(fn, flush, steps, warmup, stream):
    """Mean device time of fn() over `steps` calls, L2 flushed before each.  A short
    device-side spin after the flush keeps the GPU busy while the host marshals the
    call, so the start event is not followed by idle time waiting for the launch."""
    import torch
    spin = getattr(torch.cuda, "_sleep", None)
    for _ in range(max(3, warmup)):
        flush.zero_()
        fn()
    ev = []
    for _ in range(steps):
        flush.zero_()
        if spin is not None:
            spin(200000)   # ~100 us of device time at 2 GHz
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        ev.append((a, b))
    torch.cuda.synchronize()
    return statistics.mean(x.elapsed_time(y) for x, y in ev)


def run_aux(args):
    """Time the indexer or the prologue entry point; prints one JSON line."""
    import numpy as np
    import torch
    import oracle
    from mla_decode_attention_06_gb300 import build as libbuild
    libbuild.build()
    import mla_decode_attention_06_gb300 as M
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(device=dev, dtype=dt)
    peaks, peak_kind = load_peaks()
    clocks = ClockSampler(0)
    if args.workload == "indexer":
        p = indexer_workload()
        d = dict(q=t(p.q, torch.uint8), q_s=t(p.q_s, torch.float32),
                 off=t(p.row_offsets.astype(np.int32), torch.int32), k=t(p.k, torch.uint8),
                 ks=t(p.k_scales, torch.float32), bt=t(p.block_table, torch.int32),
                 lens=t(p.cache_lens.astype(np.int32), torch.int32))
        out = torch.empty((p.T, p.top_k), dtype=torch.int32, device=dev)

        def fn():
            M.mla_indexer_fp8(d["q"], d["q_s"], d["off"], d["k"], d["ks"], d["bt"], d["lens"],
                              page_size=p.ps, top_k=p.top_k, mask=p.mask, out=out)
        ms = time_events(fn, flush, args.steps, args.warmup, stream)
        keys = int(sum(int(n) for n in p.cache_lens))       # causal, one query per request
        macs = keys * p.H * p.D
        nbytes = keys * (p.D + 4) + p.T * p.H * (p.D + 4) + p.T * p.top_k * 4 + keys // p.ps * 4
        achieved = macs * INDEXER_OPS_PER_MAC / (ms * 1e-3)
        t0 = time.perf_counter()
        oracle.indexer(p)
        cpu_s = time.perf_counter() - t0
        line = {"metric": "FP8 indexer us/call (exact e4m3 scores, top 2048)", "value": ms * 1e3,
                "unit": "us/call", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": ms, "higher_is_better": False, "dtype": "e4m3 -> exact int64 / f64",
                "data": "synthetic (seeded)",
                "config": {"workload": f"indexer: B={p.B}, H={p.H}, D={p.D}, keys={keys}, top_k={p.top_k}, "
                                       "lengths U[1024, 8192], causal", "l2": "flushed before every step"},
                "roofline": {"bound": "alu", "achieved": achieved, "peak": INT_LANE_OPS_PER_S,
                             "unit": "int32 lane-op/s", "frac": achieved / INT_LANE_OPS_PER_S,
                             "traffic": None, "note": f"{INDEXER_OPS_PER_MAC} lane ops per exact multiply-add; "
                                                      f"HBM time of {nbytes / 1e6:.1f} MB is "
                                                      f"{nbytes / (float(peaks['hbm_gbs']) * 1e9) * 1e6:.1f} us"},
                "macs_per_call": macs, "gpu_launches": 2 * args.steps,
                "cpu_baseline": {"value": cpu_s * 1e6, "unit": "us/call", "cores": oracle.num_threads(),
                                 "kind": "oracle", "sample": "the whole call, one run"}}
    else:
        p = prologue_workload()
        from workloads.run import device_inputs
        dd = device_inputs(p, dev)
        from workloads import mla as W
        max_seq = int(p.cache_lens.max()) + 1
        freqs = t(W.rope_freqs_cis(max_seq, p.R).view(np.int16), torch.int16).view(torch.bfloat16)
        gamma = t(W.to_bf16_bits(np.ones(p.L)).view(np.int16), torch.int16).view(torch.bfloat16)
        q = dd["q"].clone()
        pool = dd["pool"]

        def fn():
            M.mla_branch_prologue(q, dd["offsets"], pool, dd["block_table"], dd["cache_lens"], freqs, gamma,
                                  page_size=p.ps, kv_lora_rank=p.L, epsilon=1e-6)
        ms = time_events(fn, flush, args.steps, args.warmup, stream)
        nbytes = 2 * (p.T * p.H * p.R * 2) + 2 * p.T * (p.L + p.R) * 2 + p.T * p.R * 2 + p.L * 2
        achieved = nbytes / (ms * 1e-3) / 1e9
        line = {"metric": "fused branch prologue us/call (RoPE + RMSNorm, in place)", "value": ms * 1e3,
                "unit": "us/call", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": ms, "higher_is_better": False, "dtype": "bf16 -> f64 -> bf16",
                "data": "synthetic (seeded)",
                "config": {"workload": workload_desc(p), "l2": "flushed before every step"},
                "roofline": {"bound": "hbm", "achieved": achieved, "peak": float(peaks["hbm_gbs"]),
                             "unit": "GB/s", "frac": achieved / float(peaks["hbm_gbs"]), "traffic": None,
                             "note": "launch-bound: the call moves "
                                     f"{nbytes / 1e6:.2f} MB"},
                "gpu_launches": args.steps}
    line["clocks"] = clocks.stop()
    print(json.dumps(line), flush=True)


def refuse_multi_gpu(args):
    """The GPU arm runs on one GPU only; under torchrun rank 0 says so and every rank exits."""
    n = max(args.gpus, world_size())
    if rank() == 0:
        print(json.dumps({"impl": "ours", "metric": METRIC, "unit": UNIT, "n_gpus": n,
                          "unavailable": "single GPU only: the decode kernel multicasts cache tiles "
                                         "within a CTA pair, and that code runs in 1-GPU processes "
                                         "only; the path needs no exchange between GPUs"}),
              flush=True)


def main():
    args = parse_args()
    p_name = args.workload
    if args.impl == "ours" and (args.gpus > 1 or world_size() > 1):
        refuse_multi_gpu(args)
        return
    if args.impl == "reference" and rank() != 0:
        return
    if args.workload in ("indexer", "prologue"):
        if args.impl == "ours":
            run_aux(args)
        else:
            print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the decode "
                                                                  "workloads only"}), flush=True)
        return
    import numpy as np  # noqa: F401
    import torch

    p = make_workload(p_name, args.profile_case)
    if args.impl == "reference":
        run_reference(args, p)
        return

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)

    from mla_decode_attention_06_gb300 import build as libbuild
    libbuild.build()
    import mla_decode_attention_06_gb300 as M
    from workloads.run import device_inputs, run_gpu, workspace_bytes

    d = device_inputs(p, dev)
    ws = torch.empty(max(256, workspace_bytes(p, args.num_splits)), dtype=torch.uint8, device=dev)
    out = torch.empty((p.T, p.H, p.V), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((p.T, p.H), dtype=torch.float32, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(timing=False, on_stream=None):
        run_gpu(p, d, num_splits=args.num_splits, out=out, lse_out=lse, workspace=ws,
                stream=on_stream or stream, timing=timing, fold_pairs=walk_arg(args))

    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    M.kernel_times()   # clear

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize()
    clocks = ClockSampler(0)
    time.sleep(0.25)
    w0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - w0
    clk = clocks.stop()
    per_step = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = statistics.mean(per_step)
    # per-kernel durations from separate steps: the library's event pairs between
    # its kernels would otherwise hold back the programmatic-launch overlap of the
    # timed calls above
    M.kernel_times()   # clear
    for _ in range(max(10, min(args.steps, 50))):
        flush.zero_()
        step(timing=True)
    torch.cuda.synchronize()
    kt, ncalls = M.kernel_times()

    alg = algorithmic(p)
    peaks, peak_kind = load_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    bf16_peak = float(peaks["bf16_tflops"])
    us = ms * 1e3
    call_gbs = alg["total_bytes"] / (ms * 1e-3) / 1e9
    call_tflops = alg["flops"] / (ms * 1e-3) / 1e12
    roof_us = max(alg["total_bytes"] / (hbm_peak * 1e9), alg["flops"] / (bf16_peak * 1e12)) * 1e6
    dec_ms = kt.get("decode_splitkv")
    dec_gbs = alg["decode_bytes"] / (dec_ms * 1e-3) / 1e9 if dec_ms else None
    dec_tflops = alg["flops_attn"] / (dec_ms * 1e-3) / 1e12 if dec_ms else None
    traffic = kernel_traffic("decode_splitkv")

    line = {
        "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if p.kv_fmt == "bf16" else "e4m3->bf16", "data": "synthetic (seeded)",
        "config": config_of(p, args),
        "hbm_gbs": call_gbs, "tflops": call_tflops,
        "roofline_call": {"bound": "hbm" if alg["total_bytes"] / hbm_peak >= alg["flops"] / (bf16_peak * 1e3) else "tensor",
                          "roofline_us": roof_us, "frac": roof_us / us},
        "roofline": {"kernel": "decode_splitkv", "bound": "hbm", "achieved": dec_gbs,
                     "peak": hbm_peak, "unit": "GB/s",
                     "frac": (dec_gbs / hbm_peak) if dec_gbs else None, "traffic": traffic,
                     "peak_source": f"hbm_gbs of {peak_kind}",
                     "algorithmic_bytes_per_launch": alg["decode_bytes"],
                     "tensor_tflops": dec_tflops,
                     "tensor_frac": (dec_tflops / bf16_peak) if dec_tflops else None},
        "kernel_ms": {k: v for k, v in kt.items()}, "kernel_calls_timed": ncalls,
        "kernel_ms_note": "separate steps with event pairs between the kernels (no launch overlap)",
        "gpu_launches": LAUNCHES_PER_CALL * args.steps,
        "clocks": clk,
        "wall_s_timed_region": wall,
    }

    line["graph"] = graph_replay(step, flush, stream, args.steps)
    if not args.no_e2e:
        line["e2e"] = e2e(p, d, args, dev, out, lse, ws, flush, stream)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(p)
    print(json.dumps(line), flush=True)


def graph_replay(step, flush, stream, steps):
    """The same call captured once in a CUDA graph and replayed (L2 flushed between replays)."""
    import torch
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step(on_stream=torch.cuda.current_stream())
        times = []
        for i in range(steps + 3):
            flush.zero_()
            s = torch.cuda.Event(enable_timing=True)
            e = torch.cuda.Event(enable_timing=True)
            s.record(stream)
            g.replay()
            e.record(stream)
            if i >= 3:
                times.append((s, e))
        torch.cuda.synchronize()
        us = statistics.mean(s.elapsed_time(e) for s, e in times) * 1e3
        return {"us_per_call": us, "replays": len(times)}
    except Exception as ex:   # capture is best effort; the eager number above is the metric
        return {"error": str(ex)[:200]}


def e2e(p, d, args, dev, out, lse, ws, flush, stream):
    """The same call through host buffers, as a serving loop runs it: every step copies its
    inputs (q, offsets, block table, cache lengths or indices) from pinned host memory and
    its output back to pinned host memory, and the copies of one step overlap the kernels
    of its neighbours (inputs and outputs double-buffered; one stream for input copies, one
    for the calls, one for output copies).  The value is the whole pipelined run's time,
    from the first input copy to the last output copy, divided by the steps.  This needs a
    step that reads more than twice the L2 (the dsv3 step reads 340 MB), so that no flush
    is due between calls; a smaller step is flushed and timed with its copies one after
    the other instead (the flush outside the timed region)."""
    import torch
    from workloads.run import run_gpu
    keys = [k for k in ("q", "offsets", "block_table", "cache_lens", "indices", "topk") if d.get(k) is not None]
    host = {k: d[k].cpu().pin_memory() for k in keys}
    bufs = [dict(d), dict(d)]
    for k in keys:
        bufs[1][k] = torch.empty_like(d[k])
    outs = [out, torch.empty_like(out)]
    out_h = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out.numel() * out.element_size()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_each = algorithmic(p)["total_bytes"] <= 2 * l2
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def run(n):
        done = [None] * n      # call i finished (its inputs and output buffer are free after)
        copied = [None] * n    # output i copied out
        first = torch.cuda.Event(enable_timing=True)
        last = torch.cuda.Event(enable_timing=True)
        for i in range(n):
            b = i & 1
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(done[i - 2])
                if i == 0:
                    first.record(s_in)
                for k in keys:
                    bufs[b][k].copy_(host[k], non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(s_in)
            with torch.cuda.stream(stream):
                stream.wait_event(ready)
                if i >= 2:
                    stream.wait_event(copied[i - 2])
                if flush_each:
                    flush.zero_()
                run_gpu(p, bufs[b], num_splits=args.num_splits, out=outs[b], lse_out=None, workspace=ws,
                        stream=stream, want_lse=False, fold_pairs=walk_arg(args))
                done[i] = torch.cuda.Event()
                done[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done[i])
                out_h[b].copy_(outs[b], non_blocking=True)
                copied[i] = torch.cuda.Event()
                copied[i].record(s_out)
        last.record(s_out)
        torch.cuda.synchronize()
        return first.elapsed_time(last) / n

    def run_serial(n):
        # a step that fits in L2: flush, then time its copies and call one after the other
        times = []
        for i in range(n):
            flush.zero_()
            s0 = torch.cuda.Event(enable_timing=True)
            s1 = torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            for k in keys:
                bufs[0][k].copy_(host[k], non_blocking=True)
            run_gpu(p, bufs[0], num_splits=args.num_splits, out=outs[0], lse_out=None, workspace=ws,
                    stream=stream, want_lse=False, fold_pairs=walk_arg(args))
            out_h[0].copy_(outs[0], non_blocking=True)
            s1.record(stream)
            times.append((s0, s1))
        torch.cuda.synchronize()
        return statistics.mean(x.elapsed_time(y) for x, y in times)

    n = max(10, min(args.steps, 50))
    if flush_each:
        run_serial(3)
        ms = run_serial(n)
        how = {"pipelined": False, "l2": "flushed before every call (a step fits in 2 x L2): copies "
                                         "and call timed one after the other"}
    else:
        run(3)   # warm-up
        ms = run(n)
        how = {"pipelined": True, "l2": "not flushed: a step reads more than 2 x L2"}
    return {"value": ms * 1e3, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": n, **how}


if __name__ == "__main__":
    main()
