#!/usr/bin/env python
"""Benchmark of the CSA2 decode step (index + sparse attention) on GB300.

One step = one pass of the whole hot path over a batch of decode queries:
append the current token (RoPE + FP4 main latent, FP4 indexer key), then for
each of the group's layers the FP8 window append, the Full / Reindex index
(or Reuse), and sparse attention.  The default workload is the 20-layer
decoder group at 131,072 entries with batch 16 ([Full + 3 Reuse] +
4 x [Reindex + 3 Reuse]).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload 128k|1m|tiny|manyq|ragged|encoder|append]

Prints one JSON line (rank 0).  Under torchrun every rank runs its own batch
(independent requests, no collective on the data path); value = all queries
over the slowest rank's time.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "CSA2 decode queries/s per layer group at 128K/1M ctx; % of HBM roofline"
UNIT = "queries/s"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def workload(name):
    from csa2_sparse_attention_gb300 import workloads as W
    return {"128k": W.group_128k, "1m": W.group_1m, "tiny": W.tiny, "manyq": W.many_query,
            "ragged": W.ragged, "encoder": W.encoder_m2}[name]()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return PEAKS_FALLBACK, "fallback"


def config_of(wl, extra=None):
    c = {"workload": wl.name, "queries_per_gpu": wl.batch,
         "context": wl.contexts[0] if len(set(wl.contexts)) == 1 else f"ragged {min(wl.contexts)}..{max(wl.contexts)}",
         "layers": "".join(wl.layers), "pool_blocks": wl.pool_blocks, "topk": wl.topk,
         "window": wl.window, "index_heads": 32, "index_dim": 128, "attn_heads": 64, "latent_dim": 512}
    c.update(extra or {})
    return c


# --------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples during the timed region (every 200 ms)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------- algorithmic bytes
# From this many queries the full scan runs as the many-query contraction
# (groups of 4 queries share each K tile); it is then tensor-bound.
MQ_MIN_QUERIES = 256
# nominal dense FP4 : bf16 tensor throughput (13.5 : 2.25 PFLOP/s)
FP4_PER_BF16 = 6.0
# Smaller batches whose candidate pool has at most this many blocks keep the
# scan's per-position scores for the Full layer's top-K.
POS_SCORE_MAX_CAND = 2048


def alg_flops_per_launch(kernel, g):
    """Algorithmic FLOPs of one scan launch: every visible position scored
    against 32 indexer heads of dim 128 (a multiply and an add each)."""
    import numpy as np
    assert kernel == "scan_blockmax"
    n = np.asarray(g.contexts, dtype=np.int64)
    return float(2 * np.sum(n) * 32 * 128)


def alg_bytes_per_launch(kernel, g):
    """Algorithmic bytes one launch of `kernel` moves for this group's step
    (average over the step's launches of that kernel)."""
    import numpy as np
    from csa2_sparse_attention_gb300 import workloads as W
    n = np.asarray(g.contexts, dtype=np.int64)
    B, P, K, Wn = g.B, g.P, g.K, g.Wn
    nb = (n + 7) // 8
    decode_scan = B < MQ_MIN_QUERIES and max(P, K) <= POS_SCORE_MAX_CAND
    if kernel == "scan_blockmax":   # indexer K stream + block maxima (+ per-position scores) + indexer Q
        return float(np.sum(n * 72 + nb * 4 + (n * 4 if decode_scan else 0)) + B * 32 * 72)
    out_bytes = 4 if getattr(g, "out_code", 1) == 1 else 2
    if kernel == "attn_split":      # selected FP4 latents + FP8 window + bf16 Q + output O (as written) + lse
        return float(np.sum(288 * np.minimum(K, n) + 512 * np.minimum(Wn, n)) + B * 64 * 512 * 2
                     + B * (64 * 512 * out_bytes + 64 * 4))
    if kernel == "attn_merge":      # output + lse
        return float(B * (64 * 512 * out_bytes + 64 * 4))
    if kernel == "pool_score":      # gathered pool blocks (8 rows x 72 B)
        # a decode batch's Full layer reads its candidates' scores from the scan instead
        n_full = 0 if decode_scan else sum(1 for m in g.layers if m == W.FULL)
        n_re = sum(1 for m in g.layers if m == W.REINDEX)
        c_full, c_re = max(P, K), P
        per = [float(np.sum(np.minimum(8 * c_full, nb * 8) * 72))] * n_full + \
              [float(np.sum(np.minimum(8 * c_re, nb * 8) * 72))] * n_re
        return sum(per) / max(1, len(per))
    if kernel == "select_blocks":
        return float(np.sum(nb * 4))
    if kernel == "select_topk":
        return float(B * 8 * P * 4)
    return None


# What limits each kernel at decode batch sizes, from its ncu capture: the
# roofline it is measured against stays HBM (or the FP4 tensor pipe), but a
# kernel whose DRAM and tensor activity are both low is latency-bound.
KERNEL_BOUND = {"scan_blockmax": "hbm", "pool_score": "hbm", "attn_split": "latency", "attn_merge": "hbm",
                "select_blocks": "latency", "select_topk": "latency", "quantize_fp4": "hbm",
                "quantize_fp8": "hbm"}


def traffic_from_profiles(kernel, wl_name):
    """dram bytes per launch from a committed ncu summary, if its recorded
    source hash still matches the kernel source; else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{wl_name}.txt")
    if not os.path.exists(path):
        return None
    meta = {}
    with open(path) as f:
        for line in f:
            if ":" in line:
                k, v = line.split(":", 1)
                meta[k.strip()] = v.strip()
    src = meta.get("source_file")
    sha = meta.get("source_sha256")
    if not src or not sha:
        return None
    with open(os.path.join(ROOT, src), "rb") as f:
        if hashlib.sha256(f.read()).hexdigest() != sha:
            return None
    try:
        return float(meta["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# --------------------------------------------------------------- CPU baseline
class OracleSample:
    """The oracle (as it stands) on a few queries of a workload: the setup
    (quantizing each query's caches) is untimed; step() runs the per-step
    work of one query (current-token append, Full/Reindex index, every
    attention layer), cycling through the prepared queries."""

    def __init__(self, wl_name, queries):
        from oracle import csa2_oracle as O
        from tests.helpers import oracle_query
        self.O = O
        self.wl = wl = workload(wl_name)
        self.preps = []
        for q in range(queries):
            inp = oracle_query(wl, q)
            kc, ks = O.quantize_fp4(inp["k_real"])
            lc, ls = O.quantize_fp4(O.rope(inp["latent_real"], inp["positions"]))
            rings = {li: O.append_swa_fp8(inp["swa_real"][li]) for li in range(len(wl.layers))}
            self.preps.append((inp, O.dequantize_fp4(kc, ks), lc, ls, rings))
        self.i = 0

    def step(self):
        O, wl = self.O, self.wl
        inp, kdq, lc, ls, rings = self.preps[self.i % len(self.preps)]
        self.i += 1
        n = inp["n"]
        O.append_main_latent(inp["latent_real"][n - 1:n], inp["positions"][n - 1:n])
        O.append_plain_fp4(inp["k_real"][n - 1:n])
        O.decode_group_step(wl.layers, inp["index_q"], inp["index_w"], kdq, lc, ls, rings,
                            inp["attn_q"], n, wl.pool_blocks, wl.topk, wl.window)


def oracle_step_sample(wl_name, queries, min_seconds):
    """(query-steps, seconds) of the oracle over at least min_seconds."""
    smp = OracleSample(wl_name, queries)
    done, t0 = 0, time.perf_counter()
    while True:
        smp.step()
        done += 1
        el = time.perf_counter() - t0
        if el >= min_seconds:
            return done, el


def _oracle_child(wl_name, queries, min_seconds, threads):
    env = dict(os.environ, OPENBLAS_NUM_THREADS=str(threads), OMP_NUM_THREADS=str(threads),
               MKL_NUM_THREADS=str(threads), CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-baseline-child", "--workload", wl_name,
           "--child-queries", str(queries), "--child-seconds", str(min_seconds)]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=900)
    if r.returncode != 0:
        return None, (r.stderr or r.stdout).strip().splitlines()[-1:] or ["failed"]
    return json.loads(r.stdout.strip().splitlines()[-1]), None


def cpu_baseline(wl_name, queries=1, min_seconds=8.0):
    """The oracle in a child process, timed twice: with every host core
    available to its BLAS (OPENBLAS/OMP/MKL threads = cores; the reported
    value) and single-threaded."""
    cores = os.cpu_count() or 1
    res, err = _oracle_child(wl_name, queries, min_seconds, cores)
    if err:
        return {"error": err}
    one, err1 = _oracle_child(wl_name, queries, min_seconds, 1)
    out = {"value": res["done"] / res["seconds"], "unit": UNIT, "cores": cores, "kind": "oracle",
           "sample": f"{res['done']} query-steps of {wl_name} ({queries} distinct queries, caches "
                     f"pre-quantized untimed), {res['seconds']:.1f} s, fp64 numpy, BLAS threads = {cores}"}
    out["single_thread"] = ({"value": one["done"] / one["seconds"], "unit": UNIT, "cores": 1,
                             "sample": f"{one['done']} query-steps, {one['seconds']:.1f} s, BLAS threads = 1"}
                            if one else {"error": err1})
    return out


# ---------------------------------------------------------------- reference
def run_reference(args):
    """The oracle timed on this host's cores on the same workload, config,
    metric and unit as the GPU arm; each step is one query through the whole
    layer group (a bounded sample of the GPU arm's 16-query step).  Warm-up
    and timed steps are the ones requested unless the timed steps would
    exceed about four minutes, in which case fewer are timed and the line
    says so."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    wl = workload(args.workload)
    smp = OracleSample(args.workload, 1)
    t0 = time.perf_counter()
    smp.step()
    est = time.perf_counter() - t0
    for _ in range(max(0, args.warmup - 1)):
        smp.step()
    timed = max(1, min(args.steps, int(240.0 / max(est, 1e-3))))
    t0 = time.perf_counter()
    for _ in range(timed):
        smp.step()
    el = time.perf_counter() - t0
    value = timed / el
    cores = os.cpu_count() or 1
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": timed, "warmup": args.warmup, "ms_per_step": 1000.0 * el / timed, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(wl, {"parallelism": f"replicas x{world}", "l2": L2_NOTE}),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{timed} single-query steps of {wl.name} (requested {args.steps}); "
                                       f"caches pre-quantized untimed; fp64 numpy, BLAS threads = {cores}"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------- ours
def run_append(args):
    """Bulk KV append: 1,048,576 tokens through the RoPE + FP4 main-latent
    append (rows layout) and the FP4 indexer-key append (BLOCK8), inputs
    resident in HBM (1.3 GB, larger than L2), one JSON line in tokens/s."""
    import torch
    from csa2_sparse_attention_gb300 import abi
    from csa2_sparse_attention_gb300 import workloads as W
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    wl = W.group_1m()
    n = 1 << 20
    lat = torch.from_numpy(W.main_latent_rows(wl, 0, 0, n)).to(torch.bfloat16).to(dev)
    ik = torch.from_numpy(W.indexer_k_rows(wl, 0, 0, n)).to(torch.bfloat16).to(dev)
    pos = torch.from_numpy(W.latent_positions(wl, 0)[:n]).to(dev)
    codes = torch.empty((n, 256), dtype=torch.uint8, device=dev)
    scales = torch.empty((n, 32), dtype=torch.uint8, device=dev)
    ik_codes = torch.empty(n // 8 * 576, dtype=torch.uint8, device=dev)  # 576-byte records (codes + scales)
    ik_scales = None
    table = torch.empty(abi.csa2_rope_table_bytes(512, n), dtype=torch.uint8, device=dev)
    ws = torch.zeros(4096, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(dev)
    abi.csa2_rope_table_init(10000.0, 512, n, table, stream)

    def step():
        abi.csa2_quantize_append(lat, n, 512, abi.FMT_FP4, abi.LAYOUT_ROWS, pos, table, n, None, n,
                                 codes, scales, ws, ws.numel(), stream)
        abi.csa2_quantize_append(ik, n, 128, abi.FMT_FP4, abi.LAYOUT_BLOCK8R, None, None, 0, None, n,
                                 ik_codes, ik_scales, ws, ws.numel(), stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    stream.synchronize()
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    torch.cuda.synchronize(dev)
    c0 = abi.csa2_launch_count()
    with ClockSampler(0) as clk:
        with torch.cuda.stream(stream):
            for k in range(K):
                ev[k][0].record(stream)
                step()
                ev[k][1].record(stream)
        torch.cuda.synchronize(dev)
    launches = abi.csa2_launch_count() - c0
    # each append alone (CUDA events around 10 back-to-back calls)
    def alone(call):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(10):
                call()
            e1.record(stream)
        stream.synchronize()
        return 1000 * e0.elapsed_time(e1) / 10
    main_us = alone(lambda: abi.csa2_quantize_append(lat, n, 512, abi.FMT_FP4, abi.LAYOUT_ROWS, pos, table, n, None, n,
                                                     codes, scales, ws, ws.numel(), stream))
    ik_us = alone(lambda: abi.csa2_quantize_append(ik, n, 128, abi.FMT_FP4, abi.LAYOUT_BLOCK8R, None, None, 0, None, n,
                                                   ik_codes, ik_scales, ws, ws.numel(), stream))
    st = abi.csa2_status_fetch(ws)
    if st[0] != 0:
        raise RuntimeError(f"append status {st}")
    ms = sum(a.elapsed_time(b) for a, b in ev)
    tok_s = n * K / (ms / 1000.0)
    pk, pk_kind = peaks()
    bpt = (1024 + 256 + 32 + 8) + (256 + 64 + 8)  # main in/out + position, indexer in/out
    achieved = bpt * tok_s / 1e9
    print(json.dumps({"metric": "KV-append tokens/s (RoPE + FP4 main latent, FP4 indexer key)", "value": tok_s,
                      "unit": "tokens/s", "n_gpus": 1, "steps": K, "warmup": args.warmup,
                      "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                      "dtype": "bf16 in, fp32 RoPE (fp64 near ties), E2M1 + E4M3 out", "data": "synthetic",
                      "config": {"workload": "bulk-append-1m", "tokens": n,
                                 "l2": "inputs (1.3 GB) larger than L2, no flush"},
                      "gpu_launches": launches,
                      "kernels": {"main_latent_us": main_us, "indexer_key_us": ik_us,
                                  "main_latent_frac": (1024 + 256 + 32 + 8) * n / (main_us * 1e-6) / 1e9 / pk["hbm_gbs"],
                                  "indexer_key_frac": (256 + 64 + 8) * n / (ik_us * 1e-6) / 1e9 / pk["hbm_gbs"]},
                      "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                                   "frac": achieved / pk["hbm_gbs"], "traffic": None, "peak_source": pk_kind,
                                   "alg_bytes_per_token": bpt},
                      "clocks": clk.summary()}), flush=True)


L2_NOTE = "GPU arm: L2 flushed between timed steps (256 MB write, then 256 MB read, untimed)"


class L2Flush:
    """Evicts the 129 MB L2 between timed steps, untimed: writes one 256 MB
    buffer, then reads another, so that the next step finds L2 full of
    clean, unrelated lines (a write alone would leave dirty lines whose
    write-back lands inside the next step's first kernel)."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(256 << 20, dtype=torch.uint8, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.max()


def max_over_ranks(x, device):
    """The largest x over all ranks of the process group (x itself when the
    job runs alone): the job's time is its slowest rank's."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(batch, world, steps, total_ms):
    """Whole-job queries/s: every rank runs `steps` steps of its own batch
    (replicas), timed by the slowest rank's total."""
    return batch * world * steps / (total_ms / 1000.0)


def measure_group(g, wl, stream, flush, dev, K, warmup, world, local):
    """Time K CUDA-graph replays of the group's step (L2 flushed between
    steps, untimed), then each kernel's device time in eager steps.  Returns
    the step times, the slowest rank's total, the clocks seen, the launches
    per step, the per-kernel table, the dominant kernel's roofline and the
    full scan's."""
    import torch
    import torch.distributed as dist
    from csa2_sparse_attention_gb300 import abi
    with torch.cuda.stream(stream):
        g.step(stream)                      # eager warm-up (sets kernel attributes)
        stream.synchronize()
        c0 = abi.csa2_launch_count()
        g.step(stream)
        stream.synchronize()
        launches_per_step = abi.csa2_launch_count() - c0
    g.capture(stream)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            flush()
            g.replay()
    stream.synchronize()

    # ---- timed region: graph replays, L2 flushed between steps (untimed)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        t_wall = time.perf_counter()
        torch.cuda.nvtx.range_push("csa2_timed")  # lets an ncu launch list select the timed steps
        with torch.cuda.stream(stream):
            for k in range(K):
                flush()
                ev[k][0].record(stream)
                g.replay()
                ev[k][1].record(stream)
        torch.cuda.synchronize(dev)
        torch.cuda.nvtx.range_pop()
        t_wall = time.perf_counter() - t_wall
    if world > 1:
        dist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(float(sum(step_ms)), dev)

    # ---- per-kernel device time (eager steps, L2 flushed, events on the launch stream)
    n_prof = max(3, min(20, K))
    kern = {}
    for kid, name in enumerate(abi.KERNELS):
        abi.csa2_timer_enable(kid, 64 * n_prof)
    with torch.cuda.stream(stream):
        for _ in range(n_prof):
            flush()
            # the GPU sleeps while the host enqueues the step, so the kernels
            # run back to back and each event pair brackets device time only
            torch.cuda._sleep(4_000_000)
            g.step(stream)
    stream.synchronize()
    for kid, name in enumerate(abi.KERNELS):
        ms, cnt = abi.csa2_timer_read(kid)
        if cnt:
            kern[name] = {"ms_per_step": ms / n_prof, "launches_per_step": cnt / n_prof, "avg_us": 1000 * ms / cnt}
    tot = sum(v["ms_per_step"] for v in kern.values())
    for v in kern.values():
        v["share"] = v["ms_per_step"] / tot if tot else None
    dom = max(kern, key=lambda k: kern[k]["ms_per_step"])
    pk, pk_kind = peaks()
    scan = kern.get("scan_blockmax")
    # the many-query scan is a dense FP4 contraction (tensor-bound); the
    # decode scan streams the indexer keys (HBM-bound)
    scan_roof = None
    if scan and g.B >= MQ_MIN_QUERIES:
        fpl = alg_flops_per_launch("scan_blockmax", g)
        achieved = fpl / (scan["avg_us"] * 1e-6) / 1e12
        fp4_peak = pk["bf16_tflops_sustained"] * FP4_PER_BF16
        scan_roof = {"achieved": achieved, "frac": achieved / fp4_peak, "unit": "TFLOP/s",
                     "alg_flops_per_launch": fpl, "avg_launch_us": scan["avg_us"]}
    elif scan:
        b = alg_bytes_per_launch("scan_blockmax", g)
        a = b / (scan["avg_us"] * 1e-6) / 1e9
        scan_roof = {"achieved": a, "frac": a / pk["hbm_gbs"], "unit": "GB/s", "alg_bytes_per_launch": b,
                     "avg_launch_us": scan["avg_us"]}
    if dom == "scan_blockmax" and g.B >= MQ_MIN_QUERIES:
        fp4_peak = pk["bf16_tflops_sustained"] * FP4_PER_BF16
        roofline = {"kernel": dom, "bound": "tensor", "achieved": scan_roof["achieved"], "peak": fp4_peak,
                    "unit": "TFLOP/s", "frac": scan_roof["frac"], "traffic": traffic_from_profiles(dom, wl.name),
                    "peak_source": pk_kind + " bf16 sustained x %g (nominal dense FP4 : bf16)" % FP4_PER_BF16,
                    "alg_flops_per_launch": scan_roof["alg_flops_per_launch"], "avg_launch_us": scan["avg_us"],
                    "note": "achieved = 2 x visible positions x 32 heads x 128 dims per query / CUDA-event "
                            "launch time; frac of the measured bf16 peak scaled to FP4"}
    else:
        bpl = alg_bytes_per_launch(dom, g)
        achieved = bpl / (kern[dom]["avg_us"] * 1e-6) / 1e9 if bpl else None
        roofline = {"kernel": dom, "bound": KERNEL_BOUND.get(dom, "hbm"), "roof": "hbm", "achieved": achieved,
                    "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": (achieved / pk["hbm_gbs"]) if achieved else None,
                    "traffic": traffic_from_profiles(dom, wl.name), "peak_source": pk_kind,
                    "alg_bytes_per_launch": bpl, "avg_launch_us": kern[dom]["avg_us"],
                    "note": "achieved = algorithmic bytes per launch / CUDA-event launch time; frac of measured "
                            "copy bandwidth; bound = what limits the kernel per its ncu capture"}
    kern = {k: {kk: (round(vv, 4) if isinstance(vv, float) else vv) for kk, vv in v.items()} for k, v in kern.items()}
    return {"step_ms": step_ms, "total_ms": total_ms, "clocks": clk.summary(), "wall_s_timed": t_wall,
            "launches_per_step": launches_per_step, "kernels": kern, "roofline": roofline, "scan_roofline": scan_roof}


# The metric is quoted at 128K and 1M context: the default line (128K) also
# carries the 1M group's figures under this workload.
SECOND_CONTEXT = {"128k": "1m"}


def run_ours(args):
    import torch
    import torch.distributed as dist
    from csa2_sparse_attention_gb300.layer_group import LayerGroup

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = workload(args.workload)
    g = LayerGroup(wl, device=dev)
    g.fill()
    stream = torch.cuda.Stream(dev)
    flush = L2Flush(dev)
    K = args.steps
    m = measure_group(g, wl, stream, flush, dev, K, args.warmup, world, local)
    value = job_throughput(wl.batch, world, K, m["total_ms"])

    # ---- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(g, stream, flush, min(K, 200), wl)

    # ---- the metric's second context, same step and timing rules
    second = None
    if SECOND_CONTEXT.get(args.workload) and not args.no_second:
        del g
        torch.cuda.empty_cache()
        wl2 = workload(SECOND_CONTEXT[args.workload])
        g2 = LayerGroup(wl2, device=dev)
        g2.fill()
        m2 = measure_group(g2, wl2, stream, flush, dev, K, args.warmup, world, local)
        second = {"workload": wl2.name, "config": config_of(wl2),
                  "value": job_throughput(wl2.batch, world, K, m2["total_ms"]), "unit": UNIT,
                  "ms_per_step": m2["total_ms"] / K, "steps": K, "warmup": args.warmup,
                  "gpu_launches": int(m2["launches_per_step"] * K), "roofline": m2["roofline"],
                  "scan_roofline": m2["scan_roofline"], "kernels": m2["kernels"], "clocks": m2["clocks"]}
        del g2

    cpu = None
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline(args.workload)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
                "warmup": args.warmup, "ms_per_step": m["total_ms"] / K, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None,
                "dtype": "fp4/fp8 storage; f16/bf16 MMA, fp32 accumulate",
                "data": "synthetic (seeded N(0,1) bf16, planted hot blocks)",
                "config": config_of(wl, {"parallelism": f"replicas x{world}", "l2": L2_NOTE}),
                "timing": "CUDA-graph replays of the whole step, CUDA events on the launching stream",
                "gpu_launches": int(m["launches_per_step"] * K),
                "roofline": m["roofline"], "scan_roofline": m["scan_roofline"],
                "kernels": m["kernels"], "clocks": m["clocks"], "wall_s_timed": m["wall_s_timed"],
                "e2e": e2e, "cpu_baseline": cpu}
        if second:
            line["second_context"] = second
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_e2e(g, stream, flush, K, wl):
    """Same metric through the same calls with host buffers: every step brings
    its inputs in from pinned host memory and reads all its outputs back.  The
    copies run on two more streams inside the step's graph (LayerGroup.step_io):
    the inputs arrive in a few growing groups of layers ahead of them and each
    layer's outputs leave in one copy as soon as it is done, while the later
    layers compute."""
    import torch
    host = g.host_buffers()
    h2d, d2h = host.flat_in.numel(), host.flat_out.numel()  # the bytes the copies move
    copy_streams = (torch.cuda.Stream(stream.device), torch.cuda.Stream(stream.device))
    g.capture_io(stream, copy_streams, host)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    with torch.cuda.stream(stream):
        for _ in range(3):
            flush()
            g.replay_io()
        for k in range(K):
            flush()
            evs[k][0].record(stream)
            g.replay_io()
            evs[k][1].record(stream)
    stream.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in evs)
    return {"value": g.B * K / (ms / 1000.0), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": K,
            "note": "host copies pipelined with the layers on two copy streams inside the step's graph: "
                    "inputs in 5 grouped copies ahead of their use, one output copy per layer"}


# ----------------------------------------------------------- ncu launch list
NCU_NAMES = (("score_tc_kernel<false", "scan_blockmax"), ("score_tc_kernel<true", "pool_score"),
             ("score_tc_kernel<0", "scan_blockmax"), ("score_tc_kernel<1", "pool_score"),
             ("select_blocks_kernel", "select_blocks"), ("select_blocks_cluster_kernel", "select_blocks"),
             ("select_topk_kernel", "select_topk"),
             ("attn_tc_kernel", "attn_split"), ("attn_query_kernel", "attn_split"), ("attn_merge_kernel", "attn_merge"),
             ("quantize_fp4_kernel", "quantize_fp4"), ("quantize_fp8_kernel", "quantize_fp8"))


def ncu_summary(csv_path, steps):
    """Per-kernel launches, device time and share from an ncu
    `--metrics gpu__time_duration.sum --csv` launch list of the timed steps."""
    import csv
    rows = []
    with open(csv_path) as f:
        lines = [ln for ln in f if ln.startswith('"')]
    for r in csv.DictReader(lines):
        if r.get("Metric Name") != "gpu__time_duration.sum":
            continue
        name = r["Kernel Name"]
        key = next((ours for pat, ours in NCU_NAMES if pat in name.replace(" ", "")), None)
        unit = r.get("Metric Unit", "ns")
        v = float(r["Metric Value"].replace(",", ""))
        ns = v * {"ns": 1.0, "nsecond": 1.0, "us": 1e3, "usecond": 1e3, "ms": 1e6, "msecond": 1e6}.get(unit, 1.0)
        rows.append((key or "other: " + name.split("(")[0][:60], ns))
    tot = sum(ns for k, ns in rows if not k.startswith("other"))
    agg = {}
    for k, ns in rows:
        a = agg.setdefault(k, [0, 0.0])
        a[0] += 1
        a[1] += ns
    out = [f"{'kernel':<28}{'launches/step':>14}{'us/step':>10}{'us/launch':>11}{'share':>8}"]
    for k, (cnt, ns) in sorted(agg.items(), key=lambda kv: -kv[1][1]):
        share = f"{ns / tot:8.3f}" if not k.startswith("other") else "       -"
        out.append(f"{k:<28}{cnt / steps:>14.1f}{ns / 1e3 / steps:>10.1f}{ns / 1e3 / cnt:>11.2f}{share}")
    out.append(f"{'sum of library kernels':<28}{'':>14}{tot / 1e3 / steps:>10.1f}")
    return "\n".join(out)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="128k",
                    choices=["128k", "1m", "tiny", "manyq", "ragged", "encoder", "append"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-second", action="store_true", help="skip the 1M group the default 128K line also reports")
    ap.add_argument("--ncu-summary", metavar="CSV",
                    help="summarize an ncu launch list of the timed steps (--steps gives their number) and exit")
    ap.add_argument("--cpu-baseline-child", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--child-queries", type=int, default=1, help=argparse.SUPPRESS)
    ap.add_argument("--child-seconds", type=float, default=10.0, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.ncu_summary:
        print(ncu_summary(args.ncu_summary, args.steps))
        return
    if args.warmup < 3 and not args.cpu_baseline_child and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    if args.cpu_baseline_child:
        done, secs = oracle_step_sample(args.workload, args.child_queries, args.child_seconds)
        print(json.dumps({"done": done, "seconds": secs}))
        return
    if args.impl == "reference":
        run_reference(args)
        return
    if args.workload == "append":
        run_append(args)
        return
    run_ours(args)


if __name__ == "__main__":
    main()
