#!/usr/bin/env python
"""Throughput of cached-KV attention: (item, query) pairs per second per
layer-attention, and the dominant kernel's achieved HBM bandwidth.

A step is one pass of the hot path over one batch: every layer of the
workload, one library launch per layer, each launch reading its layer's slice
of the cached-KV pool.  Inputs (Q, K_new, V_new, ids) are resident in HBM
before timing; they are larger than L2 (3.4 GB per launch for the gist
workload), so each launch streams from DRAM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload gist]
  python bench.py --impl reference ...   # the fp64 oracle on the host cores

Other rows: --workload {tiny,gist,qgist,wide,paged,paged_gqa}; --kv fp8 (the
same workload from an E4M3 pool, the roofline counting fp8 bytes); --fused
(QKV projection with RoPE, attention on its pre-rotated output, output
projection); --row offline | block-mass | sweep [--sweep-point K:L] (the
offline gist pass, the decode step with per-block attention mass and the
append, the k x l sweep).  --queries / --pool-items / --layers shrink a
workload for profiling captures; --no-e2e / --no-cpu-baseline skip those legs.

Under torchrun (N > 1) every rank runs an independent replica of the
workload on its own GPU (weak scaling, no collective on the data path); the
reported time is the maximum over ranks.

The plain default single-GPU run (no profiling options) also times the other
workloads and the E4M3 pools after the headline measurement, a few steps
each, and reports them under "rows" in the same JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "(item,query) pairs/s per layer-attention; achieved HBM GB/s vs GB300 peak"
UNIT = "pairs/s"
FALLBACK_HBM_GBS = 6800.0
# the dominant kernel of each workload and the sources it is built from
KERNEL_OF = {
    "gist": ("prefill_tc_kernel", ["prefill_tc.cu", "tcgen05.cuh", "common.cuh", "exact.cuh"]),
    "wide": ("prefill_tc_kernel", ["prefill_tc.cu", "tcgen05.cuh", "common.cuh", "exact.cuh"]),
    "tiny": ("prefill_tc_kernel", ["prefill_tc.cu", "tcgen05.cuh", "common.cuh", "exact.cuh"]),
    "qgist": ("decode_short_kernel", ["decode_short.cu", "frag.cuh", "common.cuh"]),
    "paged": ("decode_long_kernel", ["decode_long.cu", "common.cuh"]),
    "paged_gqa": ("decode_gqa_kernel", ["decode_gqa.cu", "frag.cuh", "common.cuh"]),
    "offline": ("prefill_long_kernel", ["prefill_long.cu", "tcgen05.cuh", "common.cuh", "exact.cuh"]),
}

DESCR = {
    "gist": "gist relevance: 24 layers, Hq=14, Hkv=2, d=64, k=8, l=64; 256 queries x 50 "
            "Zipf(1.1) candidates (12,800 pairs); pool 100k items (9.2 GiB bf16)",
    "qgist": "query also gisted: 24 layers, Hq=14, Hkv=2, d=64, l=1 against 8 item-gist + 8 "
             "query-gist positions; 500 queries x 50 Zipf(1.1) candidates (25,000 pairs)",
    "wide": "wide-KV gist: 28 layers, Hq=32, Hkv=8, d=128, k=8, l=64; 128 queries x 50 uniform "
            "candidates (6,400 pairs); pool 20k items",
    "paged": "paged decode: 32 layers, Hq=Hkv=32, d=128, l=1, 4096 cached tokens in 16 blocks "
             "of 256 behind permuted block tables; batch 32",
    "paged_gqa": "paged GQA decode: 28 layers, Hq=32, Hkv=8, d=128, l=1, 4096 cached tokens in 16 "
                 "blocks of 256 behind permuted block tables; batch 32",
    "tiny": "tiny: 1 layer, Hq=14, Hkv=2, d=64, k=8, l=64, 32 pairs, pool 16 items",
}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="gist", choices=sorted(DESCR))
    ap.add_argument("--report", default=None, help="also write a detailed JSON report here")
    ap.add_argument("--queries", type=int, default=0, help="smaller batch (profiling runs)")
    ap.add_argument("--pool-items", type=int, default=0, help="smaller pool (profiling runs)")
    ap.add_argument("--layers", type=int, default=0, help="fewer layers (profiling runs)")
    ap.add_argument("--kv", choices=["bf16", "fp8"], default="bf16",
                    help="cached-KV element type (fp8: E4M3 pool with per-block scales)")
    ap.add_argument("--fused", action="store_true",
                    help="also time the projections either side (QKV + RoPE, output projection)")
    ap.add_argument("--row", choices=["offline", "block-mass", "sweep"], default=None,
                    help="measure a widening row instead of the hot path: the offline gist "
                         "compression pass, the paged decode with per-block attention mass + append, "
                         "or the gist workload over k x l (one JSON line per point)")
    ap.add_argument("--sweep-point", default=None,
                    help="with --row sweep: only this k:l point (profiling runs)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target CPU time of the oracle sample")
    ap.add_argument("--no-extra-rows", action="store_true",
                    help="skip the other workloads' rows of the default single-GPU run")
    return ap.parse_args(argv)


# The default single-GPU run also times these (workload, KV element type) rows
# after the headline one, a few steps each, and reports them under "rows".
EXTRA_ROWS = [("wide", "bf16"), ("qgist", "bf16"), ("paged", "bf16"), ("paged_gqa", "bf16"),
              ("gist", "fp8"), ("wide", "fp8"), ("qgist", "fp8"), ("paged", "fp8"),
              ("paged_gqa", "fp8")]
EXTRA_ROWS_SECONDS = 60.0  # no further row starts after this much wall time


# ----------------------------------------------------------------- helpers ---

def algorithmic_bytes_per_launch(wl, kv_elem_bytes: int = 2) -> dict:
    """Compulsory bytes of one launch: every pair's Q, K_new, V_new, O and ids
    once, plus every distinct cached block of the layer once (with its scales
    for an fp8 pool)."""
    d = wl.dims
    P, l, Hq, Hkv, hd = d["num_pairs"], d["n_new"], d["num_q_heads"], d["num_kv_heads"], d["head_dim"]
    per_pair = 2 * l * Hq * hd * 2 + 2 * l * Hkv * hd * 2 + 4 * d["blocks_per_pair"]
    block = 2 * Hkv * d["block_len"] * hd * kv_elem_bytes + (2 * Hkv * 4 if kv_elem_bytes == 1 else 0)
    uniq = wl.meta["unique_blocks"]
    return {"per_pair": per_pair, "per_block": block, "unique_blocks": uniq,
            "total": P * per_pair + uniq * block,
            "total_per_pair_gather": P * (per_pair + d["blocks_per_pair"] * block)}


def kernel_source_hash(workload: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_OF[workload][1]:
        with open(os.path.join(ROOT, "attention_cached_kv_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal (~8 TB/s): context beside the measured copy peak


def measured_peaks() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic(workload: str, variant: str = ""):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the kernel sources as they are now; else None.  `variant` names a second
    record of the same workload (e.g. "fp8" for the E4M3 pool)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(workload + ("_" + variant if variant else ""))
    except (OSError, ValueError):
        return None
    if not rec or rec.get("kernel_sources_sha") != kernel_source_hash(workload):
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples (every 50 ms) of the SM clock and throttle reasons;
    only samples stamped inside the timed window are summarised."""
    QUERY = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.window = [None, None]

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits", "-lms", "50"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.5)

    def begin(self):
        self.window[0] = time.time()

    def end(self):
        self.window[1] = time.time()

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        import datetime as _dt
        rows = []
        for line in out.strip().splitlines():
            r = [x.strip() for x in line.split(",")]
            if len(r) < 9:
                continue
            try:
                ts = _dt.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            rows.append((ts, r))
        t0, t1 = self.window
        inside = [r for ts, r in rows if t0 is not None and t0 <= ts <= (t1 or ts)]
        use = inside if inside else [r for _, r in rows]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [v for v in (num(r[1]) for r in use) if v is not None]
        mx = [v for v in (num(r[2]) for r in use) if v is not None]
        reasons = sorted({name for r in use for name, val in zip(self.NAMES, r[5:9])
                          if val.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside),
                "note": None if inside else "no sample fell inside the timed window; all samples used"}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return ws, int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(value: float, ws: int) -> float:
    if ws == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------- CPU baseline ---

def oracle_rate(wl, layer: int, target_s: float) -> dict:
    import numpy as np
    import torch

    import oracle

    cores = len(os.sched_getaffinity(0))
    P = wl.dims["num_pairs"]

    def run(n):
        sel = np.arange(n) * max(1, P // max(n, 1)) % P
        idx = torch.from_numpy(sel).to(wl.q.device)
        q = wl.q.index_select(0, idx).cpu()
        kn = wl.k_new.index_select(0, idx).cpu()
        vn = wl.v_new.index_select(0, idx).cpu()
        dims = dict(wl.dims, num_pairs=n, num_layers=1, layer=0)
        pool = ids = table = None
        C = wl.dims["block_len"] * wl.dims["blocks_per_pair"]
        if C > 0:
            src = wl.block_table if wl.block_table is not None else wl.item_ids.view(-1, 1)
            blocks = src.index_select(0, idx).cpu().numpy()
            uniq, inv = np.unique(blocks, return_inverse=True)
            inv = inv.reshape(blocks.shape).astype(np.int32)
            pool = wl.kv_pool[:, layer].index_select(0, torch.from_numpy(uniq).to(wl.q.device).long())
            pool = pool.unsqueeze(1).contiguous().cpu()
            dims["num_blocks"] = len(uniq)
            if wl.block_table is not None:
                table = inv
            else:
                ids = inv[:, 0].copy()
        t0 = time.perf_counter()
        oracle.gist_attn(q, kn, vn, pool, item_ids=ids, block_table=table, dims=dims,
                         num_threads=cores)
        return time.perf_counter() - t0

    n0 = min(P, max(cores, 8))
    t0 = run(n0)
    want = n0 * target_s / max(t0, 1e-6)  # pairs that take about target_s
    n = int(min(P, max(n0, want)))
    # a layer that takes well under target_s is timed over as many passes as
    # that takes
    t, reps = run(n), 1
    while n == P and t < target_s:
        t += run(n)
        reps += 1
    passes = f", {reps} passes" if reps > 1 else ""
    return {"value": n * reps / t, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} of {P} pairs of layer {layer}, all heads and tokens{passes} ({t:.1f} s)"}


# -------------------------------------------------------------- our arm ---

def run_ours(args) -> dict:
    import torch

    from attention_cached_kv_gb300 import binding, workloads

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    binding.load_library()
    over = {}
    if args.queries:
        over["queries"] = args.queries
    if args.pool_items:
        over["pool_items"] = args.pool_items
    if args.layers:
        over["num_layers"] = args.layers
    wl = workloads.make(args.workload, device=dev, **over)
    L, P = wl.dims["num_layers"], wl.dims["num_pairs"]
    kv_scale = None
    if args.kv == "fp8":
        wl.kv_pool, kv_scale = workloads.make_fp8_pool(wl)
    stream = torch.cuda.Stream(device=dev)
    out = torch.empty_like(wl.q)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    dims_by_layer = [binding.make_dims(dict(wl.dims, layer=li), status) for li in range(L)]
    lib = binding.load_library()
    import ctypes
    V = ctypes.c_void_p
    ptrs = [V(t.data_ptr()) if t is not None else None for t in
            (wl.q, wl.k_new, wl.v_new, wl.kv_pool, wl.item_ids, wl.block_table, wl.pos_offset, out)]
    sh = V(stream.cuda_stream)
    if kv_scale is not None:  # fp8 entry point: the scales follow the pool pointer
        fwd = lib.gist_attn_fwd_fp8kv
        ptrs = ptrs[:4] + [V(kv_scale.data_ptr())] + ptrs[4:]
    else:
        fwd = lib.gist_attn_fwd

    def launch(li):
        rc = fwd(*ptrs, ctypes.byref(dims_by_layer[li]), sh)
        if rc != 0:
            raise binding.GistAttnError(rc, binding.status_string(rc))

    def step(ev=None):
        for li in range(L):
            if ev is not None:
                ev[li][0].record(stream)
            launch(li)
            if ev is not None:
                ev[li][1].record(stream)

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}: {binding.status_string(int(status.item()))}")

    K = args.steps
    events = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(L)] for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid if rank == 0 else None) if rank == 0 else None
    if clocks:
        clocks.start()
    barrier(ws)
    torch.cuda.synchronize(dev)
    if clocks:
        clocks.begin()
    start.record(stream)
    for k in range(K):
        step(events[k])
    end.record(stream)
    torch.cuda.synchronize(dev)
    if clocks:
        clocks.end()
    barrier(ws)
    clk = clocks.stop() if clocks else None
    elapsed_ms = start.elapsed_time(end)
    launch_ms = [events[k][li][0].elapsed_time(events[k][li][1]) for k in range(K) for li in range(L)]
    elapsed_ms = max_over_ranks(elapsed_ms, ws)
    avg_launch_ms = max_over_ranks(sum(launch_ms) / len(launch_ms), ws)

    bytes_info = algorithmic_bytes_per_launch(wl, 1 if kv_scale is not None else 2)
    peak, peak_src = measured_peaks()
    achieved = bytes_info["total"] / (avg_launch_ms * 1e-3) / 1e9
    traffic = recorded_traffic(args.workload, "fp8" if kv_scale is not None else "")
    value = P * L * K * ws / (elapsed_ms * 1e-3)
    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16; ids per the workload recipe)",
        "config": {"workload": DESCR[args.workload] + ("; E4M3 KV pool, fp32 scale per block-head"
                                                       if kv_scale is not None else ""),
                   "pairs": P, "layers_per_step": L,
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "l2": "inputs larger than L2 (no flush needed)"},
        "roofline": {"kernel": KERNEL_OF[args.workload][0],
                     "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
                     "peak_source": f"{peak_src} copy bandwidth (MEASURED_PEAKS hbm_gbs)"
                     if peak_src == "measured" else "fallback 6.8 TB/s",
                     "algorithmic_bytes_per_launch": bytes_info["total"],
                     "avg_launch_ms": avg_launch_ms},
        "gpu_launches": K * L,
        "clocks": clk,
        "impl": "ours",
    }

    if args.fused and kv_scale is None and wl.dims["n_new"] > 1:
        res["fused_layer"] = run_fused(args, wl, stream, ws)
    if not args.no_e2e and kv_scale is None:
        res["e2e"] = run_e2e(args, wl, lib, ptrs, dims_by_layer, stream, ws)
    if not args.no_cpu_baseline and rank == 0 and ws == 1:
        res["cpu_baseline"] = oracle_rate(wl, 0, args.cpu_seconds)
    return res


def run_fused(args, wl, stream, ws) -> dict:
    """One layer's projections around the attention, each timed on its own:
    QKV projection with RoPE in the epilogue, the attention on its pre-rotated
    output, the output projection (d_model = Hq * d, synthetic weights)."""
    import torch

    from attention_cached_kv_gb300 import binding

    d = wl.dims
    P, l, Hq, Hkv, hd, L = (d["num_pairs"], d["n_new"], d["num_q_heads"], d["num_kv_heads"],
                            d["head_dim"], d["num_layers"])
    dm = Hq * hd
    dev = wl.q.device
    g = torch.Generator(device=dev).manual_seed(11)
    x = torch.randn((P, l, dm), generator=g, device=dev).to(torch.bfloat16)
    wqkv = (torch.randn(((Hq + 2 * Hkv) * hd, dm), generator=g, device=dev) / dm ** 0.5).to(torch.bfloat16)
    wo = (torch.randn((dm, Hq * hd), generator=g, device=dev) / dm ** 0.5).to(torch.bfloat16)
    q, kn, vn = torch.empty_like(wl.q), torch.empty_like(wl.k_new), torch.empty_like(wl.v_new)
    attn, y = torch.empty_like(wl.q), torch.empty((P, l, dm), dtype=torch.bfloat16, device=dev)
    pre = dict(d, flags=binding.FLAG_PREROTATED)
    steps = max(1, min(args.steps, 5))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps * L)]

    def layer(li, e=None):
        dl = dict(d, layer=li)
        with torch.cuda.stream(stream):
            if e: e[0].record(stream)
            binding.gist_qkv_rope(x, wqkv, wl.pos_offset, q, kn, vn, dims=dl, stream=stream)
            if e: e[1].record(stream)
            binding.gist_attn_fwd(q, kn, vn, wl.kv_pool, wl.item_ids, wl.block_table, wl.pos_offset,
                                  attn, dims=dict(pre, layer=li), stream=stream)
            if e: e[2].record(stream)
            binding.gist_out_proj(attn, wo, y, dims=dl, stream=stream)
            if e: e[3].record(stream)

    for li in range(min(L, 3)):
        layer(li)
    torch.cuda.synchronize()
    n = 0
    for _ in range(steps):
        for li in range(L):
            layer(li, ev[n])
            n += 1
    torch.cuda.synchronize()
    t = [sum(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(n)) / n for j in range(3)]
    t = [max_over_ranks(v, ws) for v in t]
    M = P * l
    fl_qkv = 2.0 * M * dm * (Hq + 2 * Hkv) * hd
    fl_o = 2.0 * M * (Hq * hd) * dm
    peak = None
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak = float(json.load(f)["bf16_tflops"])
    except (OSError, KeyError, ValueError):
        peak = 1900.0
    tq, to = fl_qkv / (t[0] * 1e-3) / 1e12, fl_o / (t[2] * 1e-3) / 1e12
    return {"d_model": dm, "qkv_rope_ms": t[0], "attention_ms": t[1], "out_proj_ms": t[2],
            "qkv_rope_tflops": tq, "out_proj_tflops": to, "peak_tflops": peak,
            "qkv_rope_frac": tq / peak, "out_proj_frac": to / peak,
            "peak_source": "MEASURED_PEAKS bf16_tflops (burst, cuBLAS)",
            "note": "synthetic weights; per-layer launches timed one by one on the launching stream"}


def run_e2e(args, wl, lib, ptrs, dims_by_layer, stream, ws) -> dict:
    """Same metric through the C ABI with inputs in pinned host memory: every
    layer copies that layer's Q/K_new/V_new (and ids) host -> device, runs the
    kernel, and copies the output back.  Two device buffer sets and three
    streams (host->device, compute, device->host) let layer i's copies overlap
    layer i-1's kernel and read-back, as a serving loop would run them."""
    import ctypes

    import torch

    L, P = wl.dims["num_layers"], wl.dims["num_pairs"]
    ids = wl.item_ids if wl.item_ids is not None else wl.block_table
    use_ids = wl.item_ids is not None
    host = {n: t.cpu().pin_memory() for n, t in (("q", wl.q), ("k", wl.k_new), ("v", wl.v_new), ("ids", ids))}
    host_out = [torch.empty(wl.q.shape, dtype=wl.q.dtype, pin_memory=True) for _ in range(2)]
    sets = []
    for b in range(2):
        d = {"q": wl.q if b == 0 else torch.empty_like(wl.q),
             "k": wl.k_new if b == 0 else torch.empty_like(wl.k_new),
             "v": wl.v_new if b == 0 else torch.empty_like(wl.v_new),
             "ids": ids if b == 0 else torch.empty_like(ids),
             "out": torch.empty_like(wl.q)}
        p = list(ptrs)
        V = ctypes.c_void_p
        p[0], p[1], p[2], p[7] = V(d["q"].data_ptr()), V(d["k"].data_ptr()), V(d["v"].data_ptr()), V(d["out"].data_ptr())
        if use_ids:
            p[4] = V(d["ids"].data_ptr())
        else:
            p[5] = V(d["ids"].data_ptr())
        d["ptrs"] = p
        sets.append(d)
    h2d_s, d2h_s = torch.cuda.Stream(device=wl.q.device), torch.cuda.Stream(device=wl.q.device)
    sh = ctypes.c_void_p(stream.cuda_stream)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = host_out[0].numel() * host_out[0].element_size()
    ev = {n: [torch.cuda.Event() for _ in range(2)] for n in ("in", "done", "back")}

    def step():
        for li in range(L):
            b = li & 1
            d = sets[b]
            with torch.cuda.stream(h2d_s):
                h2d_s.wait_event(ev["done"][b])  # the kernel two layers back read this set
                d["q"].copy_(host["q"], non_blocking=True)
                d["k"].copy_(host["k"], non_blocking=True)
                d["v"].copy_(host["v"], non_blocking=True)
                d["ids"].copy_(host["ids"], non_blocking=True)
                ev["in"][b].record(h2d_s)
            stream.wait_event(ev["in"][b])
            stream.wait_event(ev["back"][b])  # this set's previous output has left
            rc = lib.gist_attn_fwd(*d["ptrs"], ctypes.byref(dims_by_layer[li]), sh)
            if rc != 0:
                raise RuntimeError(f"gist_attn_fwd returned {rc}")
            ev["done"][b].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(ev["done"][b])
                host_out[b].copy_(d["out"], non_blocking=True)
                ev["back"][b].record(d2h_s)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    K = max(1, args.steps)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    start.record(stream)
    h2d_s.wait_event(start)
    d2h_s.wait_event(start)
    for _ in range(K):
        step()
    stream.wait_event(ev["back"][0])
    stream.wait_event(ev["back"][1])
    end.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(start.elapsed_time(end), ws)
    return {"value": P * L * K * ws / (ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d * L,
            "d2h_bytes_per_step": d2h * L, "steps": K,
            "overlap": "two buffer sets; host->device, compute and device->host streams"}


# -------------------------------------------------------- reference arm ---

def run_reference(args) -> dict | None:
    """The fp64 oracle on the host cores, each step a bounded sample of the
    workload (a fresh seeded slice of pairs with its own cached blocks)."""
    import oracle
    from attention_cached_kv_gb300 import workloads

    ws, rank, _ = dist_env()
    if rank != 0:
        return None
    spec = workloads.SPECS[args.workload]
    cores = len(os.sched_getaffinity(0))
    # size one step to a few seconds of host time: calibrate on a small slice
    def slice_of(n, seed):
        return workloads.make_custom(n, spec.n_new, spec.num_q_heads, spec.num_kv_heads,
                                     spec.head_dim, spec.block_len, spec.blocks_per_pair, n,
                                     device="cpu", seed=seed)

    def one(wl):
        t0 = time.perf_counter()
        oracle.gist_attn(wl.q, wl.k_new, wl.v_new, wl.kv_pool, item_ids=wl.item_ids,
                         block_table=wl.block_table, dims=wl.dims, num_threads=cores)
        return time.perf_counter() - t0

    n0 = max(cores, 4)
    t0 = one(slice_of(n0, 100))
    budget_s = 150.0 / max(args.steps + args.warmup, 1)
    n = int(max(n0, min(spec.num_pairs, n0 * min(budget_s, 5.0) / max(t0, 1e-6))))
    for w in range(args.warmup):
        one(slice_of(n, 200 + w))
    times = [one(slice_of(n, 300 + k)) for k in range(args.steps)]
    total = sum(times)
    value = n * args.steps / total
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": DESCR[args.workload], "pairs_per_step": n, "layers_per_step": 1},
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{n} pairs of one layer per step (of {spec.num_pairs})"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def _timed_layers(args, L, launch, stream, ws):
    """W warm-up steps, then K steps of L layers; returns (total ms, per-layer
    ms of each phase) with CUDA events on the launching stream, max over ranks."""
    import torch

    for _ in range(max(args.warmup, 0)):
        for li in range(L):
            launch(li, None)
    torch.cuda.synchronize()
    K = args.steps
    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(L)] for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    start.record(stream)
    for k in range(K):
        for li in range(L):
            launch(li, ev[k][li])
    end.record(stream)
    torch.cuda.synchronize()
    total = max_over_ranks(start.elapsed_time(end), ws)
    ph = [max_over_ranks(sum(e[li][j].elapsed_time(e[li][j + 1]) for e in ev for li in range(L)) / (K * L), ws)
          for j in range(2)]
    return total, ph


def run_sweep(args, dev, stream, status, ws, rank, peak, peak_src):
    """The gist workload (12,800 Zipf pairs, the gist model's heads) with k in
    {1, 4, 8, 16, 32, 64} cached gist positions and l in {16, 64, 256} new
    tokens, each point through gist_attn_fwd on layers 0 and 1 of a two-layer
    pool.  Prints one JSON line per point; returns None."""
    import torch

    from attention_cached_kv_gb300 import binding, workloads

    points = [(k, l_new) for l_new in (16, 64, 256) for k in (1, 4, 8, 16, 32, 64)]
    if args.sweep_point:
        k_, l_ = (int(x) for x in args.sweep_point.split(":"))
        points = [(k_, l_)]
    for k, l_new in points:
        if True:
            over = {"num_layers": 2}
            if args.queries:
                over["queries"] = args.queries
            wl = workloads.make(workloads.sweep_spec(k, l_new), device=dev, **over)
            d = wl.dims
            P, Hq, hd = d["num_pairs"], d["num_q_heads"], d["head_dim"]
            out = torch.empty_like(wl.q)
            nws = binding.workspace_bytes(wl.dims)  # the staged path's scratch, 0 where none
            wsp = torch.empty(nws, dtype=torch.uint8, device=dev) if nws else None

            def launch(li, e, wl=wl, out=out, wsp=wsp):
                if e: e[0].record(stream)
                binding.gist_attn_fwd_ws(wl.q, wl.k_new, wl.v_new, wl.kv_pool, wl.item_ids, None, None, out,
                                         wsp, dims=dict(wl.dims, layer=li), status=status, stream=stream)
                if e:
                    e[1].record(stream)
                    e[2].record(stream)

            _, (t_attn, _) = _timed_layers(args, 2, launch, stream, ws)
            if int(status.item()) != 0:
                raise RuntimeError(f"device status {int(status.item())} at k={k} l={l_new}")
            nbytes = algorithmic_bytes_per_launch(wl)["total"]
            flops = 4.0 * hd * Hq * (l_new * k + l_new * (l_new + 1) / 2) * P  # useful: scores + PV
            gbs = nbytes / (t_attn * 1e-3) / 1e9
            # the library's dispatch: the single-pass tensor-core kernel while a
            # tile's keys fit its TMEM (288), else the staged path (pre-pass +
            # long-sequence kernel), which is when the call wants a workspace
            kernel = "stage_kernel + prefill_long_kernel" if nws else "prefill_tc_kernel"
            if rank == 0:
                print(json.dumps({
                    "metric": "(item,query) pairs/s per layer-attention", "row": "sweep", "k": k, "l": l_new,
                    "value": P * ws / (t_attn * 1e-3), "unit": "pairs/s", "n_gpus": ws,
                    "steps": args.steps, "warmup": args.warmup, "ms_per_launch": t_attn,
                    "higher_is_better": True, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16)",
                    "config": {"workload": f"gist model, {P} Zipf(1.1) pairs, k={k} cached, l={l_new} new",
                               "pairs": P, "layers_timed": 2},
                    "kernel": kernel, "algorithmic_bytes_per_launch": nbytes, "achieved_gbs": gbs,
                    "frac_of_hbm": gbs / peak, "peak_source": peak_src, "workspace_bytes": nws,
                    "tflops": flops / (t_attn * 1e-3) / 1e12}), flush=True)
            del wl, out, wsp
            torch.cuda.empty_cache()
    return None


def run_row(args) -> dict:
    """The widening rows, each through its C-ABI entry points on synthetic data.

    offline: the gist compression pass of Gist page "论文做了什么" / "在线的一次
      attention": B items of j = 1000 prompt tokens + k = 8 gist tokens (an item
      runs to about a thousand tokens on that page), the gist model (Hq 14, Hkv 2,
      d 64), per layer the causal pass over [prompt; gist] through
      gist_attn_fwd_gist_mask, then gist_kv_store of the k gist rows.
    block-mass: the paged decode workload through gist_attn_fwd_block_mass
      (Suffix page §4, §5 第三步) followed by gist_kv_append of the new token
      (KV page "Reusable-state"); the append writes the sequence's last cached
      slot, a stand-in for the next block's first one (the pool has no spare
      block), so the cache the next step reads keeps its size."""
    import torch

    from attention_cached_kv_gb300 import binding, workloads

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    binding.load_library()
    stream = torch.cuda.Stream(device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    peak, peak_src = measured_peaks()
    if args.row == "sweep":
        return run_sweep(args, dev, stream, status, ws, rank, peak, peak_src)
    if args.row == "offline":
        B, j, k = args.queries or 128, 1000, 8
        L = args.layers or 24
        l, Hq, Hkv, d = j + k, 14, 2, 64
        g = torch.Generator(device=dev).manual_seed(21)
        q = torch.randn((B, l, Hq, d), generator=g, device=dev).to(torch.bfloat16)
        kn = torch.randn((B, l, Hkv, d), generator=g, device=dev).to(torch.bfloat16)
        vn = torch.randn((B, l, Hkv, d), generator=g, device=dev).to(torch.bfloat16)
        out = torch.empty_like(q)
        pool = torch.zeros((B, L, 2, Hkv, k, d), dtype=torch.bfloat16, device=dev)
        ids = torch.arange(B, dtype=torch.int32, device=dev)
        gstart = torch.full((B,), j, dtype=torch.int32, device=dev)
        base = dict(num_pairs=B, n_new=l, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, block_len=k,
                    num_blocks=B, num_layers=L, rope_theta=1e4, softmax_scale=0.0)

        # q and k_new as the QKV projection's epilogue leaves them (rotated): the
        # attention takes them with GIST_ATTN_FLAG_PREROTATED and the store
        # writes the gist rows as they are
        pre = binding.FLAG_PREROTATED

        def launch(li, e):
            attn_dims = dict(base, blocks_per_pair=0, layer=li, flags=pre)
            store_dims = dict(base, blocks_per_pair=1, layer=li, flags=pre)
            if e: e[0].record(stream)
            binding.gist_attn_fwd(q, kn, vn, pool, None, None, None, out, dims=attn_dims,
                                  status=status, stream=stream)
            if e: e[1].record(stream)
            binding.gist_kv_store(kn, vn, pool, ids, gstart, None, dims=store_dims, status=status,
                                  stream=stream)
            if e: e[2].record(stream)

        # the same pass on pre-RoPE inputs (the general streaming kernel, gist mask entry)
        def launch_raw(li, e):
            if e: e[0].record(stream)
            binding.gist_attn_fwd_gist_mask(q, kn, vn, pool, None, None, None, gstart, k, out,
                                            dims=dict(base, blocks_per_pair=0, layer=li),
                                            status=status, stream=stream)
            if e: e[1].record(stream)
            if e: e[2].record(stream)

        _, (t_raw, _) = _timed_layers(argparse.Namespace(warmup=1, steps=1), min(L, 4), launch_raw,
                                      stream, ws)

        # the same causal pass on pre-RoPE inputs through the staged path (a
        # pre-pass rotates q and the keys into a workspace, then the long kernel)
        raw_dims = dict(base, blocks_per_pair=0, layer=0)
        wsp = torch.empty(binding.workspace_bytes(raw_dims), dtype=torch.uint8, device=dev)

        def launch_staged(li, e):
            if e: e[0].record(stream)
            binding.gist_attn_fwd_ws(q, kn, vn, pool, None, None, None, out, wsp,
                                     dims=dict(raw_dims, layer=li), status=status, stream=stream)
            if e: e[1].record(stream)
            if e: e[2].record(stream)

        _, (t_staged, _) = _timed_layers(argparse.Namespace(warmup=1, steps=2), min(L, 4), launch_staged,
                                         stream, ws)
        del wsp
        total, (t_attn, t_store) = _timed_layers(args, L, launch, stream, ws)
        if int(status.item()) != 0:
            raise RuntimeError(f"device status {int(status.item())}")
        flops = 4.0 * d * Hq * (l * (l + 1) / 2)      # useful: causal scores + PV per item-layer
        nbytes = 2 * (2 * l * Hq * d) + 2 * (2 * l * Hkv * d)  # q, out, k_new, v_new
        tfl = B * flops / (t_attn * 1e-3) / 1e12
        # the committed capture is of this 128-item pass; other sizes get none
        traffic = recorded_traffic("offline") if B == 128 else None
        bf16_peak = 1890.5
        try:
            with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
                bf16_peak = float(json.load(f)["bf16_tflops"])
        except (OSError, KeyError, ValueError):
            pass
        return {"metric": "items compressed per second per layer (offline gist pass + store)",
                "value": B * L * args.steps * ws / (total * 1e-3), "unit": "items/s",
                "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": total / args.steps, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16)",
                "config": {"workload": f"offline gist compression: {B} items x ({j} prompt + {k} gist) "
                                       f"tokens, {L} layers, Hq={Hq}, Hkv={Hkv}, d={d}; causal pass over "
                                       f"pre-rotated q/k + store of the gist rows",
                           "items": B, "layers_per_step": L},
                "roofline": {"kernel": "prefill_long_kernel", "bound": "tensor",
                             "achieved": tfl, "peak": bf16_peak, "unit": "TFLOP/s",
                             "frac": tfl / bf16_peak, "traffic": traffic,
                             "peak_source": "MEASURED_PEAKS bf16_tflops (cuBLAS burst)",
                             "useful_flops_per_item_layer": flops,
                             "hbm_bytes_per_item_layer": nbytes,
                             "achieved_gbs": B * nbytes / (t_attn * 1e-3) / 1e9,
                             "attention_ms": t_attn, "store_ms": t_store,
                             "pre_rope_streaming_ms": t_raw,
                             "pre_rope_staged_ms": t_staged,
                             "pre_rope_staged_tflops": B * flops / (t_staged * 1e-3) / 1e12,
                             "pre_rope_streaming_tflops": B * flops / (t_raw * 1e-3) / 1e12},
                "gpu_launches": 2 * L * args.steps, "impl": "ours"}
    # block-mass
    wl = workloads.make("paged", device=dev, **({"num_layers": args.layers} if args.layers else {}))
    L, P = wl.dims["num_layers"], wl.dims["num_pairs"]
    dd = wl.dims
    C = dd["block_len"] * dd["blocks_per_pair"]
    out = torch.empty_like(wl.q)
    mass = torch.empty((P, dd["num_q_heads"], dd["blocks_per_pair"]), dtype=torch.float32, device=dev)
    slot = torch.full((P,), C - 1, dtype=torch.int32, device=dev)

    def launch(li, e):
        dl = dict(dd, layer=li)
        if e: e[0].record(stream)
        binding.gist_attn_fwd_block_mass(wl.q, wl.k_new, wl.v_new, wl.kv_pool, wl.block_table, wl.pos_offset,
                                         out, mass, dims=dl, status=status, stream=stream)
        if e: e[1].record(stream)
        binding.gist_kv_append(wl.k_new, wl.v_new, wl.kv_pool, wl.block_table, slot, wl.pos_offset,
                               dims=dl, status=status, stream=stream)
        if e: e[2].record(stream)

    total, (t_dec, t_app) = _timed_layers(args, L, launch, stream, ws)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    bytes_info = algorithmic_bytes_per_launch(wl)
    nbytes = bytes_info["total"] + mass.numel() * 4
    achieved = nbytes / (t_dec * 1e-3) / 1e9
    return {"metric": "(sequence, step) pairs/s per layer: decode with per-block attention mass + KV append",
            "value": P * L * args.steps * ws / (total * 1e-3), "unit": "pairs/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16; permuted block tables)",
            "config": {"workload": DESCR["paged"] + "; per-block attention mass, then the new token appended",
                       "pairs": P, "layers_per_step": L},
            "roofline": {"kernel": "decode_long_kernel (block mass)", "bound": "hbm", "achieved": achieved,
                         "peak": peak, "unit": "GB/s", "frac": achieved / peak, "traffic": None,
                         "peak_source": f"{peak_src} copy bandwidth",
                         "algorithmic_bytes_per_launch": nbytes, "decode_ms": t_dec, "append_ms": t_app},
            "gpu_launches": 2 * L * args.steps, "impl": "ours"}


def wants_extra_rows(args, ws: int) -> bool:
    """Only the plain default run adds the other rows: one GPU, the headline
    workload, none of the options the profiling commands use."""
    return (args.impl == "ours" and ws == 1 and not args.no_extra_rows and not args.row
            and args.workload == "gist" and args.kv == "bf16" and not args.fused
            and not (args.no_e2e or args.no_cpu_baseline or args.queries or args.pool_items
                     or args.layers))


def run_extra_rows(args, run=None) -> list:
    """Each row of EXTRA_ROWS through the same measurement as the headline
    (fewer steps, no e2e or CPU leg); a row that fails is reported with its
    error instead of its numbers, and the headline line is still printed."""
    run = run or run_ours
    rows, t0 = [], time.time()
    for name, kv in EXTRA_ROWS:
        if time.time() - t0 > EXTRA_ROWS_SECONDS:
            rows.append({"workload": name, "kv": kv, "skipped": "time budget of the extra rows"})
            continue
        sub = argparse.Namespace(**vars(args))
        sub.workload, sub.kv, sub.fused = name, kv, False
        sub.steps, sub.warmup = max(1, min(args.steps, 10)), max(3, min(args.warmup, 5))
        sub.no_e2e = sub.no_cpu_baseline = True
        sub.queries = sub.pool_items = sub.layers = 0
        try:
            r = run(sub)
            roof = r["roofline"]
            rows.append({"workload": name, "kv": kv, "config": r["config"]["workload"],
                         "value": r["value"], "unit": r["unit"], "steps": sub.steps,
                         "warmup": sub.warmup, "ms_per_step": r["ms_per_step"],
                         "kernel": roof["kernel"], "avg_launch_ms": roof["avg_launch_ms"],
                         "achieved_gbs": roof["achieved"], "frac": roof["frac"],
                         "algorithmic_bytes_per_launch": roof["algorithmic_bytes_per_launch"],
                         "traffic": roof["traffic"], "gpu_launches": r["gpu_launches"],
                         "clocks": r["clocks"]})
        except Exception as e:  # keep the headline line: report the row's failure
            rows.append({"workload": name, "kv": kv, "error": f"{type(e).__name__}: {e}"[:300]})
        finally:
            try:
                import gc

                import torch
                gc.collect()
                torch.cuda.empty_cache()
            except Exception:
                pass
    return rows


def main(argv=None):
    args = parse_args(argv)
    if args.row and args.impl == "ours":
        res = run_row(args)
    else:
        res = run_reference(args) if args.impl == "reference" else run_ours(args)
    ws, rank, _ = dist_env()
    if res is not None and wants_extra_rows(args, ws):
        res["rows"] = run_extra_rows(args)
    if res is not None and rank == 0:
        line = json.dumps(res)
        print(line, flush=True)
        if args.report:
            with open(args.report, "a") as f:
                f.write(line + "\n")
    if ws > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
