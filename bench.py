"""Throughput of one paged-attention decode step on GB300, as one JSON line.

A step is the whole hot path on one batch: pa_plan + pa_decode + pa_reduce (three kernel
launches) through the C ABI, inputs resident in HBM.  The workload is the batched
grouped-query decode: B=32 sequences, 32 query heads over 8 KV heads, head dim 128, pages
of 16 tokens, context lengths uniform in [512, 4096], bf16, pool = 2x the pages needed.

value      = KV bytes read per step (every valid token's K and V rows; no padding,
             queries, tables or outputs) / device time per step, in TB/s, summed over
             ranks and divided by the slowest rank's time (weak scaling: each rank decodes
             its own batch, no collective on the data path).
e2e        = the same through the public Python binding with host buffers: every step
             copies q, block tables and lengths from pinned host memory and reads out and
             lse back, inside the timed region.  The KV cache is device state.
roofline   = the decode kernel alone (CUDA events around its launches): algorithmic bytes
             / average launch time, against the measured HBM copy peak.
cpu_baseline / --impl reference = the CPU oracle (fp32 C, OpenMP) on the host cores.

L2: two independent input sets of > 2x L2 bytes each alternate between steps, so no
step finds its KV in L2.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload NAME] [--all] [--no-cpu-baseline] [--gather]
--gather times the paged -> contiguous KV copy (pa_gather_kv) of the workload instead.
For N > 1 launch with torchrun (one process per GPU).
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode µs/call and achieved HBM TB/s on KV bytes read vs GB300 peak"
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["paged_kv_cache_work_gb300/csrc/decode_simt.cuh",
                  "paged_kv_cache_work_gb300/csrc/decode_tc.cuh",
                  "paged_kv_cache_work_gb300/csrc/decode_mma.cuh",
                  "paged_kv_cache_work_gb300/csrc/decode_common.cuh",
                  "paged_kv_cache_work_gb300/csrc/pa_internal.cuh"]


def decode_shape(wl):
    """(decode kernel name, rows per unit) the library picks for a workload: a 16-bit cache
    with head dim 128 or 256, or an fp8 cache with head dim 128 and per-tensor or no scales,
    and more than 32 query rows per kv head goes to the tcgen05 kernel in tiles of 64 or 128
    rows; other caches with a tile row of at least 128 bytes to the mma.sync kernel in tiles
    of 16, 32 or 64 rows; the rest (64-dim fp8) to the CUDA-core kernel."""
    rows = (wl.num_q_heads // wl.num_kv_heads) * wl.max_q_len
    bpe = 1 if wl.kv_dtype == "fp8" else 2
    pow2 = 1 << max(0, (rows - 1).bit_length())
    tc_fp8 = wl.head_dim == 128 and wl.scale_mode != "token"
    if wl.head_dim >= 128 and rows >= 33 and (bpe == 2 or tc_fp8):
        return "decode_tc_kernel", 64 if rows <= 64 else 128
    if wl.head_dim * bpe >= 128:
        return "decode_mma_kernel", 64 if rows >= 64 else max(16, pow2)
    return "decode_simt_kernel", min(pow2, 8)


def launches_per_step(split_merge: int) -> int:
    """Kernels one plan/decode/reduce step launches: pa_reduce launches its kernel unless
    every split unit is merged inside the decode (PA_MERGE_IN_DECODE)."""
    import paged_kv_cache_work_gb300 as pa
    return 2 if split_merge == pa.MERGE_IN_DECODE else 3


# ----------------------------------------------------------------------------- helpers
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def aggregate(local_seconds: float, local_bytes: int):
    """(max seconds over ranks, total bytes over ranks); identity without a process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return local_seconds, local_bytes
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([local_seconds], dtype=torch.float64, device=dev)
    b = torch.tensor([float(local_bytes)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(t.item()), int(b.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per decode launch from the committed ncu summary of this workload, or None
    when there is none or the kernel sources changed since it was taken."""
    src = kernel_source_hash()
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        with open(path) as f:
            text = f.read()
        w = re.search(r"^workload:\s*(\S+)", text, re.M)
        s = re.search(r"^kernel_source_sha256:\s*(\S+)", text, re.M)
        t = re.search(r"^dram_bytes_per_launch:\s*([0-9.eE+]+)", text, re.M)
        if w and s and t and w.group(1) == workload and s.group(1) == src:
            return float(t.group(1)), os.path.relpath(path, ROOT)
    return None, None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)], stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        self.t_start = time.time()

    def mark(self):
        return time.time()

    def stop(self, t0, t1):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        with open(self.file.name) as f:
            lines = [ln.strip() for ln in f if ln.strip()]
        os.unlink(self.file.name)
        rows = []
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), active=parts[4],
                                 hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        # samples are 100 ms apart: keep the ones that fall in the busy window
        n_busy = max(1, int((t1 - t0) / 0.1))
        busy = rows[-(n_busy + 2):] if len(rows) > n_busy else rows
        reasons = set()
        for r in busy:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in busy),
                "sm_max_mhz": max(r["smax"] for r in busy), "reasons": sorted(reasons),
                "samples": len(busy)}


# ------------------------------------------------------------------------ CPU oracle leg
def time_oracle(inp_cpu, budget_s: float, max_calls: int = 1000):
    """Median seconds per oracle call over as many calls as fit in budget_s (at least 1)."""
    import oracle
    times = []
    t_end = time.perf_counter() + budget_s
    while len(times) < max_calls:
        t = time.perf_counter()
        oracle.decode(inp_cpu, "f32")
        times.append(time.perf_counter() - t)
        if time.perf_counter() > t_end:
            break
    return statistics.median(times), len(times)


def oracle_sample(inp_cpu, max_seconds_per_call: float):
    """A sub-batch of the workload (whole sequences) whose oracle call takes about
    max_seconds_per_call; returns (sample, description)."""
    import oracle
    import workloads as W
    B = inp_cpu["workload"].batch
    one = _sub_batch(inp_cpu, [0])
    t = time.perf_counter()
    oracle.decode(one, "f32")
    per_seq = max(time.perf_counter() - t, 1e-6)
    n = max(1, min(B, int(max_seconds_per_call / per_seq)))
    if n >= B:
        return inp_cpu, f"the whole batch ({B} sequences)"
    return _sub_batch(inp_cpu, list(range(n))), f"the first {n} of {B} sequences"


def _sub_batch(inp, seqs):
    import torch
    w = inp["workload"].replace(batch=len(seqs))
    idx = torch.tensor(seqs, dtype=torch.long)
    out = dict(inp)
    out["workload"] = w
    for k in ("q", "block_tables", "context_lens", "q_lens"):
        out[k] = inp[k][idx].contiguous()
    return out


# ------------------------------------------------------------------------- GPU leg
def run_ours(args, rank, world, local):
    import torch
    import paged_kv_cache_work_gb300 as pa
    import workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = W.FULL[args.workload]
    pa.load()
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 0)
    seed = W.SEEDS[0] + rank
    sets = [W.make_inputs(wl, seed + 7919 * k, device=dev) for k in range(2)]
    cfg = pa.config_for(sets[0])
    step_bytes = [W.kv_bytes(s) for s in sets]
    for s in sets:
        s["out"] = torch.empty_like(s["q"])
        s["lse"] = torch.empty(s["q"].shape[:3], dtype=torch.float32, device=dev)
        s["ws"] = torch.empty(pa.workspace_size(cfg), dtype=torch.uint8, device=dev)
        s["cfg"] = pa.config_for(s)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    def step(s, ev=None):
        c = s["cfg"]
        pa.plan(c, s["block_tables"], s["context_lens"], s["q_lens"], s["ws"], sh)
        if ev is not None:
            ev[0].record(stream)
        pa.decode(c, s["q"], s["k_cache"], s["v_cache"], s["k_scale"], s["v_scale"],
                  s["block_tables"], s["context_lens"], s["q_lens"], s["out"], s["lse"],
                  s["ws"], sh)
        if ev is not None:
            ev[1].record(stream)
        pa.reduce(c, s["out"], s["lse"], s["ws"], sh)

    for k in range(args.warmup):
        step(sets[k % 2])
    torch.cuda.synchronize(dev)
    for s in sets:
        if pa.read_flags(s["ws"]) != 0:
            raise RuntimeError("device flags set on the bench inputs")

    # One CUDA graph per input set holds the step's three launches, so the timed loop
    # measures the device and not the Python launch path.
    graphs = []
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    for s in sets:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                c = s["cfg"]
                csh = cap.cuda_stream
                pa.plan(c, s["block_tables"], s["context_lens"], s["q_lens"], s["ws"], csh)
                pa.decode(c, s["q"], s["k_cache"], s["v_cache"], s["k_scale"], s["v_scale"],
                          s["block_tables"], s["context_lens"], s["q_lens"], s["out"], s["lse"],
                          s["ws"], csh)
                pa.reduce(c, s["out"], s["lse"], s["ws"], csh)
        graphs.append(g)
    stream.wait_stream(cap)
    for k in range(max(3, args.warmup)):
        graphs[k % 2].replay()
    torch.cuda.synchronize(dev)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.25)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    start.record(stream)
    total_bytes = 0
    for k in range(args.steps):
        graphs[k % 2].replay()
        total_bytes += step_bytes[k % 2]
    stop.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    t_wall1 = time.time()
    seconds = start.elapsed_time(stop) / 1e3
    max_s, all_bytes = aggregate(seconds, total_bytes)

    # The decode kernel alone: CUDA events around each launch on its stream.  The host
    # enqueues decodes faster than they run, so each pair brackets one kernel.
    n_dec = max(8, min(args.steps, 2000))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n_dec)]
    for k in range(n_dec):
        s = sets[k % 2]
        evs[k][0].record(stream)
        pa.decode(s["cfg"], s["q"], s["k_cache"], s["v_cache"], s["k_scale"], s["v_scale"],
                  s["block_tables"], s["context_lens"], s["q_lens"], s["out"], s["lse"],
                  s["ws"], sh)
        evs[k][1].record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop(t_wall0, time.time())
    decode_ms = [a.elapsed_time(b) for a, b in evs[4:]]

    # end to end through the binding with host buffers
    n_e2e = max(1, min(args.steps, 200))
    host = []
    for s in sets:
        hs = {k: s[k].cpu().pin_memory() for k in ("q", "block_tables", "context_lens", "q_lens")}
        hs["out"] = torch.empty(s["out"].shape, dtype=s["out"].dtype).pin_memory()
        hs["lse"] = torch.empty(s["lse"].shape, dtype=torch.float32).pin_memory()
        host.append(hs)
    h2d = sum(host[0][k].numel() * host[0][k].element_size()
              for k in ("q", "block_tables", "context_lens", "q_lens"))
    d2h = sum(host[0][k].numel() * host[0][k].element_size() for k in ("out", "lse"))

    def e2e_step(s, hs):
        for k in ("q", "block_tables", "context_lens", "q_lens"):
            s[k].copy_(hs[k], non_blocking=True)
        step(s)
        hs["out"].copy_(s["out"], non_blocking=True)
        hs["lse"].copy_(s["lse"], non_blocking=True)

    for k in range(3):
        e2e_step(sets[k % 2], host[k % 2])
    torch.cuda.synchronize(dev)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_bytes = 0
    e0.record(stream)
    for k in range(n_e2e):
        e2e_step(sets[k % 2], host[k % 2])
        e2e_bytes += step_bytes[k % 2]
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_s, e2e_all = aggregate(e0.elapsed_time(e1) / 1e3, e2e_bytes)

    result = None
    if rank == 0:
        peak, peak_kind = measured_hbm_peak()
        mean_decode_s = statistics.fmean(decode_ms) / 1e3
        bytes_per_launch = statistics.fmean(step_bytes)
        achieved_gbs = bytes_per_launch / mean_decode_s / 1e9
        traffic, traffic_src = profiled_traffic(wl.name)
        value = all_bytes / max_s / 1e12
        per_step_s = max_s / args.steps
        result = {
            "metric": METRIC, "value": round(value, 4), "unit": "TB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(per_step_s * 1e3, 5),
            "us_per_call": round(per_step_s * 1e6, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {
                "workload": wl.name, "batch": wl.batch, "num_q_heads": wl.num_q_heads,
                "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim,
                "block_size": wl.block_size, "context_lens": f"U[{wl.ctx_lo},{wl.ctx_hi}]",
                "max_q_len": wl.max_q_len, "kv_dtype": wl.kv_dtype, "q_dtype": wl.q_dtype,
                "kv_bytes_per_step": int(bytes_per_launch),
                "l2": (f"inputs larger than L2: 2 input sets of {int(bytes_per_launch) >> 20} MiB KV "
                       f"alternate (L2 {l2 >> 20} MiB)"),
                "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                "grid_mult": int(cfg.grid_mult) or 1,
                "split_merge": "auto (decode's last CTA merges units of few pieces, "
                               "the reduce kernel the rest)",
            },
            "roofline": {
                "kernel": decode_shape(wl)[0], "bound": "hbm", "achieved": round(achieved_gbs, 1),
                "peak": peak, "unit": "GB/s", "frac": round(achieved_gbs / peak, 4),
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                else "fallback 6.8 TB/s",
                "decode_us_mean": round(mean_decode_s * 1e6, 2),
                "decode_us_median": round(statistics.median(decode_ms) * 1e3, 2),
                "traffic": traffic, "traffic_source": traffic_src,
            },
            "e2e": {"value": round(e2e_all / e2e_s / 1e12, 4), "unit": "TB/s",
                    "us_per_call": round(e2e_s / n_e2e * 1e6, 2), "steps": n_e2e,
                    "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)},
            "gpu_launches": launches_per_step(cfg.split_merge) * args.steps,
            "timing": "device time of K CUDA-graph replays of the step (plan, decode, reduce)",
            "clocks": clocks,
        }
        if not args.no_cpu_baseline:
            inp_cpu = {k: (v.cpu() if isinstance(v, torch.Tensor) else v)
                       for k, v in sets[0].items() if k not in ("out", "lse", "ws", "cfg")}
            sample, desc = oracle_sample(inp_cpu, 2.0)
            sec, calls = time_oracle(sample, 12.0)
            import oracle
            result["cpu_baseline"] = {
                "value": round(W.kv_bytes(sample) / sec / 1e12, 6), "unit": "TB/s",
                "us_per_call": round(sec * 1e6, 1), "cores": oracle.threads(), "kind": "oracle",
                "sample": f"{desc} of the bench workload, median of {calls} calls"}
    return result


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm, on the same workload's shapes."""
    if rank != 0:
        return None
    import oracle
    import workloads as W
    wl = W.FULL[args.workload]
    inp = W.make_inputs(wl, W.SEEDS[0])
    per_step_budget = max(0.02, 120.0 / max(1, args.steps + args.warmup))
    sample, desc = oracle_sample(inp, per_step_budget)
    for _ in range(args.warmup):
        oracle.decode(sample, "f32")
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle.decode(sample, "f32")
    sec = (time.perf_counter() - t) / max(1, args.steps)
    value = W.kv_bytes(sample) / sec / 1e12
    cpu = {"value": round(value, 6), "unit": "TB/s", "cores": oracle.threads(), "kind": "oracle",
           "sample": f"{desc} of {wl.name} per step"}
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(sec * 1e3, 3), "us_per_call": round(sec * 1e6, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": wl.name, "batch": sample["workload"].batch,
                       "kv_bytes_per_step": W.kv_bytes(sample)},
            "cpu_baseline": cpu,
            "e2e": {"value": round(value, 6), "unit": "TB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_gather(args, local):
    """The paged -> contiguous copy (pa_gather_kv) of one workload's whole cache: bytes read
    plus bytes written per call over the device time of K calls (two input sets alternate,
    each larger than L2), against the measured HBM copy peak."""
    import torch
    import paged_kv_cache_work_gb300 as pa
    import workloads as W
    dev = torch.device("cuda", local)
    wl = W.FULL[args.workload]
    pa.load()
    sets = [W.make_inputs(wl, W.SEEDS[0] + 7919 * k, device=dev) for k in range(2)]
    row_elems = wl.num_kv_heads * wl.head_dim
    bufs = []
    for s in sets:
        rows = int(s["context_lens"].sum().item())
        cfg = pa.config_for(s, num_ctas=1)
        k_out = torch.empty((rows, wl.num_kv_heads, wl.head_dim), dtype=s["k_cache"].dtype,
                            device=dev)
        bufs.append((s, cfg, k_out, torch.empty_like(k_out), rows,
                     torch.zeros(1, dtype=torch.int32, device=dev)))
    bytes_per = [2 * 2 * rows * row_elems * s["k_cache"].element_size()
                 for s, _, _, _, rows, _ in bufs]  # K and V, read and written
    stream = torch.cuda.current_stream(dev)

    def call(i):
        s, cfg, k_out, v_out, rows, flags = bufs[i % 2]
        pa.gather_kv(cfg, s["k_cache"], s["v_cache"], s["block_tables"], s["context_lens"],
                     k_out, v_out, rows, None, flags, stream.cuda_stream)

    for i in range(args.warmup):
        call(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        call(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    for b in bufs:
        if int(b[5].item()):
            raise RuntimeError(f"device flags {int(b[5].item())} in the gather")
    sec = e0.elapsed_time(e1) / 1e3
    total = sum(bytes_per[i % 2] for i in range(args.steps))
    gbs = total / sec / 1e9
    peak, src = measured_hbm_peak()
    return {"metric": "paged->contiguous KV gather GB/s (bytes read + written)",
            "value": round(gbs, 1), "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "us_per_call": round(sec / args.steps * 1e6, 2),
            "higher_is_better": True, "dtype": wl.kv_dtype, "data": "synthetic",
            "config": {"workload": wl.name, "kv_bytes_read_per_call": int(statistics.fmean(bytes_per) / 2),
                       "l2": "inputs larger than L2: 2 input sets alternate"},
            "roofline": {"kernel": "gather_kernel", "bound": "hbm", "achieved": round(gbs, 1),
                         "peak": peak, "unit": "GB/s", "frac": round(gbs / peak, 4),
                         "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)"
                         if src == "measured" else src}}


def main(argv=None):
    import workloads as W
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=W.BENCH.name, choices=sorted(W.FULL))
    ap.add_argument("--all", action="store_true", help="one line per workload family")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--gather", action="store_true",
                    help="time the paged -> contiguous copy (pa_gather_kv) of the workload instead")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    rank, world, local = dist_env()
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return 0
    if args.gather:
        if rank == 0:
            print(json.dumps(run_gather(args, local)), flush=True)
        return 0
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend="nccl")
    names = sorted(W.FULL) if args.all else [args.workload]
    for name in names:
        args.workload = name
        res = run_ours(args, rank, world, local)
        if res is not None:
            print(json.dumps(res), flush=True)
        if args.all:
            args.no_cpu_baseline = True
    return 0


if __name__ == "__main__":
    sys.exit(main())
