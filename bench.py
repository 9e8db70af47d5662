"""Throughput of one paged-attention decode step on GB300, as one JSON line.

A step is the whole hot path on one batch: pa_plan + pa_decode + pa_reduce (three kernel
launches) through the C ABI, inputs resident in HBM.  The headline workload is the largest
of the decode problems that fits one GPU: B=32 sequences, 16 query heads over 16 KV heads,
head dim 256, pages of 32 tokens, 64 new tokens per sequence (causal among them), context
lengths uniform in [2048, 16384], bf16, pool = 2x the pages needed (about 4.7 GB of KV).

value      = KV bytes read per step (every valid token's K and V rows; no padding,
             queries, tables or outputs) / device time per step, in TB/s, summed over
             ranks and divided by the slowest rank's time (weak scaling: each rank decodes
             its own batch, no collective on the data path).
e2e        = the same through the public Python binding with host buffers: every step
             copies q, block tables and lengths from pinned host memory and reads out and
             lse back, inside the timed region, on two copy streams that overlap the
             neighbouring steps as a decode loop would.  The KV cache is device state.
roofline   = the decode kernel alone: algorithmic bytes / average launch time of back-to-back
             decode launches (CUDA events around the batch), against the measured HBM copy
             peak; `frac_spec` is the same against the 8 TB/s HBM3e specification; the time
             of launches bracketed one by one (with a launch gap each) is given beside it.
per_config = every decode problem family at full size: step and decode-kernel times, TB/s,
             fractions of the measured peak and of the specification, the kernel used.
gather     = the paged -> contiguous KV copy (pa_gather_kv) of the headline workload.
cpu_baseline / --impl reference = the CPU oracle (fp32 C, OpenMP) on the host cores, on a
             sample of the same inputs (the same generator, the same seeds).

L2: two independent input sets of > 2x L2 bytes each alternate between steps, so no step
finds its KV in L2.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload NAME] [--no-per-config] [--no-cpu-baseline]
For N > 1 launch with torchrun (one process per GPU).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
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
SPEC_HBM_GBS = 8000.0  # GB300 HBM3e specification, the roofline the decode is quoted against
TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SOURCES = ["paged_kv_cache_work_gb300/csrc/decode_simt.cuh",
                  "paged_kv_cache_work_gb300/csrc/decode_tc.cuh",
                  "paged_kv_cache_work_gb300/csrc/decode_mma.cuh",
                  "paged_kv_cache_work_gb300/csrc/decode_common.cuh",
                  "paged_kv_cache_work_gb300/csrc/pa_internal.cuh"]
PER_CONFIG_MIN_STEPS = 100


def decode_shape(wl):
    """(decode kernel name, rows per unit) the library picks for a workload: a 16-bit cache
    with head dim 128 or 256, or an fp8 cache with head dim 128, and more than 32 query rows
    per kv head goes to the tcgen05 kernel in tiles of 64 or 128 rows; other caches with a
    tile row of at least 128 bytes to the mma.sync kernel in tiles of 16, 32 or 64 rows; the
    rest (64-dim fp8) to the CUDA-core kernel."""
    rows = (wl.num_q_heads // wl.num_kv_heads) * wl.max_q_len
    bpe = 1 if wl.kv_dtype == "fp8" else 2
    pow2 = 1 << max(0, (rows - 1).bit_length())
    if wl.head_dim >= 128 and rows >= 33 and (bpe == 2 or wl.head_dim == 128):
        return "decode_tc_kernel", 64 if rows <= 64 else 128
    if wl.head_dim * bpe >= 128:
        return "decode_mma_kernel", 64 if rows >= 64 else max(16, pow2)
    return "decode_simt_kernel", min(pow2, 8)


def launches_per_step(split_merge: int) -> int:
    """Kernels one plan/decode/reduce step launches: pa_reduce launches its kernel unless
    every split unit is merged inside the decode (PA_MERGE_IN_DECODE)."""
    import paged_kv_cache_work_gb300 as pa
    return 2 if split_merge == pa.MERGE_IN_DECODE else 3


def compute_dtype(wl) -> str:
    """The arithmetic type of the path: 16-bit MMA operands (bf16, or f16 for fp16 and fp8
    caches) with fp32 accumulation and softmax."""
    return "bf16" if wl.kv_dtype == "bf16" else "fp16"


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
    """DRAM bytes (read + written) per decode launch of this workload from the committed ncu
    record (profiles/traffic.json), or (None, None) when there is none or the kernel sources
    changed since it was taken."""
    try:
        with open(TRAFFIC_RECORD) as f:
            records = json.load(f)["records"]
    except (OSError, KeyError, ValueError):
        return None, None
    src = kernel_source_hash()
    for r in records:
        if r.get("workload") == workload and r.get("kernel_source_sha256") == src:
            return (float(r["dram_bytes_read_per_launch"]) + float(r["dram_bytes_write_per_launch"]),
                    r.get("summary"))
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


# ------------------------------------------------------------------------- inputs
def input_device():
    """Where the seeded inputs are drawn: on the GPU when there is one (both arms of the
    bench then see the same values: the generator is the CUDA one), else on the CPU."""
    import torch
    return torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() \
        else torch.device("cpu")


def draw_sets(wl, seed: int, device):
    """The two alternating input sets of a workload (seeds seed and seed + 7919)."""
    import workloads as W
    return [W.make_inputs(wl, seed + 7919 * k, device=device) for k in range(2)]


def workload_config(wl, kv_bytes_per_step: float, l2_bytes: int, world: int) -> dict:
    """The `config` object of the JSON line, identical for both arms."""
    return {
        "workload": wl.name, "batch": wl.batch, "num_q_heads": wl.num_q_heads,
        "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim,
        "block_size": wl.block_size, "context_lens": f"U[{wl.ctx_lo},{wl.ctx_hi}]",
        "max_q_len": wl.max_q_len, "causal": bool(wl.causal), "q_dtype": wl.q_dtype,
        "kv_dtype": wl.kv_dtype, "scale_mode": wl.scale_mode,
        "kv_bytes_per_step": int(kv_bytes_per_step),
        "l2": (f"inputs larger than L2: 2 input sets of {int(kv_bytes_per_step) >> 20} MiB KV "
               f"alternate (L2 {l2_bytes >> 20} MiB)"),
        "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
    }


def l2_size() -> int:
    import torch
    if not torch.cuda.is_available():
        return 0
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    return int(getattr(props, "L2_cache_size", 0) or 0)


def compact_sample(inp, seqs):
    """The chosen sequences of a problem with only their own pages, on the host: the same
    attention problem with renumbered block tables."""
    import torch
    w = inp["workload"]
    bs = w.block_size
    ctx = inp["context_lens"].cpu()
    bt = inp["block_tables"].cpu()
    ids, tables = [], []
    for b in seqs:
        pages = (int(ctx[b]) + bs - 1) // bs
        tables.append(list(range(len(ids), len(ids) + pages)))
        ids.extend(bt[b, :pages].tolist())
    dev = inp["k_cache"].device
    idx = torch.tensor(ids, dtype=torch.long, device=dev)
    maxb = max(1, max(len(t) for t in tables))
    new_bt = torch.full((len(seqs), maxb), -1, dtype=torch.int32)
    for k, t in enumerate(tables):
        new_bt[k, :len(t)] = torch.tensor(t, dtype=torch.int32)
    sel = torch.tensor(seqs, dtype=torch.long, device=inp["q"].device)
    ks, vs = inp.get("k_scale"), inp.get("v_scale")
    if ks is not None and ks.dim() > 1:
        ks, vs = ks[idx], vs[idx]
    return dict(workload=w.replace(batch=len(seqs)), seed=inp.get("seed"),
                q=inp["q"][sel].cpu(), k_cache=inp["k_cache"][idx].cpu(),
                v_cache=inp["v_cache"][idx].cpu(),
                k_scale=None if ks is None else ks.cpu(), v_scale=None if vs is None else vs.cpu(),
                block_tables=new_bt, context_lens=ctx[seqs].clone(),
                q_lens=inp["q_lens"].cpu()[seqs].clone(), sm_scale=inp["sm_scale"])


# ------------------------------------------------------------------------ CPU oracle leg
def oracle_sample(inp, max_seconds_per_call: float):
    """The first n sequences of the problem (compacted onto the host) whose oracle call takes
    about max_seconds_per_call; returns (sample, description)."""
    import oracle
    B = inp["workload"].batch
    one = compact_sample(inp, [0])
    t = time.perf_counter()
    oracle.decode(one, "f32")
    per_seq = max(time.perf_counter() - t, 1e-6)
    n = max(1, min(B, int(max_seconds_per_call / per_seq)))
    if n == 1:
        return one, f"the first of {B} sequences"
    desc = f"the whole batch ({B} sequences)" if n >= B else f"the first {n} of {B} sequences"
    return compact_sample(inp, list(range(n))), desc


def time_oracle(sample, budget_s: float, max_calls: int = 1000):
    """Median seconds per oracle call over as many calls as fit in budget_s (at least 1)."""
    import oracle
    times = []
    t_end = time.perf_counter() + budget_s
    while len(times) < max_calls:
        t = time.perf_counter()
        oracle.decode(sample, "f32")
        times.append(time.perf_counter() - t)
        if time.perf_counter() > t_end:
            break
    return statistics.median(times), len(times)


# ------------------------------------------------------------------------- GPU leg
class Bench:
    """Two input sets of one workload on the device, their workspaces and the CUDA graphs of
    their steps."""

    def __init__(self, wl, seed, dev):
        import torch
        import paged_kv_cache_work_gb300 as pa
        import workloads as W
        self.wl, self.dev = wl, dev
        self.sets = draw_sets(wl, seed, dev)
        self.step_bytes = [W.kv_bytes(s) for s in self.sets]
        for s in self.sets:
            s["out"] = torch.empty_like(s["q"])
            s["lse"] = torch.empty(s["q"].shape[:3], dtype=torch.float32, device=dev)
            s["cfg"] = pa.config_for(s)
            s["ws"] = torch.empty(pa.workspace_size(s["cfg"]), dtype=torch.uint8, device=dev)
        self.cfg = self.sets[0]["cfg"]
        self.stream = torch.cuda.current_stream(dev)
        self.graphs = []

    def step(self, s, stream=None):
        import paged_kv_cache_work_gb300 as pa
        sh = (stream or self.stream).cuda_stream
        c = s["cfg"]
        pa.plan(c, s["block_tables"], s["context_lens"], s["q_lens"], s["ws"], sh)
        self.decode(s, stream)
        pa.reduce(c, s["out"], s["lse"], s["ws"], sh)

    def decode(self, s, stream=None):
        import paged_kv_cache_work_gb300 as pa
        sh = (stream or self.stream).cuda_stream
        pa.decode(s["cfg"], s["q"], s["k_cache"], s["v_cache"], s["k_scale"], s["v_scale"],
                  s["block_tables"], s["context_lens"], s["q_lens"], s["out"], s["lse"],
                  s["ws"], sh)

    def warm(self, warmup):
        import torch
        import paged_kv_cache_work_gb300 as pa
        for k in range(warmup):
            self.step(self.sets[k % 2])
        torch.cuda.synchronize(self.dev)
        for s in self.sets:
            if pa.read_flags(s["ws"]) != 0:
                raise RuntimeError(f"device flags set on the {self.wl.name} inputs")
        # one CUDA graph per input set holds the step's launches, so the timed loop measures
        # the device and not the Python launch path
        cap = torch.cuda.Stream(self.dev)
        cap.wait_stream(self.stream)
        for s in self.sets:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(cap):
                with torch.cuda.graph(g, stream=cap):
                    self.step(s, cap)
            self.graphs.append(g)
        self.stream.wait_stream(cap)
        for k in range(max(3, warmup)):
            self.graphs[k % 2].replay()
        torch.cuda.synchronize(self.dev)

    def time_steps(self, n):
        """(device seconds of n graph replays, KV bytes they read)."""
        import torch
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        total = 0
        start.record(self.stream)
        for k in range(n):
            self.graphs[k % 2].replay()
            total += self.step_bytes[k % 2]
        stop.record(self.stream)
        torch.cuda.synchronize(self.dev)
        return start.elapsed_time(stop) / 1e3, total

    def time_decodes(self, n):
        """Milliseconds of each of n decode launches bracketed one by one (CUDA events on the
        launching stream; the host enqueues faster than the kernels run, so each pair brackets
        one kernel).  The event between two launches stops the next decode from starting
        before the previous one has ended, so these include a launch gap per kernel."""
        import torch
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        for k in range(n):
            evs[k][0].record(self.stream)
            self.decode(self.sets[k % 2])
            evs[k][1].record(self.stream)
        torch.cuda.synchronize(self.dev)
        return [a.elapsed_time(b) for a, b in evs[min(4, n - 1):]]

    def time_decode_stream(self, n):
        """Average milliseconds per decode over n back-to-back decode launches between one pair
        of CUDA events (two input sets alternating): every launch does the whole decode, and a
        launch's set-up overlaps the end of the previous one, as in a decode loop."""
        import torch
        for k in range(4):
            self.decode(self.sets[k % 2])
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        for k in range(n):
            self.decode(self.sets[k % 2])
        e1.record(self.stream)
        torch.cuda.synchronize(self.dev)
        return e0.elapsed_time(e1) / n

    def roofline(self, decode_ms, peak, peak_kind, stream_ms=None):
        """The decode kernel's roofline: algorithmic bytes over its average launch duration,
        taken from back-to-back launches when given (stream_ms), else from the one-by-one
        brackets."""
        mean_s = (stream_ms if stream_ms is not None else statistics.fmean(decode_ms)) / 1e3
        achieved = statistics.fmean(self.step_bytes) / mean_s / 1e9
        return {"kernel": decode_shape(self.wl)[0], "bound": "hbm",
                "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "peak_source": (f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                                if peak_kind == "measured" else "fallback 6.8 TB/s"),
                "frac_spec": round(achieved / SPEC_HBM_GBS, 4),
                "spec_gbs": SPEC_HBM_GBS,
                "decode_us_mean": round(mean_s * 1e6, 2),
                "decode_timing": ("back-to-back launches, CUDA events around the batch"
                                  if stream_ms is not None else "one launch per event pair"),
                "decode_us_isolated_mean": round(statistics.fmean(decode_ms) * 1e3, 2),
                "decode_us_isolated_median": round(statistics.median(decode_ms) * 1e3, 2),
                # each input set's algorithmic bytes (launches alternate the sets, set 0
                # first: odd-numbered launches read set 0), to hold a profiled launch against
                "kv_bytes_per_set": [int(x) for x in self.step_bytes]}


def measure_config(wl, dev, seed, steps, warmup, peak, peak_kind):
    """One per_config entry: graph-replayed steps and decode-only launches of a workload."""
    b = Bench(wl, seed, dev)
    b.warm(warmup)
    n = max(steps, PER_CONFIG_MIN_STEPS)
    sec, nbytes = b.time_steps(n)
    dec = b.time_decodes(max(8, n))
    roof = b.roofline(dec, peak, peak_kind, b.time_decode_stream(n))
    step_s = sec / n
    entry = {"kernel": roof["kernel"], "q_dtype": wl.q_dtype, "kv_dtype": wl.kv_dtype,
             "scale_mode": wl.scale_mode, "kv_bytes_per_step": int(statistics.fmean(b.step_bytes)),
             "kv_bytes_per_set": [int(x) for x in b.step_bytes],
             "steps": n, "step_us": round(step_s * 1e6, 2),
             "step_tbs": round(nbytes / sec / 1e12, 4),
             "step_frac": round(nbytes / sec / 1e9 / peak, 4),
             "step_frac_spec": round(nbytes / sec / 1e9 / SPEC_HBM_GBS, 4),
             "decode_us": roof["decode_us_mean"],
             "decode_us_isolated": roof["decode_us_isolated_mean"],
             "decode_tbs": round(roof["achieved"] / 1e3, 4),
             "frac": roof["frac"], "frac_spec": roof["frac_spec"]}
    return entry


def run_gather(b, dev, n, peak, peak_kind):
    """pa_gather_kv of the headline workload's first input set: bytes read + written per call
    over the device time of n calls (the cache is larger than L2)."""
    import torch
    import paged_kv_cache_work_gb300 as pa
    s = b.sets[0]
    wl = b.wl
    rows = int(s["context_lens"].sum().item())
    cfg = pa.config_for(s, num_ctas=1)
    k_out = torch.empty((rows, wl.num_kv_heads, wl.head_dim), dtype=s["k_cache"].dtype, device=dev)
    v_out = torch.empty_like(k_out)
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    nbytes = 2 * 2 * k_out.numel() * k_out.element_size()  # K and V, read and written
    st = b.stream

    def call():
        pa.gather_kv(cfg, s["k_cache"], s["v_cache"], s["block_tables"], s["context_lens"],
                     k_out, v_out, rows, None, flags, st.cuda_stream)

    for _ in range(3):
        call()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(n):
        call()
    e1.record(st)
    torch.cuda.synchronize(dev)
    if int(flags.item()):
        raise RuntimeError(f"device flags {int(flags.item())} in the gather")
    sec = e0.elapsed_time(e1) / 1e3 / n
    gbs = nbytes / sec / 1e9
    del k_out, v_out
    return {"kernel": "gather_kernel", "workload": wl.name, "bytes_per_call": nbytes,
            "us_per_call": round(sec * 1e6, 2), "achieved": round(gbs, 1), "unit": "GB/s",
            "frac": round(gbs / peak, 4), "frac_spec": round(gbs / SPEC_HBM_GBS, 4),
            "calls": n, "peak_source": peak_kind}


def run_ours(args, rank, world, local):
    import torch
    import paged_kv_cache_work_gb300 as pa
    import workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = W.FULL[args.workload]
    pa.load()
    peak, peak_kind = measured_hbm_peak()
    seed = W.SEEDS[0] + rank
    b = Bench(wl, seed, dev)
    b.warm(args.warmup)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.25)
    barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    seconds, total_bytes = b.time_steps(args.steps)
    barrier()
    max_s, all_bytes = aggregate(seconds, total_bytes)
    dec = b.time_decodes(max(8, min(max(args.steps, 200), 2000)))
    dec_stream = b.time_decode_stream(max(8, min(max(args.steps, 200), 2000)))
    clocks = sampler.stop(t_wall0, time.time())

    # end to end through the binding with host buffers
    n_e2e = max(1, min(args.steps, 200))
    host = []
    for s in b.sets:
        hs = {k: s[k].cpu().pin_memory() for k in ("q", "block_tables", "context_lens", "q_lens")}
        hs["out"] = torch.empty(s["out"].shape, dtype=s["out"].dtype).pin_memory()
        hs["lse"] = torch.empty(s["lse"].shape, dtype=torch.float32).pin_memory()
        host.append(hs)
    h2d = sum(host[0][k].numel() * host[0][k].element_size()
              for k in ("q", "block_tables", "context_lens", "q_lens"))
    d2h = sum(host[0][k].numel() * host[0][k].element_size() for k in ("out", "lse"))

    # A decode loop's copies: step k's inputs go up on one copy stream while step k - 1
    # computes, and its outputs come down on another while step k + 1 computes.  The two
    # input sets double-buffer the device side: set i's inputs are overwritten only after
    # the step that read them has finished, and its outputs only after they reached the host.
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    computed = [torch.cuda.Event() for _ in range(2)]
    fetched = [torch.cuda.Event() for _ in range(2)]
    for i in range(2):
        computed[i].record(b.stream)
        fetched[i].record(b.stream)

    def e2e_step(k):
        i = k % 2
        s, hs = b.sets[i], host[i]
        arrived = torch.cuda.Event()
        with torch.cuda.stream(up):
            up.wait_event(computed[i])  # the step that last read set i is done with it
            for key in ("q", "block_tables", "context_lens", "q_lens"):
                s[key].copy_(hs[key], non_blocking=True)
            arrived.record(up)
        b.stream.wait_event(arrived)
        b.stream.wait_event(fetched[i])  # set i's last outputs have reached the host
        b.step(s)
        computed[i].record(b.stream)
        with torch.cuda.stream(down):
            down.wait_event(computed[i])
            hs["out"].copy_(s["out"], non_blocking=True)
            hs["lse"].copy_(s["lse"], non_blocking=True)
            fetched[i].record(down)

    for k in range(3):
        e2e_step(k)
    torch.cuda.synchronize(dev)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_bytes = 0
    e0.record(b.stream)
    up.wait_event(e0)
    down.wait_event(e0)
    for k in range(n_e2e):
        e2e_step(k)
        e2e_bytes += b.step_bytes[k % 2]
    b.stream.wait_stream(down)  # the last outputs are on the host when the clock stops
    e1.record(b.stream)
    torch.cuda.synchronize(dev)
    e2e_s, e2e_all = aggregate(e0.elapsed_time(e1) / 1e3, e2e_bytes)
    del host

    result = None
    if rank == 0:
        roof = b.roofline(dec, peak, peak_kind, dec_stream)
        traffic, traffic_src = profiled_traffic(wl.name)
        roof["traffic"] = traffic
        roof["traffic_source"] = traffic_src
        value = all_bytes / max_s / 1e12
        per_step_s = max_s / args.steps
        result = {
            "metric": METRIC, "value": round(value, 4), "unit": "TB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(per_step_s * 1e3, 5),
            "us_per_call": round(per_step_s * 1e6, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": compute_dtype(wl), "data": "synthetic",
            "config": workload_config(wl, statistics.fmean(b.step_bytes), l2_size(), world),
            "launch": {"grid_mult": int(b.cfg.grid_mult) or 1,
                       "split_merge": "auto (the reduce kernel merges every split unit)",
                       "timing": "device time of K CUDA-graph replays of the step (plan, "
                                 "decode, reduce)"},
            "roofline": roof,
            "e2e": {"value": round(e2e_all / e2e_s / 1e12, 4), "unit": "TB/s",
                    "us_per_call": round(e2e_s / n_e2e * 1e6, 2), "steps": n_e2e,
                    "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                    "timing": ("each step's inputs up from pinned host memory and its out/lse "
                               "down, on two copy streams that overlap the neighbouring steps "
                               "(the two input sets double-buffer the device side); every "
                               "step's copies are inside the timed region")},
            "gpu_launches": launches_per_step(b.cfg.split_merge) * args.steps,
            "clocks": clocks,
        }
        if not args.no_gather:
            result["gather"] = run_gather(b, dev, 10, peak, peak_kind)
        if not args.no_cpu_baseline:
            sample, desc = oracle_sample(b.sets[0], 2.0)
            sec, calls = time_oracle(sample, 12.0)
            import oracle
            result["cpu_baseline"] = {
                "value": round(W.kv_bytes(sample) / sec / 1e12, 6), "unit": "TB/s",
                "us_per_call": round(sec * 1e6, 1), "cores": oracle.threads(), "kind": "oracle",
                "sample": f"{desc} of the bench workload's first input set, median of {calls} calls"}
    del b
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_per_config:
        per = {}
        for name in W.FULL:
            per[name] = measure_config(W.FULL[name], dev, seed, args.steps, args.warmup, peak,
                                       peak_kind)
            torch.cuda.empty_cache()
        result["per_config"] = per
    return result


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm: the same workload, the same seeded inputs (drawn
    with the same generator as the GPU arm), timed on a bounded sample of whole sequences."""
    if rank != 0:
        return None
    import statistics as st
    import oracle
    import workloads as W
    wl = W.FULL[args.workload]
    sets = draw_sets(wl, W.SEEDS[0], input_device())
    mean_bytes = st.fmean(W.kv_bytes(s) for s in sets)
    per_step_budget = max(0.02, 120.0 / max(1, args.steps + args.warmup))
    sample, desc = oracle_sample(sets[0], per_step_budget)
    del sets
    for _ in range(args.warmup):
        oracle.decode(sample, "f32")
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle.decode(sample, "f32")
    sec = (time.perf_counter() - t) / max(1, args.steps)
    value = W.kv_bytes(sample) / sec / 1e12
    cpu = {"value": round(value, 6), "unit": "TB/s", "cores": oracle.threads(), "kind": "oracle",
           "sample": f"{desc} of {wl.name}'s first input set per step"}
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(sec * 1e3, 3), "us_per_call": round(sec * 1e6, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": compute_dtype(wl), "data": "synthetic",
            "config": workload_config(wl, mean_bytes, l2_size(), world),
            "cpu_baseline": cpu,
            "e2e": {"value": round(value, 6), "unit": "TB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main(argv=None):
    import workloads as W
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=W.BENCH.name, choices=sorted(W.FULL))
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only the headline workload")
    ap.add_argument("--no-gather", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    rank, world, local = dist_env()
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return 0
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend="nccl")
    res = run_ours(args, rank, world, local)
    if res is not None:
        print(json.dumps(res), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
