"""Per-shape grid multiplier: an offline tuner under CUDA-graph replay and its lookup table.

The decode's persistent grid is SMs x grid_mult x (decode CTAs resident per SM).  With
multiplier 1 the whole grid is one wave; with a larger one the planner cuts the token space
into proportionally more, smaller pieces and the GPU starts the later CTAs as earlier ones
finish, which trades more split units (and merges) for a shorter tail of unequal CTA end
times.  Which side wins depends on the shape, the device and the scale mode (the grid
multiplier of the AMD paged-attention metadata change, "[Kernel][Perf] Optimize
paged-attention metadata decode", Changes section: SMs x multiplier, default 1).

`tune()` times one plan + decode + reduce step under CUDA-graph replay for each candidate
multiplier and keeps the fastest one only when it beats multiplier 1 by more than
`min_gain`; `python -m paged_kv_cache_work_gb300.grid_tune` writes the table for the
repository's synthetic workloads.  `lookup()` reads the table (`grid_mult.csv` beside this
file): a row matches the problem's shape key and the device's SM count, and anything
without a row keeps multiplier 1.  `config_for` applies it when the caller gives neither a
grid size nor a multiplier.
"""
from __future__ import annotations

import csv
import os
from typing import Dict, Iterable, List, Optional, Sequence, Tuple

TABLE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "grid_mult.csv")
KEY_FIELDS = ("batch", "max_q_len", "num_q_heads", "num_kv_heads", "head_dim", "block_size",
              "kv_dtype", "kv_scale_mode", "sms")
COLUMNS = KEY_FIELDS + ("grid_mult", "us_per_step", "us_mult1", "workload")

_cache: Dict[str, Dict[Tuple[int, ...], int]] = {}


def shape_key(cfg, sms: int) -> Tuple[int, ...]:
    """The fields of a pa_config (and the device) a tuned multiplier is valid for."""
    return (int(cfg.batch), int(cfg.max_q_len), int(cfg.num_q_heads), int(cfg.num_kv_heads),
            int(cfg.head_dim), int(cfg.block_size), int(cfg.kv_dtype), int(cfg.kv_scale_mode),
            int(sms))


def read_table(path: str = TABLE) -> Dict[Tuple[int, ...], int]:
    """{shape key: multiplier} of a table file; empty when the file does not exist."""
    if path in _cache:
        return _cache[path]
    table: Dict[Tuple[int, ...], int] = {}
    if os.path.exists(path):
        with open(path, newline="") as f:
            for row in csv.DictReader(f):
                key = tuple(int(row[k]) for k in KEY_FIELDS)
                mult = int(row["grid_mult"])
                if mult < 1:
                    raise ValueError(f"{path}: grid_mult {mult} < 1 for {key}")
                table[key] = mult
    _cache[path] = table
    return table


def lookup(cfg, sms: int, path: str = TABLE) -> int:
    """Tuned multiplier for this shape on a device with `sms` SMs, else 1."""
    return read_table(path).get(shape_key(cfg, sms), 1)


def write_table(rows: Iterable[dict], path: str = TABLE) -> None:
    rows = sorted(rows, key=lambda r: tuple(int(r[k]) for k in KEY_FIELDS))
    with open(path, "w", newline="") as f:
        w = csv.DictWriter(f, fieldnames=COLUMNS, lineterminator="\n")
        w.writeheader()
        for r in rows:
            w.writerow({c: r[c] for c in COLUMNS})
    _cache.pop(path, None)


def choose(times: Dict[int, float], min_gain: float) -> int:
    """The multiplier to keep: the fastest, unless it beats multiplier 1 by no more than
    `min_gain` (a fraction), in which case 1."""
    best = min(times, key=lambda m: (times[m], m))
    if best != 1 and times[best] > times[1] * (1.0 - min_gain):
        return 1
    return best


def time_step(sets: Sequence[dict], mult: int, replays: int = 100, warmup: int = 5) -> float:
    """Mean device time (us) of one plan + decode + reduce step at grid multiplier `mult`: a
    CUDA graph of one step on each input set (the sets alternate, so no step finds its
    cache in L2 when each set is larger than L2) is replayed and its time divided by the
    number of sets."""
    import torch
    import paged_kv_cache_work_gb300 as pa
    dev = sets[0]["q"].device
    bufs = []
    for inp in sets:
        cfg = pa.config_for(inp, grid_mult=mult)
        q = inp["q"]
        bufs.append((inp, cfg, torch.empty_like(q),
                     torch.empty(q.shape[:3], dtype=torch.float32, device=dev),
                     torch.empty(pa.workspace_size(cfg), dtype=torch.uint8, device=dev)))
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        for inp, cfg, out, lse, ws in bufs:
            pa.paged_attention(inp, out=out, lse=lse, ws=ws, cfg=cfg, stream=s)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            for inp, cfg, out, lse, ws in bufs:
                pa.paged_attention(inp, out=out, lse=lse, ws=ws, cfg=cfg, stream=s)
        for _ in range(warmup):
            graph.replay()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(replays):
            graph.replay()
        e1.record(s)
    torch.cuda.synchronize(dev)
    for _, _, _, _, ws in bufs:
        flags = pa.read_flags(ws)
        if flags:
            raise RuntimeError(f"device flags {flags} while tuning")
    return e0.elapsed_time(e1) * 1e3 / (replays * len(bufs))


def tune(problems: Sequence[Tuple[str, Sequence[dict]]], mults: Sequence[int] = (1, 2, 3, 4),
         min_gain: float = 0.02, replays: int = 100) -> List[dict]:
    """One table row per (name, input sets on the GPU): the step time at each multiplier and
    the multiplier kept (see choose)."""
    import torch
    import paged_kv_cache_work_gb300 as pa
    if 1 not in mults:
        raise ValueError("multiplier 1 is the baseline and must be timed")
    rows = []
    for name, sets in problems:
        dev = sets[0]["q"].device
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        times = {m: time_step(sets, m, replays=replays) for m in mults}
        keep = choose(times, min_gain)
        row = dict(zip(KEY_FIELDS, shape_key(pa.config_for(sets[0], grid_mult=1), sms)))
        row.update(grid_mult=keep, us_per_step=round(times[keep], 2),
                   us_mult1=round(times[1], 2), workload=name)
        rows.append(row)
        print(f"{name:42s} " + " ".join(f"x{m}: {t:8.2f} us" for m, t in sorted(times.items()))
              + f"  -> x{keep}", flush=True)
    return rows


def main(argv: Optional[Sequence[str]] = None) -> None:
    import argparse
    import sys
    import torch
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if root not in sys.path:
        sys.path.insert(0, root)
    import workloads as W
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--workload", action="append", help="workload name (default: all full-size)")
    ap.add_argument("--mults", default="1,2,3,4")
    ap.add_argument("--min-gain", type=float, default=0.02)
    ap.add_argument("--replays", type=int, default=100)
    ap.add_argument("--out", default=TABLE)
    args = ap.parse_args(argv)
    names = args.workload or [n for n in W.FULL if not n.startswith("tiny")]
    dev = torch.device("cuda:0")
    mults = [int(m) for m in args.mults.split(",")]
    rows = []
    for n in names:  # two input sets per workload, freed before the next workload
        sets = [W.make_inputs(W.FULL[n], W.SEEDS[0] + 7919 * k, device=dev) for k in range(2)]
        rows += tune([(n, sets)], mults, args.min_gain, args.replays)
        del sets
        torch.cuda.empty_cache()
    write_table(rows, args.out)
    print(f"wrote {len(rows)} rows to {args.out}")


if __name__ == "__main__":
    main()
