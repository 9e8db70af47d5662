"""Helpers shared by the GPU tests: run one decode step through the C ABI, compare it with
the CPU oracle under the stated tolerances, and read the planner's work list back out of
the workspace (whose layout the library documents in its internal header)."""
from __future__ import annotations

import numpy as np
import torch

import paged_kv_cache_work_gb300 as pa
import workloads

# |gpu - ref| <= ATOL + RTOL * |ref| for bf16/fp16 outputs; fp8 caches: |gpu - ref| <= 3e-2
ATOL = RTOL = 8e-3
FP8_ATOL = 3e-2
# natural-log LSE is an fp32 output: fp32 logits and sums plus the approximate exp2/log2
LSE_TOL = 2e-4


def run(inp_dev: dict, num_ctas: int = 0, grid_mult: int = 0, with_lse: bool = True,
        split_merge: int = pa.MERGE_AUTO):
    cfg = pa.config_for(inp_dev, num_ctas=num_ctas, grid_mult=grid_mult, split_merge=split_merge)
    q = inp_dev["q"]
    out = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device=q.device) \
        if with_lse else None
    ws = torch.empty(pa.workspace_size(cfg), dtype=torch.uint8, device=q.device)
    out, lse, ws = pa.paged_attention(inp_dev, out=out, lse=lse, ws=ws, cfg=cfg)
    torch.cuda.synchronize()
    return out, lse, ws, cfg


def compare(out, lse, ref_out, ref_lse, kv_dtype: str):
    """Element-wise check against the oracle; returns (max abs err of out, of lse)."""
    g = out.detach().float().cpu().numpy().astype(np.float64)
    r = np.asarray(ref_out, np.float64)
    assert g.shape == r.shape
    assert np.isfinite(g).all(), "non-finite output"
    err = np.abs(g - r)
    if kv_dtype == "fp8":
        bad = err > FP8_ATOL
    else:
        bad = err > ATOL + RTOL * np.abs(r)
    assert not bad.any(), (f"{bad.sum()} of {bad.size} outputs out of tolerance; "
                           f"max abs err {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")
    lerr = 0.0
    if lse is not None:
        gl = lse.detach().cpu().numpy().astype(np.float64)
        rl = np.asarray(ref_lse, np.float64)
        assert np.array_equal(np.isfinite(gl), np.isfinite(rl)), "lse finite pattern differs"
        assert np.array_equal(gl[~np.isfinite(rl)], rl[~np.isfinite(rl)])
        f = np.isfinite(rl)
        if f.any():
            d = np.abs(gl[f] - rl[f])
            lerr = float(d.max())
            assert (d <= LSE_TOL * (1 + np.abs(rl[f]))).all(), f"lse max err {lerr:.3e}"
    return float(err.max()), lerr


# ---- workspace view ---------------------------------------------------------------
def _pow2_at_least(x):
    p = 1
    while p < x:
        p <<= 1
    return p


SIMT_MAX_ROWS = 8
TILE_BYTES = 16384
TC_STEP_TOKENS = 64
ITEM_COST_TILES = 3
TC_ITEM_COST_STEPS = 7
TC_MIN_ROWS = 33
REDUCE_WARP_PIECES = 16


def decode_merge_limit(split_merge: int, tc: bool) -> int:
    """Most pieces of a split unit that the decode kernel merges itself (pa_split_merge);
    PA_MERGE_AUTO leaves every split unit to the reduce kernel, like PA_MERGE_IN_REDUCE."""
    if split_merge == pa.MERGE_IN_DECODE:
        return 1 << 30
    return 1


def variant(cfg: pa.PaConfig, ctas: int):
    rows = (cfg.num_q_heads // cfg.num_kv_heads) * cfg.max_q_len
    bpe = 1 if cfg.kv_dtype == pa.FP8_E4M3 else 2
    tc = cfg.head_dim >= 128 and rows >= TC_MIN_ROWS and (bpe == 2 or cfg.head_dim == 128)
    if tc:  # tcgen05
        mp = 64 if rows <= 64 else 128
    elif cfg.head_dim * bpe >= 128:  # mma.sync kernel
        mp = 64 if rows >= 64 else (16 if rows <= 16 else _pow2_at_least(rows))
    else:
        mp = _pow2_at_least(rows) if rows <= SIMT_MAX_ROWS else SIMT_MAX_ROWS
    rb = -(-rows // mp)
    tt = TC_STEP_TOKENS if tc else TILE_BYTES // (cfg.head_dim * bpe)
    cost = ITEM_COST_TILES * (TILE_BYTES // (cfg.head_dim * bpe))
    return dict(rows=rows, mp=mp, rb=rb, tt=tt, units=cfg.batch * cfg.num_kv_heads * rb,
                ctas=ctas, ns_dec=decode_merge_limit(cfg.split_merge, tc),
                item_cost=TC_ITEM_COST_STEPS * TC_STEP_TOKENS if tc else -(-cost // tt) * tt)


def layout(cfg: pa.PaConfig, v: dict):
    off = 0
    out = {}

    def take(name, nbytes):
        nonlocal off
        out[name] = off
        off = -(-(off + nbytes) // 256) * 256

    C, U = v["ctas"], v["units"]
    take("header", 64 * 4)
    take("item_off", (C + 1) * 4)
    take("first_item", C * 16)
    take("items", (C + U) * 16)
    take("unit_info", U * 8)
    take("unit_cnt", U * 4)
    take("red_units", U * 4)
    take("seq_start", (cfg.batch + 1) * 4)
    take("seq_len", cfg.batch * 4)
    take("o_part", 2 * C * v["mp"] * cfg.head_dim * 4)
    take("lse_part", 2 * C * v["mp"] * 4)
    out["total"] = off
    return out


def plan_view(ws: torch.Tensor, cfg: pa.PaConfig, ctas: int):
    """Host copy of the planner's output: header, item offsets, items, unit info, partials."""
    v = variant(cfg, ctas)
    L = layout(cfg, v)
    assert L["total"] == ws.numel(), "workspace layout mirror is out of date"
    raw = ws.cpu().numpy()

    def arr(name, dtype, count):
        return raw[L[name]:L[name] + count * np.dtype(dtype).itemsize].view(dtype)

    C, U = v["ctas"], v["units"]
    hdr = arr("header", np.int32, 64)
    item_off = arr("item_off", np.int32, C + 1)
    first_item = arr("first_item", np.int32, 4 * C).reshape(-1, 4)
    items = arr("items", np.int32, 4 * (C + U)).reshape(-1, 4)
    unit_info = arr("unit_info", np.int32, 2 * U).reshape(-1, 2)
    unit_cnt = arr("unit_cnt", np.int32, U)
    n_red = int(hdr[4])
    n_red_small = int(hdr[5])
    red_units = arr("red_units", np.int32, U)[:n_red]
    o_part = arr("o_part", np.float32, 2 * C * v["mp"] * cfg.head_dim).reshape(
        2 * C, v["mp"], cfg.head_dim)
    lse_part = arr("lse_part", np.float32, 2 * C * v["mp"]).reshape(2 * C, v["mp"])
    return dict(v=v, flags=int(hdr[0]), chunk=int(hdr[1]), active=int(hdr[2]),
                n_items=int(hdr[3]), item_off=item_off.copy(), first_item=first_item.copy(),
                items=items.copy(),
                unit_info=unit_info.copy(), unit_cnt=unit_cnt.copy(), red_units=red_units.copy(),
                n_red_small=n_red_small,
                o_part=o_part.copy(), lse_part=lse_part.copy())


def sample_rows(w: workloads.Workload, ql, n: int, seed: int):
    """n distinct (b, i, h) rows, always including the first and last valid rows."""
    rng = np.random.default_rng(seed)
    rows = {(0, 0, 0), (w.batch - 1, int(ql[-1]) - 1, w.num_q_heads - 1)}
    n = min(n, int(sum(max(1, int(x)) for x in ql)) * w.num_q_heads)  # distinct rows that exist
    while len(rows) < n:
        b = int(rng.integers(w.batch))
        rows.add((b, int(rng.integers(max(1, int(ql[b])))), int(rng.integers(w.num_q_heads))))
    return np.array(sorted(rows), np.int32)
