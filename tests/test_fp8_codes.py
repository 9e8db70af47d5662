"""Every E4M3 code through the decode kernels' fp8 widening (GPU).

With one key in a sequence's context the softmax weight of that key is exactly 1, so each
output element is the key's value in that dimension: its E4M3 code decoded and times the V
scale (every finite E4M3 value times a power of two is exact in bf16).  Four sequences hold
all 256 codes in their key row, the codes of each aligned group of 16 dimensions in their
natural order for the first two sequences and with the group's two halves of 8 swapped for
the last two, so that every code meets both halves of a 16-byte chunk, the unit the kernels
widen by (a chunk's first eight codes make the low 16 bytes of its f16 row, the last eight
the high ones).  The kernel's output must equal the oracle's bit for bit, and a NaN code
must give NaN in its own dimension and nowhere else.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_run import run

pytestmark = pytest.mark.gpu

D = 128


def code_rows() -> np.ndarray:
    """[4, D] uint8: the value row of each sequence's single key."""
    d = np.arange(D)
    return np.stack([d, 128 + d, d ^ 8, 128 + (d ^ 8)]).astype(np.uint8)


def problem(num_q_heads: int, scale_mode: str) -> dict:
    """Four sequences of one key and one query row per head, one kv head, pages of 16."""
    B, bs = 4, 16
    wl = W.Workload(name=f"codes_h{num_q_heads}_{scale_mode}", batch=B, max_q_len=1,
                    num_q_heads=num_q_heads, num_kv_heads=1, head_dim=D, block_size=bs,
                    ctx_lo=1, ctx_hi=1, kv_dtype="fp8", scale_mode=scale_mode)
    pool = B + 2
    g = torch.Generator().manual_seed(1234)
    # pages hold codes that must not be read past each sequence's one key
    k_cache = torch.full((pool, bs, 1, D), 0x3C, dtype=torch.uint8)  # 1.5
    v_cache = torch.full((pool, bs, 1, D), 0x7E, dtype=torch.uint8)  # 448
    pages = [3, 0, 5, 1]
    rows = torch.from_numpy(code_rows())
    for b, pg in enumerate(pages):
        k_cache[pg, 0, 0] = torch.randint(0, 256, (D,), generator=g).to(torch.uint8) & 0x77
        v_cache[pg, 0, 0] = rows[b]
    bt = torch.tensor(pages, dtype=torch.int32).reshape(B, 1)
    k_scale = v_scale = None
    if scale_mode == "tensor":
        k_scale = torch.tensor([0.5], dtype=torch.float32)
        v_scale = torch.tensor([0.125], dtype=torch.float32)
    elif scale_mode == "token":
        k_scale = torch.full((pool, bs, 1), 2.0, dtype=torch.float32)
        v_scale = torch.full((pool, bs, 1), 0.25, dtype=torch.float32)
        v_scale[pages[2], 0, 0] = 4.0
    q = torch.randn((B, 1, num_q_heads, D), generator=g).to(torch.bfloat16)
    return dict(workload=wl, seed=0, q=q, k_cache=k_cache, v_cache=v_cache, k_scale=k_scale,
                v_scale=v_scale, block_tables=bt,
                context_lens=torch.ones(B, dtype=torch.int32),
                q_lens=torch.ones(B, dtype=torch.int32), sm_scale=D ** -0.5)


# 64 query rows per kv head go to the tcgen05 kernel, 16 to the mma.sync kernel
CASES = [(64, "none"), (64, "tensor"), (64, "token"), (16, "none"), (16, "token")]


@pytest.mark.parametrize("heads,scale_mode", CASES, ids=[f"h{h}_{m}" for h, m in CASES])
def test_every_code_widens_exactly(heads, scale_mode, cuda_device, pa):
    inp = problem(heads, scale_mode)
    ref, _ = oracle.decode(inp, "f64")
    out, _, ws, _ = run(W.to_device(inp, cuda_device))
    assert pa.read_flags(ws) == 0
    got = out.float().cpu().numpy()
    want = torch.from_numpy(np.ascontiguousarray(ref)).to(torch.bfloat16).float().numpy()
    nan_want = np.isnan(want)
    assert nan_want.sum() == 4 * heads, "two NaN codes per sequence row"
    assert np.array_equal(np.isnan(got), nan_want), "NaN outside a NaN code's dimension"
    ok = ~nan_want
    bad = np.nonzero(got[ok] != want[ok])[0]
    assert bad.size == 0, f"{bad.size} elements differ, e.g. {got[ok][bad[:4]]} vs {want[ok][bad[:4]]}"


def shaped_queries(q: torch.Tensor, seed: int) -> torch.Tensor:
    """Query rows whose magnitudes stress a kernel that rescales and splits a row: elements
    spread over six orders of magnitude, an all-zero row, a row of large values, a row of
    tiny ones (subnormal in fp16), and a row with one outlier; the rest N(0, 1)."""
    g = torch.Generator().manual_seed(seed)
    B, Sq, Hq, D_ = q.shape
    x = torch.randn((B, Sq, Hq, D_), generator=g, dtype=torch.float64)
    kind = torch.arange(B * Sq * Hq).reshape(B, Sq, Hq) % 6
    spread = 10.0 ** (torch.rand((B, Sq, Hq, D_), generator=g, dtype=torch.float64) * 6 - 3)
    x = torch.where((kind == 0)[..., None], x * spread, x)
    x = torch.where((kind == 1)[..., None], torch.zeros_like(x), x)
    x = torch.where((kind == 2)[..., None], x * 30.0, x)
    x = torch.where((kind == 3)[..., None], x * 1e-5, x)
    outlier = torch.zeros_like(x)
    outlier[..., 7] = 300.0
    x = torch.where((kind == 4)[..., None], x + outlier, x)
    return x.to(q.dtype)


RANGE_CASES = [("tcgen05", 16, "bf16", "tensor"), ("tcgen05", 16, "fp16", "token"),
               ("tcgen05", 16, "fp16", "none"), ("mma", 4, "fp16", "tensor")]


@pytest.mark.parametrize("kernel,heads,q_dtype,scale_mode", RANGE_CASES,
                         ids=[f"{k}_{q}_{m}" for k, _, q, m in RANGE_CASES])
def test_query_dynamic_range(kernel, heads, q_dtype, scale_mode, cuda_device, pa):
    """Rows of very different magnitudes against an fp8 cache, compared with the oracle at
    the fp8 tolerance (64 query rows per kv head take the tcgen05 kernel, 16 the mma.sync
    one)."""
    from pagedkv import random_problem
    from gpu_run import compare
    rng = np.random.default_rng(77 + heads)
    inp, _ = random_problem(rng, batch=3, max_q_len=4, num_q_heads=heads, num_kv_heads=1,
                            head_dim=D, block_size=64, ctx=[300, 77, 700], q_dtype=q_dtype,
                            kv_dtype="fp8", scale_mode=scale_mode, causal=True)
    inp["q"] = shaped_queries(inp["q"], 5)
    ref_out, ref_lse = oracle.decode(inp, "f32")
    out, lse, ws, _ = run(W.to_device(inp, cuda_device))
    assert pa.read_flags(ws) == 0
    compare(out, lse, ref_out, ref_lse, "fp8")
