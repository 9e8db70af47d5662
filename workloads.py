"""Seeded synthetic workloads for paged-attention decode.

This module only draws inputs: query tensors, paged K/V pools, block tables,
context lengths and (for an fp8 cache) the quantisation scales.  It holds none
of the attention arithmetic, so the CPU oracle under ``oracle/`` and the CUDA
path can both be fed from it without sharing any of the method's code.

Shapes follow the decode problems the pages study:

* "Benchmark high-perf Paged Attention (#899) vs PA unroll on a2a3" (simpler
  issue 998, Same-Shape Side-by-Side table): b1 h16 kv1 bs128 hd128 bf16 at
  context 128 and 512.
* "HSTU Paged Attention" K/V double buffering (RecSDK issue 1281, test
  method): H=16, D=256, page size 32, seeds 2026/2029/2039.
* "Optimize paged-attention metadata decode" (FlyDSL PR #910, Summary and
  Performance): block size 1024, 16 query heads, one KV head, D=128, fp8 KV
  with per-token or per-tensor scales.

The batched-GQA and long-context problems widen those to many sequences.

Conventions (each a reading of something the pages leave open):

* ``context_lens[b]`` counts every cached token of sequence b, including its
  ``q_lens[b]`` new tokens, which are the last ``q_lens[b]`` positions.
* Query head h reads KV head ``h // (Hq // Hkv)``.
* The physical pool holds twice the pages the batch needs (8 pages for the
  one-sequence problem); block tables are drawn without replacement from a
  seeded shuffle of the pool.  Table entries past a sequence's last page are -1.
* fp8 values are OCP E4M3 ("e4m3fn").  A per-tensor scale is amax/448 over the
  whole pool, separately for K and V; a per-token scale is amax/448 over one
  (block, slot, kv-head) row, or 1 where that row is all zero.  Codes come from
  torch's round-to-nearest-even cast of value/scale clamped to +-448.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

SEEDS = (2026, 2029, 2039)

DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16}


@dataclasses.dataclass(frozen=True)
class Workload:
    """One decode problem family; sizes are drawn per seed by :func:`make_inputs`."""

    name: str
    batch: int
    max_q_len: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    ctx_lo: int
    ctx_hi: int
    causal: bool = False
    q_dtype: str = "bf16"
    kv_dtype: str = "bf16"          # "bf16" | "fp16" | "fp8"
    scale_mode: str = "none"        # "none" | "tensor" | "token"
    pool_blocks: Optional[int] = None  # None: 2x the pages the batch needs

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def rows_per_kv_head(self) -> int:
        return self.group * self.max_q_len

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _wl(name, **kw) -> Workload:
    return Workload(name=name, **kw)


# The five decode problem families, at full size.
TINY_CTX128 = _wl("tiny_b1_h16_kv1_d128_bs128_ctx128", batch=1, max_q_len=1, num_q_heads=16,
                  num_kv_heads=1, head_dim=128, block_size=128, ctx_lo=128, ctx_hi=128,
                  pool_blocks=8)
TINY_CTX512 = TINY_CTX128.replace(name="tiny_b1_h16_kv1_d128_bs128_ctx512", ctx_lo=512, ctx_hi=512)
GQA_B32 = _wl("gqa_b32_h32_kv8_d128_bs16", batch=32, max_q_len=1, num_q_heads=32,
              num_kv_heads=8, head_dim=128, block_size=16, ctx_lo=512, ctx_hi=4096)
LONG_SQ1 = _wl("long_b4_h16_kv1_d128_bs1024_sq1", batch=4, max_q_len=1, num_q_heads=16,
               num_kv_heads=1, head_dim=128, block_size=1024, ctx_lo=32768, ctx_hi=131072,
               causal=True)
LONG_SQ4 = LONG_SQ1.replace(name="long_b4_h16_kv1_d128_bs1024_sq4", max_q_len=4)
FP8_TENSOR_SQ1 = _wl("fp8tensor_b64_h16_kv1_d128_bs1024_sq1", batch=64, max_q_len=1,
                     num_q_heads=16, num_kv_heads=1, head_dim=128, block_size=1024,
                     ctx_lo=8192, ctx_hi=16384, kv_dtype="fp8", scale_mode="tensor")
FP8_TENSOR_SQ4 = FP8_TENSOR_SQ1.replace(name="fp8tensor_b64_h16_kv1_d128_bs1024_sq4", max_q_len=4)
FP8_TOKEN_SQ1 = FP8_TENSOR_SQ1.replace(name="fp8token_b64_h16_kv1_d128_bs1024_sq1",
                                       scale_mode="token")
FP8_TOKEN_SQ4 = FP8_TOKEN_SQ1.replace(name="fp8token_b64_h16_kv1_d128_bs1024_sq4", max_q_len=4)


def mha_d256(batch: int, sq: int) -> Workload:
    return _wl(f"mha_b{batch}_h16_kv16_d256_bs32_sq{sq}", batch=batch, max_q_len=sq,
               num_q_heads=16, num_kv_heads=16, head_dim=256, block_size=32, ctx_lo=2048,
               ctx_hi=16384, causal=True)


MHA_D256 = [mha_d256(b, sq) for b in (8, 32) for sq in (1, 4, 16, 64)]

FULL = {w.name: w for w in [TINY_CTX128, TINY_CTX512, GQA_B32, LONG_SQ1, LONG_SQ4,
                            FP8_TENSOR_SQ1, FP8_TENSOR_SQ4, FP8_TOKEN_SQ1, FP8_TOKEN_SQ4,
                            *MHA_D256]}

# The largest problem that fits one GPU (about 4.7 GB of KV): the bench's headline workload.
BENCH = FULL["mha_b32_h16_kv16_d256_bs32_sq64"]


def reduced(w: Workload, batch: int, ctx_lo: int, ctx_hi: int) -> Workload:
    """The same head/page/dtype structure at a size the CPU oracle finishes in seconds."""
    return w.replace(name=f"{w.name}__b{batch}_ctx{ctx_lo}-{ctx_hi}", batch=batch,
                     ctx_lo=ctx_lo, ctx_hi=ctx_hi)


def _generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, g, device, chunk_elems=1 << 27):
    """Standard normal fp32, drawn in slabs along dim 0 to bound the temporary."""
    out = torch.empty(shape, dtype=torch.float32, device=device)
    flat = out.view(shape[0], -1)
    per_row = flat.shape[1]
    rows = max(1, chunk_elems // max(per_row, 1))
    for r0 in range(0, shape[0], rows):
        r1 = min(shape[0], r0 + rows)
        flat[r0:r1] = torch.randn((r1 - r0, per_row), generator=g, device=device)
    return out


def _quantise_e4m3(x: torch.Tensor, scale: torch.Tensor) -> torch.Tensor:
    """Codes of x/scale as OCP E4M3 bytes (RNE via torch's cast, clamped to +-448)."""
    y = torch.clamp(x / scale, -448.0, 448.0)
    return y.to(torch.float8_e4m3fn).view(torch.uint8)


def make_inputs(w: Workload, seed: int, device="cpu", context_lens=None, q_lens=None) -> dict:
    """Draw one seeded problem of family ``w``.

    Returns a dict of tensors on ``device``:
      q            [B, Sq, Hq, D]         bf16/fp16
      k_cache      [nb, bs, Hkv, D]       bf16/fp16, or uint8 E4M3 codes
      v_cache      [nb, bs, Hkv, D]
      k_scale      None | [1] fp32 | [nb, bs, Hkv] fp32
      v_scale      same as k_scale
      block_tables [B, max_blocks] int32  (-1 past a sequence's last page)
      context_lens [B] int32, q_lens [B] int32
    plus the python scalars sm_scale and the workload itself.
    ``context_lens``/``q_lens`` override the drawn lengths (edge-case tests).
    """
    dev = torch.device(device)
    g = _generator(seed, dev)
    B, Sq, Hq, Hkv, D, bs = (w.batch, w.max_q_len, w.num_q_heads, w.num_kv_heads,
                             w.head_dim, w.block_size)
    if context_lens is None:
        ctx = torch.randint(w.ctx_lo, w.ctx_hi + 1, (B,), generator=g, device=dev)
        ctx = ctx.to(torch.int32)
    else:
        ctx = torch.as_tensor(context_lens, dtype=torch.int32, device=dev)
    if q_lens is None:
        ql = torch.full((B,), Sq, dtype=torch.int32, device=dev)
    else:
        ql = torch.as_tensor(q_lens, dtype=torch.int32, device=dev)
    ctx_host = ctx.cpu().tolist()
    pages = [(n + bs - 1) // bs for n in ctx_host]
    needed = sum(pages)
    pool = w.pool_blocks if w.pool_blocks is not None else max(1, 2 * needed)
    if pool < needed:
        raise ValueError(f"pool of {pool} blocks cannot hold {needed} pages")
    max_blocks = max(1, max(pages) if pages else 1, -(-w.ctx_hi // bs))
    perm = torch.randperm(pool, generator=g, device=dev).to(torch.int32)
    bt = torch.full((B, max_blocks), -1, dtype=torch.int32, device=dev)
    off = 0
    for b, p in enumerate(pages):
        bt[b, :p] = perm[off:off + p]
        off += p

    qt = DTYPES[w.q_dtype]
    q = _randn((B, Sq, Hq, D), g, dev).to(qt)
    kf = _randn((pool, bs, Hkv, D), g, dev)
    vf = _randn((pool, bs, Hkv, D), g, dev)
    k_scale = v_scale = None
    if w.kv_dtype == "fp8":
        if w.scale_mode == "tensor":
            k_scale = (kf.abs().amax() / 448.0).reshape(1).float()
            v_scale = (vf.abs().amax() / 448.0).reshape(1).float()
            kc = _quantise_e4m3(kf, k_scale)
            vc = _quantise_e4m3(vf, v_scale)
        elif w.scale_mode == "token":
            ka = kf.abs().amax(dim=-1) / 448.0
            va = vf.abs().amax(dim=-1) / 448.0
            k_scale = torch.where(ka > 0, ka, torch.ones_like(ka)).contiguous()
            v_scale = torch.where(va > 0, va, torch.ones_like(va)).contiguous()
            kc = _quantise_e4m3(kf, k_scale[..., None])
            vc = _quantise_e4m3(vf, v_scale[..., None])
        else:
            one = torch.ones((), device=dev)
            kc = _quantise_e4m3(kf, one)
            vc = _quantise_e4m3(vf, one)
        k_cache, v_cache = kc.contiguous(), vc.contiguous()
    else:
        kt = DTYPES[w.kv_dtype]
        k_cache, v_cache = kf.to(kt), vf.to(kt)
    del kf, vf
    return dict(workload=w, seed=seed, q=q, k_cache=k_cache, v_cache=v_cache,
                k_scale=k_scale, v_scale=v_scale, block_tables=bt, context_lens=ctx,
                q_lens=ql, sm_scale=1.0 / math.sqrt(D))


def kv_bytes(inp: dict) -> int:
    """Algorithmic bytes one decode call must read: every valid token's K and V row for
    every KV head, plus its two fp32 scales in per-token mode.  Page-tail padding,
    queries, tables and outputs are not counted."""
    w: Workload = inp["workload"]
    tokens = int(inp["context_lens"].to(torch.int64).sum().item())
    bpe = 1 if w.kv_dtype == "fp8" else 2
    per = w.num_kv_heads * 2 * w.head_dim * bpe
    if w.kv_dtype == "fp8" and w.scale_mode == "token":
        per += w.num_kv_heads * 8
    return tokens * per


def to_device(inp: dict, device) -> dict:
    out = {}
    for k, v in inp.items():
        out[k] = v.to(device) if isinstance(v, torch.Tensor) else v
    return out
