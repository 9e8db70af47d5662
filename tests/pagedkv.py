"""Test helpers: build paged problems from contiguous per-sequence K/V, and brute-force
attention over the contiguous data in numpy float64 (scipy's softmax/logsumexp).

The brute force never looks at pages: the helper scatters each sequence's contiguous
rows into a shuffled pool through its block table, and whatever reads the pool must
gather them back through the same table to agree with it.
"""
from __future__ import annotations

import math

import numpy as np
import scipy.special
import torch

from workloads import Workload

GARBAGE = 1.0e3  # value of pool rows no sequence owns; reading one changes the answer


def decode_stored(t: torch.Tensor, kv_dtype: str) -> np.ndarray:
    """Stored values as float64 through torch's own dtype conversions."""
    if kv_dtype == "fp8":
        return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return t.to(torch.float64).numpy()


def random_problem(rng: np.random.Generator, *, batch, max_q_len, num_q_heads, num_kv_heads,
                   head_dim, block_size, ctx, q_lens=None, causal=False, q_dtype="bf16",
                   kv_dtype="bf16", scale_mode="none", sm_scale=None, extra_blocks=3):
    """A seeded problem with contiguous per-sequence K/V scattered into a shuffled pool.

    Returns (inp, contiguous) where inp has the keys of workloads.make_inputs and
    contiguous holds, per sequence, the float64 dequantised K and V rows [n, Hkv, D]."""
    B, Sq, Hq, Hkv, D, bs = batch, max_q_len, num_q_heads, num_kv_heads, head_dim, block_size
    ctx = list(ctx)
    ql = list(q_lens) if q_lens is not None else [min(Sq, n) for n in ctx]
    pages = [(n + bs - 1) // bs for n in ctx]
    pool = sum(pages) + extra_blocks
    perm = rng.permutation(pool)
    max_blocks = max(1, max(pages))
    bt = np.full((B, max_blocks), -1, np.int32)
    off = 0
    for b, p in enumerate(pages):
        bt[b, :p] = perm[off:off + p]
        off += p
    qdt = {"bf16": torch.bfloat16, "fp16": torch.float16}[q_dtype]
    q = torch.from_numpy(rng.standard_normal((B, Sq, Hq, D))).to(qdt)

    kf = np.full((pool, bs, Hkv, D), GARBAGE)
    vf = np.full((pool, bs, Hkv, D), -GARBAGE)
    seq_k = [rng.standard_normal((n, Hkv, D)) for n in ctx]
    seq_v = [rng.standard_normal((n, Hkv, D)) for n in ctx]
    for b, n in enumerate(ctx):
        for j in range(n):
            kf[bt[b, j // bs], j % bs] = seq_k[b][j]
            vf[bt[b, j // bs], j % bs] = seq_v[b][j]
    k_scale = v_scale = None
    if kv_dtype == "fp8":
        kt, vt = torch.from_numpy(kf), torch.from_numpy(vf)
        if scale_mode == "tensor":
            ks = (kt.abs().amax() / 448.0).float().reshape(1)
            vs = (vt.abs().amax() / 448.0).float().reshape(1)
            kc = (kt / ks.double()).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
            vc = (vt / vs.double()).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
        elif scale_mode == "token":
            ks = (kt.abs().amax(-1) / 448.0).float()
            vs = (vt.abs().amax(-1) / 448.0).float()
            kc = (kt / ks.double()[..., None]).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
            vc = (vt / vs.double()[..., None]).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
        else:
            ks = vs = None
            kc = kt.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
            vc = vt.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
        k_cache, v_cache, k_scale, v_scale = kc.contiguous(), vc.contiguous(), ks, vs
    else:
        kdt = {"bf16": torch.bfloat16, "fp16": torch.float16}[kv_dtype]
        k_cache = torch.from_numpy(kf).to(kdt)
        v_cache = torch.from_numpy(vf).to(kdt)

    # dequantised contiguous view, read back from the stored bytes (not from seq_k)
    kd = decode_stored(k_cache, kv_dtype)
    vd = decode_stored(v_cache, kv_dtype)
    if k_scale is not None:
        ksd = k_scale.double().numpy()
        vsd = v_scale.double().numpy()
        if scale_mode == "token":
            kd = kd * ksd[..., None]
            vd = vd * vsd[..., None]
        else:
            kd = kd * ksd[0]
            vd = vd * vsd[0]
    contiguous = []
    for b, n in enumerate(ctx):
        # the scatter above put row j of sequence b at (bt[b, j // bs], j % bs)
        idx_blk = np.array([bt[b, j // bs] for j in range(n)], dtype=np.int64)
        idx_slot = np.array([j % bs for j in range(n)], dtype=np.int64)
        contiguous.append((kd[idx_blk, idx_slot], vd[idx_blk, idx_slot]))

    w = Workload(name="random", batch=B, max_q_len=Sq, num_q_heads=Hq, num_kv_heads=Hkv,
                 head_dim=D, block_size=bs, ctx_lo=min(ctx), ctx_hi=max(ctx), causal=causal,
                 q_dtype=q_dtype, kv_dtype=kv_dtype, scale_mode=scale_mode)
    inp = dict(workload=w, seed=None, q=q, k_cache=k_cache, v_cache=v_cache, k_scale=k_scale,
               v_scale=v_scale, block_tables=torch.from_numpy(bt),
               context_lens=torch.tensor(ctx, dtype=torch.int32),
               q_lens=torch.tensor(ql, dtype=torch.int32),
               sm_scale=(1.0 / math.sqrt(D)) if sm_scale is None else sm_scale)
    return inp, contiguous


def brute_force(inp: dict, contiguous) -> tuple:
    """float64 softmax attention over each sequence's contiguous K/V rows."""
    w = inp["workload"]
    B, Sq, Hq, Hkv, D = w.batch, w.max_q_len, w.num_q_heads, w.num_kv_heads, w.head_dim
    G = Hq // Hkv
    q = inp["q"].to(torch.float64).numpy()
    sm = float(np.float32(inp["sm_scale"]))
    out = np.zeros((B, Sq, Hq, D))
    lse = np.full((B, Sq, Hq), -np.inf)
    for b in range(B):
        n = int(inp["context_lens"][b])
        ql = int(inp["q_lens"][b])
        K, V = contiguous[b]
        for i in range(ql):
            L = n - ql + i + 1 if w.causal else n
            for h in range(Hq):
                kv = h // G
                s = sm * (K[:L, kv, :] @ q[b, i, h])
                lse[b, i, h] = scipy.special.logsumexp(s)
                out[b, i, h] = scipy.special.softmax(s) @ V[:L, kv, :]
    return out, lse
