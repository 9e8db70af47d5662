"""GPU parity: the CUDA path through the C ABI against the CPU oracle (fp32 build) on the
same seeded inputs, element by element.

* every problem family at a size the oracle finishes in seconds, still spanning several
  tiles and a ragged tail, for the three seeds 2026/2029/2039;
* every problem family at full size in the bench's launch configuration, on sampled rows;
* edge cases: ragged and empty query lengths, context = new tokens, one-token contexts,
  one CTA, far more CTAs than work, every page size, fp16, head dim 64, no LSE output.

Tolerances: |gpu - ref| <= 8e-3 + 8e-3 |ref| for bf16/fp16 outputs and <= 3e-2 for an fp8
cache (against the oracle on the same dequantised values); natural-log LSE within
2e-4 (1 + |ref|).
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_run import compare, run, sample_rows
from pagedkv import random_problem

pytestmark = pytest.mark.gpu

W = workloads
REDUCED = [
    W.TINY_CTX128,
    W.TINY_CTX512,
    W.reduced(W.GQA_B32, 5, 300, 1400),
    W.reduced(W.LONG_SQ1, 2, 2500, 6000),
    W.reduced(W.LONG_SQ4, 2, 2500, 6000),
    W.reduced(W.FP8_TENSOR_SQ1, 3, 1100, 3000),
    W.reduced(W.FP8_TENSOR_SQ4, 3, 1100, 3000),
    W.reduced(W.FP8_TOKEN_SQ1, 3, 1100, 3000),
    W.reduced(W.FP8_TOKEN_SQ4, 3, 1100, 3000),
    *[W.reduced(w, 2, 200, 1300) for w in W.MHA_D256 if w.batch == 8],
]


@pytest.mark.parametrize("seed", W.SEEDS)
@pytest.mark.parametrize("wl", REDUCED, ids=lambda w: w.name)
def test_reduced_problem_matches_oracle(wl, seed, cuda_device, pa):
    inp = W.make_inputs(wl, seed)
    ref_out, ref_lse = oracle.decode(inp, "f32")
    out, lse, _, _ = run(W.to_device(inp, cuda_device))
    err, lerr = compare(out, lse, ref_out, ref_lse, wl.kv_dtype)
    print(f"{wl.name} seed {seed}: max abs err {err:.3e}, lse {lerr:.3e}")


def _compact(inp_dev, seqs):
    """The chosen sequences with only their own pages, moved to the host: the same
    attention problem (block tables renamed with the pages)."""
    w = inp_dev["workload"]
    bs = w.block_size
    ctx = inp_dev["context_lens"].cpu()
    bt = inp_dev["block_tables"].cpu()
    ids, tables = [], []
    for b in seqs:
        pages = (int(ctx[b]) + bs - 1) // bs
        tables.append(list(range(len(ids), len(ids) + pages)))
        ids.extend(bt[b, :pages].tolist())
    idx = torch.tensor(ids, dtype=torch.long, device=inp_dev["k_cache"].device)
    maxb = max(len(t) for t in tables)
    new_bt = torch.full((len(seqs), maxb), -1, dtype=torch.int32)
    for k, t in enumerate(tables):
        new_bt[k, :len(t)] = torch.tensor(t, dtype=torch.int32)
    sel = torch.tensor(seqs, dtype=torch.long, device=inp_dev["q"].device)
    ks, vs = inp_dev.get("k_scale"), inp_dev.get("v_scale")
    if ks is not None and ks.dim() > 1:
        ks, vs = ks[idx], vs[idx]
    out = dict(workload=w.replace(batch=len(seqs)), seed=inp_dev["seed"],
               q=inp_dev["q"][sel].cpu(), k_cache=inp_dev["k_cache"][idx].cpu(),
               v_cache=inp_dev["v_cache"][idx].cpu(),
               k_scale=None if ks is None else ks.cpu(), v_scale=None if vs is None else vs.cpu(),
               block_tables=new_bt, context_lens=ctx[seqs].clone(),
               q_lens=inp_dev["q_lens"].cpu()[seqs].clone(), sm_scale=inp_dev["sm_scale"])
    return out


@pytest.mark.slow
@pytest.mark.parametrize("wl", list(W.FULL.values()), ids=lambda w: w.name)
def test_full_size_sampled_rows_match_oracle(wl, cuda_device, pa):
    seed = W.SEEDS[0]
    inp = W.make_inputs(wl, seed, device=cuda_device)
    out, lse, _, _ = run(inp)
    assert torch.isfinite(out).all()
    ql = inp["q_lens"].cpu().numpy()
    rng = np.random.default_rng(seed)
    seqs = sorted({0, wl.batch - 1, *rng.choice(wl.batch, size=min(wl.batch, 4), replace=False)})
    small = _compact(inp, seqs)
    rows = sample_rows(small["workload"], ql[seqs], 48, seed)
    ref_out, ref_lse = oracle.decode_rows(small, rows, "f32")
    gb = np.array(seqs)[rows[:, 0]]
    g_out = out[torch.as_tensor(gb), torch.as_tensor(rows[:, 1]), torch.as_tensor(rows[:, 2])]
    g_lse = lse[torch.as_tensor(gb), torch.as_tensor(rows[:, 1]), torch.as_tensor(rows[:, 2])]
    err, lerr = compare(g_out, g_lse, ref_out, ref_lse, wl.kv_dtype)
    print(f"{wl.name} (full size, {len(rows)} rows): max abs err {err:.3e}, lse {lerr:.3e}")


# ------------------------------------------------------------------ edge cases
EDGE = [
    # name, kwargs for random_problem
    ("ragged_q_lens_causal", dict(batch=4, max_q_len=4, num_q_heads=8, num_kv_heads=2,
                                  head_dim=128, block_size=16, ctx=[70, 4, 33, 200],
                                  q_lens=[4, 1, 3, 2], causal=True)),
    ("ctx_equals_new_tokens", dict(batch=3, max_q_len=8, num_q_heads=4, num_kv_heads=4,
                                   head_dim=128, block_size=32, ctx=[8, 8, 5], q_lens=[8, 8, 5],
                                   causal=True)),
    ("one_token_contexts", dict(batch=5, max_q_len=1, num_q_heads=4, num_kv_heads=1,
                                head_dim=128, block_size=16, ctx=[1, 1, 2, 1, 3])),
    ("empty_sequence", dict(batch=3, max_q_len=2, num_q_heads=4, num_kv_heads=2, head_dim=64,
                            block_size=16, ctx=[0, 40, 0], q_lens=[0, 2, 0], causal=True)),
    ("fp16", dict(batch=3, max_q_len=1, num_q_heads=8, num_kv_heads=2, head_dim=128,
                  block_size=64, ctx=[500, 129, 1000], q_dtype="fp16", kv_dtype="fp16")),
    ("head_dim_64", dict(batch=3, max_q_len=2, num_q_heads=6, num_kv_heads=3, head_dim=64,
                         block_size=128, ctx=[300, 700, 1029], causal=True)),
    ("fp8_fp16_query", dict(batch=2, max_q_len=1, num_q_heads=4, num_kv_heads=4, head_dim=256,
                            block_size=32, ctx=[300, 611], q_dtype="fp16", kv_dtype="fp8",
                            scale_mode="token")),
    ("fp8_unscaled", dict(batch=2, max_q_len=2, num_q_heads=2, num_kv_heads=1, head_dim=128,
                          block_size=256, ctx=[300, 900], kv_dtype="fp8", scale_mode="none")),
    ("gqa8_sq1_rows8", dict(batch=2, max_q_len=1, num_q_heads=16, num_kv_heads=2, head_dim=128,
                            block_size=16, ctx=[257, 900])),
    ("rows_3_padded", dict(batch=2, max_q_len=3, num_q_heads=2, num_kv_heads=2, head_dim=256,
                           block_size=32, ctx=[100, 64], causal=True)),
    # mma.sync kernel: row tiles of 16, 32 and 64
    ("mma_rows12_padded", dict(batch=3, max_q_len=1, num_q_heads=24, num_kv_heads=2,
                               head_dim=128, block_size=16, ctx=[77, 300, 16])),
    ("d256_rows100", dict(batch=2, max_q_len=4, num_q_heads=25, num_kv_heads=1,
                                        head_dim=256, block_size=64, ctx=[200, 517],
                                        causal=True)),
    ("mma_fp16_rows32", dict(batch=2, max_q_len=2, num_q_heads=16, num_kv_heads=1, head_dim=128,
                             block_size=32, ctx=[150, 333], q_dtype="fp16", kv_dtype="fp16",
                             causal=True)),
    ("mma_d64_rows32", dict(batch=2, max_q_len=4, num_q_heads=8, num_kv_heads=1, head_dim=64,
                            block_size=128, ctx=[130, 700], causal=True)),
    ("mma_fp8_d256_rows16", dict(batch=2, max_q_len=16, num_q_heads=2, num_kv_heads=2,
                                 head_dim=256, block_size=32, ctx=[40, 300], kv_dtype="fp8",
                                 scale_mode="token", causal=True)),
    ("mma_d64_fp16_rows64", dict(batch=2, max_q_len=4, num_q_heads=16, num_kv_heads=1,
                                 head_dim=64, block_size=256, ctx=[260, 1000], q_dtype="fp16",
                                 kv_dtype="fp16", causal=True)),
    ("mma_fp8_fp16q_rows32", dict(batch=2, max_q_len=2, num_q_heads=16, num_kv_heads=1,
                                  head_dim=128, block_size=16, ctx=[99, 180], q_dtype="fp16",
                                  kv_dtype="fp8", scale_mode="none")),
    # per-token fp8 scales on mma.sync (up to 32 rows per kv head)
    ("mma_fp8_token_fp16q_rows32", dict(batch=3, max_q_len=2, num_q_heads=16, num_kv_heads=1,
                                        head_dim=128, block_size=16, ctx=[129, 70, 640],
                                        q_dtype="fp16", kv_dtype="fp8", scale_mode="token",
                                        causal=True)),
    ("mma_fp8_token_rows16_long_pages", dict(batch=2, max_q_len=1, num_q_heads=16,
                                             num_kv_heads=1, head_dim=128, block_size=1024,
                                             ctx=[1500, 2049], kv_dtype="fp8",
                                             scale_mode="token", causal=True)),
    ("mma_d64_fp8_stays_on_cuda_cores", dict(batch=2, max_q_len=1, num_q_heads=16,
                                             num_kv_heads=1, head_dim=64, block_size=16,
                                             ctx=[70, 130], kv_dtype="fp8", scale_mode="token")),
]


@pytest.mark.parametrize("name,kw", EDGE, ids=[e[0] for e in EDGE])
def test_edge_cases(name, kw, cuda_device, pa):
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    inp, _ = random_problem(rng, **kw)
    ref_out, ref_lse = oracle.decode(inp, "f32")
    dev = W.to_device(inp, cuda_device)
    out, lse, ws, _ = run(dev)
    compare(out, lse, ref_out, ref_lse, kw.get("kv_dtype", "bf16"))
    assert pa.read_flags(ws) == 0


# The tcgen05 kernel: 16-bit caches with head dim 128 or 256 and fp8 caches with head dim 128
# (per-tensor, per-token or no scales), more than 32 query rows per kv head (tiles of 64 or
# 128 rows, MMA always 128 rows; 64-row tiles of head dim 128 run as two token streams).
TC = [
    ("fp8_token_fp16q_rows64", dict(batch=3, max_q_len=4, num_q_heads=16, num_kv_heads=1,
                                    block_size=16, ctx=[129, 70, 640], q_dtype="fp16",
                                    kv_dtype="fp8", scale_mode="token", causal=True)),
    ("fp8_token_rows100_tile128", dict(batch=2, max_q_len=4, num_q_heads=25, num_kv_heads=1,
                                       block_size=1024, ctx=[1500, 2049], kv_dtype="fp8",
                                       scale_mode="token", causal=True)),
    ("fp8_token_rows40_partial", dict(batch=3, max_q_len=5, num_q_heads=8, num_kv_heads=1,
                                      block_size=32, ctx=[5, 191, 64], kv_dtype="fp8",
                                      scale_mode="token", causal=True)),
    ("fp8_token_two_kv_heads_ragged", dict(batch=4, max_q_len=4, num_q_heads=32,
                                           num_kv_heads=2, block_size=64, ctx=[0, 4, 300, 65],
                                           q_lens=[0, 4, 1, 3], kv_dtype="fp8",
                                           scale_mode="token", causal=True)),
    ("fp8_token_long_pages_not_causal", dict(batch=2, max_q_len=4, num_q_heads=16,
                                             num_kv_heads=1, block_size=1024, ctx=[3000, 1025],
                                             kv_dtype="fp8", scale_mode="token")),
    ("rows33_padded_causal", dict(batch=3, max_q_len=3, num_q_heads=11, num_kv_heads=1,
                                  block_size=16, ctx=[70, 300, 129], causal=True)),
    ("rows64_long_pages", dict(batch=2, max_q_len=4, num_q_heads=16, num_kv_heads=1,
                               block_size=1024, ctx=[1500, 2049], causal=True)),
    ("rows100_tile128", dict(batch=2, max_q_len=4, num_q_heads=25, num_kv_heads=1,
                             block_size=64, ctx=[200, 517], causal=True)),
    ("rows200_two_tiles", dict(batch=2, max_q_len=4, num_q_heads=100, num_kv_heads=2,
                               block_size=32, ctx=[333, 64], causal=True)),
    ("fp16_rows48", dict(batch=3, max_q_len=3, num_q_heads=32, num_kv_heads=2, block_size=128,
                         ctx=[77, 1000, 256], q_dtype="fp16", kv_dtype="fp16", causal=True)),
    ("fp8_tensor_rows64", dict(batch=2, max_q_len=4, num_q_heads=16, num_kv_heads=1,
                               block_size=256, ctx=[260, 1000], kv_dtype="fp8",
                               scale_mode="tensor", causal=True)),
    ("fp8_tensor_fp16q_rows64", dict(batch=3, max_q_len=4, num_q_heads=16, num_kv_heads=1,
                                     block_size=16, ctx=[129, 70, 640], q_dtype="fp16",
                                     kv_dtype="fp8", scale_mode="tensor", causal=True)),
    ("fp8_none_rows40_partial", dict(batch=2, max_q_len=5, num_q_heads=8, num_kv_heads=1,
                                     block_size=32, ctx=[5, 191], kv_dtype="fp8",
                                     scale_mode="none", causal=True)),
    ("fp8_none_rows100_tile128", dict(batch=2, max_q_len=4, num_q_heads=25, num_kv_heads=1,
                                      block_size=64, ctx=[200, 517], kv_dtype="fp8",
                                      scale_mode="none", causal=True)),
    ("fp8_tensor_rows200_two_tiles", dict(batch=2, max_q_len=4, num_q_heads=100,
                                          num_kv_heads=2, block_size=32, ctx=[333, 64],
                                          kv_dtype="fp8", scale_mode="tensor", causal=True)),
    ("fp8_tensor_long_pages", dict(batch=2, max_q_len=4, num_q_heads=16, num_kv_heads=1,
                                   block_size=1024, ctx=[1500, 2049], kv_dtype="fp8",
                                   scale_mode="tensor", causal=True)),
    ("ragged_and_empty", dict(batch=4, max_q_len=4, num_q_heads=16, num_kv_heads=1,
                              block_size=16, ctx=[0, 4, 63, 65], q_lens=[0, 4, 1, 3],
                              causal=True)),
    ("not_causal_tiny", dict(batch=2, max_q_len=2, num_q_heads=24, num_kv_heads=1,
                             block_size=16, ctx=[1, 3])),
    ("d256_rows64_causal", dict(head_dim=256, batch=3, max_q_len=64, num_q_heads=2,
                                num_kv_heads=2, block_size=32, ctx=[64, 300, 1029], causal=True)),
    ("d256_fp16_rows100_bs16", dict(head_dim=256, batch=2, max_q_len=4, num_q_heads=25,
                                    num_kv_heads=1, block_size=16, ctx=[200, 77], q_dtype="fp16",
                                    kv_dtype="fp16", causal=True)),
    ("d256_rows256_two_tiles", dict(head_dim=256, batch=2, max_q_len=16, num_q_heads=16,
                                    num_kv_heads=1, block_size=64, ctx=[300, 40], causal=True)),
]


@pytest.mark.parametrize("ctas", [0, 3, 40])
@pytest.mark.parametrize("name,kw", TC, ids=[c[0] for c in TC])
def test_tcgen05_kernel(name, kw, ctas, cuda_device, pa):
    rng = np.random.default_rng(zlib.crc32(name.encode()) + ctas)
    inp, _ = random_problem(rng, **{"head_dim": 128, **kw})
    ref_out, ref_lse = oracle.decode(inp, "f32")
    out, lse, ws, _ = run(W.to_device(inp, cuda_device), num_ctas=ctas)
    compare(out, lse, ref_out, ref_lse, kw.get("kv_dtype", "bf16"))
    assert pa.read_flags(ws) == 0


# The CUDA-core kernel serves caches whose rows are shorter than one 128-byte slab: 64-dim fp8.
CUDA_CORE = [
    ("rows1_tensor", dict(batch=3, max_q_len=1, num_q_heads=4, num_kv_heads=4, block_size=16,
                          ctx=[300, 17, 1200], scale_mode="tensor")),
    ("rows2_token_causal", dict(batch=2, max_q_len=2, num_q_heads=2, num_kv_heads=2,
                                block_size=32, ctx=[129, 640], scale_mode="token", causal=True)),
    ("rows4_none", dict(batch=4, max_q_len=1, num_q_heads=8, num_kv_heads=2, block_size=64,
                        ctx=[1, 64, 65, 2000], scale_mode="none")),
    ("rows8_fp16q", dict(batch=2, max_q_len=2, num_q_heads=8, num_kv_heads=2, block_size=128,
                         ctx=[700, 260], scale_mode="token", q_dtype="fp16", causal=True)),
    ("rows12_two_tiles", dict(batch=2, max_q_len=3, num_q_heads=4, num_kv_heads=1,
                              block_size=16, ctx=[90, 333], q_lens=[3, 2], scale_mode="tensor",
                              causal=True)),
    ("empty_and_ragged", dict(batch=3, max_q_len=4, num_q_heads=2, num_kv_heads=1,
                              block_size=16, ctx=[0, 5, 77], q_lens=[0, 4, 1],
                              scale_mode="token", causal=True)),
]


@pytest.mark.parametrize("ctas", [0, 5])
@pytest.mark.parametrize("name,kw", CUDA_CORE, ids=[c[0] for c in CUDA_CORE])
def test_cuda_core_kernel(name, kw, ctas, cuda_device, pa):
    rng = np.random.default_rng(zlib.crc32(name.encode()) + ctas)
    inp, _ = random_problem(rng, head_dim=64, kv_dtype="fp8", **kw)
    ref_out, ref_lse = oracle.decode(inp, "f32")
    for sm in (pa.MERGE_AUTO, pa.MERGE_IN_DECODE, pa.MERGE_IN_REDUCE):
        out, lse, ws, _ = run(W.to_device(inp, cuda_device), num_ctas=ctas, split_merge=sm)
        compare(out, lse, ref_out, ref_lse, "fp8")
        assert pa.read_flags(ws) == 0


@pytest.mark.parametrize("bs", [16, 32, 64, 128, 256, 512, 1024])
def test_every_page_size(bs, cuda_device, pa):
    rng = np.random.default_rng(bs)
    inp, _ = random_problem(rng, batch=3, max_q_len=2, num_q_heads=8, num_kv_heads=2,
                            head_dim=128, block_size=bs, ctx=[bs * 3 + 5, 17, 2 * bs],
                            causal=True, extra_blocks=2)
    ref_out, ref_lse = oracle.decode(inp, "f32")
    out, lse, _, _ = run(W.to_device(inp, cuda_device))
    compare(out, lse, ref_out, ref_lse, "bf16")


@pytest.mark.parametrize("ctas", [1, 2, 7, 152, 1000])
def test_grid_sizes(ctas, cuda_device, pa):
    inp = W.make_inputs(W.reduced(W.GQA_B32, 4, 100, 900), 2029)
    ref_out, ref_lse = oracle.decode(inp, "f32")
    out, lse, _, _ = run(W.to_device(inp, cuda_device), num_ctas=ctas)
    compare(out, lse, ref_out, ref_lse, "bf16")


def test_without_lse_output(cuda_device, pa):
    inp = W.make_inputs(W.reduced(W.LONG_SQ4, 2, 1500, 3000), 2039)
    ref_out, _ = oracle.decode(inp, "f32")
    out, _, _, _ = run(W.to_device(inp, cuda_device), with_lse=False)
    compare(out, None, ref_out, None, "bf16")


MERGE_CASES = [W.reduced(W.GQA_B32, 5, 300, 1400), W.reduced(W.LONG_SQ4, 2, 2500, 6000),
               W.reduced(W.FP8_TOKEN_SQ4, 3, 1100, 3000), W.reduced(W.mha_d256(8, 16), 2, 200, 1300)]


@pytest.mark.parametrize("mode", ["in_reduce", "in_decode"])
@pytest.mark.parametrize("ctas", [0, 40])
@pytest.mark.parametrize("wl", MERGE_CASES, ids=lambda w: w.name)
def test_split_merge_modes(wl, ctas, mode, cuda_device, pa):
    """Every split merged by the reduce kernel, or every one by the decode's last CTA."""
    inp = W.make_inputs(wl, 2039)
    ref_out, ref_lse = oracle.decode(inp, "f32")
    sm = pa.MERGE_IN_REDUCE if mode == "in_reduce" else pa.MERGE_IN_DECODE
    out, lse, ws, _ = run(W.to_device(inp, cuda_device), num_ctas=ctas, split_merge=sm)
    compare(out, lse, ref_out, ref_lse, wl.kv_dtype)
    assert pa.read_flags(ws) == 0


def test_empty_sequences_with_reduce_kernel(cuda_device, pa):
    rng = np.random.default_rng(5)
    inp, _ = random_problem(rng, batch=4, max_q_len=2, num_q_heads=4, num_kv_heads=2,
                            head_dim=128, block_size=16, ctx=[0, 90, 0, 33], q_lens=[0, 2, 0, 1],
                            causal=True)
    ref_out, ref_lse = oracle.decode(inp, "f32")
    out, lse, _, _ = run(W.to_device(inp, cuda_device), num_ctas=7, split_merge=pa.MERGE_IN_REDUCE)
    compare(out, lse, ref_out, ref_lse, "bf16")

# Grid multipliers above 1 (more CTAs than one wave; the later ones start as earlier ones
# finish): every kernel family, compared with the oracle.
GRID_CASES = [W.reduced(W.GQA_B32, 6, 300, 2000), W.reduced(W.LONG_SQ4, 2, 3000, 9000),
              W.reduced(W.FP8_TENSOR_SQ4, 3, 1000, 4000), W.reduced(W.mha_d256(4, 64), 2, 300, 1500)]


@pytest.mark.parametrize("mult", [2, 4])
@pytest.mark.parametrize("wl", GRID_CASES, ids=lambda w: w.name)
def test_grid_multiplier(wl, mult, cuda_device, pa):
    inp = W.make_inputs(wl, W.SEEDS[1])
    ref_out, ref_lse = oracle.decode(inp, "f32")
    out, lse, ws, cfg = run(W.to_device(inp, cuda_device), grid_mult=mult)
    assert cfg.grid_mult == mult
    compare(out, lse, ref_out, ref_lse, wl.kv_dtype)
    assert pa.read_flags(ws) == 0
