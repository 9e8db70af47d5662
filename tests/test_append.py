"""GPU parity of the quantise-on-write KV append (pa_append_kv) against the oracle's append,
bit for bit: the whole cache (codes or 16-bit rows) and every per-token scale after the
call, on the same seeded problems.

Covered: 16-bit caches (bf16, fp16), fp8 with per-token, per-tensor and no scales, bf16 and
fp16 new rows, head dims 64/128/256, pages of 16 and 1024 tokens (appends that straddle a
page boundary), ragged and empty q_lens, several kv heads, a bad block id (flagged, that row
not written) and bad lengths (flagged, that sequence not written).
"""
import numpy as np
import pytest
import torch

import oracle
from test_append_oracle import random_append_problem

pytestmark = pytest.mark.gpu

CASES = [
    # name, kwargs of random_append_problem
    ("bf16_d128", dict(kv_dtype="bf16", q_dtype="bf16", scale_mode="none", head_dim=128,
                       block_size=16)),
    ("fp16_d64", dict(kv_dtype="fp16", q_dtype="fp16", scale_mode="none", head_dim=64,
                      block_size=32)),
    ("bf16_d256_two_heads", dict(kv_dtype="bf16", q_dtype="bf16", scale_mode="none",
                                 head_dim=256, num_kv_heads=2, block_size=16)),
    ("fp8_token_d128", dict(kv_dtype="fp8", scale_mode="token", head_dim=128, block_size=16)),
    ("fp8_token_fp16_d256", dict(kv_dtype="fp8", scale_mode="token", q_dtype="fp16",
                                 head_dim=256, num_kv_heads=3, block_size=16)),
    ("fp8_token_d64_big_pages", dict(kv_dtype="fp8", scale_mode="token", head_dim=64,
                                     block_size=1024, batch=3, max_q_len=4)),
    ("fp8_tensor_d128", dict(kv_dtype="fp8", scale_mode="tensor", head_dim=128,
                             block_size=32)),
    ("fp8_none_fp16_d128", dict(kv_dtype="fp8", scale_mode="none", q_dtype="fp16",
                                head_dim=128, block_size=16)),
    ("fp8_token_many_seqs", dict(kv_dtype="fp8", scale_mode="token", head_dim=128,
                                 block_size=16, batch=37, max_q_len=5, num_kv_heads=2)),
]


def _cfg(pa, inp):
    w = inp["workload"]
    dt = {"bf16": pa.BF16, "fp16": pa.FP16, "fp8": pa.FP8_E4M3}
    sm = {"none": pa.SCALE_NONE, "tensor": pa.SCALE_PER_TENSOR, "token": pa.SCALE_PER_TOKEN}
    return pa.PaConfig(batch=w.batch, max_q_len=w.max_q_len, num_q_heads=w.num_kv_heads,
                       num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                       block_size=w.block_size,
                       max_blocks_per_seq=inp["block_tables"].shape[1],
                       num_blocks=inp["k_cache"].shape[0], q_dtype=dt[w.q_dtype],
                       kv_dtype=dt[w.kv_dtype],
                       kv_scale_mode=sm[w.scale_mode] if w.kv_dtype == "fp8" else pa.SCALE_NONE,
                       causal=0, sm_scale=1.0)


def _run(pa, inp, kn, vn, dev):
    d = {k: (v.to(dev).clone() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    pa.append_kv(_cfg(pa, inp), kn.to(dev), vn.to(dev), d["block_tables"], d["context_lens"],
                 d["q_lens"], d["k_cache"], d["v_cache"], d["k_scale"], d["v_scale"], flags)
    torch.cuda.synchronize()
    return d, int(flags.item())


def _bits(t):
    t = t.detach().cpu().contiguous()
    return t.view(torch.uint8) if t.element_size() == 1 else t.view(torch.int16)


def _assert_same(d, kc, vc, ks, vs):
    assert torch.equal(_bits(d["k_cache"]), _bits(kc)), "K cache differs from the oracle"
    assert torch.equal(_bits(d["v_cache"]), _bits(vc)), "V cache differs from the oracle"
    if ks is not None:
        assert torch.equal(d["k_scale"].cpu().view(torch.int32), ks.view(torch.int32))
        assert torch.equal(d["v_scale"].cpu().view(torch.int32), vs.view(torch.int32))


@pytest.mark.parametrize("seed", [2026, 2029, 2039])
@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_append_matches_oracle_bitwise(name, kw, seed, cuda_device, pa):
    inp, kn, vn = random_append_problem(seed, **kw)
    kc, vc, ks, vs = oracle.append_kv(inp, kn, vn)
    d, flags = _run(pa, inp, kn, vn, cuda_device)
    assert flags == 0
    _assert_same(d, kc, vc, ks, vs)


def test_append_then_decode_matches_oracle(cuda_device, pa):
    """The decode reads back what the append wrote: appending the new rows into an fp8
    per-token cache and decoding equals the oracle decode of the oracle's appended cache."""
    import workloads as W
    from gpu_run import compare, run
    wl = W.reduced(W.FP8_TOKEN_SQ4, 3, 300, 900)
    inp = W.make_inputs(wl, 2026)
    rng = np.random.default_rng(7)
    B, Sq, H, D = wl.batch, wl.max_q_len, wl.num_kv_heads, wl.head_dim
    kn = torch.from_numpy(rng.standard_normal((B, Sq, H, D)) * 2).to(torch.bfloat16)
    vn = torch.from_numpy(rng.standard_normal((B, Sq, H, D))).to(torch.bfloat16)
    kc, vc, ks, vs = oracle.append_kv(inp, kn, vn)
    ref_inp = dict(inp, k_cache=kc, v_cache=vc, k_scale=ks, v_scale=vs)
    ref_out, ref_lse = oracle.decode(ref_inp, "f32")
    d, flags = _run(pa, inp, kn, vn, cuda_device)
    assert flags == 0
    _assert_same(d, kc, vc, ks, vs)
    out, lse, ws, _ = run(d)
    compare(out, lse, ref_out, ref_lse, "fp8")
    assert pa.read_flags(ws) == 0


def test_append_bad_block_id_is_flagged_and_skipped(cuda_device, pa):
    inp, kn, vn = random_append_problem(2029, kv_dtype="fp8", scale_mode="token", head_dim=128,
                                        block_size=16, batch=4)
    bs = inp["workload"].block_size
    b = 0
    n, ql = int(inp["context_lens"][b]), int(inp["q_lens"][b])
    page = (n - ql) // bs  # the page of the sequence's first new row
    good = dict(inp)
    bad = dict(inp)
    bad["block_tables"] = inp["block_tables"].clone()
    bad["block_tables"][b, page] = inp["k_cache"].shape[0] + 5
    d, flags = _run(pa, bad, kn, vn, cuda_device)
    assert flags & pa.FLAG_BAD_BLOCK_ID
    # every row but the ones on that page matches the oracle's append with the good table;
    # the rows of that page were not written (the cache keeps its old contents there)
    kc, vc, ks, vs = oracle.append_kv(good, kn, vn)
    blk = int(inp["block_tables"][b, page])
    kc[blk] = inp["k_cache"][blk]
    vc[blk] = inp["v_cache"][blk]
    ks[blk] = inp["k_scale"][blk]
    vs[blk] = inp["v_scale"][blk]
    # other sequences never write block blk (tables are drawn without replacement)
    _assert_same(d, kc, vc, ks, vs)


def test_append_bad_lengths_are_flagged_and_skipped(cuda_device, pa):
    inp, kn, vn = random_append_problem(2039, kv_dtype="bf16", q_dtype="bf16",
                                        scale_mode="none", head_dim=64, block_size=16, batch=4)
    bad = dict(inp)
    bad["context_lens"] = inp["context_lens"].clone()
    bad["q_lens"] = inp["q_lens"].clone()
    bad["q_lens"][0] = 2
    bad["context_lens"][0] = 1  # fewer cached tokens than new ones
    d, flags = _run(pa, bad, kn, vn, cuda_device)
    assert flags & pa.FLAG_BAD_LENGTHS
    # sequence 0 writes nothing; the others as the oracle writes them
    ok = dict(inp)
    ok["q_lens"] = inp["q_lens"].clone()
    ok["q_lens"][0] = 0
    kc, vc, _, _ = oracle.append_kv(ok, kn, vn)
    _assert_same(d, kc, vc, None, None)


def test_append_rejects_bad_arguments(cuda_device, pa):
    inp, kn, vn = random_append_problem(2026, kv_dtype="fp8", scale_mode="token", head_dim=128,
                                        block_size=16)
    dev = cuda_device
    cfg = _cfg(pa, inp)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    with pytest.raises(pa.PaError) as e:  # scales missing with a scale mode
        pa.append_kv(cfg, kn.to(dev), vn.to(dev), d["block_tables"], d["context_lens"],
                     d["q_lens"], d["k_cache"], d["v_cache"], None, None)
    assert e.value.status == 1
    cfg.head_dim = 96
    with pytest.raises(pa.PaError) as e:
        pa.append_kv(cfg, kn.to(dev), vn.to(dev), d["block_tables"], d["context_lens"],
                     d["q_lens"], d["k_cache"], d["v_cache"], d["k_scale"], d["v_scale"])
    assert e.value.status == 2
