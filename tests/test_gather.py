"""The paged -> contiguous copy (pa_gather_kv): the oracle's gather pinned on CPU, and the
CUDA copy bit-exact against it on GPU."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W


def _bits(t):
    t = t.detach().cpu().contiguous()
    return (t.view(torch.uint8) if t.element_size() == 1 else t.view(torch.int16)).numpy()


# ---- the oracle's gather (CPU) ----------------------------------------------------------
PIN_CASES = [W.reduced(W.GQA_B32, 3, 20, 60), W.reduced(W.FP8_TOKEN_SQ1, 2, 700, 1500),
             W.reduced(W.mha_d256(8, 4), 2, 40, 90)]


@pytest.mark.parametrize("wl", PIN_CASES, ids=lambda w: w.name)
def test_oracle_gather_scatters_back_into_the_cache(wl):
    """Writing each gathered row back through the block table reproduces the cache at
    every position the batch uses, and nothing is gathered twice or left out."""
    inp = W.make_inputs(wl, W.SEEDS[0])
    k_rows, v_rows, off = oracle.gather_kv(inp)
    ctx = inp["context_lens"].numpy()
    assert off[0] == 0 and np.array_equal(np.diff(off), ctx) and len(k_rows) == ctx.sum()
    bt = inp["block_tables"].numpy()
    bs = wl.block_size
    for name, rows in (("k_cache", k_rows), ("v_cache", v_rows)):
        cache = _bits(inp[name])
        rebuilt = np.zeros_like(cache)
        used = np.zeros(cache.shape[:2], bool)
        r = 0
        for b, n in enumerate(ctx):
            for j in range(n):
                blk, slot = bt[b][j // bs], j % bs
                assert not used[blk, slot]
                rebuilt[blk, slot] = rows[r]
                used[blk, slot] = True
                r += 1
        assert r == len(rows)
        assert np.array_equal(rebuilt[used], cache[used])


def test_oracle_gather_of_an_identity_table_is_a_reshape():
    """Pages laid out in order (block b * pages + p for page p of sequence b): each
    sequence's rows are the first n_b rows of its pages' memory, read as one array."""
    wl = W.reduced(W.GQA_B32, 3, 20, 60)
    inp = W.make_inputs(wl, W.SEEDS[1])
    bs = wl.block_size
    pages = inp["block_tables"].shape[1]
    ctx = inp["context_lens"]
    inp["block_tables"] = torch.arange(wl.batch * pages, dtype=torch.int32).view(wl.batch, pages)
    need = wl.batch * pages
    for name in ("k_cache", "v_cache"):
        c = inp[name]
        inp[name] = torch.cat([c, c[:1].expand(max(0, need - c.shape[0]), *c.shape[1:])])[:need]
    k_rows, _, off = oracle.gather_kv(inp)
    flat = _bits(inp["k_cache"]).reshape(wl.batch, pages * bs, wl.num_kv_heads, wl.head_dim)
    for b in range(wl.batch):
        assert np.array_equal(k_rows[off[b]:off[b + 1]], flat[b, :int(ctx[b])])


def test_oracle_gather_skips_empty_sequences():
    wl = W.reduced(W.GQA_B32, 4, 20, 60)
    inp = W.make_inputs(wl, W.SEEDS[0], context_lens=[5, 0, 17, 0], q_lens=[1, 0, 1, 0])
    k_rows, v_rows, off = oracle.gather_kv(inp)
    assert list(off) == [0, 5, 5, 22, 22] and k_rows.shape[0] == v_rows.shape[0] == 22


# ---- the CUDA copy (GPU) -----------------------------------------------------------------
GATHER_CASES = [
    ("gqa_bs16", W.reduced(W.GQA_B32, 7, 1, 900), None),
    ("long_bs1024", W.reduced(W.LONG_SQ1, 2, 1500, 5000), None),
    ("fp8_bs1024", W.reduced(W.FP8_TENSOR_SQ1, 3, 700, 3000), None),
    ("mha_d256_bs32", W.reduced(W.mha_d256(8, 4), 5, 30, 1200), None),   # 256 KB pages
    ("ragged_and_empty", W.reduced(W.GQA_B32, 6, 1, 50), [0, 1, 17, 0, 16, 33]),
    ("tiny_bs128", W.TINY_CTX512, None),
]


def _sentinel(t):
    return 0x55 if t.element_size() == 1 else 0x5555


def _run_gather(pa, inp_dev, cfg, max_rows, flags):
    """k_out, v_out filled with a sentinel bit pattern first, and the offsets with -1."""
    dev = inp_dev["k_cache"].device
    k_out = torch.empty((max_rows, *inp_dev["k_cache"].shape[2:]), dtype=inp_dev["k_cache"].dtype,
                        device=dev)
    v_out = torch.empty_like(k_out)
    for t in (k_out, v_out):
        (t.view(torch.uint8) if t.element_size() == 1 else t.view(torch.int16)).fill_(_sentinel(t))
    offs = torch.full((cfg.batch + 1,), -1, dtype=torch.int32, device=dev)
    pa.gather_kv(cfg, inp_dev["k_cache"], inp_dev["v_cache"], inp_dev["block_tables"],
                 inp_dev["context_lens"], k_out, v_out, max_rows, offs, flags)
    torch.cuda.synchronize()
    return k_out, v_out, offs


@pytest.mark.gpu
@pytest.mark.parametrize("name,wl,lens", GATHER_CASES, ids=[c[0] for c in GATHER_CASES])
def test_gather_matches_oracle_bitwise(name, wl, lens, cuda_device, pa):
    q_lens = None if lens is None else [min(1, n) for n in lens]
    inp = W.make_inputs(wl, W.SEEDS[2], context_lens=lens, q_lens=q_lens)
    k_ref, v_ref, off = oracle.gather_kv(inp)
    dev_inp = W.to_device(inp, cuda_device)
    cfg = pa.config_for(dev_inp, num_ctas=1)
    flags = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    total = int(off[-1])
    k_out, v_out, offs = _run_gather(pa, dev_inp, cfg, total + 3, flags)
    assert int(flags.item()) == 0
    assert np.array_equal(offs.cpu().numpy(), off.astype(np.int32))
    assert np.array_equal(_bits(k_out)[:total], k_ref)
    assert np.array_equal(_bits(v_out)[:total], v_ref)
    assert (_bits(k_out)[total:] == _sentinel(k_out)).all()


@pytest.mark.gpu
def test_gather_flags_a_bad_block_and_skips_only_its_page(cuda_device, pa):
    wl = W.reduced(W.GQA_B32, 3, 100, 200)
    inp = W.make_inputs(wl, W.SEEDS[0])
    k_ref, v_ref, off = oracle.gather_kv(inp)
    bad = inp["block_tables"].clone()
    bad[1, 2] = inp["k_cache"].shape[0] + 5  # page 2 of sequence 1: rows 32 .. 47 of it
    inp_bad = dict(inp, block_tables=bad)
    dev_inp = W.to_device(inp_bad, cuda_device)
    cfg = pa.config_for(dev_inp, num_ctas=1)
    flags = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    total = int(off[-1])
    k_out, v_out, _ = _run_gather(pa, dev_inp, cfg, total, flags)
    assert int(flags.item()) & pa.FLAG_BAD_BLOCK_ID
    skipped = np.zeros(total, bool)
    skipped[off[1] + 32:off[1] + 48] = True
    assert np.array_equal(_bits(k_out)[~skipped], k_ref[~skipped])
    assert np.array_equal(_bits(v_out)[~skipped], v_ref[~skipped])
    assert (_bits(k_out)[skipped] == 0x5555).all()


@pytest.mark.gpu
def test_gather_copies_nothing_when_the_rows_do_not_fit(cuda_device, pa):
    wl = W.reduced(W.GQA_B32, 3, 100, 200)
    inp = W.make_inputs(wl, W.SEEDS[0])
    _, _, off = oracle.gather_kv(inp)
    dev_inp = W.to_device(inp, cuda_device)
    cfg = pa.config_for(dev_inp, num_ctas=1)
    flags = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    k_out, v_out, offs = _run_gather(pa, dev_inp, cfg, int(off[-1]) - 1, flags)
    assert int(flags.item()) & pa.FLAG_BAD_LENGTHS
    assert (_bits(k_out) == 0x5555).all() and (_bits(v_out) == 0x5555).all()
    assert np.array_equal(offs.cpu().numpy(), off.astype(np.int32))  # offsets still written


@pytest.mark.gpu
def test_gather_bad_lengths_count_as_empty_sequences(cuda_device, pa):
    """A negative length, or one beyond max_blocks_per_seq * block_size, is flagged and that
    sequence counts as empty: it gets no rows, the offsets stay consistent, and every other
    sequence is copied bit for bit."""
    wl = W.reduced(W.GQA_B32, 4, 20, 60)
    inp = W.make_inputs(wl, W.SEEDS[1], context_lens=[40, 17, 33, 5], q_lens=[1, 1, 1, 1])
    cap = inp["block_tables"].shape[1] * wl.block_size
    lens = [-3, 17, cap + 1, 5]
    ref_inp = dict(inp, context_lens=torch.tensor([0, 17, 0, 5], dtype=torch.int32))
    k_ref, v_ref, off = oracle.gather_kv(ref_inp)
    bad = dict(inp, context_lens=torch.tensor(lens, dtype=torch.int32))
    dev_inp = W.to_device(bad, cuda_device)
    cfg = pa.config_for(dev_inp, num_ctas=1)
    flags = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    total = int(off[-1])
    k_out, v_out, offs = _run_gather(pa, dev_inp, cfg, total + 4, flags)
    assert int(flags.item()) & pa.FLAG_BAD_LENGTHS
    assert list(offs.cpu().numpy()) == [0, 0, 17, 17, 22] == list(off.astype(np.int32))
    assert np.array_equal(_bits(k_out)[:total], k_ref)
    assert np.array_equal(_bits(v_out)[:total], v_ref)
    assert (_bits(k_out)[total:] == _sentinel(k_out)).all()
