"""The planner's work list, read back from the workspace (GPU).

* bit-exact coverage: every (sequence, kv head, row tile, token) lies in exactly one work
  item, and items never reach past a sequence's context;
* every CTA's items are exactly the units its piece of the concatenated token space
  overlaps (each unit its tile-padded length plus a fixed item cost), with the token range
  the piece holds, and the chunk is the smallest tile multiple that fits the space in C
  pieces;
* the partial slots of units cut into several pieces are CTA c's slots 2c / 2c + 1, and
  the unit table points at them;
* the reduce list holds exactly the units of more pieces than the decode merges itself, in
  unit order, and a finished decode leaves every merge counter at zero;
* each partial the decode kernel wrote equals the oracle's attention over that item's
  key range (so the split mode is checked on its own, before the reducer).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_run import REDUCE_WARP_PIECES, plan_view, run
from pagedkv import random_problem

pytestmark = pytest.mark.gpu


def check_plan(view, ctx, ctas, hkv):
    """Exact checks of the work list against the cutting rule stated in plan.cu: units laid
    end to end, each its tile-padded length plus the fixed item cost (none for an empty
    unit), the space cut into equal tile-aligned pieces, one per CTA."""
    v = view["v"]
    tt, U, rb, cost = v["tt"], v["units"], v["rb"], v["item_cost"]
    per_seq = hkv * rb
    lens = np.array([ctx[u // per_seq] for u in range(U)], np.int64)
    plen = -(-lens // tt) * tt
    stride = np.where(lens > 0, plen + cost, 0)
    start = np.concatenate([[0], np.cumsum(stride)])
    T = int(start[-1])
    chunk = view["chunk"]
    if T > 0:
        assert chunk == -(-(-(-T // ctas)) // tt) * tt
        assert view["active"] == -(-T // chunk) <= ctas
    else:
        assert view["active"] == 0
    item_off, items = view["item_off"], view["items"]
    assert item_off[0] == 0 and (np.diff(item_off) >= 0).all()
    assert item_off[-1] == view["n_items"]
    # each CTA's first item is repeated in its own slot, (0, 0, 0, -1) for an empty list
    for c in range(ctas):
        want_first = items[item_off[c]] if item_off[c] < item_off[c + 1] else [0, 0, 0, -1]
        assert view["first_item"][c].tolist() == list(want_first), f"CTA {c} first item"
    covered = [np.zeros(int(n), np.int32) for n in lens]
    slots = {}
    for c in range(ctas):
        got = [tuple(int(x) for x in items[it]) for it in range(item_off[c], item_off[c + 1])]
        want = []
        if c < view["active"]:
            lo, hi = c * chunk, min((c + 1) * chunk, T)
            for u in range(U):
                st = int(start[u])
                if stride[u] == 0 or st >= hi or st + stride[u] <= lo:
                    continue
                t0, t1 = max(lo, st) - st, min(hi - st, int(lens[u]))
                if t1 <= t0:
                    want.append((u, 0, 0, -1))  # only the unit's item-cost stretch
                    continue
                split = (st + plen[u] - 1) // chunk != st // chunk
                want.append((u, t0, t1, 2 * c + (1 if want else 0) if split else -1))
        assert got == want, f"CTA {c}: {got} != {want}"
        for k, (u, t0, t1, slot) in enumerate(got):
            if t1 <= t0:
                continue
            assert t0 % tt == 0 and (t1 % tt == 0 or t1 == lens[u])
            covered[u][t0:t1] += 1
            slots.setdefault(u, []).append(slot)
            if slot >= 0:  # only a piece's first or last item can be split
                assert k == 0 or k == len(got) - 1
    for u in range(U):
        assert (covered[u] == 1).all(), f"unit {u} not covered exactly once"
        info = view["unit_info"][u]
        ns = len(slots.get(u, []))
        assert int(info[1]) == ns
        if ns == 1:
            assert slots[u] == [-1]
        elif ns > 1:
            first = int(info[0])
            assert slots[u] == [first] + [2 * (first // 2 + s) for s in range(1, ns)]
    # units left to the reduce kernel: the few-piece ones first, then the rest, each in order
    ns_of = [int(view["unit_info"][u][1]) for u in range(U)]
    small = [u for u in range(U) if v["ns_dec"] < ns_of[u] <= REDUCE_WARP_PIECES]
    large = [u for u in range(U) if ns_of[u] > max(v["ns_dec"], REDUCE_WARP_PIECES)]
    assert view["red_units"].tolist() == small + large
    assert view["n_red_small"] == len(small)
    assert (view["unit_cnt"] == 0).all(), "merge counters not reset by the decode"
    return T


CASES = [
    ("gqa", W.reduced(W.GQA_B32, 7, 1, 3000), [152, 5, 1, 1000]),
    ("long_sq4", W.reduced(W.LONG_SQ4, 3, 4, 20000), [152, 3]),
    ("mha_sq16", W.reduced(W.mha_d256(8, 16), 3, 16, 4000), [152, 64]),
    ("fp8_token", W.reduced(W.FP8_TOKEN_SQ1, 5, 1, 5000), [152, 9]),
    # a tcgen05 decode's planner keeps prefix sums of at most 1024 sequences in shared memory
    ("long_sq4_many_sequences", W.reduced(W.LONG_SQ4, 1100, 4, 300), [152]),
]


@pytest.mark.parametrize("name,wl,grids", CASES, ids=[c[0] for c in CASES])
def test_work_list_covers_every_token_once(name, wl, grids, cuda_device, pa):
    for seed in W.SEEDS:
        inp = W.make_inputs(wl, seed, device=cuda_device)
        ctx = inp["context_lens"].cpu().numpy()
        for ctas in grids:
            for sm in (pa.MERGE_AUTO, pa.MERGE_IN_DECODE, pa.MERGE_IN_REDUCE):
                _, _, ws, cfg = run(inp, num_ctas=ctas, split_merge=sm)
                view = plan_view(ws, cfg, ctas)
                assert view["flags"] == 0
                check_plan(view, ctx, ctas, wl.num_kv_heads)


def test_random_shapes_coverage(cuda_device, pa):
    rng = np.random.default_rng(99)
    for trial in range(12):
        B = int(rng.integers(1, 9))
        ctx = [int(x) for x in rng.integers(0, 700, size=B)]
        ctx[0] = max(ctx[0], 1)
        kw = dict(batch=B, max_q_len=1, num_q_heads=4, num_kv_heads=int(rng.choice([1, 2, 4])),
                  head_dim=int(rng.choice([64, 128])), block_size=int(rng.choice([16, 32, 128])),
                  ctx=ctx, q_lens=[min(1, n) for n in ctx])
        inp, _ = random_problem(rng, **kw)
        dev = W.to_device(inp, cuda_device)
        for ctas in (1, 3, 152):
            _, _, ws, cfg = run(dev, num_ctas=ctas)
            check_plan(plan_view(ws, cfg, ctas), ctx, ctas, kw["num_kv_heads"])


def test_partials_equal_oracle_ranges(cuda_device, pa):
    wl = W.reduced(W.LONG_SQ4, 2, 3000, 7000)
    inp = W.make_inputs(wl, 2026)
    dev = W.to_device(inp, cuda_device)
    ctas = 16
    _, _, ws, cfg = run(dev, num_ctas=ctas)
    view = plan_view(ws, cfg, ctas)
    v = view["v"]
    G = wl.num_q_heads // wl.num_kv_heads
    checked = 0
    for it in range(view["n_items"]):
        u, t0, t1, slot = (int(x) for x in view["items"][it])
        if slot < 0 or t1 <= t0:
            continue
        b = u // (wl.num_kv_heads * v["rb"])
        g = (u // v["rb"]) % wl.num_kv_heads
        rb = u % v["rb"]
        for r in range(v["mp"]):
            rg = rb * v["mp"] + r
            if rg >= v["rows"]:
                continue
            i, h = rg // G, g * G + rg % G
            o, lse = oracle.attend_range(inp, b, i, h, t0, t1, "f64")
            got_o = view["o_part"][slot, r]
            got_l = view["lse_part"][slot, r] * np.log(2.0)
            if not np.isfinite(lse):
                assert got_l == -np.inf and np.all(got_o == 0)
                continue
            assert np.abs(got_o - o).max() <= 2e-3 + 2e-3 * np.abs(o).max()
            assert abs(got_l - lse) <= 2e-4 * (1 + abs(lse))
            checked += 1
    assert checked > 0
