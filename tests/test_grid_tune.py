"""The grid-multiplier table and its lookup (CPU); parity at multipliers above 1 is in
test_parity.py (GPU)."""
import csv
import os

import pytest

import paged_kv_cache_work_gb300 as pa
from paged_kv_cache_work_gb300 import grid_tune
import workloads as W


def _cfg(**kw):
    base = dict(batch=32, max_q_len=1, num_q_heads=32, num_kv_heads=8, head_dim=128,
                block_size=16, kv_dtype=pa.BF16, kv_scale_mode=pa.SCALE_NONE)
    base.update(kw)
    return pa.PaConfig(**base)


def test_choose_keeps_one_unless_a_larger_multiplier_wins_clearly():
    assert grid_tune.choose({1: 100.0, 2: 99.0, 3: 101.0}, 0.02) == 1   # 1 % is noise
    assert grid_tune.choose({1: 100.0, 2: 97.0, 4: 90.0}, 0.02) == 4
    assert grid_tune.choose({1: 100.0, 2: 90.0, 3: 90.0}, 0.02) == 2    # ties: the smaller
    assert grid_tune.choose({1: 80.0, 2: 90.0}, 0.0) == 1


def test_table_round_trip_and_lookup(tmp_path):
    path = str(tmp_path / "grid.csv")
    a, b = _cfg(), _cfg(head_dim=256, num_kv_heads=16, num_q_heads=16)
    rows = []
    for cfg, mult, name in ((a, 2, "gqa"), (b, 3, "mha")):
        r = dict(zip(grid_tune.KEY_FIELDS, grid_tune.shape_key(cfg, 152)))
        r.update(grid_mult=mult, us_per_step=1.0, us_mult1=2.0, workload=name)
        rows.append(r)
    grid_tune.write_table(rows, path)
    assert grid_tune.lookup(a, 152, path) == 2
    assert grid_tune.lookup(b, 152, path) == 3
    assert grid_tune.lookup(a, 148, path) == 1              # another device: default
    assert grid_tune.lookup(_cfg(batch=31), 152, path) == 1  # another shape: default
    assert grid_tune.lookup(a, 152, str(tmp_path / "missing.csv")) == 1


def test_table_rejects_a_multiplier_below_one(tmp_path):
    path = str(tmp_path / "bad.csv")
    r = dict(zip(grid_tune.KEY_FIELDS, grid_tune.shape_key(_cfg(), 152)))
    r.update(grid_mult=0, us_per_step=1.0, us_mult1=1.0, workload="x")
    grid_tune.write_table([r], path)
    with pytest.raises(ValueError):
        grid_tune.read_table(path)


def test_key_distinguishes_scale_mode_and_dtype():
    k1 = grid_tune.shape_key(_cfg(kv_dtype=pa.FP8_E4M3, kv_scale_mode=pa.SCALE_PER_TENSOR), 152)
    k2 = grid_tune.shape_key(_cfg(kv_dtype=pa.FP8_E4M3, kv_scale_mode=pa.SCALE_PER_TOKEN), 152)
    k3 = grid_tune.shape_key(_cfg(), 152)
    assert len({k1, k2, k3}) == 3


def test_committed_table_is_well_formed():
    if not os.path.exists(grid_tune.TABLE):
        pytest.skip("no tuned table")
    with open(grid_tune.TABLE, newline="") as f:
        rows = list(csv.DictReader(f))
    assert rows and tuple(rows[0].keys()) == grid_tune.COLUMNS
    for r in rows:
        assert r["workload"] in W.FULL
        wl = W.FULL[r["workload"]]
        assert (int(r["batch"]), int(r["max_q_len"]), int(r["num_q_heads"]),
                int(r["num_kv_heads"]), int(r["head_dim"]), int(r["block_size"])) == (
            wl.batch, wl.max_q_len, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
            wl.block_size)
        assert int(r["grid_mult"]) >= 1
        assert float(r["us_per_step"]) <= float(r["us_mult1"])
    assert len(grid_tune.read_table()) == len(rows)  # one row per key


def test_config_for_leaves_cpu_inputs_alone():
    inp = W.make_inputs(W.reduced(W.GQA_B32, 2, 100, 200), W.SEEDS[0])
    assert pa.config_for(inp).grid_mult == 0
    assert pa.config_for(inp, grid_mult=3).grid_mult == 3
