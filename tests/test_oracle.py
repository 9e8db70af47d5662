"""Pins of the CPU oracle to facts other than itself (CPU only).

* hand-derived tiny problems (tests/golden/hand_cases.json);
* brute-force float64 attention over contiguous K/V (numpy + scipy) on tiny problems
  whose pools were written by scattering through a random block table;
* paging invariance, split invariance of the log-sum-exp merge;
* closed forms: one key, identical keys, zero scale, causal first row;
* the E4M3 / fp16 / bf16 decoders against torch's dtype casts and the OCP table.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from pagedkv import brute_force, random_problem

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden", "hand_cases.json")

TOL = {"f64": 1e-11, "f32": 2e-5}


def _close(a, b, tol):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape
    fin = np.isfinite(b)
    assert np.array_equal(np.isfinite(a), fin), "finite/infinite pattern differs"
    assert np.array_equal(a[~fin], b[~fin])
    err = np.abs(a[fin] - b[fin]) / (1.0 + np.abs(b[fin]))
    assert err.size == 0 or err.max() <= tol, f"max rel err {err.max():.3e} > {tol:.1e}"


# --------------------------------------------------------------------------- golden
def _golden_inputs(case):
    c = case["cfg"]
    w = workloads.Workload(name=case["name"], batch=c["batch"], max_q_len=c["max_q_len"],
                           num_q_heads=c["num_q_heads"], num_kv_heads=c["num_kv_heads"],
                           head_dim=c["head_dim"], block_size=c["block_size"], ctx_lo=0,
                           ctx_hi=0, causal=c["causal"], q_dtype=c["q_dtype"],
                           kv_dtype=c["kv_dtype"], scale_mode=c["scale_mode"])
    q = torch.tensor(case["q"], dtype=torch.float64).to(torch.bfloat16)
    assert torch.equal(q.double(), torch.tensor(case["q"], dtype=torch.float64))
    if c["kv_dtype"] == "fp8":
        k = torch.tensor(case["k_cache_codes"], dtype=torch.uint8)
        v = torch.tensor(case["v_cache_codes"], dtype=torch.uint8)
        ks = torch.tensor(case["k_scale"], dtype=torch.float32)
        vs = torch.tensor(case["v_scale"], dtype=torch.float32)
    else:
        k = torch.tensor(case["k_cache"], dtype=torch.float64).to(torch.bfloat16)
        v = torch.tensor(case["v_cache"], dtype=torch.float64).to(torch.bfloat16)
        ks = vs = None
    return dict(workload=w, seed=None, q=q, k_cache=k, v_cache=v, k_scale=ks, v_scale=vs,
                block_tables=torch.tensor(case["block_tables"], dtype=torch.int32),
                context_lens=torch.tensor(case["context_lens"], dtype=torch.int32),
                q_lens=torch.tensor(case["q_lens"], dtype=torch.int32),
                sm_scale=c["sm_scale"])


def _golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)


@pytest.mark.parametrize("precision", ["f64", "f32"])
@pytest.mark.parametrize("idx", range(4))
def test_golden_hand_cases(idx, precision):
    case = _golden_cases()["cases"][idx]
    out, lse = oracle.decode(_golden_inputs(case), precision)
    np.testing.assert_allclose(out, np.array(case["expected_out"], np.float64), rtol=1e-6,
                               atol=1e-6)
    np.testing.assert_allclose(lse, np.array(case["expected_lse"], np.float64), rtol=1e-6,
                               atol=1e-6)


def test_golden_e4m3_table():
    table = _golden_cases()["e4m3"]["codes"]
    for code, val in table.items():
        got = oracle.e4m3(int(code))
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == val and math.copysign(1, got) == math.copysign(1, val), (code, got)


# --------------------------------------------------------------------- decoders
def test_e4m3_all_codes_match_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    for prec in ("f64", "f32"):
        got = np.array([oracle.e4m3(c, prec) for c in range(256)])
        r = ref.numpy()
        assert np.array_equal(np.isnan(got), np.isnan(r))
        m = ~np.isnan(r)
        assert np.array_equal(got[m], r[m])
        assert np.array_equal(np.signbit(got[m]), np.signbit(r[m]))


@pytest.mark.parametrize("kind", ["bf16", "fp16"])
def test_16bit_decoders_all_codes(kind):
    codes = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    dt = torch.bfloat16 if kind == "bf16" else torch.float16
    ref = codes.view(dt).to(torch.float64).numpy()
    fn = oracle.bf16 if kind == "bf16" else oracle.fp16
    got = np.array([fn(c) for c in range(65536)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    m = ~np.isnan(ref)
    assert np.array_equal(got[m], ref[m])
    assert np.array_equal(np.signbit(got[m]), np.signbit(ref[m]))


# ------------------------------------------------------------------ brute force
BRUTE_CASES = [
    # (B, Sq, Hq, Hkv, D, bs, ctx, q_lens, causal, kv_dtype, scale_mode)
    (1, 1, 1, 1, 8, 1, [1], None, False, "bf16", "none"),
    (2, 1, 4, 2, 8, 2, [5, 17], None, False, "bf16", "none"),
    (2, 1, 6, 3, 16, 4, [33, 40], None, False, "bf16", "none"),
    (1, 3, 4, 1, 8, 16, [37], None, True, "bf16", "none"),
    (2, 3, 2, 2, 16, 4, [3, 29], [3, 2], True, "bf16", "none"),
    (2, 4, 8, 2, 8, 2, [9, 12], [4, 1], False, "fp16", "none"),
    (2, 2, 4, 4, 16, 16, [16, 31], None, True, "fp16", "none"),
    (2, 1, 4, 1, 16, 4, [21, 40], None, False, "fp8", "tensor"),
    (2, 2, 4, 2, 8, 2, [11, 26], None, True, "fp8", "token"),
    (1, 1, 2, 1, 8, 1, [40], None, False, "fp8", "token"),
]


def _brute_problem(case, seed):
    B, Sq, Hq, Hkv, D, bs, ctx, ql, causal, kvd, sm = case
    rng = np.random.default_rng(seed)
    q_dtype = "fp16" if kvd == "fp16" else "bf16"
    return random_problem(rng, batch=B, max_q_len=Sq, num_q_heads=Hq, num_kv_heads=Hkv,
                          head_dim=D, block_size=bs, ctx=ctx, q_lens=ql, causal=causal,
                          q_dtype=q_dtype, kv_dtype=kvd, scale_mode=sm)


@pytest.mark.parametrize("precision", ["f64", "f32"])
@pytest.mark.parametrize("ci", range(len(BRUTE_CASES)))
def test_oracle_matches_contiguous_brute_force(ci, precision):
    inp, contiguous = _brute_problem(BRUTE_CASES[ci], 100 + ci)
    ref_out, ref_lse = brute_force(inp, contiguous)
    out, lse = oracle.decode(inp, precision)
    _close(out, ref_out, TOL[precision])
    _close(lse, ref_lse, TOL[precision])


def test_rows_and_ranges_agree_with_full_decode():
    inp, _ = _brute_problem(BRUTE_CASES[4], 7)
    out, lse = oracle.decode(inp, "f64")
    rows = np.array([[0, 0, 1], [1, 1, 0], [1, 2, 1], [0, 2, 0]], np.int32)
    o2, l2 = oracle.decode_rows(inp, rows, "f64")
    for t, (b, i, h) in enumerate(rows):
        assert np.array_equal(o2[t], out[b, i, h]) and l2[t] == lse[b, i, h]
    # a range covering every visible key is the full row
    o3, l3 = oracle.attend_range(inp, 1, 0, 1, 0, 10 ** 6, "f64")
    assert np.array_equal(o3, out[1, 0, 1]) and l3 == lse[1, 0, 1]


# ------------------------------------------------------------------- invariances
@pytest.mark.parametrize("precision", ["f64", "f32"])
def test_paging_invariance_bitwise(precision):
    inp, _ = _brute_problem(BRUTE_CASES[2], 11)
    out, lse = oracle.decode(inp, precision)
    nb = inp["k_cache"].shape[0]
    perm = torch.from_numpy(np.random.default_rng(5).permutation(nb)).long()
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(nb)
    moved = dict(inp)
    # block p moves to physical slot perm[p]; the table is renamed the same way
    moved["k_cache"] = inp["k_cache"][inv].contiguous()
    moved["v_cache"] = inp["v_cache"][inv].contiguous()
    bt = inp["block_tables"].long()
    moved["block_tables"] = torch.where(bt >= 0, perm[bt.clamp(min=0)], bt).to(torch.int32)
    out2, lse2 = oracle.decode(moved, precision)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


@pytest.mark.parametrize("precision", ["f64", "f32"])
@pytest.mark.parametrize("nsplit", [2, 3, 7, 40])
def test_split_invariance(nsplit, precision):
    for ci in (2, 4, 8):
        inp, _ = _brute_problem(BRUTE_CASES[ci], 21 + ci)
        out, lse = oracle.decode(inp, precision)
        o2, l2 = oracle.decode(inp, precision, nsplit=nsplit)
        _close(o2, out, 1e-12 if precision == "f64" else 1e-5)
        _close(l2, lse, 1e-12 if precision == "f64" else 1e-5)


def test_merge_of_empty_splits():
    o = np.zeros((3, 4))
    o[1] = [1, 2, 3, 4]
    lse = np.array([-np.inf, 0.5, -np.inf])
    mo, ml = oracle.merge(o, lse)
    assert np.array_equal(mo, o[1]) and ml == 0.5
    mo, ml = oracle.merge(np.zeros((2, 4)), np.array([-np.inf, -np.inf]))
    assert np.all(mo == 0) and ml == -np.inf


# ----------------------------------------------------------------- closed forms
@pytest.mark.parametrize("precision", ["f64", "f32"])
def test_single_key_returns_its_value_row(precision):
    rng = np.random.default_rng(3)
    inp, contiguous = random_problem(rng, batch=3, max_q_len=1, num_q_heads=4, num_kv_heads=2,
                                     head_dim=16, block_size=4, ctx=[1, 1, 1])
    out, lse = oracle.decode(inp, precision)
    q = inp["q"].double().numpy()
    sm = float(np.float32(inp["sm_scale"]))
    for b in range(3):
        K, V = contiguous[b]
        for h in range(4):
            assert np.array_equal(out[b, 0, h], V[0, h // 2].astype(out.dtype))
            assert abs(lse[b, 0, h] - sm * (K[0, h // 2] @ q[b, 0, h])) < 1e-5


@pytest.mark.parametrize("precision", ["f64", "f32"])
def test_identical_keys_give_mean_of_values(precision):
    rng = np.random.default_rng(4)
    inp, contiguous = random_problem(rng, batch=1, max_q_len=1, num_q_heads=2, num_kv_heads=1,
                                     head_dim=8, block_size=2, ctx=[13])
    kc = inp["k_cache"].clone()
    bt = inp["block_tables"][0]
    first = kc[bt[0], 0].clone()
    for j in range(13):
        kc[bt[j // 2], j % 2] = first
    inp["k_cache"] = kc
    out, lse = oracle.decode(inp, precision)
    Vmean = contiguous[0][1][:, 0].mean(axis=0)
    for h in range(2):
        np.testing.assert_allclose(out[0, 0, h], Vmean, rtol=1e-5, atol=1e-6)
        s0 = float(np.float32(inp["sm_scale"])) * (first[0].double().numpy() @
                                                    inp["q"][0, 0, h].double().numpy())
        assert abs(lse[0, 0, h] - (s0 + math.log(13))) < 1e-5


@pytest.mark.parametrize("precision", ["f64", "f32"])
def test_zero_scale_gives_mean_over_visible_keys(precision):
    rng = np.random.default_rng(6)
    inp, contiguous = random_problem(rng, batch=2, max_q_len=3, num_q_heads=2, num_kv_heads=2,
                                     head_dim=8, block_size=4, ctx=[7, 10], q_lens=[3, 2],
                                     causal=True, sm_scale=0.0)
    out, lse = oracle.decode(inp, precision)
    for b, (n, ql) in enumerate([(7, 3), (10, 2)]):
        V = contiguous[b][1]
        for i in range(3):
            for h in range(2):
                if i >= ql:
                    assert np.all(out[b, i, h] == 0) and lse[b, i, h] == -np.inf
                    continue
                L = n - ql + i + 1
                np.testing.assert_allclose(out[b, i, h], V[:L, h].mean(axis=0), rtol=1e-5,
                                           atol=1e-6)
                assert abs(lse[b, i, h] - math.log(L)) < 1e-6


@pytest.mark.parametrize("precision", ["f64", "f32"])
def test_causal_first_row_sees_only_first_key(precision):
    rng = np.random.default_rng(8)
    inp, contiguous = random_problem(rng, batch=1, max_q_len=5, num_q_heads=3, num_kv_heads=1,
                                     head_dim=8, block_size=2, ctx=[5], causal=True)
    out, _ = oracle.decode(inp, precision)
    V0 = contiguous[0][1][0, 0]
    for h in range(3):
        assert np.array_equal(out[0, 0, h], V0.astype(out.dtype))


def test_invalid_lengths_rejected():
    inp, _ = _brute_problem(BRUTE_CASES[1], 1)
    bad = dict(inp)
    bad["q_lens"] = torch.tensor([2, 1], dtype=torch.int32)  # > max_q_len
    with pytest.raises(ValueError):
        oracle.decode(bad, "f64")
    bad = dict(inp)
    bad["block_tables"] = inp["block_tables"].clone()
    bad["block_tables"][1, 0] = 10 ** 6  # page outside the pool
    with pytest.raises(ValueError):
        oracle.decode(bad, "f64")


def test_f32_build_tracks_f64_on_a_workload():
    w = workloads.reduced(workloads.GQA_B32, 3, 100, 300)
    inp = workloads.make_inputs(w, workloads.SEEDS[0])
    o32, l32 = oracle.decode(inp, "f32")
    o64, l64 = oracle.decode(inp, "f64")
    assert np.abs(o32 - o64).max() < 1e-4 and np.abs(l32 - l64).max() < 1e-4
