"""Pins of the oracle's quantise-on-write KV append to facts other than itself (CPU only).

* hand-derived tiny appends (tests/golden/append_cases.json): codes, scales and the rows
  the block table sends them to;
* the E4M3 encoder against torch's float8_e4m3fn cast (round to nearest even, after the
  clamp to +-448) on every grid point, every midpoint between neighbours and values just
  off them, and against a brute-force nearest-code search over torch's decoding of all 256
  codes;
* placement: every new row lands at slot (n - q_len + i) % bs of block
  table[b][(n - q_len + i) // bs] and no other pool row changes;
* per-token scales: amax / 448 in fp32, the largest-magnitude element encodes to +-448, and
  decoding the written codes returns every value within half a grid step.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden", "append_cases.json")

SENTINEL_16 = 1000.0
SENTINEL_CODE = 0x11
SENTINEL_SCALE = 9.0


def _torch_codes(x: torch.Tensor) -> torch.Tensor:
    """torch's E4M3 encoding of fp32 values after the clamp to +-448."""
    return torch.clamp(x.float(), -448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)


def _all_code_values() -> np.ndarray:
    """float64 value of each of the 256 codes, through torch's own decoding."""
    return torch.arange(256, dtype=torch.int32).to(torch.uint8).view(
        torch.float8_e4m3fn).to(torch.float64).numpy()


def _encode_all(xs: np.ndarray) -> np.ndarray:
    return np.array([oracle.e4m3_encode(float(x)) for x in xs.astype(np.float32)], np.int64)


# ------------------------------------------------------------------------- encoder
def _grid_points_and_midpoints():
    vals = _all_code_values()
    finite = np.unique(np.abs(vals[np.isfinite(vals)]))  # 0 .. 448, ascending
    mids = (finite[:-1] + finite[1:]) / 2  # exact in fp32 (one more bit than E4M3)
    pts = np.concatenate([finite, mids])
    f32 = pts.astype(np.float32)
    assert np.array_equal(f32.astype(np.float64), pts), "midpoints must be exact in fp32"
    up = np.nextafter(f32, np.float32(np.inf))
    dn = np.nextafter(f32, np.float32(0))
    out = np.concatenate([f32, up, dn, [448.0, 449.0, 463.99, 464.0, 465.0, 480.0, 1e6, 3e38]])
    out = out.astype(np.float32)
    return np.concatenate([out, -out])


def test_e4m3_encode_matches_torch_on_grid_midpoints_and_neighbours():
    xs = _grid_points_and_midpoints()
    got = _encode_all(xs)
    want = _torch_codes(torch.from_numpy(xs)).numpy().astype(np.int64)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(xs[i]), hex(got[i]), hex(want[i])) for i in bad[:8]]


def test_e4m3_encode_matches_torch_on_random_values():
    rng = np.random.default_rng(2026)
    xs = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.05, 1.0, 30.0, 400.0)])
    xs = xs.astype(np.float32)
    got = _encode_all(xs)
    want = _torch_codes(torch.from_numpy(xs)).numpy().astype(np.int64)
    assert np.array_equal(got, want)


def test_e4m3_encode_is_the_nearest_code_ties_to_even():
    """Brute force: the chosen code's value is the nearest finite E4M3 value to the clamped
    input, and on a tie its mantissa is even."""
    vals = _all_code_values()
    codes = np.arange(256)
    fin = np.isfinite(vals)
    rng = np.random.default_rng(2029)
    xs = np.concatenate([_grid_points_and_midpoints(),
                         (rng.standard_normal(3000) * 50).astype(np.float32)])
    for x, c in zip(xs, _encode_all(xs)):
        xc = min(max(float(x), -448.0), 448.0)
        dist = np.abs(vals[fin] - xc)
        best = dist.min()
        assert abs(vals[c] - xc) == best, (float(x), hex(c))
        ties = codes[fin][dist == best]
        # a signed zero tie is between 0x00 and 0x80: both have an even mantissa
        if ties.size > 1 and best > 0:
            assert c & 1 == 0, (float(x), hex(c), [hex(t) for t in ties])


def test_e4m3_encode_nan():
    assert oracle.e4m3_encode(float("nan")) & 0x7f == 0x7f


# ---------------------------------------------------------------------- golden cases
def _golden():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


def _case_problem(case):
    c = case["cfg"]
    new_k = torch.tensor(case["new_k"], dtype=torch.float64)
    B, Sq, H, D = new_k.shape
    bt = torch.tensor(case["block_tables"], dtype=torch.int32)
    w = workloads.Workload(name=case["name"], batch=B, max_q_len=Sq, num_q_heads=H,
                           num_kv_heads=H, head_dim=D, block_size=c["block_size"], ctx_lo=0,
                           ctx_hi=0, kv_dtype=c["kv_dtype"], scale_mode=c["scale_mode"])
    nb, bs = c["num_blocks"], c["block_size"]
    if c["kv_dtype"] == "fp8":
        k = torch.full((nb, bs, H, D), SENTINEL_CODE, dtype=torch.uint8)
        v = k.clone()
        if c["scale_mode"] == "token":
            ks = torch.full((nb, bs, H), SENTINEL_SCALE, dtype=torch.float32)
            vs = ks.clone()
        elif c["scale_mode"] == "tensor":
            ks = torch.tensor([c["k_scale"]], dtype=torch.float32)
            vs = torch.tensor([c["v_scale"]], dtype=torch.float32)
        else:
            ks = vs = None
    else:
        k = torch.full((nb, bs, H, D), SENTINEL_16, dtype=torch.bfloat16)
        v = k.clone()
        ks = vs = None
    inp = dict(workload=w, q=torch.zeros((B, Sq, H, D), dtype=torch.bfloat16), k_cache=k,
               v_cache=v, k_scale=ks, v_scale=vs, block_tables=bt,
               context_lens=torch.tensor(case["context_lens"], dtype=torch.int32),
               q_lens=torch.tensor(case["q_lens"], dtype=torch.int32), sm_scale=1.0)
    kn = new_k.to(torch.bfloat16)
    vn = torch.tensor(case["new_v"], dtype=torch.float64).to(torch.bfloat16)
    assert torch.equal(kn.double(), new_k), "golden inputs must be exact in bf16"
    return inp, kn, vn


@pytest.mark.parametrize("precision", ["f64", "f32"])
@pytest.mark.parametrize("idx", range(5))
def test_golden_append_cases(idx, precision):
    case = _golden()[idx]
    inp, kn, vn = _case_problem(case)
    kc, vc, ks, vs = oracle.append_kv(inp, kn, vn, precision)
    fp8 = case["cfg"]["kv_dtype"] == "fp8"
    written = set()
    for r in case["expected_rows"]:
        blk, slot, h = r["block"], r["slot"], r["head"]
        written.add((blk, slot, h))
        if fp8:
            assert kc[blk, slot, h].tolist() == r["k_codes"]
            assert vc[blk, slot, h].tolist() == r["v_codes"]
            if "k_scale" in r:
                assert float(ks[blk, slot, h]) == r["k_scale"]
                assert float(vs[blk, slot, h]) == r["v_scale"]
        else:
            assert kc[blk, slot, h].double().tolist() == r["k"]
            assert vc[blk, slot, h].double().tolist() == r["v"]
    nb, bs, H, _ = kc.shape
    for blk in range(nb):
        for slot in range(bs):
            for h in range(H):
                if (blk, slot, h) in written:
                    continue
                if fp8:
                    assert (kc[blk, slot, h] == SENTINEL_CODE).all()
                    assert (vc[blk, slot, h] == SENTINEL_CODE).all()
                    if case["cfg"]["scale_mode"] == "token":
                        assert float(ks[blk, slot, h]) == SENTINEL_SCALE
                else:
                    assert (kc[blk, slot, h].double() == SENTINEL_16).all()
    if fp8 and case["cfg"]["scale_mode"] == "tensor":
        assert float(ks[0]) == case["cfg"]["k_scale"] and float(vs[0]) == case["cfg"]["v_scale"]


# ------------------------------------------------------------- random problems, pinned
def random_append_problem(seed, *, batch=4, max_q_len=3, num_kv_heads=2, head_dim=16,
                          block_size=4, kv_dtype="fp8", scale_mode="token", q_dtype="bf16",
                          zero_rows=True):
    """A pool with sentinel contents, random lengths (some sequences appending fewer rows
    than max_q_len, one appending none) and new rows, some of them all zero."""
    rng = np.random.default_rng(seed)
    B, Sq, H, D, bs = batch, max_q_len, num_kv_heads, head_dim, block_size
    ql = rng.integers(0, Sq + 1, size=B)
    ql[0] = Sq
    ctx = ql + rng.integers(0, 3 * bs, size=B)
    pages = [(int(n) + bs - 1) // bs for n in ctx]
    nb = sum(pages) + 3
    perm = rng.permutation(nb)
    maxb = max(1, max(pages))
    bt = np.full((B, maxb), -1, np.int32)
    off = 0
    for b, p in enumerate(pages):
        bt[b, :p] = perm[off:off + p]
        off += p
    qdt = {"bf16": torch.bfloat16, "fp16": torch.float16}[q_dtype]
    kn = torch.from_numpy(rng.standard_normal((B, Sq, H, D)) * 3).to(qdt)
    vn = torch.from_numpy(rng.standard_normal((B, Sq, H, D)) * 0.2).to(qdt)
    if zero_rows:
        kn[0, 0, 0] = 0
        vn[0, Sq - 1, H - 1] = 0
    w = workloads.Workload(name="append", batch=B, max_q_len=Sq, num_q_heads=H,
                           num_kv_heads=H, head_dim=D, block_size=bs, ctx_lo=0, ctx_hi=0,
                           q_dtype=q_dtype, kv_dtype=kv_dtype, scale_mode=scale_mode)
    if kv_dtype == "fp8":
        k = torch.from_numpy(rng.integers(0, 0x7e, size=(nb, bs, H, D), dtype=np.uint8))
        v = torch.from_numpy(rng.integers(0, 0x7e, size=(nb, bs, H, D), dtype=np.uint8))
        if scale_mode == "token":
            ks = torch.from_numpy(rng.uniform(1, 2, size=(nb, bs, H)).astype(np.float32))
            vs = torch.from_numpy(rng.uniform(1, 2, size=(nb, bs, H)).astype(np.float32))
        elif scale_mode == "tensor":
            ks = torch.tensor([0.021], dtype=torch.float32)
            vs = torch.tensor([0.0017], dtype=torch.float32)
        else:
            ks = vs = None
    else:
        k = torch.from_numpy(rng.standard_normal((nb, bs, H, D))).to(qdt)
        v = torch.from_numpy(rng.standard_normal((nb, bs, H, D))).to(qdt)
        ks = vs = None
    inp = dict(workload=w, q=torch.zeros((B, Sq, H, D), dtype=qdt), k_cache=k, v_cache=v,
               k_scale=ks, v_scale=vs, block_tables=torch.from_numpy(bt),
               context_lens=torch.from_numpy(ctx.astype(np.int32)),
               q_lens=torch.from_numpy(ql.astype(np.int32)), sm_scale=1.0)
    return inp, kn, vn


def _targets(inp):
    """(b, i, block, slot) of every appended row, from the block table by hand."""
    bs = inp["workload"].block_size
    out = []
    for b in range(inp["workload"].batch):
        n, ql = int(inp["context_lens"][b]), int(inp["q_lens"][b])
        for i in range(ql):
            pos = n - ql + i
            out.append((b, i, int(inp["block_tables"][b, pos // bs]), pos % bs))
    return out


@pytest.mark.parametrize("kv_dtype,q_dtype", [("bf16", "bf16"), ("fp16", "fp16")])
def test_16bit_append_places_rows_bitwise(kv_dtype, q_dtype):
    inp, kn, vn = random_append_problem(2026, kv_dtype=kv_dtype, q_dtype=q_dtype,
                                        scale_mode="none")
    kc, vc, _, _ = oracle.append_kv(inp, kn, vn)
    k0 = inp["k_cache"].view(torch.int16).clone()
    v0 = inp["v_cache"].view(torch.int16).clone()
    for b, i, blk, slot in _targets(inp):
        k0[blk, slot] = kn[b, i].view(torch.int16)
        v0[blk, slot] = vn[b, i].view(torch.int16)
    assert torch.equal(kc.view(torch.int16), k0)
    assert torch.equal(vc.view(torch.int16), v0)


@pytest.mark.parametrize("scale_mode", ["token", "tensor", "none"])
@pytest.mark.parametrize("q_dtype", ["bf16", "fp16"])
def test_fp8_append_codes_and_scales(scale_mode, q_dtype):
    inp, kn, vn = random_append_problem(2039, scale_mode=scale_mode, q_dtype=q_dtype)
    kc, vc, ks, vs = oracle.append_kv(inp, kn, vn)
    k0, v0 = inp["k_cache"].clone(), inp["v_cache"].clone()
    ks0 = None if inp["k_scale"] is None else inp["k_scale"].clone()
    vs0 = None if inp["v_scale"] is None else inp["v_scale"].clone()
    for b, i, blk, slot in _targets(inp):
        for new, c0, s0, name in ((kn, k0, ks0, "k"), (vn, v0, vs0, "v")):
            x = new[b, i].float()  # [H, D]
            if scale_mode == "token":
                amax = x.abs().amax(dim=-1)
                s = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
                s0[blk, slot] = s
                # the largest magnitude of a non-zero row lands on the code of +-448 (the
                # fp32 quotient amax / (amax / 448) is 448 to within two ulps)
                for h in range(x.shape[0]):
                    if amax[h] > 0:
                        j = int(x[h].abs().argmax())
                        qv = float((x[h, j] / s[h]).abs())
                        assert abs(qv - 448.0) <= 2 * 448.0 * 2.0 ** -23
                        assert oracle.e4m3_encode(float(x[h, j] / s[h])) & 0x7f == 0x7e
            elif scale_mode == "tensor":
                s = s0.expand(x.shape[0])
            else:
                s = torch.ones(x.shape[0])
            c0[blk, slot] = _torch_codes(x / s[:, None])
    assert torch.equal(kc, k0) and torch.equal(vc, v0)
    if scale_mode == "token":
        assert torch.equal(ks, ks0) and torch.equal(vs, vs0)
    elif scale_mode == "tensor":
        assert torch.equal(ks, inp["k_scale"]) and torch.equal(vs, inp["v_scale"])


def test_fp8_append_round_trip_within_half_a_step():
    """Decoding the written codes (the oracle's own, separately pinned decoder) times the
    written scale returns each input within half the E4M3 grid step at that magnitude."""
    inp, kn, vn = random_append_problem(2029, scale_mode="token", batch=3, head_dim=32)
    kc, vc, ks, vs = oracle.append_kv(inp, kn, vn)
    dec = np.array([oracle.e4m3(c) for c in range(256)])
    for b, i, blk, slot in _targets(inp):
        for new, cache, sc in ((kn, kc, ks), (vn, vc, vs)):
            x = new[b, i].double().numpy()
            s = sc[blk, slot].double().numpy()[:, None]
            y = dec[cache[blk, slot].numpy().astype(np.int64)] * s
            a = np.abs(x / s)
            e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
            half_step = 2.0 ** (e - 4) * s
            assert (np.abs(y - x) <= half_step * (1 + 1e-6) + 1e-30).all()


def test_append_rejects_bad_block_id_and_lengths():
    inp, kn, vn = random_append_problem(2026, scale_mode="token")
    bad = dict(inp)
    bad["block_tables"] = inp["block_tables"].clone()
    b, i, _, _ = _targets(inp)[0]
    pos = int(inp["context_lens"][b]) - int(inp["q_lens"][b]) + i
    bad["block_tables"][b, pos // inp["workload"].block_size] = inp["k_cache"].shape[0]
    with pytest.raises(ValueError):
        oracle.append_kv(bad, kn, vn)
    bad = dict(inp)
    bad["context_lens"] = inp["context_lens"].clone()
    bad["context_lens"][0] = int(inp["q_lens"][0]) - 1
    with pytest.raises(ValueError):
        oracle.append_kv(bad, kn, vn)
