"""The planner's integer division by a runtime divisor (plan.cu, div_small): floor(x / d)
from the float estimate x * rd, rd a reciprocal of d within one ulp (the approximate
reciprocal instruction's bound), truncated and corrected by one either way.  The claim is
that this is exact for 0 <= x, d < 2^31 with a quotient below 2^21, whichever float within
one ulp of 1/d the reciprocal returns; numpy's float32 arithmetic is IEEE round-to-nearest,
so the same steps run here with each of the three candidates (the correctly rounded
reciprocal and its two neighbours) and are checked against exact integer division, on random
operands and on the boundaries where the estimate is closest to an integer
(x = q d - 1, q d, q d + d - 1), up to the largest quotients and divisors allowed."""
import numpy as np


def div_small(x: np.ndarray, d: np.ndarray, ulp: int) -> np.ndarray:
    xf = x.astype(np.float32)                        # round to nearest
    rd = np.float32(1.0) / d.astype(np.float32)      # correctly rounded reciprocal
    if ulp:                                          # a neighbour, one ulp away
        rd = np.nextafter(rd, np.float32(np.inf if ulp > 0 else 0.0))
    q = np.trunc(xf * rd).astype(np.int64)           # product rounded, then truncated
    qd = q * d
    q = np.where(qd > x, q - 1, np.where(x - qd >= d, q + 1, q))
    return q


def _check(x, d):
    x = np.asarray(x, np.int64)
    d = np.asarray(d, np.int64)
    ok = (x >= 0) & (x < 2**31) & (d > 0) & (d < 2**31) & (x // d < 2**21)
    x, d = x[ok], d[ok]
    for ulp in (-1, 0, 1):
        got = div_small(x, d, ulp)
        bad = np.nonzero(got != x // d)[0]
        assert bad.size == 0, f"ulp {ulp}: x={x[bad[:5]]} d={d[bad[:5]]} got={got[bad[:5]]}"
    return x.size


def test_random_operands():
    rng = np.random.default_rng(7)
    n = 0
    for dmax in (2**4, 2**10, 2**16, 2**24, 2**31 - 1):
        d = rng.integers(1, dmax, size=200_000, dtype=np.int64)
        q = rng.integers(0, 2**21, size=d.size, dtype=np.int64)
        x = np.minimum(q * d + rng.integers(0, d, dtype=np.int64), 2**31 - 1)
        n += _check(x, d)
    assert n > 500_000


def test_boundaries():
    rng = np.random.default_rng(8)
    q = np.concatenate([np.arange(0, 4096), 2**21 - 1 - np.arange(0, 4096),
                        rng.integers(0, 2**21, size=20_000)]).astype(np.int64)
    for d in (1, 2, 3, 7, 128, 1000, 4096, 65535, 1 << 20, (1 << 24) + 1, 2**31 - 1):
        d = np.full(q.shape, d, np.int64)
        for off in (-1, 0, 1):
            _check(q * d + off, d)
        _check(q * d + d - 1, d)
    # divisors near 2^31 / q for large q: the products the correction forms stay below 2^32
    qq = 2**21 - 1 - np.arange(0, 2000, dtype=np.int64)
    dd = (2**31 - 1) // qq
    for off in (-1, 0, 1):
        _check(qq * dd + off, dd)
