"""ctypes wrapper of the CPU oracle for paged-attention decode (``pa_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the bench's
CPU-baseline leg may use this module; the product path never imports it.  It
does not import the CUDA package either: the two sides meet only in the seeded
inputs drawn by ``workloads.py``.

Two builds of the same C source are loaded: ``precision="f32"`` (every sum,
exp and log in float, the CPU FP32 reference of the pages' correctness check)
and ``precision="f64"`` (double, used to pin the float build).
"""
from __future__ import annotations

import contextlib
import ctypes
import os
from typing import Optional

import numpy as np
import torch

from .build import LIBS, build as _build

_HERE = os.path.dirname(os.path.abspath(__file__))

_DTYPE_CODE = {"bf16": 0, "fp16": 1, "fp8": 2}
_SCALE_CODE = {"none": 0, "tensor": 1, "token": 2}


class OracleCfg(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "max_q_len", "num_q_heads", "num_kv_heads", "head_dim", "block_size",
        "max_blocks_per_seq", "num_blocks", "q_dtype", "kv_dtype", "scale_mode", "causal")] + [
        ("sm_scale", ctypes.c_double)]


_libs: dict = {}
_lib_dir = _HERE


@contextlib.contextmanager
def libs_from(directory: str):
    """Load the oracle from another build directory for the duration of the block
    (the planted-mistake tests use this to run the pins against a patched build)."""
    global _libs, _lib_dir
    saved = (_libs, _lib_dir)
    _libs, _lib_dir = {}, directory
    try:
        yield
    finally:
        _libs, _lib_dir = saved


def lib(precision: str = "f32"):
    """Load (building on first use if needed) the oracle shared library."""
    if precision not in _libs:
        path = os.path.join(_lib_dir, LIBS[precision])
        if not os.path.exists(path):
            if _lib_dir != _HERE:
                raise FileNotFoundError(path)
            _build()
        L = ctypes.CDLL(path)
        vp, i32p = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)
        real = ctypes.c_float if precision == "f32" else ctypes.c_double
        rp = ctypes.POINTER(real)
        fp = ctypes.POINTER(ctypes.c_float)
        cp = ctypes.POINTER(OracleCfg)
        L.oracle_real_bytes.restype = ctypes.c_int
        L.oracle_decode.argtypes = [cp, vp, vp, vp, fp, fp, i32p, i32p, i32p, ctypes.c_int, rp, rp]
        L.oracle_decode.restype = ctypes.c_int
        L.oracle_decode_rows.argtypes = [cp, vp, vp, vp, fp, fp, i32p, i32p, i32p, ctypes.c_int,
                                         i32p, rp, rp]
        L.oracle_decode_rows.restype = ctypes.c_int
        L.oracle_attend_range.argtypes = [cp, vp, vp, vp, fp, fp, i32p, i32p, i32p, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          rp, rp]
        L.oracle_attend_range.restype = ctypes.c_int
        L.oracle_merge.argtypes = [ctypes.c_int, ctypes.c_int, rp, rp, rp, rp]
        L.oracle_merge.restype = None
        for name in ("oracle_bf16", "oracle_fp16"):
            getattr(L, name).argtypes = [ctypes.c_uint16]
            getattr(L, name).restype = real
        L.oracle_e4m3.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3.restype = real
        L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        L.oracle_e4m3_encode.restype = ctypes.c_uint8
        L.oracle_append_kv.argtypes = [cp, vp, vp, i32p, i32p, i32p, vp, vp, fp, fp]
        L.oracle_append_kv.restype = ctypes.c_int
        assert L.oracle_real_bytes() == (4 if precision == "f32" else 8)
        _libs[precision] = (L, real)
    return _libs[precision]


def _np_real(precision):
    return np.float32 if precision == "f32" else np.float64


def _host(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return t.detach().cpu().contiguous()


def _ptr(t: Optional[torch.Tensor], ctype=ctypes.c_void_p):
    if t is None:
        return None
    if ctype is ctypes.c_void_p:
        return ctypes.c_void_p(t.data_ptr())
    return ctypes.cast(t.data_ptr(), ctypes.POINTER(ctype))


class _Prepared:
    """Host copies of one problem's tensors, kept alive for the duration of a call."""

    def __init__(self, inp: dict):
        w = inp["workload"]
        self.w = w
        self.q = _host(inp["q"])
        self.k = _host(inp["k_cache"])
        self.v = _host(inp["v_cache"])
        self.ks = _host(inp.get("k_scale"))
        self.vs = _host(inp.get("v_scale"))
        self.bt = _host(inp["block_tables"]).to(torch.int32)
        self.ctx = _host(inp["context_lens"]).to(torch.int32)
        self.ql = _host(inp["q_lens"]).to(torch.int32)
        if self.ks is not None:
            self.ks = self.ks.float()
            self.vs = self.vs.float()
        # The library takes sm_scale as an fp32 argument; hand the oracle the same value.
        sm = float(np.float32(inp["sm_scale"]))
        self.cfg = OracleCfg(w.batch, w.max_q_len, w.num_q_heads, w.num_kv_heads, w.head_dim,
                             w.block_size, self.bt.shape[1], self.k.shape[0],
                             _DTYPE_CODE[w.q_dtype], _DTYPE_CODE[w.kv_dtype],
                             _SCALE_CODE[w.scale_mode if w.kv_dtype == "fp8" else "none"],
                             int(w.causal), sm)

    def args(self):
        f = ctypes.c_float
        i = ctypes.c_int32
        return (ctypes.byref(self.cfg), _ptr(self.q), _ptr(self.k), _ptr(self.v),
                _ptr(self.ks, f), _ptr(self.vs, f), _ptr(self.bt, i), _ptr(self.ctx, i),
                _ptr(self.ql, i))


def decode(inp: dict, precision: str = "f32", nsplit: int = 0):
    """Every output row of one problem.

    Returns (out [B, Sq, Hq, D], lse [B, Sq, Hq]) as numpy arrays of the oracle's
    precision.  ``nsplit > 1`` computes each row as that many key ranges merged by
    the log-sum-exp rule (used to pin the merge)."""
    L, real = lib(precision)
    p = _Prepared(inp)
    w = p.w
    out = np.empty((w.batch, w.max_q_len, w.num_q_heads, w.head_dim), _np_real(precision))
    lse = np.empty((w.batch, w.max_q_len, w.num_q_heads), _np_real(precision))
    rc = L.oracle_decode(*p.args(), int(nsplit), out.ctypes.data_as(ctypes.POINTER(real)),
                         lse.ctypes.data_as(ctypes.POINTER(real)))
    if rc != 0:
        raise ValueError(f"oracle_decode rejected the problem (code {rc})")
    return out, lse


def decode_rows(inp: dict, rows_bih, precision: str = "f32"):
    """Selected rows only: ``rows_bih`` is an (n, 3) int array of (b, i, h)."""
    L, real = lib(precision)
    p = _Prepared(inp)
    rows = np.ascontiguousarray(np.asarray(rows_bih, dtype=np.int32).reshape(-1, 3))
    n = rows.shape[0]
    out = np.empty((n, p.w.head_dim), _np_real(precision))
    lse = np.empty((n,), _np_real(precision))
    rc = L.oracle_decode_rows(*p.args(), n, rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                              out.ctypes.data_as(ctypes.POINTER(real)),
                              lse.ctypes.data_as(ctypes.POINTER(real)))
    if rc != 0:
        raise ValueError(f"oracle_decode_rows rejected the problem (code {rc})")
    return out, lse


def attend_range(inp: dict, b: int, i: int, h: int, j0: int, j1: int, precision: str = "f32"):
    """Partial result (o, lse) of row (b, i, h) over keys [j0, j1) of its visible keys."""
    L, real = lib(precision)
    p = _Prepared(inp)
    o = np.empty((p.w.head_dim,), _np_real(precision))
    lse = np.empty((1,), _np_real(precision))
    rc = L.oracle_attend_range(*p.args(), b, i, h, j0, j1, o.ctypes.data_as(ctypes.POINTER(real)),
                               lse.ctypes.data_as(ctypes.POINTER(real)))
    if rc != 0:
        raise ValueError(f"oracle_attend_range rejected the problem (code {rc})")
    return o, float(lse[0])


def merge(o_s: np.ndarray, lse_s: np.ndarray, precision: str = "f64"):
    """LSE merge of partials: o_s (n, D), lse_s (n,)."""
    L, real = lib(precision)
    t = _np_real(precision)
    o_s = np.ascontiguousarray(o_s, dtype=t)
    lse_s = np.ascontiguousarray(lse_s, dtype=t)
    n, D = o_s.shape
    o = np.empty((D,), t)
    lse = np.empty((1,), t)
    P = ctypes.POINTER(real)
    L.oracle_merge(n, D, o_s.ctypes.data_as(P), lse_s.ctypes.data_as(P), o.ctypes.data_as(P),
                   lse.ctypes.data_as(P))
    return o, float(lse[0])


def e4m3(code: int, precision: str = "f64") -> float:
    return float(lib(precision)[0].oracle_e4m3(code))


def e4m3_encode(x: float, precision: str = "f64") -> int:
    """OCP E4M3 code of the float32 value x: clamped to +-448, nearest grid point, ties to
    the even code (the encoding step of the quantise-on-write append)."""
    return int(lib(precision)[0].oracle_e4m3_encode(float(np.float32(x))))


def bf16(bits: int, precision: str = "f64") -> float:
    return float(lib(precision)[0].oracle_bf16(bits))


def fp16(bits: int, precision: str = "f64") -> float:
    return float(lib(precision)[0].oracle_fp16(bits))


def threads() -> int:
    """Host threads the oracle's OpenMP loops use (OMP_NUM_THREADS, else the affinity mask)."""
    env = os.environ.get("OMP_NUM_THREADS")
    if env and env.isdigit():
        return int(env)
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


__all__ = ["decode", "decode_rows", "attend_range", "merge", "e4m3", "e4m3_encode", "bf16",
           "fp16", "lib", "libs_from", "threads", "gather_kv", "append_kv"]


def gather_kv(inp: dict):
    """Paged -> contiguous copy of every cached token's K and V rows (the copy from the paged
    KV cache into the attention's workspace, "HSTU Paged Attention" K/V double-buffering
    issue, background section), written out from its definition: sequence b's token j,
    0 <= j < context_lens[b], is row j % block_size of block block_tables[b][j // block_size],
    and the sequences follow one another in batch order.

    Returns (k_rows, v_rows, row_offsets): the rows as the cache stores them (numpy arrays of
    the cache's element bits, [total_tokens, Hkv, D]) and the int64 offsets [B + 1]."""
    w = inp["workload"]
    bs = w.block_size
    bt = inp["block_tables"].cpu().numpy()
    ctx = inp["context_lens"].cpu().numpy().astype(np.int64)
    out = []
    for name in ("k_cache", "v_cache"):
        cache = inp[name].detach().cpu().contiguous()
        bits = cache.view(torch.uint8) if cache.element_size() == 1 else cache.view(torch.int16)
        cache_np = bits.numpy()
        parts = []
        for b in range(len(ctx)):
            j = np.arange(ctx[b])
            parts.append(cache_np[bt[b][j // bs], j % bs])
        out.append(np.concatenate(parts, axis=0) if parts else cache_np[:0, 0])
    offsets = np.concatenate([[0], np.cumsum(ctx)])
    return out[0], out[1], offsets


def append_kv(inp: dict, k_new: torch.Tensor, v_new: torch.Tensor, precision: str = "f64"):
    """Quantise-on-write KV append, written out from its definition in pa_oracle.c: new row
    i < q_lens[b] of sequence b (k_new / v_new [B, Sq, Hkv, D] in the query dtype) goes to
    position context_lens[b] - q_lens[b] + i of that sequence, i.e. slot pos % block_size of
    block block_tables[b][pos // block_size]; an fp8 cache receives E4M3 codes of the row over
    its scale (per-token scales amax/448 are written too; a per-tensor scale is read).

    ``inp`` holds the cache as workloads.make_inputs lays it out.  Returns new host tensors
    (k_cache, v_cache, k_scale, v_scale); the inputs are not modified."""
    L, _ = lib(precision)
    w = inp["workload"]
    cfg = _Prepared(inp).cfg
    kc = _host(inp["k_cache"]).clone()
    vc = _host(inp["v_cache"]).clone()
    ks = _host(inp.get("k_scale"))
    vs = _host(inp.get("v_scale"))
    ks = None if ks is None else ks.float().clone()
    vs = None if vs is None else vs.float().clone()
    kn = _host(k_new)
    vn = _host(v_new)
    qdt = {"bf16": torch.bfloat16, "fp16": torch.float16}[w.q_dtype]
    assert kn.dtype == qdt and vn.dtype == qdt, "new rows are in the query dtype"
    assert tuple(kn.shape) == (w.batch, w.max_q_len, w.num_kv_heads, w.head_dim)
    bt = _host(inp["block_tables"]).to(torch.int32)
    ctx = _host(inp["context_lens"]).to(torch.int32)
    ql = _host(inp["q_lens"]).to(torch.int32)
    i32 = ctypes.c_int32
    f = ctypes.c_float
    rc = L.oracle_append_kv(ctypes.byref(cfg), _ptr(kn), _ptr(vn), _ptr(bt, i32), _ptr(ctx, i32),
                            _ptr(ql, i32), _ptr(kc), _ptr(vc), _ptr(ks, f), _ptr(vs, f))
    if rc != 0:
        raise ValueError(f"oracle_append_kv rejected the problem (code {rc})")
    return kc, vc, ks, vs
