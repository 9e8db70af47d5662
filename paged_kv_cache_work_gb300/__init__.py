"""Paged-attention decode on GB300: Python binding of libpa103.so (include/pa.h).

This module only marshals arguments: every step of the decode (planning, page gather,
attention, split merge) runs in the library's CUDA kernels.  PyTorch tensors supply the
device memory and the current stream.  If the library has not been built the first call
raises; there is no fallback.

Build the library with ``python -m paged_kv_cache_work_gb300.build`` (or
``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

__all__ = ["PaConfig", "PaError", "load", "workspace_size", "plan", "decode", "reduce",
           "decode_step_static", "STATIC_SCRATCH_BYTES", "append_kv", "gather_kv",
           "read_flags", "status_string", "config_for", "paged_attention", "LIB_PATH",
           "BF16", "FP16", "FP8_E4M3", "SCALE_NONE", "SCALE_PER_TENSOR", "SCALE_PER_TOKEN",
           "FLAG_BAD_LENGTHS", "FLAG_BAD_BLOCK_ID", "FLAG_WAIT_TIMEOUT", "FLAG_STALE_PLAN",
           "EXPORTED_SYMBOLS",
           "MERGE_AUTO", "MERGE_IN_DECODE", "MERGE_IN_REDUCE"]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpa103.so")

# pa_status
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_DEVICE = range(6)
# pa_dtype, pa_scale_mode, flags
BF16, FP16, FP8_E4M3 = 0, 1, 2
SCALE_NONE, SCALE_PER_TENSOR, SCALE_PER_TOKEN = 0, 1, 2
FLAG_BAD_LENGTHS, FLAG_BAD_BLOCK_ID, FLAG_WAIT_TIMEOUT, FLAG_STALE_PLAN = 1, 2, 4, 8
MERGE_AUTO, MERGE_IN_DECODE, MERGE_IN_REDUCE = 0, 1, 2

EXPORTED_SYMBOLS = ("pa_workspace_size", "pa_plan", "pa_decode", "pa_reduce", "pa_read_flags",
                    "pa_status_string", "pa_decode_step_static", "pa_gather_kv", "pa_append_kv")

# Bytes of the device array behind pa_decode_step_static (PA_STATIC_SCRATCH_BYTES).
STATIC_SCRATCH_BYTES = 16 << 20


class PaConfig(ctypes.Structure):
    """Mirror of pa_config."""
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "max_q_len", "num_q_heads", "num_kv_heads", "head_dim", "block_size",
        "max_blocks_per_seq", "num_blocks", "q_dtype", "kv_dtype", "kv_scale_mode", "causal")] + [
        ("sm_scale", ctypes.c_float), ("num_ctas", ctypes.c_int32), ("grid_mult", ctypes.c_int32),
        ("split_merge", ctypes.c_int32)]


class PaError(RuntimeError):
    def __init__(self, call: str, status: int):
        super().__init__(f"{call}: {status_string(status)} (status {status})")
        self.status = status


_lib = None


def load(path: str = LIB_PATH):
    """Load the library (once).  Raises if it is missing: there is no CPU fallback."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built; run python -m paged_kv_cache_work_gb300.build")
    L = ctypes.CDLL(path)
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    cfgp = ctypes.POINTER(PaConfig)
    L.pa_workspace_size.argtypes = [cfgp, ctypes.POINTER(sz)]
    L.pa_plan.argtypes = [cfgp, vp, vp, vp, vp, sz, vp]
    L.pa_decode.argtypes = [cfgp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.pa_reduce.argtypes = [cfgp, vp, vp, vp, sz, vp]
    L.pa_read_flags.argtypes = [vp, sz, ctypes.POINTER(ctypes.c_int32), vp]
    for f in ("pa_workspace_size", "pa_plan", "pa_decode", "pa_reduce", "pa_read_flags"):
        getattr(L, f).restype = ctypes.c_int
    L.pa_decode_step_static.argtypes = [cfgp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.pa_decode_step_static.restype = ctypes.c_int
    L.pa_gather_kv.argtypes = [cfgp, vp, vp, vp, vp, vp, vp, ctypes.c_int64, vp, vp, vp]
    L.pa_gather_kv.restype = ctypes.c_int
    L.pa_append_kv.argtypes = [cfgp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.pa_append_kv.restype = ctypes.c_int
    L.pa_status_string.argtypes = [ctypes.c_int]
    L.pa_status_string.restype = ctypes.c_char_p
    _lib = L
    return L


def status_string(status: int) -> str:
    return load().pa_status_string(int(status)).decode()


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(call: str, status: int):
    if status != OK:
        raise PaError(call, status)


def workspace_size(cfg: PaConfig) -> int:
    n = ctypes.c_size_t(0)
    _check("pa_workspace_size", load().pa_workspace_size(ctypes.byref(cfg), ctypes.byref(n)))
    return n.value


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def plan(cfg: PaConfig, block_tables, context_lens, q_lens, ws, stream=None):
    _check("pa_plan", load().pa_plan(ctypes.byref(cfg), _ptr(block_tables), _ptr(context_lens),
                                     _ptr(q_lens), _ptr(ws), _nbytes(ws), _stream(stream)))


def decode(cfg: PaConfig, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
           q_lens, out, lse, ws, stream=None):
    _check("pa_decode", load().pa_decode(
        ctypes.byref(cfg), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
        _ptr(block_tables), _ptr(context_lens), _ptr(q_lens), _ptr(out), _ptr(lse), _ptr(ws),
        _nbytes(ws), _stream(stream)))


def reduce(cfg: PaConfig, out, lse, ws, stream=None):
    _check("pa_reduce", load().pa_reduce(ctypes.byref(cfg), _ptr(out), _ptr(lse), _ptr(ws),
                                         _nbytes(ws), _stream(stream)))


def read_flags(ws, stream=None) -> int:
    """Synchronise and return the device flags of the last step run in ``ws``."""
    f = ctypes.c_int32(0)
    st = load().pa_read_flags(_ptr(ws), _nbytes(ws), ctypes.byref(f), _stream(stream))
    if st not in (OK, ERR_DEVICE):
        raise PaError("pa_read_flags", st)
    return f.value


def decode_step_static(cfg: PaConfig, q, k_cache, v_cache, k_scale, v_scale, block_tables,
                       context_lens, q_lens, out, lse, stream=None):
    """One decode step on the library's static device scratch, for callers that cannot
    allocate device memory (no workspace argument; see pa_decode_step_static in pa.h)."""
    _check("pa_decode_step_static", load().pa_decode_step_static(
        ctypes.byref(cfg), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
        _ptr(block_tables), _ptr(context_lens), _ptr(q_lens), _ptr(out), _ptr(lse),
        _stream(stream)))


def gather_kv(cfg: PaConfig, k_cache, v_cache, block_tables, context_lens, k_out, v_out,
              max_rows: int, row_offsets=None, flags=None, stream=None):
    """Paged -> contiguous copy of the batch's K and V rows (see pa_gather_kv in pa.h):
    sequence b lands at rows row_offsets[b] .. row_offsets[b + 1] - 1 of k_out and v_out."""
    _check("pa_gather_kv", load().pa_gather_kv(
        ctypes.byref(cfg), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        _ptr(k_out), _ptr(v_out), int(max_rows), _ptr(row_offsets), _ptr(flags),
        _stream(stream)))


def append_kv(cfg: PaConfig, k_new, v_new, block_tables, context_lens, q_lens, k_cache, v_cache,
              k_scale=None, v_scale=None, flags=None, stream=None):
    """Write a step's new K/V rows into their pages, quantised to fp8 for an fp8 cache (see
    pa_append_kv in pa.h): new row i of sequence b lands at position
    context_lens[b] - q_lens[b] + i.  Per-token scales are written into k_scale / v_scale."""
    _check("pa_append_kv", load().pa_append_kv(
        ctypes.byref(cfg), _ptr(k_new), _ptr(v_new), _ptr(block_tables), _ptr(context_lens),
        _ptr(q_lens), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(flags),
        _stream(stream)))


_DT = {"bf16": BF16, "fp16": FP16, "fp8": FP8_E4M3}
_SM = {"none": SCALE_NONE, "tensor": SCALE_PER_TENSOR, "token": SCALE_PER_TOKEN}


def config_for(inp: dict, num_ctas: int = 0, grid_mult: int = 0,
               split_merge: int = MERGE_AUTO) -> PaConfig:
    """pa_config of a problem laid out as workloads.make_inputs returns it.  With neither a
    grid size nor a multiplier given and the inputs on a GPU, the multiplier comes from the
    tuned table (grid_tune.lookup: 1 for shapes it does not list)."""
    w = inp["workload"]
    cfg = PaConfig(batch=w.batch, max_q_len=w.max_q_len, num_q_heads=w.num_q_heads,
                   num_kv_heads=w.num_kv_heads, head_dim=w.head_dim, block_size=w.block_size,
                   max_blocks_per_seq=inp["block_tables"].shape[1],
                   num_blocks=inp["k_cache"].shape[0], q_dtype=_DT[w.q_dtype],
                   kv_dtype=_DT[w.kv_dtype],
                   kv_scale_mode=_SM[w.scale_mode] if w.kv_dtype == "fp8" else SCALE_NONE,
                   causal=int(w.causal), sm_scale=float(inp["sm_scale"]), num_ctas=num_ctas,
                   grid_mult=grid_mult, split_merge=split_merge)
    q = inp["q"]
    if num_ctas == 0 and grid_mult == 0 and getattr(q, "is_cuda", False):
        import torch
        from . import grid_tune
        sms = torch.cuda.get_device_properties(q.device).multi_processor_count
        cfg.grid_mult = grid_tune.lookup(cfg, sms)
    return cfg


def paged_attention(inp: dict, out=None, lse=None, ws=None, cfg: Optional[PaConfig] = None,
                    stream=None):
    """One decode step (plan, decode, reduce) on tensors already on the GPU.

    Allocates out [B, Sq, Hq, D], lse [B, Sq, Hq] and the workspace with torch when they are
    not given.  Returns (out, lse, ws)."""
    import torch
    cfg = cfg if cfg is not None else config_for(inp)
    q = inp["q"]
    dev = q.device
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    if ws is None:
        ws = torch.empty(workspace_size(cfg), dtype=torch.uint8, device=dev)
    plan(cfg, inp["block_tables"], inp["context_lens"], inp["q_lens"], ws, stream)
    decode(cfg, q, inp["k_cache"], inp["v_cache"], inp.get("k_scale"), inp.get("v_scale"),
           inp["block_tables"], inp["context_lens"], inp["q_lens"], out, lse, ws, stream)
    reduce(cfg, out, lse, ws, stream)
    return out, lse, ws
