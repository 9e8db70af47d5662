"""The C ABI without a GPU: the library loads, exports exactly the calls include/pa.h
declares, and rejects malformed or unsupported configurations on the host with the
documented status codes (no kernel is launched by any of these calls)."""
import ctypes
import os
import re
import subprocess

import pytest

import paged_kv_cache_work_gb300 as pa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa.h")


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(pa.LIB_PATH):
        from paged_kv_cache_work_gb300.build import build
        build()
    return pa.load()


def test_header_declares_the_binding_calls():
    assert declared_functions() == sorted(pa.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_library_exports_nothing_else():
    out = subprocess.run(["nm", "-D", "--defined-only", pa.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    names = sorted({line.split()[-1] for line in out.splitlines() if line.strip()})
    names = [n for n in names if not n.startswith("_") and n not in ("_init", "_fini")]
    assert names == sorted(pa.EXPORTED_SYMBOLS), names


def base_cfg(**kw):
    c = dict(batch=2, max_q_len=1, num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
             max_blocks_per_seq=8, num_blocks=32, q_dtype=pa.BF16, kv_dtype=pa.BF16,
             kv_scale_mode=pa.SCALE_NONE, causal=0, sm_scale=0.088, num_ctas=4, grid_mult=0)
    c.update(kw)
    return pa.PaConfig(**c)


def ws_size(lib, cfg):
    n = ctypes.c_size_t(0)
    st = lib.pa_workspace_size(ctypes.byref(cfg), ctypes.byref(n))
    return st, n.value


def test_workspace_size_for_supported_shapes(lib):
    for D in (64, 128, 256):
        for bs in (16, 32, 64, 128, 256, 512, 1024):
            for kv, sm in ((pa.BF16, 0), (pa.FP8_E4M3, 0), (pa.FP8_E4M3, 1), (pa.FP8_E4M3, 2)):
                st, n = ws_size(lib, base_cfg(head_dim=D, block_size=bs, kv_dtype=kv,
                                              kv_scale_mode=sm))
                assert st == pa.OK and n > 0
    st16, _ = ws_size(lib, base_cfg(q_dtype=pa.FP16, kv_dtype=pa.FP16))
    assert st16 == pa.OK


def test_workspace_grows_with_grid_and_batch(lib):
    _, a = ws_size(lib, base_cfg(num_ctas=4))
    _, b = ws_size(lib, base_cfg(num_ctas=400))
    _, c = ws_size(lib, base_cfg(num_ctas=4, batch=64))
    assert b > a and c > a


@pytest.mark.parametrize("kw,expect", [
    (dict(head_dim=96), pa.ERR_UNSUPPORTED),
    (dict(head_dim=512), pa.ERR_UNSUPPORTED),
    (dict(block_size=8), pa.ERR_UNSUPPORTED),
    (dict(block_size=48), pa.ERR_UNSUPPORTED),
    (dict(block_size=2048), pa.ERR_UNSUPPORTED),
    (dict(num_q_heads=6, num_kv_heads=4), pa.ERR_UNSUPPORTED),
    (dict(q_dtype=pa.FP8_E4M3, kv_dtype=pa.FP8_E4M3), pa.ERR_UNSUPPORTED),
    (dict(q_dtype=pa.BF16, kv_dtype=pa.FP16), pa.ERR_UNSUPPORTED),
    (dict(kv_scale_mode=pa.SCALE_PER_TOKEN), pa.ERR_UNSUPPORTED),
    (dict(batch=0), pa.ERR_INVALID_ARG),
    (dict(max_q_len=0), pa.ERR_INVALID_ARG),
    (dict(num_kv_heads=0), pa.ERR_INVALID_ARG),
    (dict(num_blocks=0), pa.ERR_INVALID_ARG),
    (dict(causal=2), pa.ERR_INVALID_ARG),
    (dict(sm_scale=float("nan")), pa.ERR_INVALID_ARG),
    (dict(sm_scale=float("inf")), pa.ERR_INVALID_ARG),
    (dict(q_dtype=7), pa.ERR_INVALID_ARG),
    (dict(kv_scale_mode=5), pa.ERR_INVALID_ARG),
    (dict(num_ctas=-1), pa.ERR_INVALID_ARG),
    (dict(split_merge=3), pa.ERR_INVALID_ARG),
    (dict(split_merge=-1), pa.ERR_INVALID_ARG),
])
def test_rejections(lib, kw, expect):
    st, _ = ws_size(lib, base_cfg(**kw))
    assert st == expect, pa.status_string(st)


def test_null_arguments_rejected_before_any_launch(lib):
    cfg = base_cfg()
    n = ctypes.c_size_t(0)
    assert lib.pa_workspace_size(None, ctypes.byref(n)) == pa.ERR_INVALID_ARG
    assert lib.pa_workspace_size(ctypes.byref(cfg), None) == pa.ERR_INVALID_ARG
    _, need = ws_size(lib, cfg)
    fake = 1 << 20  # never dereferenced: every call below is rejected on the host
    assert lib.pa_plan(ctypes.byref(cfg), None, fake, fake, fake, need, None) == pa.ERR_INVALID_ARG
    assert lib.pa_plan(ctypes.byref(cfg), fake, fake, fake, None, need, None) == pa.ERR_INVALID_ARG
    assert lib.pa_plan(ctypes.byref(cfg), fake, fake, fake, fake + 8, need, None) == pa.ERR_INVALID_ARG
    assert lib.pa_plan(ctypes.byref(cfg), fake, fake, fake, fake, need - 1, None) == pa.ERR_WORKSPACE
    dec = lambda q, out, ws, nb, ks=None, vs=None, c=cfg: lib.pa_decode(
        ctypes.byref(c), q, fake, fake, ks, vs, fake, fake, fake, out, None, ws, nb, None)
    assert dec(None, fake, fake, need) == pa.ERR_INVALID_ARG
    assert dec(fake + 2, fake, fake, need) == pa.ERR_INVALID_ARG       # q not 16-byte aligned
    assert dec(fake, fake + 8, fake, need) == pa.ERR_INVALID_ARG       # out not aligned
    assert dec(fake, fake, fake, need - 1) == pa.ERR_WORKSPACE
    c8 = base_cfg(kv_dtype=pa.FP8_E4M3, kv_scale_mode=pa.SCALE_PER_TENSOR)
    _, need8 = ws_size(lib, c8)
    assert dec(fake, fake, fake, need8, None, fake, c8) == pa.ERR_INVALID_ARG  # missing scale
    assert lib.pa_reduce(ctypes.byref(cfg), None, None, fake, need, None) == pa.ERR_INVALID_ARG
    assert lib.pa_reduce(ctypes.byref(cfg), fake, None, fake, need - 1, None) == pa.ERR_WORKSPACE
    f = ctypes.c_int32(0)
    assert lib.pa_read_flags(None, 1024, ctypes.byref(f), None) == pa.ERR_INVALID_ARG
    assert lib.pa_read_flags(fake, 1024, None, None) == pa.ERR_INVALID_ARG


def test_gather_arguments_rejected_before_any_launch(lib):
    fake = 1 << 20  # never dereferenced: every call below is rejected on the host
    g = lambda c, kc=fake, vc=fake, bt=fake, cl=fake, ko=fake, vo=fake, rows=1000: \
        lib.pa_gather_kv(ctypes.byref(c), kc, vc, bt, cl, ko, vo, rows, None, None, None)
    cfg = base_cfg()
    assert lib.pa_gather_kv(None, fake, fake, fake, fake, fake, fake, 10, None, None,
                            None) == pa.ERR_INVALID_ARG
    for kw in (dict(kc=None), dict(vc=None), dict(bt=None), dict(cl=None), dict(ko=None),
               dict(vo=None)):
        assert g(cfg, **kw) == pa.ERR_INVALID_ARG, kw
    assert g(cfg, kc=fake + 8) == pa.ERR_INVALID_ARG   # cache not 16-byte aligned
    assert g(cfg, vo=fake + 4) == pa.ERR_INVALID_ARG   # output not aligned
    assert g(cfg, rows=-1) == pa.ERR_INVALID_ARG
    assert g(base_cfg(head_dim=96)) == pa.ERR_UNSUPPORTED
    assert g(base_cfg(block_size=24)) == pa.ERR_UNSUPPORTED
    assert g(base_cfg(batch=8193)) == pa.ERR_UNSUPPORTED
    assert g(base_cfg(batch=0)) == pa.ERR_INVALID_ARG


def test_status_strings(lib):
    seen = set()
    for s in range(6):
        txt = pa.status_string(s)
        assert txt and txt != "unknown status"
        seen.add(txt)
    assert len(seen) == 6
    assert pa.status_string(99) == "unknown status"


def test_binding_raises_on_missing_library(tmp_path):
    saved = pa._lib
    pa._lib = None
    try:
        with pytest.raises(RuntimeError):
            pa.load(str(tmp_path / "missing.so"))
    finally:
        pa._lib = saved
