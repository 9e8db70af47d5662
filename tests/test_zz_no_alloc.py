"""pa_decode_step_static: the decode step for callers that cannot allocate device memory
(a plugin or framework interface without an allocator, a serving loop that must not call
cudaMalloc after start-up, or code under stream capture).  It keeps its scratch in a
static device array inside the library.  Checked here (GPU) through the C ABI against the
workspace-based entry points and against the CPU oracle, within the parity tolerances, on
two calls in a row; and a problem too large for the static array is refused before anything
runs.

This file is collected last on purpose: the entry point's first call on a device looks the
array up, and the test must pass both alone in a fresh process and after every other test.
"""
import ctypes

import pytest
import torch

import oracle
import paged_kv_cache_work_gb300 as pa
import workloads as W
from gpu_run import compare

pytestmark = pytest.mark.gpu

CASES = [W.reduced(W.GQA_B32, 6, 300, 2500), W.reduced(W.LONG_SQ1, 2, 3000, 9000),
         W.reduced(W.FP8_TOKEN_SQ1, 4, 1000, 4000), W.reduced(W.mha_d256(8, 4), 3, 200, 1500),
         W.reduced(W.mha_d256(8, 16), 2, 200, 900)]


def _static_call(lib, cfg, inp, out, lse):
    return lib.pa_decode_step_static(
        ctypes.byref(cfg), inp["q"].data_ptr(), inp["k_cache"].data_ptr(),
        inp["v_cache"].data_ptr(),
        None if inp["k_scale"] is None else inp["k_scale"].data_ptr(),
        None if inp["v_scale"] is None else inp["v_scale"].data_ptr(),
        inp["block_tables"].data_ptr(), inp["context_lens"].data_ptr(),
        inp["q_lens"].data_ptr(), out.data_ptr(), lse.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_static_step_matches_workspace_step_twice(wl, cuda_device):
    lib = pa.load()
    inp = W.make_inputs(wl, 2029, device=cuda_device)
    cfg = pa.config_for(inp)
    assert pa.workspace_size(cfg) <= pa.STATIC_SCRATCH_BYTES
    ref_out, ref_lse, _ = pa.paged_attention(inp, cfg=cfg)
    torch.cuda.synchronize()
    ref_out = ref_out.float().cpu().numpy()
    ref_lse = ref_lse.cpu().numpy()
    orc_out, orc_lse = oracle.decode(W.to_device(inp, "cpu"), "f32")
    for _ in range(2):
        out = torch.full_like(inp["q"], float("nan"))
        lse = torch.full(inp["q"].shape[:3], float("nan"), dtype=torch.float32,
                         device=cuda_device)
        assert _static_call(lib, cfg, inp, out, lse) == pa.OK
        torch.cuda.synchronize()
        compare(out, lse, ref_out, ref_lse, wl.kv_dtype)
        compare(out, lse, orc_out, orc_lse, wl.kv_dtype)


def test_static_step_refuses_problems_beyond_its_scratch(cuda_device):
    lib = pa.load()
    inp = W.make_inputs(W.reduced(W.GQA_B32, 2, 16, 64), 2026, device=cuda_device)
    cfg = pa.config_for(inp)
    while pa.workspace_size(cfg) <= pa.STATIC_SCRATCH_BYTES:
        cfg.batch *= 2  # the work list grows with the batch until it no longer fits
    assert cfg.batch > inp["workload"].batch
    out = torch.empty(1, device=cuda_device)
    lse = torch.empty(1, device=cuda_device)
    assert _static_call(lib, cfg, inp, out, lse) == pa.ERR_WORKSPACE
