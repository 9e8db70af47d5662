"""Inputs the host cannot check (device-resident lengths and block tables) are caught on
the device (GPU), the calls still return OK and pa_read_flags reports what was wrong.  Bad
lengths: the planner empties the work list (output zeros, lse = -inf).  A block id outside
the pool: the decode kernel's range check skips that page (only that sequence's rows are
affected).  Either way no kernel reads outside its inputs."""
import numpy as np
import pytest
import torch

import paged_kv_cache_work_gb300 as pa
import workloads as W
from gpu_run import run

pytestmark = pytest.mark.gpu


def _inputs(device):
    return W.make_inputs(W.reduced(W.GQA_B32, 4, 200, 600), 2026, device=device)


def test_context_shorter_than_new_tokens(cuda_device):
    inp = _inputs(cuda_device)
    inp["q_lens"][2] = 2  # > max_q_len = 1
    out, lse, ws, _ = run(inp)
    assert pa.read_flags(ws) == pa.FLAG_BAD_LENGTHS
    assert torch.all(out == 0) and torch.all(lse == -np.inf)


def test_context_longer_than_block_table(cuda_device):
    inp = _inputs(cuda_device)
    inp["context_lens"][1] = inp["block_tables"].shape[1] * 16 + 1
    out, _, ws, _ = run(inp)
    assert pa.read_flags(ws) == pa.FLAG_BAD_LENGTHS
    assert torch.all(out == 0)


@pytest.mark.parametrize("bad", [-5, 10 ** 7])
def test_block_id_outside_pool(bad, cuda_device):
    inp = _inputs(cuda_device)
    inp["block_tables"][3, 2] = bad
    out, _, ws, _ = run(inp)
    assert pa.read_flags(ws) == pa.FLAG_BAD_BLOCK_ID
    # the other sequences are unaffected by the skipped page
    inp["block_tables"][3, 2] = 0
    ref, _, ws2, _ = run(inp)
    assert pa.read_flags(ws2) == 0
    assert torch.equal(out[:3].view(torch.int16), ref[:3].view(torch.int16))


def test_block_table_changed_after_planning(cuda_device):
    inp = _inputs(cuda_device)
    cfg = pa.config_for(inp)
    q = inp["q"]
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=cuda_device)
    ws = torch.empty(pa.workspace_size(cfg), dtype=torch.uint8, device=cuda_device)
    pa.plan(cfg, inp["block_tables"], inp["context_lens"], inp["q_lens"], ws)
    bt = inp["block_tables"].clone()
    bt[0, 1] = -1
    pa.decode(cfg, q, inp["k_cache"], inp["v_cache"], None, None, bt, inp["context_lens"],
              inp["q_lens"], out, lse, ws)
    pa.reduce(cfg, out, lse, ws)
    assert pa.read_flags(ws) == pa.FLAG_BAD_BLOCK_ID
    # the other sequences are unaffected
    ref, _, ws2, _ = run(inp)
    assert pa.read_flags(ws2) == 0
    assert torch.equal(out[1:].view(torch.int16), ref[1:].view(torch.int16))


def test_flags_reset_by_next_plan(cuda_device):
    inp = _inputs(cuda_device)
    cfg = pa.config_for(inp)
    ws = torch.empty(pa.workspace_size(cfg), dtype=torch.uint8, device=cuda_device)
    good_q = inp["q_lens"].clone()
    inp["q_lens"][0] = 7
    pa.paged_attention(inp, ws=ws, cfg=cfg)
    assert pa.read_flags(ws) == pa.FLAG_BAD_LENGTHS
    inp["q_lens"] = good_q
    pa.paged_attention(inp, ws=ws, cfg=cfg)
    assert pa.read_flags(ws) == 0


def test_lengths_changed_after_planning(cuda_device):
    """The tcgen05 decode derives each CTA's first work item from the lengths and checks it
    against the planner's: lengths changed between pa_plan and pa_decode (shorter, so every
    key the changed plan reaches is still inside its sequence's pages) raise
    PA_FLAG_STALE_PLAN, and nothing is read outside the inputs."""
    wl = W.reduced(W.LONG_SQ4, 3, 3000, 6000)  # 64 query rows per kv head: tcgen05
    inp = W.make_inputs(wl, 2026, device=cuda_device)
    cfg = pa.config_for(inp)
    q = inp["q"]
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=cuda_device)
    ws = torch.empty(pa.workspace_size(cfg), dtype=torch.uint8, device=cuda_device)
    pa.plan(cfg, inp["block_tables"], inp["context_lens"], inp["q_lens"], ws)
    ctx = (inp["context_lens"] // 2).clone()
    pa.decode(cfg, q, inp["k_cache"], inp["v_cache"], None, None, inp["block_tables"], ctx,
              inp["q_lens"], out, lse, ws)
    torch.cuda.synchronize()
    assert pa.read_flags(ws) & pa.FLAG_STALE_PLAN
