"""Bitwise determinism (GPU): two eager calls, and a CUDA-graph capture of the whole step
(plan, decode, reduce) replayed, give identical bytes.  The RecSDK HSTU paged-attention
issue (1281, correctness section) asks the same of its kernel: eager repeats and
eager-vs-graph runs bitwise equal.  The work list is fixed per input and no float atomics
are used, so this holds by construction."""
import pytest
import torch

import paged_kv_cache_work_gb300 as pa
import workloads as W

pytestmark = pytest.mark.gpu

CASES = [W.reduced(W.GQA_B32, 8, 300, 3000), W.reduced(W.LONG_SQ4, 2, 20000, 40000),
         W.reduced(W.FP8_TOKEN_SQ4, 4, 2000, 5000), W.reduced(W.mha_d256(8, 4), 4, 500, 3000),
         # the tcgen05 kernel at head dim 256 and with an fp8 cache
         W.reduced(W.mha_d256(8, 64), 3, 500, 3000), W.reduced(W.FP8_TENSOR_SQ4, 4, 2000, 5000)]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_eager_repeat_and_graph_replay_bitwise(wl, cuda_device):
    inp = W.make_inputs(wl, 2026, device=cuda_device)
    cfg = pa.config_for(inp)
    q = inp["q"]
    ws = torch.empty(pa.workspace_size(cfg), dtype=torch.uint8, device=cuda_device)
    outs = []
    for _ in range(2):
        out = torch.empty_like(q)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=cuda_device)
        pa.paged_attention(inp, out=out, lse=lse, ws=ws, cfg=cfg)
        outs.append((out, lse))
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0].view(torch.int16), outs[1][0].view(torch.int16))
    assert torch.equal(outs[0][1].view(torch.int32), outs[1][1].view(torch.int32))

    g_out = torch.empty_like(q)
    g_lse = torch.empty(q.shape[:3], dtype=torch.float32, device=cuda_device)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            pa.paged_attention(inp, out=g_out, lse=g_lse, ws=ws, cfg=cfg, stream=s)
    for _ in range(2):
        g_out.zero_()
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0].view(torch.int16), g_out.view(torch.int16))
    assert torch.equal(outs[0][1].view(torch.int32), g_lse.view(torch.int32))
    assert pa.read_flags(ws) == 0


@pytest.mark.parametrize("mode", ["auto", "in_decode", "in_reduce"])
@pytest.mark.parametrize("wl", CASES[:2], ids=lambda w: w.name)
def test_decode_repeats_on_one_plan(wl, mode, cuda_device):
    """pa_plan once, then decode + reduce twice: the merge counters the last CTA of each unit
    sets back to zero let the second decode merge exactly like the first."""
    sm = {"auto": pa.MERGE_AUTO, "in_decode": pa.MERGE_IN_DECODE,
          "in_reduce": pa.MERGE_IN_REDUCE}[mode]
    inp = W.make_inputs(wl, 2029, device=cuda_device)
    cfg = pa.config_for(inp, split_merge=sm)
    q = inp["q"]
    ws = torch.empty(pa.workspace_size(cfg), dtype=torch.uint8, device=cuda_device)
    pa.plan(cfg, inp["block_tables"], inp["context_lens"], inp["q_lens"], ws)
    outs = []
    for _ in range(2):
        out = torch.full_like(q, float("nan"))
        lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device=cuda_device)
        pa.decode(cfg, q, inp["k_cache"], inp["v_cache"], inp["k_scale"], inp["v_scale"],
                  inp["block_tables"], inp["context_lens"], inp["q_lens"], out, lse, ws)
        pa.reduce(cfg, out, lse, ws)
        outs.append((out, lse))
    torch.cuda.synchronize()
    assert not torch.isnan(outs[0][0]).any()
    assert torch.equal(outs[0][0].view(torch.int16), outs[1][0].view(torch.int16))
    assert torch.equal(outs[0][1].view(torch.int32), outs[1][1].view(torch.int32))
