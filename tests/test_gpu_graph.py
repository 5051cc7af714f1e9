"""The decode step and the prefill captured in a CUDA graph and replayed: every per-step
decision (the split plan, the lengths, the page ids) is made on the device from device
arrays, so a graph captured once serves later steps whose queries and lengths are written
into the same buffers.  Replays are compared bit for bit with eager calls on the same inputs."""
import numpy as np
import pytest
import torch

from mla_absorbed_latent_decode_gb300 import workloads as W
from mla_absorbed_latent_decode_gb300.runner import DecodeSession, bf16_tensor

pytestmark = pytest.mark.gpu


def test_decode_step_replays_from_a_graph():
    wl = W.make_decode("graph_decode", 81, 128, [700, 64, 1500, 3, 4096])
    s = DecodeSession(wl)
    s.prefill()
    rows, seq, pos = s.step_inputs()
    s.append_step(rows, seq, pos)
    eager = s.decode().clone()                       # also sets the kernels' attributes before capture
    out = torch.empty_like(eager)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        s.mla.kv_append(rows, seq, pos, s.block_table, s.cache, wl.num_pages, stream=side)
        s.mla.decode(s.q, s.ctx_len, wl.max_ctx, s.block_table, s.cache, wl.num_pages, s.workspace, out, stream=side)
    g.replay()
    torch.cuda.synchronize()
    assert s.status() == 0
    assert torch.equal(out, eager)
    # later steps: new queries and shorter lengths in the captured buffers (a different split plan)
    rng = np.random.default_rng(7)
    for lens in ([699, 1, 1500, 3, 2000], [5, 64, 65, 1, 4096]):
        s.q.copy_(bf16_tensor(W.to_bf16_bits(rng.standard_normal((wl.B, wl.n_h, 192))), s.device))
        s.ctx_len.copy_(torch.tensor(lens, dtype=torch.int32, device=s.device))
        g.replay()
        ref = s.decode().clone()                      # eager, same inputs (the append rewrites the same rows)
        torch.cuda.synchronize()
        assert s.status() == 0
        assert torch.equal(out, ref)
    s.close()


def test_prefill_replays_from_a_graph():
    wl = W.make_prefill("graph_prefill", 82, 16, [300, 129, 64], [300, 100, 1])
    s = DecodeSession(wl)
    s.append_rows()
    p = wl.extra["prefill"]
    dev = s.device
    q = bf16_tensor(p["q"], dev)
    qs = torch.from_numpy(p["q_start"]).to(dev)
    ql = torch.from_numpy(p["q_len"]).to(dev)
    ws = torch.empty(s.mla.prefill_workspace_size(wl.B, wl.max_ctx), dtype=torch.uint8, device=dev)
    eager = torch.empty((q.shape[0], wl.n_h, 128), dtype=torch.bfloat16, device=dev)
    s.mla.prefill(q, qs, ql, 300, s.ctx_len, wl.max_ctx, s.block_table, s.cache, wl.num_pages, ws, eager)
    out = torch.empty_like(eager)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        s.mla.prefill(q, qs, ql, 300, s.ctx_len, wl.max_ctx, s.block_table, s.cache, wl.num_pages, ws, out,
                      stream=side)
    g.replay()
    torch.cuda.synchronize()
    assert s.status() == 0
    assert torch.equal(out, eager)
    s.close()
