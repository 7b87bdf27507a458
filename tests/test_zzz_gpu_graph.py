"""The decode calls inside a CUDA graph.  A serving loop replays one captured decode step per token
instead of paying the host-side launch path every time.  The decode launchers make no host-side
CUDA call other than the launch itself, so a step captures; each replay must equal an eager call
on the same inputs bit for bit.  The file name makes pytest run it last."""
import pytest
import torch

import gated_deltanet_recurrence_gb300 as gdn
from gated_deltanet_recurrence_gb300 import synthetic
from tests._util import oracle_gates

pytestmark = pytest.mark.gpu


def _decode_inputs(T=None):
    cfg = synthetic.workload("decode", N=16, H=8, d=128, dtype=torch.bfloat16, seed=41)
    inp = synthetic.decode_inputs(cfg)
    g, b = oracle_gates(inp)
    dev = "cuda"
    if T is None:
        return (inp["q"].to(dev), inp["k"].to(dev), inp["v"].to(dev), g.to(dev), b.to(dev),
                inp["state"].to(dev))
    rep = lambda x: x.unsqueeze(1).repeat_interleave(T, 1).contiguous().to(dev)  # noqa: E731
    return rep(inp["q"]), rep(inp["k"]), rep(inp["v"]), rep(g), rep(b), inp["state"].to(dev)


def test_decode_step_replays_from_a_cuda_graph():
    q, k, v, g, b, state = _decode_inputs()
    out = torch.empty(q.shape[0], v.shape[1], v.shape[2], device="cuda", dtype=torch.float32)
    s_eager = state.clone()
    gdn.gdn_recurrent_step(q, k, v, g, b, s_eager, out=torch.empty_like(out))   # warm-up, eager
    torch.cuda.synchronize()
    s_eager.copy_(state)
    s_graph = state.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gdn.gdn_recurrent_step(q, k, v, g, b, s_graph, out=out)
    s_graph.copy_(state)                       # capture does not run the kernel; start from S0
    out_eager = torch.empty_like(out)
    for _ in range(3):                         # three tokens: the state advances in place
        graph.replay()
        gdn.gdn_recurrent_step(q, k, v, g, b, s_eager, out=out_eager)
        torch.cuda.synchronize()
        assert torch.equal(out, out_eager)
        assert torch.equal(s_graph, s_eager)
    assert gdn.gdn_get_device_error() == 0


def test_multi_token_decode_replays_from_a_cuda_graph():
    T = 4                                      # the streamed form (blocks of four tokens)
    q, k, v, g, b, pool = _decode_inputs(T)
    idx = torch.arange(q.shape[0] - 1, -1, -1, dtype=torch.int32, device="cuda")
    out = torch.empty(q.shape[0], T, v.shape[2], v.shape[3], device="cuda", dtype=torch.float32)
    p_eager = pool.clone()
    gdn.gdn_recurrent_multi_step(q, k, v, g, b, p_eager, state_indices=idx, out=torch.empty_like(out))
    torch.cuda.synchronize()
    p_eager.copy_(pool)
    p_graph = pool.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gdn.gdn_recurrent_multi_step(q, k, v, g, b, p_graph, state_indices=idx, out=out)
    p_graph.copy_(pool)
    out_eager = torch.empty_like(out)
    for _ in range(2):
        graph.replay()
        gdn.gdn_recurrent_multi_step(q, k, v, g, b, p_eager, state_indices=idx, out=out_eager)
        torch.cuda.synchronize()
        assert torch.equal(out, out_eager)
        assert torch.equal(p_graph, p_eager)
    assert gdn.gdn_get_device_error() == 0
