"""The forward captured in a CUDA graph: a replay gives the eager result, and
a replay after new inputs are copied into the same buffers recomputes them."""
import numpy as np
import pytest
import torch

from moe_expert_ffn_route_gb300 import binding as mb
from moe_expert_ffn_route_gb300 import synth

pytestmark = pytest.mark.gpu


def _up(a):
    a = np.ascontiguousarray(a)
    return torch.from_numpy(a.view(np.int32) if a.dtype == np.uint32 else a).cuda()


def test_forward_replays_in_a_cuda_graph():
    wl = synth.Workload("graph", 96, 512, 256, 6, 2, 51)
    inp = synth.make_inputs(wl)
    inp2 = synth.make_inputs(synth.Workload("graph2", 96, 512, 256, 6, 2, 52))
    prob = mb.problem(wl.T, wl.H, wl.I, wl.E, wl.k)
    prepared = mb.prepare_weights(prob, _up(inp["w1"]), _up(inp["w1_sf"]), _up(inp["w2"]), _up(inp["w2_sf"]))
    logits, x, x_sf = _up(inp["logits"]), _up(inp["x"]), _up(inp["x_sf"])

    def eager(lg, xx, xs):
        i, w = mb.route_topk(lg, wl.k)
        ws = mb.empty_workspace(prob)
        y = mb.forward(prob, xx, xs, i, w, prepared, ws)
        torch.cuda.synchronize()
        assert mb.device_status(prob, ws)[0] == mb.OK
        return y.clone()

    y_ref = eager(logits, x, x_sf)
    idx = torch.empty((wl.T, wl.k), dtype=torch.int64, device="cuda")
    w = torch.empty((wl.T, wl.k), dtype=torch.float32, device="cuda")
    ws = mb.empty_workspace(prob)
    y = torch.empty_like(y_ref)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        mb.route_topk(logits, wl.k, idx, w)
        mb.forward(prob, x, x_sf, idx, w, prepared, ws, y)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        mb.route_topk(logits, wl.k, idx, w)
        mb.forward(prob, x, x_sf, idx, w, prepared, ws, y)

    y.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert mb.device_status(prob, ws)[0] == mb.OK
    assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))

    # new tokens and router logits in the captured buffers
    lg2, x2, xs2 = _up(inp2["logits"]), _up(inp2["x"]), _up(inp2["x_sf"])
    y_ref2 = eager(lg2, x2, xs2)
    logits.copy_(lg2)
    x.copy_(x2)
    x_sf.copy_(xs2)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y_ref2.view(torch.int16))
    assert not torch.equal(y_ref2.view(torch.int16), y_ref.view(torch.int16))
