"""The forward captured in a CUDA graph: a replay gives the eager result, and
a replay after new inputs are copied into the same buffers recomputes them.
Each replay is also checked against the oracle: routing and schedule tables
bit-exact, y within the forward's tolerances."""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_ffn_route_gb300 import binding as mb
from moe_expert_ffn_route_gb300 import synth
from parity_helpers import bf16_bits, y_errors

pytestmark = pytest.mark.gpu


def _up(a):
    a = np.ascontiguousarray(a)
    return torch.from_numpy(a.view(np.int32) if a.dtype == np.uint32 else a).cuda()


def _check_oracle(inp, k, prob, ws, idx, y):
    ridx, rw = oracle.route(inp["logits"], k)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    E, N = prob.num_experts, prob.num_tokens * k
    lay = oracle.layout(ridx, E)
    q = lambda name: mb.query(prob, ws, name).view(torch.int32)
    assert np.array_equal(q("counts")[:E].cpu().numpy(), lay["counts"])
    assert np.array_equal(q("offsets")[: E + 1].cpu().numpy(), lay["offsets"])
    assert np.array_equal(q("slots")[:N].cpu().numpy().reshape(-1, k), lay["slots"])
    ref = oracle.forward(inp, ridx, rw)
    max_rel, mean_rel = y_errors(bf16_bits(y), ref["y"])
    assert max_rel <= 2e-2 and mean_rel <= 5e-3, (max_rel, mean_rel)


@pytest.mark.parametrize("T", [96, 600])
def test_forward_replays_in_a_cuda_graph(T):
    # T = 96: 32-row tiles; T = 600: paired 144-row tiles (200 rows per expert expected)
    wl = synth.Workload("graph", T, 512, 256, 6, 2, 51)
    inp = synth.make_inputs(wl)
    inp2 = synth.make_inputs(synth.Workload("graph2", T, 512, 256, 6, 2, 52))
    prob = mb.problem(wl.T, wl.H, wl.I, wl.E, wl.k)
    assert mb.paired_tiles(prob) == (T == 600)
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
    _check_oracle(inp, wl.k, prob, ws, idx, y)

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
    assert mb.device_status(prob, ws)[0] == mb.OK
    # the graph's weights are the first input set's; its tokens and logits the second's
    mixed = dict(inp, logits=inp2["logits"], x=inp2["x"], x_sf=inp2["x_sf"])
    _check_oracle(mixed, wl.k, prob, ws, idx, y)
