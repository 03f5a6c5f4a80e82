"""The allocation-free schedule-table entry point.

It exists for callers that may not allocate device memory when they need
the routing tables (a fixed memory budget reserved at start-up, or a loop
that must not enter the allocator because it can synchronise the device).
Its tables must equal the ones moeffn_forward builds in its workspace, call
after call, although every call reuses the same static scratch.
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from moe_expert_ffn_route_gb300 import binding as mb
from moe_expert_ffn_route_gb300 import synth
from parity_helpers import GpuRun

pytestmark = pytest.mark.gpu


def _tables_noalloc(idx: np.ndarray, E: int):
    T, k = idx.shape
    d_idx = torch.from_numpy(np.ascontiguousarray(idx, np.int64)).cuda()
    counts = torch.full((E,), -7, dtype=torch.int32, device="cuda")
    offsets = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    slots = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
    mb.schedule_tables_noalloc(d_idx, E, counts, offsets, slots)
    torch.cuda.synchronize()
    return counts.cpu().numpy(), offsets.cpu().numpy(), slots.cpu().numpy().reshape(T, k)


def _case(T, H, I, E, k, seed, empty=0.0):
    inp = synth.make_inputs(synth.Workload(f"noalloc{seed}", T, H, I, E, k, seed))
    idx, w = oracle.route(inp["logits"], k)
    if empty:
        idx = idx.copy()
        idx[np.random.default_rng(seed).random(idx.shape) < empty] = -1
    return inp, idx, w


def test_noalloc_tables_match_forward_on_consecutive_calls():
    # a larger call first, then a smaller one: stale scratch from the first
    # call must not leak into the second
    cases = [_case(3000, 256, 128, 64, 8, 41), _case(77, 256, 128, 12, 3, 42, empty=0.2)]
    for inp, idx, w in cases:
        run = GpuRun(inp, idx, w)
        ref = run.tables()
        counts, offsets, slots = _tables_noalloc(idx, run.E)
        assert np.array_equal(counts, ref["counts"])
        assert np.array_equal(offsets, ref["offsets"])
        assert np.array_equal(slots, ref["slots"])


def test_noalloc_rejects_problems_beyond_its_scratch():
    L = mb.load()
    f = ctypes.c_void_p(1 << 20)
    # 64 + 4*N + 4*ceil(N/1024)*E bytes > 4 MiB
    assert L.moeffn_schedule_tables_noalloc(f, 200000, 256, 8, f, f, f, None) == mb.ERR_WORKSPACE_TOO_SMALL
    assert L.moeffn_schedule_tables_noalloc(f, 10, 0, 1, f, f, f, None) == mb.ERR_INVALID_ARG
