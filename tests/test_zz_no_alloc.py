"""The allocation-free schedule-table entry point.

It exists for callers that may not allocate device memory when they need
the routing tables (a fixed memory budget reserved at start-up, or a loop
that must not enter the allocator because it can synchronise the device).
Its tables must equal the oracle's and the ones moeffn_forward builds in its
workspace, call after call, although every call reuses the same static
scratch.  This file is collected last on purpose.
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


class _Buffers:
    """Device buffers of one call, allocated before the call is made."""

    def __init__(self, idx: np.ndarray, E: int):
        T, k = idx.shape
        self.T, self.k, self.E = T, k, E
        self.idx = torch.from_numpy(np.ascontiguousarray(idx, np.int64)).cuda()
        self.counts = torch.full((E,), -7, dtype=torch.int32, device="cuda")
        self.offsets = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
        self.slots = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")

    def call(self):
        mb.schedule_tables_noalloc(self.idx, self.E, self.counts, self.offsets, self.slots)

    def result(self):
        torch.cuda.synchronize()
        return (self.counts.cpu().numpy(), self.offsets.cpu().numpy(),
                self.slots.cpu().numpy().reshape(self.T, self.k))


def _tables_noalloc(idx: np.ndarray, E: int):
    b = _Buffers(idx, E)
    b.call()
    return b.result()


def _case(T, H, I, E, k, seed, empty=0.0):
    inp = synth.make_inputs(synth.Workload(f"noalloc{seed}", T, H, I, E, k, seed))
    idx, w = oracle.route(inp["logits"], k)
    if empty:
        idx = idx.copy()
        idx[np.random.default_rng(seed).random(idx.shape) < empty] = -1
    return inp, idx, w


def _assert_oracle_tables(got, idx, E):
    ref = oracle.layout(idx, E)
    counts, offsets, slots = got
    assert np.array_equal(counts, ref["counts"])
    assert np.array_equal(offsets, ref["offsets"])
    assert np.array_equal(slots, ref["slots"])


def test_noalloc_tables_match_oracle_and_forward_on_consecutive_calls():
    # a larger call first, then a smaller one: stale scratch from the first
    # call must not leak into the second
    cases = [_case(3000, 256, 128, 64, 8, 41), _case(77, 256, 128, 12, 3, 42, empty=0.2)]
    for inp, idx, w in cases:
        run = GpuRun(inp, idx, w)
        ref = run.tables()
        got = _tables_noalloc(idx, run.E)
        _assert_oracle_tables(got, idx, run.E)
        counts, offsets, slots = got
        assert np.array_equal(counts, ref["counts"])
        assert np.array_equal(offsets, ref["offsets"])
        assert np.array_equal(slots, ref["slots"])


def test_noalloc_ids_outside_the_experts_are_empty_entries():
    rng = np.random.default_rng(5)
    E, k = 24, 4
    idx = np.stack([rng.permutation(E)[:k] for _ in range(700)]).astype(np.int64)
    bad = rng.random(idx.shape) < 0.05
    idx[bad] = np.where(rng.random(bad.sum()) < 0.5, E, E + 5)
    got = _tables_noalloc(idx, E)
    eff = np.where(idx >= E, -1, idx)
    _assert_oracle_tables(got, eff, E)
    assert np.all(got[2][bad] == -1)


def test_noalloc_multi_chunk_calls_with_different_expert_counts():
    # more than 1024 entries each (several per-chunk histograms), different E:
    # the second call must not see the first call's histograms
    rng = np.random.default_rng(6)
    for T, E, k in [(300, 64, 8), (500, 20, 4), (1100, 7, 2)]:
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int64)
        _assert_oracle_tables(_tables_noalloc(idx, E), idx, E)


def test_noalloc_calls_take_no_device_memory():
    rng = np.random.default_rng(7)
    idx = np.stack([rng.permutation(32)[:4] for _ in range(900)]).astype(np.int64)
    b = _Buffers(idx, 32)
    b.call()                               # the first call on the device loads the module
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        b.call()
    got = b.result()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    _assert_oracle_tables(got, idx, 32)


def test_noalloc_rejects_problems_beyond_its_scratch():
    L = mb.load()
    f = ctypes.c_void_p(1 << 20)
    # 64 + 4*N + 4*ceil(N/1024)*E bytes > 4 MiB
    assert L.moeffn_schedule_tables_noalloc(f, 200000, 256, 8, f, f, f, None) == mb.ERR_WORKSPACE_TOO_SMALL
    assert L.moeffn_schedule_tables_noalloc(f, 10, 0, 1, f, f, f, None) == mb.ERR_INVALID_ARG
