"""The bounds-checked build of the library (MOEFFN_BOUNDS_CHECK).

There is no sanitizer to run on this GPU, so a second build of the same
sources checks, before each access, every pool-row, token-tile and
128-row-block index the table, gather and combine kernels use against its
buffer (the grouped GEMM's rows and tiles come from the tile records, whose
ranges are checked where they are written).  An index out of range is
reported through the workspace status word and the access is skipped.

The parity cases below run on that build, over every stage layout: no index
is out of range, and the results equal the oracle's.  The reporting path
itself is checked by a small program, and the host's reading of the status
bit by a status word set by hand.
"""
import os
import subprocess
import tempfile

import numpy as np
import pytest
import torch

import oracle
from moe_expert_ffn_route_gb300 import binding as mb
from moe_expert_ffn_route_gb300 import build as mbuild
from moe_expert_ffn_route_gb300 import synth
from parity_helpers import GpuRun, y_errors

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bounds_library():
    lib = mb.open_library(mbuild.build(variant="bounds"))
    saved = mb._lib
    mb._lib = lib
    yield lib
    mb._lib = saved


def _routed(T, H, I, E, k, seed, empty=0.0, skew=False, first_empty=False):
    inp = synth.make_inputs(synth.Workload(f"bounds{seed}", T, H, I, E, k, seed))
    logits = inp["logits"].copy()
    if skew:
        logits[:, 0] += 5.0
        logits[:, E - 1] -= 50.0
    if first_empty:
        logits[:, 0] -= 50.0                    # expert 0 gets no rows (empty first segment)
    idx, w = oracle.route(logits, k)
    if empty:
        idx = idx.copy()
        idx[np.random.default_rng(seed).random(idx.shape) < empty] = -1
    return inp, idx, w


# (T, H, I, E, k, tile_n, extra): 32-row tiles; paired 48-row tiles with a
# skewed expert; one-tile-per-stage 144; 224; empty entries; H = 384 (an L2
# tail half, paired); one expert; expert 0 without rows, paired
CASES = [
    (96, 512, 256, 6, 2, 0, {}),
    (200, 512, 256, 5, 2, 48, {"skew": True}),
    (160, 512, 256, 6, 2, 144, {}),
    (300, 512, 256, 4, 2, 224, {}),
    (37, 512, 256, 7, 3, 0, {"empty": 0.3}),
    (300, 384, 128, 3, 2, 0, {}),
    (200, 512, 256, 1, 1, 0, {}),
    (300, 512, 256, 5, 2, 48, {"first_empty": True}),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_no_index_out_of_bounds(bounds_library, case):
    T, H, I, E, k, tile_n, extra = CASES[case]
    inp, idx, w = _routed(T, H, I, E, k, 70 + case, **extra)
    run = GpuRun(inp, idx, w, tile_n=tile_n)
    st, code, _ = run.status()
    assert st == mb.OK and code == 0, (st, code)
    lay = oracle.layout(idx, E)
    tabs = run.tables()
    for key in ("counts", "offsets", "slots", "row2tk", "slack"):
        assert np.array_equal(tabs[key], lay[key]), key
    ref = oracle.forward(inp, idx, w)
    max_rel, mean_rel = y_errors(run.y_bits(), ref["y"])
    assert max_rel <= 2e-2 and mean_rel <= 5e-3, (max_rel, mean_rel)


def test_out_of_bounds_report():
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "bounds_check")
        cmd = [mbuild.nvcc()] + mbuild.ARCH + ["-O3", "-std=c++17", "-DMOEFFN_BOUNDS_CHECK", "-I", mbuild.INCLUDE,
                                               "-I", mbuild.CSRC, os.path.join(ROOT, "tests", "bounds_check.cu"),
                                               "-o", exe]
        subprocess.run(cmd, check=True, capture_output=True, timeout=300)
        out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=60).stdout.split()
    vals = dict(zip(out[::2], (int(v) for v in out[1::2])))
    assert vals == {"code": 4, "where": 42, "index": 5, "ok": 5}, vals


def test_status_word_reads_as_out_of_bounds():
    prob = mb.problem(16, 256, 128, 4, 2)
    ws = mb.empty_workspace(prob)
    status = mb.query(prob, ws, "status").view(torch.int32)
    status.zero_()
    status[0] = 4                               # the bounds bit of the status word
    assert mb.device_status(prob, ws)[0] == mb.ERR_OUT_OF_BOUNDS
    status[0] = 4 | 2                           # with a timeout as well: the bounds report wins
    assert mb.device_status(prob, ws)[0] == mb.ERR_OUT_OF_BOUNDS
