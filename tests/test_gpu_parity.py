"""Parity of the CUDA path (through the C ABI) with the oracle.

Bars: routing indices, counts, padded offsets, slot table, inverse map,
slack and gathered bytes bit-exact; >= 99.9 % of the requantised L1 E4M3
codes identical and the rest within one E4M3 step; y within
max|y - y_ref| <= 2e-2 max|y_ref| and sum|y - y_ref| / sum|y_ref| <= 5e-3.
The tiny and decode workloads are checked on every token.  The medium,
prefill and skewed workloads are checked on the tokens that own these pool
rows (the oracle computes those tokens one by one): in every token tile of
the grouped GEMMs, its first row, its last valid row (the short last tile
of each expert included) and the first row the pair's second CTA stages;
plus 40-96 random tokens, the 8 rows with the largest activation scales
and the last token.  Every token tile of the run has checked rows; the
test asserts it and reports rows checked / pool rows.  With the default
144-row tile bound that is, for medium, 128 tiles, ~340 of 2048 tokens,
~2.7k of 16384 routed rows; prefill 518 tiles (paired: an even number per
expert), ~1.1k of 8192 tokens, ~8.9k of 65536 rows; skewed 381 tiles,
~930 of 4000 tokens, ~7.4k of 32000 rows.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_ffn_route_gb300 import binding as mb
from moe_expert_ffn_route_gb300 import synth
from parity_helpers import GpuRun, compare_l1_codes, up, upload_weights, y_errors

pytestmark = pytest.mark.gpu

Y_MAX_REL, Y_MEAN_REL, CODE_FRAC = 2e-2, 5e-3, 0.999
CONFIGS = ["tiny", "medium", "decode", "prefill", "skewed"]
SAMPLE = {"tiny": None, "medium": 96, "decode": None, "prefill": 40, "skewed": 40}

_cache = {}


def tile_probe_rows(tabs):
    """Pool rows probing every token tile of the grouped GEMMs: its first row,
    its last valid row and the first row of the half the pair's second CTA
    stages (tile geometry from the run's tile tables)."""
    rows = []
    off, counts, tiles, per = tabs["offsets"], tabs["counts"], tabs["tiles"], tabs["tile_rows"]
    for e in range(len(counts)):
        n, r = int(counts[e]), int(per[e])
        for t in range(int(tiles[e + 1] - tiles[e])):
            lo, hi = t * r, min(n, (t + 1) * r)
            for q in (lo, hi - 1, lo + r // 2):
                if lo <= q < hi:
                    rows.append(int(off[e]) + q)
    return np.unique(np.asarray(rows, np.int64))


def case(name):
    if name in _cache:
        return _cache[name]
    wl = synth.WORKLOADS[name]
    inp = synth.make_inputs(wl)
    idx, w = oracle.route(inp["logits"], wl.k)
    run = GpuRun(inp, idx, w)
    n = SAMPLE[name]
    if n is None:
        tokens = np.arange(wl.T)
    else:
        rng = np.random.default_rng(100 + wl.seed)
        tokens = rng.choice(wl.T, size=n, replace=False)
        # the rows with the largest activation scales (outliers) and the ragged tail
        big = np.argsort(-inp["x_sf"].view(np.uint8).max(axis=1), kind="stable")[:8]
        lay = oracle.layout(idx, wl.E)
        probe = tile_probe_rows(run.tables())
        owners = lay["row2tk"][probe] // wl.k
        assert np.all(lay["row2tk"][probe] >= 0)
        tokens = np.unique(np.concatenate([tokens, big, [wl.T - 1], owners]))
    ref = oracle.forward(inp, idx, w, tokens=tokens, want_codes=True)
    _cache[name] = (wl, inp, idx, w, run, tokens, ref)
    return _cache[name]


@pytest.mark.parametrize("name", [c for c in CONFIGS if SAMPLE[c] is not None])
def test_checked_rows_cover_every_token_tile(name):
    wl, inp, idx, w, run, tokens, _ = case(name)
    tabs = run.tables()
    slots = tabs["slots"][tokens].reshape(-1)
    checked = np.zeros(tabs["P"], bool)
    checked[slots[slots >= 0]] = True
    off, counts, tiles, per = tabs["offsets"], tabs["counts"], tabs["tiles"], tabs["tile_rows"]
    n_tiles = n_empty = 0
    for e in range(wl.E):
        for t in range(int(tiles[e + 1] - tiles[e])):
            lo = int(off[e]) + t * int(per[e])
            hi = int(off[e]) + min(int(counts[e]), (t + 1) * int(per[e]))
            if hi <= lo:
                # the second tile of an expert with at most 16 rows (an even
                # number of tiles): it owns no rows, and no output comes from it
                assert mb.paired_tiles(run.prob) and t == 1 and counts[e] <= 16, (e, t)
                n_empty += 1
                continue
            assert checked[lo] and checked[hi - 1], (e, t)
            n_tiles += 1
    print(f"{name}: {int(checked.sum())} of {int(counts.sum())} pool rows checked, "
          f"{len(tokens)} of {wl.T} tokens, {n_tiles} token tiles (+ {n_empty} without rows)")


@pytest.mark.parametrize("name", CONFIGS)
def test_route_parity(name):
    wl = synth.WORKLOADS[name]
    inp = synth.make_inputs(wl)
    ridx, rw = oracle.route(inp["logits"], wl.k)
    gidx, gw = mb.route_topk(up(inp["logits"]), wl.k)
    torch.cuda.synchronize()
    assert np.array_equal(gidx.cpu().numpy(), ridx)
    np.testing.assert_allclose(gw.cpu().numpy(), rw, rtol=2e-6, atol=1e-7)


@pytest.mark.parametrize("E,k", [(40, 6), (256, 8)])
def test_route_nan_logits(E, k):
    """NaN logits rank below every number (the oracle's reading); every id is
    valid and distinct, also for a token with fewer finite logits than k."""
    rng = np.random.default_rng(E)
    logits = rng.standard_normal((96, E)).astype(np.float32)
    logits[rng.random(logits.shape) < 0.3] = np.nan
    logits[7, :] = np.nan
    logits[7, 3] = 1.0                            # one finite logit
    logits[8, :] = -np.inf
    ridx, rw = oracle.route(logits, k)
    gidx, gw = mb.route_topk(up(logits), k)
    torch.cuda.synchronize()
    gidx, gw = gidx.cpu().numpy(), gw.cpu().numpy()
    assert np.array_equal(gidx, ridx)
    assert ((gidx >= 0) & (gidx < E)).all()
    assert all(len(set(r)) == k for r in gidx.tolist())
    fin = np.isfinite(rw).all(axis=1)
    assert not fin[8] and fin.sum() == 95            # all -inf: 0/0 weights, as in the oracle
    np.testing.assert_allclose(gw[fin], rw[fin], rtol=2e-6, atol=1e-7)


@pytest.mark.parametrize("name", ["medium", "prefill"])
def test_forward_is_deterministic(name):
    """A second forward on the same inputs, into a fresh workspace, gives the
    same y (every token) and the same L1 codes and scales (the sampled tokens,
    every token tile among them) bit for bit: no step sums in an order that
    depends on timing."""
    import copy
    wl, inp, idx, w, run, tokens, _ = case(name)
    run2 = copy.copy(run)
    run2.ws = mb.empty_workspace(run.prob)
    run2.y = mb.forward(run.prob, run.x, run.x_sf, run.idx, run.w, run.prepared, run2.ws)
    torch.cuda.synchronize()
    assert run2.status()[0] == mb.OK
    assert torch.equal(run2.y.view(torch.int16), run.y.view(torch.int16))
    c1, e1 = _l1_codes(run, run.tables(), tokens)
    c2, e2 = _l1_codes(run2, run2.tables(), tokens)
    assert np.array_equal(c1, c2) and np.array_equal(e1, e2)


@pytest.mark.parametrize("E,k", [(40, 6), (256, 8), (1000, 8)])
def test_route_ties_and_signed_zeros(E, k):
    """Logits from a handful of values (many ties, +0 and -0 among them): the
    ids equal the oracle's, which breaks ties by the lower expert index."""
    rng = np.random.default_rng(E + 1)
    levels = np.array([-1.0, -0.0, 0.0, 0.5, 0.5, 2.0], np.float32)
    logits = levels[rng.integers(0, len(levels), size=(64, E))]
    logits[5, :] = -0.0
    logits[6, :] = 0.0
    logits[6, ::2] = -0.0
    ridx, rw = oracle.route(logits, k)
    gidx, gw = mb.route_topk(up(logits), k)
    torch.cuda.synchronize()
    assert np.array_equal(gidx.cpu().numpy(), ridx)
    np.testing.assert_allclose(gw.cpu().numpy(), rw, rtol=2e-6, atol=1e-7)


@pytest.mark.parametrize("name", CONFIGS)
def test_layout_parity(name):
    wl, inp, idx, w, run, _, _ = case(name)
    assert run.status()[0] == mb.OK
    ref = oracle.layout(idx, wl.E)
    got = run.tables()
    for key in ("counts", "offsets", "slots", "row2tk", "slack"):
        assert np.array_equal(got[key], ref[key]), key
    assert got["P"] == ref["P"]
    ntile = -(-ref["counts"] // run.tile_n)
    if mb.paired_tiles(run.prob):
        ntile += ntile & 1                            # an even number of tiles per expert
    assert np.array_equal(got["tiles"], np.concatenate([[0], np.cumsum(ntile)]))
    # equal tiles, rounded up to the 16-row quantum of the tile layout
    per = np.where(ntile > 0, -(-ref["counts"] // np.maximum(ntile, 1)), 16)
    assert np.array_equal(got["tile_rows"], -(-per // 16) * 16)
    s = ref["slots"].reshape(-1)
    assert np.array_equal(got["wpool"][s], w.reshape(-1))
    pad = ref["row2tk"] < 0
    assert np.all(got["wpool"][pad] == 0)


@pytest.mark.parametrize("name", CONFIGS)
def test_gather_parity(name):
    wl, inp, idx, w, run, tokens, _ = case(name)
    tabs = run.tables()
    slots = tabs["slots"][tokens].reshape(-1)
    toks = np.repeat(tokens, wl.k)
    ok = slots >= 0
    slots, toks = slots[ok], toks[ok]
    rows = run.pool_rows("xpool", slots, wl.H)
    assert np.array_equal(rows, inp["x"][toks])
    sf = run.sf_bytes("xpool_sf", slots, wl.H // 128, tabs)
    assert np.array_equal(sf, inp["x_sf"][toks].view(np.uint8))


def _l1_codes(run, tabs, tokens):
    """E4M3 codes [n, k, I] and exponents [n, k, I/32] of the requantised L1
    output of the listed tokens; entries with an empty slot are left zero."""
    I = run.I
    slots = tabs["slots"][tokens].reshape(-1)
    ok = slots >= 0
    codes = np.zeros((len(slots), I), np.uint8)
    exps = np.zeros((len(slots), I // 32), np.int32)
    codes[ok] = run.pool_rows("hpool", slots[ok], I)
    exps[ok] = run.sf_bytes("hpool_sf", slots[ok], I // 128, tabs).astype(np.int32) - 127
    return codes.reshape(len(tokens), run.k, I), exps.reshape(len(tokens), run.k, I // 32)


@pytest.mark.parametrize("name", CONFIGS)
def test_l1_codes_parity(name):
    wl, inp, idx, w, run, tokens, ref = case(name)
    codes, exps = _l1_codes(run, run.tables(), tokens)
    frac, within, n_diff = compare_l1_codes(codes, exps, ref["q"], ref["qe"])
    assert frac >= CODE_FRAC, (frac, n_diff)
    assert within


@pytest.mark.parametrize("name", CONFIGS)
def test_y_parity(name):
    wl, inp, idx, w, run, tokens, ref = case(name)
    y = run.y_bits()[tokens]
    max_rel, mean_rel = y_errors(y, ref["y"])
    assert max_rel <= Y_MAX_REL and mean_rel <= Y_MEAN_REL, (max_rel, mean_rel)


# ------------------------------------------------------------------ edge cases

def _small(T=96, H=512, I=256, E=6, k=2, seed=31, empty=0.0, skew=False):
    inp = synth.make_inputs(synth.Workload(f"edge{seed}", T, H, I, E, k, seed))
    logits = inp["logits"].copy()
    if skew:
        logits[:, 0] += 5.0          # expert 0 takes almost everything
        logits[:, E - 1] -= 50.0     # expert E-1 gets nothing
    idx, w = oracle.route(logits, k)
    if empty:
        rng = np.random.default_rng(seed)
        idx = idx.copy()
        idx[rng.random(idx.shape) < empty] = -1
    return inp, idx, w


def _check_full(inp, idx, w, run, clamp=0.0):
    T = inp["x"].shape[0]
    ref = oracle.forward(inp, idx, w, want_codes=True, clamp=clamp)
    lay = oracle.layout(idx, run.E)
    tabs = run.tables()
    for key in ("counts", "offsets", "slots", "row2tk", "slack"):
        assert np.array_equal(tabs[key], lay[key]), key
    valid = idx >= 0
    tokens = np.arange(T)
    if valid.any():
        codes, exps = _l1_codes(run, tabs, tokens)
        frac, within, _ = compare_l1_codes(codes[valid], exps[valid], ref["q"][valid], ref["qe"][valid])
        assert frac >= CODE_FRAC and within, frac
    max_rel, mean_rel = y_errors(run.y_bits(), ref["y"])
    assert max_rel <= Y_MAX_REL and mean_rel <= Y_MEAN_REL, (max_rel, mean_rel)


@pytest.mark.parametrize("tile_n,T", [(32, 200), (48, 200), (64, 200), (96, 200), (128, 200), (144, 200),
                                      (160, 200), (192, 200), (224, 200), (96, 700), (144, 700)])
def test_every_token_tile(tile_n, T):
    # T = 200 pairs tiles at bounds 48 and 64 (80 rows per expert expected),
    # T = 700 at 96 and 144 as well (280 rows)
    inp, idx, w = _small(T=T, E=5, k=2, skew=True)
    run = GpuRun(inp, idx, w, tile_n=tile_n)
    assert run.tile_n == tile_n and run.status()[0] == mb.OK
    assert mb.paired_tiles(run.prob) == (tile_n in (48, 64) or (T == 700 and tile_n in (96, 144)))
    _check_full(inp, idx, w, run)


@pytest.mark.parametrize("clamp", [10.0, 0.5])
def test_activation_clamp(clamp):
    # 10 is the pages' default threshold; 0.5 clamps a large share of gate and up values
    inp, idx, w = _small(T=120, E=5, k=2, seed=41)
    run = GpuRun(inp, idx, w, act_clamp=clamp)
    assert run.status()[0] == mb.OK
    _check_full(inp, idx, w, run, clamp=clamp)
    if clamp < 1.0:
        # the clamp is live: the clamped oracle and the plain one differ here
        plain = oracle.forward(inp, idx, w)["y"]
        assert not np.array_equal(run.y_bits(), plain)


def test_fast_math_meets_the_same_bars():
    # approximate exp and reciprocal in SiLU, against the exact oracle
    inp, idx, w = _small(T=160, E=6, k=2, seed=43)
    run = GpuRun(inp, idx, w, fast_math=1)
    assert run.status()[0] == mb.OK
    _check_full(inp, idx, w, run)


@pytest.mark.parametrize("T,tile_n", [(37, 0), (200, 48)])
def test_empty_entries_and_ragged_tokens(T, tile_n):
    # (200, 48): paired 48-row tiles (~86 rows per expert expected)
    inp, idx, w = _small(T=T, E=7, k=3, empty=0.3)
    run = GpuRun(inp, idx, w, tile_n=tile_n)
    assert mb.paired_tiles(run.prob) == (tile_n == 48)
    _check_full(inp, idx, w, run)


@pytest.mark.parametrize("T", [50, 200])
def test_single_expert_top1(T):
    # T = 200: one expert with 200 rows, paired into two 112-row tiles
    inp, idx, w = _small(T=T, E=1, k=1)
    run = GpuRun(inp, idx, w)
    assert mb.paired_tiles(run.prob) == (T == 200)
    _check_full(inp, idx, w, run)


def test_all_experts_per_token():
    inp, idx, w = _small(T=40, E=4, k=4)
    run = GpuRun(inp, idx, w)
    _check_full(inp, idx, w, run)


@pytest.mark.parametrize("T", [64, 300])
def test_hidden_not_multiple_of_256(T):
    """L2 output channel tiles of 256 with a 128-wide remainder; I = 128, so
    an L2 item has one K block.  T = 300 pairs the token tiles (200 rows per
    expert expected against 144-row tiles)."""
    inp, idx, w = _small(T=T, H=384, I=128, E=3, k=2)
    run = GpuRun(inp, idx, w)
    assert mb.paired_tiles(run.prob) == (T == 300)
    _check_full(inp, idx, w, run)


@pytest.mark.parametrize("shape", [dict(T=300, E=6, k=2), dict(T=700, H=1024, I=384, E=12, k=4, skew=True)])
def test_one_launch_equals_two_launches(shape):
    """The persistent launch (L2 items wait for their token tile's L1 items)
    and the two-launch form give the same bytes: L1 codes, their scales and y."""
    inp, idx, w = _small(seed=61, **shape)
    fused = GpuRun(inp, idx, w)
    split = GpuRun(inp, idx, w, debug_flags=mb.DEBUG_SPLIT_LAYERS, weights=fused.prepared)
    assert fused.status()[0] == mb.OK and split.status()[0] == mb.OK
    assert np.array_equal(fused.y_bits(), split.y_bits())
    tabs = fused.tables()
    rows = np.nonzero(tabs["row2tk"] >= 0)[0]
    assert np.array_equal(fused.pool_rows("hpool", rows, fused.I), split.pool_rows("hpool", rows, split.I))
    kb = fused.I // 128
    assert np.array_equal(fused.sf_bytes("hpool_sf", rows, kb, tabs), split.sf_bytes("hpool_sf", rows, kb, tabs))
    _check_full(inp, idx, w, fused)


def test_bad_expert_id_is_reported_and_skipped():
    inp, idx, w = _small(T=32, E=6, k=2)
    bad = idx.copy()
    bad[3, 1] = 77
    bad[9, 0] = -5
    run = GpuRun(inp, bad, w)
    st, code, _ = run.status()
    assert st == mb.ERR_INVALID_ARG and code & 1
    eff = bad.copy()
    eff[(eff < 0) | (eff >= 6)] = -1
    _check_full(inp, eff, w, run)


def test_zero_tokens():
    inp, idx, w = _small(T=16)
    prob = mb.problem(0, 512, 256, 6, 2)
    ws = mb.empty_workspace(prob)
    empty8 = torch.empty(0, dtype=torch.uint8, device="cuda")
    y = torch.empty((0, 512), dtype=torch.bfloat16, device="cuda")
    prepared = upload_weights(inp, prob)
    mb.forward(prob, empty8, torch.empty(0, dtype=torch.int32, device="cuda"),
               torch.empty(0, dtype=torch.int64, device="cuda"), torch.empty(0, dtype=torch.float32, device="cuda"),
               prepared, ws, y=y)
    assert mb.device_status(prob, ws)[0] == mb.OK


def test_l1_accumulators_match_exact_products():
    """Raw FP32 accumulators of the block-scaled tensor-core GEMM against the
    fp64 sum of exactly representable products."""
    from oracle.grouped import _dequant_act, _dequant_w
    # (tile bound, tokens): 70 tokens give one tile per stage at every bound;
    # 48-row tiles with 120 tokens (80 rows per expert) are paired
    for tile_n, T in ((32, 70), (96, 70), (144, 70), (224, 70), (48, 120)):
        inp, idx, w = _small(T=T, H=1024, I=256, E=3, k=2, seed=5)
        run = GpuRun(inp, idx, w, tile_n=tile_n, debug_flags=mb.DEBUG_DUMP_L1_ACC)
        assert mb.paired_tiles(run.prob) == (tile_n == 48)
        tabs = run.tables()
        z = run.view("ypool", torch.float32)[: tabs["P"] * 2 * run.I].view(tabs["P"], 2 * run.I).cpu().numpy()
        assert run.status()[0] == mb.OK
        xd = _dequant_act(inp["x"], inp["x_sf"])
        for e in range(run.E):
            W = _dequant_w(inp["w1"][e], inp["w1_sf"][e])
            rows = np.arange(2 * run.I).reshape(run.I // 8, 2, 8)
            Wg, Wu = W[rows[:, 0].reshape(-1)], W[rows[:, 1].reshape(-1)]
            sel = np.nonzero(idx == e)
            t = sel[0]
            s = tabs["slots"][sel]
            ref = np.concatenate([xd[t] @ Wg.T, xd[t] @ Wu.T], axis=1)
            mag = np.concatenate([np.abs(xd[t]) @ np.abs(Wg).T, np.abs(xd[t]) @ np.abs(Wu).T], axis=1)
            err = np.abs(z[s] - ref)
            assert np.all(err <= 1e-5 * mag + 1e-30), (e, tile_n, float((err / (mag + 1e-30)).max()))


@pytest.mark.parametrize("tile_n,T", [(0, 64), (48, 200)])
def test_bounded_wait_reports_timeout_and_context_survives(tile_n, T):
    # (0, 64): 32-row tiles, one ring per MMA warp; (48, 200): paired tiles, one ring
    inp, idx, w = _small(T=T, E=4, k=2)
    run = GpuRun(inp, idx, w, tile_n=tile_n, debug_flags=mb.DEBUG_STARVE_L1, wait_timeout_us=20000)
    assert mb.paired_tiles(run.prob) == (tile_n == 48)
    st, code, detail = run.status()
    # any pipeline wait may be the first of the grid to expire (a race), but it is one of them
    assert st == mb.ERR_TIMEOUT and code & 2 and 1 <= detail <= 7
    # the context is still usable: a normal forward afterwards is correct
    run2 = GpuRun(inp, idx, w)
    assert run2.status()[0] == mb.OK
    _check_full(inp, idx, w, run2)
