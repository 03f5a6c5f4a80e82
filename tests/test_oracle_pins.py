"""Pins for the oracle against things other than itself: torch's format
dtypes, closed forms, brute force, invariants, the pages' worked example,
and a second (grouped) formulation of the forward."""
import itertools
import os

import numpy as np
import pytest
import torch

import oracle
from oracle.grouped import forward_grouped
from moe_expert_ffn_route_gb300.synth import Workload, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- formats

def test_e4m3_decode_all_codes_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = oracle.e4m3_decode(codes)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def test_ue8m0_decode_all_codes_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e8m0fnu).double().numpy()
    got = oracle.ue8m0_decode(codes)
    assert np.isnan(got[255]) and np.isnan(ref[255])
    assert np.array_equal(ref[:255], got[:255])


def _minifloat(code, ebits, mbits, bias, nan_codes=()):
    """Generic sign/exponent/mantissa decoder with subnormals and no Inf."""
    s = (code >> (ebits + mbits)) & 1
    e = (code >> mbits) & ((1 << ebits) - 1)
    m = code & ((1 << mbits) - 1)
    if code in nan_codes:
        return float("nan")
    if e == 0:
        v = m / (1 << mbits) * 2.0 ** (1 - bias)
    else:
        v = (1 + m / (1 << mbits)) * 2.0 ** (e - bias)
    return -v if s else v


def test_generic_minifloat_matches_torch_then_pins_e2m1():
    # validate the generic decoder on the two 8-bit formats torch implements ...
    e4 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    for c in range(256):
        v = _minifloat(c, 4, 3, 7, nan_codes=(0x7F, 0xFF))
        assert (np.isnan(v) and np.isnan(e4[c])) or v == e4[c]
    e5 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e5m2).double().numpy()
    for c in range(256):
        if (c & 0x7C) == 0x7C:
            continue  # E5M2 has Inf/NaN in its top exponent; E2M1 has neither
        assert _minifloat(c, 5, 2, 15) == e5[c]
    # ... then apply it to E2M1 (1 sign, 2 exponent, 1 mantissa bit, bias 1)
    ref = np.array([_minifloat(c, 2, 1, 1) for c in range(16)])
    got = oracle.e2m1_decode(np.arange(16, dtype=np.uint8))
    assert np.array_equal(ref, got)
    assert sorted(set(np.abs(got))) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


def _e4m3_values():
    return torch.arange(0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def test_e4m3_encode_rne_vs_torch():
    vals = _e4m3_values()
    mids = (vals[:-1] + vals[1:]) / 2          # exact midpoints (ties)
    rng = np.random.default_rng(7)
    rnd = rng.uniform(-448, 448, 4000)
    small = rng.uniform(-2.0 ** -5, 2.0 ** -5, 2000)
    grid = np.concatenate([vals, -vals, mids, -mids, rnd, small,
                           np.nextafter(mids, 0), np.nextafter(mids, 1000)]).astype(np.float32)
    grid = grid[np.abs(grid) <= 448]
    ref = torch.from_numpy(grid).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(grid.astype(np.float64))
    # +-0 both decode to zero; compare decoded values for zeros, codes elsewhere
    nz = grid != 0
    assert np.array_equal(ref[nz], got[nz])
    # saturation: the encoder saturates (torch's cast does not)
    assert oracle.e4m3_encode(np.array([1e6, -500.0])).tolist() == [0x7E, 0xFE]


def test_bf16_round_vs_torch():
    rng = np.random.default_rng(3)
    a = (rng.standard_normal(20000) * np.exp2(rng.integers(-60, 60, 20000))).astype(np.float32)
    # exact ties: 8 significant bits + a half ulp
    m = rng.integers(128, 256, 2000).astype(np.float64)
    ties = np.ldexp(m + 0.5, rng.integers(-40, 40, 2000) - 7).astype(np.float32)
    v = np.concatenate([a, ties, -ties])
    ref = torch.from_numpy(v).to(torch.bfloat16).double().numpy()
    got = oracle.bf16_round(v.astype(np.float64))
    assert np.array_equal(ref, got)


def test_requant_exponent_definition():
    rng = np.random.default_rng(5)
    amax = np.concatenate([np.abs(rng.standard_normal(3000)) * np.exp2(rng.integers(-30, 30, 3000)),
                           448.0 * np.exp2(np.arange(-20, 20.0)),
                           np.nextafter(448.0 * np.exp2(np.arange(-20, 20.0)), np.inf)])
    e = oracle.requant_exponent(amax)
    assert np.all(amax <= 448.0 * np.exp2(e.astype(np.float64)))
    assert np.all(amax > 448.0 * np.exp2(e - 1.0))
    assert oracle.requant_exponent(np.array([0.0]))[0] == 0
    # codes never saturate under this rule
    assert np.all(np.abs(amax / np.exp2(e.astype(np.float64))) <= 448.0)


def test_silu_closed_form():
    x = np.linspace(-30, 30, 601)
    got = oracle.silu(x)
    ref = torch.nn.functional.silu(torch.from_numpy(x)).numpy()
    assert np.allclose(got, ref, rtol=1e-14, atol=1e-300)
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    assert np.allclose(got - oracle.silu(-x), x, rtol=1e-14, atol=1e-14)   # silu(x)-silu(-x)=x
    assert abs(oracle.silu(np.array([40.0]))[0] - 40.0) < 1e-12


# ---------------------------------------------------------------- routing

def test_route_bruteforce_small():
    rng = np.random.default_rng(11)
    for E, k in [(5, 1), (6, 2), (7, 3), (8, 8)]:
        logits = rng.standard_normal((40, E)).astype(np.float32)
        logits[0, :] = 0.5                     # all tied: lowest indices first
        idx, w = oracle.route(logits, k)
        for t in range(logits.shape[0]):
            l = logits[t].astype(np.float64)
            best = max(itertools.combinations(range(E), k),
                       key=lambda s: (sum(l[list(s)]), [-i for i in s]))
            assert sorted(idx[t].tolist()) == sorted(best)
            order = sorted(best, key=lambda e: (-l[e], e))
            assert idx[t].tolist() == order
            ref = torch.softmax(torch.from_numpy(l[order]), 0).numpy()
            assert np.allclose(w[t], ref, rtol=2e-7, atol=0)
            assert abs(w[t].astype(np.float64).sum() - 1) < 1e-6


def test_route_nan_logits_rank_last():
    """The pages leave NaN router logits undefined; the reading taken is that a
    NaN ranks below every number.  Checked against torch's top-k over the
    logits with NaN replaced by -inf (torch.sort is stable: ties keep the
    lower index first) and torch's softmax over the chosen values."""
    rng = np.random.default_rng(12)
    T, E, k = 64, 40, 6
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[rng.random((T, E)) < 0.3] = np.nan
    logits[5, :E - 3] = np.nan                  # fewer finite logits than k
    logits[5, E - 3:] = [0.5, -1.0, 2.0]
    logits[6, 0] = -np.inf
    idx, w = oracle.route(logits, k)
    clean = torch.from_numpy(np.where(np.isnan(logits), -np.inf, logits).astype(np.float64))
    order = torch.sort(clean, dim=1, descending=True, stable=True).indices[:, :k]
    assert np.array_equal(idx, order.numpy())
    sel = torch.gather(clean, 1, order)
    ref = torch.softmax(sel, 1).numpy()
    ok = np.isfinite(sel.numpy()).all(axis=1)
    assert np.allclose(w[ok], ref[ok], rtol=2e-7, atol=1e-30)
    # with fewer than k finite logits the -inf entries get weight 0
    assert np.all(w[5, 3:] == 0) and np.allclose(w[5, :3].sum(), 1.0, rtol=1e-6)
    assert sorted(idx[5, 3:].tolist()) == list(range(3))


# ---------------------------------------------------------------- layout

def _check_layout(idx, E, lay, block=128):
    T, k = idx.shape
    counts, offsets, slots, row2tk, slack, P = (lay[n] for n in
                                                 ("counts", "offsets", "slots", "row2tk", "slack", "P"))
    flat = idx.reshape(-1)
    assert np.array_equal(counts, np.bincount(flat[flat >= 0], minlength=E))
    assert offsets[0] == 0 and offsets[-1] == P
    assert np.array_equal(np.diff(offsets), -(-counts // block) * block)
    valid = flat >= 0
    s = slots.reshape(-1)
    assert np.all(s[~valid] == -1)
    assert len(np.unique(s[valid])) == valid.sum()              # injective
    for e in range(E):                                           # rows of e in its range
        se = s[flat == e]
        assert np.all((se >= offsets[e]) & (se < offsets[e] + counts[e]))
        # stable in t*k+j order
        assert np.array_equal(se, offsets[e] + np.arange(counts[e]))
    inv = np.full(P, -1)
    inv[s[valid]] = np.nonzero(valid)[0]
    assert np.array_equal(inv, row2tk)                           # bijection with row2tk
    real = (row2tk.reshape(-1, block) >= 0).sum(1) if P else np.zeros(0)
    assert np.array_equal(real + slack, np.full(P // block, block))
    assert slack.sum() == P - valid.sum()
    # against a library stable sort
    order = np.argsort(np.where(valid, flat, E), kind="stable")[: valid.sum()]
    ref = np.empty_like(s)
    ref[order] = offsets[flat[order]] + (np.arange(valid.sum()) - np.repeat(
        np.concatenate([[0], np.cumsum(counts)[:-1]]), counts))
    assert np.array_equal(ref[valid], s[valid])


@pytest.mark.parametrize("T,E,k,empty", [(128, 8, 2, 0.0), (300, 16, 4, 0.1), (257, 64, 8, 0.0),
                                         (5, 32, 3, 0.5), (1, 4, 4, 0.0)])
def test_layout_invariants(T, E, k, empty):
    rng = np.random.default_rng(T * 131 + E)
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int64)
    idx[rng.random(idx.shape) < empty] = -1
    idx[:, :] = np.where(idx == 3, 5 % E, idx) if E > 5 else idx   # some experts unused
    lay = oracle.layout(idx, E)
    _check_layout(idx, E, lay)


def test_layout_all_empty():
    idx = -np.ones((7, 2), np.int64)
    lay = oracle.layout(idx, 4)
    assert lay["P"] == 0 and np.all(lay["slots"] == -1)


def _golden(name):
    d = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            key, val = line.split()
            d[key] = int(val)
    return d


def test_pool_capacity_worked_example():
    g = _golden("pool_sizing.txt")
    R, T, k, E_loc, bm = (g["num_ranks"], g["num_max_tokens_per_rank"], g["num_topk"],
                          g["num_experts_per_rank"], g["block_m"])
    assert g["num_experts"] // R == E_loc
    # the printed terms: R*T*min(k, E_loc) and E_loc*(B_M-1)
    assert oracle.pool_capacity(R, T, k, E_loc, 1, 1) == g["recv_term"]
    assert oracle.pool_capacity(0, T, k, E_loc, bm, 1) == g["padding_term"]
    # the capacity is their aligned sum (the printed total does not follow; see header)
    cap = oracle.pool_capacity(R, T, k, E_loc, bm, bm)
    assert cap == -(-(g["recv_term"] + g["padding_term"]) // bm) * bm
    # SF pool relation on the printed pair
    assert oracle.sf_pool_rows(g["printed_pool"], bm) == g["printed_sf_pool"]


# ---------------------------------------------------------------- forward

def _tiny(T=24, H=256, I=256, E=4, k=2, seed=9, empty=0.1):
    inp = make_inputs(Workload("pin", T, H, I, E, k, seed))
    idx, w = oracle.route(inp["logits"], k)
    rng = np.random.default_rng(seed)
    idx = idx.copy()
    idx[rng.random(idx.shape) < empty] = -1
    return inp, idx, w


def test_grouped_equals_direct():
    for args in [dict(), dict(T=33, H=384, I=128, E=3, k=3, seed=4, empty=0.0)]:
        inp, idx, w = _tiny(**args)
        d = oracle.forward(inp, idx, w, want_codes=True)
        y, q, qe = forward_grouped(inp, idx, w)
        assert np.array_equal(d["qe"], qe)
        assert np.array_equal(d["q"], q)
        assert np.array_equal(d["y"], y)


def test_activation_clamp_pins():
    """The optional clamp (MegaMoE notes, "Activation clamp": gate limited above,
    up on both sides): grouped and direct forms agree; a clamp above every value
    changes nothing; a small clamp bounds every requantised activation."""
    inp, idx, w = _tiny(T=30, H=256, I=128, E=3, k=2, seed=12, empty=0.0)
    plain = oracle.forward(inp, idx, w, want_codes=True)
    # no-op when the threshold exceeds every gate and up value
    big = oracle.forward(inp, idx, w, want_codes=True, clamp=1e30)
    assert np.array_equal(big["y"], plain["y"]) and np.array_equal(big["q"], plain["q"])
    for c in (0.5, 2.0, 10.0):
        d = oracle.forward(inp, idx, w, want_codes=True, clamp=c)
        y, q, qe = forward_grouped(inp, idx, w, clamp=c)
        assert np.array_equal(d["qe"], qe) and np.array_equal(d["q"], q) and np.array_equal(d["y"], y)
    # with c = 0.5: |h| = |silu(g) u w| <= max(silu(c), -min silu) * c * w; the decoded E4M3
    # value is within half a step (1/16 relative) of h
    c = 0.5
    d = oracle.forward(inp, idx, w, want_codes=True, clamp=c)
    assert not np.array_equal(d["y"], plain["y"])        # the clamp is live on these inputs
    hdec = _e4m3_table()[d["q"]] * np.ldexp(1.0, d["qe"].astype(np.int64))[..., None].repeat(32, -1).reshape(d["q"].shape)
    bound = max(c / (1 + np.exp(-c)), 0.2785) * c * w[..., None] * (1 + 1 / 16)
    assert np.all(np.abs(hdec) <= bound)
    # and without the clamp the same inputs exceed that bound somewhere
    hplain = _e4m3_table()[plain["q"]] * np.ldexp(1.0, plain["qe"].astype(np.int64))[..., None].repeat(32, -1).reshape(plain["q"].shape)
    assert np.any(np.abs(hplain) > bound)


def _e4m3_table():
    return torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def _e2m1_to_torch(codes):
    """E2M1 code -> value via an E4M3 bit pattern (bias 1 -> bias 7) and torch."""
    c = codes.astype(np.int32)
    s, e, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
    e4 = np.where(e == 0, np.where(m == 1, 6 << 3, 0), ((e + 6) << 3) | (m << 2))
    e4 = (e4 | (s << 7)).astype(np.uint8)
    return torch.from_numpy(e4).view(torch.float8_e4m3fn).double()


def test_dense_special_case_matches_textbook_mlp():
    """E=1, k=1, w=1: y = bf16(W2 . requant(silu(bf16(Wg x)) * bf16(Wu x)))."""
    T, H, I = 8, 256, 128
    inp = make_inputs(Workload("dense", T, H, I, 1, 1, 21))
    idx = np.zeros((T, 1), np.int64)
    w = np.ones((T, 1), np.float32)
    got = oracle.forward(inp, idx, w)["y"]

    def scales(sf, K):
        return torch.from_numpy(np.ascontiguousarray(sf).view(np.uint8).copy()).view(
            torch.float8_e8m0fnu).double().repeat_interleave(32, dim=-1)[..., :K]

    x = torch.from_numpy(inp["x"]).view(torch.float8_e4m3fn).double() * scales(inp["x_sf"], H)
    w1 = inp["w1"][0]
    w1c = np.stack([w1 & 0xF, w1 >> 4], -1).reshape(2 * I, H)
    W1 = _e2m1_to_torch(w1c) * scales(inp["w1_sf"][0], H)
    rows = torch.arange(2 * I).view(I // 8, 2, 8)
    Wg, Wu = W1[rows[:, 0].reshape(-1)], W1[rows[:, 1].reshape(-1)]
    g = (x @ Wg.T).to(torch.bfloat16).double()
    u = (x @ Wu.T).to(torch.bfloat16).double()
    h = torch.nn.functional.silu(g) * u
    hb = h.view(T, I // 32, 32)
    amax = hb.abs().amax(-1)
    e = torch.ceil(torch.log2(amax / 448.0))
    e = torch.where(amax <= 448.0 * torch.exp2(e - 1), e - 1, e)
    e = torch.where(amax > 448.0 * torch.exp2(e), e + 1, e)
    hq = (hb * torch.exp2(-e)[..., None]).float().to(torch.float8_e4m3fn).double() * torch.exp2(e)[..., None]
    w2 = inp["w2"][0]
    W2 = _e2m1_to_torch(np.stack([w2 & 0xF, w2 >> 4], -1).reshape(H, I)) * scales(inp["w2_sf"][0], I)
    y = (hq.view(T, I) @ W2.T).to(torch.bfloat16)
    ref = y.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)
