"""The seeded input generator: encoders, determinism, workload structure."""
import numpy as np
import torch

from moe_expert_ffn_route_gb300 import synth


def test_e2m1_encoder_is_nearest_even():
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
    mids = (grid[:-1] + grid[1:]) / 2
    v = np.concatenate([grid, mids, np.linspace(0, 6, 1201)]).astype(np.float32)
    v = np.concatenate([v, -v])
    codes = synth._encode_e2m1(v)
    mag = grid[codes & 7]
    d = np.abs(np.abs(v)[:, None] - grid[None, :])
    best = d.min(1)
    assert np.allclose(np.abs(np.abs(v) - mag), best)
    tie = (d == best[:, None]).sum(1) > 1
    assert np.all((codes[tie] & 1) == 0)               # ties -> even code
    assert np.all(((codes >> 3) & 1) == np.signbit(v))


def test_activation_encoding_roundtrip():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((16, 256)).astype(np.float32)
    x[3] *= 64
    x[5] = 0
    codes, sf = synth._quantize(x, "e4m3")
    e = sf.astype(np.int32) - 127
    dec = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    xh = dec * np.exp2(np.repeat(e, 32, axis=1))
    blk = np.abs(x).reshape(16, 8, 32).max(-1)
    assert np.all(blk <= 448 * np.exp2(e)) and np.all((blk == 0) | (blk > 448 * np.exp2(e - 1)))
    # RNE error at most half a step of E4M3 (2^-3 relative, subnormals absolute)
    assert np.all(np.abs(xh - x) <= np.maximum(np.abs(x) * 2.0 ** -4, np.exp2(np.repeat(e, 32, 1) - 10)))


def test_deterministic_and_worker_independent():
    w = synth.Workload("t", 8, 256, 128, 3, 2, 5)
    a = synth.make_inputs.__wrapped__(w, workers=1)
    b = synth.make_inputs.__wrapped__(w, workers=2)
    for key in a:
        assert np.array_equal(a[key], b[key]), key
    assert a["w1"].shape == (3, 256, 128) and a["w1_sf"].shape == (3, 256, 2)
    assert a["w2"].shape == (3, 256, 64) and a["w2_sf"].shape == (3, 256, 1)


def test_skewed_routing_structure():
    w = synth.WORKLOADS["skewed"]
    logits = synth._logits(w)
    top = np.argsort(-logits, axis=1, kind="stable")[:, : w.k]
    counts = np.bincount(top.reshape(-1), minlength=w.E)
    assert (counts == 0).sum() >= 20
    assert counts.max() >= 3000
    assert w.T % 128 != 0


def test_skewed_outlier_rows():
    # 1 % of the 4000 rows (40, distinct) scaled by 64 = 2^6 before encoding: their
    # block exponents sit about 6 above the rest
    w = synth.WORKLOADS["skewed"]
    codes, sf = synth._activations(w)
    sfb = sf.view(np.uint8).reshape(w.T, -1).astype(np.int32)
    row_mean = sfb.mean(axis=1)
    typical = np.median(row_mean)
    hot = np.flatnonzero(row_mean > typical + 3)
    assert len(hot) == 40
    assert np.all(np.abs(row_mean[hot] - typical - 6) < 1)
    assert codes.shape == (w.T, w.H) and codes.dtype == np.uint8
