"""Seeded synthetic inputs for the fused MoE expert forward.

This module only *draws* inputs and stores them in the formats the forward
consumes: E4M3 activation codes, E2M1 weight codes (two per byte, element 2i
in the low nibble), and UE8M0 scale codes packed four per uint32 along K.
It implements none of the forward's own steps (routing, layout, gather, the
two grouped GEMMs, SwiGLU, requantisation, combine). Both the oracle tests
and the CUDA path take their inputs from here; neither is imported here.

Workloads (MegaMoE pages, "test default shape" table of the code-reading
notes, and the TP-MoE practice page's problem setting) are described by
`Workload`. The draw recipe:

* router logits: N(0, 1) fp32 [T, E] ("uniform" routing), or, for the
  skewed workload, log p_rank(e) + Gumbel(0, 1) with p_r proportional to
  r^-s over a seeded permutation of the experts, the coldest `n_cold`
  experts at -inf, so that top-k by logit samples experts without
  replacement by Zipf popularity;
* x: N(0, 1) fp32 [T, H]; for the skewed workload a seeded 1 % of the rows
  are multiplied by 64 before encoding;
* W1: gate [I, H] and up [I, H] per expert, each N(0, std = 1/sqrt(H)),
  encoded, then interleaved by 8 rows (gate 0..7, up 0..7, gate 8..15, ...)
  as the MegaMoE weight transform does ("L1 weight interleave" section);
* W2: [H, I] per expert, N(0, std = 1/sqrt(I)).

Encoding of a block of 32 consecutive K values v: the UE8M0 exponent is the
smallest integer e in [-127, 127] with max|v| <= FMAX * 2^e (FMAX = 448 for
E4M3 activations, 6 for E2M1 weights; e = 0 for an all-zero block); the
element codes are the round-to-nearest-even encodings of v * 2^-e.
"""
from __future__ import annotations

import dataclasses
import functools
import multiprocessing as mp
import os
from typing import Dict, Optional

import numpy as np

__all__ = ["Workload", "WORKLOADS", "make_inputs"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int            # tokens
    H: int            # d_model (hidden)
    I: int            # d_ff per expert (intermediate)
    E: int            # experts
    k: int            # top-k
    seed: int
    routing: str = "uniform"      # "uniform" | "zipf"
    zipf_s: float = 1.2
    n_cold: int = 0
    outlier_frac: float = 0.0
    outlier_scale: float = 1.0

    @property
    def N(self) -> int:
        return self.T * self.k

    def useful_flops(self) -> float:
        """2 * N * 3 * H * I (gate + up + down over routed rows)."""
        return 2.0 * self.N * 3.0 * self.H * self.I


WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", 128, 1024, 512, 8, 2, 0),
    "medium": Workload("medium", 2048, 4096, 1536, 64, 8, 1),
    "decode": Workload("decode", 128, 7168, 2048, 256, 8, 2),
    "prefill": Workload("prefill", 8192, 7168, 2048, 256, 8, 3),
    "skewed": Workload("skewed", 4000, 7168, 2048, 256, 8, 4, routing="zipf",
                       zipf_s=1.2, n_cold=24, outlier_frac=0.01, outlier_scale=64.0),
    # the prefill and decode shapes at E = 32: the same rows per expert (256 and
    # 4), so the same token tiles and per-tile work, with 1/8 of the weights;
    # small enough for hardware-counter captures of single GEMM launches
    "prefill_e32": Workload("prefill_e32", 1024, 7168, 2048, 32, 8, 5),
    "decode_e32": Workload("decode_e32", 16, 7168, 2048, 32, 8, 6),
}


# ----------------------------------------------------------------------------
# storage-format encoders (input synthesis only)
# ----------------------------------------------------------------------------

def _block_exponents(blocks: np.ndarray, fmax_m: float, fmax_q: int) -> np.ndarray:
    """Smallest e with amax <= FMAX*2^e, FMAX = fmax_m * 2^fmax_q, fmax_m in [0.5,1)."""
    amax = np.abs(blocks).max(axis=-1)
    m, q = np.frexp(amax)
    e = q.astype(np.int32) - fmax_q + (m > fmax_m).astype(np.int32)
    e = np.where(amax == 0, 0, e)
    return np.clip(e, -127, 127).astype(np.int32)


def _encode_e4m3(v: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _encode_e2m1(v: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even onto {0, .5, 1, 1.5, 2, 3, 4, 6}; |v| <= 6 assumed."""
    a = np.abs(v).astype(np.float32)
    c_lo = np.rint(a * 2.0)             # [0, 2): codes 0..4 (spacing 0.5)
    c_mid = np.rint(a) + 2.0            # [2, 4): codes 4..6 (spacing 1)
    c_hi = np.rint(a * 0.5) + 4.0       # [4, 6]: codes 6..7 (spacing 2)
    code = np.where(a < 2.0, c_lo, np.where(a < 4.0, c_mid, c_hi)).astype(np.uint8)
    sign = (np.signbit(v)).astype(np.uint8) << 3
    return code | sign


def _quantize(v: np.ndarray, kind: str):
    """v [..., K] fp32 -> (codes [..., K] uint8, scale codes [..., K/32] uint8)."""
    K = v.shape[-1]
    blocks = v.reshape(v.shape[:-1] + (K // 32, 32))
    if kind == "e4m3":
        e = _block_exponents(blocks, 0.875, 9)      # 448 = 0.875 * 2^9
    else:
        e = _block_exponents(blocks, 0.75, 3)       # 6 = 0.75 * 2^3
    scaled = np.ldexp(blocks, -e[..., None]).astype(np.float32)
    codes = _encode_e4m3(scaled) if kind == "e4m3" else _encode_e2m1(scaled)
    return codes.reshape(v.shape), (e + 127).astype(np.uint8)


def _pack_nibbles(codes: np.ndarray) -> np.ndarray:
    return (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)


def _pack_scales(sf: np.ndarray) -> np.ndarray:
    """[..., K/32] uint8 -> [..., K/128] uint32 (byte b of word w covers [128w+32b, +32))."""
    return np.ascontiguousarray(sf).view("<u4")


def _interleave8(gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    I = gate.shape[0]
    g = gate.reshape((I // 8, 8) + gate.shape[1:])
    u = up.reshape((I // 8, 8) + up.shape[1:])
    return np.stack([g, u], axis=1).reshape((2 * I,) + gate.shape[1:])


# ----------------------------------------------------------------------------
# draws
# ----------------------------------------------------------------------------

_TAG_LOGITS, _TAG_X, _TAG_W1, _TAG_W2, _TAG_OUTLIERS = 0, 1, 2, 3, 4


def _rng(seed: int, tag: int, sub: int = 0) -> np.random.Generator:
    return np.random.default_rng([seed, tag, sub])


def _expert(args):
    seed, e, H, I = args
    r1 = _rng(seed, _TAG_W1, e)
    gate = r1.standard_normal((I, H), dtype=np.float32) * np.float32(1.0 / np.sqrt(H))
    up = r1.standard_normal((I, H), dtype=np.float32) * np.float32(1.0 / np.sqrt(H))
    gc, gs = _quantize(gate, "e2m1")
    uc, us = _quantize(up, "e2m1")
    del gate, up
    w1 = _interleave8(_pack_nibbles(gc), _pack_nibbles(uc))
    w1_sf = _interleave8(_pack_scales(gs), _pack_scales(us))
    r2 = _rng(seed, _TAG_W2, e)
    down = r2.standard_normal((H, I), dtype=np.float32) * np.float32(1.0 / np.sqrt(I))
    dc, ds = _quantize(down, "e2m1")
    return e, w1, w1_sf, _pack_nibbles(dc), _pack_scales(ds)


def _logits(w: Workload) -> np.ndarray:
    r = _rng(w.seed, _TAG_LOGITS)
    if w.routing == "uniform":
        return r.standard_normal((w.T, w.E), dtype=np.float32)
    if w.routing == "zipf":
        perm = r.permutation(w.E)
        n_hot = w.E - w.n_cold
        ranks = np.arange(1, n_hot + 1, dtype=np.float64)
        p = ranks ** (-w.zipf_s)
        p /= p.sum()
        logp = np.full(w.E, -np.inf)
        logp[perm[:n_hot]] = np.log(p)
        g = r.gumbel(size=(w.T, w.E))
        return (logp[None, :] + g).astype(np.float32)
    raise ValueError(w.routing)


def _activations(w: Workload):
    r = _rng(w.seed, _TAG_X)
    x = r.standard_normal((w.T, w.H), dtype=np.float32)
    if w.outlier_frac > 0:
        ro = _rng(w.seed, _TAG_OUTLIERS)
        n_out = int(round(w.outlier_frac * w.T))
        rows = ro.choice(w.T, size=n_out, replace=False)
        x[rows] *= np.float32(w.outlier_scale)
    codes, sf = _quantize(x, "e4m3")
    return codes, _pack_scales(sf)


@functools.lru_cache(maxsize=4)
def make_inputs(w: Workload, workers: Optional[int] = None) -> Dict[str, np.ndarray]:
    """All inputs of one workload as numpy arrays (cached per process).

    Returns logits f32 [T,E]; x u8 [T,H]; x_sf u32 [T,H/128];
    w1 u8 [E,2I,H/2]; w1_sf u32 [E,2I,H/128]; w2 u8 [E,H,I/2]; w2_sf u32 [E,H,I/128].
    Expert weights are drawn per expert from their own seed, so the result does
    not depend on `workers`.
    """
    T, H, I, E = w.T, w.H, w.I, w.E
    assert H % 128 == 0 and I % 128 == 0
    out: Dict[str, np.ndarray] = {"logits": _logits(w)}
    out["x"], out["x_sf"] = _activations(w)
    w1 = np.empty((E, 2 * I, H // 2), np.uint8)
    w1_sf = np.empty((E, 2 * I, H // 128), np.uint32)
    w2 = np.empty((E, H, I // 2), np.uint8)
    w2_sf = np.empty((E, H, I // 128), np.uint32)
    jobs = [(w.seed, e, H, I) for e in range(E)]
    n_el = E * 3 * H * I
    if workers is None:
        workers = min(os.cpu_count() or 1, 32) if n_el > 50_000_000 else 1
    if workers > 1:
        # spawn: never fork a process that may already hold a CUDA context
        with mp.get_context("spawn").Pool(workers) as pool:
            # a bounded get: a pool whose workers cannot start raises instead of waiting forever
            results = pool.map_async(_expert, jobs, chunksize=1).get(timeout=1800)
            for e, a, b, c, d in results:
                w1[e], w1_sf[e], w2[e], w2_sf[e] = a, b, c, d
    else:
        for job in jobs:
            e, a, b, c, d = _expert(job)
            w1[e], w1_sf[e], w2[e], w2_sf[e] = a, b, c, d
    out.update(w1=w1, w1_sf=w1_sf, w2=w2, w2_sf=w2_sf)
    return out
