"""Grouped restatement of the forward (TEST INFRASTRUCTURE ONLY).

A second formulation of the same mathematics, organised the way the pages'
data flow is (MegaMoE code-reading notes, "End-to-end data flow": L1 pool
-> L1 GEMM -> SwiGLU + requant -> L2 pool -> L2 GEMM -> combine buffer ->
top-k reduce), written with numpy fp64 matmuls over expert-sorted pools.
It exists to pin the direct loop in ``oracle.c``: on tiny inputs both must
agree bit for bit on the E4M3 codes and on y.  It decodes formats and
de-interleaves weights with its own code (bit manipulation on arrays) so
that a mistake in either formulation shows up as a mismatch.
"""
from __future__ import annotations

import numpy as np


def _e4m3(codes: np.ndarray) -> np.ndarray:
    c = codes.astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 7
    v = np.where(e == 0, m * 2.0 ** -9, (8 + m) * np.exp2(e - 10.0))
    return s * v


def _e2m1(codes: np.ndarray) -> np.ndarray:
    c = codes.astype(np.int64)
    s = np.where(c & 8, -1.0, 1.0)
    e = (c >> 1) & 3
    m = c & 1
    v = np.where(e == 0, 0.5 * m, (2 + m) * np.exp2(e - 2.0))
    return s * v


def _scales(sf_u32: np.ndarray) -> np.ndarray:
    """[..., K/128] packed uint32 -> [..., K/32] fp64 power-of-two scales."""
    b = np.ascontiguousarray(sf_u32).view(np.uint8).astype(np.int64)
    return np.exp2(b - 127.0)


def _dequant_act(codes: np.ndarray, sf: np.ndarray) -> np.ndarray:
    v = _e4m3(codes)
    s = _scales(sf)
    return (v.reshape(v.shape[:-1] + (-1, 32)) * s[..., None]).reshape(v.shape)


def _dequant_w(packed: np.ndarray, sf: np.ndarray) -> np.ndarray:
    lo = packed & 0xF
    hi = packed >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(packed.shape[:-1] + (-1,))
    v = _e2m1(codes)
    s = _scales(sf)
    return (v.reshape(v.shape[:-1] + (-1, 32)) * s[..., None]).reshape(v.shape)


def _bf16(v: np.ndarray) -> np.ndarray:
    """Nearest bfloat16 value (8 significant bits), ties to even, for normal
    magnitudes: round the fp64 significand directly."""
    m, q = np.frexp(v)
    return np.ldexp(np.rint(np.ldexp(m, 8)), q - 8)


def _e4m3_rne(v: np.ndarray) -> np.ndarray:
    """Codes for |v| <= 448 by exhaustive nearest search over the 127 finite
    non-negative E4M3 values (ties -> even code)."""
    table = _e4m3(np.arange(0x7F))                      # 0x00..0x7E
    a = np.abs(v)
    d = np.abs(a[..., None] - table)                    # distance to each value
    best = d.min(axis=-1, keepdims=True)
    cand = d == best
    # ties: prefer the even code
    even = cand & ((np.arange(0x7F) & 1) == 0)
    pick = np.where(even.any(axis=-1), even.argmax(axis=-1), cand.argmax(axis=-1))
    return (pick | np.where(np.signbit(v), 0x80, 0)).astype(np.uint8)


def forward_grouped(inp: dict, idx: np.ndarray, w: np.ndarray, block: int = 128, clamp: float = 0.0):
    """Returns (y bf16 bits [T,H], q codes [T,k,I], qe exponents [T,k,I/32]).
    clamp > 0: the optional activation clamp of the L1 epilogue (MegaMoE notes,
    "Activation clamp"): gate limited above, up on both sides, after the BF16 cast."""
    x, x_sf = inp["x"], inp["x_sf"]
    T, H = x.shape
    E, I2, _ = inp["w1"].shape
    I = I2 // 2
    k = idx.shape[1]
    xd = _dequant_act(x, x_sf)                                 # [T,H]
    # expert-sorted pool (stable in t*k+j), padded per expert to `block` rows
    flat = idx.reshape(-1)
    order = np.argsort(np.where(flat < 0, E, flat), kind="stable")
    q = np.zeros((T, k, I), np.uint8)
    qe = np.zeros((T, k, I // 32), np.int8)
    yslots = np.zeros((T, k, H))
    for e in range(E):
        ent = order[flat[order] == e]
        if ent.size == 0:
            continue
        tok, jj = ent // k, ent % k
        X = xd[tok]                                            # pool rows of e
        W1 = _dequant_w(inp["w1"][e], inp["w1_sf"][e])         # [2I,H]
        rows = np.arange(2 * I).reshape(I // 8, 2, 8)
        Wg, Wu = W1[rows[:, 0, :].reshape(-1)], W1[rows[:, 1, :].reshape(-1)]
        g = _bf16(X @ Wg.T)
        u = _bf16(X @ Wu.T)
        if clamp > 0:
            g = np.minimum(g, clamp)
            u = np.clip(u, -clamp, clamp)
        Hm = g / (1.0 + np.exp(-g)) * u * w[tok, jj][:, None].astype(np.float64)
        grp = Hm.reshape(len(ent), I // 32, 32)
        amax = np.abs(grp).max(axis=-1)
        es = np.zeros(amax.shape, np.int64)
        pos = amax > 0
        # smallest e with amax <= 448*2^e: ceil(log2(amax/448)) done exactly
        mm, qq = np.frexp(amax / 448.0)                        # amax/448 exact? not always
        cand = np.where(mm == 0.5, qq - 1, qq)
        # correct the (rare) inexact division by checking the definition
        cand = np.where(amax > np.ldexp(448.0, cand), cand + 1, cand)
        cand = np.where(amax <= np.ldexp(448.0, cand - 1), cand - 1, cand)
        es[pos] = cand[pos]
        es = np.clip(es, -127, 127)
        codes = _e4m3_rne(np.ldexp(grp, -es[..., None]))
        q[tok, jj] = codes.reshape(len(ent), I)
        qe[tok, jj] = es.astype(np.int8)
        Hq = np.ldexp(_e4m3(codes), es[..., None]).reshape(len(ent), I)
        W2 = _dequant_w(inp["w2"][e], inp["w2_sf"][e])         # [H,I]
        yslots[tok, jj] = _bf16(Hq @ W2.T)
    ysum = yslots.sum(axis=1)
    yb = _bf16(ysum).astype(np.float32)
    y = (yb.view(np.uint32) >> 16).astype(np.uint16)
    return y, q, qe
