"""Oracle for the fused MoE expert forward (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product path (the CUDA library and its
Python binding) never imports, links or runs anything under ``oracle/``.

``oracle.c`` is a plain fp64 C restatement of what the pages define (see its
header for the passages).  This module builds it with gcc, loads it with
ctypes and marshals numpy arrays; it does no arithmetic of its own beyond
what ``grouped.py`` restates for the grouped-vs-direct pin.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(format tables against torch dtypes, closed forms, brute force, invariants
and the pages' worked pool-size example).
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import platform
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_lib = None


def _so_path() -> str:
    return os.path.join(_HERE, "_build", platform.machine(), "liboracle.so")


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (plain C11, fp64, OpenMP)."""
    so = _so_path()
    os.makedirs(os.path.dirname(so), exist_ok=True)
    with open(_SRC, "rb") as f:
        digest = hashlib.sha256(f.read()).hexdigest()
    stamp = so + ".stamp"
    if not force and os.path.exists(so) and os.path.exists(stamp):
        if open(stamp).read().strip() == digest:
            return so
    # -ffp-contract=off: no fused multiply-adds, identical results on x86 and Arm
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", so + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(so + ".tmp", so)
    with open(stamp, "w") as f:
        f.write(digest)
    return so


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        d, u8, i32, i64, p = ctypes.c_double, ctypes.c_uint8, ctypes.c_int, ctypes.c_int64, ctypes.c_void_p
        L.oracle_e4m3_decode.restype = d; L.oracle_e4m3_decode.argtypes = [u8]
        L.oracle_e2m1_decode.restype = d; L.oracle_e2m1_decode.argtypes = [u8]
        L.oracle_ue8m0_decode.restype = d; L.oracle_ue8m0_decode.argtypes = [u8]
        L.oracle_e4m3_encode.restype = u8; L.oracle_e4m3_encode.argtypes = [d]
        L.oracle_bf16_round.restype = d; L.oracle_bf16_round.argtypes = [d]
        L.oracle_bf16_bits.restype = ctypes.c_uint16; L.oracle_bf16_bits.argtypes = [d]
        L.oracle_silu.restype = d; L.oracle_silu.argtypes = [d]
        L.oracle_requant_exponent.restype = i32; L.oracle_requant_exponent.argtypes = [d]
        L.oracle_route.restype = None
        L.oracle_route.argtypes = [p, i32, i32, i32, p, p]
        L.oracle_layout.restype = i32
        L.oracle_layout.argtypes = [p, i32, i32, i32, i32, p, p, p, p, p]
        L.oracle_pool_capacity.restype = i64
        L.oracle_pool_capacity.argtypes = [i64] * 6
        L.oracle_sf_pool_rows.restype = i64
        L.oracle_sf_pool_rows.argtypes = [i64, i64]
        L.oracle_forward.restype = None
        L.oracle_forward.argtypes = [i32, i32, i32, i32, i32, p, p, p, p, p, p, p, p, p, i32,
                                     p, p, p, d, i32]
        L.oracle_num_threads.restype = i32
        _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------------------
# scalar helpers (vectorised over numpy arrays for the pin tests)
# ---------------------------------------------------------------------------

def e4m3_decode(codes) -> np.ndarray:
    L = lib()
    return np.array([L.oracle_e4m3_decode(int(c)) for c in np.ravel(codes)]).reshape(np.shape(codes))


def e2m1_decode(codes) -> np.ndarray:
    L = lib()
    return np.array([L.oracle_e2m1_decode(int(c)) for c in np.ravel(codes)]).reshape(np.shape(codes))


def ue8m0_decode(codes) -> np.ndarray:
    L = lib()
    return np.array([L.oracle_ue8m0_decode(int(c)) for c in np.ravel(codes)]).reshape(np.shape(codes))


def e4m3_encode(v) -> np.ndarray:
    L = lib()
    return np.array([L.oracle_e4m3_encode(float(x)) for x in np.ravel(v)], np.uint8).reshape(np.shape(v))


def bf16_round(v) -> np.ndarray:
    L = lib()
    return np.array([L.oracle_bf16_round(float(x)) for x in np.ravel(v)]).reshape(np.shape(v))


def silu(v) -> np.ndarray:
    L = lib()
    return np.array([L.oracle_silu(float(x)) for x in np.ravel(v)]).reshape(np.shape(v))


def requant_exponent(amax) -> np.ndarray:
    L = lib()
    return np.array([L.oracle_requant_exponent(float(x)) for x in np.ravel(amax)], np.int32).reshape(np.shape(amax))


def pool_capacity(R, T, k, E_loc, block_m, align_to) -> int:
    return int(lib().oracle_pool_capacity(R, T, k, E_loc, block_m, align_to))


def sf_pool_rows(pool, block_m) -> int:
    return int(lib().oracle_sf_pool_rows(pool, block_m))


# ---------------------------------------------------------------------------
# array entry points
# ---------------------------------------------------------------------------

def route(logits: np.ndarray, k: int):
    """softmax -> top-k -> renormalise; returns (idx int64 [T,k], w float32 [T,k])."""
    logits = np.ascontiguousarray(logits, np.float32)
    T, E = logits.shape
    idx = np.empty((T, k), np.int64)
    w = np.empty((T, k), np.float32)
    lib().oracle_route(_ptr(logits), T, E, k, _ptr(idx), _ptr(w))
    return idx, w


def layout(idx: np.ndarray, E: int, block: int = 128):
    """Naive schedule tables: counts, offsets, slots, row2tk, slack, P."""
    idx = np.ascontiguousarray(idx, np.int64)
    T, k = idx.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    slots = np.empty((T, k), np.int32)
    L = lib()
    P = L.oracle_layout(_ptr(idx), T, k, E, block, _ptr(counts), _ptr(offsets), _ptr(slots), None, None)
    row2tk = np.empty(max(P, 1), np.int32)
    slack = np.empty(max(P // block, 1), np.int32)
    L.oracle_layout(_ptr(idx), T, k, E, block, _ptr(counts), _ptr(offsets), _ptr(slots),
                    _ptr(row2tk), _ptr(slack))
    return dict(counts=counts, offsets=offsets, slots=slots, row2tk=row2tk[:P],
                slack=slack[:P // block], P=int(P))


def forward(inp: dict, idx: np.ndarray, w: np.ndarray, tokens=None, want_codes: bool = False,
            clamp: float = 0.0, threads: int = 0):
    """Direct per-(token, k) loop.  Returns dict(y=uint16 bf16 bits [n,H],
    q=uint8 [n,k,I] E4M3 codes, qe=int8 [n,k,I/32] exponents) for the listed tokens."""
    x, x_sf = inp["x"], inp["x_sf"]
    w1, w1_sf, w2, w2_sf = inp["w1"], inp["w1_sf"], inp["w2"], inp["w2_sf"]
    T, H = x.shape
    E, I2, _ = w1.shape
    I = I2 // 2
    k = idx.shape[1]
    idx = np.ascontiguousarray(idx, np.int64)
    w = np.ascontiguousarray(w, np.float32)
    tl = None if tokens is None else np.ascontiguousarray(tokens, np.int32)
    n = T if tl is None else len(tl)
    y = np.empty((n, H), np.uint16)
    q = np.empty((n, k, I), np.uint8) if want_codes else None
    qe = np.empty((n, k, I // 32), np.int8) if want_codes else None
    for a in (x, x_sf, w1, w1_sf, w2, w2_sf):
        assert a.flags.c_contiguous
    lib().oracle_forward(T, H, I, E, k, _ptr(x), _ptr(x_sf), _ptr(idx), _ptr(w),
                         _ptr(w1), _ptr(w1_sf), _ptr(w2), _ptr(w2_sf),
                         _ptr(tl), n, _ptr(y), _ptr(q), _ptr(qe), float(clamp), int(threads))
    return dict(y=y, q=q, qe=qe)


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint32) << 16).view(np.float32)
