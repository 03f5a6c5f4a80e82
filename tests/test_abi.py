"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every symbol include/moeffn.h declares, validates arguments synchronously,
and sizes its buffers from the pool-capacity formula."""
import ctypes
import os
import re

import pytest

import oracle
from moe_expert_ffn_route_gb300 import binding as mb

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moeffn.h")


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MOEFFN_API\s+[\w\s\*]+?\b(moeffn_\w+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    L = mb.load()
    names = declared_symbols()
    assert len(names) >= 11
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(mb.SIGNATURES)
    assert L.moeffn_abi_version() == 1


def test_status_strings():
    for s in range(7):
        assert mb.status_string(s) != "unknown status"
    assert mb.status_string(99) == "unknown status"


@pytest.mark.parametrize("kw,status", [
    (dict(), mb.OK),
    (dict(H=1000), mb.ERR_INVALID_ARG),
    (dict(I=200), mb.ERR_INVALID_ARG),
    (dict(E=0), mb.ERR_INVALID_ARG),
    (dict(E=1025), mb.ERR_INVALID_ARG),
    (dict(k=9, E=8), mb.ERR_INVALID_ARG),
    (dict(k=0), mb.ERR_INVALID_ARG),
    (dict(k=33, E=64), mb.ERR_INVALID_ARG),
    (dict(T=-1), mb.ERR_INVALID_ARG),
    (dict(tile_n=40), mb.ERR_INVALID_ARG),
    (dict(tile_n=48), mb.OK),
    (dict(tile_n=56), mb.ERR_INVALID_ARG),
    (dict(tile_n=16), mb.ERR_INVALID_ARG),
    (dict(tile_n=256), mb.ERR_INVALID_ARG),
    (dict(tile_n=96), mb.OK),
    (dict(tile_n=192), mb.OK),
    (dict(tile_n=224), mb.OK),
    (dict(act_clamp=10.0), mb.OK),
    (dict(act_clamp=float("nan")), mb.ERR_INVALID_ARG),
    (dict(fast_math=1), mb.OK),
    (dict(fast_math=2), mb.ERR_UNSUPPORTED),
    (dict(debug_flags=4), mb.OK),
    (dict(debug_flags=8), mb.ERR_INVALID_ARG),
    (dict(debug_flags=2, H=1024, I=512), mb.ERR_UNSUPPORTED),
    (dict(debug_flags=2, H=1024, I=256), mb.OK),
    (dict(T=0), mb.OK),
])
def test_check_problem(kw, status):
    base = dict(T=128, H=1024, I=512, E=8, k=2)
    base.update(kw)
    p = mb.problem(base.pop("T"), base.pop("H"), base.pop("I"), base.pop("E"), base.pop("k"), **base)
    assert mb.check_problem(p) == status


def test_tile_n_choice():
    assert mb.tile_n(mb.problem(128, 7168, 2048, 256, 8)) == 32       # decode: ~4 rows per expert
    assert mb.tile_n(mb.problem(8192, 7168, 2048, 256, 8)) == 144     # prefill: ~256 rows per expert
    assert mb.tile_n(mb.problem(8192, 7168, 2048, 64, 8)) == 224      # ~1024 rows per expert
    assert mb.tile_n(mb.problem(128, 1024, 512, 8, 2, tile_n=128)) == 128


def test_paired_tiles_choice():
    # pairs of token tiles per weight stage when an expert expects more than one
    # tile (T*k > tile_n*E) and the tile bound is 48..144
    assert mb.paired_tiles(mb.problem(8192, 7168, 2048, 256, 8))           # prefill: 256 > 144 rows
    assert mb.paired_tiles(mb.problem(2048, 4096, 1536, 64, 8))            # 256 rows per expert
    assert not mb.paired_tiles(mb.problem(4000, 7168, 2048, 256, 8))       # 125 rows per expert
    assert not mb.paired_tiles(mb.problem(128, 7168, 2048, 256, 8))        # decode: 32-row tiles
    assert not mb.paired_tiles(mb.problem(8192, 7168, 2048, 64, 8))        # 224-row tiles
    assert mb.paired_tiles(mb.problem(200, 256, 128, 5, 2, tile_n=48))     # 80 > 48 rows
    assert not mb.paired_tiles(mb.problem(200, 256, 128, 5, 2, tile_n=96))
    assert not mb.paired_tiles(mb.problem(200, 256, 128, 5, 2, tile_n=160))


@pytest.mark.parametrize("T,H,I,E,k", [(128, 1024, 512, 8, 2), (8192, 7168, 2048, 256, 8),
                                       (4000, 7168, 2048, 256, 8), (0, 256, 128, 4, 1)])
def test_buffer_sizes(T, H, I, E, k):
    p = mb.problem(T, H, I, E, k)
    ws = mb.workspace_bytes(p)
    P_max = oracle.pool_capacity(1, T, k, E, 128, 128)
    # the pools dominate: Xpool (H B/row) + Hpool (I) + Ypool (2H)
    assert ws >= P_max * (3 * H + I)
    assert ws < P_max * (3 * H + I) * 1.1 + (1 << 24)
    pw = mb.prepared_weight_bytes(p)
    # E2M1 data (1/2 byte per element) + UE8M0 scales (1/32 byte per element)
    assert pw >= E * 3 * H * I * (1 / 2 + 1 / 32) and pw < E * 3 * H * I * (1 / 2 + 1 / 32) + (1 << 20)
    # views tile the workspace without overlap
    fake = ctypes.c_void_p(1 << 40)
    spans = []
    L = mb.load()
    for name, v in mb.VIEWS.items():
        ptr, n = ctypes.c_void_p(), ctypes.c_size_t()
        assert L.moeffn_query(ctypes.byref(p), fake, v, ctypes.byref(ptr), ctypes.byref(n)) == mb.OK
        off = ptr.value - fake.value
        assert off % 1024 == 0 and off + n.value <= ws
        spans.append((off, off + n.value))
    spans.sort()
    for a, b in zip(spans, spans[1:]):
        assert a[1] <= b[0]
    if T:
        ptr, n = ctypes.c_void_p(), ctypes.c_size_t()
        L.moeffn_query(ctypes.byref(p), fake, mb.VIEWS["xpool"], ctypes.byref(ptr), ctypes.byref(n))
        assert n.value == P_max * H


def test_forward_argument_errors_are_synchronous():
    """Rejected before any CUDA call, so these pass without a GPU."""
    L = mb.load()
    p = mb.problem(128, 1024, 512, 8, 2)
    f = ctypes.c_void_p(1 << 20)
    ws = mb.workspace_bytes(p)
    fwd = L.moeffn_forward
    assert fwd(ctypes.byref(p), None, f, f, f, f, f, ws, f, None) == mb.ERR_INVALID_ARG        # null x
    assert fwd(ctypes.byref(p), f, f, f, f, None, f, ws, f, None) == mb.ERR_INVALID_ARG        # null prepared
    assert fwd(ctypes.byref(p), f, f, f, f, f, f, ws - 1, f, None) == mb.ERR_WORKSPACE_TOO_SMALL
    mis = ctypes.c_void_p((1 << 20) + 8)
    assert fwd(ctypes.byref(p), mis, f, f, f, f, f, ws, f, None) == mb.ERR_INVALID_ARG         # misaligned x
    bad = mb.problem(128, 1000, 512, 8, 2)
    assert fwd(ctypes.byref(bad), f, f, f, f, f, f, ws, f, None) == mb.ERR_INVALID_ARG
    prep = L.moeffn_prepare_weights
    assert prep(ctypes.byref(p), None, f, f, f, f, mb.prepared_weight_bytes(p), None) == mb.ERR_INVALID_ARG
    assert prep(ctypes.byref(p), f, f, f, f, f, 10, None) == mb.ERR_WORKSPACE_TOO_SMALL
    route = L.moeffn_route_topk
    assert route(f, 4, 8, 9, f, f, None) == mb.ERR_INVALID_ARG
    assert route(f, 4, 2000, 2, f, f, None) == mb.ERR_INVALID_ARG
    assert route(None, 4, 8, 2, f, f, None) == mb.ERR_INVALID_ARG
    q = L.moeffn_query
    ptr, n = ctypes.c_void_p(), ctypes.c_size_t()
    assert q(ctypes.byref(p), f, 99, ctypes.byref(ptr), ctypes.byref(n)) == mb.ERR_INVALID_ARG
