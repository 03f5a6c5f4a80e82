"""Python binding of libmoeffn (argument marshalling only).

Every function here checks tensor dtypes/devices, passes raw device
pointers and the current CUDA stream to the C ABI declared in
``include/moeffn.h``, and raises ``MoeffnError`` on a non-OK status.  All
computation runs in the library's CUDA kernels; there is no CPU fallback:
if the library cannot be loaded, ``load()`` raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

from . import build as _build

c_int32, c_float, c_void_p, c_size_t = ctypes.c_int32, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t


class Problem(ctypes.Structure):
    """Mirror of ``moeffn_problem``."""
    _fields_ = [
        ("num_tokens", c_int32),
        ("hidden", c_int32),
        ("intermediate", c_int32),
        ("num_experts", c_int32),
        ("topk", c_int32),
        ("act_clamp", c_float),
        ("fast_math", c_int32),
        ("tile_n", c_int32),
        ("wait_timeout_us", c_int32),
        ("debug_flags", c_int32),
    ]


STATUS = {0: "MOEFFN_OK", 1: "MOEFFN_ERR_INVALID_ARG", 2: "MOEFFN_ERR_UNSUPPORTED",
          3: "MOEFFN_ERR_WORKSPACE_TOO_SMALL", 4: "MOEFFN_ERR_CUDA", 5: "MOEFFN_ERR_TIMEOUT",
          6: "MOEFFN_ERR_OUT_OF_BOUNDS"}
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE_TOO_SMALL, ERR_CUDA, ERR_TIMEOUT, ERR_OUT_OF_BOUNDS = range(7)
DEBUG_STARVE_L1 = 1
DEBUG_DUMP_L1_ACC = 2
DEBUG_SPLIT_LAYERS = 4

VIEWS = {"status": 0, "counts": 1, "offsets": 2, "tiles": 3, "slots": 4, "row2tk": 5, "wpool": 6,
         "slack": 7, "xpool": 8, "xpool_sf": 9, "hpool": 10, "hpool_sf": 11, "ypool": 12,
         "tile_rows": 13}

# every symbol include/moeffn.h declares: (restype, argtypes)
SIGNATURES = {
    "moeffn_status_string": (ctypes.c_char_p, [c_int32]),
    "moeffn_abi_version": (c_int32, []),
    "moeffn_check_problem": (c_int32, [ctypes.POINTER(Problem)]),
    "moeffn_tile_n": (c_int32, [ctypes.POINTER(Problem), ctypes.POINTER(c_int32)]),
    "moeffn_paired_tiles": (c_int32, [ctypes.POINTER(Problem), ctypes.POINTER(c_int32)]),
    "moeffn_workspace_bytes": (c_int32, [ctypes.POINTER(Problem), ctypes.POINTER(c_size_t)]),
    "moeffn_prepared_weight_bytes": (c_int32, [ctypes.POINTER(Problem), ctypes.POINTER(c_size_t)]),
    "moeffn_prepare_weights": (c_int32, [ctypes.POINTER(Problem), c_void_p, c_void_p, c_void_p, c_void_p,
                                         c_void_p, c_size_t, c_void_p]),
    "moeffn_route_topk": (c_int32, [c_void_p, c_int32, c_int32, c_int32, c_void_p, c_void_p, c_void_p]),
    "moeffn_forward": (c_int32, [ctypes.POINTER(Problem), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                 c_void_p, c_size_t, c_void_p, c_void_p]),
    "moeffn_forward_profiled": (c_int32, [ctypes.POINTER(Problem), c_void_p, c_void_p, c_void_p, c_void_p,
                                          c_void_p, c_void_p, c_size_t, c_void_p, c_void_p,
                                          ctypes.POINTER(c_void_p)]),
    "moeffn_query": (c_int32, [ctypes.POINTER(Problem), c_void_p, c_int32, ctypes.POINTER(c_void_p),
                               ctypes.POINTER(c_size_t)]),
    "moeffn_get_device_status": (c_int32, [ctypes.POINTER(Problem), c_void_p, c_void_p,
                                           ctypes.POINTER(ctypes.c_uint32)]),
    "moeffn_schedule_tables_noalloc": (c_int32, [c_void_p, c_int32, c_int32, c_int32, c_void_p, c_void_p,
                                                 c_void_p, c_void_p]),
}


class MoeffnError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)}")
        self.status = status


_lib: Optional[ctypes.CDLL] = None


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libmoeffn.so (building it first if absent).  Raises if it cannot."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.lib_path()
    if not os.path.exists(path):
        if not build_if_missing:
            raise FileNotFoundError(f"CUDA library not built: {path}")
        path = _build.build()
    _lib = open_library(path)
    return _lib


def open_library(path: str) -> ctypes.CDLL:
    """Open a build of the library (e.g. the bounds-checked variant) with the
    entry points' signatures set; load() opens the product build."""
    L = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


def _check(status: int, what: str) -> None:
    if status != OK:
        raise MoeffnError(status, what)


def problem(T: int, H: int, I: int, E: int, k: int, tile_n: int = 0, wait_timeout_us: int = 0,
            debug_flags: int = 0, act_clamp: float = 0.0, fast_math: int = 0) -> Problem:
    return Problem(T, H, I, E, k, act_clamp, fast_math, tile_n, wait_timeout_us, debug_flags)


# --------------------------------------------------------------------- host-only calls

def check_problem(prob: Problem) -> int:
    return load().moeffn_check_problem(ctypes.byref(prob))


def tile_n(prob: Problem) -> int:
    v = c_int32()
    _check(load().moeffn_tile_n(ctypes.byref(prob), ctypes.byref(v)), "moeffn_tile_n")
    return v.value


def paired_tiles(prob: Problem) -> bool:
    v = c_int32()
    _check(load().moeffn_paired_tiles(ctypes.byref(prob), ctypes.byref(v)), "moeffn_paired_tiles")
    return v.value == 1


def workspace_bytes(prob: Problem) -> int:
    v = c_size_t()
    _check(load().moeffn_workspace_bytes(ctypes.byref(prob), ctypes.byref(v)), "moeffn_workspace_bytes")
    return v.value


def prepared_weight_bytes(prob: Problem) -> int:
    v = c_size_t()
    _check(load().moeffn_prepared_weight_bytes(ctypes.byref(prob), ctypes.byref(v)),
           "moeffn_prepared_weight_bytes")
    return v.value


def status_string(status: int) -> str:
    return load().moeffn_status_string(status).decode()


# --------------------------------------------------------------------- device calls

def _torch():
    import torch
    return torch


def _stream(stream=None):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return c_void_p(s.cuda_stream)


def _dev(t, name: str, elem_size: int):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.element_size() != elem_size:
        raise TypeError(f"{name}: element size {t.element_size()} != {elem_size}")
    return c_void_p(t.data_ptr())


def empty_workspace(prob: Problem, device=None):
    torch = _torch()
    return torch.empty(workspace_bytes(prob), dtype=torch.uint8, device=device or "cuda")


def prepare_weights(prob: Problem, w1, w1_sf, w2, w2_sf, prepared=None, stream=None):
    """Returns the prepared-weight buffer (uint8 CUDA tensor)."""
    torch = _torch()
    nbytes = prepared_weight_bytes(prob)
    if prepared is None:
        prepared = torch.empty(nbytes, dtype=torch.uint8, device=w1.device)
    E, H, I = prob.num_experts, prob.hidden, prob.intermediate
    if w1.numel() != E * 2 * I * H // 2 or w2.numel() != E * H * I // 2:
        raise ValueError("weight shapes do not match the problem")
    if w1_sf.numel() != E * 2 * I * H // 128 or w2_sf.numel() != E * H * I // 128:
        raise ValueError("weight scale shapes do not match the problem")
    _check(load().moeffn_prepare_weights(ctypes.byref(prob), _dev(w1, "w1", 1), _dev(w1_sf, "w1_sf", 4),
                                         _dev(w2, "w2", 1), _dev(w2_sf, "w2_sf", 4),
                                         _dev(prepared, "prepared", 1), nbytes, _stream(stream)),
           "moeffn_prepare_weights")
    return prepared


def route_topk(logits, k: int, topk_idx=None, topk_w=None, stream=None) -> Tuple:
    torch = _torch()
    T, E = logits.shape
    if logits.dtype != torch.float32:
        raise TypeError("logits must be float32")
    if topk_idx is None:
        topk_idx = torch.empty((T, k), dtype=torch.int64, device=logits.device)
    if topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    _check(load().moeffn_route_topk(_dev(logits, "logits", 4), T, E, k, _dev(topk_idx, "topk_idx", 8),
                                    _dev(topk_w, "topk_w", 4), _stream(stream)), "moeffn_route_topk")
    return topk_idx, topk_w


def forward(prob: Problem, x, x_sf, topk_idx, topk_w, prepared, workspace, y=None, stream=None):
    """y (uint16 BF16 bits [T, H], or a bfloat16 tensor if given) of the fused expert forward."""
    torch = _torch()
    T, H, k = prob.num_tokens, prob.hidden, prob.topk
    if y is None:
        y = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    if x.numel() != T * H or x_sf.numel() != T * H // 128:
        raise ValueError("x / x_sf shape does not match the problem")
    if topk_idx.numel() != T * k or topk_w.numel() != T * k:
        raise ValueError("topk shape does not match the problem")
    if topk_idx.dtype != torch.int64 or topk_w.dtype != torch.float32:
        raise TypeError("topk_idx must be int64 and topk_w float32")
    _check(load().moeffn_forward(ctypes.byref(prob), _dev(x, "x", 1), _dev(x_sf, "x_sf", 4),
                                 _dev(topk_idx, "topk_idx", 8), _dev(topk_w, "topk_w", 4),
                                 _dev(prepared, "prepared", 1), _dev(workspace, "workspace", 1),
                                 workspace.numel(), _dev(y, "y", 2), _stream(stream)),
           "moeffn_forward")
    return y


def forward_profiled(prob: Problem, x, x_sf, topk_idx, topk_w, prepared, workspace, y, events, stream=None):
    """forward() recording five torch.cuda.Event objects at the stage boundaries
    (before tables, after gather, after L1, after L2, after combine)."""
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    for ev in events:
        ev.record(s)              # materialise the underlying cudaEvent_t
    handles = (c_void_p * 5)(*[ev.cuda_event for ev in events])
    _check(load().moeffn_forward_profiled(ctypes.byref(prob), _dev(x, "x", 1), _dev(x_sf, "x_sf", 4),
                                          _dev(topk_idx, "topk_idx", 8), _dev(topk_w, "topk_w", 4),
                                          _dev(prepared, "prepared", 1), _dev(workspace, "workspace", 1),
                                          workspace.numel(), _dev(y, "y", 2), c_void_p(s.cuda_stream), handles),
           "moeffn_forward_profiled")
    return y


def query(prob: Problem, workspace, view: str):
    """A uint8 view of one region of the workspace (see moeffn_view)."""
    ptr, n = c_void_p(), c_size_t()
    _check(load().moeffn_query(ctypes.byref(prob), c_void_p(workspace.data_ptr()), VIEWS[view],
                               ctypes.byref(ptr), ctypes.byref(n)), "moeffn_query")
    off = ptr.value - workspace.data_ptr()
    return workspace[off: off + n.value]


def device_status(prob: Problem, workspace, stream=None) -> Tuple[int, int, int]:
    """(status, raw error bits, detail) after synchronising the stream."""
    words = (ctypes.c_uint32 * 2)()
    st = load().moeffn_get_device_status(ctypes.byref(prob), c_void_p(workspace.data_ptr()),
                                         _stream(stream), words)
    return st, words[0], words[1]


def schedule_tables_noalloc(topk_idx, num_experts: int, counts, offsets, slots, stream=None) -> None:
    """Routing tables without any device allocation (see moeffn_schedule_tables_noalloc):
    fills the caller's counts [E], offsets [E+1] and slots [T*k] int32 tensors."""
    T, k = topk_idx.shape
    _check(load().moeffn_schedule_tables_noalloc(_dev(topk_idx, "topk_idx", 8), T, num_experts, k,
                                                 _dev(counts, "counts", 4), _dev(offsets, "offsets", 4),
                                                 _dev(slots, "slots", 4), _stream(stream)),
           "moeffn_schedule_tables_noalloc")
