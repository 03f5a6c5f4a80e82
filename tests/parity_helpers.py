"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
on seeded inputs and compare it with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from moe_expert_ffn_route_gb300 import binding as mb


def up(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def dims(inp):
    T, H = inp["x"].shape
    E, I2, _ = inp["w1"].shape
    return T, H, I2 // 2, E


class GpuRun:
    """One forward on the GPU; keeps the device tensors for inspection."""

    def __init__(self, inp, idx, w, tile_n=0, debug_flags=0, wait_timeout_us=0, weights=None,
                 act_clamp=0.0, fast_math=0):
        T, H, I, E = dims(inp)
        k = idx.shape[1]
        self.prob = mb.problem(T, H, I, E, k, tile_n=tile_n, debug_flags=debug_flags,
                               wait_timeout_us=wait_timeout_us, act_clamp=act_clamp, fast_math=fast_math)
        self.tile_n = mb.tile_n(self.prob)
        self.T, self.H, self.I, self.E, self.k = T, H, I, E, k
        if weights is None:
            weights = upload_weights(inp, self.prob)
        self.prepared = weights
        self.x, self.x_sf = up(inp["x"]), up(inp["x_sf"])
        self.idx, self.w = up(idx.astype(np.int64)), up(w.astype(np.float32))
        self.ws = mb.empty_workspace(self.prob)
        self.y = mb.forward(self.prob, self.x, self.x_sf, self.idx, self.w, self.prepared, self.ws)
        torch.cuda.synchronize()

    def view(self, name, dtype=torch.int32):
        return mb.query(self.prob, self.ws, name).view(dtype)

    def status(self):
        return mb.device_status(self.prob, self.ws)

    def y_bits(self):
        return bf16_bits(self.y)

    def tables(self):
        E, N = self.E, self.T * self.k
        off = self.view("offsets")[: E + 1].cpu().numpy()
        P = int(off[-1])
        return dict(counts=self.view("counts")[:E].cpu().numpy(), offsets=off,
                    tiles=self.view("tiles")[: E + 1].cpu().numpy(),
                    tile_rows=self.view("tile_rows")[:E].cpu().numpy(),
                    slots=self.view("slots")[:N].cpu().numpy().reshape(self.T, self.k),
                    row2tk=self.view("row2tk")[:P].cpu().numpy(),
                    slack=self.view("slack")[: P // 128].cpu().numpy(),
                    wpool=self.view("wpool", torch.float32)[:P].cpu().numpy(), P=P)

    def sf_bytes(self, view: str, rows: np.ndarray, kblocks: int, tabs) -> np.ndarray:
        """UE8M0 codes [len(rows), 4*kblocks] of pool rows from a tile-layout view."""
        raw = self.view(view, torch.uint8)
        rows = np.asarray(rows, np.int64)
        assert rows.size == 0 or (rows.min() >= 0 and rows.max() < tabs["P"]), "pool row out of range"
        e_of = np.searchsorted(tabs["offsets"], rows, side="right") - 1
        r = rows - tabs["offsets"][e_of]
        tr = tabs["tile_rows"][e_of]
        chunk = tabs["tiles"][e_of] + r // tr
        rt = r % tr
        word = (rt // 128) * 128 + (rt % 32) * 4 + (rt % 128) // 32
        kb = np.arange(kblocks)
        byte = ((chunk[:, None] * kblocks + kb[None, :]) * 256 + word[:, None]) * 4
        idx = (byte[:, :, None] + np.arange(4)[None, None, :]).reshape(len(rows), -1)
        assert idx.size == 0 or (idx.min() >= 0 and idx.max() < raw.numel()), "scale index out of range"
        return raw[torch.from_numpy(idx).cuda()].cpu().numpy()

    def pool_rows(self, view: str, rows: np.ndarray, width: int, dtype=torch.uint8) -> np.ndarray:
        """Rows of a [P_max][width] pool view, indices checked on the host first."""
        pool = self.view(view, dtype).view(-1, width)
        rows = np.asarray(rows, np.int64)
        assert rows.size == 0 or (rows.min() >= 0 and rows.max() < pool.shape[0]), "pool row out of range"
        return pool[torch.from_numpy(rows).cuda()].cpu().numpy()


def upload_weights(inp, prob):
    return mb.prepare_weights(prob, up(inp["w1"]), up(inp["w1_sf"]), up(inp["w2"]), up(inp["w2_sf"]))


def e4m3_ulp(v_scaled: np.ndarray) -> np.ndarray:
    """Spacing of E4M3 at |v| (in scaled units, |v| <= 448)."""
    a = np.abs(v_scaled)
    ex = np.floor(np.log2(np.maximum(a, 2.0 ** -9)))
    return np.exp2(np.maximum(ex, -6) - 3)


def compare_l1_codes(gpu_codes, gpu_exp, ref_codes, ref_exp):
    """Fraction of identical L1 codes (a group with a different scale counts
    as 32 non-identical codes) and whether every other value is within one
    E4M3 step of the oracle's value at the oracle's scale."""
    from oracle.grouped import _e4m3
    gc = gpu_codes.reshape(gpu_exp.shape + (32,))
    rc = ref_codes.reshape(ref_exp.shape + (32,))
    same_scale = gpu_exp == ref_exp
    zero = (gc & 0x7F) == 0
    same = (gc == rc) | (zero & ((rc & 0x7F) == 0))
    ident = same & same_scale[..., None]
    frac = ident.mean()
    gv = _e4m3(gc) * np.exp2(gpu_exp[..., None].astype(np.float64))
    rv_scaled = _e4m3(rc)
    rv = rv_scaled * np.exp2(ref_exp[..., None].astype(np.float64))
    ulp = e4m3_ulp(rv_scaled) * np.exp2(ref_exp[..., None].astype(np.float64))
    within = np.abs(gv - rv) <= ulp * (1 + 1e-12)
    return frac, bool(np.all(within | ident)), int((~ident).sum())


def y_errors(y_gpu_bits, y_ref_bits):
    g = oracle.bf16_bits_to_float(y_gpu_bits).astype(np.float64)
    r = oracle.bf16_bits_to_float(y_ref_bits).astype(np.float64)
    d = np.abs(g - r)
    max_rel = d.max() / max(np.abs(r).max(), 1e-30)
    mean_rel = d.sum() / max(np.abs(r).sum(), 1e-30)
    return max_rel, mean_rel
