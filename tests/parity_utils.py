"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and compare it, chunk by chunk, with the double-precision oracle.

Tolerances (per element):
* masked entries and padded rows: the output bits are exactly +0.0;
* fp32 IO: |gpu - oracle| <= 2e-6 (oracle in double, not rounded);
* bf16 / fp16 IO: the gpu value is within 1 ulp of the oracle rounded once
  to the IO dtype (distance counted in representable values; +0 and -0 are
  the same point).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import seeded_inputs as si

F32_ABS_TOL = 2e-6
HALF_ULP_TOL = 1

_BITS = {"f32": torch.int32, "bf16": torch.int16, "f16": torch.int16}
_NP_BITS = {"f32": np.uint32, "bf16": np.uint16, "f16": np.uint16}


def to_bits(t: torch.Tensor, dtype: str) -> np.ndarray:
    """Raw element bits of a (CPU or CUDA) tensor as a numpy unsigned array."""
    return t.detach().contiguous().view(_BITS[dtype]).cpu().numpy().view(_NP_BITS[dtype])


def from_bits(bits: np.ndarray, dtype: str, device) -> torch.Tensor:
    arr = np.ascontiguousarray(bits.astype(_NP_BITS[dtype], copy=False))
    signed = arr.view(np.int32 if dtype == "f32" else np.int16)
    return torch.from_numpy(signed.copy()).to(device).view(si.TORCH_DTYPES[dtype])


def decode(bits: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return bits.view(np.float32).astype(np.float64)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def ordered(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Map sign-magnitude float bits to integers ordered like the values (+0 == -0)."""
    width = 32 if dtype == "f32" else 16
    b = bits.astype(np.int64)
    sign = b >> (width - 1)
    mag = b & ((1 << (width - 1)) - 1)
    return np.where(sign == 1, -mag, mag)


class Stats:
    def __init__(self):
        self.max_abs = 0.0
        self.max_ulp = 0
        self.ulp_hist = np.zeros(4, dtype=np.int64)   # 0, 1, 2, >2
        self.live = 0
        self.masked = 0
        self.bad_masked = 0
        self.bad_live = 0

    def __repr__(self):
        return (f"Stats(live={self.live}, masked={self.masked}, max_abs={self.max_abs:.3g}, "
                f"max_ulp={self.max_ulp}, ulp_hist={self.ulp_hist.tolist()}, bad_masked={self.bad_masked}, "
                f"bad_live={self.bad_live})")

    @property
    def ok(self):
        return self.bad_masked == 0 and self.bad_live == 0


def compare_rows(gpu_bits: np.ndarray, ref: np.ndarray, kept, dtype: str, stats: Stats):
    """gpu_bits [rows, S] raw bits, ref [rows, S] float64 oracle, kept = (c0, c1) kept column range per row."""
    S = gpu_bits.shape[1]
    c0, c1 = kept
    col = np.arange(S)[None, :]
    live = (col >= c0[:, None]) & (col < c1[:, None])
    stats.live += int(live.sum())
    stats.masked += int((~live).sum())
    stats.bad_masked += int(np.count_nonzero(gpu_bits[~live]))
    if not live.any():
        return
    g = gpu_bits[live]
    r = ref[live]
    if dtype == "f32":
        err = np.abs(decode(g, dtype) - r)
        err = np.where(np.isnan(err), np.inf, err)
        stats.max_abs = max(stats.max_abs, float(err.max()))
        stats.bad_live += int(np.count_nonzero(err > F32_ABS_TOL))
    else:
        code = si.DTYPE_CODES[dtype]
        rb = oracle.round_to(r, code)
        ulp = np.abs(ordered(g, dtype) - ordered(rb, dtype))
        stats.max_ulp = max(stats.max_ulp, int(ulp.max()))
        stats.ulp_hist += np.bincount(np.minimum(ulp, 3), minlength=4)[:4]
        stats.max_abs = max(stats.max_abs, float(np.abs(decode(g, dtype) - r).max()))
        stats.bad_live += int(np.count_nonzero(ulp > HALF_ULP_TOL))


def kept_for_rows(seq_lens: np.ndarray, M: int, S: int, q0: int, q1: int, mask_kind=0, window=0):
    """(c0, c1) kept column range of each row q in [q0, q1)."""
    c0, c1 = oracle.kept_ranges(seq_lens, S, mask_kind, window)          # [B, S]
    q = np.arange(q0, q1)
    b, r = q // (M * S), q % S
    return c0[b, r], c1[b, r]


def check_forward(x_bits_rows, y_bits_rows, seq_lens, B, M, S, scale, dtype, q0, q1, stats, threads=8,
                  mask_kind=0, window=0):
    """Oracle forward on rows [q0, q1) (x given as raw bits) vs the GPU's y bits."""
    ref = oracle.forward(x_bits_rows, seq_lens, B, M, S, scale, si.DTYPE_CODES[dtype], q0, q1, threads=threads,
                         mask_kind=mask_kind, window=window)
    compare_rows(y_bits_rows.reshape(q1 - q0, S), ref, kept_for_rows(seq_lens, M, S, q0, q1, mask_kind, window),
                 dtype, stats)


def check_backward(y_bits_rows, dy_bits_rows, dx_bits_rows, seq_lens, B, M, S, scale, dtype, q0, q1, stats,
                   threads=8, mask_kind=0, window=0):
    ref = oracle.backward(y_bits_rows, dy_bits_rows, seq_lens, B, M, S, scale, si.DTYPE_CODES[dtype], q0, q1,
                          threads=threads, mask_kind=mask_kind, window=window)
    compare_rows(dx_bits_rows.reshape(q1 - q0, S), ref, kept_for_rows(seq_lens, M, S, q0, q1, mask_kind, window),
                 dtype, stats)


def row_chunks(q0: int, q1: int, S: int, max_elems: int = 1 << 23):
    step = max(1, max_elems // max(1, S))
    for a in range(q0, q1, step):
        yield a, min(q1, a + step)


def oracle_forward_bits(x_bits: np.ndarray, seq_lens, B, M, S, scale, dtype, threads=8, mask_kind=0,
                        window=0) -> np.ndarray:
    """Oracle forward of a whole small tensor, rounded once to the IO dtype (raw bits)."""
    out = np.empty(B * M * S * S, dtype=_NP_BITS[dtype])
    flat = x_bits.reshape(-1)
    for a, b in row_chunks(0, B * M * S, S):
        ref = oracle.forward(flat[a * S:b * S], seq_lens, B, M, S, scale, si.DTYPE_CODES[dtype], a, b,
                             threads=threads, mask_kind=mask_kind, window=window)
        out[a * S:b * S] = oracle.round_to(ref, si.DTYPE_CODES[dtype]).reshape(-1)
    return out.reshape(B, M, S, S)


def masked_bits_all_zero(out: torch.Tensor, seq_lens_dev: torch.Tensor, dtype: str, mask_kind=0, window=0) -> bool:
    """On the device, for every row of every batch: no masked element has a nonzero bit."""
    B, M, S, _ = out.shape
    bits = out.view(_BITS[dtype])
    col = torch.arange(S, device=out.device)
    row = torch.arange(S, device=out.device)
    for b in range(B):
        L = int(seq_lens_dev[b].clamp(0, S).item())
        if mask_kind == 1:
            kept = (col[None, :] < L) & (row[:, None] < L)
        else:
            kept = (col[None, :] <= row[:, None]) & (row[:, None] < L)
            if mask_kind == 2:
                kept &= col[None, :] > row[:, None] - window
        if bool(((bits[b] != 0) & ~kept).any().item()):
            return False
    return True


def live_row_sums_close_to_one(y: torch.Tensor, seq_lens_dev: torch.Tensor, tol: float) -> bool:
    """On the device: every live row of y sums to 1 within tol (padded rows sum to 0)."""
    B, M, S, _ = y.shape
    for b in range(B):
        L = int(seq_lens_dev[b].clamp(0, S).item())
        sums = y[b].to(torch.float64).sum(-1)                     # [M, S]
        if L > 0 and float((sums[:, :L] - 1.0).abs().max().item()) > tol:
            return False
        if L < S and float(sums[:, L:].abs().max().item()) != 0.0:
            return False
    return True
