"""Double-precision CPU oracle for the grouped-tril masked softmax (fwd + bwd).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
legs of ``bench.py`` may import this package. It shares no code with the CUDA
library in ``masked_softmax_attention_gb300`` and neither side imports the
other; the product path never falls back to it.

The arithmetic lives in ``gtms_oracle.c`` (plain loops, double accumulation,
one row at a time); this module compiles it with the host C compiler and
wraps it with ctypes. Every function cites the passage it follows:

* mask and forward -- "Attention-Mask-Optimization" README, section
  "算子行为（融合下面的计算）" (operator behaviour) and its printed output;
  scale inside the exponent -- "优化ScaledMaskSoftmax算子", section 4.1.
* backward -- "ops(8): self-attention 的 CUDA 实现及优化 (下)", section 2.1
  (Softmax 求导) and section 2.2 (scale applied in the softmax backward).

Parity pins (``tests/test_oracle_pins.py``) tie every function here to the
pages' worked example, closed forms, finite differences and independent
library routines; no function is "parity unpinned".
"""
from __future__ import annotations

import concurrent.futures as _cf
import ctypes
import os
import subprocess
import threading

import numpy as np

F32, BF16, F16, F64 = 0, 1, 2, 3
_ELEM_BYTES = {F32: 4, BF16: 2, F16: 2, F64: 8}
_BITS_DTYPE = {F32: np.uint32, BF16: np.uint16, F16: np.uint16, F64: np.float64}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gtms_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libgtms_oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        cc = os.environ.get("CC", "cc")
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call([cc, "-O2", "-fno-fast-math", "-std=c11", "-fPIC", "-shared",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            i64, vp, dp = ctypes.c_int64, ctypes.c_void_p, ctypes.c_double
            lib.gtms_oracle_forward.argtypes = [vp, ctypes.c_int, vp, i64, i64, i64, dp, i64, i64, vp]
            lib.gtms_oracle_backward.argtypes = [vp, vp, ctypes.c_int, vp, i64, i64, i64, dp, i64, i64, vp]
            ci = ctypes.c_int
            lib.gtms_oracle_forward_masked.argtypes = [vp, ci, vp, i64, i64, i64, dp, ci, i64, i64, i64, vp]
            lib.gtms_oracle_backward_masked.argtypes = [vp, vp, ci, vp, i64, i64, i64, dp, ci, i64, i64, i64, vp]
            lib.gtms_oracle_forward_masked.restype = ctypes.c_int
            lib.gtms_oracle_backward_masked.restype = ctypes.c_int
            lib.gtms_oracle_forward_explicit.argtypes = [vp, ci, vp, i64, i64, i64, i64, dp, i64, i64, vp]
            lib.gtms_oracle_backward_explicit.argtypes = [vp, vp, ci, vp, i64, i64, i64, i64, dp, i64, i64, vp]
            lib.gtms_oracle_forward_explicit.restype = ctypes.c_int
            lib.gtms_oracle_backward_explicit.restype = ctypes.c_int
            lib.gtms_oracle_attn_dscores.argtypes = [vp, vp, vp, ci, vp, i64, i64, i64, i64, dp, i64, i64, vp]
            lib.gtms_oracle_attn_dscores.restype = ctypes.c_int
            lib.gtms_oracle_round.argtypes = [vp, i64, ctypes.c_int, vp]
            lib.gtms_oracle_decode.argtypes = [vp, i64, ctypes.c_int, vp]
            for f in (lib.gtms_oracle_forward, lib.gtms_oracle_backward,
                      lib.gtms_oracle_round, lib.gtms_oracle_decode):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _as_bits(a: np.ndarray, dtype: int) -> np.ndarray:
    """View an array of raw element bits (or float32 / float64 values) as contiguous storage."""
    a = np.ascontiguousarray(a)
    if a.itemsize != _ELEM_BYTES[dtype]:
        raise ValueError(f"element size {a.itemsize} does not match dtype code {dtype}")
    return a


def _row_chunks(row_begin: int, row_end: int, threads: int):
    n = row_end - row_begin
    if threads <= 1 or n < 2 * threads:
        return [(row_begin, row_end)]
    step = -(-n // (threads * 4))
    return [(r, min(r + step, row_end)) for r in range(row_begin, row_end, step)]


def _run_rows(kernel, ins, dtype, seq_lens, B, M, S, scale, row_begin, row_end, threads, mask=None):
    lib = _load()
    seq = np.ascontiguousarray(seq_lens, dtype=np.int32)
    if seq.shape != (B,):
        raise ValueError("seq_lens must have shape [B]")
    rows = row_end - row_begin
    out = np.empty((rows, S), dtype=np.float64)
    arrs = [_as_bits(a, dtype).reshape(-1) for a in ins]
    for a in arrs:
        if a.size != rows * S:
            raise ValueError("input rows do not match the requested row range")
    eb = _ELEM_BYTES[dtype]

    def work(chunk):
        r0, r1 = chunk
        off = (r0 - row_begin) * S
        ptrs = [ctypes.c_void_p(a.ctypes.data + off * eb) for a in arrs]
        extra = () if mask is None else (int(mask[0]), int(mask[1]))
        rc = getattr(lib, kernel)(*ptrs, dtype, seq.ctypes.data, B, M, S, float(scale), *extra, r0, r1,
                                  ctypes.c_void_p(out.ctypes.data + off * 8))
        if rc != 0:
            raise ValueError(f"{kernel} rejected its arguments")

    chunks = _row_chunks(row_begin, row_end, threads)
    if len(chunks) == 1:
        work(chunks[0])
    else:
        with _cf.ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(work, chunks))
    return out


MASK_GROUPED_TRIL, MASK_LENGTH, MASK_SLIDING_WINDOW = 0, 1, 2


def forward(x, seq_lens, B, M, S, scale, dtype, row_begin=0, row_end=None, threads=1, mask_kind=0, window=0):
    """Masked softmax of rows [row_begin, row_end) of X[B,M,S,S] in double.

    ``x`` holds exactly those rows (raw element bits for bf16/fp16, uint32 bits
    or float32 values for fp32, float64 for F64). Returns float64 [rows, S].
    ``mask_kind``: 0 grouped tril (default), 1 length mask, 2 sliding causal
    window of width ``window`` (see gtms_oracle.c).
    """
    row_end = B * M * S if row_end is None else row_end
    return _run_rows("gtms_oracle_forward_masked", [x], dtype, seq_lens, B, M, S, scale,
                     row_begin, row_end, threads, mask=(mask_kind, window))


def backward(y, dy, seq_lens, B, M, S, scale, dtype, row_begin=0, row_end=None, threads=1, mask_kind=0,
             window=0):
    """Softmax backward dx = scale*y*(dy - rowsum(dy*y)) under the same mask, in double."""
    row_end = B * M * S if row_end is None else row_end
    return _run_rows("gtms_oracle_backward_masked", [y, dy], dtype, seq_lens, B, M, S, scale,
                     row_begin, row_end, threads, mask=(mask_kind, window))


def _run_explicit(kernel, ins, dtype, mask, B, M, S, scale, row_begin, row_end, threads):
    lib = _load()
    mk = np.ascontiguousarray(mask, dtype=np.uint8)
    if mk.ndim != 3 or mk.shape[1:] != (S, S) or mk.shape[0] not in (1, B):
        raise ValueError("mask must be uint8 [1 or B, S, S]")
    rows = row_end - row_begin
    out = np.empty((rows, S), dtype=np.float64)
    arrs = [_as_bits(a, dtype).reshape(-1) for a in ins]
    eb = _ELEM_BYTES[dtype]

    def work(chunk):
        r0, r1 = chunk
        off = (r0 - row_begin) * S
        ptrs = [ctypes.c_void_p(a.ctypes.data + off * eb) for a in arrs]
        rc = getattr(lib, kernel)(*ptrs, dtype, mk.ctypes.data, mk.shape[0], B, M, S, float(scale), r0, r1,
                                  ctypes.c_void_p(out.ctypes.data + off * 8))
        if rc != 0:
            raise ValueError(f"{kernel} rejected its arguments")

    chunks = _row_chunks(row_begin, row_end, threads)
    if len(chunks) == 1:
        work(chunks[0])
    else:
        with _cf.ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(work, chunks))
    return out


def forward_explicit(x, mask, B, M, S, scale, dtype, row_begin=0, row_end=None, threads=1):
    """Softmax of scale*x over the entries whose mask byte is nonzero ("优化ScaledMaskSoftmax算子",
    sections 2.2 / 3.1 / 4.1); ``mask`` uint8 [1 or B, S, S], shared by the heads. Float64 [rows, S]."""
    row_end = B * M * S if row_end is None else row_end
    return _run_explicit("gtms_oracle_forward_explicit", [x], dtype, mask, B, M, S, scale, row_begin, row_end,
                         threads)


def backward_explicit(y, dy, mask, B, M, S, scale, dtype, row_begin=0, row_end=None, threads=1):
    """Backward of forward_explicit: dx = scale*y*(dy - rowsum(dy*y)) on kept entries, 0 elsewhere."""
    row_end = B * M * S if row_end is None else row_end
    return _run_explicit("gtms_oracle_backward_explicit", [y, dy], dtype, mask, B, M, S, scale, row_begin, row_end,
                         threads)


def attn_dscores(p, dout, v, seq_lens, B, M, S, d, scale, dtype, row_begin=0, row_end=None, threads=1):
    """Attention-backward step dS = scale * P * (dP - rowsum(dP * P)), dP = dO V^T, grouped tril mask
    ("ops(8): self-attention 的 CUDA 实现及优化 (下)", section 2.1). ``p`` holds rows [row_begin, row_end)
    of P [B,M,S,S]; ``dout`` and ``v`` are whole [B,M,S,d] tensors. Float64 [rows, S]."""
    lib = _load()
    row_end = B * M * S if row_end is None else row_end
    seq = np.ascontiguousarray(seq_lens, dtype=np.int32)
    pa = _as_bits(np.asarray(p), dtype).reshape(-1)
    da = _as_bits(np.asarray(dout), dtype).reshape(-1)
    va = _as_bits(np.asarray(v), dtype).reshape(-1)
    rows = row_end - row_begin
    if seq.shape != (B,) or pa.size != rows * S or da.size != B * M * S * d or va.size != B * M * S * d:
        raise ValueError("attn_dscores: shapes do not match")
    out = np.empty((rows, S), dtype=np.float64)
    eb = _ELEM_BYTES[dtype]

    def work(chunk):
        r0, r1 = chunk
        off = (r0 - row_begin) * S
        rc = lib.gtms_oracle_attn_dscores(ctypes.c_void_p(pa.ctypes.data + off * eb), da.ctypes.data, va.ctypes.data,
                                          dtype, seq.ctypes.data, B, M, S, d, float(scale), r0, r1,
                                          ctypes.c_void_p(out.ctypes.data + off * 8))
        if rc != 0:
            raise ValueError("gtms_oracle_attn_dscores rejected its arguments")

    chunks = _row_chunks(row_begin, row_end, threads)
    if len(chunks) == 1:
        work(chunks[0])
    else:
        with _cf.ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(work, chunks))
    return out


def round_to(values, dtype: int) -> np.ndarray:
    """Round doubles once (to nearest, ties to even) into raw bits of ``dtype``."""
    lib = _load()
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, dtype=_BITS_DTYPE[dtype])
    if lib.gtms_oracle_round(v.ctypes.data, v.size, dtype, out.ctypes.data) != 0:
        raise ValueError("bad dtype")
    return out


def decode(bits, dtype: int) -> np.ndarray:
    """Decode raw element bits of ``dtype`` into float64."""
    lib = _load()
    b = _as_bits(np.asarray(bits), dtype)
    out = np.empty(b.shape, dtype=np.float64)
    if lib.gtms_oracle_decode(b.ctypes.data, b.size, dtype, out.ctypes.data) != 0:
        raise ValueError("bad dtype")
    return out


def kept_prefix_lengths(seq_lens, M: int, S: int) -> np.ndarray:
    """n_r per (b, r): the kept-prefix length, as the oracle's mask defines it.

    Returned shape [B, S]; the same for every head m (README, operator behaviour).
    """
    L = np.clip(np.asarray(seq_lens, dtype=np.int64), 0, S)[:, None]
    r = np.arange(S, dtype=np.int64)[None, :]
    return np.where(r < L, r + 1, 0)


def kept_ranges(seq_lens, S: int, mask_kind: int = 0, window: int = 0):
    """(c0, c1) per (b, r), each [B, S]: the kept column range of every mask family."""
    L = np.clip(np.asarray(seq_lens, dtype=np.int64), 0, S)[:, None]
    r = np.arange(S, dtype=np.int64)[None, :]
    live = r < L
    if mask_kind == 1:
        c1 = np.where(live, L, 0)
        c0 = np.zeros_like(c1)
    else:
        c1 = np.where(live, r + 1, 0)
        c0 = np.where(live, np.maximum(r - window + 1, 0), 0) if mask_kind == 2 else np.zeros_like(c1)
    return c0, c1
