"""Grouped-tril masked softmax for GB300 (sm_103a): thin Python binding of libgtms.

The compute runs in hand-written CUDA kernels behind the C ABI of
``include/gtms.h``. This module only marshals arguments: it passes device
pointers, sizes and the current CUDA stream to ``gtms_forward`` /
``gtms_backward`` and turns a non-zero status into an exception. There is no
CPU or PyTorch fallback: if ``libgtms.so`` is missing or cannot be loaded,
every call raises.

Operation ("Attention-Mask-Optimization" README, operator behaviour): for
X[B,M,S,S] and per-batch lengths L_b = seq_lens[b], row r keeps columns
c <= r when r < L_b; kept entries get softmax(scale * x), the rest +0.0.
Backward ("ops(8): self-attention 的 CUDA 实现及优化 (下)", section 2.1):
dx = scale * y * (dy - rowsum(dy * y)) on kept entries, +0.0 elsewhere.
"""
from __future__ import annotations

import ctypes
import os
import threading

from ._build import LIB_PATH, build_library  # noqa: F401  (re-exported for build scripts)

GTMS_F32, GTMS_BF16, GTMS_F16 = 0, 1, 2
GTMS_OK, GTMS_ERR_INVALID_ARG, GTMS_ERR_UNSUPPORTED, GTMS_ERR_CUDA, GTMS_ERR_TIMEOUT = 0, 1, 2, 3, 4
GTMS_MAX_S = 65536
GTMS_MASK_GROUPED_TRIL, GTMS_MASK_LENGTH, GTMS_MASK_SLIDING_WINDOW = 0, 1, 2

EXPORTED_SYMBOLS = ("gtms_forward", "gtms_backward", "gtms_status_string", "gtms_version",
                    "gtms_kernel_name", "gtms_kernel_name_masked", "gtms_kernel_name_explicit",
                    "gtms_device_pointer_of_host",
                    "gtms_forward_masked",
                    "gtms_backward_masked", "gtms_forward_explicit", "gtms_backward_explicit",
                    "gtms_attention_softmax_backward", "gtms_forward_staged")

_lib = None
_lock = threading.Lock()


class GtmsError(RuntimeError):
    """A libgtms call returned a non-zero status."""

    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libgtms.so (built in-tree by ``build_library``); raise if it is absent."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"libgtms.so not found at {p}: build it with "
                               "masked_softmax_attention_gb300.build_library() (needs nvcc); "
                               "there is no fallback implementation")
        lib = ctypes.CDLL(p)
        vp, i64 = ctypes.c_void_p, ctypes.c_int64
        lib.gtms_forward.argtypes = [vp, vp, vp, i64, i64, i64, ctypes.c_float, ctypes.c_int, vp]
        lib.gtms_forward.restype = ctypes.c_int
        lib.gtms_backward.argtypes = [vp, vp, vp, vp, i64, i64, i64, ctypes.c_float, ctypes.c_int, vp]
        lib.gtms_backward.restype = ctypes.c_int
        lib.gtms_forward_staged.argtypes = [vp, vp, vp, i64, i64, i64, ctypes.c_float, ctypes.c_int, vp]
        lib.gtms_forward_staged.restype = ctypes.c_int
        lib.gtms_forward_masked.argtypes = [vp, vp, vp, i64, i64, i64, ctypes.c_float, ctypes.c_int, i64,
                                            ctypes.c_int, vp]
        lib.gtms_forward_masked.restype = ctypes.c_int
        lib.gtms_backward_masked.argtypes = [vp, vp, vp, vp, i64, i64, i64, ctypes.c_float, ctypes.c_int, i64,
                                             ctypes.c_int, vp]
        lib.gtms_backward_masked.restype = ctypes.c_int
        lib.gtms_forward_explicit.argtypes = [vp, vp, vp, i64, i64, i64, i64, ctypes.c_float, ctypes.c_int, vp]
        lib.gtms_forward_explicit.restype = ctypes.c_int
        lib.gtms_backward_explicit.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, ctypes.c_float, ctypes.c_int, vp]
        lib.gtms_backward_explicit.restype = ctypes.c_int
        lib.gtms_attention_softmax_backward.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, ctypes.c_float,
                                                        ctypes.c_int, vp, vp]
        lib.gtms_attention_softmax_backward.restype = ctypes.c_int
        lib.gtms_status_string.argtypes = [ctypes.c_int]
        lib.gtms_status_string.restype = ctypes.c_char_p
        lib.gtms_version.argtypes = []
        lib.gtms_version.restype = ctypes.c_int
        lib.gtms_kernel_name.argtypes = [ctypes.c_int, i64, ctypes.c_int, ctypes.c_int]
        lib.gtms_kernel_name.restype = ctypes.c_char_p
        lib.gtms_kernel_name_masked.argtypes = [ctypes.c_int, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int, i64]
        lib.gtms_kernel_name_masked.restype = ctypes.c_char_p
        lib.gtms_kernel_name_explicit.argtypes = [ctypes.c_int, i64, ctypes.c_int]
        lib.gtms_kernel_name_explicit.restype = ctypes.c_char_p
        lib.gtms_device_pointer_of_host.argtypes = [vp, ctypes.POINTER(ctypes.c_void_p)]
        lib.gtms_device_pointer_of_host.restype = ctypes.c_int
        if path is None:
            _lib = lib
        return lib


# ---------------------------------------------------------------------------
# Raw C-ABI calls: integer pointers in, status code out.
# ---------------------------------------------------------------------------

def gtms_forward(x, y, seq_lens, B, M, S, scale, dtype, stream) -> int:
    return load_library().gtms_forward(x, y, seq_lens, B, M, S, scale, dtype, stream)


def gtms_backward(y, dy, dx, seq_lens, B, M, S, scale, dtype, stream) -> int:
    return load_library().gtms_backward(y, dy, dx, seq_lens, B, M, S, scale, dtype, stream)


def gtms_forward_staged(x, y, seq_lens, B, M, S, scale, dtype, stream) -> int:
    return load_library().gtms_forward_staged(x, y, seq_lens, B, M, S, scale, dtype, stream)


def gtms_forward_masked(x, y, seq_lens, B, M, S, scale, mask_kind, window, dtype, stream) -> int:
    return load_library().gtms_forward_masked(x, y, seq_lens, B, M, S, scale, mask_kind, window, dtype, stream)


def gtms_backward_masked(y, dy, dx, seq_lens, B, M, S, scale, mask_kind, window, dtype, stream) -> int:
    return load_library().gtms_backward_masked(y, dy, dx, seq_lens, B, M, S, scale, mask_kind, window, dtype, stream)


def gtms_forward_explicit(x, y, mask, mask_batches, B, M, S, scale, dtype, stream) -> int:
    return load_library().gtms_forward_explicit(x, y, mask, mask_batches, B, M, S, scale, dtype, stream)


def gtms_backward_explicit(y, dy, dx, mask, mask_batches, B, M, S, scale, dtype, stream) -> int:
    return load_library().gtms_backward_explicit(y, dy, dx, mask, mask_batches, B, M, S, scale, dtype, stream)


def gtms_attention_softmax_backward(p, dout, v, ds, seq_lens, B, M, S, head_dim, scale, dtype, status,
                                    stream) -> int:
    return load_library().gtms_attention_softmax_backward(p, dout, v, ds, seq_lens, B, M, S, head_dim, scale, dtype,
                                                          status, stream)


def status_string(status: int) -> str:
    return load_library().gtms_status_string(status).decode()


def gtms_version() -> int:
    return load_library().gtms_version()


def kernel_name(direction: int, S: int, dtype: int, aligned16: bool = True) -> str:
    return load_library().gtms_kernel_name(direction, S, dtype, 1 if aligned16 else 0).decode()


def kernel_name_masked(direction: int, S: int, dtype: int, mask_kind: int, window: int = 0,
                       aligned16: bool = True) -> str:
    return load_library().gtms_kernel_name_masked(direction, S, dtype, 1 if aligned16 else 0, mask_kind,
                                                  window).decode()


def kernel_name_explicit(direction: int, S: int, dtype: int) -> str:
    return load_library().gtms_kernel_name_explicit(direction, S, dtype).decode()


def device_pointer_of_host(host_ptr: int) -> int:
    """Device address of a page-locked host buffer (``gtms_device_pointer_of_host``)."""
    out = ctypes.c_void_p()
    rc = load_library().gtms_device_pointer_of_host(host_ptr, ctypes.byref(out))
    if rc != GTMS_OK:
        raise GtmsError("gtms_device_pointer_of_host", rc)
    return out.value


# ---------------------------------------------------------------------------
# Tensor API (torch provides device memory and the stream, nothing else).
# ---------------------------------------------------------------------------

def _dtype_code(t) -> int:
    import torch

    codes = {torch.float32: GTMS_F32, torch.bfloat16: GTMS_BF16, torch.float16: GTMS_F16}
    if t.dtype not in codes:
        raise TypeError(f"unsupported dtype {t.dtype}; expected float32, bfloat16 or float16")
    return codes[t.dtype]


def _check_scores(name, t):
    if t.dim() != 4 or t.shape[-1] != t.shape[-2]:
        raise ValueError(f"{name} must be [B, M, S, S], got {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _check_lens(seq_lens, B, device):
    import torch

    if seq_lens.dtype != torch.int32 or seq_lens.shape != (B,) or seq_lens.device != device \
            or not seq_lens.is_contiguous():
        raise ValueError("seq_lens must be a contiguous int32 CUDA tensor of shape [B] on the scores' device")


def forward(x, seq_lens, scale: float = 1.0, out=None, mask_kind: int = GTMS_MASK_GROUPED_TRIL, window: int = 0):
    """y = masked softmax(scale * x) (grouped tril by default); ``out`` may be ``x`` (in place)."""
    import torch

    _check_scores("x", x)
    B, M, S, _ = x.shape
    _check_lens(seq_lens, B, x.device)
    y = torch.empty_like(x) if out is None else out
    if y.shape != x.shape or y.dtype != x.dtype or y.device != x.device or not y.is_contiguous():
        raise ValueError("out must match x in shape, dtype, device and be contiguous")
    stream = torch.cuda.current_stream(x.device).cuda_stream
    rc = gtms_forward_masked(x.data_ptr(), y.data_ptr(), seq_lens.data_ptr(), B, M, S, float(scale),
                             int(mask_kind), int(window), _dtype_code(x), stream)
    if rc != GTMS_OK:
        raise GtmsError("gtms_forward_masked", rc)
    return y


def forward_staged(x, seq_lens, scale: float = 1.0, out=None):
    """``forward`` computed by the staged kernel (gtms_forward_staged: rows brought into shared
    memory by TMA bulk copies); the same values within the parity tolerances."""
    import torch

    _check_scores("x", x)
    B, M, S, _ = x.shape
    _check_lens(seq_lens, B, x.device)
    y = torch.empty_like(x) if out is None else out
    if y.shape != x.shape or y.dtype != x.dtype or y.device != x.device or not y.is_contiguous():
        raise ValueError("out must match x in shape, dtype, device and be contiguous")
    stream = torch.cuda.current_stream(x.device).cuda_stream
    rc = gtms_forward_staged(x.data_ptr(), y.data_ptr(), seq_lens.data_ptr(), B, M, S, float(scale), _dtype_code(x),
                             stream)
    if rc != GTMS_OK:
        raise GtmsError("gtms_forward_staged", rc)
    return y


def backward(y, dy, seq_lens, scale: float = 1.0, out=None, mask_kind: int = GTMS_MASK_GROUPED_TRIL,
             window: int = 0):
    """dx = scale * y * (dy - rowsum(dy * y)) under the mask; ``out`` may be ``y`` or ``dy``."""
    import torch

    _check_scores("y", y)
    _check_scores("dy", dy)
    if dy.shape != y.shape or dy.dtype != y.dtype or dy.device != y.device:
        raise ValueError("dy must match y in shape, dtype and device")
    B, M, S, _ = y.shape
    _check_lens(seq_lens, B, y.device)
    dx = torch.empty_like(y) if out is None else out
    if dx.shape != y.shape or dx.dtype != y.dtype or dx.device != y.device or not dx.is_contiguous():
        raise ValueError("out must match y in shape, dtype, device and be contiguous")
    stream = torch.cuda.current_stream(y.device).cuda_stream
    rc = gtms_backward_masked(y.data_ptr(), dy.data_ptr(), dx.data_ptr(), seq_lens.data_ptr(), B, M, S,
                              float(scale), int(mask_kind), int(window), _dtype_code(y), stream)
    if rc != GTMS_OK:
        raise GtmsError("gtms_backward_masked", rc)
    return dx


def _check_mask(mask, B, S, device):
    import torch

    if mask.dtype != torch.uint8 or mask.dim() != 3 or mask.shape[1:] != (S, S) or mask.shape[0] not in (1, B) \
            or mask.device != device or not mask.is_contiguous():
        raise ValueError("mask must be a contiguous uint8 CUDA tensor [1 or B, S, S] on the scores' device")


def forward_explicit(x, mask, scale: float = 1.0, out=None):
    """Softmax of scale * x over the entries whose mask byte is nonzero (mask uint8 [1 or B, S, S],
    shared by the heads); +0.0 elsewhere, all-masked rows zero. ``out`` may be ``x``."""
    import torch

    _check_scores("x", x)
    B, M, S, _ = x.shape
    _check_mask(mask, B, S, x.device)
    y = torch.empty_like(x) if out is None else out
    if y.shape != x.shape or y.dtype != x.dtype or y.device != x.device or not y.is_contiguous():
        raise ValueError("out must match x in shape, dtype, device and be contiguous")
    stream = torch.cuda.current_stream(x.device).cuda_stream
    rc = gtms_forward_explicit(x.data_ptr(), y.data_ptr(), mask.data_ptr(), mask.shape[0], B, M, S, float(scale),
                               _dtype_code(x), stream)
    if rc != GTMS_OK:
        raise GtmsError("gtms_forward_explicit", rc)
    return y


def backward_explicit(y, dy, mask, scale: float = 1.0, out=None):
    """Backward of forward_explicit over the same kept entries; ``out`` may be ``y`` or ``dy``."""
    import torch

    _check_scores("y", y)
    _check_scores("dy", dy)
    if dy.shape != y.shape or dy.dtype != y.dtype or dy.device != y.device:
        raise ValueError("dy must match y in shape, dtype and device")
    B, M, S, _ = y.shape
    _check_mask(mask, B, S, y.device)
    dx = torch.empty_like(y) if out is None else out
    if dx.shape != y.shape or dx.dtype != y.dtype or dx.device != y.device or not dx.is_contiguous():
        raise ValueError("out must match y in shape, dtype, device and be contiguous")
    stream = torch.cuda.current_stream(y.device).cuda_stream
    rc = gtms_backward_explicit(y.data_ptr(), dy.data_ptr(), dx.data_ptr(), mask.data_ptr(), mask.shape[0], B, M, S,
                                float(scale), _dtype_code(y), stream)
    if rc != GTMS_OK:
        raise GtmsError("gtms_backward_explicit", rc)
    return dx


def attention_softmax_backward(p, dout, v, seq_lens, scale: float = 1.0, out=None, status=None):
    """dS = scale * P * (dO V^T - rowsum(dO V^T * P)) on the grouped-tril kept entries, with the GEMM on the
    tensor cores; ``p`` [B,M,S,S], ``dout`` / ``v`` [B,M,S,d] (d 64 or 128), bf16 or fp16. ``status`` (an
    optional int32 CUDA tensor of one element) receives 1 if an internal wait of the kernel ran out."""
    import torch

    _check_scores("p", p)
    B, M, S, _ = p.shape
    for name, t in (("dout", dout), ("v", v)):
        if t.dim() != 4 or t.shape[:3] != p.shape[:3] or t.dtype != p.dtype or t.device != p.device \
                or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [B, M, S, d] tensor matching p")
    if dout.shape != v.shape:
        raise ValueError("dout and v must have the same shape")
    _check_lens(seq_lens, B, p.device)
    ds = torch.empty_like(p) if out is None else out
    if ds.shape != p.shape or ds.dtype != p.dtype or ds.device != p.device or not ds.is_contiguous():
        raise ValueError("out must match p in shape, dtype, device and be contiguous")
    stream = torch.cuda.current_stream(p.device).cuda_stream
    rc = gtms_attention_softmax_backward(p.data_ptr(), dout.data_ptr(), v.data_ptr(), ds.data_ptr(),
                                         seq_lens.data_ptr(), B, M, S, dout.shape[3], float(scale), _dtype_code(p),
                                         None if status is None else status.data_ptr(), stream)
    if rc != GTMS_OK:
        raise GtmsError("gtms_attention_softmax_backward", rc)
    return ds


def attention_softmax_backward_host(p, dout, v, seq_lens, scale: float = 1.0, out=None, status=None, device=None):
    """``attention_softmax_backward`` on pinned host tensors: the kernel reads P, dO, V and writes dS in host
    memory (see ``forward_host``). ``status``, if given, is an int32 CUDA tensor of one element."""
    import torch

    for name, t in (("p", p), ("dout", dout), ("v", v), ("seq_lens", seq_lens)):
        _check_pinned(name, t)
    if p.dim() != 4 or p.shape[-1] != p.shape[-2] or dout.dim() != 4 or dout.shape != v.shape \
            or dout.shape[:3] != p.shape[:3] or dout.dtype != p.dtype or v.dtype != p.dtype:
        raise ValueError("p must be [B, M, S, S]; dout and v [B, M, S, d] of p's dtype")
    if seq_lens.dtype != torch.int32 or seq_lens.shape != p.shape[:1]:
        raise ValueError("seq_lens must be int32 [B]")
    ds = torch.empty_like(p).pin_memory() if out is None else out
    _check_pinned("out", ds)
    B, M, S, _ = p.shape
    stream = torch.cuda.current_stream(device).cuda_stream
    dp = device_pointer_of_host
    rc = gtms_attention_softmax_backward(dp(p.data_ptr()), dp(dout.data_ptr()), dp(v.data_ptr()),
                                         dp(ds.data_ptr()), dp(seq_lens.data_ptr()), B, M, S, dout.shape[3],
                                         float(scale), _dtype_code(p), None if status is None else status.data_ptr(),
                                         stream)
    if rc != GTMS_OK:
        raise GtmsError("gtms_attention_softmax_backward", rc)
    return ds


def _check_pinned(name, t):
    if t.is_cuda or not t.is_pinned() or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous page-locked (pinned) CPU tensor")


def forward_host(x, seq_lens, scale: float = 1.0, out=None, device=None):
    """Forward on pinned host tensors: the kernels read x and write y in host memory.

    ``x`` [B,M,S,S], ``seq_lens`` int32 [B] and ``out`` (allocated pinned if
    omitted) stay in page-locked host memory; the call is enqueued on the
    current stream of ``device`` and returns at once (synchronise before
    reading ``out``).
    """
    import torch

    _check_pinned("x", x)
    _check_pinned("seq_lens", seq_lens)
    if x.dim() != 4 or x.shape[-1] != x.shape[-2] or seq_lens.dtype != torch.int32 or seq_lens.shape != x.shape[:1]:
        raise ValueError("x must be [B, M, S, S] and seq_lens int32 [B]")
    y = torch.empty_like(x).pin_memory() if out is None else out
    _check_pinned("out", y)
    B, M, S, _ = x.shape
    stream = torch.cuda.current_stream(device).cuda_stream
    rc = gtms_forward(device_pointer_of_host(x.data_ptr()), device_pointer_of_host(y.data_ptr()),
                      device_pointer_of_host(seq_lens.data_ptr()), B, M, S, float(scale), _dtype_code(x), stream)
    if rc != GTMS_OK:
        raise GtmsError("gtms_forward", rc)
    return y


def backward_host(y, dy, seq_lens, scale: float = 1.0, out=None, device=None):
    """Backward on pinned host tensors (see ``forward_host``)."""
    import torch

    for name, t in (("y", y), ("dy", dy), ("seq_lens", seq_lens)):
        _check_pinned(name, t)
    if dy.shape != y.shape or dy.dtype != y.dtype or y.dim() != 4 or seq_lens.dtype != torch.int32 \
            or seq_lens.shape != y.shape[:1]:
        raise ValueError("y and dy must be matching [B, M, S, S] tensors and seq_lens int32 [B]")
    dx = torch.empty_like(y).pin_memory() if out is None else out
    _check_pinned("out", dx)
    B, M, S, _ = y.shape
    stream = torch.cuda.current_stream(device).cuda_stream
    rc = gtms_backward(device_pointer_of_host(y.data_ptr()), device_pointer_of_host(dy.data_ptr()),
                       device_pointer_of_host(dx.data_ptr()), device_pointer_of_host(seq_lens.data_ptr()),
                       B, M, S, float(scale), _dtype_code(y), stream)
    if rc != GTMS_OK:
        raise GtmsError("gtms_backward", rc)
    return dx


def _autograd_function():
    import torch

    class GroupedTrilMaskSoftmax(torch.autograd.Function):
        """Autograd wrapper: forward and backward both run the CUDA kernels."""

        @staticmethod
        def forward(ctx, x, seq_lens, scale):
            y = forward(x.contiguous(), seq_lens, scale)
            ctx.save_for_backward(y, seq_lens)
            ctx.scale = scale
            return y

        @staticmethod
        def backward(ctx, dy):
            y, seq_lens = ctx.saved_tensors
            return backward(y, dy.contiguous(), seq_lens, ctx.scale), None, None

    return GroupedTrilMaskSoftmax


_fn = None


def grouped_tril_mask_softmax(x, seq_lens, scale: float = 1.0):
    """Differentiable op: ``y = grouped_tril_mask_softmax(x, seq_lens, scale)``."""
    global _fn
    if _fn is None:
        _fn = _autograd_function()
    return _fn.apply(x, seq_lens, float(scale))
