"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Element-by-element on seeded inputs at sizes the oracle finishes in seconds
(several rows per team, ragged kept prefixes, partial 16-byte units), on edge
sizes, and at the full workload sizes on sampled (b, m) slices plus
properties checked on every row. Backward inputs y are the oracle's own
forward output rounded to the IO dtype, never the GPU's.
"""
import numpy as np
import pytest
import torch

import masked_softmax_attention_gb300 as gtms
import oracle
import seeded_inputs as si
from parity_utils import (Stats, check_backward, check_forward, from_bits, live_row_sums_close_to_one,
                          masked_bits_all_zero, oracle_forward_bits, row_chunks, to_bits)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gtms.build_library()
    gtms.load_library()
    return torch.device("cuda:0")


def _lens_dev(w, dev):
    return torch.from_numpy(si.seq_lens(w)).to(dev)


def run_and_check(w, dev, backward=True, x_cpu=None, offset_elems=0, mask_kind=0, window=0):
    """Full element-wise parity of forward (and backward) for a small workload."""
    mk = dict(mask_kind=mask_kind, window=window)
    B, M, S = w.B, w.M, w.S
    lens = si.seq_lens(w)
    lens_d = torch.from_numpy(lens).to(dev)
    x = si.make_x(w, "cpu") if x_cpu is None else x_cpu
    x_bits = to_bits(x, w.dtype).reshape(-1)

    def place(t):
        if offset_elems == 0:
            return t.to(dev)
        buf = torch.empty(t.numel() + offset_elems, dtype=t.dtype, device=dev)
        view = buf[offset_elems:].view(t.shape)
        view.copy_(t)
        return view

    y = place(torch.zeros_like(x))
    gtms.forward(place(x), lens_d, w.scale, out=y, **mk)
    torch.cuda.synchronize()
    y_bits = to_bits(y, w.dtype).reshape(-1)
    st = Stats()
    for a, b in row_chunks(0, w.rows, S):
        check_forward(x_bits[a * S:b * S], y_bits[a * S:b * S], lens, B, M, S, w.scale, w.dtype, a, b, st, **mk)
    assert st.ok, f"forward {w.describe()} {mk}: {st}"
    if not backward:
        return st, None
    y_or = oracle_forward_bits(x_bits, lens, B, M, S, w.scale, w.dtype, **mk)
    dy = si.make_dy(w, "cpu")
    dy_bits = to_bits(dy, w.dtype).reshape(-1)
    dx = place(torch.zeros_like(dy))
    gtms.backward(place(from_bits(y_or, w.dtype, "cpu")), place(dy), lens_d, w.scale, out=dx, **mk)
    torch.cuda.synchronize()
    dx_bits = to_bits(dx, w.dtype).reshape(-1)
    yb = y_or.reshape(-1)
    sb = Stats()
    for a, b in row_chunks(0, w.rows, S):
        check_backward(yb[a * S:b * S], dy_bits[a * S:b * S], dx_bits[a * S:b * S], lens, B, M, S, w.scale,
                       w.dtype, a, b, sb, **mk)
    assert sb.ok, f"backward {w.describe()} {mk}: {sb}"
    return st, sb


# ---------------------------------------------------------------------------
# Workload-shaped cases small enough for a full comparison
# ---------------------------------------------------------------------------

REDUCED = [
    si.WORKLOADS["worked_example"],
    si.custom("s1000_f32", 2, 3, 1000, "f32", 1.0, seq_lens=(1000, 637), seed=11),
    si.custom("s1000_f32_u", 3, 2, 1000, "f32", 1.0, seq_len_range=(1, 1000), seed=12),
    si.custom("s2048_bf16", 2, 2, 2048, "bf16", 0.125, seq_lens=(2048, 1500), x_std=2.0, seed=13),
    si.custom("s4096_bf16", 2, 1, 4096, "bf16", 0.125, seq_lens=(4096, 3001), x_std=2.0, seed=14),
    si.custom("s8192_f16", 1, 2, 8192, "f16", 0.125, seq_lens=(8192,), spike_prob=0.01, seed=15),
    si.custom("s8192_f32", 1, 1, 8192, "f32", 1.0, seq_lens=(6001,), seed=16),
    si.custom("s8192_bf16", 1, 1, 8192, "bf16", 0.125, seq_lens=(8192,), x_std=2.0, seed=17),
]


@pytest.mark.parametrize("w", REDUCED, ids=[w.name for w in REDUCED])
def test_reduced_workloads(dev, w):
    run_and_check(w, dev)


EDGE_S = [1, 2, 3, 5, 7, 8, 9, 15, 16, 17, 31, 32, 33, 63, 64, 65, 100, 127, 128, 129, 255, 256, 257,
          511, 512, 513, 1000, 1023, 1024, 1025, 2047, 2048, 2049, 4095, 4096, 4097, 8191, 8192]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("S", EDGE_S)
def test_edge_sizes(dev, S, dtype):
    """Lengths -1 (clamped to 0), 0, 1, S//2+1 and S+3 (clamped to S) in one call."""
    M = 2 if S <= 1024 else 1
    w = si.custom(f"edge{S}", 5, M, S, dtype, 0.125 if dtype != "f32" else 1.0,
                  seq_lens=(-1, 0, 1, S // 2 + 1, S + 3), x_std=2.0, seed=S)
    run_and_check(w, dev)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("S", [5, 64, 1000, 2048, 8192])
def test_element_aligned_buffers(dev, S, dtype):
    """Buffers offset by one element: the element-granular path, same tolerances."""
    w = si.custom(f"unaligned{S}", 2, 1, S, dtype, 0.5, seq_lens=(S, S // 3 + 1), seed=100 + S)
    run_and_check(w, dev, offset_elems=1)


def test_zero_length_batches_produce_all_zero_output(dev):
    w = si.custom("zeros", 3, 2, 256, "f32", 1.0, seq_lens=(0, 0, 0), seed=3)
    x = si.make_x(w, dev)
    lens = _lens_dev(w, dev)
    y = torch.full_like(x, float("nan"))
    gtms.forward(x, lens, 1.0, out=y)
    dx = torch.full_like(x, float("nan"))
    gtms.backward(x, x, lens, 1.0, out=dx)
    torch.cuda.synchronize()
    assert bool((y.view(torch.int32) == 0).all()) and bool((dx.view(torch.int32) == 0).all())


# ---------------------------------------------------------------------------
# Properties: masked inputs are never read, every output is written, aliasing
# ---------------------------------------------------------------------------

def _kept_mask(lens, M, S, dev):
    n = torch.from_numpy(oracle.kept_prefix_lengths(lens, M, S)).to(dev)        # [B, S]
    col = torch.arange(S, device=dev)
    return (col[None, None, :] < n[:, :, None])[:, None]                        # [B, 1, S, S]


@pytest.mark.parametrize("dtype,S", [("f32", 1000), ("bf16", 2048), ("f16", 8192), ("f32", 5), ("bf16", 33),
                                     ("f32", 8192), ("bf16", 16384)])
def test_masked_inputs_are_not_read(dev, dtype, S):
    w = si.custom("sentinel", 3, 2, S, dtype, 0.125, seq_lens=(S, S // 2 + 1, 0), seed=21)
    lens = si.seq_lens(w)
    lens_d = torch.from_numpy(lens).to(dev)
    kept = _kept_mask(lens, w.M, S, dev)
    x = si.make_x(w, dev)
    dy = si.make_dy(w, dev)
    y_ref = gtms.forward(x, lens_d, w.scale)
    dx_ref = gtms.backward(y_ref, dy, lens_d, w.scale)
    nan = torch.tensor(float("nan"), dtype=x.dtype, device=dev)
    x_nan = torch.where(kept, x, nan)
    y_in = torch.where(kept, y_ref, nan)
    dy_nan = torch.where(kept, dy, nan)
    y = gtms.forward(x_nan, lens_d, w.scale)
    dx = gtms.backward(y_in, dy_nan, lens_d, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16 if dtype != "f32" else torch.int32),
                       y_ref.view(torch.int16 if dtype != "f32" else torch.int32))
    assert torch.equal(dx.view(torch.int16 if dtype != "f32" else torch.int32),
                       dx_ref.view(torch.int16 if dtype != "f32" else torch.int32))


@pytest.mark.parametrize("dtype,S", [("f32", 1000), ("bf16", 2048), ("f16", 8192), ("f32", 7), ("f32", 8192),
                                     ("bf16", 16384)])
def test_every_output_element_is_written(dev, dtype, S):
    w = si.custom("prefill", 2, 2, S, dtype, 1.0, seq_lens=(S, S // 3), seed=22)
    lens_d = _lens_dev(w, dev)
    x = si.make_x(w, dev)
    ref = gtms.forward(x, lens_d, 1.0)
    y = torch.full_like(x, float("nan"))
    gtms.forward(x, lens_d, 1.0, out=y)
    dref = gtms.backward(ref, x, lens_d, 1.0)
    dx = torch.full_like(x, float("nan"))
    gtms.backward(ref, x, lens_d, 1.0, out=dx)
    torch.cuda.synchronize()
    assert not bool(torch.isnan(y).any()) and not bool(torch.isnan(dx).any())
    assert torch.equal(y, ref) and torch.equal(dx, dref)
    assert masked_bits_all_zero(y, lens_d, dtype) and masked_bits_all_zero(dx, lens_d, dtype)


@pytest.mark.parametrize("dtype,S", [("f32", 1000), ("bf16", 2048), ("f16", 8192), ("f32", 5), ("f32", 8192),
                                     ("bf16", 16384)])
def test_exact_aliasing_is_in_place(dev, dtype, S):
    w = si.custom("alias", 2, 3, S, dtype, 0.125, seq_lens=(S, S // 2 + 3), seed=23)
    lens_d = _lens_dev(w, dev)
    x = si.make_x(w, dev)
    dy = si.make_dy(w, dev)
    y_ref = gtms.forward(x, lens_d, w.scale)
    dx_ref = gtms.backward(y_ref, dy, lens_d, w.scale)
    xi = x.clone()
    gtms.forward(xi, lens_d, w.scale, out=xi)
    dyi = dy.clone()
    gtms.backward(y_ref, dyi, lens_d, w.scale, out=dyi)
    yi = y_ref.clone()
    gtms.backward(yi, dy, lens_d, w.scale, out=yi)
    torch.cuda.synchronize()
    assert torch.equal(xi, y_ref)
    assert torch.equal(dyi, dx_ref)
    assert torch.equal(yi, dx_ref)


@pytest.mark.parametrize("offset", [0, 1])
@pytest.mark.parametrize("dtype,S", [("f32", 1000), ("bf16", 2048), ("f16", 8192), ("f32", 5), ("f32", 8192)])
def test_guard_bands_untouched(dev, dtype, S, offset):
    """Canary bytes around each output stay intact (compute-sanitizer stand-in)."""
    w = si.custom("guard", 2, 2, S, dtype, 1.0, seq_lens=(S, 1), seed=24)
    lens_d = _lens_dev(w, dev)
    x = si.make_x(w, dev)
    n = x.numel()
    pad = 4096 + offset
    for direction in ("fwd", "bwd"):
        buf = torch.full((n + 2 * pad,), -7.0, dtype=x.dtype, device=dev)
        canary = buf.clone()
        out = buf[pad:pad + n].view(x.shape)
        if direction == "fwd":
            gtms.forward(x, lens_d, 1.0, out=out)
        else:
            gtms.backward(x, x, lens_d, 1.0, out=out)
        torch.cuda.synchronize()
        assert torch.equal(buf[:pad], canary[:pad]) and torch.equal(buf[pad + n:], canary[pad + n:])


def test_row0_is_exactly_one_hot(dev):
    for dtype, S in (("f32", 1000), ("bf16", 2048), ("f16", 8192), ("f32", 5), ("f32", 8192), ("bf16", 16384)):
        w = si.custom("row0", 3, 4, S, dtype, 0.37, seq_lens=(S, 1, 2), x_std=3.0, seed=25)
        y = gtms.forward(si.make_x(w, dev), _lens_dev(w, dev), w.scale)
        torch.cuda.synchronize()
        assert bool((y[:, :, 0, 0].float() == 1.0).all())
        assert bool((y[:, :, 0, 1:].float() == 0.0).all())


def test_side_stream_and_determinism(dev):
    w = si.custom("stream", 4, 8, 1000, "f32", 1.0, seq_len_range=(1, 1000), seed=26)
    lens_d = _lens_dev(w, dev)
    x = si.make_x(w, dev)
    dy = si.make_dy(w, dev)
    y0 = gtms.forward(x, lens_d)
    d0 = gtms.backward(y0, dy, lens_d)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        y1 = gtms.forward(x, lens_d)
        d1 = gtms.backward(y1, dy, lens_d)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1) and torch.equal(d0, d1)


def test_autograd_function(dev):
    w = si.custom("autograd", 2, 2, 64, "f32", 0.5, seq_lens=(64, 20), seed=27)
    lens_d = _lens_dev(w, dev)
    x = si.make_x(w, dev).requires_grad_(True)
    dy = si.make_dy(w, dev)
    y = gtms.grouped_tril_mask_softmax(x, lens_d, 0.5)
    y.backward(dy)
    torch.cuda.synchronize()
    ref_y = gtms.forward(x.detach(), lens_d, 0.5)
    ref_dx = gtms.backward(ref_y, dy, lens_d, 0.5)
    assert torch.equal(y.detach(), ref_y) and torch.equal(x.grad, ref_dx)


# ---------------------------------------------------------------------------
# Full workload sizes, in the launch configuration the benchmark times
# ---------------------------------------------------------------------------

FULL = ["worked_example", "s1000_b3", "s1000_b12", "s2048_bf16", "s8192_f16", "s4096_bf16"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload(dev, name):
    w = si.WORKLOADS[name]
    B, M, S = w.B, w.M, w.S
    lens = si.seq_lens(w)
    lens_d = torch.from_numpy(lens).to(dev)
    x = si.make_x(w, dev)
    y = gtms.forward(x, lens_d, w.scale)
    torch.cuda.synchronize()
    # every row: masked bits zero, live rows sum to 1
    assert masked_bits_all_zero(y, lens_d, w.dtype)
    tol = {"f32": 1e-5, "bf16": 2.0 ** -7, "f16": 2.0 ** -9}[w.dtype]
    assert live_row_sums_close_to_one(y, lens_d, tol)
    # sampled slices: element-wise against the oracle
    slices = si.sample_slices(w, 6)
    st = Stats()
    for b, m in slices:
        xs = to_bits(x[b, m], w.dtype).reshape(-1)
        ys = to_bits(y[b, m], w.dtype).reshape(-1)
        q_base = (b * M + m) * S
        for a, e in row_chunks(0, S, S):
            check_forward(xs[a * S:e * S], ys[a * S:e * S], lens, B, M, S, w.scale, w.dtype,
                          q_base + a, q_base + e, st)
    assert st.ok, f"forward {w.describe()}: {st}"
    if not w.backward:
        return
    # backward: y input = GPU forward everywhere except the sampled slices,
    # which hold the oracle's own forward (those are the slices compared).
    dy = si.make_dy(w, dev)
    y_in = y
    for b, m in slices:
        xs = to_bits(x[b, m], w.dtype).reshape(1, 1, S, S)
        ref = oracle_forward_bits(xs, lens[b:b + 1], 1, 1, S, w.scale, w.dtype)
        y_in[b, m].copy_(from_bits(ref, w.dtype, "cpu").view(S, S))
    dx = gtms.backward(y_in, dy, lens_d, w.scale)
    torch.cuda.synchronize()
    assert masked_bits_all_zero(dx, lens_d, w.dtype)
    assert bool(torch.isfinite(dx).all())
    sb = Stats()
    for b, m in slices:
        ys = to_bits(y_in[b, m], w.dtype).reshape(-1)
        gs = to_bits(dy[b, m], w.dtype).reshape(-1)
        ds = to_bits(dx[b, m], w.dtype).reshape(-1)
        q_base = (b * M + m) * S
        for a, e in row_chunks(0, S, S):
            check_backward(ys[a * S:e * S], gs[a * S:e * S], ds[a * S:e * S], lens, B, M, S, w.scale, w.dtype,
                           q_base + a, q_base + e, sb)
    assert sb.ok, f"backward {w.describe()}: {sb}"
    del x, y, dy, dx, y_in
    torch.cuda.empty_cache()


@pytest.mark.parametrize("chunk", [1, 2, 5])
def test_host_pipeline_matches_device_calls(dev, chunk):
    """Pinned host buffers through the chunked 3-stream pipeline give the same
    bits as the device calls on resident tensors."""
    from masked_softmax_attention_gb300.pipeline import HostPipeline

    w = si.custom("pipe", 5, 3, 1000, "f32", 1.0, seq_len_range=(1, 1000), seed=31)
    lens = si.seq_lens(w)
    lens_d = torch.from_numpy(lens).to(dev)
    x = si.make_x(w, dev)
    dy = si.make_dy(w, dev)
    y_ref = gtms.forward(x, lens_d, 1.0)
    dx_ref = gtms.backward(y_ref, dy, lens_d, 1.0)
    x_h, dy_h = x.cpu().pin_memory(), dy.cpu().pin_memory()
    y_h = torch.full_like(x_h, float("nan")).pin_memory()
    dx_h = torch.full_like(x_h, float("nan")).pin_memory()
    pipe = HostPipeline(w.B, w.M, w.S, torch.float32, dev, chunk_batches=chunk)
    for _ in range(2):
        pipe.run(x_h, torch.from_numpy(lens).pin_memory(), 1.0, y_h, dy_h, dx_h)
        torch.cuda.current_stream().synchronize()
        assert torch.equal(y_h, y_ref.cpu()) and torch.equal(dx_h, dx_ref.cpu())


# ---------------------------------------------------------------------------
# Staged forward (gtms_forward_staged): each row's kept units brought into shared
# memory by one TMA bulk copy, several rows ahead
# ---------------------------------------------------------------------------

STAGED = [
    si.custom("st1000_f32", 2, 3, 1000, "f32", 1.0, seq_lens=(1000, 637), seed=111),
    si.custom("st2048_bf16", 2, 2, 2048, "bf16", 0.125, seq_lens=(2048, 1500), x_std=2.0, seed=112),
    si.custom("st4096_bf16", 2, 1, 4096, "bf16", 0.125, seq_lens=(4096, 3001), x_std=2.0, seed=113),
    si.custom("st8192_f16", 1, 2, 8192, "f16", 0.125, seq_lens=(8192,), spike_prob=0.01, seed=114),
    si.custom("st4096_f32", 2, 1, 4096, "f32", 0.7, seq_lens=(4096, 2049), seed=115),
] + [si.custom(f"stedge{S}_{dt}", 5, 2, S, dt, -0.5 if S == 64 else 0.125, seq_lens=(-1, 0, 1, S // 2 + 1, S + 3),
               x_std=2.0, seed=S + 116) for S, dt in ((8, "f32"), (64, "bf16"), (1024, "f16"), (1032, "f32"),
                                                       (2056, "bf16"))]


def _staged_run_and_check(w, dev, call=None, x_cpu=None):
    """Full element-wise parity of a staged forward against the oracle; the output buffer starts as NaN,
    so every element must be written."""
    S = w.S
    lens = si.seq_lens(w)
    x = si.make_x(w, "cpu") if x_cpu is None else x_cpu
    x_bits = to_bits(x, w.dtype).reshape(-1)
    x_d = x.to(dev)
    y = torch.full_like(x_d, float("nan"))
    lens_d = torch.from_numpy(lens).to(dev)
    if call is None:
        gtms.forward_staged(x_d, lens_d, w.scale, out=y)
    else:
        call(x_d, y, lens_d)
    torch.cuda.synchronize()
    y_bits = to_bits(y, w.dtype).reshape(-1)
    st = Stats()
    for a, b in row_chunks(0, w.rows, S):
        check_forward(x_bits[a * S:b * S], y_bits[a * S:b * S], lens, w.B, w.M, S, w.scale, w.dtype, a, b, st)
    assert st.ok, f"staged forward {w.describe()}: {st}"
    return y


@pytest.mark.parametrize("w", STAGED, ids=[w.name for w in STAGED])
def test_staged_forward_matches_oracle(dev, w):
    _staged_run_and_check(w, dev)


@pytest.mark.parametrize("dtype,S", [("f32", 1000), ("bf16", 2048), ("f16", 8192)])
def test_staged_forward_agrees_with_forward_and_does_not_read_masked_inputs(dev, dtype, S):
    """Where the staged kernel's team shape is the forward's (a team of 64 with 4 units per thread),
    the arithmetic is the same, so the bits are; NaN in every masked input changes nothing."""
    w = si.custom("staged_eq", 3, 2, S, dtype, 0.125, seq_lens=(S, S // 2 + 1, 0), seed=117)
    lens_d = torch.from_numpy(si.seq_lens(w)).to(dev)
    x = si.make_x(w, dev)
    y = gtms.forward_staged(x, lens_d, w.scale)
    nan = torch.tensor(float("nan"), dtype=x.dtype, device=dev)
    y_nan = gtms.forward_staged(torch.where(_kept_mask(si.seq_lens(w), w.M, S, dev), x, nan), lens_d, w.scale)
    torch.cuda.synchronize()
    bits = torch.int32 if dtype == "f32" else torch.int16
    assert torch.equal(y_nan.view(bits), y.view(bits))
    if gtms.kernel_name(2, S, w.dtype_code).split(",")[1:3] == gtms.kernel_name(0, S, w.dtype_code).split(",")[1:3]:
        assert torch.equal(y.view(bits), gtms.forward(x, lens_d, w.scale).view(bits))


def _build_staged_give_up_probe():
    """Compile tests/staged_give_up_probe.cu (the staged forward with no copy ever issued) into a library
    of its own under _build/; libgtms.so is not touched."""
    import ctypes
    import os
    import subprocess

    from masked_softmax_attention_gb300 import _build as b

    src = os.path.join(b.ROOT, "tests", "staged_give_up_probe.cu")
    out_dir = os.path.join(b.ROOT, "_build", "test_probe")
    os.makedirs(out_dir, exist_ok=True)
    lib_path = os.path.join(out_dir, "libgtms_staged_give_up_probe.so")
    deps = [src] + [os.path.join(b.CSRC, f) for f in os.listdir(b.CSRC)] + [os.path.join(b.INCLUDE, "gtms.h")]
    if not os.path.exists(lib_path) or any(os.path.getmtime(d) > os.path.getmtime(lib_path) for d in deps):
        tmp = lib_path + f".{os.getpid()}.tmp"
        subprocess.run([b.nvcc_path(), *b.ARCH, *b.NVCC_FLAGS, "-shared", src, "-o", tmp], check=True,
                       capture_output=True, text=True)
        os.replace(tmp, lib_path)
    lib = ctypes.CDLL(lib_path)
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    lib.gtms_test_staged_no_copies.argtypes = [vp, vp, vp, i64, i64, i64, ctypes.c_float, ctypes.c_int, vp,
                                               ctypes.c_uint64]
    lib.gtms_test_staged_no_copies.restype = ctypes.c_int
    return lib


@pytest.mark.parametrize("dtype,S", [("f32", 1000), ("bf16", 2048)])
def test_staged_forward_gives_up_on_copies_that_never_arrive(dev, dtype, S):
    """Failure path without a GPU fault: in a test build that issues no copy, every team's first wait
    runs out (after 100 us), the team stops staging and reads its rows from global memory. The kernel
    must end promptly and its output must still match the oracle element by element."""
    import time

    probe = _build_staged_give_up_probe()
    w = si.custom("staged_give_up", 2, 4, S, dtype, 0.125, seq_lens=(S, S // 3 + 1), x_std=2.0, seed=118)
    t0 = time.monotonic()

    def call(x_d, y, lens_d):
        rc = probe.gtms_test_staged_no_copies(x_d.data_ptr(), y.data_ptr(), lens_d.data_ptr(), w.B, w.M, S,
                                              w.scale, w.dtype_code, torch.cuda.current_stream().cuda_stream,
                                              100_000)
        assert rc == 0

    _staged_run_and_check(w, dev, call=call)
    assert time.monotonic() - t0 < 60.0


# ---------------------------------------------------------------------------
# Long rows (up to S = 65536): rows of 32 KB and more stream in two passes, one CTA per row
# ---------------------------------------------------------------------------

LONG_FULL = [(8200, "f32"), (8200, "bf16"), (12288, "f16"), (16384, "f32"), (16384, "bf16")]


@pytest.mark.parametrize("S,dtype", LONG_FULL)
def test_long_rows_full_comparison(dev, S, dtype):
    """Every element, lengths S, S//2+1, 1 and 0 (rows of several stream batches, ragged last batch)."""
    w = si.custom(f"long{S}", 4, 1, S, dtype, 0.125 if dtype != "f32" else 0.7,
                  seq_lens=(S, S // 2 + 1, 1, 0), x_std=2.0, seed=S + 7)
    run_and_check(w, dev)


@pytest.mark.parametrize("S,dtype,L", [(32768, "f32", 20001), (32768, "bf16", 32768), (65536, "bf16", 40000),
                                       (65536, "f16", 65536), (65536, "f32", 30001)])
def test_long_rows_sampled(dev, S, dtype, L):
    """Largest rows (two-pass stream kernels, up to 256 KB rows): sampled rows
    element by element, every row's masked bits and live row sums on the device."""
    w = si.custom(f"long{S}", 1, 1, S, dtype, 0.125, seq_lens=(L,), seed=S + L)
    lens = si.seq_lens(w)
    lens_d = torch.from_numpy(lens).to(dev)
    x = si.make_x(w, dev)
    y = gtms.forward(x, lens_d, w.scale)
    dy = si.make_dy(w, dev)
    rng = np.random.default_rng(S)
    rows = sorted({0, 1, 2, L - 1, L - 2, L // 2, L, S - 1} | set(rng.integers(0, L, 12).tolist()))
    rows = [r for r in rows if 0 <= r < S]
    # backward input: the oracle's own forward on the sampled rows, the GPU's elsewhere
    y_in = y.clone()
    for r in rows:
        xs = to_bits(x[0, 0, r:r + 1], w.dtype).reshape(-1)
        ref = oracle.forward(xs, lens, 1, 1, S, w.scale, w.dtype_code, r, r + 1)
        y_in[0, 0, r].copy_(from_bits(oracle.round_to(ref, w.dtype_code), w.dtype, "cpu").view(S))
    dx = gtms.backward(y_in, dy, lens_d, w.scale)
    torch.cuda.synchronize()
    assert masked_bits_all_zero(y, lens_d, w.dtype) and masked_bits_all_zero(dx, lens_d, w.dtype)
    tol = {"f32": 1e-5, "bf16": 2.0 ** -7, "f16": 2.0 ** -9}[w.dtype]
    assert live_row_sums_close_to_one(y, lens_d, tol)
    st, sb = Stats(), Stats()
    for r in rows:
        check_forward(to_bits(x[0, 0, r:r + 1], w.dtype).reshape(-1), to_bits(y[0, 0, r:r + 1], w.dtype).reshape(-1),
                      lens, 1, 1, S, w.scale, w.dtype, r, r + 1, st)
        check_backward(to_bits(y_in[0, 0, r:r + 1], w.dtype).reshape(-1), to_bits(dy[0, 0, r:r + 1], w.dtype).reshape(-1),
                       to_bits(dx[0, 0, r:r + 1], w.dtype).reshape(-1), lens, 1, 1, S, w.scale, w.dtype, r, r + 1, sb)
    assert st.ok, f"forward {w.describe()}: {st}"
    assert sb.ok, f"backward {w.describe()}: {sb}"
    del x, y, dy, dx, y_in
    torch.cuda.empty_cache()


@pytest.mark.parametrize("S,dtype,scale", [(16384, "bf16", 0.125), (16384, "f32", -0.5), (2048, "bf16", 0.125),
                                           (65536, "bf16", 0.125)])
def test_infinite_inputs_before_the_extreme(dev, S, dtype, scale):
    """Kept inputs at columns 1 .. 4999 are -inf (+inf for a negative scale), so their exponentials are 0:
    the stream kernels' threads see whole batches of them before the first finite value (column 0 and
    columns >= 5000), and their running sums must start cleanly, as the row-in-registers kernels do."""
    inf = float("-inf") if scale > 0 else float("inf")
    if S <= 16384:
        w = si.custom(f"inf{S}", 2, 1, S, dtype, scale, seq_lens=(S, S // 2 + 1), x_std=2.0, seed=S + 41)
        x = si.make_x(w, "cpu")
        x[:, :, :, 1:5000] = inf
        run_and_check(w, dev, x_cpu=x)
        return
    L = 40000   # one row of 64K elements: sampled rows against the oracle
    w = si.custom(f"inf{S}", 1, 1, S, dtype, scale, seq_lens=(L,), x_std=2.0, seed=S + 41)
    lens = si.seq_lens(w)
    x = si.make_x(w, dev)
    x[:, :, :, 1:5000] = inf
    y = gtms.forward(x, torch.from_numpy(lens).to(dev), w.scale)
    torch.cuda.synchronize()
    st = Stats()
    for r in (0, 1, 4999, 5000, 5001, 20000, L - 1, S - 1):
        check_forward(to_bits(x[0, 0, r:r + 1], w.dtype).reshape(-1), to_bits(y[0, 0, r:r + 1], w.dtype).reshape(-1),
                      lens, w.B, 1, S, w.scale, w.dtype, r, r + 1, st)
    assert st.ok, f"forward {w.describe()}: {st}"


SCALE_CASES = [(1000, "f32", -0.7), (2048, "bf16", -0.125), (37, "f16", -2.0), (4096, "f16", -0.25),
               (8192, "f32", -1.0), (16384, "bf16", -0.125), (1000, "f32", 0.0), (16384, "bf16", 0.0)]


@pytest.mark.parametrize("S,dtype,scale", SCALE_CASES)
def test_negative_and_zero_scale(dev, S, dtype, scale):
    """scale < 0 makes the row minimum the reference point of the exponentials; scale = 0 gives
    1/n on every kept element. Warp, CTA, element and stream kernels, forward and backward."""
    w = si.custom(f"scale{S}", 2, 1, S, dtype, scale, seq_lens=(S, S // 3 + 1), x_std=2.0, seed=S + 31)
    run_and_check(w, dev)


def test_long_rows_that_are_not_16_byte_multiples_are_rejected(dev):
    lens = torch.ones(1, dtype=torch.int32, device=dev)
    x = torch.zeros(1, 1, 8196, 8196, dtype=torch.float16, device=dev)
    with pytest.raises(gtms.GtmsError, match="UNSUPPORTED"):
        gtms.forward(x, lens)
    with pytest.raises(gtms.GtmsError, match="UNSUPPORTED"):
        gtms.backward(x, x, lens)


def test_host_resident_buffers_match_device_calls(dev):
    """Pinned host tensors passed straight to the kernels (no staging copy) give
    the same bits as device-resident tensors."""
    w = si.custom("hostres", 3, 4, 1000, "f32", 1.0, seq_len_range=(1, 1000), seed=41)
    lens = si.seq_lens(w)
    lens_d = torch.from_numpy(lens).to(dev)
    x = si.make_x(w, dev)
    dy = si.make_dy(w, dev)
    y_ref = gtms.forward(x, lens_d, 1.0)
    dx_ref = gtms.backward(y_ref, dy, lens_d, 1.0)
    x_h, dy_h = x.cpu().pin_memory(), dy.cpu().pin_memory()
    lens_h = torch.from_numpy(lens).pin_memory()
    y_h = gtms.forward_host(x_h, lens_h, 1.0, device=dev)
    dx_h = gtms.backward_host(y_h, dy_h, lens_h, 1.0, device=dev)
    torch.cuda.synchronize()
    assert torch.equal(y_h, y_ref.cpu()) and torch.equal(dx_h, dx_ref.cpu())


# ---------------------------------------------------------------------------
# Mask families ("优化ScaledMaskSoftmax算子" section 6): length mask, sliding window
# ---------------------------------------------------------------------------

MASK_CASES = [
    (1, 0, 1000, "f32"), (1, 0, 2048, "bf16"), (1, 0, 37, "f16"), (1, 0, 8192, "f16"), (1, 0, 16384, "bf16"),
    (2, 1, 1000, "f32"), (2, 7, 1000, "f32"), (2, 100, 2048, "bf16"), (2, 257, 33, "f16"), (2, 300, 8192, "f16"),
    (2, 5000, 16384, "f32"), (2, 8, 64, "bf16"), (2, 9, 5, "f32"),
    (2, 900, 4096, "bf16"), (2, 1500, 8192, "f16"), (2, 256, 2048, "bf16"),
    (2, 1017, 2048, "bf16"),   # the widest window a 4-unit band lane set holds: 128 units at every offset
]


@pytest.mark.parametrize("kind,window,S,dtype", MASK_CASES)
def test_mask_families(dev, kind, window, S, dtype):
    """Length mask and sliding causal window: every element, head and tail partial units, per-row and
    stream kernels, 16-byte and element paths."""
    M = 2 if S <= 2048 else 1
    w = si.custom(f"mask{kind}_{S}", 4, M, S, dtype, 0.125 if dtype != "f32" else 1.0,
                  seq_lens=(S, S // 2 + 3, 1, 0), x_std=2.0, seed=S + 31 * kind + window)
    run_and_check(w, dev, mask_kind=kind, window=window)


@pytest.mark.parametrize("S,dtype,window,scale", [(2048, "bf16", 256, -0.125), (1000, "f32", 7, 0.0),
                                                  (4096, "f16", 129, -0.5)])
def test_band_kernels_negative_and_zero_scale(dev, S, dtype, window, scale):
    """Narrow sliding windows (warp-per-row band kernels) with the row minimum as the reference point
    (scale < 0) and with scale = 0 (1/n on every kept element)."""
    w = si.custom(f"band{S}", 3, 2, S, dtype, scale, seq_lens=(S, S // 2 + 5, 1), x_std=2.0, seed=S + window)
    run_and_check(w, dev, mask_kind=2, window=window)


def test_mask_family_sentinels_and_aliasing(dev):
    """Masked inputs of the window family are never read; in-place works."""
    S, win = 1000, 33
    w = si.custom("winsent", 2, 2, S, "f32", 1.0, seq_lens=(S, 500), seed=33)
    lens = si.seq_lens(w)
    lens_d = torch.from_numpy(lens).to(dev)
    c0, c1 = oracle.kept_ranges(lens, S, 2, win)
    col = torch.arange(S, device=dev)
    kept = ((col[None, None, :] >= torch.from_numpy(c0).to(dev)[:, :, None])
            & (col[None, None, :] < torch.from_numpy(c1).to(dev)[:, :, None]))[:, None]
    x = si.make_x(w, dev)
    ref = gtms.forward(x, lens_d, 1.0, mask_kind=2, window=win)
    y = gtms.forward(torch.where(kept, x, float("nan")), lens_d, 1.0, mask_kind=2, window=win)
    xi = x.clone()
    gtms.forward(xi, lens_d, 1.0, out=xi, mask_kind=2, window=win)
    torch.cuda.synchronize()
    assert torch.equal(y, ref) and torch.equal(xi, ref)
    assert masked_bits_all_zero(ref, lens_d, "f32", mask_kind=2, window=win)


def test_wide_window_equals_default_op(dev):
    w = si.custom("widewin", 2, 2, 1000, "f32", 1.0, seq_lens=(1000, 700), seed=34)
    lens_d = _lens_dev(w, dev)
    x = si.make_x(w, dev)
    dy = si.make_dy(w, dev)
    y0 = gtms.forward(x, lens_d)
    y2 = gtms.forward(x, lens_d, mask_kind=2, window=1000)
    d0 = gtms.backward(y0, dy, lens_d)
    d2 = gtms.backward(y0, dy, lens_d, mask_kind=2, window=5000)
    torch.cuda.synchronize()
    assert torch.equal(y0, y2) and torch.equal(d0, d2)


# ---------------------------------------------------------------------------
# Explicit keep mask ("优化ScaledMaskSoftmax算子" sections 2.2 / 3.1 / 4.1)
# ---------------------------------------------------------------------------

def _random_keep_mask(mb, S, seed, density=0.3):
    g = torch.Generator().manual_seed(seed)
    m = (torch.rand(mb, S, S, generator=g) < density).to(torch.uint8)
    m[:, 1, :] = 0                 # an all-masked row
    m[:, 2, :] = 1                 # a fully kept row
    m[:, 3, :] = 0
    m[:, 3, S - 1] = 1             # one kept entry, in the row's last unit
    return m


@pytest.mark.parametrize("S,dtype,mb", [(64, "f32", 1), (1000, "f32", 2), (2048, "bf16", 1), (2048, "f16", 2),
                                        (8192, "f16", 1), (8192, "f32", 2), (24, "bf16", 2)])
def test_explicit_mask_matches_oracle(dev, S, dtype, mb):
    B, M = 2, 2 if S <= 2048 else 1
    w = si.custom("explicit", B, M, S, dtype, 0.125 if dtype != "f32" else 1.0, seq_lens=(S,) * B, x_std=2.0,
                  seed=S + mb)
    mask = _random_keep_mask(mb, S, seed=S * 3 + mb)
    mask_d = mask.to(dev)
    x = si.make_x(w, "cpu")
    dy = si.make_dy(w, "cpu")
    y = gtms.forward_explicit(x.to(dev), mask_d, w.scale)
    torch.cuda.synchronize()
    xb, yb = to_bits(x, dtype).reshape(-1), to_bits(y, dtype).reshape(-1)
    keep = mask.numpy().astype(bool)
    code = w.dtype_code
    ref = oracle.forward_explicit(xb, mask.numpy(), B, M, S, w.scale, code, threads=8)
    st = Stats()
    q = np.arange(B * M * S)
    kept_rows = keep[(q // (M * S)) if mb == B else np.zeros_like(q), q % S]          # [rows, S]
    _compare_explicit(yb.reshape(-1, S), ref, kept_rows, dtype, st)
    assert st.ok, f"explicit forward {w.describe()}: {st}"
    y_or = oracle.round_to(ref, code)
    dx = gtms.backward_explicit(from_bits(y_or, dtype, "cpu").view(x.shape).to(dev), dy.to(dev), mask_d, w.scale)
    torch.cuda.synchronize()
    refb = oracle.backward_explicit(y_or, to_bits(dy, dtype).reshape(-1), mask.numpy(), B, M, S, w.scale, code,
                                    threads=8)
    sb = Stats()
    _compare_explicit(to_bits(dx, dtype).reshape(-1, S), refb, kept_rows, dtype, sb)
    assert sb.ok, f"explicit backward {w.describe()}: {sb}"


def _compare_explicit(gpu_bits, ref, kept_rows, dtype, stats):
    """compare_rows with an arbitrary kept set: masked bits must be zero, kept values within tolerance."""
    from parity_utils import compare_rows

    S = gpu_bits.shape[1]
    # kept entries are compared through compare_rows one row at a time via their (c0, c1) = (0, S) and a
    # zeroed reference where masked; masked bits are checked separately
    stats.bad_masked += int(np.count_nonzero(gpu_bits[~kept_rows]))
    g = np.where(kept_rows, gpu_bits, 0).astype(gpu_bits.dtype)
    full = (np.zeros(len(g), np.int64), np.full(len(g), S, np.int64))
    compare_rows(g, np.where(kept_rows, ref, 0.0), full, dtype, stats)


def test_explicit_mask_inputs_not_read_and_tril_equivalence(dev):
    S, B, M = 1000, 2, 2
    w = si.custom("explicit_tril", B, M, S, "f32", 1.0, seq_lens=(S, 600), seed=77)
    lens = si.seq_lens(w)
    r, c = torch.arange(S)[:, None], torch.arange(S)[None, :]
    tril = torch.stack([((c <= r) & (r < int(L))) for L in lens]).to(torch.uint8).to(dev)
    x = si.make_x(w, dev)
    dy = si.make_dy(w, dev)
    lens_d = torch.from_numpy(lens).to(dev)
    y_ref = gtms.forward(x, lens_d)
    y = gtms.forward_explicit(x, tril)
    x_nan = torch.where(tril[:, None].bool(), x, float("nan"))
    y_nan = gtms.forward_explicit(x_nan, tril)
    d_ref = gtms.backward(y_ref, dy, lens_d)
    d = gtms.backward_explicit(y_ref, torch.where(tril[:, None].bool(), dy, float("nan")), tril)
    torch.cuda.synchronize()
    # same kept set and same arithmetic as the grouped-tril kernel, up to reduction order
    assert torch.equal(y_nan, y)
    assert float((y - y_ref).abs().max()) <= 2e-6 and float((d - d_ref).abs().max()) <= 2e-6
    assert masked_bits_all_zero(y, lens_d, "f32") and masked_bits_all_zero(d, lens_d, "f32")


# ---------------------------------------------------------------------------
# Attention-backward step fused with its tensor-core GEMM ("ops(8)" section 2.1)
# ---------------------------------------------------------------------------

def _attn_case(dev, B, M, S, d, dtype, lens, seed, scale=0.125):
    """P = the oracle's forward of seeded scores (rounded to the IO dtype), dO, V ~ N(0,1)."""
    w = si.custom("attn", B, M, S, dtype, scale, seq_lens=lens, x_std=2.0, seed=seed)
    x_bits = to_bits(si.make_x(w, "cpu"), dtype)
    p_bits = oracle_forward_bits(x_bits, si.seq_lens(w), B, M, S, scale, dtype)
    g = torch.Generator().manual_seed(seed + 1)
    tdt = si.TORCH_DTYPES[dtype]
    dout = torch.randn(B, M, S, d, generator=g).to(tdt)
    v = torch.randn(B, M, S, d, generator=g).to(tdt)
    return w, p_bits, dout, v


def _attn_check(w, d, p_bits, dout, v, ds_dev, tag):
    """Element-wise: masked entries +0.0 bits; kept entries within
        ulp(ref) + scale * P_rc * 2^-23 * (d * A_rc + (d + 3) * max_c' A_rc' + (N_r - 1 + d / 8) * F_r),
    with A = |dO| |V|^T, N_r = 128 * (r // 128) the columns left of the diagonal tile of row r's
    128-row block, and F_r = sum over those columns of P_rc' A_rc'. Every addition inside the tensor
    cores is taken to round with a relative error of at most 2^-23 (one ulp: round to nearest and
    truncation both qualify), whatever the order:
    * dP_rc sums d exact products: off by at most d * 2^-23 * A_rc, and that reaches dS_rc directly;
    * the row sum over the diagonal tile (float-float over unit sums of 8 products, an FMA chain):
      the same dP error weighted by P (which sums to at most 1.004 after 16-bit rounding) plus
      5 * 2^-24 per unit sum, at most (d + 3) * 2^-23 * max A -- the whole row sum of the per-tile
      form is bounded by this term too;
    * the kernel that takes the columns left of the diagonal tile as dO_r . (P V)_r: (P V)_rk sums
      N_r exact products, off by at most (N_r - 1) * 2^-23 * sum_c' P_rc' |V_c'k|, which the dot
      with dO_r weights into (N_r - 1) * 2^-23 * F_r; the fp32 dot itself (d / 4 terms per thread,
      FMA chain, merged as float-float) adds at most (d / 8) * 2^-23 * F_r.
    The fp32 steps after the row sum are far inside the second half-ulp. The bound covers both kernels
    (the per-tile row sum of the cp.async kernel is the case F_r weighted by zero)."""
    B, M, S, dt = w.B, w.M, w.S, w.dtype
    lens = si.seq_lens(w)
    code = w.dtype_code
    db, vb = to_bits(dout, dt), to_bits(v, dt)
    ref = oracle.attn_dscores(p_bits, db, vb, lens, B, M, S, d, w.scale, code, threads=8).reshape(B, M, S, S)
    got = to_bits(ds_dev, dt).reshape(B, M, S, S)
    pv = oracle.decode(p_bits, code).reshape(B, M, S, S)
    A = np.abs(oracle.decode(db, code)) @ np.swapaxes(np.abs(oracle.decode(vb, code)), -1, -2)   # [B,M,S,S]
    c0, c1 = oracle.kept_ranges(lens, S)
    col = np.arange(S)[None, None, None, :]
    kept = (col >= c0[:, None, :, None]) & (col < c1[:, None, :, None])
    kept = np.broadcast_to(kept, ref.shape)
    assert np.count_nonzero(got[~kept]) == 0, f"{tag}: masked output not +0.0"
    Amax = np.where(kept, A, 0.0).max(axis=-1, keepdims=True)
    n_left = (128 * (np.arange(S) // 128))[None, None, :, None]          # N_r, per row
    F = np.where(kept & (col < n_left), pv * A, 0.0).sum(axis=-1, keepdims=True)
    # one ulp of the IO dtype at |ref|: the gap to the next representable magnitude
    rb = oracle.round_to(np.abs(ref), code).astype(np.int64)
    top = 0x7BFF if dt == "f16" else 0x7F7F
    nb = np.where(rb < top, rb + 1, rb - 1)
    ulp = np.abs(oracle.decode(nb.astype(np.uint16), code) - oracle.decode(rb.astype(np.uint16), code))
    tol = ulp + abs(w.scale) * pv * 2.0 ** -23 * (d * A + (d + 3) * Amax + (np.maximum(n_left - 1, 0) + d / 8) * F)
    err = np.abs(oracle.decode(got, code) - ref)
    bad = kept & (err > tol)
    assert not bad.any(), f"{tag}: {int(bad.sum())} of {int(kept.sum())} kept entries out of tolerance, " \
                          f"worst excess {float((err - tol)[kept].max()):.3g}"


@pytest.mark.parametrize("S,d,dtype,lens", [(8, 64, "bf16", (8, 3)), (128, 64, "bf16", (128, 77)),
                                             (200, 128, "f16", (200, 0)), (1000, 64, "bf16", (1000, 513)),
                                             (1024, 128, "bf16", (700, 1024)), (2048, 64, "f16", (2048, 1300))])
def test_attention_softmax_backward_matches_oracle(dev, S, d, dtype, lens):
    B, M = 2, 2 if S <= 1024 else 1
    w, p_bits, dout, v = _attn_case(dev, B, M, S, d, dtype, lens, seed=S + d)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    p_d = from_bits(p_bits, dtype, "cpu").view(B, M, S, S).to(dev)
    ds = torch.full_like(p_d, float("nan"))
    gtms.attention_softmax_backward(p_d, dout.to(dev), v.to(dev), torch.from_numpy(si.seq_lens(w)).to(dev),
                                    w.scale, out=ds, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _attn_check(w, d, p_bits, dout, v, ds, f"S={S} d={d} {dtype}")


def test_attention_softmax_backward_in_place_and_masked_p_not_read(dev):
    B, M, S, d, dtype = 2, 2, 384, 64, "bf16"
    w, p_bits, dout, v = _attn_case(dev, B, M, S, d, dtype, (384, 200), seed=90)
    lens_d = torch.from_numpy(si.seq_lens(w)).to(dev)
    p_d = from_bits(p_bits, dtype, "cpu").view(B, M, S, S).to(dev)
    ref = gtms.attention_softmax_backward(p_d, dout.to(dev), v.to(dev), lens_d, w.scale)
    # NaN in every masked P entry must not reach dS; dS may overwrite P
    kept = torch.from_numpy(oracle.kept_prefix_lengths(si.seq_lens(w), M, S)).to(dev)
    col = torch.arange(S, device=dev)
    keep = (col[None, None, :] < kept[:, :, None])[:, None]
    p_nan = torch.where(keep, p_d, torch.tensor(float("nan"), dtype=p_d.dtype, device=dev))
    got = gtms.attention_softmax_backward(p_nan, dout.to(dev), v.to(dev), lens_d, w.scale, out=p_nan)
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


def test_attention_softmax_backward_many_items_per_cta(dev):
    """512 (slice, row block) items: each persistent CTA takes several, so the stage ring, both
    tensor-memory accumulators and both dO buffers wrap around many times."""
    B, M, S, d, dtype = 4, 16, 1024, 64, "bf16"
    w, p_bits, dout, v = _attn_case(dev, B, M, S, d, dtype, (1024, 700, 513, 1), seed=91)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    p_d = from_bits(p_bits, dtype, "cpu").view(B, M, S, S).to(dev)
    ds = torch.full_like(p_d, float("nan"))
    gtms.attention_softmax_backward(p_d, dout.to(dev), v.to(dev), torch.from_numpy(si.seq_lens(w)).to(dev),
                                    w.scale, out=ds, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _attn_check(w, d, p_bits, dout, v, ds, "B=4 M=16 S=1024")


@pytest.mark.parametrize("S,d,dtype,lens", [(1000, 64, "bf16", (1000, 513)), (384, 128, "f16", (300, 384))])
def test_attention_softmax_backward_host_resident(dev, S, d, dtype, lens):
    """Operands in mapped pinned host memory (the kernel that copies with cp.async)."""
    B, M = 2, 2
    w, p_bits, dout, v = _attn_case(dev, B, M, S, d, dtype, lens, seed=S + 7)
    p_h = from_bits(p_bits, dtype, "cpu").view(B, M, S, S).pin_memory()
    ds_h = torch.full_like(p_h, float("nan")).pin_memory()
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    gtms.attention_softmax_backward_host(p_h, dout.pin_memory(), v.pin_memory(),
                                         torch.from_numpy(si.seq_lens(w)).pin_memory(), w.scale, out=ds_h,
                                         status=status, device=dev)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _attn_check(w, d, p_bits, dout, v, ds_h, f"host S={S} d={d} {dtype}")


@pytest.mark.parametrize("name", ["attn_s2048_bf16", "attn_d128_s2048_f16"])
def test_attention_softmax_backward_full_size_sampled(dev, name):
    """The benchmark's workloads (P[32,16,2048,2048] bf16 with head dim 64, fp16 with head dim 128) in the
    benchmark's launch: masked bits zero everywhere; sampled slices, whose P is the oracle's own forward,
    element-wise against the oracle."""
    w = si.WORKLOADS[name]
    B, M, S, d = w.B, w.M, w.S, w.head_dim
    lens = si.seq_lens(w)
    lens_d = torch.from_numpy(lens).to(dev)
    x = si.make_x(w, dev)
    p = gtms.forward(x, lens_d, w.scale)
    dout, v = si.make_head_operands(w, dev)
    slices = si.sample_slices(w, 4)
    p_ref = {}
    for b, m in slices:
        xs = to_bits(x[b, m], w.dtype).reshape(1, 1, S, S)
        p_ref[(b, m)] = oracle_forward_bits(xs, lens[b:b + 1], 1, 1, S, w.scale, w.dtype)
        p[b, m].copy_(from_bits(p_ref[(b, m)], w.dtype, "cpu").view(S, S))
    del x
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ds = gtms.attention_softmax_backward(p, dout, v, lens_d, w.scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert masked_bits_all_zero(ds, lens_d, w.dtype)
    assert bool(torch.isfinite(ds).all())
    for b, m in slices:
        ws = si.custom("attn_slice", 1, 1, S, w.dtype, w.scale, seq_lens=(int(lens[b]),))
        _attn_check(ws, d, p_ref[(b, m)], dout[b, m].reshape(1, 1, S, d).cpu(), v[b, m].reshape(1, 1, S, d).cpu(),
                    ds[b, m].reshape(1, 1, S, S), f"full size slice ({b},{m})")
    del p, ds, dout, v
    torch.cuda.empty_cache()


def _build_give_up_probe():
    """Compile tests/attn_give_up_probe.cu (the TMA attention kernel with its copies left out) into a
    library of its own under _build/; libgtms.so is not touched."""
    import ctypes
    import os
    import subprocess

    from masked_softmax_attention_gb300 import _build as b

    src = os.path.join(b.ROOT, "tests", "attn_give_up_probe.cu")
    out_dir = os.path.join(b.ROOT, "_build", "test_probe")
    os.makedirs(out_dir, exist_ok=True)
    lib_path = os.path.join(out_dir, "libgtms_attn_give_up_probe.so")
    deps = [src] + [os.path.join(b.CSRC, f) for f in os.listdir(b.CSRC)] + [os.path.join(b.INCLUDE, "gtms.h")]
    if not os.path.exists(lib_path) or any(os.path.getmtime(d) > os.path.getmtime(lib_path) for d in deps):
        tmp = lib_path + f".{os.getpid()}.tmp"
        subprocess.run([b.nvcc_path(), *b.ARCH, *b.NVCC_FLAGS, "-shared", src, "-o", tmp], check=True,
                       capture_output=True, text=True)
        os.replace(tmp, lib_path)
    lib = ctypes.CDLL(lib_path)
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    lib.gtms_test_attn_no_loads.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, ctypes.c_float, vp, vp,
                                            ctypes.c_uint64]
    lib.gtms_test_attn_no_loads.restype = ctypes.c_int
    return lib


def test_attention_kernel_gives_up_when_its_waits_run_out(dev):
    """Failure detection of the TMA attention kernel, without a GPU fault: in a test build whose producer
    issues no copies, every consumer wait runs out (after 200 us here). The launch must succeed, the
    kernel must end promptly with GTMS_ERR_TIMEOUT in the status word, and the context must stay usable:
    a normal call right after it matches the oracle."""
    import time

    probe = _build_give_up_probe()
    B, M, S, d, dtype = 2, 4, 1024, 64, "bf16"
    w, p_bits, dout, v = _attn_case(dev, B, M, S, d, dtype, (1024, 700), seed=97)
    lens_d = torch.from_numpy(si.seq_lens(w)).to(dev)
    p_d = from_bits(p_bits, dtype, "cpu").view(B, M, S, S).to(dev)
    dout_d, v_d = dout.to(dev), v.to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ds = torch.zeros_like(p_d)
    torch.cuda.synchronize()
    t0 = time.monotonic()
    rc = probe.gtms_test_attn_no_loads(p_d.data_ptr(), dout_d.data_ptr(), v_d.data_ptr(), ds.data_ptr(),
                                       lens_d.data_ptr(), B, M, S, w.scale, status.data_ptr(),
                                       torch.cuda.current_stream().cuda_stream, 200_000)
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    assert rc == 0
    assert int(status.item()) == gtms.GTMS_ERR_TIMEOUT
    assert elapsed < 20.0
    status.zero_()
    out = torch.full_like(p_d, float("nan"))
    gtms.attention_softmax_backward(p_d, dout_d, v_d, lens_d, w.scale, out=out, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _attn_check(w, d, p_bits, dout, v, out, "after a give-up")


@pytest.mark.parametrize("lens", [(0, 0), (-5, 3000)])
def test_attention_softmax_backward_padded_and_clamped_lengths(dev, lens):
    """All-padded batches give an all-zero dS; seq_lens outside [0, S] are clamped."""
    B, M, S, d, dtype = 2, 2, 256, 64, "bf16"
    clamped = tuple(min(max(v, 0), S) for v in lens)
    w, p_bits, dout, v = _attn_case(dev, B, M, S, d, dtype, clamped, seed=95)
    p_d = from_bits(p_bits, dtype, "cpu").view(B, M, S, S).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    raw_lens = torch.tensor(lens, dtype=torch.int32, device=dev)
    ds = torch.full_like(p_d, float("nan"))
    gtms.attention_softmax_backward(p_d, dout.to(dev), v.to(dev), raw_lens, w.scale, out=ds, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _attn_check(w, d, p_bits, dout, v, ds, f"lens {lens}")


def test_attention_softmax_backward_long_rows(dev):
    """S = 8192: 64 row blocks, up to 64 tiles per block and 128 tile iterations per work item."""
    B, M, S, d, dtype = 1, 1, 8192, 64, "bf16"
    w, p_bits, dout, v = _attn_case(dev, B, M, S, d, dtype, (6001,), seed=96)
    p_d = from_bits(p_bits, dtype, "cpu").view(B, M, S, S).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ds = torch.full_like(p_d, float("nan"))
    gtms.attention_softmax_backward(p_d, dout.to(dev), v.to(dev), torch.from_numpy(si.seq_lens(w)).to(dev),
                                    w.scale, out=ds, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _attn_check(w, d, p_bits, dout, v, ds, "S=8192")
