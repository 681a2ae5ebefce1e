"""Host-side tests of the C ABI (no GPU needed).

Every call here fails argument validation, or is an empty no-op, before the
library touches CUDA; the fake pointer values are never dereferenced. The
tests check that libgtms.so loads, exports exactly what include/gtms.h
declares, and maps each kind of bad argument to its documented status.
"""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

import masked_softmax_attention_gb300 as gtms

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gtms.h")

OK, INVALID, UNSUPPORTED = gtms.GTMS_OK, gtms.GTMS_ERR_INVALID_ARG, gtms.GTMS_ERR_UNSUPPORTED
F32, BF16, F16 = gtms.GTMS_F32, gtms.GTMS_BF16, gtms.GTMS_F16

# Distinct, 256-byte aligned fake device addresses, far apart. Never dereferenced.
X, Y, DY, LENS = 0x10_0000_0000, 0x20_0000_0000, 0x30_0000_0000, 0x40_0000_0000


def _cuda_visible():
    import torch

    return torch.cuda.is_available() or os.path.exists("/dev/nvidia0")


# These tests hand the library fake device addresses. Each call is meant to be
# rejected on the host, but on a machine with a GPU a slip in a test would
# launch a kernel on them, so the module runs only where no GPU is visible.
pytestmark = pytest.mark.skipif(_cuda_visible(), reason="fake-pointer host tests run only without a GPU")


@pytest.fixture(scope="module")
def lib():
    gtms.build_library()
    return gtms.load_library()


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    return sorted(set(re.findall(r"^\s*(?:int|const char\*)\s+(gtms_\w+)\s*\(", text, re.M)))


def test_header_declares_the_public_api():
    assert declared_functions() == sorted(gtms.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_library_exports_nothing_else(lib):
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", "--defined-only", gtms.LIB_PATH], capture_output=True, text=True).stdout
    exported = sorted({ln.split()[-1] for ln in out.splitlines() if " T " in ln and ln.split()[-1].startswith("gtms")})
    assert exported == declared_functions()


def test_version_and_status_strings(lib):
    assert gtms.gtms_version() == 1
    assert gtms.status_string(OK) == "GTMS_OK"
    assert gtms.status_string(INVALID) == "GTMS_ERR_INVALID_ARG"
    assert gtms.status_string(UNSUPPORTED) == "GTMS_ERR_UNSUPPORTED"
    assert gtms.status_string(gtms.GTMS_ERR_CUDA) == "GTMS_ERR_CUDA"
    assert gtms.status_string(gtms.GTMS_ERR_TIMEOUT) == "GTMS_ERR_TIMEOUT"
    assert gtms.status_string(99) == "GTMS_UNKNOWN_STATUS"


def test_kernel_choice(lib):
    # vector kernels: a warp or a small CTA per row, sized by the row's 16-byte units
    assert gtms.kernel_name(0, 1000, F32) == "gtms_fwd_vec_kernel<f32,team64,x4,minb0>"
    assert gtms.kernel_name(1, 1000, F32) == "gtms_bwd_vec_kernel<f32,team32,x8,minb5>"
    assert gtms.kernel_name(0, 2048, BF16) == "gtms_fwd_heads_kernel<bf16,team64,x4,minb12>"
    assert gtms.kernel_name(1, 2048, BF16) == "gtms_bwd_vec_kernel<bf16,team32,x8,minb5>"
    assert gtms.kernel_name(1, 8192, F16) == "gtms_bwd_vec_kernel<f16,team128,x8,minb0>"
    assert gtms.kernel_name(0, 4096, F32) == "gtms_fwd_vec_kernel<f32,team256,x4,minb0>"
    assert gtms.kernel_name(0, 1024, F16) == "gtms_fwd_vec_kernel<f16,team32,x4,minb6>"
    assert gtms.kernel_name(0, 8200, F16) == "gtms_fwd_heads_kernel<f16,team512,x4,minb1>"
    assert gtms.kernel_name(0, 16376, BF16) == "gtms_fwd_heads_kernel<bf16,team512,x4,minb1>"   # 32752-byte rows
    # 16-bit forwards of CTA-team rows: a team per (batch, row) pair runs its heads in turn
    assert gtms.kernel_name(0, 8192, F16) == "gtms_fwd_heads_kernel<f16,team256,x4,minb3>"
    assert gtms.kernel_name(0, 4096, BF16) == "gtms_fwd_heads_kernel<bf16,team128,x4,minb6>"
    assert gtms.kernel_name(0, 1024, BF16) == "gtms_fwd_vec_kernel<bf16,team32,x4,minb6>"
    assert gtms.kernel_name(1, 4096, BF16) == "gtms_bwd_vec_kernel<bf16,team64,x8,minb0>"
    # rows whose byte length is not a multiple of 16, or unaligned buffers: element kernels
    assert gtms.kernel_name(0, 5, F32) == "gtms_fwd_elem_kernel<f32,team32,x1>"
    assert gtms.kernel_name(0, 1000, F32, aligned16=False) == "gtms_fwd_elem_kernel<f32,team32,x32>"
    assert gtms.kernel_name(1, 8191, F16) == "gtms_bwd_elem_kernel<f16,team256,x32>"
    # rows of 32 KB and more: one CTA per row streams the kept units in two passes, 16-byte units only
    assert gtms.kernel_name(0, 8192, F32) == "gtms_fwd_stream_kernel<f32,team128,x4,minb8>"
    assert gtms.kernel_name(0, 16384, BF16) == "gtms_fwd_stream_kernel<bf16,team128,x4,minb8>"
    assert gtms.kernel_name(0, 16384, F32) == "gtms_fwd_stream_kernel<f32,team256,x4,minb4>"
    assert gtms.kernel_name(0, 32768, BF16) == "gtms_fwd_stream_kernel<bf16,team256,x4,minb4>"
    assert gtms.kernel_name(0, 65536, F32) == "gtms_fwd_stream_kernel<f32,team256,x4,minb4>"
    assert gtms.kernel_name(1, 8192, F32) == "gtms_bwd_stream_kernel<f32,team256,x2,minb4>"
    assert gtms.kernel_name(1, 32768, BF16) == "gtms_bwd_stream_kernel<bf16,team256,x2,minb4>"
    assert gtms.kernel_name(1, 65536, BF16) == "gtms_bwd_stream_kernel<bf16,team256,x2,minb4>"
    assert gtms.kernel_name(0, 16384, F32, aligned16=False) == "none"
    # mask families: the row-length variant with the mask kind, or a warp-per-row band kernel for a
    # narrow sliding window in a row longer than one warp's 128 units
    assert gtms.kernel_name_masked(0, 2048, BF16, 1) == "gtms_fwd_heads_kernel<bf16,team64,x4,minb12,mask1>"
    assert gtms.kernel_name_masked(0, 2048, BF16, 0) == gtms.kernel_name(0, 2048, BF16)
    assert gtms.kernel_name_masked(0, 2048, BF16, 2, 256) == "gtms_fwd_band_kernel<bf16,x2,minb8>"
    assert gtms.kernel_name_masked(1, 2048, BF16, 2, 256) == "gtms_bwd_band_kernel<bf16,x2,minb4>"
    assert gtms.kernel_name_masked(0, 2048, BF16, 2, 100) == "gtms_fwd_band_kernel<bf16,x1,minb8>"
    assert gtms.kernel_name_masked(0, 8192, F16, 2, 300) == "gtms_fwd_band_kernel<f16,x2,minb8>"
    assert gtms.kernel_name_masked(1, 1000, F32, 2, 1000) == "gtms_bwd_vec_kernel<f32,team32,x8,minb5,mask2>"
    assert gtms.kernel_name_masked(0, 1000, F32, 2, 7) == "gtms_fwd_band_kernel<f32,x1,minb8>"
    assert gtms.kernel_name_masked(0, 512, F32, 2, 7) == "gtms_fwd_vec_kernel<f32,team32,x4,minb8,mask2>"
    assert gtms.kernel_name_masked(0, 1000, F32, 2, 7, aligned16=False) == "gtms_fwd_elem_kernel<f32,team32,x32,mask2>"
    assert gtms.kernel_name_masked(0, 16384, F32, 2, 5000) == "gtms_fwd_stream_kernel<f32,team256,x4,minb4,mask2>"
    # the band holds every run of w columns: (w + 2 * EPU - 2) // EPU units at most
    assert gtms.kernel_name_masked(0, 2048, BF16, 2, 241) == "gtms_fwd_band_kernel<bf16,x1,minb8>"
    assert gtms.kernel_name_masked(0, 2048, BF16, 2, 250) == "gtms_fwd_band_kernel<bf16,x2,minb8>"
    assert gtms.kernel_name_masked(0, 2048, BF16, 2, 1017) == "gtms_fwd_band_kernel<bf16,x4,minb6>"
    assert gtms.kernel_name_masked(0, 2048, BF16, 2, 1018) == "gtms_fwd_heads_kernel<bf16,team64,x4,minb12,mask2>"
    assert gtms.kernel_name_masked(1, 2048, BF16, 2, 1018) == "gtms_bwd_vec_kernel<bf16,team32,x8,minb5,mask2>"
    assert gtms.kernel_name_masked(0, 2048, BF16, 2, 0) == "none"
    assert gtms.kernel_name_masked(0, 2048, BF16, 3, 1) == "none"
    # explicit-mask kernels: the vector rows, the forward with its own register caps, up to S = 8192
    assert gtms.kernel_name_explicit(0, 2048, BF16) == "gtms_fwd_explicit_kernel<bf16,team64,x4,minb12>"
    assert gtms.kernel_name_explicit(1, 2048, BF16) == "gtms_bwd_explicit_kernel<bf16,team32,x8,minb5>"
    assert gtms.kernel_name_explicit(0, 1000, F32) == "gtms_fwd_explicit_kernel<f32,team64,x4,minb0>"
    assert gtms.kernel_name_explicit(0, 8192, F32) == "gtms_fwd_explicit_kernel<f32,team512,x4,minb1>"
    assert gtms.kernel_name_explicit(0, 16384, BF16) == "none"
    assert gtms.kernel_name_explicit(0, 1001, F32) == "none"
    # out of range
    assert gtms.kernel_name(0, 8193, F32) == "none"
    assert gtms.kernel_name(0, 65537, BF16) == "none"
    assert gtms.kernel_name(0, 0, F32) == "none"
    assert gtms.kernel_name(3, 100, F32) == "none"
    # the staged forward (direction 2): a CTA team per row, rows of 16-byte units below 32 KB
    assert gtms.kernel_name(2, 1000, F32) == "gtms_fwd_staged_kernel<f32,team64,x4,slots6,minb12>"
    assert gtms.kernel_name(2, 2048, BF16) == "gtms_fwd_staged_kernel<bf16,team64,x4,slots2,minb10>"
    assert gtms.kernel_name(2, 4096, BF16) == "gtms_fwd_staged_kernel<bf16,team128,x4,slots2,minb5>"
    assert gtms.kernel_name(2, 8192, F16) == "gtms_fwd_staged_kernel<f16,team256,x4,slots2,minb3>"
    assert gtms.kernel_name(2, 4096, F32) == "gtms_fwd_staged_kernel<f32,team256,x4,slots2,minb3>"
    assert gtms.kernel_name(2, 8192, F32) == "none"      # 32 KB rows: stream rows
    assert gtms.kernel_name(2, 1001, F32) == "none"      # not a 16-byte multiple
    assert gtms.kernel_name(2, 1000, F32, aligned16=False) == "none"
    assert gtms.kernel_name(0, 100, 7) == "none"


def fwd(x=X, y=Y, lens=LENS, B=2, M=3, S=64, scale=1.0, dtype=F32):
    return gtms.gtms_forward(x, y, lens, B, M, S, scale, dtype, None)


def bwd(y=X, dy=DY, dx=Y, lens=LENS, B=2, M=3, S=64, scale=1.0, dtype=F32):
    return gtms.gtms_backward(y, dy, dx, lens, B, M, S, scale, dtype, None)


@pytest.mark.parametrize("call", [fwd, bwd])
def test_shape_and_scale_errors(lib, call):
    assert call(B=-1) == INVALID
    assert call(M=-2) == INVALID
    assert call(S=-5) == INVALID
    assert call(scale=float("nan")) == INVALID
    assert call(scale=float("inf")) == INVALID
    assert call(dtype=3) == UNSUPPORTED
    assert call(dtype=-1) == UNSUPPORTED
    assert call(S=gtms.GTMS_MAX_S + 1) == UNSUPPORTED
    # byte count overflows int64
    assert call(B=1 << 30, M=1 << 30, S=4096) == INVALID


def test_mask_arguments(lib):
    for fn, ptrs in ((gtms.gtms_forward_masked, (X, Y, LENS)), (gtms.gtms_backward_masked, (X, DY, Y, LENS))):
        assert fn(*ptrs, 2, 3, 64, 1.0, 3, 0, F32, None) == UNSUPPORTED      # unknown mask kind
        assert fn(*ptrs, 2, 3, 64, 1.0, -1, 0, F32, None) == UNSUPPORTED
        assert fn(*ptrs, 2, 3, 64, 1.0, 2, 0, F32, None) == INVALID          # window must be >= 1
        assert fn(*ptrs, 2, 3, 64, 1.0, 2, -4, F32, None) == INVALID
        assert fn(*ptrs, 0, 3, 64, 1.0, 2, 4, F32, None) == OK               # empty work
        assert fn(*ptrs, 2, 3, 64, float("nan"), 1, 0, F32, None) == INVALID


def test_attention_softmax_backward_arguments(lib):
    fn = gtms.gtms_attention_softmax_backward
    DO, V, DS, ST = 0x60_0000_0000, 0x70_0000_0000, 0x80_0000_0000, 0x90_0000_0000
    args = dict(B=2, M=3, S=256, d=64, scale=0.125, dtype=BF16)

    def call(p=X, dout=DO, v=V, ds=DS, lens=LENS, status=ST, **kw):
        a = {**args, **kw}
        return fn(p, dout, v, ds, lens, a["B"], a["M"], a["S"], a["d"], a["scale"], a["dtype"], status, None)

    assert call(dtype=F32) == UNSUPPORTED          # tensor-core path is 16-bit only
    assert call(d=96) == UNSUPPORTED                # head dims 64 and 128
    assert call(S=260) == UNSUPPORTED               # S multiple of 8
    assert call(S=gtms.GTMS_MAX_S + 8) == UNSUPPORTED
    assert call(d=-64) == INVALID
    assert call(p=None) == INVALID and call(v=None) == INVALID and call(lens=None) == INVALID
    assert call(dout=DO + 8) == INVALID             # 16-byte alignment
    assert call(status=ST + 2) == INVALID
    assert call(ds=X + 32) == INVALID               # partial overlap with p
    assert call(ds=DO + 64) == INVALID              # overlap with dO
    assert call(status=DS + 4) == INVALID           # status inside the output
    assert call(B=0, p=None, dout=None, v=None, ds=None, lens=None) == OK
    assert call(scale=float("inf")) == INVALID


def test_explicit_mask_arguments(lib):
    MASK = 0x50_0000_0000
    f, b = gtms.gtms_forward_explicit, gtms.gtms_backward_explicit
    for fn, ptrs in ((f, (X, Y)), (b, (X, DY, Y))):
        assert fn(*ptrs, None, 1, 2, 3, 64, 1.0, F32, None) == INVALID          # null mask
        assert fn(*ptrs, MASK + 4, 1, 2, 3, 64, 1.0, F32, None) == INVALID      # mask not 8-byte aligned
        assert fn(*ptrs, MASK, 3, 2, 3, 64, 1.0, F32, None) == INVALID          # mask_batches not 1 or B
        assert fn(*ptrs, Y + 64, 2, 2, 3, 64, 1.0, F32, None) == INVALID        # mask inside the output
        assert fn(*ptrs, MASK, 1, 2, 3, 63, 1.0, F32, None) == UNSUPPORTED      # rows not 16-byte multiples
        assert fn(*ptrs, MASK, 1, 2, 3, 8200, 1.0, F32, None) == UNSUPPORTED    # longer than 8192
        assert fn(*ptrs, MASK, 1, 0, 3, 64, 1.0, F32, None) == OK               # empty work
        assert fn(*ptrs, MASK, 1, 2, 3, 64, 1.0, 5, None) == UNSUPPORTED        # unknown dtype


def test_staged_forward_arguments(lib):
    fn = gtms.gtms_forward_staged

    def call(x=X, y=Y, lens=LENS, B=2, M=3, S=64, scale=1.0, dtype=F32):
        return fn(x, y, lens, B, M, S, scale, dtype, None)

    assert call(B=-1) == INVALID and call(scale=float("nan")) == INVALID
    assert call(dtype=3) == UNSUPPORTED
    assert call(x=None) == INVALID and call(lens=None) == INVALID
    assert call(y=X + 16) == INVALID                   # partial overlap of y with x
    assert call(S=63) == UNSUPPORTED                   # rows not 16-byte multiples
    assert call(x=X + 4) == UNSUPPORTED                # buffers only element-aligned
    assert call(S=8192) == UNSUPPORTED                 # 32 KB rows (stream rows)
    assert call(S=16384, dtype=BF16) == UNSUPPORTED
    assert call(B=0, x=None, y=None, lens=None) == OK  # empty work


@pytest.mark.parametrize("call", [fwd, bwd])
def test_long_rows_need_16_byte_units(lib, call):
    assert call(S=8193) == UNSUPPORTED                  # fp32 row of 32772 bytes
    assert call(S=8196, dtype=F16) == UNSUPPORTED       # 16392 bytes
    assert call(S=65536 + 8) == UNSUPPORTED             # beyond GTMS_MAX_S


@pytest.mark.parametrize("call", [fwd, bwd])
def test_empty_work_is_an_ok_noop_even_with_null_pointers(lib, call):
    if call is fwd:
        assert fwd(x=None, y=None, lens=None, B=0) == OK
        assert fwd(x=None, y=None, lens=None, M=0) == OK
        assert fwd(x=None, y=None, lens=None, S=0) == OK
    else:
        assert bwd(y=None, dy=None, dx=None, lens=None, B=0) == OK
        assert bwd(y=None, dy=None, dx=None, lens=None, S=0) == OK


def test_forward_pointer_errors(lib):
    assert fwd(x=None) == INVALID
    assert fwd(y=None) == INVALID
    assert fwd(lens=None) == INVALID
    assert fwd(x=X + 2) == INVALID                    # fp32 element not 4-byte aligned
    assert fwd(y=Y + 1, dtype=BF16) == INVALID        # 16-bit element not 2-byte aligned
    assert fwd(lens=LENS + 2) == INVALID              # int32 seq_lens not 4-byte aligned
    nbytes = 2 * 3 * 64 * 64 * 4
    assert fwd(y=X + 16) == INVALID                   # partial overlap of y with x
    assert fwd(y=X - nbytes + 16) == INVALID
    assert fwd(lens=Y + nbytes - 4) == INVALID        # seq_lens inside the output


def test_backward_pointer_errors(lib):
    assert bwd(y=None) == INVALID
    assert bwd(dy=None) == INVALID
    assert bwd(dx=None) == INVALID
    assert bwd(lens=None) == INVALID
    assert bwd(dx=Y + 1, dtype=F16) == INVALID        # 16-bit element not 2-byte aligned
    nbytes = 2 * 3 * 64 * 64 * 4
    assert bwd(dx=DY + 64) == INVALID                 # partial overlap with dy
    assert bwd(dx=X + nbytes - 4) == INVALID          # partial overlap with y
    assert bwd(lens=Y + 128) == INVALID               # seq_lens inside dx
    assert bwd(dy=DY + 1) == INVALID


def test_device_pointer_of_host_rejects_bad_arguments(lib):
    out = ctypes.c_void_p()
    assert lib.gtms_device_pointer_of_host(None, ctypes.byref(out)) == INVALID
    buf = ctypes.create_string_buffer(64)
    assert lib.gtms_device_pointer_of_host(ctypes.addressof(buf), None) == INVALID


def test_tensor_api_rejects_cpu_tensors(lib):
    import torch

    x = torch.zeros(1, 1, 4, 4)
    lens = torch.ones(1, dtype=torch.int32)
    with pytest.raises(ValueError):
        gtms.forward(x, lens)
    with pytest.raises(ValueError):
        gtms.backward(x, x, lens)
    p = torch.zeros(1, 1, 4, 4, dtype=torch.bfloat16)
    dv = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        gtms.attention_softmax_backward(p, dv, dv, lens)
    # the host-resident forms want page-locked tensors: ordinary CPU tensors are refused
    with pytest.raises(ValueError):
        gtms.attention_softmax_backward_host(p, dv, dv, lens)
    with pytest.raises(ValueError):
        gtms.forward_host(x, lens)


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="no fallback"):
        gtms.load_library(str(tmp_path / "libgtms.so"))


def test_ctypes_signatures_match_header(lib):
    text = open(HEADER, encoding="utf-8").read()
    fwd_decl = re.search(r"int gtms_forward\(([^)]*)\)", text, re.S).group(1)
    bwd_decl = re.search(r"int gtms_backward\(([^)]*)\)", text, re.S).group(1)
    assert len(fwd_decl.split(",")) == len(lib.gtms_forward.argtypes) == 9
    assert len(bwd_decl.split(",")) == len(lib.gtms_backward.argtypes) == 10
    assert lib.gtms_forward.argtypes[6] is ctypes.c_float
