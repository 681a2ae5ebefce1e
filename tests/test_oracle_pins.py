"""Pins for the CPU oracle, independent of the oracle itself (no GPU).

Each test ties one part of ``oracle/`` to something fixed outside it: the
worked example printed in the "Attention-Mask-Optimization" README (operator
behaviour section), closed forms of the softmax, textbook routines from
torch / scipy run in float64, central finite differences, the softmax Jacobian
of "ops(8): self-attention 的 CUDA 实现及优化 (下)" section 2.1, and numpy / torch
conversions for the IEEE rounding helpers. A plausible slip in the oracle (a
dropped max, a wrong sign, a transposed mask, a missing scale, a bad rounding
tie) fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle

F32, BF16, F16, F64 = oracle.F32, oracle.BF16, oracle.F16, oracle.F64


def _fwd64(x, seq_lens, scale=1.0):
    """Oracle forward on a float64 array x[B,M,S,S]; returns float64 of the same shape."""
    B, M, S, _ = x.shape
    y = oracle.forward(np.ascontiguousarray(x, dtype=np.float64), seq_lens, B, M, S, scale, F64)
    return y.reshape(B, M, S, S)


def _bwd64(y, dy, seq_lens, scale=1.0):
    B, M, S, _ = y.shape
    dx = oracle.backward(np.ascontiguousarray(y, np.float64), np.ascontiguousarray(dy, np.float64),
                         seq_lens, B, M, S, scale, F64)
    return dx.reshape(B, M, S, S)


# ---------------------------------------------------------------------------
# The README's worked example
# ---------------------------------------------------------------------------

def test_golden_fixture_is_self_consistent(golden_worked_example):
    """The transcription itself: printed zeros are exactly the printed mask,
    row 0 prints 1.0000 and each live row sums to 1 up to 4-decimal rounding."""
    seq_lens, mask, out = golden_worked_example
    assert list(seq_lens) == [3, 4, 5]
    for b in range(3):
        for m in range(2):
            assert np.array_equal(out[b, m] == 0.0, mask[b])
            assert out[b, m, 0, 0] == 1.0
            for r in range(5):
                if not mask[b, r].all():
                    assert abs(out[b, m, r].sum() - 1.0) <= 5 * 0.5e-4 + 1e-12


def test_worked_example_mask_pattern(golden_worked_example):
    """The oracle's zero pattern equals the printed causal_mask for every head."""
    seq_lens, mask, _ = golden_worked_example
    rng = np.random.default_rng(1)
    x = rng.standard_normal((3, 2, 5, 5))
    y = _fwd64(x, seq_lens)
    for b in range(3):
        for m in range(2):
            assert np.array_equal(y[b, m] == 0.0, mask[b])


def test_worked_example_values_from_printed_output(golden_worked_example):
    """Softmax is shift invariant, so logits x = log(printed y) on the kept
    entries reproduce the printed values up to the print rounding. NaN placed in
    every masked input must not reach the output (masked entries are not read)."""
    seq_lens, mask, out = golden_worked_example
    x = np.where(mask[:, None], np.nan, np.log(np.where(out > 0, out, 1.0)))
    x = x + np.arange(6).reshape(3, 2, 1, 1) * 0.37  # arbitrary per-slice shift
    y = _fwd64(x, seq_lens)
    assert not np.isnan(y).any()
    assert np.all(y[np.broadcast_to(mask[:, None], y.shape)] == 0.0)
    assert np.max(np.abs(y - out)) <= 2e-4


def test_row0_is_one_hot():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((2, 3, 7, 7)) * 5
    y = _fwd64(x, np.array([7, 1], np.int32), scale=0.3)
    assert np.all(y[:, :, 0, 0] == 1.0)
    assert np.all(y[:, :, 0, 1:] == 0.0)


# ---------------------------------------------------------------------------
# Closed forms of the forward
# ---------------------------------------------------------------------------

def test_equal_inputs_give_uniform_rows():
    S = 9
    x = np.full((1, 1, S, S), 3.25)
    y = _fwd64(x, np.array([S], np.int32), scale=1.7)
    for r in range(S):
        np.testing.assert_allclose(y[0, 0, r, : r + 1], 1.0 / (r + 1), rtol=1e-15)
        assert np.all(y[0, 0, r, r + 1:] == 0.0)


def test_two_entry_row_is_logistic():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((1, 4, 2, 2)) * 3
    for scale in (1.0, 0.125, -2.0):
        y = _fwd64(x, np.array([2], np.int32), scale=scale)
        for m in range(4):
            x0, x1 = x[0, m, 1, 0], x[0, m, 1, 1]
            expect0 = 1.0 / (1.0 + math.exp(scale * (x1 - x0)))
            assert abs(y[0, m, 1, 0] - expect0) <= 1e-15
            assert abs(y[0, m, 1, 1] - (1.0 - expect0)) <= 1e-15


def test_zero_scale_gives_uniform_rows():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((1, 1, 6, 6)) * 10
    y = _fwd64(x, np.array([6], np.int32), scale=0.0)
    for r in range(6):
        np.testing.assert_allclose(y[0, 0, r, : r + 1], 1.0 / (r + 1), rtol=1e-15)


def test_large_offsets_do_not_overflow():
    """exp(800) overflows double: only a max-subtracted softmax survives this."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((1, 2, 8, 8))
    y0 = _fwd64(x, np.array([8], np.int32))
    y1 = _fwd64(x + 800.0, np.array([8], np.int32))
    assert np.all(np.isfinite(y1))
    np.testing.assert_allclose(y1, y0, rtol=0, atol=1e-12)


def test_negative_scale_equals_negated_input():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((2, 2, 6, 6))
    sl = np.array([4, 6], np.int32)
    assert np.array_equal(_fwd64(x, sl, scale=-0.5), _fwd64(-x, sl, scale=0.5))


def test_live_rows_sum_to_one_and_are_positive():
    rng = np.random.default_rng(7)
    B, M, S = 3, 2, 40
    x = rng.standard_normal((B, M, S, S)) * 4
    sl = np.array([40, 17, 1], np.int32)
    y = _fwd64(x, sl, scale=0.9)
    n = oracle.kept_prefix_lengths(sl, M, S)
    for b in range(B):
        for r in range(S):
            if n[b, r]:
                np.testing.assert_allclose(y[b, :, r].sum(-1), 1.0, rtol=0, atol=1e-14)
                assert np.all(y[b, :, r, : n[b, r]] > 0)
            else:
                assert np.all(y[b, :, r] == 0)


# ---------------------------------------------------------------------------
# Textbook routines in float64 (library code, not the oracle)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("S,L", [(1, 1), (5, 5), (16, 16), (33, 20), (64, 1), (64, 64)])
def test_matches_torch_causal_softmax(S, L):
    """With L = S the op is the textbook causal softmax; rows >= L become zero."""
    g = torch.Generator().manual_seed(100 + S + L)
    x = torch.randn(1, 3, S, S, generator=g, dtype=torch.float64) * 2
    scale = 0.7
    causal = torch.triu(torch.ones(S, S, dtype=torch.bool), 1)
    ref = torch.softmax((x * scale).masked_fill(causal, float("-inf")), dim=-1)
    ref[:, :, L:, :] = 0.0
    y = _fwd64(x.numpy(), np.array([L], np.int32), scale=scale)
    np.testing.assert_allclose(y, ref.numpy(), rtol=0, atol=1e-15)


def test_matches_scipy_softmax_per_row():
    scipy_special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(8)
    S = 23
    x = rng.standard_normal((2, 1, S, S)) * 3
    sl = np.array([23, 11], np.int32)
    y = _fwd64(x, sl, scale=1.3)
    for b in range(2):
        for r in range(sl[b]):
            ref = scipy_special.softmax(1.3 * x[b, 0, r, : r + 1])
            np.testing.assert_allclose(y[b, 0, r, : r + 1], ref, rtol=1e-14, atol=1e-16)


def test_seq_len_is_clamped():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((4, 1, 6, 6))
    y = _fwd64(x, np.array([-3, 0, 6, 99], np.int32))
    assert np.all(y[0] == 0) and np.all(y[1] == 0)
    np.testing.assert_array_equal(y[3], _fwd64(x[3:4], np.array([6], np.int32))[0])


# ---------------------------------------------------------------------------
# Backward
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("L", range(0, 8))
def test_backward_matches_central_differences(L):
    """dx is the gradient of F(x) = sum_c dy_c * y_c(x): central differences of
    the oracle's own forward, h = 1e-6, agree to 1e-8."""
    S, scale, h = 7, 0.8, 1e-6
    rng = np.random.default_rng(10 + L)
    x = rng.standard_normal((1, 1, S, S))
    dy = rng.standard_normal((1, 1, S, S))
    sl = np.array([L], np.int32)
    y = _fwd64(x, sl, scale)
    dx = _bwd64(y, dy, sl, scale)
    num = np.zeros_like(x)
    for r in range(S):
        for c in range(S):
            xp, xm = x.copy(), x.copy()
            xp[0, 0, r, c] += h
            xm[0, 0, r, c] -= h
            num[0, 0, r, c] = ((_fwd64(xp, sl, scale) * dy).sum() - (_fwd64(xm, sl, scale) * dy).sum()) / (2 * h)
    np.testing.assert_allclose(dx, num, rtol=0, atol=1e-8)


@pytest.mark.parametrize("S,L,scale", [(9, 9, 1.0), (17, 12, 0.125), (40, 3, -1.5)])
def test_backward_matches_torch_autograd(S, L, scale):
    g = torch.Generator().manual_seed(7 * S + L)
    x = torch.randn(2, 2, S, S, generator=g, dtype=torch.float64).requires_grad_(True)
    dy = torch.randn(2, 2, S, S, generator=g, dtype=torch.float64)
    causal = torch.triu(torch.ones(S, S, dtype=torch.bool), 1)
    ref_y = torch.softmax((x * scale).masked_fill(causal, float("-inf")), dim=-1)
    keep = torch.zeros(S, S, dtype=torch.float64)
    keep[:L] = 1.0
    ref_y = ref_y * keep
    (ref_y * dy).sum().backward()
    sl = np.array([L, L], np.int32)
    dx = _bwd64(ref_y.detach().numpy(), dy.numpy(), sl, scale)
    np.testing.assert_allclose(dx, x.grad.numpy(), rtol=0, atol=1e-13)


def test_backward_jacobian_entrywise():
    """dx = scale * J^T dy with J_ij = y_i (delta_ij - y_j) (section 2.1's Jacobian)."""
    rng = np.random.default_rng(11)
    S, scale = 6, 0.6
    x = rng.standard_normal((1, 1, S, S))
    dy = rng.standard_normal((1, 1, S, S))
    sl = np.array([S], np.int32)
    y = _fwd64(x, sl, scale)
    dx = _bwd64(y, dy, sl, scale)
    for r in range(S):
        n = r + 1
        yr = y[0, 0, r, :n]
        J = np.empty((n, n))
        for i in range(n):
            for j in range(n):
                J[i, j] = yr[i] * ((1.0 if i == j else 0.0) - yr[j])
        np.testing.assert_allclose(dx[0, 0, r, :n], scale * J.T @ dy[0, 0, r, :n], rtol=0, atol=1e-15)


def test_backward_invariants():
    rng = np.random.default_rng(12)
    B, M, S = 2, 2, 30
    x = rng.standard_normal((B, M, S, S)) * 2
    sl = np.array([30, 9], np.int32)
    y = _fwd64(x, sl, 0.5)
    # gradients of a softmax sum to zero over the kept prefix
    dx = _bwd64(y, rng.standard_normal((B, M, S, S)), sl, 0.5)
    np.testing.assert_allclose(dx.sum(-1), 0.0, atol=1e-14)
    # a constant upstream gradient leaves the softmax gradient at zero
    dx_const = _bwd64(y, np.full((B, M, S, S), -3.5), sl, 0.5)
    assert np.max(np.abs(dx_const)) <= 1e-15
    # masked positions: exactly zero, and never read (NaN sentinels in masked y / dy)
    n = oracle.kept_prefix_lengths(sl, M, S)
    masked = np.arange(S)[None, None, :] >= n[:, :, None]          # [B, S(rows), S(cols)]
    masked = np.broadcast_to(masked[:, None], dx.shape)
    dy = rng.standard_normal((B, M, S, S))
    dy_nan, y_nan = dy.copy(), y.copy()
    dy_nan[masked] = np.nan
    y_nan[masked] = np.nan
    ref = _bwd64(y, dy, sl, 0.5)
    got = _bwd64(y_nan, dy_nan, sl, 0.5)
    assert np.array_equal(got, ref)
    assert np.all(got[masked] == 0.0)


# ---------------------------------------------------------------------------
# Element decoding and rounding (IEEE 754 binary16 / bfloat16 / binary32)
# ---------------------------------------------------------------------------

def test_decode_f16_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.decode(bits, F16)
    ref = bits.view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def test_decode_bf16_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.decode(bits, BF16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def _rounding_probe_values(rng):
    mags = np.exp(rng.uniform(np.log(1e-9), np.log(7e4), 200000))
    v = mags * rng.choice([-1.0, 1.0], mags.size)
    # exact midpoints between consecutive binary16 values, and their neighbours
    h = np.arange(0, 0x7bff, 7, dtype=np.uint16).view(np.float16).astype(np.float64)
    h_next = (np.arange(0, 0x7bff, 7, dtype=np.uint16) + 1).view(np.float16).astype(np.float64)
    mid = (h + h_next) / 2
    extra = np.concatenate([mid, -mid, np.nextafter(mid, 0), np.nextafter(mid, 1e9),
                            [65504.0, 65519.99, 65520.0, 65536.0, 1e-8, 2.0**-25, 2.0**-24 * 1.5,
                             -0.0, 0.0, np.inf, -np.inf]])
    return np.concatenate([v, extra])


def test_round_f16_matches_numpy():
    v = _rounding_probe_values(np.random.default_rng(13))
    got = oracle.round_to(v, F16)
    ref = v.astype(np.float16).view(np.uint16)   # numpy converts double -> half directly
    assert np.array_equal(got, ref)


def test_round_bf16_matches_torch_on_float32_values():
    rng = np.random.default_rng(14)
    f = (rng.standard_normal(200000) * np.exp(rng.uniform(-60, 60, 200000))).astype(np.float32)
    # exact bfloat16 midpoints (low 16 bits = 0x8000), both parities
    mids = (rng.integers(0x00800000, 0x7f000000, 20000, dtype=np.uint32) & 0xffff0000) | 0x8000
    f = np.concatenate([f, mids.view(np.float32)])
    got = oracle.round_to(f.astype(np.float64), BF16)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


def test_round_bf16_is_nearest_with_ties_to_even():
    """Brute force on doubles: the result is the nearest bfloat16, even on ties."""
    rng = np.random.default_rng(15)
    v = rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))
    got = oracle.round_to(v, BF16)
    for val, b in zip(v[:3000], got[:3000]):
        cand = np.array([int(b) - 1, int(b), int(b) + 1], dtype=np.int64) & 0xffff
        vals = oracle.decode(cand.astype(np.uint16), BF16)
        d = np.abs(vals - val)
        assert d[1] <= d[0] and d[1] <= d[2]
        if d[1] == d[0] or d[1] == d[2]:
            assert int(b) % 2 == 0


def test_round_f32_matches_numpy():
    rng = np.random.default_rng(16)
    v = rng.standard_normal(100000) * np.exp(rng.uniform(-80, 80, 100000))
    assert np.array_equal(oracle.round_to(v, F32), v.astype(np.float32).view(np.uint32))


# ---------------------------------------------------------------------------
# Host logic of the oracle wrapper
# ---------------------------------------------------------------------------

def test_row_ranges_and_threads_are_bit_identical():
    rng = np.random.default_rng(17)
    B, M, S = 3, 4, 37
    x = rng.standard_normal((B, M, S, S)).astype(np.float32)
    sl = np.array([37, 20, 5], np.int32)
    whole = oracle.forward(x, sl, B, M, S, 0.125, F32)
    threaded = oracle.forward(x, sl, B, M, S, 0.125, F32, threads=4)
    assert np.array_equal(whole, threaded)
    rows = x.reshape(B * M * S, S)
    part = oracle.forward(rows[100:250], sl, B, M, S, 0.125, F32, row_begin=100, row_end=250)
    assert np.array_equal(part, whole[100:250])
    dy = rng.standard_normal((B, M, S, S)).astype(np.float32)
    yb = oracle.round_to(whole, F32)
    g1 = oracle.backward(yb, dy, sl, B, M, S, 0.125, F32)
    g2 = oracle.backward(yb, dy, sl, B, M, S, 0.125, F32, threads=3)
    assert np.array_equal(g1, g2)


def test_half_precision_inputs_are_decoded_exactly():
    """Forward on bf16 / fp16 bits equals forward on their exact float64 values."""
    rng = np.random.default_rng(18)
    B, M, S = 1, 2, 12
    x = rng.standard_normal((B, M, S, S)) * 3
    sl = np.array([10], np.int32)
    for code in (BF16, F16):
        bits = oracle.round_to(x, code)
        a = oracle.forward(bits, sl, B, M, S, 0.125, code)
        b = oracle.forward(oracle.decode(bits, code), sl, B, M, S, 0.125, F64)
        assert np.array_equal(a, b)


# ---------------------------------------------------------------------------
# Mask families ("优化ScaledMaskSoftmax算子" section 6): length mask, sliding window
# ---------------------------------------------------------------------------

def _fwd64_kind(x, seq_lens, scale, kind, window=0):
    B, M, S, _ = x.shape
    y = oracle.forward(np.ascontiguousarray(x, np.float64), seq_lens, B, M, S, scale, F64, mask_kind=kind,
                       window=window)
    return y.reshape(B, M, S, S)


def _bwd64_kind(y, dy, seq_lens, scale, kind, window=0):
    B, M, S, _ = y.shape
    dx = oracle.backward(np.ascontiguousarray(y, np.float64), np.ascontiguousarray(dy, np.float64), seq_lens,
                         B, M, S, scale, F64, mask_kind=kind, window=window)
    return dx.reshape(B, M, S, S)


@pytest.mark.parametrize("S,L", [(6, 6), (20, 13), (33, 1), (16, 0)])
def test_length_mask_matches_torch_key_padding_softmax(S, L):
    """Kind 1: torch.softmax with a key-padding mask (c >= L masked), padded query rows zero."""
    g = torch.Generator().manual_seed(200 + S + L)
    x = torch.randn(2, 2, S, S, generator=g, dtype=torch.float64) * 2
    scale = 0.9
    key_pad = (torch.arange(S) >= L)[None, :].expand(S, S)
    ref = torch.softmax((x * scale).masked_fill(key_pad, float("-inf")), dim=-1)
    ref[:, :, L:, :] = 0.0
    ref = torch.nan_to_num(ref, nan=0.0)
    y = _fwd64_kind(x.numpy(), np.array([L, L], np.int32), scale, 1)
    np.testing.assert_allclose(y, ref.numpy(), rtol=0, atol=1e-15)


@pytest.mark.parametrize("S,L,w", [(9, 9, 3), (20, 15, 1), (20, 20, 7), (17, 10, 40)])
def test_sliding_window_matches_torch_band_softmax(S, L, w):
    """Kind 2: torch.softmax with a causal band of width w masked outside."""
    g = torch.Generator().manual_seed(300 + S + L + w)
    x = torch.randn(1, 3, S, S, generator=g, dtype=torch.float64) * 2
    r = torch.arange(S)[:, None]
    c = torch.arange(S)[None, :]
    outside = (c > r) | (c <= r - w)
    ref = torch.softmax((x * 0.6).masked_fill(outside, float("-inf")), dim=-1)
    ref[:, :, L:, :] = 0.0
    y = _fwd64_kind(x.numpy(), np.array([L], np.int32), 0.6, 2, w)
    np.testing.assert_allclose(y, ref.numpy(), rtol=0, atol=1e-15)


def test_window_special_cases():
    rng = np.random.default_rng(19)
    x = rng.standard_normal((2, 2, 12, 12)) * 3
    sl = np.array([12, 7], np.int32)
    # width 1: each live row keeps only its diagonal -> exactly one-hot
    y1 = _fwd64_kind(x, sl, 1.3, 2, 1)
    eye = np.eye(12)[None, None]
    live = (np.arange(12)[None, :] < sl[:, None])[:, None, :, None]
    assert np.array_equal(y1, np.broadcast_to(np.where(live, eye, 0.0), y1.shape))
    # a window as wide as the row is the default grouped-tril op
    assert np.array_equal(_fwd64_kind(x, sl, 1.3, 2, 12), _fwd64(x, sl, 1.3))
    assert np.array_equal(_fwd64_kind(x, sl, 1.3, 2, 500), _fwd64(x, sl, 1.3))
    # bad arguments: unknown kind, window < 1 for the sliding window
    with pytest.raises(ValueError):
        _fwd64_kind(x, sl, 1.0, 3)
    with pytest.raises(ValueError):
        _fwd64_kind(x, sl, 1.0, 2, 0)


@pytest.mark.parametrize("kind,w", [(1, 0), (2, 3)])
def test_mask_family_backward_matches_central_differences(kind, w):
    S, scale, h = 6, 0.7, 1e-6
    rng = np.random.default_rng(20 + kind)
    x = rng.standard_normal((1, 1, S, S))
    dy = rng.standard_normal((1, 1, S, S))
    sl = np.array([5], np.int32)
    y = _fwd64_kind(x, sl, scale, kind, w)
    dx = _bwd64_kind(y, dy, sl, scale, kind, w)
    num = np.zeros_like(x)
    for r in range(S):
        for c in range(S):
            xp, xm = x.copy(), x.copy()
            xp[0, 0, r, c] += h
            xm[0, 0, r, c] -= h
            num[0, 0, r, c] = ((_fwd64_kind(xp, sl, scale, kind, w) * dy).sum()
                               - (_fwd64_kind(xm, sl, scale, kind, w) * dy).sum()) / (2 * h)
    np.testing.assert_allclose(dx, num, rtol=0, atol=1e-8)


@pytest.mark.parametrize("kind,w", [(0, 0), (1, 0), (2, 4)])
def test_kept_ranges_match_oracle_zero_pattern(kind, w):
    rng = np.random.default_rng(21)
    S = 10
    x = rng.standard_normal((3, 1, S, S))
    sl = np.array([10, 6, 0], np.int32)
    y = _fwd64_kind(x, sl, 1.0, kind, w)
    c0, c1 = oracle.kept_ranges(sl, S, kind, w)
    col = np.arange(S)[None, None, :]
    kept = (col >= c0[:, :, None]) & (col < c1[:, :, None])
    assert np.array_equal(y[:, 0] != 0.0, kept)


# ---------------------------------------------------------------------------
# Explicit mask ("优化ScaledMaskSoftmax算子" sections 2.2 / 3.1 / 4.1)
# ---------------------------------------------------------------------------

def _fwd64_explicit(x, mask, scale=1.0):
    B, M, S, _ = x.shape
    return oracle.forward_explicit(np.ascontiguousarray(x, np.float64), mask, B, M, S, scale, F64).reshape(B, M, S, S)


def _bwd64_explicit(y, dy, mask, scale=1.0):
    B, M, S, _ = y.shape
    return oracle.backward_explicit(np.ascontiguousarray(y, np.float64), np.ascontiguousarray(dy, np.float64), mask,
                                    B, M, S, scale, F64).reshape(B, M, S, S)


def test_explicit_mask_matches_torch_masked_softmax():
    """Random keep-mask with some all-masked rows: torch softmax of a -inf-filled
    input (NaN rows of all-masked inputs become 0, as the section 4.1 guard does)."""
    g = torch.Generator().manual_seed(400)
    B, M, S = 3, 2, 19
    x = torch.randn(B, M, S, S, generator=g, dtype=torch.float64) * 2
    keep = torch.rand(B, S, S, generator=g) < 0.4
    keep[:, 3, :] = False
    keep[1, 7, :] = True
    ref = torch.nan_to_num(torch.softmax((x * 0.8).masked_fill(~keep[:, None], float("-inf")), dim=-1), nan=0.0)
    y = _fwd64_explicit(x.numpy(), keep.numpy().astype(np.uint8), 0.8)
    np.testing.assert_allclose(y, ref.numpy(), rtol=0, atol=1e-15)
    assert np.all(y[:, :, 3, :] == 0.0)


def test_explicit_mask_reduces_to_the_grouped_families():
    """A tril keep-mask restricted to r, c < L is the grouped-tril op; a length
    mask is kind 1; one [1, S, S] mask broadcasts over the batches."""
    rng = np.random.default_rng(22)
    B, M, S = 3, 2, 14
    x = rng.standard_normal((B, M, S, S)) * 2
    sl = np.array([14, 9, 0], np.int32)
    r, c = np.arange(S)[:, None], np.arange(S)[None, :]
    tril = np.stack([((c <= r) & (r < L)) for L in sl]).astype(np.uint8)
    length = np.stack([((c < L) & (r < L)) for L in sl]).astype(np.uint8)
    assert np.array_equal(_fwd64_explicit(x, tril, 0.5), _fwd64(x, sl, 0.5))
    assert np.array_equal(_fwd64_explicit(x, length, 0.5), _fwd64_kind(x, sl, 0.5, 1))
    one = (c <= r).astype(np.uint8)[None]
    assert np.array_equal(_fwd64_explicit(x, one, 0.5), _fwd64(x, np.array([S, S, S], np.int32), 0.5))
    with pytest.raises(ValueError):
        _fwd64_explicit(x, np.ones((2, S, S), np.uint8))


def test_explicit_mask_backward_matches_central_differences():
    rng = np.random.default_rng(23)
    S, scale, h = 6, 0.9, 1e-6
    x = rng.standard_normal((1, 1, S, S))
    dy = rng.standard_normal((1, 1, S, S))
    keep = (rng.random((1, S, S)) < 0.5).astype(np.uint8)
    keep[0, 2, :] = 0
    y = _fwd64_explicit(x, keep, scale)
    dx = _bwd64_explicit(y, dy, keep, scale)
    num = np.zeros_like(x)
    for r in range(S):
        for c in range(S):
            xp, xm = x.copy(), x.copy()
            xp[0, 0, r, c] += h
            xm[0, 0, r, c] -= h
            num[0, 0, r, c] = ((_fwd64_explicit(xp, keep, scale) * dy).sum()
                               - (_fwd64_explicit(xm, keep, scale) * dy).sum()) / (2 * h)
    np.testing.assert_allclose(dx, num, rtol=0, atol=1e-8)
    assert np.all(dx[0, 0][keep[0] == 0] == 0.0)


# ---------------------------------------------------------------------------
# Attention-backward step ("ops(8)" section 2.1): dS from P, dO, V
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("S,d,L", [(8, 4, 8), (17, 16, 11), (33, 8, 0)])
def test_attn_dscores_matches_autograd_through_pv(S, d, L):
    """X.grad of O = masked_softmax(scale * X) V under upstream dO is the fused step's dS."""
    g = torch.Generator().manual_seed(500 + S + d + L)
    B, M, scale = 2, 2, 0.35
    x = (torch.randn(B, M, S, S, generator=g, dtype=torch.float64) * 2).requires_grad_(True)
    v = torch.randn(B, M, S, d, generator=g, dtype=torch.float64)
    dout = torch.randn(B, M, S, d, generator=g, dtype=torch.float64)
    causal = torch.triu(torch.ones(S, S, dtype=torch.bool), 1)
    keep = torch.zeros(S, S, dtype=torch.float64)
    keep[:L] = 1.0
    p = torch.softmax((x * scale).masked_fill(causal, float("-inf")), dim=-1) * keep
    (p @ v).backward(dout)
    sl = np.array([L, L], np.int32)
    ds = oracle.attn_dscores(p.detach().numpy(), dout.numpy(), v.numpy(), sl, B, M, S, d, scale, F64)
    np.testing.assert_allclose(ds.reshape(B, M, S, S), x.grad.numpy(), rtol=0, atol=1e-13)


def test_attn_dscores_is_softmax_backward_of_dp():
    rng = np.random.default_rng(24)
    B, M, S, d = 2, 1, 12, 5
    x = rng.standard_normal((B, M, S, S))
    v = rng.standard_normal((B, M, S, d))
    dout = rng.standard_normal((B, M, S, d))
    sl = np.array([12, 7], np.int32)
    p = _fwd64(x, sl, 0.5)
    dp = dout @ np.swapaxes(v, -1, -2)
    ds = oracle.attn_dscores(p, dout, v, sl, B, M, S, d, 0.5, F64, threads=3).reshape(B, M, S, S)
    np.testing.assert_allclose(ds, _bwd64(p, dp, sl, 0.5), rtol=0, atol=1e-13)
