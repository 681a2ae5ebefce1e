/*
 * gtms_oracle.c -- plain, slow, double-precision CPU oracle for the
 * grouped-tril masked softmax (forward) and its softmax backward.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path links, loads or calls
 * this file: only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline /
 * reference leg use it. It shares no code, header, table or helper with the
 * CUDA library.
 *
 * What it computes (one row at a time, no blocking, no fusion):
 *
 *   Mask. "Attention-Mask-Optimization" README, section "算子行为（融合下面的计算）"
 *   (operator behaviour): for batch b with valid length L = seq_len[b], entry
 *   (row, col) of the [S,S] score matrix is kept iff row < L, col < L and
 *   col <= row; the same mask applies to every head m. Because col <= row < L
 *   implies col < L, the kept set of row r is the prefix col in [0, n) with
 *   n = r + 1 when r < L and n = 0 otherwise.
 *
 *   Forward. Softmax over the kept entries of each row, with the scale applied
 *   inside the exponent as in "优化ScaledMaskSoftmax算子", section 4.1
 *   (exp(input*scale)). Masked entries and whole padded rows are exactly +0.0
 *   (reading taken: the README's post-hoc `attn == 1/S` zeroing is an artefact
 *   of its fill-with-minus-max reference; the printed output shows plain zeros).
 *
 *   Backward. "ops(8): self-attention 的 CUDA 实现及优化 (下)", section 2.1
 *   (Softmax 求导): dy_i/dx_j = y_i (delta_ij - y_j). Through z = scale*x the
 *   chain rule gives dx_c = scale * y_c * (dy_c - sum_j dy_j y_j) on kept
 *   entries (section 2.2 applies the scale in the softmax backward pass);
 *   masked entries get +0.0.
 *
 *   Rounding. Results are produced in double. oracle_round() rounds a double
 *   once, to nearest with ties to even, into fp32 / bf16 / fp16 bit patterns
 *   (reading taken: the pages never state a rounding rule; IEEE 754 default).
 *
 * seq_len values outside [0, S] are clamped to that range (reading taken: the
 * pages only show 1 <= seq_len <= S).
 *
 * Mask families ("优化ScaledMaskSoftmax算子", section 6, lists a local window
 * mask and a length mask besides the default). Every family keeps a
 * contiguous column range [c0, c1) of row r < L and nothing of rows r >= L:
 *   kind 0, grouped tril (default): [0, r + 1);
 *   kind 1, length mask:            [0, L)          (key padding; r < L only);
 *   kind 2, sliding causal window:  [max(0, r - w + 1), r + 1), window w >= 1.
 * Reading taken for kind 2: the section's garbled tril(window_size) snippet
 * under the heading "local window attention" is read as the usual causal band
 * of width w. Reading taken for kind 1: padded query rows stay all-zero, as in
 * the default op.
 *
 * Explicit mask ("优化ScaledMaskSoftmax算子", sections 2.2 and 3.1: the op takes
 * the input, a mask tensor and the scale). Reading taken: a nonzero mask byte
 * marks a kept entry -- the article's own masks are ones(L, L).tril(...) and
 * arange(L) < lengths, both 1 where attention is allowed -- and a row with no
 * kept entry is all +0.0 (section 4.1 guards the all-masked row). The mask is
 * uint8 [mask_batches, S, S] with mask_batches 1 (one mask for every batch) or
 * B, and is shared by the M heads.
 *
 * Attention-backward step ("ops(8): self-attention 的 CUDA 实现及优化 (下)", section
 * 2.1: with P = softmax(S), O = P V the backward runs dP = dO V^T, then
 * dS = softmax-backward(dP, P)). gtms_oracle_attn_dscores forms, for each row,
 * dP_rc = sum_k dO_rk V_ck on the kept columns (grouped tril mask) and
 * dS_rc = scale * P_rc * (dP_rc - sum_c' dP_rc' P_rc'), +0.0 elsewhere; dO and
 * V are [B, M, S, d].
 *
 * Build: cc -O2 -fno-fast-math -fPIC -shared gtms_oracle.c -o libgtms_oracle.so -lm
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F16 = 2, ORC_F64 = 3 };
enum { ORC_OK = 0, ORC_BAD_ARG = 1 };

/* ---- element decoding (IEEE 754 binary32 / binary16, and bfloat16 = top half of binary32) ---- */

static double f32_bits_to_double(uint32_t bits)
{
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static double f16_bits_to_double(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int expo = (h >> 10) & 0x1f;
    const int frac = h & 0x3ff;
    double mag;
    if (expo == 0)
        mag = ldexp((double)frac, -24);                  /* zero or subnormal: frac * 2^-24 */
    else if (expo == 31)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(1024 + frac), expo - 25);   /* (1 + frac/2^10) * 2^(expo-15) */
    return sign ? -mag : mag;
}

static double load_elem(const void* base, int64_t i, int dtype)
{
    switch (dtype) {
    case ORC_F32: {
        uint32_t b;
        memcpy(&b, (const char*)base + 4 * i, 4);
        return f32_bits_to_double(b);
    }
    case ORC_BF16: {
        uint16_t b;
        memcpy(&b, (const char*)base + 2 * i, 2);
        return f32_bits_to_double((uint32_t)b << 16);
    }
    case ORC_F16: {
        uint16_t b;
        memcpy(&b, (const char*)base + 2 * i, 2);
        return f16_bits_to_double(b);
    }
    default: {
        double d;
        memcpy(&d, (const char*)base + 8 * i, 8);
        return d;
    }
    }
}

/* ---- rounding a double once, to nearest, ties to even ----
 * Format with p significand bits (implicit bit included), minimum normal
 * exponent emin and maximum exponent emax. Returns the rounded value as a
 * double (exactly representable in the target format) or +-inf on overflow. */
static double round_to_format(double v, int p, int emin, int emax)
{
    if (isnan(v) || isinf(v) || v == 0.0)
        return v;
    int e2;
    frexp(fabs(v), &e2);           /* |v| = f * 2^e2, f in [0.5, 1): leading bit is 2^(e2-1) */
    int lead = e2 - 1;
    if (lead < emin)
        lead = emin;               /* subnormal range: fixed quantum */
    const double quantum = ldexp(1.0, lead - (p - 1));
    const double q = nearbyint(v / quantum);   /* exact scaling; default mode rounds ties to even */
    const double r = q * quantum;
    const double max_finite = ldexp(2.0 - ldexp(1.0, 1 - p), emax);
    if (fabs(r) > max_finite)
        return copysign(INFINITY, v);
    return r;
}

static uint16_t double_to_f16_bits(double v)
{
    if (isnan(v))
        return 0x7e00;
    const double r = round_to_format(v, 11, -14, 15);
    const uint16_t sign = signbit(r) ? 0x8000 : 0;
    const double a = fabs(r);
    if (isinf(a))
        return sign | 0x7c00;
    if (a == 0.0)
        return sign;
    if (a < ldexp(1.0, -14))                            /* subnormal: a = frac * 2^-24 */
        return sign | (uint16_t)(a / ldexp(1.0, -24));
    int e2;
    frexp(a, &e2);
    const int expo = e2 - 1;                            /* a in [2^expo, 2^(expo+1)) */
    const uint16_t frac = (uint16_t)((a / ldexp(1.0, expo) - 1.0) * 1024.0);
    return sign | (uint16_t)((expo + 15) << 10) | frac;
}

static uint16_t double_to_bf16_bits(double v)
{
    if (isnan(v))
        return 0x7fc0;
    const float r = (float)round_to_format(v, 8, -126, 127);   /* exact in binary32 */
    uint32_t b;
    memcpy(&b, &r, 4);
    return (uint16_t)(b >> 16);
}

static void store_rounded(void* out, int64_t i, double v, int dtype)
{
    switch (dtype) {
    case ORC_F32: {
        const float f = (float)v;   /* C conversion: round to nearest even in the default mode */
        memcpy((char*)out + 4 * i, &f, 4);
        break;
    }
    case ORC_BF16: {
        const uint16_t b = double_to_bf16_bits(v);
        memcpy((char*)out + 2 * i, &b, 2);
        break;
    }
    case ORC_F16: {
        const uint16_t b = double_to_f16_bits(v);
        memcpy((char*)out + 2 * i, &b, 2);
        break;
    }
    default:
        memcpy((char*)out + 8 * i, &v, 8);
    }
}

/* ---- mask ---- */

/* Kept column range [*c0, *c1) of row q (flat row id over [B, M, S]); empty
 * when *c1 <= *c0. */
static void kept_range(const int32_t* seq_lens, int64_t M, int64_t S, int kind, int64_t window, int64_t q,
                       int64_t* c0, int64_t* c1)
{
    const int64_t b = q / (M * S);
    const int64_t r = q % S;
    int64_t L = seq_lens[b];
    if (L < 0)
        L = 0;
    if (L > S)
        L = S;
    *c0 = 0;
    *c1 = 0;
    if (r >= L)
        return;
    if (kind == 1) {
        *c1 = L;
    } else {
        *c1 = r + 1;
        if (kind == 2 && r - window + 1 > 0)
            *c0 = r - window + 1;
    }
}

static int bad_shape(int64_t B, int64_t M, int64_t S, int64_t row_begin, int64_t row_end)
{
    if (B < 0 || M < 0 || S < 0 || row_begin < 0 || row_end < row_begin)
        return 1;
    return row_end > B * M * S;
}

static int bad_mask(int kind, int64_t window)
{
    return kind < 0 || kind > 2 || (kind == 2 && window < 1);
}

/* ---- forward ----
 * x: rows [row_begin, row_end) of X[B,M,S,S], contiguous, element type dtype.
 * y: (row_end - row_begin) * S doubles. */
int gtms_oracle_forward_masked(const void* x, int dtype, const int32_t* seq_lens,
                               int64_t B, int64_t M, int64_t S, double scale, int kind, int64_t window,
                               int64_t row_begin, int64_t row_end, double* y)
{
    if (dtype < ORC_F32 || dtype > ORC_F64 || bad_shape(B, M, S, row_begin, row_end) || bad_mask(kind, window))
        return ORC_BAD_ARG;
    for (int64_t q = row_begin; q < row_end; ++q) {
        const int64_t base = (q - row_begin) * S;
        int64_t c0, c1;
        kept_range(seq_lens, M, S, kind, window, q, &c0, &c1);
        double* yr = y + base;
        for (int64_t c = 0; c < S; ++c)
            yr[c] = 0.0;
        if (c1 <= c0)
            continue;
        /* z_c = scale * x_c; the row maximum is subtracted before exp so that
         * large scores cannot overflow (the result is unchanged mathematically). */
        double zmax = -INFINITY;
        for (int64_t c = c0; c < c1; ++c) {
            const double z = scale * load_elem(x, base + c, dtype);
            if (z > zmax)
                zmax = z;
        }
        double sum = 0.0;
        for (int64_t c = c0; c < c1; ++c) {
            const double e = exp(scale * load_elem(x, base + c, dtype) - zmax);
            yr[c] = e;
            sum += e;
        }
        for (int64_t c = c0; c < c1; ++c)
            yr[c] = yr[c] / sum;
    }
    return ORC_OK;
}

int gtms_oracle_forward(const void* x, int dtype, const int32_t* seq_lens,
                        int64_t B, int64_t M, int64_t S, double scale,
                        int64_t row_begin, int64_t row_end, double* y)
{
    return gtms_oracle_forward_masked(x, dtype, seq_lens, B, M, S, scale, 0, 0, row_begin, row_end, y);
}

/* ---- backward ----
 * y, dy: rows [row_begin, row_end), element type dtype (ORC_F64 accepted for
 * unrounded inputs). dx: (row_end - row_begin) * S doubles. */
int gtms_oracle_backward_masked(const void* y, const void* dy, int dtype, const int32_t* seq_lens,
                                int64_t B, int64_t M, int64_t S, double scale, int kind, int64_t window,
                                int64_t row_begin, int64_t row_end, double* dx)
{
    if (dtype < ORC_F32 || dtype > ORC_F64 || bad_shape(B, M, S, row_begin, row_end) || bad_mask(kind, window))
        return ORC_BAD_ARG;
    for (int64_t q = row_begin; q < row_end; ++q) {
        const int64_t base = (q - row_begin) * S;
        int64_t c0, c1;
        kept_range(seq_lens, M, S, kind, window, q, &c0, &c1);
        double* dxr = dx + base;
        for (int64_t c = 0; c < S; ++c)
            dxr[c] = 0.0;
        if (c1 <= c0)
            continue;
        double dot = 0.0;   /* sum_j dy_j * y_j over the kept range */
        for (int64_t c = c0; c < c1; ++c)
            dot += load_elem(dy, base + c, dtype) * load_elem(y, base + c, dtype);
        for (int64_t c = c0; c < c1; ++c) {
            const double yc = load_elem(y, base + c, dtype);
            const double dyc = load_elem(dy, base + c, dtype);
            dxr[c] = scale * yc * (dyc - dot);
        }
    }
    return ORC_OK;
}

int gtms_oracle_backward(const void* y, const void* dy, int dtype, const int32_t* seq_lens,
                         int64_t B, int64_t M, int64_t S, double scale,
                         int64_t row_begin, int64_t row_end, double* dx)
{
    return gtms_oracle_backward_masked(y, dy, dtype, seq_lens, B, M, S, scale, 0, 0, row_begin, row_end, dx);
}

/* ---- attention-backward step: dS from P, dO, V ----
 * p: rows [row_begin, row_end) of P[B,M,S,S]; dout, v: the whole [B,M,S,d]
 * tensors. ds: (row_end - row_begin) * S doubles. */
int gtms_oracle_attn_dscores(const void* p, const void* dout, const void* v, int dtype, const int32_t* seq_lens,
                             int64_t B, int64_t M, int64_t S, int64_t d, double scale,
                             int64_t row_begin, int64_t row_end, double* ds)
{
    if (dtype < ORC_F32 || dtype > ORC_F64 || bad_shape(B, M, S, row_begin, row_end) || d < 1)
        return ORC_BAD_ARG;
    for (int64_t q = row_begin; q < row_end; ++q) {
        const int64_t base = (q - row_begin) * S;
        int64_t c0, c1;
        kept_range(seq_lens, M, S, 0, 0, q, &c0, &c1);
        const int64_t slice = q / S;               /* (b, m) */
        const int64_t r = q % S;
        double* dsr = ds + base;
        for (int64_t c = 0; c < S; ++c)
            dsr[c] = 0.0;
        if (c1 <= c0)
            continue;
        double dot = 0.0;                          /* sum_c dP_rc P_rc */
        for (int64_t c = c0; c < c1; ++c) {
            double dp = 0.0;
            for (int64_t k = 0; k < d; ++k)
                dp += load_elem(dout, (slice * S + r) * d + k, dtype) * load_elem(v, (slice * S + c) * d + k, dtype);
            dsr[c] = dp;                           /* dP held here until the second loop */
            dot += dp * load_elem(p, base + c, dtype);
        }
        for (int64_t c = c0; c < c1; ++c)
            dsr[c] = scale * load_elem(p, base + c, dtype) * (dsr[c] - dot);
    }
    return ORC_OK;
}

/* ---- explicit mask ---- */

static const uint8_t* mask_row(const uint8_t* mask, int64_t mask_batches, int64_t M, int64_t S, int64_t q)
{
    const int64_t b = mask_batches == 1 ? 0 : q / (M * S);
    return mask + (b * S + q % S) * S;
}

int gtms_oracle_forward_explicit(const void* x, int dtype, const uint8_t* mask, int64_t mask_batches,
                                 int64_t B, int64_t M, int64_t S, double scale,
                                 int64_t row_begin, int64_t row_end, double* y)
{
    if (dtype < ORC_F32 || dtype > ORC_F64 || bad_shape(B, M, S, row_begin, row_end) ||
        (mask_batches != 1 && mask_batches != B))
        return ORC_BAD_ARG;
    for (int64_t q = row_begin; q < row_end; ++q) {
        const int64_t base = (q - row_begin) * S;
        const uint8_t* keep = mask_row(mask, mask_batches, M, S, q);
        double* yr = y + base;
        double zmax = -INFINITY;
        int any = 0;
        for (int64_t c = 0; c < S; ++c) {
            yr[c] = 0.0;
            if (keep[c]) {
                const double z = scale * load_elem(x, base + c, dtype);
                if (!any || z > zmax)
                    zmax = z;
                any = 1;
            }
        }
        if (!any)
            continue;
        double sum = 0.0;
        for (int64_t c = 0; c < S; ++c)
            if (keep[c]) {
                yr[c] = exp(scale * load_elem(x, base + c, dtype) - zmax);
                sum += yr[c];
            }
        for (int64_t c = 0; c < S; ++c)
            if (keep[c])
                yr[c] = yr[c] / sum;
    }
    return ORC_OK;
}

int gtms_oracle_backward_explicit(const void* y, const void* dy, int dtype, const uint8_t* mask,
                                  int64_t mask_batches, int64_t B, int64_t M, int64_t S, double scale,
                                  int64_t row_begin, int64_t row_end, double* dx)
{
    if (dtype < ORC_F32 || dtype > ORC_F64 || bad_shape(B, M, S, row_begin, row_end) ||
        (mask_batches != 1 && mask_batches != B))
        return ORC_BAD_ARG;
    for (int64_t q = row_begin; q < row_end; ++q) {
        const int64_t base = (q - row_begin) * S;
        const uint8_t* keep = mask_row(mask, mask_batches, M, S, q);
        double* dxr = dx + base;
        double dot = 0.0;
        for (int64_t c = 0; c < S; ++c) {
            dxr[c] = 0.0;
            if (keep[c])
                dot += load_elem(dy, base + c, dtype) * load_elem(y, base + c, dtype);
        }
        for (int64_t c = 0; c < S; ++c)
            if (keep[c])
                dxr[c] = scale * load_elem(y, base + c, dtype) * (load_elem(dy, base + c, dtype) - dot);
    }
    return ORC_OK;
}

/* ---- element conversion helpers (used by the tests to form expected bits) ---- */

int gtms_oracle_round(const double* v, int64_t n, int dtype, void* out)
{
    if (dtype < ORC_F32 || dtype > ORC_F64 || n < 0)
        return ORC_BAD_ARG;
    for (int64_t i = 0; i < n; ++i)
        store_rounded(out, i, v[i], dtype);
    return ORC_OK;
}

int gtms_oracle_decode(const void* in, int64_t n, int dtype, double* out)
{
    if (dtype < ORC_F32 || dtype > ORC_F64 || n < 0)
        return ORC_BAD_ARG;
    for (int64_t i = 0; i < n; ++i)
        out[i] = load_elem(in, i, dtype);
    return ORC_OK;
}
