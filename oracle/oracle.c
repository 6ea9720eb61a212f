/*
 * Oracle for 3-D max pooling over NCDHW tensors: forward with argmax
 * (fixed and adaptive windows) and the backward that routes each output
 * gradient to its argmax input.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path (the CUDA library,
 * its headers or its Python binding) includes, links or calls this file.
 * Only the tests, the smoke check and the CPU-baseline / reference legs of
 * the benchmark load it. It shares no code, header, table or helper with
 * the CUDA path.
 *
 * Style: plain, single-threaded, unblocked C that follows the definition of
 * each result directly, so that a reader can check it against the pages by
 * eye. There is no tiling, no separable reduction and no reordering.
 *
 * Sources (web pages on the subject):
 *  [MPF]  teenygrad API docs, "Struct Maxpool3dForward": description
 *         ("3-D max-pooling forward pass") and its "Constraints" paragraph
 *         (no padding; OD = (D - KD)/STRIDE_D + 1, likewise OH and OW).
 *  [AMPB] FlagGems-Experimental PR #308, "Add adaptive_max_pool3d_backward
 *         Moore Threads specialized operator", section "Summary": the
 *         backward scatters each output window's gradient back to its
 *         argmax input position; in the divisible case windows tile the
 *         input disjointly, in the non-divisible case windows overlap and
 *         contributions to one input accumulate.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - Adaptive window i along an axis of input size I and output size O is
 *    [floor(i*I/O), ceil((i+1)*I/O)), computed in exact integer arithmetic.
 *  - Ties among equal maxima go to the first occurrence in (d, h, w)
 *    row-major order. +0 and -0 compare equal. A NaN beats every number;
 *    among NaNs the first occurrence wins. The output value is a bit copy
 *    of the winning input element.
 *  - The argmax index is the int64 flat offset d*H*W + h*W + w inside the
 *    element's own (n, c) plane.
 *  - Backward: each input's gradient is the sum, in ascending output order
 *    (od, oh, ow), of the gradients of the outputs whose argmax is that
 *    input, evaluated left to right in binary32 starting from the first
 *    term, then rounded once (round to nearest, ties to even) to the data
 *    type. An input that no output selects gets +0. A single contribution
 *    is therefore copied exactly.
 *  - Comparisons are made on the exact values widened to binary64.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2 };

enum {
    OR_OK = 0,
    OR_ERR_SHAPE = 1,   /* a size or window that the definition rejects */
    OR_ERR_DTYPE = 2,
    OR_ERR_INDEX = 3,   /* backward: an index outside its plane          */
    OR_ERR_NOMEM = 4
};

/* ------------------------------------------------------------------ */
/* Number formats (IEEE 754 binary16, and bfloat16 = the upper 16 bits  */
/* of binary32), written from the format definitions.                  */
/* ------------------------------------------------------------------ */

/* binary16 -> binary32: sign, 5-bit exponent (bias 15), 10-bit fraction.
 * Normal numbers keep sign and fraction and move the exponent from bias 15
 * to bias 127; subnormals are frac * 2^-24 (exact in binary32); infinity
 * and NaN keep sign and fraction (the NaN payload moves to the top of the
 * binary32 fraction). */
float oracle_f16_to_f32(uint16_t h)
{
    uint32_t sign = (uint32_t)(h >> 15) << 31;
    uint32_t e = (h >> 10) & 0x1F;
    uint32_t frac = h & 0x3FF;
    uint32_t bits;
    float f;
    if (e == 0) {
        f = (float)frac * 0x1p-24f;                         /* zero or subnormal */
        return sign ? -f : f;
    }
    if (e == 0x1F)
        bits = sign | (0xFFu << 23) | (frac << 13);         /* infinity or NaN */
    else
        bits = sign | ((e - 15 + 127) << 23) | (frac << 13); /* normal */
    memcpy(&f, &bits, 4);
    return f;
}

/* bfloat16 -> binary32: bfloat16 is the high half of a binary32 pattern. */
float oracle_bf16_to_f32(uint16_t b)
{
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, 4);
    return f;
}

/* Round a (a positive finite binary32 value held exactly in a double) to
 * the nearest value of a binary format with `mbits` fraction bits and
 * minimum normal exponent `emin`, ties to even. Returns the rounded
 * magnitude (exact in a double). The caller handles overflow. */
static double round_to_format(double a, int mbits, int emin)
{
    int e;
    double q, n, fl, frac, r;
    if (a == 0.0)
        return 0.0;
    frexp(a, &e);                 /* a = m * 2^e with 0.5 <= m < 1 */
    e -= 1;                       /* now 2^e <= a < 2^(e+1)        */
    if (e < emin)
        e = emin;                 /* subnormal range: fixed spacing */
    q = ldexp(1.0, e - mbits);    /* spacing of representable values */
    n = a / q;                    /* exact: q is a power of two      */
    fl = floor(n);
    frac = n - fl;
    if (frac > 0.5)
        r = fl + 1.0;
    else if (frac < 0.5)
        r = fl;
    else
        r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;   /* tie: to even */
    return r * q;
}

/* Encode a magnitude v that is representable in the target format. */
static uint16_t encode_small_float(int sign, double v, int mbits, int emin, int ebias, int ebits)
{
    int e;
    uint32_t field, frac;
    uint32_t emax_field = (1u << ebits) - 1;
    if (v == 0.0)
        return (uint16_t)(sign << 15);
    if (v < ldexp(1.0, emin)) {
        /* subnormal: v = frac * 2^(emin - mbits) */
        frac = (uint32_t)(v / ldexp(1.0, emin - mbits));
        return (uint16_t)((sign << 15) | frac);
    }
    frexp(v, &e);
    e -= 1;                                    /* 2^e <= v < 2^(e+1) */
    field = (uint32_t)(e + ebias);
    if (field >= emax_field)                   /* rounded past the largest finite */
        return (uint16_t)((sign << 15) | (emax_field << mbits));
    frac = (uint32_t)(v / ldexp(1.0, e - mbits)) - (1u << mbits);
    return (uint16_t)((sign << 15) | (field << mbits) | frac);
}

/* binary32 -> binary16, round to nearest, ties to even; overflow gives
 * infinity; NaN stays NaN (sign and top payload bits kept, quiet bit set). */
uint16_t oracle_f32_to_f16(float f)
{
    uint32_t bits;
    int sign;
    double r;
    memcpy(&bits, &f, 4);
    sign = (int)(bits >> 31);
    if (isnan(f))
        return (uint16_t)((sign << 15) | 0x7C00 | 0x200 | ((bits >> 13) & 0x3FF));
    if (isinf(f))
        return (uint16_t)((sign << 15) | 0x7C00);
    r = round_to_format(fabs((double)f), 10, -14);
    if (r >= 65536.0)                          /* 2^16: beyond binary16 range */
        return (uint16_t)((sign << 15) | 0x7C00);
    return encode_small_float(sign, r, 10, -14, 15, 5);
}

/* binary32 -> bfloat16 (8 exponent bits, 7 fraction bits), round to
 * nearest, ties to even; overflow gives infinity; NaN stays NaN. */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t bits;
    int sign;
    double r;
    memcpy(&bits, &f, 4);
    sign = (int)(bits >> 31);
    if (isnan(f))
        return (uint16_t)((sign << 15) | 0x7F80 | 0x40 | ((bits >> 16) & 0x7F));
    if (isinf(f))
        return (uint16_t)((sign << 15) | 0x7F80);
    r = round_to_format(fabs((double)f), 7, -126);
    if (r >= ldexp(1.0, 128))
        return (uint16_t)((sign << 15) | 0x7F80);
    return encode_small_float(sign, r, 7, -126, 127, 8);
}

static int elem_size(int dtype)
{
    switch (dtype) {
    case OR_F32: return 4;
    case OR_F16: return 2;
    case OR_BF16: return 2;
    default: return 0;
    }
}

/* Exact value of element i of a buffer of the given type, as a double. */
static double load_value(int dtype, const void* base, int64_t i)
{
    if (dtype == OR_F32)
        return (double)((const float*)base)[i];
    if (dtype == OR_F16)
        return (double)oracle_f16_to_f32(((const uint16_t*)base)[i]);
    return (double)oracle_bf16_to_f32(((const uint16_t*)base)[i]);
}

/* Value of a gradient element as binary32 (exact for all three types). */
static float load_f32(int dtype, const void* base, int64_t i)
{
    if (dtype == OR_F32)
        return ((const float*)base)[i];
    if (dtype == OR_F16)
        return oracle_f16_to_f32(((const uint16_t*)base)[i]);
    return oracle_bf16_to_f32(((const uint16_t*)base)[i]);
}

static void store_rounded(int dtype, void* base, int64_t i, float v)
{
    if (dtype == OR_F32)
        ((float*)base)[i] = v;
    else if (dtype == OR_F16)
        ((uint16_t*)base)[i] = oracle_f32_to_f16(v);
    else
        ((uint16_t*)base)[i] = oracle_f32_to_bf16(v);
}

/* ------------------------------------------------------------------ */
/* Window geometry                                                      */
/* ------------------------------------------------------------------ */

/* [MPF] Constraints: no padding, O = (I - K) / S + 1 (integer division).
 * Returns 0 when the window does not fit (I < K) or an argument is < 1. */
int64_t oracle_fixed_out_size(int64_t I, int64_t K, int64_t S)
{
    if (I < 1 || K < 1 || S < 1 || I < K)
        return 0;
    return (I - K) / S + 1;
}

/* Fixed window o along one axis: [o*S, o*S + K). */
void oracle_fixed_window(int64_t o, int64_t K, int64_t S, int64_t* start, int64_t* end)
{
    *start = o * S;
    *end = o * S + K;
}

/* Adaptive window i along an axis (input size I, output size O):
 * [floor(i*I/O), ceil((i+1)*I/O)). */
void oracle_adaptive_window(int64_t i, int64_t I, int64_t O, int64_t* start, int64_t* end)
{
    *start = (i * I) / O;
    *end = ((i + 1) * I + O - 1) / O;
}

/* ------------------------------------------------------------------ */
/* Forward                                                              */
/* ------------------------------------------------------------------ */

/* "v beats the current maximum m": larger, or a NaN against a number. */
static int beats(double v, double m)
{
    if (isnan(v))
        return !isnan(m);
    return v > m;
}

/* Max and argmax over the box [ds,de) x [hs,he) x [ws,we) of plane p,
 * scanning d, then h, then w in ascending order and replacing the running
 * maximum only when a later element beats it (so the first occurrence of
 * the maximum is kept). Writes the winning element's bytes to y[o] and its
 * in-plane offset to idx[o]. */
static void reduce_window(int dtype, const void* x, void* y, int64_t* idx,
                          int64_t p, int64_t H, int64_t W, int64_t vol, int64_t o,
                          int64_t ds, int64_t de, int64_t hs, int64_t he,
                          int64_t ws, int64_t we)
{
    int es = elem_size(dtype);
    int64_t best = -1;
    double m = 0.0;
    int64_t d, h, w;
    for (d = ds; d < de; d++)
        for (h = hs; h < he; h++)
            for (w = ws; w < we; w++) {
                int64_t off = (d * H + h) * W + w;
                double v = load_value(dtype, x, p * vol + off);
                if (best < 0 || beats(v, m)) {
                    m = v;
                    best = off;
                }
            }
    memcpy((char*)y + o * es, (const char*)x + (p * vol + best) * es, (size_t)es);
    idx[o] = best;
}

/* Fixed-window forward ([MPF]): y[p,od,oh,ow] = max over
 * d in [od*sd, od*sd+kd), h in [oh*sh, oh*sh+kh), w in [ow*sw, ow*sw+kw). */
int oracle_maxpool3d_fwd(int dtype, const void* x, void* y, int64_t* idx,
                         int64_t P, int64_t D, int64_t H, int64_t W,
                         int64_t kd, int64_t kh, int64_t kw,
                         int64_t sd, int64_t sh, int64_t sw)
{
    int64_t OD = oracle_fixed_out_size(D, kd, sd);
    int64_t OH = oracle_fixed_out_size(H, kh, sh);
    int64_t OW = oracle_fixed_out_size(W, kw, sw);
    int64_t vol = D * H * W, p, od, oh, ow, o = 0;
    if (elem_size(dtype) == 0)
        return OR_ERR_DTYPE;
    if (P < 0 || OD < 1 || OH < 1 || OW < 1)
        return OR_ERR_SHAPE;
    for (p = 0; p < P; p++)
        for (od = 0; od < OD; od++)
            for (oh = 0; oh < OH; oh++)
                for (ow = 0; ow < OW; ow++) {
                    int64_t ds, de, hs, he, ws, we;
                    oracle_fixed_window(od, kd, sd, &ds, &de);
                    oracle_fixed_window(oh, kh, sh, &hs, &he);
                    oracle_fixed_window(ow, kw, sw, &ws, &we);
                    reduce_window(dtype, x, y, idx, p, H, W, vol, o, ds, de, hs, he, ws, we);
                    o++;
                }
    return OR_OK;
}

/* Adaptive-window forward: the same max/argmax over the adaptive windows. */
int oracle_adaptive_maxpool3d_fwd(int dtype, const void* x, void* y, int64_t* idx,
                                  int64_t P, int64_t D, int64_t H, int64_t W,
                                  int64_t OD, int64_t OH, int64_t OW)
{
    int64_t vol = D * H * W, p, od, oh, ow, o = 0;
    if (elem_size(dtype) == 0)
        return OR_ERR_DTYPE;
    if (P < 0 || D < 1 || H < 1 || W < 1 || OD < 1 || OH < 1 || OW < 1)
        return OR_ERR_SHAPE;
    for (p = 0; p < P; p++)
        for (od = 0; od < OD; od++)
            for (oh = 0; oh < OH; oh++)
                for (ow = 0; ow < OW; ow++) {
                    int64_t ds, de, hs, he, ws, we;
                    oracle_adaptive_window(od, D, OD, &ds, &de);
                    oracle_adaptive_window(oh, H, OH, &hs, &he);
                    oracle_adaptive_window(ow, W, OW, &ws, &we);
                    reduce_window(dtype, x, y, idx, p, H, W, vol, o, ds, de, hs, he, ws, we);
                    o++;
                }
    return OR_OK;
}

/* ------------------------------------------------------------------ */
/* Padding, dilation and ceil-mode output sizes: the fixed-window forward */
/* beyond [MPF]'s "no padding" constraint (the usual max_pool3d surface). */
/* ------------------------------------------------------------------ */

/* Output length along one axis with padding p on both sides, dilation dl
 * and ceil mode, following the usual max_pool3d definition (the pages fix
 * only the unpadded case). The window of output o takes the positions
 * o*S - p + k*dl, k = 0 .. K-1, that lie inside [0, I); its span is
 * e = dl*(K-1) + 1. O = floor((I + 2p - e) / S) + 1, or
 * floor((I + 2p - e + S - 1) / S) + 1 in ceil mode, where a last window starting
 * at or past I + p (wholly in the right padding) is dropped. Returns 0 for
 * invalid arguments: K, S or dl < 1, p < 0, p more than half the kernel
 * size (2p > K), or no output. */
int64_t oracle_ex_out_size(int64_t I, int64_t K, int64_t S, int64_t p, int64_t dl, int ceil_mode)
{
    int64_t e, num, O;
    if (I < 1 || K < 1 || S < 1 || dl < 1 || p < 0)
        return 0;
    if (2 * p > K)
        return 0;
    e = dl * (K - 1) + 1;
    num = I + 2 * p - e;
    if (ceil_mode)
        num += S - 1;
    O = (num >= 0 ? num / S : -((-num + S - 1) / S)) + 1;   /* floor division */
    if (ceil_mode && (O - 1) * S >= I + p)
        O--;
    return O < 1 ? 0 : O;
}

/* Forward with padding and dilation: y[p,od,oh,ow] = max over the window
 * positions (d, h, w) = (od*sd - pd + a*dd, oh*sh - ph + b*dh,
 * ow*sw - pw + c*dw), a < kd, b < kh, c < kw, that lie inside the input,
 * scanned in ascending a, b, c (so ascending d, h, w; padding is never
 * chosen). A window with no position inside the input makes the geometry
 * invalid (OR_ERR_SHAPE). */
int oracle_maxpool3d_fwd_ex(int dtype, const void* x, void* y, int64_t* idx,
                            int64_t P, int64_t D, int64_t H, int64_t W,
                            int64_t kd, int64_t kh, int64_t kw,
                            int64_t sd, int64_t sh, int64_t sw,
                            int64_t pd, int64_t ph, int64_t pw,
                            int64_t dd, int64_t dh, int64_t dw, int ceil_mode)
{
    int64_t OD = oracle_ex_out_size(D, kd, sd, pd, dd, ceil_mode);
    int64_t OH = oracle_ex_out_size(H, kh, sh, ph, dh, ceil_mode);
    int64_t OW = oracle_ex_out_size(W, kw, sw, pw, dw, ceil_mode);
    int64_t vol = D * H * W, p, od, oh, ow, o = 0;
    int es = elem_size(dtype);
    if (es == 0)
        return OR_ERR_DTYPE;
    if (P < 0 || OD < 1 || OH < 1 || OW < 1)
        return OR_ERR_SHAPE;
    for (p = 0; p < P; p++)
        for (od = 0; od < OD; od++)
            for (oh = 0; oh < OH; oh++)
                for (ow = 0; ow < OW; ow++) {
                    int64_t best = -1, a, b, c;
                    double m = 0.0;
                    for (a = 0; a < kd; a++) {
                        int64_t d = od * sd - pd + a * dd;
                        if (d < 0 || d >= D)
                            continue;
                        for (b = 0; b < kh; b++) {
                            int64_t h = oh * sh - ph + b * dh;
                            if (h < 0 || h >= H)
                                continue;
                            for (c = 0; c < kw; c++) {
                                int64_t w = ow * sw - pw + c * dw;
                                int64_t off;
                                double v;
                                if (w < 0 || w >= W)
                                    continue;
                                off = (d * H + h) * W + w;
                                v = load_value(dtype, x, p * vol + off);
                                if (best < 0 || beats(v, m)) {
                                    m = v;
                                    best = off;
                                }
                            }
                        }
                    }
                    if (best < 0)
                        return OR_ERR_SHAPE;
                    memcpy((char*)y + o * es, (const char*)x + es * (p * vol + best), (size_t)es);
                    idx[o] = best;
                    o++;
                }
    return OR_OK;
}

/* ------------------------------------------------------------------ */
/* Backward ([AMPB] Summary)                                            */
/* ------------------------------------------------------------------ */

/* grad_in[p, j] = sum over outputs o of plane p with idx[p, o] == j of
 * grad_out[p, o], summed in ascending o (that is, ascending (od, oh, ow))
 * in binary32, first term as the initial value, rounded once to the type;
 * +0 where no output selects j. in_vol = D*H*W, out_vol = OD*OH*OW.
 * The window geometry does not enter: the routing is fixed by idx alone. */
int oracle_maxpool3d_bwd(int dtype, const void* g, const int64_t* idx, void* gin,
                         int64_t P, int64_t in_vol, int64_t out_vol)
{
    float* acc;
    unsigned char* seen;
    int64_t p, o, j;
    if (elem_size(dtype) == 0)
        return OR_ERR_DTYPE;
    if (P < 0 || in_vol < 1 || out_vol < 1)
        return OR_ERR_SHAPE;
    acc = (float*)malloc((size_t)in_vol * sizeof(float));
    seen = (unsigned char*)malloc((size_t)in_vol);
    if (!acc || !seen) {
        free(acc);
        free(seen);
        return OR_ERR_NOMEM;
    }
    for (p = 0; p < P; p++) {
        memset(seen, 0, (size_t)in_vol);
        for (o = 0; o < out_vol; o++) {
            int64_t target = idx[p * out_vol + o];
            float gv = load_f32(dtype, g, p * out_vol + o);
            if (target < 0 || target >= in_vol) {
                free(acc);
                free(seen);
                return OR_ERR_INDEX;
            }
            if (!seen[target]) {
                acc[target] = gv;
                seen[target] = 1;
            } else {
                acc[target] = acc[target] + gv;   /* binary32 add */
            }
        }
        for (j = 0; j < in_vol; j++)
            store_rounded(dtype, gin, p * in_vol + j, seen[j] ? acc[j] : 0.0f);
    }
    free(acc);
    free(seen);
    return OR_OK;
}
