/*
 * CPU oracle of the reduced-vocabulary draft head. TEST INFRASTRUCTURE ONLY:
 * only the tests, the smoke check and the benchmark's CPU baseline load it.
 * It shares no code, header, table or constant with the CUDA library.
 *
 * Plain, slow, single-threaded C11. Decisions that produce integer codes are
 * taken in fp32, as the pages' PyTorch code does (`w.float()`); everything
 * else (dequantised weights, GEMV, logits) is computed in fp64.
 *
 * Sources, by page title and section:
 *  [Q38]  "q38_draft.py" (Qwen3.8-Flash-Next MTP drafter patch), functions
 *         load_draft_model (keep mask -> dh_idx, padding to N % 64, row gather),
 *         get_top_tokens (argmax over kept rows, mapped through dh_idx) and
 *         compute_logits (-inf row, index_copy_ of the kept logits).
 *  [FP8]  "FP8 MTP draft stack for vLLM - +6.6% decode on modelopt NVFP4
 *         Qwen3.5-family checkpoints", function _fp8_convert_draft_head
 *         (per-tensor E4M3 head), _Fp8DraftHeadMethod.apply (per-token dynamic
 *         E4M3 activations, scaled matmul) and Qwen3_5MTP.compute_logits.
 *  [H98K] "Qwen3.8-Flash-Next-ABLITERATED - MTP drafter, NVFP4 experts + 98K FP8
 *         head", section "How it was built": NVFP4 = global scale amax/(6*448),
 *         E4M3 block scales per 16 elements, e2m1 round-to-nearest-even.
 *  [SPARK] "autotrust/Qwen3.8-27B-NVFP4-DGX-SPARK", section "Repository layout":
 *         a 248,320-entry keep mask with 64,026 kept ids.
 *
 * Readings taken where the pages are silent (each is also a parity-unpinned
 * choice of operation order, see the header of or_nvfp4_quantize):
 *  - an empty keep mask is an error (the pages' idx[:1] would be empty);
 *  - the NVFP4 amax is clamped below at 1e-12 as the FP8 head's amax is;
 *  - block scale t = bamax / fp32(6*g); element x = w / fp32(dec(s)*g);
 *  - a block whose decoded scale is 0 encodes every element as a signed zero;
 *  - codes are packed two per byte, element 2i in the low nibble;
 *  - the per-token activation scale is amax_m / 448 with amax_m clamped below
 *    at 1e-12 and codes E4M3_RNE(clamp(h / s, +-448)), the head's own recipe
 *    applied per row (the page calls a library quantiser whose code is not on
 *    the pages).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_ERR_ARG 1
#define OR_ERR_SHAPE 2

/* ------------------------------------------------------------------------ */
/* Number formats                                                           */
/* ------------------------------------------------------------------------ */

/* BF16 bits -> float (exact: BF16 is the upper half of an IEEE single). */
static float bf16_value(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* E2M1 (FP4) value of a 4-bit code: bit 3 sign, bits 2..1 exponent with bias 1,
 * bit 0 mantissa; exponent field 0 is subnormal (0 or 0.5). [H98K] */
double or_e2m1_decode(int code)
{
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

/* E4M3 ("fn": no infinities) value of a byte: bit 7 sign, bits 6..3 exponent
 * with bias 7, bits 2..0 mantissa; exponent field 0 is subnormal (m * 2^-9);
 * 0x7F / 0xFF are NaN. Largest finite value 448. [H98K], [FP8] */
double or_e4m3_decode(int byte)
{
    int s = (byte >> 7) & 1, e = (byte >> 3) & 15, m = byte & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    v = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* Nearest E2M1 code to x, ties to the code with an even mantissa bit
 * (round-to-nearest-even), magnitudes beyond 6 clamp to 6. The sign bit
 * follows the sign of x, so a negative value that rounds to zero gives 0x8.
 * Written as a search over the eight magnitudes. [H98K] */
int or_e2m1_encode(float x)
{
    static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    double a = fabs((double)x);
    int sign = signbit(x) ? 8 : 0;
    int best = 0, c;
    double bd = a;
    if (a >= 6.0)
        return sign | 7;
    for (c = 1; c < 8; c++) {
        double d = fabs(a - mag[c]);
        if (d < bd || (d == bd && (c & 1) == 0)) {
            best = c;
            bd = d;
        }
    }
    return sign | best;
}

/* Nearest E4M3 byte to t, ties to even mantissa, saturating to +-448
 * (values beyond 448 give 448). NaN gives 0x7F. [FP8] (`.to(float8_e4m3fn)`
 * after a clamp to +-448), [H98K] (E4M3 block scales). */
int or_e4m3_encode(float t)
{
    int sign = signbit(t) ? 0x80 : 0;
    double a = fabs((double)t), q, n, v;
    int e, E;
    if (isnan(t))
        return 0x7F;
    if (a == 0.0)
        return sign;
    (void)frexp(a, &e); /* a = f * 2^e, f in [0.5, 1) */
    E = e - 1;          /* 2^E <= a < 2^(E+1) */
    if (E < -6)
        E = -6;         /* below the smallest normal the spacing stays 2^-9 */
    q = ldexp(1.0, E - 3);
    n = nearbyint(a / q); /* default rounding mode: nearest, ties to even */
    v = n * q;
    if (v > 448.0)
        v = 448.0;
    if (v < ldexp(1.0, -6))
        return sign | (int)(v / ldexp(1.0, -9)); /* subnormal (or 0) */
    (void)frexp(v, &e);
    E = e - 1;
    return sign | ((E + 7) << 3) | (int)((v / ldexp(1.0, E) - 1.0) * 8.0);
}

/* ------------------------------------------------------------------------ */
/* Head build: index, NVFP4 and FP8 quantisation                            */
/* ------------------------------------------------------------------------ */

/* dh_idx from a keep mask [Q38 load_draft_model]: the kept ids in ascending
 * order (keep.nonzero()), then pad = (-n) mod 64 copies of the first kept id so
 * that N % 64 == 0. Writes N ids to idx (cap entries available). */
int or_build_index(const uint8_t *keep, int V, int32_t *idx, int cap,
                   int *n_kept, int *N)
{
    int n = 0, v, pad, i;
    if (!keep || !idx || !n_kept || !N || V <= 0)
        return OR_ERR_ARG;
    for (v = 0; v < V; v++)
        if (keep[v]) {
            if (n >= cap)
                return OR_ERR_SHAPE;
            idx[n++] = v;
        }
    if (n == 0)
        return OR_ERR_ARG;
    pad = (64 - n % 64) % 64;
    if (n + pad > cap)
        return OR_ERR_SHAPE;
    for (i = 0; i < pad; i++)
        idx[n + i] = idx[0];
    *n_kept = n;
    *N = n + pad;
    return OR_OK;
}

/* Largest |W[idx[n], k]| over the gathered rows (exact, as float). */
static float gathered_amax(const uint16_t *W, int K, const int32_t *idx, int N)
{
    float amax = 0.0f;
    int n, k;
    for (n = 0; n < N; n++)
        for (k = 0; k < K; k++) {
            float a = fabsf(bf16_value(W[(size_t)idx[n] * K + k]));
            if (a > amax)
                amax = a;
        }
    return amax;
}

static int check_gather(int V, int K, const int32_t *idx, int N)
{
    int n;
    if (V <= 0 || K <= 0 || N <= 0 || K % 16 != 0)
        return OR_ERR_SHAPE;
    for (n = 0; n < N; n++)
        if (idx[n] < 0 || idx[n] >= V)
            return OR_ERR_ARG;
    return OR_OK;
}

/* NVFP4 quantisation of the gathered rows W[idx[n], :] [H98K "How it was
 * built"; Q38 load_draft_model: make_linear(W[idx].contiguous(), "marlin")].
 *   g   = fp32(max(amax, 1e-12) / 2688)            2688 = 6 * 448
 *   per block of 16 consecutive k in a row:
 *   t   = fp32(bamax / fp32(6 * g)),  s = E4M3_RNE_sat(t)
 *   d   = fp32(dec(s) * g)
 *   x   = fp32(w / d) clamped to [-6, 6],  c = E2M1_RNE(x)   (d == 0: signed 0)
 * Output: q [N][K/2] (code 2i in the low nibble of byte i), sf [N][K/16], g.
 * Parity unpinned: the pages state the recipe, not this operation order. */
int or_nvfp4_quantize(const uint16_t *W, int V, int K, const int32_t *idx, int N,
                      uint8_t *q, uint8_t *sf, float *g_out)
{
    float amax, g, den;
    int n, b, k, st;
    if (!W || !idx || !q || !sf || !g_out)
        return OR_ERR_ARG;
    if ((st = check_gather(V, K, idx, N)) != OR_OK)
        return st;
    amax = gathered_amax(W, K, idx, N);
    if (amax < 1e-12f)
        amax = 1e-12f;
    g = amax / 2688.0f;
    den = 6.0f * g;
    for (n = 0; n < N; n++) {
        const uint16_t *row = W + (size_t)idx[n] * K;
        for (b = 0; b < K / 16; b++) {
            float bamax = 0.0f, d;
            int s, codes[16];
            for (k = 0; k < 16; k++) {
                float a = fabsf(bf16_value(row[16 * b + k]));
                if (a > bamax)
                    bamax = a;
            }
            s = or_e4m3_encode(bamax / den);
            d = (float)or_e4m3_decode(s) * g;
            for (k = 0; k < 16; k++) {
                float w = bf16_value(row[16 * b + k]);
                if (d == 0.0f) {
                    codes[k] = signbit(w) ? 8 : 0;
                } else {
                    float x = w / d;
                    if (x > 6.0f)
                        x = 6.0f;
                    if (x < -6.0f)
                        x = -6.0f;
                    codes[k] = or_e2m1_encode(x);
                }
            }
            sf[(size_t)n * (K / 16) + b] = (uint8_t)s;
            for (k = 0; k < 16; k += 2)
                q[(size_t)n * (K / 2) + 8 * b + k / 2] =
                    (uint8_t)(codes[k] | (codes[k + 1] << 4));
        }
    }
    *g_out = g;
    return OR_OK;
}

/* Per-tensor FP8 E4M3 quantisation of the gathered rows [FP8
 * _fp8_convert_draft_head]: amax = max|w| clamped below at 1e-12,
 * scale = fp32(amax / 448), q = E4M3_RNE(clamp(fp32(w / scale), +-448)).
 * Stored row-major q [N][K] (the page keeps the transpose; same bytes). */
int or_fp8_quantize(const uint16_t *W, int V, int K, const int32_t *idx, int N,
                    uint8_t *q, float *scale_out)
{
    float amax, scale;
    int n, k, st;
    if (!W || !idx || !q || !scale_out)
        return OR_ERR_ARG;
    if ((st = check_gather(V, K, idx, N)) != OR_OK)
        return st;
    amax = gathered_amax(W, K, idx, N);
    if (amax < 1e-12f)
        amax = 1e-12f;
    scale = amax / 448.0f;
    for (n = 0; n < N; n++)
        for (k = 0; k < K; k++) {
            float x = bf16_value(W[(size_t)idx[n] * K + k]) / scale;
            if (x > 448.0f)
                x = 448.0f;
            if (x < -448.0f)
                x = -448.0f;
            q[(size_t)n * K + k] = (uint8_t)or_e4m3_encode(x);
        }
    *scale_out = scale;
    return OR_OK;
}

/* Dynamic per-token FP8 quantisation of the draft hidden states, the
 * activation half of the W8A8 head [FP8 _Fp8DraftHeadMethod.apply:
 * scaled_fp8_quant(x, use_per_token_if_dynamic=True) before the scaled
 * matmul]. Per row m: amax_m = max_k |h[m, k]| clamped below at 1e-12 (as the
 * head's own amax is), s_m = fp32(amax_m / 448),
 * qx[m, k] = E4M3_RNE(clamp(fp32(h[m, k] / s_m), +-448)). Same recipe as the
 * head's per-tensor quantisation, one scale per row. */
int or_fp8_act_quantize(const uint16_t *h, int M, int K, uint8_t *qx, float *sx)
{
    int m, k;
    if (!h || !qx || !sx || M <= 0 || K <= 0)
        return OR_ERR_ARG;
    for (m = 0; m < M; m++) {
        float amax = 0.0f, s;
        for (k = 0; k < K; k++) {
            float a = fabsf(bf16_value(h[(size_t)m * K + k]));
            if (a > amax)
                amax = a;
        }
        if (amax < 1e-12f)
            amax = 1e-12f;
        s = amax / 448.0f;
        for (k = 0; k < K; k++) {
            float x = bf16_value(h[(size_t)m * K + k]) / s;
            if (x > 448.0f)
                x = 448.0f;
            if (x < -448.0f)
                x = -448.0f;
            qx[(size_t)m * K + k] = (uint8_t)or_e4m3_encode(x);
        }
        sx[m] = s;
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Draft step: GEMV, argmax, id map, logits scatter                         */
/* ------------------------------------------------------------------------ */

/* W8A8 FP8 head [FP8 _Fp8DraftHeadMethod.apply: cutlass_scaled_mm(qx, W, sx,
 * weight_scale)]: y[m, n] = scale * sx[m] * sum_k dec(q[n, k]) * dec(qx[m, k]),
 * in fp64 (every product of two E4M3 values is exact), and A[m, n] the same
 * sum of |products| (tolerance scale). q row-major [N][K], qx [M][K] as
 * written by or_fp8_act_quantize. A may be NULL. */
int or_gemv_w8a8(const uint8_t *q, float scale, int N, int K, const uint8_t *qx,
                 const float *sx, int M, double *y, double *A)
{
    double e4[256];
    int m, n, k;
    if (!q || !qx || !sx || !y || N <= 0 || K <= 0 || M <= 0)
        return OR_ERR_ARG;
    for (k = 0; k < 256; k++)
        e4[k] = or_e4m3_decode(k);
    for (n = 0; n < N; n++)
        for (m = 0; m < M; m++) {
            const double ws = (double)scale * (double)sx[m];
            double s = 0.0, a = 0.0;
            for (k = 0; k < K; k++) {
                double p = e4[q[(size_t)n * K + k]] * e4[qx[(size_t)m * K + k]];
                s += p;
                a += fabs(p);
            }
            y[(size_t)m * N + n] = s * ws;
            if (A)
                A[(size_t)m * N + n] = a * fabs(ws);
        }
    return OR_OK;
}

/* y[m, n] = sum_k w'[n, k] * h[m, k] in fp64, and A[m, n] = sum_k |w'[n, k] h[m, k]|
 * (the scale of the logits tolerance) [Q38 get_top_tokens / compute_logits:
 * draft_head(h)]. fmt: 1 = NVFP4 (q, sf, scale = g), 2 = FP8 (q, scale),
 * 3 = BF16 (q holds the BF16 head, scale unused). Each head row is first
 * dequantised into w'[0..K) (exact in fp64), then dotted with every h row.
 * Rows are those of the head as stored (N of them). y and A are [M][N];
 * A may be NULL. */
int or_gemv(int fmt, const uint8_t *q, const uint8_t *sf, float scale, int N, int K,
            const uint16_t *h, int M, double *y, double *A)
{
    double e2[16], e4[256], *w, *hv;
    int m, n, k;
    if (!q || !h || !y || N <= 0 || K <= 0 || M <= 0 || K % 16 != 0)
        return OR_ERR_ARG;
    if ((fmt == 1 && !sf) || fmt < 1 || fmt > 3)
        return OR_ERR_ARG;
    for (k = 0; k < 16; k++)
        e2[k] = or_e2m1_decode(k);
    for (k = 0; k < 256; k++)
        e4[k] = or_e4m3_decode(k);
    w = (double *)malloc(sizeof(double) * (size_t)K);
    hv = (double *)malloc(sizeof(double) * (size_t)K * (size_t)M);
    if (!w || !hv) {
        free(w);
        free(hv);
        return OR_ERR_ARG;
    }
    for (m = 0; m < M; m++)
        for (k = 0; k < K; k++)
            hv[(size_t)m * K + k] = bf16_value(h[(size_t)m * K + k]);
    for (n = 0; n < N; n++) {
        for (k = 0; k < K; k++) {
            if (fmt == 1) {
                int byte = q[(size_t)n * (K / 2) + k / 2];
                int code = (k & 1) ? (byte >> 4) : (byte & 15);
                w[k] = e2[code] * e4[sf[(size_t)n * (K / 16) + k / 16]] * (double)scale;
            } else if (fmt == 2) {
                w[k] = e4[q[(size_t)n * K + k]] * (double)scale;
            } else {
                w[k] = bf16_value(((const uint16_t *)q)[(size_t)n * K + k]);
            }
        }
        for (m = 0; m < M; m++) {
            const double *x = hv + (size_t)m * K;
            double s = 0.0, a = 0.0;
            for (k = 0; k < K; k++) {
                double p = w[k] * x[k];
                s += p;
                a += fabs(p);
            }
            y[(size_t)m * N + n] = s;
            if (A)
                A[(size_t)m * N + n] = a;
        }
    }
    free(w);
    free(hv);
    return OR_OK;
}

/* First index of the maximum of y[0..n) (torch.argmax semantics on finite
 * values: the lowest index wins a tie). */
int or_argmax(const double *y, int n)
{
    int i, best = 0;
    for (i = 1; i < n; i++)
        if (y[i] > y[best])
            best = i;
    return best;
}

/* get_top_tokens [Q38]: per draft m, r* = argmax over the N head rows of
 * y[m, :], then ids[m] = idx[r*] (idx = NULL: the row is the id, as for the
 * full-vocabulary head). rows[m] = r* if rows is not NULL. */
int or_top_tokens(const double *y, int M, int N, const int32_t *idx,
                  int32_t *ids, int32_t *rows)
{
    int m;
    if (!y || !ids || M <= 0 || N <= 0)
        return OR_ERR_ARG;
    for (m = 0; m < M; m++) {
        int r = or_argmax(y + (size_t)m * N, N);
        ids[m] = idx ? idx[r] : r;
        if (rows)
            rows[m] = r;
    }
    return OR_OK;
}

/* compute_logits [Q38 compute_logits; FP8 page Qwen3_5MTP.compute_logits]:
 * out[m, :] = -inf over the whole target vocabulary V, then
 * out[m, idx[n]] = fp32(y[m, n]) for the kept rows n < n_kept (the padding
 * rows repeat idx[0] and carry row 0's values, so they are not written). */
int or_scatter_logits(const double *y, int M, int N, const int32_t *idx, int n_kept,
                      int V, float *out)
{
    int m, n, v;
    if (!y || !idx || !out || M <= 0 || n_kept <= 0 || n_kept > N || V <= 0)
        return OR_ERR_ARG;
    for (n = 0; n < n_kept; n++)
        if (idx[n] < 0 || idx[n] >= V)
            return OR_ERR_ARG;
    for (m = 0; m < M; m++) {
        for (v = 0; v < V; v++)
            out[(size_t)m * V + v] = -INFINITY;
        for (n = 0; n < n_kept; n++)
            out[(size_t)m * V + idx[n]] = (float)y[(size_t)m * N + n];
    }
    return OR_OK;
}
