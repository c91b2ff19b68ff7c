/*
 * Plain CPU oracle for the Hadamard route: rotate each 32-block of activations
 * with a 32-point Walsh-Hadamard transform, round it to 4-bit (or 8-bit) codes
 * with one fp32 scale, and take block-scaled integer dot products against
 * Q4_0 weights that were rotated the same way.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the bench load this file's library.  It shares no code,
 * header, constant or helper with the CUDA path, and nothing in the product
 * path calls it.
 *
 * Sources (page titles and sections of the pages the method comes from):
 *   [Rot]  "509 tokens a second of prompt: the Hadamard route ships", section
 *          "The rotation": blocks of 32 values share one scale; each block is
 *          rotated by a 32-point Walsh-Hadamard transform before rounding; the
 *          weights are rotated the same way offline, and x.w = (Hx).(Hw)
 *          because the transform is orthogonal.
 *   [PP]   "Qwen3.8-27B at 45.7 tok/s ...", section "Prompt processing: 4-bit
 *          activations, rotated first": same facts; the rotation runs inside
 *          the activation quantizer; the exact route uses 8-bit activations.
 *   [Q40]  Both posts, section "Why prompts are a matrix-unit problem" /
 *          "Prompt processing ...": a Q4_0 code q means q - 8.
 *
 * Readings where the pages leave a step open (each one is listed with its
 * reason in the design notes):
 *   - The transform is the Sylvester-ordered Hadamard matrix scaled by the
 *     fp32 number nearest to 1/sqrt(32); it is evaluated as the in-place
 *     butterfly with strides 1, 2, 4, 8, 16 in that order, each add/sub
 *     rounded to fp32, then one fp32 multiply by that constant.
 *   - Activation scale d = amax / 7 (or / 127) in fp32; codes are the
 *     nearest-even integers of y * (1/d), clamped to [-8, 7] (or [-127, 127]).
 *     An all-zero block has d = 0 and all codes 0.  Where 1/d is not finite
 *     (a block of subnormal size) or the rotation overflowed, the code is
 *     y / d by an IEEE divide instead (zeros stay 0), inf / inf read as its
 *     limit +-qmax; weights likewise.
 *   - 4-bit codes are packed in the Q4_0 nibble order: byte j of a block holds
 *     element j in its low nibble and element j + 16 in its high nibble.
 *   - Weight codes follow the ordinary Q4_0 rule without an importance matrix:
 *     the signed value of largest magnitude (first one on ties) maps to -8,
 *     d = max / -8, code = min(15, trunc(y * (1/d) + 8.5)), and d is stored
 *     as fp16 rounded to nearest even.
 *   - The fp32 result accumulates the blocks in order b = 0, 1, ... with
 *     acc = fma(fp32(d_w * d_x), S_b, acc), starting from +0.
 *
 * Parity pins: every function here is pinned by a test that checks it against
 * something other than itself (closed forms, a library Hadamard matrix,
 * brute force, exhaustive decode tables, hand-derived golden blocks).
 *
 * Build: plain C99, -O2 -ffp-contract=off, no fast-math, single threaded.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Basic conversions                                                         */
/* ------------------------------------------------------------------------ */

/* bf16 -> fp32 is exact: the bf16 bits are the top half of the fp32 bits. */
void o_bf16_to_f32(const uint16_t *in, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) {
        uint32_t u = ((uint32_t)in[i]) << 16;
        memcpy(&out[i], &u, 4);
    }
}

/* fp32 -> fp16 with round-to-nearest-even (the compiler's conversion). */
static uint16_t f32_to_f16_bits(float f)
{
    _Float16 h = (_Float16)f;
    uint16_t b;
    memcpy(&b, &h, 2);
    return b;
}

static float f16_bits_to_f32(uint16_t b)
{
    _Float16 h;
    memcpy(&h, &b, 2);
    return (float)h;
}

void o_f32_to_f16(const float *in, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_f16_bits(in[i]);
}

void o_f16_to_f32(const uint16_t *in, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = f16_bits_to_f32(in[i]);
}

/* ------------------------------------------------------------------------ */
/* The 32-point Walsh-Hadamard rotation [Rot], [PP]                          */
/* ------------------------------------------------------------------------ */

/* fp32 nearest to 1/sqrt(32); the tests pin it against an exact value. */
static float h32_scale_f32(void) { return (float)(1.0 / sqrt(32.0)); }

/* In-place butterfly: for h = 1, 2, 4, 8, 16, every pair (i, i + h) with
 * bit h of i clear becomes (a + c, a - c).  Then one multiply by 1/sqrt(32). */
static void fwht32_f32(float v[32])
{
    for (int h = 1; h < 32; h <<= 1) {
        for (int i = 0; i < 32; ++i) {
            if ((i & h) == 0) {
                float a = v[i];
                float c = v[i + h];
                v[i] = a + c;
                v[i + h] = a - c;
            }
        }
    }
    const float s = h32_scale_f32();
    for (int i = 0; i < 32; ++i) v[i] = v[i] * s;
}

/* The same butterfly in fp64, used for the invariance check x.w = (Hx).(Hw). */
static void fwht32_f64(double v[32])
{
    for (int h = 1; h < 32; h <<= 1) {
        for (int i = 0; i < 32; ++i) {
            if ((i & h) == 0) {
                double a = v[i];
                double c = v[i + h];
                v[i] = a + c;
                v[i + h] = a - c;
            }
        }
    }
    const double s = 1.0 / sqrt(32.0);
    for (int i = 0; i < 32; ++i) v[i] = v[i] * s;
}

/* ------------------------------------------------------------------------ */
/* Larger rotations, 64 and 128 points, with the scales still per 32-block   */
/* ("Qwen3.8-27B at 45.7 tok/s ...", section "What's next": a larger         */
/* rotation is the next step).  Same Sylvester transform and stage order:    */
/* strides 1, 2, ..., n/2, then one multiply by the fp32 nearest 1/sqrt(n).  */
/* ------------------------------------------------------------------------ */

static float rot_scale_f32(int n) { return (float)(1.0 / sqrt((double)n)); }

static void fwht_n_f32(float *v, int n)
{
    for (int h = 1; h < n; h <<= 1) {
        for (int i = 0; i < n; ++i) {
            if ((i & h) == 0) {
                float a = v[i];
                float c = v[i + h];
                v[i] = a + c;
                v[i + h] = a - c;
            }
        }
    }
    const float s = rot_scale_f32(n);
    for (int i = 0; i < n; ++i) v[i] = v[i] * s;
}

static void fwht_n_f64(double *v, int n)
{
    for (int h = 1; h < n; h <<= 1) {
        for (int i = 0; i < n; ++i) {
            if ((i & h) == 0) {
                double a = v[i];
                double c = v[i + h];
                v[i] = a + c;
                v[i + h] = a - c;
            }
        }
    }
    const double s = 1.0 / sqrt((double)n);
    for (int i = 0; i < n; ++i) v[i] = v[i] * s;
}

/* Rotate consecutive n-blocks (n = 32, 64 or 128); `count` values in all. */
void o_fwht_n_f32(const float *in, float *out, int64_t count, int n)
{
    for (int64_t b = 0; b + n <= count; b += n) {
        float v[128];
        memcpy(v, in + b, sizeof(float) * (size_t)n);
        fwht_n_f32(v, n);
        memcpy(out + b, v, sizeof(float) * (size_t)n);
    }
}

void o_fwht_n_f64(const double *in, double *out, int64_t count, int n)
{
    for (int64_t b = 0; b + n <= count; b += n) {
        double v[128];
        memcpy(v, in + b, sizeof(double) * (size_t)n);
        fwht_n_f64(v, n);
        memcpy(out + b, v, sizeof(double) * (size_t)n);
    }
}

float o_rot_scale(int n) { return rot_scale_f32(n); }

/* rotate argument of the quantizers: 0 = none, 1 or 32 = 32 points, 64, 128 */
static int rot_points(int rotate) { return rotate == 1 ? 32 : rotate; }

/* Rotate n consecutive 32-blocks. */
void o_fwht32_f32(const float *in, float *out, int64_t nblocks)
{
    for (int64_t b = 0; b < nblocks; ++b) {
        float v[32];
        memcpy(v, in + 32 * b, sizeof v);
        fwht32_f32(v);
        memcpy(out + 32 * b, v, sizeof v);
    }
}

void o_fwht32_f64(const double *in, double *out, int64_t nblocks)
{
    for (int64_t b = 0; b < nblocks; ++b) {
        double v[32];
        memcpy(v, in + 32 * b, sizeof v);
        fwht32_f64(v);
        memcpy(out + 32 * b, v, sizeof v);
    }
}

float o_h32_scale(void) { return h32_scale_f32(); }

/* ------------------------------------------------------------------------ */
/* Symmetric activation codes, one fp32 scale per 32-block [Rot], [PP]       */
/* ------------------------------------------------------------------------ */

/* y: one (rotated) block.  qmax = 7 (4-bit) or 127 (8-bit); qmin = -8 / -127. */
static void quantize_block_sym(const float y[32], int qmin, int qmax, int q[32], float *d_out)
{
    float amax = 0.0f;
    for (int i = 0; i < 32; ++i) {
        float a = fabsf(y[i]);
        if (a > amax) amax = a;
    }
    float d = amax / (float)qmax;
    float id = (d != 0.0f) ? 1.0f / d : 0.0f;
    /* A degenerate block: 1/d overflows (d below 2^-128, a block of subnormal
     * size) or the rotation itself overflowed (amax, and so d, infinite).
     * There the code is y / d by an IEEE divide, so exact zeros stay 0 and
     * the element of largest magnitude gets +-qmax; an infinite element of an
     * overflowed block (inf / inf) takes the limit of y / d, +-qmax. */
    int degenerate = isinf(id) || isinf(amax);
    for (int i = 0; i < 32; ++i) {
        float t;
        if (!degenerate) {
            t = y[i] * id;
        } else {
            t = y[i] / d;
            if (isnan(t)) t = copysignf((float)qmax, y[i]);
        }
        /* clamp first (max then min), then round to nearest even */
        t = fmaxf(t, (float)qmin);
        t = fminf(t, (float)qmax);
        q[i] = (int)rintf(t);
    }
    *d_out = d;
}

/* x: fp32 activations [M][K] row-major (bf16 inputs are widened first with
 * o_bf16_to_f32).  bits = 4: xq is [M][K/2] bytes in Q4_0 nibble order,
 * two's-complement nibbles.  bits = 8: xq is [M][K] int8.  xd is [M][K/32].
 * rotate = 0 skips the Walsh-Hadamard step (the unrotated 4-bit route); 1 or 32
 * rotates each 32-block; 64 or 128 rotates each 64- or 128-block (K a multiple
 * of it) and still takes one scale per 32-block of the rotated values. */
void o_quantize_act(const float *x, int64_t M, int64_t K, int bits, int rotate,
                    uint8_t *xq, float *xd)
{
    const int64_t nb = K / 32;
    const int qmax = (bits == 4) ? 7 : 127;
    const int qmin = (bits == 4) ? -8 : -127;
    const int n = rot_points(rotate);
    for (int64_t m = 0; m < M; ++m) {
        float row[128];
        for (int64_t b = 0; b < nb; ++b) {
            float v[32];
            if (n > 32) {
                /* the first block of each n-block rotates all n values */
                if ((32 * b) % n == 0) {
                    memcpy(row, x + m * K + 32 * b, sizeof(float) * (size_t)n);
                    fwht_n_f32(row, n);
                }
                memcpy(v, row + (32 * b) % n, sizeof v);
            } else {
                memcpy(v, x + m * K + 32 * b, sizeof v);
                if (n == 32) fwht32_f32(v);
            }
            int q[32];
            float d;
            quantize_block_sym(v, qmin, qmax, q, &d);
            xd[m * nb + b] = d;
            if (bits == 4) {
                uint8_t *dst = xq + m * (K / 2) + 16 * b;
                for (int j = 0; j < 16; ++j)
                    dst[j] = (uint8_t)((q[j] & 0xF) | ((q[j + 16] & 0xF) << 4));
            } else {
                int8_t *dst = (int8_t *)xq + m * K + 32 * b;
                for (int j = 0; j < 32; ++j) dst[j] = (int8_t)q[j];
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Q4_0 weights, rotated offline [Rot] "Making the file is part of the engine" */
/* ------------------------------------------------------------------------ */

static void q4_0_block(const float y[32], uint8_t qs[16], uint16_t *d16)
{
    float amax = 0.0f, mx = 0.0f;
    for (int i = 0; i < 32; ++i) {
        float a = fabsf(y[i]);
        if (a > amax) {
            amax = a;
            mx = y[i];
        }
    }
    float d = mx / -8.0f;
    float id = (d != 0.0f) ? 1.0f / d : 0.0f;
    /* degenerate blocks as for the activations: where 1/d overflows or the
     * rotation overflowed, y / d by an IEEE divide (a zero stays at code 8,
     * the signed maximum gets code 0); inf / inf takes its limit, -8 when y
     * has the sign of the signed maximum, else +8 */
    int degenerate = isinf(id) || isinf(amax);
    int c[32];
    for (int i = 0; i < 32; ++i) {
        /* two roundings, the product then the sum: -ffp-contract=off keeps
         * the compiler from fusing them */
        float u;
        if (!degenerate) {
            u = y[i] * id + 8.5f;
        } else {
            float t = y[i] / d;
            if (isnan(t)) t = ((signbit(y[i]) != 0) == (signbit(mx) != 0)) ? -8.0f : 8.0f;
            u = t + 8.5f;
        }
        u = fmaxf(u, 0.0f);
        u = fminf(u, 15.0f);
        c[i] = (int)u; /* truncation; u >= 0 here */
    }
    for (int j = 0; j < 16; ++j) qs[j] = (uint8_t)(c[j] | (c[j + 16] << 4));
    *d16 = f32_to_f16_bits(d);
}

/* w: fp32 [N][K] -> wq [N][K/2] (codes 0..15, Q4_0 nibble order),
 * wd [N][K/32] fp16 bits.  rotate = 0 gives plain Q4_0; 1/32, 64, 128 as for
 * the activations. */
void o_quantize_weights_q4_0(const float *w, int64_t N, int64_t K, int rotate,
                             uint8_t *wq, uint16_t *wd)
{
    const int64_t nb = K / 32;
    const int rn = rot_points(rotate);
    for (int64_t n = 0; n < N; ++n) {
        float row[128];
        for (int64_t b = 0; b < nb; ++b) {
            float v[32];
            if (rn > 32) {
                if ((32 * b) % rn == 0) {
                    memcpy(row, w + n * K + 32 * b, sizeof(float) * (size_t)rn);
                    fwht_n_f32(row, rn);
                }
                memcpy(v, row + (32 * b) % rn, sizeof v);
            } else {
                memcpy(v, w + n * K + 32 * b, sizeof v);
                if (rn == 32) fwht32_f32(v);
            }
            q4_0_block(v, wq + n * (K / 2) + 16 * b, wd + n * nb + b);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Decoding codes (plain definitions, not the bit-flip)                      */
/* ------------------------------------------------------------------------ */

/* element k of a row stored in Q4_0 nibble order */
static int nibble_at(const uint8_t *row, int64_t k)
{
    int64_t b = k / 32, j = k % 32;
    uint8_t byte = row[16 * b + (j & 15)];
    return (j < 16) ? (byte & 0xF) : (byte >> 4);
}

static int act4_value(const uint8_t *row, int64_t k)
{
    int u = nibble_at(row, k);
    return (u < 8) ? u : u - 16; /* two's complement */
}

static int w4_value(const uint8_t *row, int64_t k)
{
    return nibble_at(row, k) - 8; /* Q4_0: code q means q - 8 */
}

/* Exposed for the pins: decode whole rows to int8 values. */
void o_decode_act4(const uint8_t *xq, int64_t M, int64_t K, int8_t *out)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k) out[m * K + k] = (int8_t)act4_value(xq + m * (K / 2), k);
}

void o_decode_w4(const uint8_t *wq, int64_t N, int64_t K, int8_t *out)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) out[n * K + k] = (int8_t)w4_value(wq + n * (K / 2), k);
}

/* ------------------------------------------------------------------------ */
/* Block dot products and the scale epilogue                                 */
/* ------------------------------------------------------------------------ */

/* Exact integer sum of one 32-block, in int64. xbits = 4 or 8. */
static int64_t block_sum(const uint8_t *wrow, const uint8_t *xrow, int xbits, int64_t b)
{
    int64_t s = 0;
    for (int64_t j = 0; j < 32; ++j) {
        int64_t k = 32 * b + j;
        int64_t xv = (xbits == 4) ? act4_value(xrow, k) : ((const int8_t *)xrow)[k];
        s += xv * (int64_t)w4_value(wrow, k);
    }
    return s;
}

/* One output element: y32 in the fixed fp32 order, y64 in fp64, and
 * (optionally) the block sums. */
static void one_output(const uint8_t *wrow, const uint16_t *wdrow, const uint8_t *xrow,
                       const float *xdrow, int xbits, int64_t nb,
                       float *y32, double *y64, int64_t *S_out)
{
    float acc = 0.0f;
    double acc64 = 0.0;
    for (int64_t b = 0; b < nb; ++b) {
        int64_t S = block_sum(wrow, xrow, xbits, b);
        if (S_out) S_out[b] = S;
        float dw = f16_bits_to_f32(wdrow[b]);
        float dx = xdrow[b];
        float s = dw * dx;
        acc = fmaf(s, (float)S, acc);
        acc64 += (double)dw * (double)dx * (double)S;
    }
    *y32 = acc;
    *y64 = acc64;
}

static int64_t act_row_bytes(int64_t K, int xbits) { return (xbits == 4) ? K / 2 : K; }

/* Full GEMM: y[m][n] for all m < M, n < N.  S (nullable) is [M][N][K/32]. */
void o_gemm(const uint8_t *wq, const uint16_t *wd, const uint8_t *xq, const float *xd,
            int xbits, int64_t M, int64_t N, int64_t K,
            float *y32, double *y64, int64_t *S)
{
    const int64_t nb = K / 32, xrb = act_row_bytes(K, xbits);
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            one_output(wq + n * (K / 2), wd + n * nb, xq + m * xrb, xd + m * nb, xbits, nb,
                       &y32[m * N + n], &y64[m * N + n], S ? S + (m * N + n) * nb : 0);
}

/* Sampled GEMM: the outputs (m_idx[i], n_idx[i]) only.  S (nullable) is [P][K/32]. */
void o_gemm_sampled(const uint8_t *wq, const uint16_t *wd, const uint8_t *xq, const float *xd,
                    int xbits, int64_t K, int64_t P, const int64_t *m_idx, const int64_t *n_idx,
                    float *y32, double *y64, int64_t *S)
{
    const int64_t nb = K / 32, xrb = act_row_bytes(K, xbits);
    for (int64_t i = 0; i < P; ++i) {
        int64_t m = m_idx[i], n = n_idx[i];
        one_output(wq + n * (K / 2), wd + n * nb, xq + m * xrb, xd + m * nb, xbits, nb,
                   &y32[i], &y64[i], S ? S + i * nb : 0);
    }
}

/* Expert-batched GEMM, sampled: row r (grouped order) belongs to the expert e
 * with off[e] <= r < off[e+1] and reads activation row row_idx[r] (or r when
 * row_idx is null).  Weights wq [E][N][K/2], wd [E][N][K/32]. */
void o_gemm_experts_sampled(const uint8_t *wq, const uint16_t *wd, int64_t E,
                            const uint8_t *xq, const float *xd, const int32_t *row_idx,
                            const int32_t *expert_off, int64_t N, int64_t K,
                            int64_t P, const int64_t *r_idx, const int64_t *n_idx,
                            float *y32, double *y64, int64_t *S)
{
    const int64_t nb = K / 32;
    for (int64_t i = 0; i < P; ++i) {
        int64_t r = r_idx[i], n = n_idx[i];
        int64_t e = 0;
        while (e < E && !(expert_off[e] <= r && r < expert_off[e + 1])) ++e;
        if (e == E) { /* row outside every group: not computed */
            y32[i] = NAN;
            y64[i] = NAN;
            continue;
        }
        int64_t xr = row_idx ? row_idx[r] : r;
        one_output(wq + (e * N + n) * (K / 2), wd + (e * N + n) * nb, xq + xr * (K / 2),
                   xd + xr * nb, 4, nb, &y32[i], &y64[i], S ? S + i * nb : 0);
    }
}

/* ------------------------------------------------------------------------ */
/* Expert routing and the weighted combine around the expert-batched GEMM    */
/* ------------------------------------------------------------------------ */
/* [MoE] "Where the engine is going: HRX and the NPU", section "4-bit
 * activations reach the MoE experts": the route covers the expert matmuls of
 * a mixture-of-experts model.  The pages do not spell out the router around
 * them; the readings taken:
 *   - a token takes the k experts of largest logit (the softmax is monotonic,
 *     so these are its k most probable experts), ties to the lower expert id,
 *     listed by decreasing logit;
 *   - choice j weighs w_j = exp(l_j - l_max) / sum_i exp(l_i - l_max) over
 *     the k chosen logits, which is the full softmax's top-k probabilities
 *     renormalised to sum to 1; in fp32: one difference and one exp per
 *     choice, the sum taken in choice order from +0, one IEEE divide each;
 *   - rows are grouped by expert id, and within an expert by token;
 *   - the combine adds the k expert rows of a token in choice order,
 *     acc = fma(w_j, y_j, acc) from +0. */

/* Logits that are not finite (masked experts, a broken router) follow the
 * limits of the same rule: a NaN ranks below every number, -inf included
 * (NaNs among themselves by id); the unnormalised weight e_j of a choice is
 * exp(l_j - l_max) when the largest chosen logit l_max is finite (0 for a
 * chosen -inf or NaN), 1 for the choices equal to +inf (0 for the others)
 * when l_max = +inf, and 1 for every choice when l_max is -inf or NaN (all
 * logits masked: equal weights). */

/* does logit a (expert ia) rank before logit b (expert ib)? */
static int ranks_before(float a, int64_t ia, float b, int64_t ib)
{
    if (isnan(a) || isnan(b)) {
        if (isnan(a) && isnan(b)) return ia < ib;
        return isnan(b);
    }
    return a > b || (a == b && ia < ib);
}

static float unnormalised_weight(float l, float lmax)
{
    if (isfinite(lmax)) return isnan(l) ? 0.0f : expf(l - lmax);
    if (lmax > 0.0f) return (l == lmax) ? 1.0f : 0.0f; /* lmax = +inf */
    return 1.0f;                                         /* -inf or NaN */
}

/* logits [T][E] -> topk_id [T][k], topk_w [T][k], expert_off [E+1],
 * row_idx [T*k] (the token of grouped row r), row_of [T][k] (the grouped row
 * of choice j of token t). */
void o_moe_route(const float *logits, int64_t T, int64_t E, int64_t k, int32_t *topk_id,
                 float *topk_w, int32_t *expert_off, int32_t *row_idx, int32_t *row_of)
{
    for (int64_t t = 0; t < T; ++t) {
        const float *l = logits + t * E;
        int32_t *id = topk_id + t * k;
        for (int64_t j = 0; j < k; ++j) {
            int64_t best = -1;
            for (int64_t e = 0; e < E; ++e) {
                int taken = 0;
                for (int64_t i = 0; i < j; ++i)
                    if (id[i] == e) taken = 1;
                if (taken) continue;
                if (best < 0 || ranks_before(l[e], e, l[best], best)) best = e;
            }
            id[j] = (int32_t)best;
        }
        const float lmax = l[id[0]];
        float s = 0.0f;
        for (int64_t j = 0; j < k; ++j) s = s + unnormalised_weight(l[id[j]], lmax);
        for (int64_t j = 0; j < k; ++j)
            topk_w[t * k + j] = unnormalised_weight(l[id[j]], lmax) / s;
    }
    int64_t r = 0;
    for (int64_t e = 0; e < E; ++e) {
        expert_off[e] = (int32_t)r;
        for (int64_t t = 0; t < T; ++t)
            for (int64_t j = 0; j < k; ++j)
                if (topk_id[t * k + j] == e) {
                    row_idx[r] = (int32_t)t;
                    row_of[t * k + j] = (int32_t)r;
                    ++r;
                }
    }
    expert_off[E] = (int32_t)r;
}

/* out [T][H] = sum over j < k of topk_w[t][j] * y[row_of[t][j]][:] (y [R][ldy]) */
void o_moe_combine(const float *y, int64_t ldy, const int32_t *row_of, const float *topk_w,
                   int64_t T, int64_t k, int64_t H, float *out)
{
    for (int64_t t = 0; t < T; ++t)
        for (int64_t h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int64_t j = 0; j < k; ++j)
                acc = fmaf(topk_w[t * k + j], y[(int64_t)row_of[t * k + j] * ldy + h], acc);
            out[t * H + h] = acc;
        }
}
