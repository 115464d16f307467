/*
 * jetq oracle: a plain, slow, obviously-correct CPU statement of the
 * block-scaled FP8 (E4M3) quantize-and-GEMM precision flow.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library calls this code; only the
 * tests, __graft_entry__.smoke() and bench.py's CPU-baseline leg load it.  It
 * shares no code, header, table or constant with the CUDA path.
 *
 * Sources (web pages, cited by title and section):
 *   [JR]  "Jet-RL: Enabling On-Policy FP8 Reinforcement Learning with Unified
 *         Training and Rollout Precision Flow" (paper-graph-ui explainer),
 *         section "GEMM Quantization: Granularity, Layout, and Kernel Design"
 *         and "The Three GEMM Operations and Their Quantization Configuration".
 *   [JR2] the papercache summary of the same paper, section 2.1 (quantizer
 *         equation: X^ = round(X / S_X), S_X = max|X| / Delta_max,
 *         Delta_max = 448 for E4M3), section 2.2 (the shapes of FProp, WGrad,
 *         DGrad) and section 4.2 (1x128 activations, 128x128 weights, the
 *         WGrad operands grouped along the token axis).
 *   [MB]  the Miles "Blackwell-native RL recipes" post, MXFP8 section
 *         (one E8M0 scale per 32 consecutive E4M3 values, a power of two
 *         rounded upward so that the largest value of a block still fits;
 *         the row-wise and column-wise copies each come from full precision).
 *
 * Readings where the pages are silent or garbled (each is listed in the
 * design notes):
 *   - round() is round-to-nearest, ties to even, saturating at +-448.
 *   - the scale is an FP32 number S = fl32(amax / 448) and the quotient is
 *     taken in FP32, q = E4M3(fl32(x / S)): two roundings, in that order.
 *   - an all-zero group has S = 0 and every code 0x00 (MX: scale byte 127).
 *   - column groups never cross segment bounds; a partial group's amax
 *     covers only its valid rows; each segment of the column copy starts at a
 *     multiple of the group size and its padding codes are 0x00.
 *
 * Build: plain C99, -O2 -ffp-contract=off, no fast-math.  Arithmetic is
 * IEEE binary32/binary64 as written; FLT_EVAL_METHOD must be 0.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#if FLT_EVAL_METHOD != 0
#error "the oracle needs FLT_EVAL_METHOD == 0 (float arithmetic rounded to float)"
#endif

#define E4M3_MAX 448.0

/* ------------------------------------------------------------------------ */
/* BF16 and FP32 bit views                                                  */
/* ------------------------------------------------------------------------ */

static float bf16_value(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16; /* bf16 is the top half of a binary32 */
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* ------------------------------------------------------------------------ */
/* E4M3 ("FN" variant of the OCP 8-bit float spec cited by [JR2] 2.1):      */
/* sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no infinities,   */
/* S.1111.111 is NaN, largest finite magnitude 1.75 * 2^8 = 448.            */
/* ------------------------------------------------------------------------ */

double jo_e4m3_decode(uint8_t code)
{
    int sign = code >> 7;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9); /* subnormal: m/8 * 2^(1-7) */
    else
        mag = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/*
 * Nearest finite E4M3 value to v, ties to the code with an even mantissa
 * (the last code bit), magnitudes above 448 saturated to 448, sign of zero
 * kept.  Positive finite codes 0x00..0x7E are increasing in value, so the
 * search is over that ordered list; the comparison is against the exact
 * midpoint of two neighbours (a binary64 number), so no rounding enters.
 */
uint8_t jo_e4m3_encode(double v)
{
    uint8_t sign;
    double a, mid;
    int lo, hi;
    if (isnan(v))
        return 0x7F;
    sign = signbit(v) ? 0x80 : 0x00;
    a = fabs(v);
    lo = 0;
    hi = 0x7E;
    while (lo < hi) { /* largest code c with decode(c) <= a */
        int c = (lo + hi + 1) / 2;
        if (jo_e4m3_decode((uint8_t)c) <= a)
            lo = c;
        else
            hi = c - 1;
    }
    if (lo == 0x7E)
        return (uint8_t)(sign | 0x7E); /* saturate */
    mid = 0.5 * (jo_e4m3_decode((uint8_t)lo) + jo_e4m3_decode((uint8_t)(lo + 1)));
    if (a < mid)
        return (uint8_t)(sign | lo);
    if (a > mid)
        return (uint8_t)(sign | (lo + 1));
    return (uint8_t)(sign | ((lo & 1) ? lo + 1 : lo)); /* tie: even mantissa */
}

/* ------------------------------------------------------------------------ */
/* FP32-scale group quantizer, [JR2] 2.1 and [JR] "GEMM Quantization":      */
/*   S = fl32(amax / 448),  q = E4M3(fl32(x / S)).                          */
/* ------------------------------------------------------------------------ */

static float scale_of(float amax)
{
    return amax / (float)E4M3_MAX; /* binary32 division, round to nearest */
}

static uint8_t quant_value(float x, float s)
{
    if (s == 0.0f)
        return 0x00; /* all-zero group */
    return jo_e4m3_encode((double)(x / s)); /* x / s rounded to binary32 */
}

/*
 * Row-wise groups of `gs` consecutive columns ([JR] 1x128 activation
 * quantization: one scale per token and 128-channel group).
 *   x  : bf16 [rows x cols], row stride ldx (elements)
 *   q  : codes [rows x cols], row stride ldq (bytes)
 *   s  : scales [cols/gs x rows], group-major: s[g * rows + r]
 */
void jo_quant_rowgroups(const uint16_t *x, int64_t rows, int64_t cols, int64_t ldx, int64_t gs,
                        uint8_t *q, int64_t ldq, float *s)
{
    int64_t r, g, j;
    for (r = 0; r < rows; ++r) {
        for (g = 0; g < cols / gs; ++g) {
            float amax = 0.0f, sc;
            for (j = 0; j < gs; ++j) {
                float v = fabsf(bf16_value(x[r * ldx + g * gs + j]));
                if (v > amax)
                    amax = v;
            }
            sc = scale_of(amax);
            s[g * rows + r] = sc;
            for (j = 0; j < gs; ++j)
                q[r * ldq + g * gs + j] = quant_value(bf16_value(x[r * ldx + g * gs + j]), sc);
        }
    }
}

/* padded start of every segment in the column copy: pad[e] = sum_{j<e} ceil(n_j/gs)*gs */
static void padded_starts(const int64_t *off, int nseg, int64_t gs, int64_t *pad)
{
    int e;
    pad[0] = 0;
    for (e = 0; e < nseg; ++e) {
        int64_t n = off[e + 1] - off[e];
        pad[e + 1] = pad[e] + ((n + gs - 1) / gs) * gs;
    }
}

/* total padded length of the column copy (a multiple of gs) */
int64_t jo_colcopy_length(const int64_t *off, int nseg, int64_t gs)
{
    int64_t *pad = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nseg + 1));
    int64_t total;
    padded_starts(off, nseg, gs, pad);
    total = pad[nseg];
    free(pad);
    return total;
}

/*
 * Column-wise groups of `gs` consecutive rows, stored transposed ([JR2] 4.2:
 * the WGrad operands are grouped 128 along the token axis; [MB]: the
 * column-wise copy is quantized from full precision).
 *   x    : bf16 [rows x cols], row stride ldx
 *   off  : segment bounds, off[0] = 0 <= ... <= off[nseg] = rows
 *   qc   : codes [cols x ldqc]; segment e occupies columns pad[e] .. ,
 *          padding codes inside a segment's last group are 0x00
 *   sc   : scales [P/gs x cols], sc[(pad[e]/gs + t) * cols + c]
 */
void jo_quant_colgroups(const uint16_t *x, int64_t rows, int64_t cols, int64_t ldx, int64_t gs,
                        const int64_t *off, int nseg, uint8_t *qc, int64_t ldqc, float *sc)
{
    int64_t *pad = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nseg + 1));
    int e;
    (void)rows;
    padded_starts(off, nseg, gs, pad);
    for (e = 0; e < nseg; ++e) {
        int64_t n_e = off[e + 1] - off[e];
        int64_t t, c, i;
        for (t = 0; t * gs < n_e; ++t) {
            int64_t r0 = off[e] + t * gs;
            int64_t valid = (n_e - t * gs < gs) ? n_e - t * gs : gs;
            int64_t col0 = pad[e] + t * gs;
            for (c = 0; c < cols; ++c) {
                float amax = 0.0f, s;
                for (i = 0; i < valid; ++i) {
                    float v = fabsf(bf16_value(x[(r0 + i) * ldx + c]));
                    if (v > amax)
                        amax = v;
                }
                s = scale_of(amax);
                sc[(col0 / gs) * cols + c] = s;
                for (i = 0; i < gs; ++i)
                    qc[c * ldqc + col0 + i] =
                        (i < valid) ? quant_value(bf16_value(x[(r0 + i) * ldx + c]), s) : 0x00;
            }
        }
    }
    free(pad);
}

/*
 * Column copy re-quantized from the FP8 row copy ([JR] requantize_for_dgrad:
 * the 1x128 copy is taken back through dequantization and quantized again
 * along the token dimension; [MB] calls this the DeepSeek-V3 style).  Every
 * value is first rebuilt in binary32,
 *     v = fl32(decode(q_row[r, k]) * S_row[k/gs, r]),
 * then quantized exactly as jo_quant_colgroups quantizes BF16 input
 * (segments start on multiples of gs, gs x 1 groups, padding codes 0).
 *   q_row : [rows x cols] ; s_row : [cols/gs x rows]
 */
static float requant_value(const uint8_t *q_row, const float *s_row, int64_t rows, int64_t cols, int64_t gs,
                           int64_t r, int64_t c)
{
    return (float)jo_e4m3_decode(q_row[r * cols + c]) * s_row[(c / gs) * rows + r];
}

void jo_requant_colgroups(const uint8_t *q_row, const float *s_row, int64_t rows, int64_t cols, int64_t gs,
                          const int64_t *off, int nseg, uint8_t *qc, int64_t ldqc, float *sc)
{
    int64_t *pad = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nseg + 1));
    int e;
    padded_starts(off, nseg, gs, pad);
    for (e = 0; e < nseg; ++e) {
        int64_t n_e = off[e + 1] - off[e];
        int64_t t, c, i;
        for (t = 0; t * gs < n_e; ++t) {
            int64_t r0 = off[e] + t * gs;
            int64_t valid = (n_e - t * gs < gs) ? n_e - t * gs : gs;
            int64_t col0 = pad[e] + t * gs;
            for (c = 0; c < cols; ++c) {
                float amax = 0.0f, s;
                for (i = 0; i < valid; ++i) {
                    float v = fabsf(requant_value(q_row, s_row, rows, cols, gs, r0 + i, c));
                    if (v > amax)
                        amax = v;
                }
                s = scale_of(amax);
                sc[(col0 / gs) * cols + c] = s;
                for (i = 0; i < gs; ++i)
                    qc[c * ldqc + col0 + i] =
                        (i < valid) ? quant_value(requant_value(q_row, s_row, rows, cols, gs, r0 + i, c), s) : 0x00;
            }
        }
    }
    free(pad);
}

/*
 * BF16 round-to-nearest-even of a binary64 value (used on exact products:
 * a 4-bit E4M3 significand times a 24-bit scale is exact in binary64, so the
 * dequantized BF16 value is rounded once).  bf16 keeps 8 significant bits;
 * below 2^-126 the quantum stays 2^-133 (subnormals).
 */
static uint16_t bf16_rne(double v)
{
    double a = fabs(v), quantum, m;
    float f;
    uint32_t u;
    int k;
    if (a == 0.0)
        return signbit(v) ? 0x8000u : 0u;
    (void)frexp(a, &k); /* a = f * 2^k, f in [0.5, 1): leading bit 2^(k-1) */
    quantum = ldexp(1.0, (k - 1 < -126 ? -126 : k - 1) - 7);
    m = nearbyint(a / quantum); /* a / quantum is exact; default mode rounds half to even */
    f = (float)(m * quantum);   /* exactly a bf16 value */
    memcpy(&u, &f, sizeof u);
    return (uint16_t)((u >> 16) | (signbit(v) ? 0x8000u : 0u));
}

/* Dequantization to BF16 of a row-group copy (gs groups along each row) or of
 * bs x bs blocks: out = BF16(decode(q) * S), S from the copy's scale layout. */
void jo_dequant_rowgroups_bf16(const uint8_t *q, int64_t rows, int64_t cols, int64_t gs, const float *s,
                               uint16_t *out)
{
    int64_t r, c;
    for (r = 0; r < rows; ++r)
        for (c = 0; c < cols; ++c)
            out[r * cols + c] = bf16_rne(jo_e4m3_decode(q[r * cols + c]) * (double)s[(c / gs) * rows + r]);
}

void jo_dequant_blocks_bf16(const uint8_t *q, int64_t rows, int64_t cols, int64_t bs, const float *s, uint16_t *out)
{
    int64_t r, c;
    for (r = 0; r < rows; ++r)
        for (c = 0; c < cols; ++c)
            out[r * cols + c] =
                bf16_rne(jo_e4m3_decode(q[r * cols + c]) * (double)s[(r / bs) * (cols / bs) + c / bs]);
}

/* ------------------------------------------------------------------------ */
/* Producers fused with the 1x128 quantizer ([JR] the activation quantizer  */
/* sits in the kernel that produces the tensor; the pages name RMSNorm and  */
/* the SwiGLU product as producers).  The producer output is the BF16 value */
/* the unfused layer would store, defined operation by operation in          */
/* binary32 so that the GPU can reproduce it bit for bit; it is then         */
/* quantized exactly as jo_quant_rowgroups / jo_quant_colgroups quantize     */
/* BF16 input.                                                               */
/* ------------------------------------------------------------------------ */

static uint16_t bf16_of_float(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    u += 0x7FFFu + ((u >> 16) & 1u); /* round to nearest even (finite values) */
    return (uint16_t)(u >> 16);
}

static float float_of_bits(uint32_t u)
{
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/*
 * exp in binary32 by Cody-Waite reduction and a Taylor polynomial (textbook
 * method, e.g. Muller, "Elementary Functions", ch. 11): n = rint(x log2 e),
 * r = x - n ln2 with ln2 split in two constants, exp(r) = sum_{k<=7} r^k/k!
 * in Horner form with fmaf, result p * 2^n (2^n built from its bits).
 * Inputs above 88 give +inf, below -87 give 0 (flushed).
 */
float jo_expf_fixed(float x)
{
    const float log2e = 1.44269502f, ln2_hi = 0.693145751953125f, ln2_lo = 1.42860677e-06f;
    const float c[8] = {1.0f, 1.0f, 0.5f, 0.166666672f, 0.0416666679f, 0.00833333377f, 0.00138888892f,
                        0.000198412701f};
    float n, r, p;
    int k;
    if (x > 88.0f)
        return float_of_bits(0x7F800000u);
    if (x < -87.0f)
        return 0.0f;
    n = rintf(x * log2e);
    r = fmaf(-n, ln2_hi, x);
    r = fmaf(-n, ln2_lo, r);
    p = c[7];
    for (k = 6; k >= 0; --k)
        p = fmaf(p, r, c[k]);
    return p * float_of_bits((uint32_t)((int)n + 127) << 23);
}

/* SwiGLU product: h = BF16(fl32(fl32(g * fl32(1 / fl32(1 + exp(-g)))) * u)) */
void jo_swiglu_bf16(const uint16_t *gate, const uint16_t *up, int64_t count, uint16_t *h)
{
    int64_t i;
    for (i = 0; i < count; ++i) {
        float gv = bf16_value(gate[i]), uv = bf16_value(up[i]);
        float e = jo_expf_fixed(-gv);
        float sg = 1.0f / (1.0f + e);
        h[i] = bf16_of_float((gv * sg) * uv);
    }
}

/*
 * RMSNorm: per row, the sum of squares in binary32 in a fixed order (each
 * 128-column group summed left to right with fmaf, then the group sums added
 * left to right), rstd = 1 / sqrt(sum / cols + eps) (IEEE division and square
 * root), y = BF16(fl32(fl32(x * rstd) * w)).  rstd is returned per row.
 */
void jo_rmsnorm_bf16(const uint16_t *x, const uint16_t *w, int64_t rows, int64_t cols, int64_t ldx, float eps,
                     uint16_t *y, float *rstd)
{
    int64_t r, c, g;
    for (r = 0; r < rows; ++r) {
        float total = 0.0f, rs;
        for (g = 0; g < cols / 128; ++g) {
            float part = 0.0f;
            for (c = g * 128; c < (g + 1) * 128; ++c) {
                float v = bf16_value(x[r * ldx + c]);
                part = fmaf(v, v, part);
            }
            total = total + part;
        }
        rs = 1.0f / sqrtf(total / (float)cols + eps);
        rstd[r] = rs;
        for (c = 0; c < cols; ++c)
            y[r * cols + c] = bf16_of_float((bf16_value(x[r * ldx + c]) * rs) * bf16_value(w[c]));
    }
}

/*
 * Square blocks of bs x bs ([JR] 128x128 per-block weight quantization,
 * S_W(i,j) = max|W_tile(i,j)| / 448, W^ = round(W / S_W)).
 *   w  : bf16 [rows x cols], row stride ldw
 *   q  : codes [rows x cols] (dense), s : [rows/bs x cols/bs] row-major
 *   qT : optional transposed codes [cols x rows], sT : [cols/bs x rows/bs]
 *        ([JR]: DGrad takes the quantized weight merely transposed).
 */
void jo_quant_blocks(const uint16_t *w, int64_t rows, int64_t cols, int64_t ldw, int64_t bs,
                     uint8_t *q, float *s, uint8_t *qT, float *sT)
{
    int64_t bi, bj, i, j;
    for (bi = 0; bi < rows / bs; ++bi) {
        for (bj = 0; bj < cols / bs; ++bj) {
            float amax = 0.0f, sc;
            for (i = 0; i < bs; ++i)
                for (j = 0; j < bs; ++j) {
                    float v = fabsf(bf16_value(w[(bi * bs + i) * ldw + bj * bs + j]));
                    if (v > amax)
                        amax = v;
                }
            sc = scale_of(amax);
            s[bi * (cols / bs) + bj] = sc;
            if (sT)
                sT[bj * (rows / bs) + bi] = sc;
            for (i = 0; i < bs; ++i)
                for (j = 0; j < bs; ++j) {
                    int64_t r = bi * bs + i, c = bj * bs + j;
                    uint8_t code = quant_value(bf16_value(w[r * ldw + c]), sc);
                    q[r * cols + c] = code;
                    if (qT)
                        qT[c * rows + r] = code;
                }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* MXFP8 ([MB], MXFP8 section): blocks of 32 consecutive values share one   */
/* E8M0 scale 2^e, rounded upward so the block maximum stays in range:     */
/* e is the smallest integer with amax <= 448 * 2^e, clamped to [-127,127]; */
/* the scale byte is e + 127 and q = E4M3(x * 2^-e) (the product is exact   */
/* in binary64, so there is exactly one rounding).  All-zero block: byte    */
/* 127 (scale 1) and codes 0x00.                                            */
/* ------------------------------------------------------------------------ */

int jo_e8m0_exponent(float amax)
{
    int e;
    double a = (double)amax;
    if (a == 0.0)
        return 0;
    /* frexp: a = f * 2^k with f in [0.5, 1); start from a bound below the answer */
    {
        int k;
        (void)frexp(a, &k);
        e = k - 10; /* 448 * 2^(k-10) < 2^(k-1) <= a, so the answer is larger */
    }
    while (a > E4M3_MAX * ldexp(1.0, e)) /* exact comparisons in binary64 */
        ++e;
    if (e < -127)
        e = -127;
    if (e > 127)
        e = 127;
    return e;
}

static uint8_t mx_value(float x, int e, int zero_block)
{
    if (zero_block)
        return 0x00;
    return jo_e4m3_encode((double)x * ldexp(1.0, -e));
}

/*
 * Row-wise MX blocks of `bs` consecutive columns.
 *   x : bf16 [rows x cols] stride ldx ; q : [rows x cols] stride ldq
 *   e8: logical scale bytes [rows x cols/bs] (row-major)
 */
void jo_quant_mx_rows(const uint16_t *x, int64_t rows, int64_t cols, int64_t ldx, int64_t bs,
                      uint8_t *q, int64_t ldq, uint8_t *e8)
{
    int64_t r, g, j;
    for (r = 0; r < rows; ++r) {
        for (g = 0; g < cols / bs; ++g) {
            float amax = 0.0f;
            int e;
            for (j = 0; j < bs; ++j) {
                float v = fabsf(bf16_value(x[r * ldx + g * bs + j]));
                if (v > amax)
                    amax = v;
            }
            e = jo_e8m0_exponent(amax);
            e8[r * (cols / bs) + g] = (uint8_t)(e + 127);
            for (j = 0; j < bs; ++j)
                q[r * ldq + g * bs + j] = mx_value(bf16_value(x[r * ldx + g * bs + j]), e, amax == 0.0f);
        }
    }
}

/*
 * Power-of-two bs x bs weight blocks (the blockwise recipe with its FP32
 * scales constrained to powers of two: [SK] "Deep dive: FP8 quantization with
 * FP32 and power-of-two block scales"; the only block scaling Blackwell
 * tensor cores take).  The exponent follows the rule above: per block e is
 * the smallest integer with amax <= 448 * 2^e, the byte is e + 127 and
 * q = E4M3(w * 2^-e).
 *   w : bf16 [rows x cols] stride ldw ; q : [rows x cols] ; e8 : [rows/bs x cols/bs]
 *   qT, e8T (optional): the transposed codes [cols x rows] and bytes [cols/bs x rows/bs]
 */
void jo_quant_blocks_pow2(const uint16_t *w, int64_t rows, int64_t cols, int64_t ldw, int64_t bs,
                          uint8_t *q, uint8_t *e8, uint8_t *qT, uint8_t *e8T)
{
    int64_t bi, bj, i, j;
    for (bi = 0; bi < rows / bs; ++bi) {
        for (bj = 0; bj < cols / bs; ++bj) {
            float amax = 0.0f;
            int e;
            for (i = 0; i < bs; ++i)
                for (j = 0; j < bs; ++j) {
                    float v = fabsf(bf16_value(w[(bi * bs + i) * ldw + bj * bs + j]));
                    if (v > amax)
                        amax = v;
                }
            e = jo_e8m0_exponent(amax);
            e8[bi * (cols / bs) + bj] = (uint8_t)(e + 127);
            if (e8T)
                e8T[bj * (rows / bs) + bi] = (uint8_t)(e + 127);
            for (i = 0; i < bs; ++i)
                for (j = 0; j < bs; ++j) {
                    int64_t r = bi * bs + i, c = bj * bs + j;
                    uint8_t code = mx_value(bf16_value(w[r * ldw + c]), e, amax == 0.0f);
                    q[r * cols + c] = code;
                    if (qT)
                        qT[c * rows + r] = code;
                }
        }
    }
}

/*
 * Column-wise MX blocks of `bs` consecutive rows inside each segment, stored
 * transposed like jo_quant_colgroups; segments start at multiples of `seg_align`
 * (a multiple of bs) in the column copy.
 *   qc : [cols x ldqc] ; e8 : logical scale bytes [cols x P/bs] (row-major)
 */
void jo_quant_mx_cols(const uint16_t *x, int64_t rows, int64_t cols, int64_t ldx, int64_t bs,
                      int64_t seg_align, const int64_t *off, int nseg, uint8_t *qc, int64_t ldqc,
                      uint8_t *e8)
{
    int64_t *pad = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nseg + 1));
    int64_t P;
    int e;
    (void)rows;
    padded_starts(off, nseg, seg_align, pad);
    P = pad[nseg];
    for (e = 0; e < nseg; ++e) {
        int64_t n_e = off[e + 1] - off[e];
        int64_t t, c, i;
        for (t = 0; t * bs < ((n_e + seg_align - 1) / seg_align) * seg_align; ++t) {
            int64_t r0 = off[e] + t * bs;
            int64_t valid = n_e - t * bs;
            int64_t col0 = pad[e] + t * bs;
            if (valid < 0)
                valid = 0;
            if (valid > bs)
                valid = bs;
            for (c = 0; c < cols; ++c) {
                float amax = 0.0f;
                int ex;
                for (i = 0; i < valid; ++i) {
                    float v = fabsf(bf16_value(x[(r0 + i) * ldx + c]));
                    if (v > amax)
                        amax = v;
                }
                ex = jo_e8m0_exponent(amax);
                e8[c * (P / bs) + col0 / bs] = (uint8_t)(ex + 127);
                for (i = 0; i < bs; ++i)
                    qc[c * ldqc + col0 + i] =
                        (i < valid) ? mx_value(bf16_value(x[(r0 + i) * ldx + c]), ex, amax == 0.0f) : 0x00;
            }
        }
    }
    free(pad);
}

/* ------------------------------------------------------------------------ */
/* Dequantizers: x^ = decode(q) * S, in binary64, back to the natural       */
/* [rows x cols] layout of the tensor the copy was made from.               */
/* ------------------------------------------------------------------------ */

void jo_dequant_rowgroups(const uint8_t *q, int64_t rows, int64_t cols, int64_t ldq, int64_t gs,
                          const float *s, double *out)
{
    int64_t r, c;
    for (r = 0; r < rows; ++r)
        for (c = 0; c < cols; ++c)
            out[r * cols + c] = jo_e4m3_decode(q[r * ldq + c]) * (double)s[(c / gs) * rows + r];
}

void jo_dequant_colgroups(const uint8_t *qc, int64_t ldqc, const float *sc, int64_t rows, int64_t cols,
                          int64_t gs, const int64_t *off, int nseg, double *out)
{
    int64_t *pad = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nseg + 1));
    int e;
    (void)rows;
    padded_starts(off, nseg, gs, pad);
    for (e = 0; e < nseg; ++e) {
        int64_t i, c;
        for (i = 0; i < off[e + 1] - off[e]; ++i) {
            int64_t col = pad[e] + i; /* position in the column copy */
            for (c = 0; c < cols; ++c)
                out[(off[e] + i) * cols + c] =
                    jo_e4m3_decode(qc[c * ldqc + col]) * (double)sc[(col / gs) * cols + c];
        }
    }
    free(pad);
}

void jo_dequant_blocks(const uint8_t *q, int64_t rows, int64_t cols, int64_t bs, const float *s,
                       double *out)
{
    int64_t r, c;
    for (r = 0; r < rows; ++r)
        for (c = 0; c < cols; ++c)
            out[r * cols + c] = jo_e4m3_decode(q[r * cols + c]) * (double)s[(r / bs) * (cols / bs) + c / bs];
}

/* power-of-two blocks: value = decode(q) * 2^(byte - 127) */
void jo_dequant_blocks_pow2(const uint8_t *q, int64_t rows, int64_t cols, int64_t bs, const uint8_t *e8, double *out)
{
    int64_t r, c;
    for (r = 0; r < rows; ++r)
        for (c = 0; c < cols; ++c)
            out[r * cols + c] =
                jo_e4m3_decode(q[r * cols + c]) * ldexp(1.0, (int)e8[(r / bs) * (cols / bs) + c / bs] - 127);
}

void jo_dequant_mx_rows(const uint8_t *q, int64_t rows, int64_t cols, int64_t ldq, int64_t bs,
                        const uint8_t *e8, double *out)
{
    int64_t r, c;
    for (r = 0; r < rows; ++r)
        for (c = 0; c < cols; ++c)
            out[r * cols + c] =
                jo_e4m3_decode(q[r * ldq + c]) * ldexp(1.0, (int)e8[r * (cols / bs) + c / bs] - 127);
}

void jo_dequant_mx_cols(const uint8_t *qc, int64_t ldqc, const uint8_t *e8, int64_t P, int64_t rows,
                        int64_t cols, int64_t bs, int64_t seg_align, const int64_t *off, int nseg,
                        double *out)
{
    int64_t *pad = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nseg + 1));
    int e;
    (void)rows;
    padded_starts(off, nseg, seg_align, pad);
    for (e = 0; e < nseg; ++e) {
        int64_t i, c;
        for (i = 0; i < off[e + 1] - off[e]; ++i) {
            int64_t col = pad[e] + i;
            for (c = 0; c < cols; ++c)
                out[(off[e] + i) * cols + c] =
                    jo_e4m3_decode(qc[c * ldqc + col]) * ldexp(1.0, (int)e8[c * (P / bs) + col / bs] - 127);
        }
    }
    free(pad);
}

/* ------------------------------------------------------------------------ */
/* The three linear-layer GEMMs of [JR2] 2.2, in binary64 on dequantized    */
/* operands given in their natural layouts:                                 */
/*   FProp  Y[n,d]   = sum_c X[n,c]  W[d,c]      (Y = X W^T)                */
/*   DGrad  dX[n,c]  = sum_d dY[n,d] W[d,c]      (dX = dY W)                */
/*   WGrad  dW[d,c]  = sum_n dY[n,d] X[n,c]      (dW = dY^T X)              */
/* Each output also gets bound = sum |term|, the scale of its rounding      */
/* error.  `at` lists (i, j) output coordinates (count pairs); NULL means    */
/* every output, written row-major into y / bound.                          */
/* ------------------------------------------------------------------------ */

static void dot_terms(const double *a, int64_t sa, const double *b, int64_t sb, int64_t k, double *y,
                      double *bound)
{
    double acc = 0.0, mag = 0.0;
    int64_t i;
    for (i = 0; i < k; ++i) {
        double t = a[i * sa] * b[i * sb];
        acc += t;
        mag += fabs(t);
    }
    *y = acc;
    *bound = mag;
}

void jo_fprop(const double *X, const double *W, int64_t N, int64_t D, int64_t C, const int64_t *at,
              int64_t count, double *y, double *bound)
{
    int64_t i;
    if (!at) {
        int64_t n, d;
        for (n = 0; n < N; ++n)
            for (d = 0; d < D; ++d)
                dot_terms(X + n * C, 1, W + d * C, 1, C, &y[n * D + d], &bound[n * D + d]);
        return;
    }
    for (i = 0; i < count; ++i)
        dot_terms(X + at[2 * i] * C, 1, W + at[2 * i + 1] * C, 1, C, &y[i], &bound[i]);
}

void jo_dgrad(const double *dY, const double *W, int64_t N, int64_t D, int64_t C, const int64_t *at,
              int64_t count, double *y, double *bound)
{
    int64_t i;
    if (!at) {
        int64_t n, c;
        for (n = 0; n < N; ++n)
            for (c = 0; c < C; ++c)
                dot_terms(dY + n * D, 1, W + c, C, D, &y[n * C + c], &bound[n * C + c]);
        return;
    }
    for (i = 0; i < count; ++i)
        dot_terms(dY + at[2 * i] * D, 1, W + at[2 * i + 1], C, D, &y[i], &bound[i]);
}

void jo_wgrad(const double *dY, const double *X, int64_t N, int64_t D, int64_t C, const int64_t *at,
              int64_t count, double *y, double *bound)
{
    int64_t i;
    if (!at) {
        int64_t d, c;
        for (d = 0; d < D; ++d)
            for (c = 0; c < C; ++c)
                dot_terms(dY + d, D, X + c, C, N, &y[d * C + c], &bound[d * C + c]);
        return;
    }
    for (i = 0; i < count; ++i)
        dot_terms(dY + at[2 * i], D, X + at[2 * i + 1], C, N, &y[i], &bound[i]);
}

/* ------------------------------------------------------------------------ */
/* NVFP4 ([MB] NVFP4 section): FP4 E2M1 values with one E4M3 scale per      */
/* block of 16 consecutive values (rounded to the nearest E4M3 value) and    */
/* one FP32 scale for a larger scope: one per token (row) for activations,   */
/* one per tensor (shared by a gate/up pair) for weights.  The pages give    */
/* no formula; the readings, in the order of the FP8 recipe above:           */
/*   S_g = fl32(amax_scope / 2688)          (2688 = 448 * 6: the largest     */
/*                                           E4M3 scale times the largest    */
/*                                           E2M1 value)                     */
/*   block b:  e_b = E4M3(fl32(fl32(amax_b / 6) / S_g))                      */
/*             D_b = fl32(decode(e_b) * S_g)                                 */
/*             q   = E2M1(fl32(x / D_b)),  D_b = 0: every code 0x0           */
/* E2M1: sign, 2 exponent bits (bias 1), 1 mantissa bit; magnitudes 0, 0.5,  */
/* 1, 1.5, 2, 3, 4, 6; nearest value, ties to the even code, saturating at   */
/* 6, sign of zero kept.  Two codes per byte, element 2j in the low nibble.  */
/* ------------------------------------------------------------------------ */

double jo_e2m1_decode(uint8_t code)
{
    static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    double m = mag[code & 7];
    return (code & 8) ? -m : m;
}

uint8_t jo_e2m1_encode(double v)
{
    uint8_t sign = signbit(v) ? 8 : 0;
    double a = fabs(v), mid;
    int lo = 0;
    while (lo < 7 && jo_e2m1_decode((uint8_t)(lo + 1)) <= a) /* largest code with decode <= a */
        ++lo;
    if (lo == 7)
        return (uint8_t)(sign | 7); /* saturate */
    mid = 0.5 * (jo_e2m1_decode((uint8_t)lo) + jo_e2m1_decode((uint8_t)(lo + 1)));
    if (a < mid)
        return (uint8_t)(sign | lo);
    if (a > mid)
        return (uint8_t)(sign | (lo + 1));
    return (uint8_t)(sign | ((lo & 1) ? lo + 1 : lo)); /* tie: even code */
}

/*
 *   x   : bf16 [rows x cols], row stride ldx; cols a multiple of 16
 *   scope_amax : NULL for one scale per row (the row's max |x|), else the
 *         max |x| of the tensor scope, one scale for every row
 *   q   : packed codes [rows x cols/2];  sb : E4M3 block scales [rows x cols/16]
 *   sg  : FP32 scope scales, [rows] (per row) or [1]
 */
void jo_quant_nvfp4(const uint16_t *x, int64_t rows, int64_t cols, int64_t ldx, const float *scope_amax,
                    uint8_t *q, uint8_t *sb, float *sg)
{
    int64_t r, b, j;
    for (r = 0; r < rows; ++r) {
        float amax = 0.0f, s;
        if (scope_amax) {
            amax = *scope_amax;
        } else {
            for (j = 0; j < cols; ++j) {
                float v = fabsf(bf16_value(x[r * ldx + j]));
                if (v > amax)
                    amax = v;
            }
        }
        s = amax / 2688.0f;
        if (!scope_amax || r == 0)
            sg[scope_amax ? 0 : r] = s;
        for (b = 0; b < cols / 16; ++b) {
            float ab = 0.0f, d;
            uint8_t e;
            for (j = 0; j < 16; ++j) {
                float v = fabsf(bf16_value(x[r * ldx + b * 16 + j]));
                if (v > ab)
                    ab = v;
            }
            e = s > 0.0f ? jo_e4m3_encode((double)((ab / 6.0f) / s)) : 0x00;
            sb[r * (cols / 16) + b] = e;
            d = (float)jo_e4m3_decode(e) * s; /* binary32 product */
            for (j = 0; j < 16; j += 2) {
                uint8_t c0 = 0, c1 = 0;
                if (d != 0.0f) {
                    c0 = jo_e2m1_encode((double)(bf16_value(x[r * ldx + b * 16 + j]) / d));
                    c1 = jo_e2m1_encode((double)(bf16_value(x[r * ldx + b * 16 + j + 1]) / d));
                }
                q[r * (cols / 2) + b * 8 + j / 2] = (uint8_t)(c0 | (c1 << 4));
            }
        }
    }
}

/* out = e2m1 * decode(e_b) * S_g in binary64 (exact: a 2-bit times a 4-bit
 * times a 24-bit significand), the operand value the NVFP4 GEMM multiplies
 * (Miles "Blackwell-native RL recipes", NVFP4 section: E2M1 values, one E4M3
 * scale per 16 values, one FP32 scale for a larger scope).  Codes packed two
 * per byte, element 2j in the low nibble; sg per row (per_row) or one. */
void jo_dequant_nvfp4(const uint8_t *q, const uint8_t *sb, const float *sg, int64_t rows, int64_t cols,
                      int per_row, double *out)
{
    int64_t r, c;
    for (r = 0; r < rows; ++r)
        for (c = 0; c < cols; ++c) {
            uint8_t byte = q[r * (cols / 2) + c / 2];
            uint8_t code = (c & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
            out[r * cols + c] =
                jo_e2m1_decode(code) * jo_e4m3_decode(sb[r * (cols / 16) + c / 16]) * (double)sg[per_row ? r : 0];
        }
}

/* out = BF16(e2m1 * decode(e_b) * S_g), rounded once: the product of a 2-bit,
 * a 4-bit and a 24-bit significand is exact in binary64. */
void jo_dequant_nvfp4_bf16(const uint8_t *q, const uint8_t *sb, const float *sg, int64_t rows, int64_t cols,
                           int per_row, uint16_t *out)
{
    int64_t r, c;
    for (r = 0; r < rows; ++r)
        for (c = 0; c < cols; ++c) {
            uint8_t byte = q[r * (cols / 2) + c / 2];
            uint8_t code = (c & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
            out[r * cols + c] = bf16_rne(jo_e2m1_decode(code) * jo_e4m3_decode(sb[r * (cols / 16) + c / 16]) *
                                         (double)sg[per_row ? r : 0]);
        }
}
