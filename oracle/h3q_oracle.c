/*
 * h3q_oracle.c -- plain, slow CPU oracle for the fused NVFP4 activation producers.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library calls this file.  It is
 * loaded by the tests, by the smoke check and by the benchmark's CPU-baseline
 * leg, and by nothing else.  It shares no code, header, table or constant with
 * the CUDA path: every definition below is written out again from the pages'
 * description of the method, in IEEE binary32 arithmetic, one rounding per
 * operation.  Build flags: -O2 -ffp-contract=off, no fast-math, so that the C
 * compiler neither fuses a multiply into an add nor reorders a sum.
 *
 * Sources (web pages; the oracle follows what they compute, not how):
 *   [FV-API]  FastVideo API page "fastvideo.models.vaes.minimax_h3_nvfp4_fused":
 *             module introduction (E4M3 block scales, layout_128x4 swizzle,
 *             zeroed padding rows, no FMA contraction where eager rounds) and
 *             the new_quantized / quantize / swiglu_quantize sources (buffer
 *             shapes [m, k/2] and [pad128(m), k/16]).
 *   [FV-CUH]  FastVideo compare "fasth3-spark-exact-perf", file
 *             fastvideo-kernel/csrc/quantization/minimax_h3_swiglu_quant.cuh:
 *             scale_float (E4M3 decode), fp4_pair (nibble order), swiglu_bf16
 *             (value * silu(gate), bf16 rounded) and quant_probe (block amax,
 *             scale = e4m3(gsf * amax / 6), codes = e2m1(y / (scale / gsf)),
 *             swizzled scale index).
 *   [TRT]     TensorRT-LLM PR #21483 "Fuse the MiniMax-H3 NVFP4 activation
 *             quantize into the AdaLN, SwiGLU and attention-output producers":
 *             summary and commit messages (AdaLN RMSNorm + modulation producer,
 *             SiLU-and-mul producer, attention-output quantize).
 *   [FV-LOG]  FastVideo commit log, branch vae-parallel-decode: the modulation
 *             index contract [0, table_rows) and the int64 indexing fix.
 *   [FV-CUH]  also minimax_h3_swiglu_gemm.cu on the same compare page
 *             (launch_gemm_swiglu, h3_epilogue::Store): the block-scaled NVFP4
 *             GEMM with value/gate-paired columns and the SwiGLU + NVFP4
 *             epilogue.
 *   [FV-API], NVFP4DecoderLinear; [FlashRT] FlashRT PR #142 "FP8/NVFP4
 *             kernelized inference pipeline", commit "...amax pipeline": the
 *             dynamic (per-call abs-max) and calibrated (running-max) scales.
 *
 * Readings where the pages are silent or use approximate arithmetic are
 * stated next to each function (division and reciprocal are correctly
 * rounded; the SiLU exponential is the fixed operation sequence exp_c).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* bit views                                                                 */
/* ------------------------------------------------------------------------ */

static uint32_t bits_of(float f) { uint32_t u; memcpy(&u, &f, sizeof u); return u; }
static float float_of(uint32_t u) { float f; memcpy(&f, &u, sizeof f); return f; }

/* ------------------------------------------------------------------------ */
/* bfloat16: the top 16 bits of a binary32, rounded to nearest, ties to even */
/* ------------------------------------------------------------------------ */

uint16_t orc_bf16_bits(float v)
{
    uint32_t u = bits_of(v);
    if (isnan(v))
        return (uint16_t)((u >> 16) | 0x0040u); /* quiet NaN, sign kept */
    uint32_t kept = u >> 16;          /* value truncated toward zero        */
    uint32_t dropped = u & 0xFFFFu;   /* what truncation threw away          */
    /* The next bf16 away from zero is kept + 1 (a carry into the exponent
     * field is the correct next value, up to and including infinity). */
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
        kept += 1u;
    return (uint16_t)kept;
}

float orc_bf16_value(uint16_t b) { return float_of((uint32_t)b << 16); }

float orc_bf16_round(float v) { return orc_bf16_value(orc_bf16_bits(v)); }

/* ------------------------------------------------------------------------ */
/* E4M3 (OCP FP8, "fn" variant: no infinities, max finite 448)               */
/* ------------------------------------------------------------------------ */

/* Decode of a non-negative finite code 0x00..0x7E: exponent bias 7, three
 * mantissa bits, subnormals m * 2^-9.  Same values as scale_float in [FV-CUH]. */
float orc_e4m3_value(uint8_t code)
{
    int e = (code >> 3) & 15;
    int m = code & 7;
    if (e == 0)
        return ldexpf((float)m, -9);
    return ldexpf(1.0f + (float)m / 8.0f, e - 7);
}

/* Encode of s >= 0: the nearest E4M3 value, ties to the even code (even
 * mantissa); anything at or above 448, including +inf, saturates to 448
 * (code 0x7E).  This is what "round to nearest even, satfinite" means for the
 * E4M3 block scale in [FV-CUH] scale_fp8.  Negative and NaN s never occur
 * (s = gsf * amax / 6 with gsf > 0). */
uint8_t orc_e4m3_encode(float s)
{
    if (!(s < 448.0f))
        return 0x7E;
    /* largest code whose value does not exceed s (values rise with the code) */
    int k = 0;
    for (int c = 0; c <= 0x7E; ++c)
        if (orc_e4m3_value((uint8_t)c) <= s)
            k = c;
    double lo = orc_e4m3_value((uint8_t)k);
    if (lo == (double)s)
        return (uint8_t)k;
    double hi = orc_e4m3_value((uint8_t)(k + 1)); /* k < 0x7E because s < 448 */
    double below = (double)s - lo;                /* exact in binary64       */
    double above = hi - (double)s;
    if (below < above)
        return (uint8_t)k;
    if (above < below)
        return (uint8_t)(k + 1);
    return (uint8_t)((k & 1) ? k + 1 : k);
}

/* ------------------------------------------------------------------------ */
/* E2M1 (FP4): magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}, code = sign<<3 | idx */
/* ------------------------------------------------------------------------ */

static const float E2M1_MAGNITUDE[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

float orc_e2m1_value(uint8_t code)
{
    float m = E2M1_MAGNITUDE[code & 7];
    return (code & 8) ? -m : m;
}

/* Nearest grid point, ties to the even index (even mantissa), saturating at
 * 6; the sign bit is the sign of v, also for -0 and for negatives that round
 * to zero (IEEE conversions keep the sign of a zero result; the pages do not
 * say otherwise). */
uint8_t orc_e2m1_encode(float v)
{
    uint8_t sign = signbit(v) ? 8 : 0;
    float a = fabsf(v);
    int idx;
    if (!(a < 6.0f)) {
        idx = 7;
    } else {
        int k = 0;
        for (int i = 0; i < 8; ++i)
            if (E2M1_MAGNITUDE[i] <= a)
                k = i;
        double below = (double)a - E2M1_MAGNITUDE[k];
        double above = (double)E2M1_MAGNITUDE[k + 1] - (double)a;
        if (below < above)
            idx = k;
        else if (above < below)
            idx = k + 1;
        else
            idx = (k & 1) ? k + 1 : k;
    }
    return (uint8_t)(sign | idx);
}

/* ------------------------------------------------------------------------ */
/* exp_c: the fixed binary32 exponential used by SiLU                        */
/* ------------------------------------------------------------------------ */
/*
 * The pages' SiLU uses the hardware ex2.approx and div.full ([FV-CUH]
 * swiglu_bf16), which no CPU reproduces.  The reading taken: an exponential
 * that is a fixed sequence of correctly rounded binary32 operations, written
 * separately here and in the kernel.  Method: Cody and Waite's additive
 * argument reduction (W. J. Cody, W. Waite, "Software Manual for the
 * Elementary Functions", 1980) with a two-part ln 2 applied by fused
 * multiply-adds, and the degree-7 Taylor polynomial of e^r in Horner form:
 *
 *   z > 89            ->  +inf
 *   z < -104          ->  +0
 *   t  = fl(z * L2E)                    L2E = fl(1 / ln 2)
 *   kf = rint(t)                        round half to even
 *   r  = fma(-kf, C1, z)                C1  = fl(ln 2)
 *   r  = fma(-kf, C2, r)                C2  = fl(ln 2 - C1)
 *   p  = P7; p = fma(p, r, Pn) for n = 6..2; p = fma(p, r, 1); p = fma(p, r, 1)
 *                                       Pn  = fl(1 / n!)
 *   k1 = trunc(k / 2), k2 = k - k1      (k = kf as an integer)
 *   result = fl(fl(p * 2^k1) * 2^k2)    (the first product is exact)
 *
 * Constants are binary32 values of the named real numbers.
 */
static const float EXPC_L2E = 0x1.715476p+0f;   /* fl(1/ln 2)        */
static const float EXPC_C1 = 0x1.62e430p-1f;    /* fl(ln 2)          */
static const float EXPC_C2 = -0x1.05c610p-29f;  /* fl(ln 2 - C1)     */
static const float EXPC_P[8] = {
    1.0f,                 /* 1/0! (unused; the last two steps add 1)  */
    1.0f,                 /* 1/1!                                     */
    0.5f,                 /* 1/2!                                     */
    0x1.555556p-3f,       /* fl(1/3!)                                 */
    0x1.555556p-5f,       /* fl(1/4!)                                 */
    0x1.111112p-7f,       /* fl(1/5!)                                 */
    0x1.6c16c2p-10f,      /* fl(1/6!)                                 */
    0x1.a01a02p-13f,      /* fl(1/7!)                                 */
};

void orc_exp_constants(float out[11])
{
    out[0] = EXPC_L2E;
    out[1] = EXPC_C1;
    out[2] = EXPC_C2;
    for (int n = 0; n < 8; ++n)
        out[3 + n] = EXPC_P[n];
}

float orc_exp(float z)
{
    if (z > 89.0f)
        return INFINITY;
    if (z < -104.0f)
        return 0.0f;
    float t = z * EXPC_L2E;
    float kf = rintf(t);
    float r = fmaf(-kf, EXPC_C1, z);
    r = fmaf(-kf, EXPC_C2, r);
    float p = EXPC_P[7];
    for (int n = 6; n >= 2; --n)
        p = fmaf(p, r, EXPC_P[n]);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    int k = (int)kf;
    int k1 = k / 2;
    int k2 = k - k1;
    float scaled = p * ldexpf(1.0f, k1);
    return scaled * ldexpf(1.0f, k2);
}

/* SwiGLU value: silu(gate) * up, rounded once to bf16 at the end, as
 * swiglu_bf16 in [FV-CUH] does (there: value * (gate * sigmoid)).  The
 * sigmoid is 1 / (1 + exp_c(-gate)) with a correctly rounded division. */
float orc_swiglu_value(float gate, float up)
{
    float e = orc_exp(-gate);
    float d = 1.0f + e;
    float sigmoid = 1.0f / d;
    float s = gate * sigmoid;
    return orc_bf16_round(s * up);
}

/* ------------------------------------------------------------------------ */
/* NVFP4 block quantize                                                       */
/* ------------------------------------------------------------------------ */
/*
 * One block is 16 consecutive elements of a row.  Following quant_probe in
 * [FV-CUH] with every approximate reciprocal replaced by a correctly rounded
 * division:
 *   amax = max |y_i|
 *   s    = fl(gsf * fl(amax / 6))
 *   sf   = E4M3(s)                      (round to nearest even, satfinite)
 *   dec  = fl(E4M3value(sf) / gsf)
 *   inv  = dec != 0 ? fl(1 / dec) : 0
 *   c_i  = E2M1(fl(y_i * inv))
 * Codes are packed two per byte, the even element in the low nibble
 * ([FV-CUH] fp4_pair).
 */
void orc_quantize_block(const float y[16], float gsf, uint8_t *sf_out, uint8_t packed[8])
{
    float amax = 0.0f;
    for (int i = 0; i < 16; ++i) {
        float a = fabsf(y[i]);
        if (a > amax)
            amax = a;
    }
    float t = amax / 6.0f;
    float s = gsf * t;
    uint8_t sf = orc_e4m3_encode(s);
    float dec = orc_e4m3_value(sf) / gsf;
    float inv = (dec != 0.0f) ? 1.0f / dec : 0.0f;
    for (int j = 0; j < 8; ++j) {
        uint8_t lo = orc_e2m1_encode(y[2 * j] * inv);
        uint8_t hi = orc_e2m1_encode(y[2 * j + 1] * inv);
        packed[j] = (uint8_t)(lo | (hi << 4));
    }
    *sf_out = sf;
}

/* Static per-tensor global scale: the block holding the tensor amax gets the
 * largest E4M3 scale (448) with its largest element on the largest E2M1
 * magnitude (6): gsf = fl(448 * 6 / amax). */
float orc_global_scale(float amax) { return 2688.0f / amax; }

/* Dynamic and calibrated scales.  [FV-API] NVFP4DecoderLinear: a dynamic
 * layer scales each call by the abs-max of its input; a calibrating layer folds
 * each call's abs-max into a persistent running maximum (input_amax).
 * [FlashRT] commit "...amax pipeline": the abs-max is taken on the device in a
 * pass of its own and read by the quantize pass, with no host synchronisation.
 *
 * orc_amax_bf16: max |v| over n bf16 values (exact; 0 for n = 0; NaN is outside
 * the contract).  orc_global_scale_from_amax: the global scale of an abs-max,
 * with two readings where the formula has no finite positive value: amax = 0
 * (an all-zero tensor, whose codes and scales are zero under any scale) gives 1,
 * and amax = +inf (a producer output that overflowed bf16) is clamped to the
 * largest finite binary32 first. */
float orc_amax_bf16(const uint16_t *v, int64_t n)
{
    float m = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(orc_bf16_value(v[i]));
        if (a > m) m = a;
    }
    return m;
}

float orc_global_scale_from_amax(float amax)
{
    if (amax == 0.0f) return 1.0f;
    if (amax > FLT_MAX) amax = FLT_MAX;
    return 2688.0f / amax;
}

/* ------------------------------------------------------------------------ */
/* 128x4 scale layout                                                         */
/* ------------------------------------------------------------------------ */
/*
 * The scale matrix is [pad128(rows), cols/16] bytes, tiled into 512-byte
 * atoms of 128 rows x 4 scale columns.  Atoms are laid out row-tile major
 * (cols/64 atoms per 128-row tile).  Inside an atom, row r sits at
 * (r % 32) * 16 + ((r / 32) % 4) * 4 and scale column g at g % 4 -- the
 * "layout_128x4" index written out in quant_probe in [FV-CUH].  Rows beyond
 * the tensor's rows are zero ([FV-API] introduction, "zeroed padding rows").
 */
int64_t orc_scale_offset(int64_t row, int64_t group, int64_t cols)
{
    int64_t atoms_per_tile_row = cols / 64;
    int64_t atom = (row / 128) * atoms_per_tile_row + group / 4;
    int64_t inside = (row % 32) * 16 + ((row / 32) % 4) * 4 + group % 4;
    return atom * 512 + inside;
}

int64_t orc_padded_rows(int64_t rows) { return (rows + 127) / 128 * 128; }

/* Offsets of every scale of the listed rows: out is [n, cols/16]. */
void orc_scale_offsets_rows(const int64_t *rows, int64_t n, int64_t cols, int64_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        for (int64_t g = 0; g < cols / 16; ++g)
            out[i * (cols / 16) + g] = orc_scale_offset(rows[i], g, cols);
}

/* sf_logical is [rows, cols/16]; out is pad128(rows) * cols/16 bytes. */
void orc_swizzle_scales(const uint8_t *sf_logical, int64_t rows, int64_t cols, uint8_t *out)
{
    int64_t groups = cols / 16;
    int64_t total = orc_padded_rows(rows) * groups;
    memset(out, 0, (size_t)total);
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t g = 0; g < groups; ++g)
            out[orc_scale_offset(r, g, cols)] = sf_logical[r * groups + g];
}

/* ------------------------------------------------------------------------ */
/* Row producers.  Each takes nrows rows of bf16 input (row stride ld, in     */
/* elements) and writes codes [nrows, cols/2] and logical (unswizzled) block  */
/* scales [nrows, cols/16].  cols is a multiple of 64.                       */
/* ------------------------------------------------------------------------ */

static void quantize_row_values(const float *y, int64_t cols, float gsf, uint8_t *codes_row,
                                uint8_t *sf_row)
{
    for (int64_t b = 0; b < cols / 16; ++b)
        orc_quantize_block(y + 16 * b, gsf, &sf_row[b], &codes_row[8 * b]);
}

/* standalone quantize, e.g. of the attention output ([TRT] commit
 * "quantize the attention output with a bandwidth-bound kernel";
 * [FV-API] quantize). */
void orc_quantize_rows(const uint16_t *x, int64_t nrows, int64_t cols, int64_t ld, float gsf,
                       float *scratch_row, uint8_t *codes, uint8_t *sf)
{
    for (int64_t r = 0; r < nrows; ++r) {
        for (int64_t j = 0; j < cols; ++j)
            scratch_row[j] = orc_bf16_value(x[r * ld + j]);
        quantize_row_values(scratch_row, cols, gsf, codes + r * (cols / 2), sf + r * (cols / 16));
    }
}

/*
 * Sum of squares in the canonical order.  This is the one routine behind every
 * RMS statistic of the oracle (bf16 rows, fp32 rows of the residual fold, and
 * the heads of the QKV epilogue); the order is a definition of this build,
 * fixed here and pinned bit for bit by hand-derived rows, and kernels follow it.
 *
 * The n values (n a multiple of 8) form 8-element chunks, chunk c = values
 * 8c..8c+7.  Chunks are dealt round-robin to `lanes` lanes (chunk c to lane
 * c % lanes).  Each lane keeps eight fp32 partials starting at +0; element e of
 * each of its chunks, chunks in increasing order, goes into partial e through a
 * fused multiply-add ("sequential FMA per thread", [FV-API] introduction).  A
 * lane's total is ((p0+p1)+(p2+p3))+((p4+p5)+(p6+p7)).  The lanes form groups
 * of G = min(lanes, 32) consecutive lanes; inside a group a butterfly -- for
 * o = G/2, ..., 2, 1 every lane adds the total of lane (l xor o) -- leaves each
 * lane holding the group total.  One group: that total is the sum.  Four groups
 * (lanes = 128, the rows): ss = (T_0 + T_1) + (T_2 + T_3).
 * `lanes` is 128 for rows and hd/8 (a power of two up to 32) for heads.
 * Values come from `b16` (bf16 bit patterns, exact in binary32) when it is not
 * NULL, else from `f32`.
 */
static float canonical_sumsq(const uint16_t *b16, const float *f32, int64_t n, int lanes)
{
    int64_t chunks = n / 8;
    float lane[128];
    for (int l = 0; l < lanes; ++l) {
        float p[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
        for (int64_t c = l; c < chunks; c += lanes)
            for (int e = 0; e < 8; ++e) {
                float v = b16 ? orc_bf16_value(b16[8 * c + e]) : f32[8 * c + e];
                p[e] = fmaf(v, v, p[e]);
            }
        lane[l] = ((p[0] + p[1]) + (p[2] + p[3])) + ((p[4] + p[5]) + (p[6] + p[7]));
    }
    int width = lanes < 32 ? lanes : 32;
    float total[4];
    for (int w = 0; w < lanes / width; ++w) {
        float g[32];
        memcpy(g, lane + width * w, sizeof(float) * (size_t)width);
        for (int o = width / 2; o >= 1; o /= 2) {
            float next[32];
            for (int l = 0; l < width; ++l)
                next[l] = g[l] + g[l ^ o];
            memcpy(g, next, sizeof(float) * (size_t)width);
        }
        total[w] = g[0];
    }
    if (lanes / width == 1)
        return total[0];
    return (total[0] + total[1]) + (total[2] + total[3]);
}

/* rstd = fl(1 / fl(sqrt(fl(fl(ss / n) + eps)))): correctly rounded division and
 * square root, eps added after the mean. */
static float rstd_of_sumsq(float ss, int64_t n, float eps)
{
    float mean = ss / (float)n;
    float root = sqrtf(mean + eps);
    return 1.0f / root;
}

/* The canonical sum of squares of n values (bf16 bits or binary32) with the given
 * number of lanes (128 for a row; hd/8 for a head of hd values). */
float orc_sumsq_bf16(const uint16_t *v, int64_t n, int lanes) { return canonical_sumsq(v, NULL, n, lanes); }
float orc_sumsq_f32(const float *v, int64_t n, int lanes) { return canonical_sumsq(NULL, v, n, lanes); }

/* rstd of one bf16 row (128 lanes). */
float orc_row_rstd(const uint16_t *xrow, int64_t cols, float eps)
{
    return rstd_of_sumsq(canonical_sumsq(xrow, NULL, cols, 128), cols, eps);
}

/* rstd of one fp32 row (128 lanes): the residual fold's statistics. */
float orc_row_rstd_f32(const float *row, int64_t cols, float eps)
{
    return rstd_of_sumsq(canonical_sumsq(NULL, row, cols, 128), cols, eps);
}

/*
 * RMSNorm with fp32 statistics, then AdaLN modulation, then NVFP4
 * ([TRT] commit "...emit the packed E2M1 codes and swizzled E4M3 block
 * scales directly" for the AdaLN RMSNorm + modulation producer).
 * The modulation table is bf16 [frames, 2, cols]: [t][0] is the shift and
 * [t][1] the scale.  frame_of_row[i] is the frame of input row i.
 * Per element, one rounding per operation and a single bf16 rounding at the
 * end (products are never fused into the following add):
 *   n = fl(x * rstd); h = fl(n * gamma); a = fl(1 + scale); m = fl(h * a);
 *   o = fl(m + shift); y = bf16(o)
 * y_out (optional, [nrows, cols] bf16 bits) receives y.
 */
void orc_adaln_rows(const uint16_t *x, int64_t nrows, int64_t cols, int64_t ld,
                    const uint16_t *gamma, const uint16_t *table, const int64_t *frame_of_row,
                    float eps, float gsf, float *scratch_row, uint8_t *codes, uint8_t *sf,
                    float *rstd_out, uint16_t *y_out)
{
    for (int64_t r = 0; r < nrows; ++r) {
        const uint16_t *xr = x + r * ld;
        float rstd = orc_row_rstd(xr, cols, eps);
        const uint16_t *shift = table + frame_of_row[r] * 2 * cols;
        const uint16_t *scale = shift + cols;
        for (int64_t j = 0; j < cols; ++j) {
            float n = orc_bf16_value(xr[j]) * rstd;
            float h = n * orc_bf16_value(gamma[j]);
            float a = 1.0f + orc_bf16_value(scale[j]);
            float m = h * a;
            float o = m + orc_bf16_value(shift[j]);
            scratch_row[j] = orc_bf16_round(o);
            if (y_out)
                y_out[r * cols + j] = orc_bf16_bits(o);
        }
        if (rstd_out)
            rstd_out[r] = rstd;
        if (codes)
            quantize_row_values(scratch_row, cols, gsf, codes + r * (cols / 2),
                                sf + r * (cols / 16));
    }
}

/* SwiGLU silu(gate) * up, then NVFP4 ([TRT] SiLU-and-mul producer;
 * [FV-CUH] swiglu_bf16).  y_out as above. */
/*
 * SwiGLU of a value-first packed projection with its bias.
 * [FV-API] swiglu_quantize: o is [M, 2F], value first (columns 0..F-1), gate
 * second, the bias not yet added.  Reading: each half gets its bias in binary32
 * and is rounded to bf16, as the projection's own output would be,
 *   v = bf16(fl(o_v + b_v)),  g = bf16(fl(o_g + b_g))   (no add without a bias)
 * and then the SwiGLU spec: y = bf16(fl(fl(g * sigma(g)) * v)), quantized.
 */
void orc_swiglu_packed_rows(const uint16_t *o, int64_t ld_o, const uint16_t *bias, int64_t nrows,
                            int64_t f, float gsf, float *scratch_row, uint8_t *codes, uint8_t *sf,
                            uint16_t *y_out)
{
    for (int64_t r = 0; r < nrows; ++r) {
        const uint16_t *orow = o + r * ld_o;
        for (int64_t j = 0; j < f; ++j) {
            float v = orc_bf16_value(orow[j]);
            float g = orc_bf16_value(orow[f + j]);
            if (bias) {
                v = orc_bf16_round(v + orc_bf16_value(bias[j]));
                g = orc_bf16_round(g + orc_bf16_value(bias[f + j]));
            }
            float y = orc_swiglu_value(g, v);
            scratch_row[j] = y;
            if (y_out)
                y_out[r * f + j] = orc_bf16_bits(y);
        }
        if (codes)
            quantize_row_values(scratch_row, f, gsf, codes + r * (f / 2), sf + r * (f / 16));
    }
}

/* ------------------------------------------------------------------------ */
/* QKV epilogue: bias + per-head RMSNorm + partial RoPE                     */
/* ------------------------------------------------------------------------ */
/*
 * [FV-API] qkv_epilogue: projected q/k/v [M, H*HD] bf16 with the bias not yet
 * added -> roped q, k and biased v, each [M, H, HD]; cos/sin are bf16 [M, ROT]
 * (the eager path's cos.to(query.dtype)).  [FV-LOG] names the kernel a q/k
 * norm with partial RoPE.  Readings (the pages print only the wrapper):
 *   x' = bf16(fl(x + b))                       every tensor (v stops here)
 *   per head of q and k: rstd over the HD values of x' in the canonical order
 *   with HD/8 lanes (chunk c of the head on lane c, eight fmaf partials, the
 *   lane total, a butterfly over the lanes), rstd = fl(1/fl(sqrt(fl(fl(ss/HD)
 *   + eps)))), no weight (the wrapper takes none), n = bf16(fl(x' * rstd));
 *   rotate-half RoPE on the first ROT values of each head, each bf16 op of the
 *   eager path rounded to bf16:
 *     r_i = -n_{i+ROT/2} (i < ROT/2), n_{i-ROT/2} (ROT/2 <= i < ROT)
 *     out_i = bf16(fl(bf16(fl(n_i * cos_i)) + bf16(fl(r_i * sin_i))))   i < ROT
 *     out_i = n_i                                                         i >= ROT
 *   or, with `interleaved`, the pairs (2j, 2j+1) rotated together ([FlashRT]
 *   commit "...fused RMSNorm+RoPE kernels": interleaved RoPE on the native
 *   [B, S, H, D] layout): r_{2j} = -n_{2j+1}, r_{2j+1} = n_{2j}, same out_i.
 */
/* rstd of one head of hd values (hd a power of two, 16..256): the canonical
 * order with hd/8 lanes, one chunk per lane. */
float orc_head_rstd(const float *v, int64_t hd, float eps)
{
    return rstd_of_sumsq(canonical_sumsq(NULL, v, hd, (int)(hd / 8)), hd, eps);
}

void orc_qkv_epilogue_rows(const uint16_t *x, int64_t ld_x, const uint16_t *bias, int64_t nrows,
                           int64_t heads, int64_t hd, int is_v, const uint16_t *cos_t,
                           const uint16_t *sin_t, int64_t rot, int interleaved, float eps,
                           uint16_t *out)
{
    float xb[1024], n[1024];
    for (int64_t r = 0; r < nrows; ++r) {
        for (int64_t hh = 0; hh < heads; ++hh) {
            const uint16_t *xh = x + r * ld_x + hh * hd;
            const uint16_t *bh = bias + hh * hd;
            uint16_t *oh = out + (r * heads + hh) * hd;
            for (int64_t i = 0; i < hd; ++i)
                xb[i] = orc_bf16_round(orc_bf16_value(xh[i]) + orc_bf16_value(bh[i]));
            if (is_v) {
                for (int64_t i = 0; i < hd; ++i)
                    oh[i] = orc_bf16_bits(xb[i]);
                continue;
            }
            float rstd = orc_head_rstd(xb, hd, eps);
            for (int64_t i = 0; i < hd; ++i)
                n[i] = orc_bf16_round(xb[i] * rstd);
            for (int64_t i = 0; i < hd; ++i) {
                if (i >= rot) {
                    oh[i] = orc_bf16_bits(n[i]);
                    continue;
                }
                float rr;
                if (interleaved)
                    rr = (i & 1) ? n[i - 1] : -n[i + 1];
                else
                    rr = i < rot / 2 ? -n[i + rot / 2] : n[i - rot / 2];
                float a = orc_bf16_round(n[i] * orc_bf16_value(cos_t[r * rot + i]));
                float b = orc_bf16_round(rr * orc_bf16_value(sin_t[r * rot + i]));
                oh[i] = orc_bf16_bits(a + b);
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Residual fold + RMSNorm + AdaLN                                          */
/* ------------------------------------------------------------------------ */
/*
 * [TRT] commit "...norm1 ... from a second table": a block folds its MLP
 * residual into the next block's norm1 kernel, reading the gate from its own
 * AdaLN table while the scale and shift come from the next block's.
 * [FV-API] residual_norm_quantize: in place h += bf16(o + bias) * scale on a
 * contiguous fp32 residual h, then NVFP4 of the normed h.
 *
 * Reading: with the gate g[t] of the row's frame (bf16 table [T, cols]),
 *   u = bf16(fl(o + bias))   (u = o when there is no bias)
 *   h' = fl(h + fl(u * g))   written back to h
 * and then the RMSNorm + AdaLN spec above on the fp32 values h' (the same
 * canonical reduction order, squares by fmaf of fp32 values).
 */
void orc_residual_adaln_rows(float *h, int64_t nrows, int64_t cols, int64_t ld_h,
                             const uint16_t *o, int64_t ld_o, const uint16_t *bias,
                             const uint16_t *gate, const uint16_t *gamma, const uint16_t *table,
                             const int64_t *frame_of_row, float eps, float gsf, float *scratch_row,
                             uint8_t *codes, uint8_t *sf, float *rstd_out, uint16_t *y_out)
{
    for (int64_t r = 0; r < nrows; ++r) {
        float *hr = h + r * ld_h;
        const uint16_t *orow = o + r * ld_o;
        const uint16_t *g = gate + frame_of_row[r] * cols;
        for (int64_t j = 0; j < cols; ++j) {
            float u = bias ? orc_bf16_round(orc_bf16_value(orow[j]) + orc_bf16_value(bias[j]))
                           : orc_bf16_value(orow[j]);
            float t = u * orc_bf16_value(g[j]);
            hr[j] = hr[j] + t;
        }
        float rstd = orc_row_rstd_f32(hr, cols, eps);
        const uint16_t *shift = table + frame_of_row[r] * 2 * cols;
        const uint16_t *scale = shift + cols;
        for (int64_t j = 0; j < cols; ++j) {
            float n = hr[j] * rstd;
            float hh = n * orc_bf16_value(gamma[j]);
            float a = 1.0f + orc_bf16_value(scale[j]);
            float m = hh * a;
            float out = m + orc_bf16_value(shift[j]);
            scratch_row[j] = orc_bf16_round(out);
            if (y_out)
                y_out[r * cols + j] = orc_bf16_bits(out);
        }
        if (rstd_out)
            rstd_out[r] = rstd;
        if (codes)
            quantize_row_values(scratch_row, cols, gsf, codes + r * (cols / 2),
                                sf + r * (cols / 16));
    }
}

void orc_swiglu_rows(const uint16_t *gate, int64_t ld_gate, const uint16_t *up, int64_t ld_up,
                     int64_t nrows, int64_t cols, float gsf, float *scratch_row, uint8_t *codes,
                     uint8_t *sf, uint16_t *y_out)
{
    for (int64_t r = 0; r < nrows; ++r) {
        for (int64_t j = 0; j < cols; ++j) {
            float y = orc_swiglu_value(orc_bf16_value(gate[r * ld_gate + j]),
                                       orc_bf16_value(up[r * ld_up + j]));
            scratch_row[j] = y;
            if (y_out)
                y_out[r * cols + j] = orc_bf16_bits(y);
        }
        if (codes)
            quantize_row_values(scratch_row, cols, gsf, codes + r * (cols / 2),
                                sf + r * (cols / 16));
    }
}

/* ------------------------------------------------------------------------ */
/* Block-scaled NVFP4 GEMM, then the SwiGLU + NVFP4 epilogue                 */
/* ------------------------------------------------------------------------ */
/*
 * [FV-CMP] minimax_h3_swiglu_gemm.cu (launch_gemm_swiglu, h3_epilogue::Store):
 * the FFN-up projection as a block-scaled NVFP4 GEMM whose epilogue applies the
 * SwiGLU on value/gate-paired columns and writes NVFP4 directly.  A is the
 * activation [m, k] and B the weight [n, k], both NVFP4 (E2M1 codes, one E4M3
 * scale per 16 elements along k); n = 2F, and output j pairs column 2j (the
 * value) with column 2j + 1 (the gate).
 *
 * The GEMM: acc[i][j] = fl(sum over k of a_ik * b_jk) with a_ik =
 * E2M1value(code) * E4M3value(scale), each product and the whole sum taken
 * exactly and rounded once to binary32.  (Every element is an integer times
 * 2^-10, every product an integer times 2^-20, so the sum is an exact integer
 * in int64 for k <= 2^19; converting it to binary32 is one correctly rounded
 * conversion, and the scaling by 2^-20 is exact.)  A tensor core adds its
 * partial products in its own order; this exact sum is what it approximates.
 *
 * The epilogue (reading of h3_epilogue::Store with the SwiGLU and the block
 * quantize of this library):
 *   u = bf16(fl(alpha * acc[2j])),  g = bf16(fl(alpha * acc[2j + 1]))
 *   y = bf16(fl(fl(g * sigma(g)) * u)),  sigma(g) = fl(1 / fl(1 + exp_c(-g)))
 * and y [m, F] is block-quantized with the global scale gsf.
 */

/* E2M1value(code) * E4M3value(sf) as an integer times 2^-10.  The E4M3 value
 * is mant * 2^(e - 10) for a normal code (mant = 8 + m) and m * 2^-9 for a
 * subnormal one; the E2M1 magnitude is i / 2 with i in {0,1,2,3,4,6,8,12}. */
static int64_t nvfp4_units(uint8_t code, uint8_t sf)
{
    static const int twice_e2m1[8] = {0, 1, 2, 3, 4, 6, 8, 12};
    int e = (sf >> 3) & 15;
    int m = sf & 7;
    int64_t mant = e == 0 ? m : 8 + m;
    int shift = e == 0 ? 0 : e - 1; /* value * 2^10 = i * mant * 2^shift */
    int64_t v = ((int64_t)twice_e2m1[code & 7] * mant) << shift;
    return (code & 8) ? -v : v;
}

/* One operand row as integers (units of 2^-10): codes [k/2] (even element in
 * the low nibble) and logical scales [k/16]. */
static void nvfp4_row_units(const uint8_t *codes, const uint8_t *sf, int64_t k, int64_t *out)
{
    for (int64_t e = 0; e < k; ++e) {
        uint8_t byte = codes[e / 2];
        uint8_t c = (e % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
        out[e] = nvfp4_units(c, sf[e / 16]);
    }
}

/* acc [m, n] (rows i0..i1 of it) of A codes [m, k/2] with logical scales
 * [m, k/16] and B codes [n, k/2] with logical scales [n, k/16].  a_units is
 * scratch of (i1 - i0) * k int64 (A's rows as integers), b_units of k. */
void orc_nvfp4_gemm_rows(const uint8_t *a, const uint8_t *sfa, int64_t i0, int64_t i1, int64_t k,
                         const uint8_t *b, const uint8_t *sfb, int64_t n, int64_t *a_units,
                         int64_t *b_units, float *acc)
{
    for (int64_t i = i0; i < i1; ++i)
        nvfp4_row_units(a + i * (k / 2), sfa + i * (k / 16), k, a_units + (i - i0) * k);
    for (int64_t j = 0; j < n; ++j) {
        nvfp4_row_units(b + j * (k / 2), sfb + j * (k / 16), k, b_units);
        for (int64_t i = i0; i < i1; ++i) {
            const int64_t *au = a_units + (i - i0) * k;
            int64_t sum = 0;
            for (int64_t e = 0; e < k; ++e)
                sum += au[e] * b_units[e];
            acc[(i - i0) * n + j] = ldexpf((float)sum, -20);
        }
    }
}

/* The SwiGLU + NVFP4 epilogue of nrows rows of acc [nrows, n]: y [nrows, n/2],
 * quantized into codes [nrows, n/4] and logical scales [nrows, n/32]. */
void orc_swiglu_epilogue_rows(const float *acc, int64_t nrows, int64_t n, float alpha, float gsf,
                              float *scratch_row, uint8_t *codes, uint8_t *sf, uint16_t *y_out)
{
    int64_t f = n / 2;
    for (int64_t r = 0; r < nrows; ++r) {
        for (int64_t j = 0; j < f; ++j) {
            float u = orc_bf16_round(alpha * acc[r * n + 2 * j]);
            float g = orc_bf16_round(alpha * acc[r * n + 2 * j + 1]);
            float y = orc_swiglu_value(g, u);
            scratch_row[j] = y;
            if (y_out)
                y_out[r * f + j] = orc_bf16_bits(y);
        }
        if (codes)
            quantize_row_values(scratch_row, f, gsf, codes + r * (f / 2), sf + r * (f / 16));
    }
}

/* Dequantize (checking path): x = fl((E2M1value(c) * E4M3value(sf)) / gsf).
 * The product is exact (at most 2 x 4 significant bits), so there is one
 * rounding: the value an NVFP4 GEMM sees for the element, divided by the
 * global scale. */
void orc_dequantize_rows(const uint8_t *codes, const uint8_t *sf, int64_t nrows, int64_t cols,
                         float gsf, float *out)
{
    for (int64_t r = 0; r < nrows; ++r)
        for (int64_t j = 0; j < cols; ++j) {
            uint8_t byte = codes[r * (cols / 2) + j / 2];
            uint8_t c = (j % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
            float scale = orc_e4m3_value(sf[r * (cols / 16) + j / 16]);
            out[r * cols + j] = (orc_e2m1_value(c) * scale) / gsf;
        }
}

/* ------------------------------------------------------------------------ */
/* Element-wise entry points used by the pin tests                           */
/* ------------------------------------------------------------------------ */

void orc_bf16_bits_array(const float *v, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_bf16_bits(v[i]);
}

void orc_e4m3_encode_array(const float *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e4m3_encode(v[i]);
}

void orc_e2m1_encode_array(const float *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e2m1_encode(v[i]);
}

void orc_exp_array(const float *v, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_exp(v[i]);
}

void orc_swiglu_value_array(const float *g, const float *u, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_swiglu_value(g[i], u[i]);
}
