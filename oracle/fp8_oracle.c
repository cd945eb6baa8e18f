/*
 * fp8_oracle.c -- plain, slow, scalar CPU reference for FP8 scaled quantization.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call this file:
 * only the tests, the smoke check and the benchmark's CPU-baseline leg use it.
 * It shares no code, header, table or constant generator with the CUDA
 * library; it is written from the format definitions and the scaling
 * recipes as the pages state them, one element at a time, in the order the
 * pages give.
 *
 * Sources (page title, section):
 *   "Megatron FP8" §2  FP8 formats E4M3 / E5M2: bias 2^(k-1)-1, max finite
 *                      (2-2^-M)*2^emax, E4M3FN has no Inf and saturates to
 *                      +-448, E5M2 keeps Inf/NaN, min normals 2^-6 / 2^-14.
 *   "Megatron FP8" §3  the set of representable values.
 *   "Megatron FP8" §4  tensor scale: amax = max|x|, s* = amax/FP8_MAX,
 *                      2^margin headroom, clamp to +-FP8_MAX, scale_inv = 1/s
 *                      cached so dequantize is one multiply.
 *   "Megatron FP8" §5  delayed scaling: amax history ring, slot step % len,
 *                      algo max / most_recent, scale 1 while history is 0.
 *   "Megatron FP8" §10 margin semantics; multiplier form fp8_max / amax.
 *   "Megatron FP8" §23 dequantize = fp8 value * scale.
 *   "Low Precision Training and Rollout", "BF16 Training with FP8 Rollout"
 *                      and "FP8 Quick Start": 128x128 blocks, FP32 block
 *                      scales; "MXFP8 (Blackwell only)": the stored block
 *                      factor of block FP8 is the inverse scale.
 *
 * Where the pages are silent or garbled, the reading taken is stated next to
 * the code it governs.
 *
 * Floating point: every fp32 operation below is a single IEEE-754 binary32
 * operation rounded to nearest-even (compile with -ffp-contract=off, no fast
 * math).  Encoding and decoding use fp64 only where the value is exact in
 * fp64 (every fp32 and FP8 value is).
 */
#include <float.h>
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#if !defined(FLT_EVAL_METHOD) || FLT_EVAL_METHOD != 0
#error "the oracle needs fp32 arithmetic evaluated in fp32 (FLT_EVAL_METHOD 0)"
#endif

#define OREF_E4M3 0
#define OREF_E5M2 1
#define OREF_BF16 0
#define OREF_FP32 1
#define OREF_ALGO_MAX 0
#define OREF_ALGO_MOST_RECENT 1

/* ------------------------------------------------------------------------ */
/* Format description ("Megatron FP8" §2)                                    */
/* ------------------------------------------------------------------------ */

static int fmt_exp_bits(int fmt) { return fmt == OREF_E4M3 ? 4 : 5; }
static int fmt_mant_bits(int fmt) { return fmt == OREF_E4M3 ? 3 : 2; }
static int fmt_bias(int fmt) { return (1 << (fmt_exp_bits(fmt) - 1)) - 1; }

/* Classify a code: 0 finite, 1 infinity, 2 NaN.
 * E5M2 follows IEEE: all-ones exponent with zero mantissa is Inf, non-zero
 * mantissa is NaN.  E4M3FN ("FN" = finite + NaN): the all-ones exponent is
 * an ordinary binade except mantissa 111, the only NaN; there is no Inf. */
static int code_class(uint8_t code, int fmt) {
    int E = fmt_exp_bits(fmt), M = fmt_mant_bits(fmt);
    int e = (code >> M) & ((1 << E) - 1);
    int m = code & ((1 << M) - 1);
    if (fmt == OREF_E5M2 && e == (1 << E) - 1) return m == 0 ? 1 : 2;
    if (fmt == OREF_E4M3 && e == (1 << E) - 1 && m == (1 << M) - 1) return 2;
    return 0;
}

/* Exact value of a code, in fp64. */
double oref_decode_f64(uint8_t code, int fmt) {
    int E = fmt_exp_bits(fmt), M = fmt_mant_bits(fmt), bias = fmt_bias(fmt);
    int sign = code >> 7;
    int e = (code >> M) & ((1 << E) - 1);
    int m = code & ((1 << M) - 1);
    double v;
    int cls = code_class(code, fmt);
    if (cls == 2) return NAN;
    if (cls == 1) return sign ? -INFINITY : INFINITY;
    if (e == 0)
        v = ldexp((double)m, 1 - bias - M);          /* subnormal: m * 2^(1-bias-M) */
    else
        v = ldexp((double)((1 << M) + m), e - bias - M); /* (1 + m/2^M) * 2^(e-bias) */
    return sign ? -v : v;
}

float oref_decode(uint8_t code, int fmt) { return (float)oref_decode_f64(code, fmt); }

/* Largest finite value, found by walking all codes (not a stored constant). */
double oref_max_finite(int fmt) {
    double best = 0.0;
    for (int c = 0; c < 256; ++c) {
        if (code_class((uint8_t)c, fmt) != 0) continue;
        double v = oref_decode_f64((uint8_t)c, fmt);
        if (v > best) best = v;
    }
    return best;
}

/* Smallest positive normal value: 2^(1-bias). */
double oref_min_normal(int fmt) { return ldexp(1.0, 1 - fmt_bias(fmt)); }

/* (bias, e_max, max_finite) with e_max the unbiased exponent of the largest
 * finite value -- the triple "Megatron FP8" §2 prints for E4M3 and E5M2. */
void oref_format_stats(int fmt, int* bias, int* e_max, double* max_finite) {
    double mx = oref_max_finite(fmt);
    int ex = 0;
    frexp(mx, &ex); /* mx = f * 2^ex, f in [0.5, 1) */
    *bias = fmt_bias(fmt);
    *e_max = ex - 1;
    *max_finite = mx;
}

/* Code of the largest finite positive value. */
static uint8_t max_code(int fmt) {
    uint8_t best = 0;
    double bv = -1.0;
    for (int c = 0; c < 128; ++c) {
        if (code_class((uint8_t)c, fmt) != 0) continue;
        double v = oref_decode_f64((uint8_t)c, fmt);
        if (v > bv) { bv = v; best = (uint8_t)c; }
    }
    return best;
}

/* Facts about a format, derived once per top-level call from the code walk
 * above (so a per-element loop does not redo the 256-code walk). */
typedef struct {
    int fmt, M, bias;
    double max_finite, min_normal;
    uint8_t max_code;
} fmt_info;

static fmt_info make_info(int fmt) {
    fmt_info f;
    f.fmt = fmt;
    f.M = fmt_mant_bits(fmt);
    f.bias = fmt_bias(fmt);
    f.max_finite = oref_max_finite(fmt);
    f.min_normal = oref_min_normal(fmt);
    f.max_code = max_code(fmt);
    return f;
}

/* The byte a NaN input becomes.  The pages do not say; the reading taken is
 * the positive canonical NaN code 0x7F (all exponent and mantissa bits set)
 * in both formats, sign dropped. */
#define OREF_NAN_CODE 0x7F

/* ------------------------------------------------------------------------ */
/* Encoding: round-to-nearest-even onto the FP8 grid, saturating            */
/* ------------------------------------------------------------------------ */

/* Round a non-negative finite real a (< max finite) to the FP8 grid with
 * ties to even, and return the code of the result (positive sign).
 * Inside a binade [2^e, 2^(e+1)) the grid step is 2^(e-M); below the
 * smallest normal the step is the subnormal quantum 2^(1-bias-M). */
static uint8_t round_to_code(double a, const fmt_info* f) {
    int M = f->M, bias = f->bias;
    int e; /* unbiased exponent of the binade holding a */
    if (a < f->min_normal) {
        e = 1 - bias;
    } else {
        int ex;
        frexp(a, &ex); /* a = g * 2^ex, g in [0.5, 1)  =>  a in [2^(ex-1), 2^ex) */
        e = ex - 1;
    }
    double quantum = ldexp(1.0, e - M);
    double t = a / quantum; /* exact: a has at most 24 significant bits */
    double fl = floor(t);
    double frac = t - fl;
    double r;
    if (frac > 0.5)
        r = fl + 1.0;
    else if (frac < 0.5)
        r = fl;
    else
        r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0; /* tie: to the even neighbour */
    double v = r * quantum; /* the rounded value, exact */

    /* Code of v (v may have moved up into the next binade). */
    if (v == 0.0) return 0;
    if (v < f->min_normal) {
        int m = (int)(v / ldexp(1.0, 1 - bias - M)); /* subnormal mantissa */
        return (uint8_t)m;
    }
    int ex;
    frexp(v, &ex);
    int ev = ex - 1;
    int m = (int)(v / ldexp(1.0, ev - M)) - (1 << M);
    return (uint8_t)(((ev + bias) << M) | m);
}

/* Encode one already-scaled fp32 value p.
 *   NaN           -> canonical NaN code.
 *   |p| >= max    -> +-max code (saturation; this also covers p = +-Inf that
 *                    comes from an fp32 product overflowing).
 *   otherwise     -> nearest grid value, ties to even; results that round to
 *                    zero keep their sign (0x80 for negative). */
static uint8_t encode_saturating(float p, const fmt_info* f) {
    if (isnan(p)) return OREF_NAN_CODE;
    uint8_t sign = signbit(p) ? 0x80 : 0x00;
    double a = fabs((double)p);
    if (a >= f->max_finite) return sign | f->max_code;
    return sign | round_to_code(a, f);
}

uint8_t oref_encode_saturating(float p, int fmt) {
    fmt_info f = make_info(fmt);
    return encode_saturating(p, &f);
}

/* Quantize one input element x with multiplier scale ("Megatron FP8" §4:
 * scale, then clamp to +-FP8_MAX; §2: E5M2 keeps Inf, E4M3FN saturates).
 *   x NaN          -> canonical NaN code.
 *   x = +-Inf      -> E5M2: +-Inf code (0x7C / 0xFC); E4M3FN: +-448.
 *   x finite       -> encode_saturating(fl32(x * scale)).
 * *saturated is set when x is finite and |fl32(x * scale)| > FP8_MAX. */
static uint8_t quantize_element(float x, float scale, const fmt_info* f, int* saturated) {
    *saturated = 0;
    if (isnan(x)) return OREF_NAN_CODE;
    if (isinf(x)) {
        uint8_t sign = signbit(x) ? 0x80 : 0x00;
        if (f->fmt == OREF_E5M2) return sign | 0x7C;
        return sign | f->max_code;
    }
    float p = x * scale; /* one fp32 multiply, round to nearest even */
    if (fabs((double)p) > f->max_finite) *saturated = 1;
    return encode_saturating(p, f);
}

uint8_t oref_quantize_element(float x, float scale, int fmt, int* saturated) {
    fmt_info f = make_info(fmt);
    return quantize_element(x, scale, &f, saturated);
}

/* ------------------------------------------------------------------------ */
/* Input element access                                                      */
/* ------------------------------------------------------------------------ */

/* BF16 is the upper half of an fp32 bit pattern, so widening is exact. */
float oref_bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* fp32 -> BF16, round to nearest even on the dropped 16 bits.  NaN becomes
 * the canonical BF16 NaN 0x7FFF (reading: the pages do not fix NaN bits). */
uint16_t oref_f32_to_bf16(float f) {
    if (isnan(f)) return 0x7FFF;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint32_t upper = u >> 16;
    uint32_t dropped = u & 0xFFFFu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (upper & 1u))) upper += 1u;
    return (uint16_t)upper;
}

static float load_elem(const void* x, int dt, int64_t i) {
    if (dt == OREF_BF16) return oref_bf16_to_f32(((const uint16_t*)x)[i]);
    return ((const float*)x)[i];
}

/* ------------------------------------------------------------------------ */
/* amax and scale ("Megatron FP8" §4, §5, §10)                               */
/* ------------------------------------------------------------------------ */

/* Canonical NaN of an amax that saw a NaN (reading: NaN propagates, as
 * torch's x.abs().max() does; the bits are fixed to the quiet NaN 0x7FC00000). */
static float canonical_nan_f32(void) {
    uint32_t u = 0x7FC00000u;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* amax = max_i |x_i|; an empty input has amax 0. */
float oref_amax(const void* x, int dt, int64_t n) {
    float m = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(load_elem(x, dt, i));
        if (isnan(a)) return canonical_nan_f32();
        if (a > m) m = a;
    }
    return m;
}

/* Current-scaling factor from an amax, multiplier convention:
 *   scale     = fl32( fl32(FP8_MAX / amax) * 2^-margin )
 *   scale_inv = fl32( 1 / scale )
 * Readings (the pages leave these open):
 *   amax == 0, negative, NaN or Inf   -> scale = scale_inv = 1
 *     ("Megatron FP8" §5: scale 1 while the history maximum is 0);
 *   scale above FLT_MAX (overflow)    -> FLT_MAX;
 *   scale below FLT_MIN               -> FLT_MIN,
 * so scale and scale_inv are always finite and positive. */
void oref_compute_scale(float amax, int fmt, int margin, float* scale, float* scale_inv) {
    if (!(amax > 0.0f) || isinf(amax)) {
        *scale = 1.0f;
        *scale_inv = 1.0f;
        return;
    }
    float fp8_max = (float)oref_max_finite(fmt);
    float s = fp8_max / amax;                 /* fp32 division, round to nearest */
    float headroom = ldexpf(1.0f, -margin);   /* exact power of two, |margin| <= 126 */
    s = s * headroom;                         /* fp32 multiply, round to nearest */
    if (s > FLT_MAX) s = FLT_MAX;
    if (s < FLT_MIN) s = FLT_MIN;
    *scale = s;
    *scale_inv = 1.0f / s;
}

/* ------------------------------------------------------------------------ */
/* Per-tensor quantize, cast-transpose, delayed update                      */
/* ------------------------------------------------------------------------ */

/* q[i] = quantize(x[i], scale); returns the saturated-element count. */
uint64_t oref_quantize(const void* x, int dt, int64_t n, int fmt, float scale, uint8_t* q) {
    fmt_info f = make_info(fmt);
    uint64_t sat = 0;
    for (int64_t i = 0; i < n; ++i) {
        int s;
        q[i] = quantize_element(load_elem(x, dt, i), scale, &f, &s);
        sat += (uint64_t)s;
    }
    return sat;
}

/* Rowwise and columnwise copies under one scale (the columnwise copy is the
 * layout a transposed FP8 GEMM operand needs; "Megatron FP8" §6 and the
 * columnwise storage of "[Pytorch][Common] Hybrid quantization #2817").
 *   q_row[r*cols + c] = quantize(x[r*cols + c])
 *   q_col[c*rows + r] = quantize(x[r*cols + c])
 * Each copy is computed from x on its own. */
void oref_cast_transpose(const void* x, int dt, int64_t rows, int64_t cols, int fmt, float scale,
                         uint8_t* q_row, uint8_t* q_col) {
    fmt_info f = make_info(fmt);
    int s;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c)
            q_row[r * cols + c] = quantize_element(load_elem(x, dt, r * cols + c), scale, &f, &s);
    for (int64_t c = 0; c < cols; ++c)
        for (int64_t r = 0; r < rows; ++r)
            q_col[c * rows + r] = quantize_element(load_elem(x, dt, r * cols + c), scale, &f, &s);
}

/* Delayed-scaling update ("Megatron FP8" §5, update_fp8_meta):
 *   1. if new_amax is given, history[step % len] = *new_amax;
 *   2. eff = max(history) for algo max, history[step % len] for most_recent
 *      (max propagates NaN, like torch's max);
 *   3. scale / scale_inv from eff as in oref_compute_scale. */
void oref_update_delayed(float* history, int len, int64_t step, const float* new_amax, int algo,
                         int fmt, int margin, float* scale, float* scale_inv) {
    int64_t slot = step % len;
    if (new_amax) history[slot] = *new_amax;
    float eff;
    if (algo == OREF_ALGO_MAX) {
        eff = history[0];
        for (int i = 1; i < len; ++i) {
            if (isnan(eff)) break;
            if (isnan(history[i]) || history[i] > eff) eff = history[i];
        }
    } else {
        eff = history[slot];
    }
    oref_compute_scale(eff, fmt, margin, scale, scale_inv);
}

/* ------------------------------------------------------------------------ */
/* Blockwise quantize and dequantize                                        */
/* ------------------------------------------------------------------------ */

/* Block-scaled quantize: for every br x bc block of the row-major [rows,cols]
 * input, amax over the block's elements (edge blocks: the elements that
 * exist), scale and scale_inv as in oref_compute_scale with margin 0, codes
 * with that block's scale.  scale_inv is stored row-major
 * [ceil(rows/br), ceil(cols/bc)]. */
void oref_quantize_block(const void* x, int dt, int64_t rows, int64_t cols, int br, int bc, int fmt,
                         uint8_t* q, float* scale_inv_out) {
    fmt_info f = make_info(fmt);
    int64_t nbr = (rows + br - 1) / br, nbc = (cols + bc - 1) / bc;
    for (int64_t bi = 0; bi < nbr; ++bi) {
        for (int64_t bj = 0; bj < nbc; ++bj) {
            int64_t r0 = bi * br, c0 = bj * bc;
            int64_t r1 = r0 + br < rows ? r0 + br : rows;
            int64_t c1 = c0 + bc < cols ? c0 + bc : cols;
            float amax = 0.0f;
            int saw_nan = 0;
            for (int64_t r = r0; r < r1; ++r)
                for (int64_t c = c0; c < c1; ++c) {
                    float a = fabsf(load_elem(x, dt, r * cols + c));
                    if (isnan(a)) saw_nan = 1;
                    else if (a > amax) amax = a;
                }
            if (saw_nan) amax = canonical_nan_f32();
            float scale, scale_inv;
            oref_compute_scale(amax, fmt, 0, &scale, &scale_inv);
            scale_inv_out[bi * nbc + bj] = scale_inv;
            int s;
            for (int64_t r = r0; r < r1; ++r)
                for (int64_t c = c0; c < c1; ++c)
                    q[r * cols + c] = quantize_element(load_elem(x, dt, r * cols + c), scale, &f, &s);
        }
    }
}

/* Dequantize ("Megatron FP8" §4 and §23): y = decode(q) * scale_inv, one
 * fp32 multiply, then (BF16 output) one round-to-nearest-even to BF16.
 * br = bc = 0 means one per-tensor scale_inv[0]; otherwise scale_inv is the
 * row-major [ceil(rows/br), ceil(cols/bc)] block grid.
 * A NaN result is written as the canonical NaN of the output type (BF16
 * 0x7FFF, fp32 0x7FFFFFFF) -- a reading, the pages do not fix NaN bits. */
void oref_dequantize(const uint8_t* q, int fmt, int64_t rows, int64_t cols, const float* scale_inv,
                     int br, int bc, void* y, int out_dt) {
    int64_t nbc = bc > 0 ? (cols + bc - 1) / bc : 1;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < cols; ++c) {
            float si = (br > 0) ? scale_inv[(r / br) * nbc + (c / bc)] : scale_inv[0];
            float v = oref_decode(q[r * cols + c], fmt) * si; /* fp32 multiply */
            if (out_dt == OREF_BF16) {
                ((uint16_t*)y)[r * cols + c] = oref_f32_to_bf16(v);
            } else {
                if (isnan(v)) {
                    uint32_t u = 0x7FFFFFFFu;
                    memcpy(&((float*)y)[r * cols + c], &u, sizeof u);
                } else {
                    ((float*)y)[r * cols + c] = v;
                }
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* MXFP8: one E8M0 power-of-two scale per 32 consecutive elements           */
/* ------------------------------------------------------------------------ */
/* "Megatron FP8" §10 and §16: every 32 consecutive elements share one E8M0
 * scale -- 8 exponent bits, no mantissa, no sign, 2^-127 .. 2^127 -- the OCP
 * Microscaling (MX) format; applying it is an exponent add.  "Low Precision
 * Training and Rollout", "MXFP8 (Blackwell only)": E4M3 values with UE8M0
 * scales per 32-element group.
 *
 * Readings (the pages give the format, not the rule that picks the scale):
 *   - the OCP MX rule: shared_exp = floor(log2(amax_block)) - emax_elem,
 *     emax_elem = unbiased exponent of the element format's largest finite
 *     value (8 for E4M3, 15 for E5M2), clamped to [-127, 127]; an all-zero
 *     block takes -127;
 *   - elements: encode_saturating(fl32(x * 2^-shared_exp));
 *   - a block holding a NaN or an infinity gets the NaN scale code 0xFF and
 *     every element of that block the NaN code 0x7F;
 *   - E8M0 code = shared_exp + 127; code 0xFF is NaN. */

#define OREF_MX_BLOCK 32

/* E8M0 value: 2^(code - 127); code 255 is NaN. */
double oref_e8m0_decode(uint8_t code) {
    if (code == 0xFF) return NAN;
    return ldexp(1.0, (int)code - 127);
}

/* The shared exponent of a block from its amax (finite, >= 0). */
static int mx_shared_exp(double amax, const fmt_info* f) {
    if (amax == 0.0) return -127;
    int ex;
    frexp(amax, &ex); /* amax in [2^(ex-1), 2^ex) => floor(log2(amax)) = ex - 1 */
    int mex;
    frexp(f->max_finite, &mex);
    int e_max_elem = mex - 1; /* 8 for E4M3 (448 = 1.75 * 2^8), 15 for E5M2 */
    int se = (ex - 1) - e_max_elem;
    if (se < -127) se = -127;
    if (se > 127) se = 127;
    return se;
}

/* Rowwise MX quantize of a row-major [rows, cols] input: blocks are 32
 * consecutive elements of a row (the last block of a row may be shorter);
 * scales are row-major [rows, ceil(cols / 32)] E8M0 codes. */
void oref_quantize_mx(const void* x, int dt, int64_t rows, int64_t cols, int fmt, uint8_t* q, uint8_t* scales) {
    fmt_info f = make_info(fmt);
    int64_t nb = (cols + OREF_MX_BLOCK - 1) / OREF_MX_BLOCK;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            int64_t c0 = b * OREF_MX_BLOCK, c1 = c0 + OREF_MX_BLOCK < cols ? c0 + OREF_MX_BLOCK : cols;
            double amax = 0.0;
            int special = 0;
            for (int64_t c = c0; c < c1; ++c) {
                double v = fabs((double)load_elem(x, dt, r * cols + c));
                if (isnan(v) || isinf(v)) special = 1;
                else if (v > amax) amax = v;
            }
            if (special) {
                scales[r * nb + b] = 0xFF;
                for (int64_t c = c0; c < c1; ++c) q[r * cols + c] = OREF_NAN_CODE;
                continue;
            }
            int se = mx_shared_exp(amax, &f);
            scales[r * nb + b] = (uint8_t)(se + 127);
            float m = (float)ldexp(1.0, -se); /* 2^-se, exact in fp32 for |se| <= 127 */
            for (int64_t c = c0; c < c1; ++c) {
                float p = load_elem(x, dt, r * cols + c) * m; /* one fp32 multiply */
                q[r * cols + c] = encode_saturating(p, &f);
            }
        }
    }
}

/* MX dequantize (rowwise layout): y = decode(q) * 2^(scale - 127), one fp32
 * multiply, then BF16 (round to nearest even) or fp32.  A NaN scale makes
 * the block NaN; NaN results use the canonical NaN of the output type. */
void oref_dequantize_mx(const uint8_t* q, const uint8_t* scales, int64_t rows, int64_t cols, int fmt, void* y,
                        int out_dt) {
    int64_t nb = (cols + OREF_MX_BLOCK - 1) / OREF_MX_BLOCK;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < cols; ++c) {
            float s = (float)oref_e8m0_decode(scales[r * nb + c / OREF_MX_BLOCK]);
            float v = oref_decode(q[r * cols + c], fmt) * s;
            if (out_dt == OREF_BF16) {
                ((uint16_t*)y)[r * cols + c] = oref_f32_to_bf16(v);
            } else if (isnan(v)) {
                uint32_t u = 0x7FFFFFFFu;
                memcpy(&((float*)y)[r * cols + c], &u, sizeof u);
            } else {
                ((float*)y)[r * cols + c] = v;
            }
        }
    }
}

/* Lossless re-blocking of 128 x 128 block scales into 1 x 32 E8M0 scales
 * ("Low Precision Training and Rollout", "MXFP8 (Blackwell only)": block-FP8
 * [128,128] sources are rescaled to [1,32] without dequantizing when the
 * scales are powers of two).  The codes are unchanged; each 1 x 32 block takes
 * the E8M0 code of its 128 x 128 block's scale_inv.  A scale_inv that is not
 * a power of two in [2^-127, 2^127] cannot be represented: its blocks get
 * 0xFF and the function returns how many 128 x 128 blocks were like that. */
int64_t oref_block128_scales_to_mx(const float* scale_inv, int64_t rows, int64_t cols, uint8_t* mx_scales) {
    int64_t nbc128 = (cols + 127) / 128, nb32 = (cols + OREF_MX_BLOCK - 1) / OREF_MX_BLOCK;
    int64_t bad = 0;
    int64_t nbr128 = (rows + 127) / 128;
    for (int64_t i = 0; i < nbr128; ++i)
        for (int64_t j = 0; j < nbc128; ++j) {
            double s = (double)scale_inv[i * nbc128 + j];
            int ex;
            double frac = frexp(s, &ex); /* s = frac * 2^ex, frac in [0.5, 1) */
            if (!(s > 0.0) || isinf(s) || frac != 0.5 || ex - 1 < -127 || ex - 1 > 127) ++bad;
        }
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb32; ++b) {
            double s = (double)scale_inv[(r / 128) * nbc128 + (b * OREF_MX_BLOCK) / 128];
            int ex;
            double frac = frexp(s, &ex);
            uint8_t code = 0xFF;
            if (s > 0.0 && !isinf(s) && frac == 0.5 && ex - 1 >= -127 && ex - 1 <= 127) code = (uint8_t)(ex - 1 + 127);
            mx_scales[r * nb32 + b] = code;
        }
    return bad;
}

/* ------------------------------------------------------------------------ */
/* Hybrid per-direction quantization                                         */
/* ------------------------------------------------------------------------ */
/* "[Pytorch][Common] Hybrid quantization #2817": the rowwise and columnwise
 * copies may use different formats and scalings (per-tensor Float8, any
 * per-direction combination), and the columnwise copy is quantized either
 * from the original tensor (columnwise_source = original) or from the
 * dequantized rowwise value (columnwise_source = rowwise_dequantized).
 * Reading: the dequantized rowwise value is what fp8_dequantize produces --
 * fl32(decode(q_row) * fl32(1 / scale_row)) rounded to BF16 -- and the
 * columnwise copy is written transposed [cols, rows], as in cast-transpose. */
#define OREF_SRC_ORIGINAL 0
#define OREF_SRC_ROWWISE_DEQUANTIZED 1

void oref_quantize_hybrid(const void* x, int dt, int64_t rows, int64_t cols, int fmt_row, float scale_row,
                          int fmt_col, float scale_col, int source, uint8_t* q_row, uint8_t* q_col) {
    fmt_info fr = make_info(fmt_row), fc = make_info(fmt_col);
    float scale_inv_row = 1.0f / scale_row;
    int s;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c)
            q_row[r * cols + c] = quantize_element(load_elem(x, dt, r * cols + c), scale_row, &fr, &s);
    for (int64_t c = 0; c < cols; ++c)
        for (int64_t r = 0; r < rows; ++r) {
            float v;
            if (source == OREF_SRC_ORIGINAL) {
                v = load_elem(x, dt, r * cols + c);
            } else {
                uint8_t code = quantize_element(load_elem(x, dt, r * cols + c), scale_row, &fr, &s);
                float y = oref_decode(code, fmt_row) * scale_inv_row; /* fp32 multiply */
                v = oref_bf16_to_f32(oref_f32_to_bf16(y));            /* the BF16 dequantized value */
            }
            q_col[c * rows + r] = quantize_element(v, scale_col, &fc, &s);
        }
}
