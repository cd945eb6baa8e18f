// fp8q_device.cuh -- device helpers of the sm_103a FP8 quantization kernels.
//
// Numerics ("Megatron FP8" §2, §4): one fp32 multiply x * scale rounded to
// nearest-even (__fmul_rn, never contracted), then one round-to-nearest-even
// saturating conversion to E4M3FN / E5M2 (cvt.rn.satfinite, two values per
// instruction).  Inf / NaN inputs and the saturation count are handled off
// the fast path: a chunk whose largest |x| bit pattern is Inf/NaN, or whose
// largest |x| * scale exceeds FP8_MAX, is re-done element by element.  Both
// tests are exact because fl32(|x| * s) is monotone in |x|.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "fp8q.h"

namespace fp8q {

constexpr int kE4M3 = FP8_E4M3;
constexpr int kE5M2 = FP8_E5M2;

// Largest finite magnitude of each format ("Megatron FP8" §2).
template <int FMT> struct Fmt;
template <> struct Fmt<kE4M3> {
    static constexpr float kMax = 448.0f;
    static constexpr uint32_t kMaxCode = 0x7E;  // S.1111.110
    static constexpr uint32_t kInfCode = 0x7E;  // no Inf: +-Inf saturates
};
template <> struct Fmt<kE5M2> {
    static constexpr float kMax = 57344.0f;
    static constexpr uint32_t kMaxCode = 0x7B;  // S.11110.11
    static constexpr uint32_t kInfCode = 0x7C;  // S.11111.00
};
constexpr uint32_t kNaNCode = 0x7F;

// ---------------------------------------------------------------- conversions

// Two fp32 -> two FP8 codes in the low 16 bits: `lo` in bits 0-7, `hi` in 8-15.
// cvt with two f32 sources puts its first source in the upper half.
template <int FMT>
__device__ __forceinline__ uint32_t cvt2(float lo, float hi) {
    uint16_t r;
    if constexpr (FMT == kE4M3)
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Four fp32 -> four FP8 codes in one word (a in bits 0-7, b 8-15, c 16-23,
// d 24-31): two two-value converts written into the halves of one register.
template <int FMT>
__device__ __forceinline__ uint32_t cvt4(float a, float b, float c, float d) {
    uint32_t r;
    if constexpr (FMT == kE4M3)
        asm("{\n\t.reg .b16 lo, hi;\n\t"
            "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
            "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
            "mov.b32 %0, {lo, hi};\n\t}"
            : "=r"(r) : "f"(a), "f"(b), "f"(c), "f"(d));
    else
        asm("{\n\t.reg .b16 lo, hi;\n\t"
            "cvt.rn.satfinite.e5m2x2.f32 lo, %2, %1;\n\t"
            "cvt.rn.satfinite.e5m2x2.f32 hi, %4, %3;\n\t"
            "mov.b32 %0, {lo, hi};\n\t}"
            : "=r"(r) : "f"(a), "f"(b), "f"(c), "f"(d));
    return r;
}

// Two FP8 codes (low 16 bits of `c2`) -> two exact f16 values (f16x2).
template <int FMT>
__device__ __forceinline__ uint32_t fp8x2_to_f16x2(uint32_t c2) {
    uint32_t r;
    if constexpr (FMT == kE4M3) {
        uint16_t in = (uint16_t)c2;
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(in));
    } else {
        // E5M2 is the upper byte of binary16: place each code in the high byte.
        r = __byte_perm(c2, 0u, 0x1404);  // bytes: [0, c0, 0, c1]
    }
    return r;
}

__device__ __forceinline__ float f16_lo_to_f32(uint32_t h2) {
    float f;
    asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %1; cvt.f32.f16 %0, lo; }" : "=f"(f) : "r"(h2));
    return f;
}
__device__ __forceinline__ float f16_hi_to_f32(uint32_t h2) {
    float f;
    asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %1; cvt.f32.f16 %0, hi; }" : "=f"(f) : "r"(h2));
    return f;
}

// Two fp32 -> BF16x2 (round to nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// BF16 pair packed in a word -> fp32 (exact).
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// a * s and b * s, each the round-to-nearest-even fp32 product (subnormals
// kept), in one packed two-lane multiply (mul.rn.f32x2, sm_100 and later):
// the same values as two __fmul_rn calls, half the multiply instructions.
__device__ __forceinline__ float2 fmul2_rn(float a, float b, float s) {
    unsigned long long r;
    asm("{\n\t.reg .b64 x, y;\n\t"
        "mov.b64 x, {%1, %2};\n\t"
        "mov.b64 y, {%3, %3};\n\t"
        "mul.rn.f32x2 %0, x, y;\n\t}"
        : "=l"(r) : "r"(__float_as_uint(a)), "r"(__float_as_uint(b)), "r"(__float_as_uint(s)));
    return make_float2(__uint_as_float((uint32_t)r), __uint_as_float((uint32_t)(r >> 32)));
}

// Lane-wise unsigned 16-bit maximum of two BF16 pairs.
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// |x| bit patterns of a BF16 pair; fold a u16x2 max into one fp32 bit pattern.
__device__ __forceinline__ uint32_t abs_bf16x2(uint32_t w) { return w & 0x7FFF7FFFu; }
__device__ __forceinline__ uint32_t fold_u16x2_to_f32bits(uint32_t m) {
    uint32_t a = m & 0xFFFFu, b = m >> 16;
    return (a > b ? a : b) << 16;
}

// Exact 2^k as fp32 for -126 <= k <= 127.
__device__ __forceinline__ float exp2i(int k) { return __uint_as_float((uint32_t)(k + 127) << 23); }

// -------------------------------------------------------------- scale rule

// Current scale from an amax bit pattern ("Megatron FP8" §4, §10; the
// multiplier form FP8_MAX / amax with 2^-margin headroom).
template <int FMT>
__device__ __forceinline__ void scale_from_amax(float amax, int margin, float* scale, float* scale_inv) {
    if (!(amax > 0.0f) || isinf(amax)) {
        *scale = 1.0f;
        *scale_inv = 1.0f;
        return;
    }
    float s = __fdiv_rn(Fmt<FMT>::kMax, amax);
    s = __fmul_rn(s, exp2i(-margin));
    if (s > 3.402823466e+38f) s = 3.402823466e+38f;  // +Inf -> FLT_MAX
    if (s < 1.175494351e-38f) s = 1.175494351e-38f;  // below FLT_MIN -> FLT_MIN
    *scale = s;
    *scale_inv = __fdiv_rn(1.0f, s);
}

__device__ __forceinline__ float scale_from_amax_rt(int fmt, float amax, int margin, float* scale_inv) {
    float s;
    if (fmt == kE4M3) scale_from_amax<kE4M3>(amax, margin, &s, scale_inv);
    else scale_from_amax<kE5M2>(amax, margin, &s, scale_inv);
    return s;
}

// ------------------------------------------- block scales of a BF16 amax
//
// A BF16 magnitude a = (1 + i/128) * 2^(E-127) has a 7-bit fraction i, so
// FP8_MAX / a = T[i] * 2^(127-E) with T[i] = FP8_MAX / (1 + i/128): rounding
// commutes with the power of two while the result stays a normal fp32
// number, so RN(FP8_MAX / a) = RN(T[i]) * 2^(127-E), and likewise
// RN(1 / s) = RN(1 / RN(T[i])) * 2^(E-127).  The two 128-entry tables per
// format are built at compile time in integer arithmetic with round half to
// even, so they hold what a correctly rounded fp32 division gives; two table
// reads and two exponent adds replace the two divisions of the scale rule for
// every block of BF16 data (margin 0, the block recipes' rule).

// RN-even fp32 bit pattern of num / den for positive integers whose quotient
// is a normal fp32 number and for which num * 2^48 and den * 2^48 fit in 64 bits.
constexpr uint32_t rn_quotient_bits(uint64_t num, uint64_t den) {
    int k = 0;  // quotient = q * 2^-k
    while (num < (den << 23)) { num <<= 1; ++k; }
    while (num >= (den << 24)) { den <<= 1; --k; }
    uint64_t q = num / den;
    const uint64_t r = num % den;
    if (2 * r > den || (2 * r == den && (q & 1))) ++q;
    if (q == (1ull << 24)) { q >>= 1; --k; }
    return (uint32_t)((150 - k) << 23) | (uint32_t)(q - (1ull << 23));
}

struct Bf16ScaleTables {
    uint32_t s[2][128];   // RN(FP8_MAX / (1 + i/128)), per format
    uint32_t si[2][128];  // RN(1 / s)
};

constexpr Bf16ScaleTables make_bf16_scale_tables() {
    Bf16ScaleTables t{};
    for (int f = 0; f < 2; ++f) {
        const uint64_t fmax = f == kE4M3 ? 448 : 57344;
        for (int i = 0; i < 128; ++i) {
            const uint32_t sb = rn_quotient_bits(fmax * 128, 128 + (uint64_t)i);
            t.s[f][i] = sb;
            // s = (2^23 + m) * 2^(e - 150), so 1 / s = 2^(150 - e) / (2^23 + m)
            t.si[f][i] = rn_quotient_bits(1ull << (150 - (sb >> 23)), (1ull << 23) | (sb & 0x7FFFFFu));
        }
    }
    return t;
}

static __device__ const Bf16ScaleTables g_bf16_scale_tables = make_bf16_scale_tables();

// One format's tables in shared memory: word i < 128 is s[i], word 128 + i is
// si[i].  A kernel reads its word of the table (table_word, one per thread of
// a 256-thread CTA) before its dependency wait -- the tables are constants that
// no kernel writes -- stores it after issuing its own loads, and synchronises
// before the first lookup, so the lookups are shared-memory reads.
template <int FMT>
__device__ __forceinline__ uint32_t table_word(int t) {
    return t < 128 ? __ldg(&g_bf16_scale_tables.s[FMT][t]) : __ldg(&g_bf16_scale_tables.si[FMT][t - 128]);
}

// scale and scale_inv of a block whose amax bits are those of a BF16 value
// (low 16 bits zero), margin 0, from the shared table `tab`: exactly what
// scale_from_amax gives.  Any other amax (fp32 data, zero, subnormal, Inf,
// NaN) and results outside the normal range go through scale_from_amax.
template <int FMT>
__device__ __forceinline__ void block_scale_bf16(const uint32_t* tab, uint32_t bits, float* scale, float* scale_inv) {
    const int e = (int)(bits >> 23);
    if ((bits & 0xFFFFu) == 0 && e >= 1 && e <= 254) {
        const uint32_t i = (bits >> 16) & 0x7Fu;
        const uint32_t sb = tab[i], ib = tab[128 + i];
        const int es = (int)(sb >> 23) + 127 - e, ei = (int)(ib >> 23) + e - 127;
        if (es >= 1 && es <= 254 && ei >= 1 && ei <= 254) {
            *scale = __uint_as_float(((uint32_t)es << 23) | (sb & 0x7FFFFFu));
            *scale_inv = __uint_as_float(((uint32_t)ei << 23) | (ib & 0x7FFFFFu));
            return;
        }
    }
    scale_from_amax<FMT>(__uint_as_float(bits), 0, scale, scale_inv);
}

// ------------------------------------------------------- element-exact path

// One element with every special case spelled out; used by the slow path.
template <int FMT>
__device__ __forceinline__ uint32_t quant_one(float x, float scale, uint32_t* sat) {
    uint32_t xb = __float_as_uint(x);
    uint32_t sign = (xb >> 24) & 0x80u;
    if (isnan(x)) { *sat = 0; return kNaNCode; }
    if (isinf(x)) { *sat = 0; return sign | Fmt<FMT>::kInfCode; }
    float p = __fmul_rn(x, scale);
    *sat = fabsf(p) > Fmt<FMT>::kMax ? 1u : 0u;
    return cvt2<FMT>(p, 0.0f) & 0xFFu;
}

// ------------------------------------------------------------ 8 BF16 -> 8 codes

// Result of converting one 16-byte chunk (8 BF16) into 8 codes.
struct Codes8 {
    uint32_t lo, hi;  // codes 0-3, 4-7 (code i in byte i % 4)
};

// Convert 8 BF16 values (4 words) with `scale`.  `absmax` receives the u16x2
// max of |x| over the chunk.  Special values and saturation are fixed up by
// fixup_bf16x8 when the caller's chunk test asks for it.
template <int FMT>
__device__ __forceinline__ Codes8 cvt_bf16x8(uint4 v, float scale, uint32_t* absmax) {
    Codes8 c;
    const float2 p0 = fmul2_rn(bf16lo(v.x), bf16hi(v.x), scale);
    const float2 p1 = fmul2_rn(bf16lo(v.y), bf16hi(v.y), scale);
    const float2 p2 = fmul2_rn(bf16lo(v.z), bf16hi(v.z), scale);
    const float2 p3 = fmul2_rn(bf16lo(v.w), bf16hi(v.w), scale);
    c.lo = cvt4<FMT>(p0.x, p0.y, p1.x, p1.y);
    c.hi = cvt4<FMT>(p2.x, p2.y, p3.x, p3.y);
    *absmax = max_u16x2(max_u16x2(abs_bf16x2(v.x), abs_bf16x2(v.y)),
                        max_u16x2(abs_bf16x2(v.z), abs_bf16x2(v.w)));
    return c;
}

// The same 8 codes without the |x| maximum, for callers that already know
// whether the values hold Inf / NaN (the block kernels, from the block amax).
template <int FMT>
__device__ __forceinline__ Codes8 cvt_bf16x8_nomax(uint4 v, float scale) {
    Codes8 c;
    const float2 p0 = fmul2_rn(bf16lo(v.x), bf16hi(v.x), scale);
    const float2 p1 = fmul2_rn(bf16lo(v.y), bf16hi(v.y), scale);
    const float2 p2 = fmul2_rn(bf16lo(v.z), bf16hi(v.z), scale);
    const float2 p3 = fmul2_rn(bf16lo(v.w), bf16hi(v.w), scale);
    c.lo = cvt4<FMT>(p0.x, p0.y, p1.x, p1.y);
    c.hi = cvt4<FMT>(p2.x, p2.y, p3.x, p3.y);
    return c;
}

// True when the chunk needs the element-exact path: some |x| is Inf/NaN, or
// (when counting saturation) the largest |x| * scale exceeds FP8_MAX.
template <int FMT, bool COUNT_SAT>
__device__ __forceinline__ bool chunk_needs_fixup(uint32_t absmax_f32bits, float scale) {
    if (absmax_f32bits >= 0x7F800000u) return true;
    if constexpr (COUNT_SAT) {
        return __fmul_rn(__uint_as_float(absmax_f32bits), scale) > Fmt<FMT>::kMax;
    } else {
        return false;
    }
}

// Redo 8 BF16 elements exactly.  The out-of-line part returns codes and the
// saturated count by value, so the caller's code words never need a stack
// slot (a pointer argument would force them into local memory on every chunk,
// fixed up or not); the inline wrapper keeps the call sites' form.
struct Fixed8 {
    uint32_t lo, hi, sat;
};

template <int FMT>
__device__ __noinline__ Fixed8 fixup_bf16x8_exact(uint4 v, float scale) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    Fixed8 r = {0u, 0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float x = (i & 1) ? bf16hi(w[i >> 1]) : bf16lo(w[i >> 1]);
        uint32_t s;
        const uint32_t code = quant_one<FMT>(x, scale, &s);
        r.sat += s;
        if (i < 4) r.lo |= code << (8 * i);
        else r.hi |= code << (8 * (i - 4));
    }
    return r;
}

// Returns the saturated-element count; *c receives the 8 codes.
template <int FMT>
__device__ __forceinline__ uint32_t fixup_bf16x8(uint4 v, float scale, Codes8* c) {
    const Fixed8 r = fixup_bf16x8_exact<FMT>(v, scale);
    c->lo = r.lo;
    c->hi = r.hi;
    return r.sat;
}

// ----------------------------------------------------------- fp32 inputs

// Convert 4 fp32 values into 4 codes (one word).
template <int FMT>
__device__ __forceinline__ uint32_t cvt_f32x4(float4 v, float scale, uint32_t* absmax) {
    const float2 p0 = fmul2_rn(v.x, v.y, scale);
    const float2 p1 = fmul2_rn(v.z, v.w, scale);
    uint32_t a = __float_as_uint(v.x) & 0x7FFFFFFFu, b = __float_as_uint(v.y) & 0x7FFFFFFFu;
    uint32_t c = __float_as_uint(v.z) & 0x7FFFFFFFu, d = __float_as_uint(v.w) & 0x7FFFFFFFu;
    *absmax = umax(umax(a, b), umax(c, d));
    return cvt4<FMT>(p0.x, p0.y, p1.x, p1.y);
}

// Redo 4 fp32 elements exactly (by value, as fixup_bf16x8_exact).
template <int FMT>
__device__ __noinline__ uint2 fixup_f32x4_exact(float4 v, float scale) {
    const float e[4] = {v.x, v.y, v.z, v.w};
    uint32_t out = 0, sat = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t s;
        out |= quant_one<FMT>(e[i], scale, &s) << (8 * i);
        sat += s;
    }
    return make_uint2(out, sat);
}

// Returns the saturated-element count; *code4 receives the 4 codes.
template <int FMT>
__device__ __forceinline__ uint32_t fixup_f32x4(float4 v, float scale, uint32_t* code4) {
    const uint2 r = fixup_f32x4_exact<FMT>(v, scale);
    *code4 = r.x;
    return r.y;
}

// ----------------------------------------------------------- reductions

__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) { return __reduce_max_sync(0xFFFFFFFFu, v); }
__device__ __forceinline__ uint32_t warp_sum_u32(uint32_t v) { return __reduce_add_sync(0xFFFFFFFFu, v); }

// Block-wide max / sum for blockDim.x a multiple of 32 (<= 1024).  `smem`
// holds 32 words; the result is valid in every thread.
__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, uint32_t* smem) {
    v = warp_max_u32(v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    __syncthreads();
    if (lane == 0) smem[warp] = v;
    __syncthreads();
    v = lane < nw ? smem[lane] : 0u;
    return warp_max_u32(v);
}

__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long v, unsigned long long* smem) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    __syncthreads();
    if (lane == 0) smem[warp] = v;
    __syncthreads();
    v = lane < nw ? smem[lane] : 0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// ------------------------------------------------------ reductions across CTAs

// Programmatic dependent launch: every kernel of the library is launched so
// that it may become resident while the previous kernel on the stream drains.
// It waits here, before touching any global memory, until that kernel has
// completed and its writes are visible, then lets its own dependents launch.
// Without the launch attribute both instructions are no-ops.
__device__ __forceinline__ void pdl_begin() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Per-(device, stream) workspace of the reducing casts: each CTA stores its
// partial max |x| (fp32 bits) and saturated count in its own slot with plain
// stores -- no atomics or fences, so a CTA retires as soon as its stores are
// issued -- and a one-CTA finalize kernel launched right after reduces them.
constexpr int kMaxPartials = 8192;
struct Workspace {
    uint32_t amax[kMaxPartials];
    unsigned long long sat[kMaxPartials];
    float scratch[4];  // device scalars for calls whose caller passed none
};

// What a launch that reduced into the workspace leaves to the finalize kernel
// (kept for the allocation-free amax, which finishes in its last CTA).
struct FinishArgs {
    float* amax_out;                     // nullable
    float* scale_out;                    // nullable
    float* scale_inv_out;                // nullable
    unsigned long long* sat_out;         // nullable
    int fmt;
    int margin;
};

// ------------------------------------------------------------ memory ops

// L2 eviction-priority policies (createpolicy, sm_80+).  Current scaling reads
// x twice (amax, then the cast); the cast runs right after the amax pass in
// reverse chunk order, so it starts on the part of x the amax pass touched
// last (still in L2), and marks its loads evict_first: they are x's last use.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint4 ldg_stream_hint(const void* p, uint64_t policy) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p), "l"(policy));
    return v;
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ void stg_stream(void* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// Evict-first (streaming) 16-byte store, for outputs that the same chain of
// kernels does not read again (the dequantized values): their dirty lines
// leave L2 while the storing kernel runs instead of during the next kernel's
// reads.  Measured on the E5M2 gradient chain (32 x 8192^2 cast + dequantize):
// 5% less time than plain stores; the codes keep plain stores because the
// dequantize reads them back from L2.
__device__ __forceinline__ void stg_evict_first(void* p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void stg_stream(void* p, uint2 v) {
    asm volatile("st.global.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

}  // namespace fp8q
