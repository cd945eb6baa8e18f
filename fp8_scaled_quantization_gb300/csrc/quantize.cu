// quantize.cu -- per-tensor scaled cast BF16/FP32 -> E4M3FN/E5M2 with an
// optional fused amax (the delayed recipe records it) and saturation count,
// and the fused delayed-scaling step (cast + history update).
//
// "Megatron FP8" §4 (x * scale, clamp to +-FP8_MAX), §2 (E4M3FN saturates,
// E5M2 keeps Inf), §5 (delayed scaling: record amax, update the history, derive
// the next scale), §6 (cast_to_fp8 feeding the FP8 GEMM), §24 (overflow counts
// per layer).
//
// HBM-bound: each thread moves items of one 16-byte load (8 BF16 / 4 fp32
// elements in, 8 / 4 codes out) and keeps 8 loads in flight; one CTA per fixed
// chunk of 16384 (BF16) / 8192 (fp32) elements.
// Chunks run in reverse order with evict_first loads: after an amax pass over
// x (current scaling) the end of x is the part still in L2.  Reductions store
// one partial per CTA in the stream workspace (plain stores, so a CTA retires
// as soon as its stores are issued); the finalize kernel reduces them.
#include "fp8q_device.cuh"
#include "fp8q_host.h"

namespace fp8q {
namespace {

constexpr int kThreads = 256;

// Items of one 16-byte load (8 BF16 / 4 fp32 elements -> 8 / 4 codes): a warp
// loads 512 contiguous bytes and stores 256 / 128 contiguous bytes per item
// (16-byte loads at a 32- or 64-byte lane stride, each touching half or a
// quarter of every sector, measured slower); 8 items in flight per thread.
template <bool BF16> struct VecCfg {
    static constexpr int kPer = BF16 ? 8 : 4;  // elements per item
    static constexpr int kItems = 8;
    static constexpr int64_t kItemsPerCta = (int64_t)kThreads * kItems;
};

// Current scaling inside the cast: the amax kernel left one partial per CTA;
// every CTA of the cast reduces them (after issuing its own loads of x) and
// derives the scale; CTA 0 writes amax / scale / scale_inv.
struct CurArgs {
    const uint32_t* part = nullptr;
    int nparts = 0;
    int margin = 0;
    float* amax_out = nullptr;
    float* scale_out = nullptr;
    float* scale_inv_out = nullptr;
};

// fp8_quantize_current lets the cast CTAs reduce the amax partials only up to
// this many partials (about 6M BF16 elements); beyond, each CTA's partial
// reads cost more than the finalize launch they replace (measured on
// 8192 x 8192: 93.3 vs 91.6 us per amax + cast + dequantize chain).
constexpr int kCastReducesUpTo = 256;

// The tensor's current scale from the amax partials (every thread of the CTA
// calls this; the result is valid in all of them).
template <int FMT>
__device__ __forceinline__ float scale_from_partials(const CurArgs& cur, uint32_t* red) {
    uint32_t m = 0;
    for (int i = threadIdx.x; i < cur.nparts; i += kThreads) m = umax(m, __ldcg(cur.part + i));
    uint32_t bits = block_max_u32(m, red);
    if (bits > 0x7F800000u) bits = 0x7FC00000u;  // canonical NaN
    const float amax = __uint_as_float(bits);
    float s, si;
    scale_from_amax<FMT>(amax, cur.margin, &s, &si);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        if (cur.amax_out) *cur.amax_out = amax;
        if (cur.scale_out) *cur.scale_out = s;
        if (cur.scale_inv_out) *cur.scale_inv_out = si;
    }
    return s;
}

// The plain cast fits 48 registers, so 5 CTAs (1280 threads, 160 KB of loads
// in flight) share an SM; the reducing and current-scale variants need more
// (at 48 the reducing ones spill inside the loop) and take 64 registers, 4
// CTAs per SM.
template <int FMT, bool BF16, bool AMAX, bool SAT, bool CUR = false>
__global__ void __launch_bounds__(kThreads, (AMAX || SAT || CUR) ? 4 : 5)
quantize_vec_kernel(const uint8_t* __restrict__ x, uint8_t* __restrict__ q, int64_t n, const float* scale_ptr,
                    uint32_t* __restrict__ part_amax, unsigned long long* __restrict__ part_sat, CurArgs cur) {
    pdl_begin();
    using C = VecCfg<BF16>;
    const int64_t nitems = n / C::kPer;
    const int64_t nchunks = (nitems + C::kItemsPerCta - 1) / C::kItemsPerCta;
    const uint64_t pol = l2_policy_evict_first();
    __shared__ uint32_t cur_red[CUR ? 32 : 1];
    float scale = CUR ? 0.0f : *scale_ptr;
    bool have_scale = !CUR;
    uint32_t am16 = 0;  // BF16: u16x2 max of |x|
    uint32_t am32 = 0;  // fp32 bits max of |x|
    uint32_t sat = 0;
    for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
        const int64_t chunk = nchunks - 1 - c;  // reverse order
        const int64_t ibase = chunk * C::kItemsPerCta + threadIdx.x;
        uint4 v[C::kItems];
#pragma unroll
        for (int k = 0; k < C::kItems; ++k) {
            const int64_t i = ibase + (int64_t)k * kThreads;
            if (i < nitems) v[k] = ldg_stream_hint(x + i * 16, pol);
        }
        if constexpr (CUR) {
            if (!have_scale) {  // the loads above are in flight meanwhile
                scale = scale_from_partials<FMT>(cur, cur_red);
                have_scale = true;
            }
        }
#pragma unroll
        for (int k = 0; k < C::kItems; ++k) {
            const int64_t i = ibase + (int64_t)k * kThreads;
            if (i >= nitems) break;
            if constexpr (BF16) {
                uint32_t m;
                Codes8 cd = cvt_bf16x8<FMT>(v[k], scale, &m);
                if (chunk_needs_fixup<FMT, SAT>(fold_u16x2_to_f32bits(m), scale)) sat += fixup_bf16x8<FMT>(v[k], scale, &cd);
                if constexpr (AMAX) am16 = max_u16x2(am16, m);
                stg_stream(q + i * 8, make_uint2(cd.lo, cd.hi));
            } else {
                const float4 f = make_float4(__uint_as_float(v[k].x), __uint_as_float(v[k].y), __uint_as_float(v[k].z),
                                             __uint_as_float(v[k].w));
                uint32_t m;
                uint32_t w = cvt_f32x4<FMT>(f, scale, &m);
                if (chunk_needs_fixup<FMT, SAT>(m, scale)) sat += fixup_f32x4<FMT>(f, scale, &w);
                if constexpr (AMAX) am32 = umax(am32, m);
                __stcs(reinterpret_cast<unsigned int*>(q + i * 4), w);
            }
        }
    }

    if constexpr (CUR) {
        if (!have_scale) scale = scale_from_partials<FMT>(cur, cur_red);  // a CTA without chunks (tiny n)
    }
    // Tail (< one item): CTA 0.
    if (blockIdx.x == 0) {
        for (int64_t i = nitems * C::kPer + threadIdx.x; i < n; i += kThreads) {
            float xv;
            uint32_t b;
            if constexpr (BF16) {
                uint16_t h = reinterpret_cast<const uint16_t*>(x)[i];
                xv = __uint_as_float((uint32_t)h << 16);
                b = (uint32_t)(h & 0x7FFFu) << 16;
            } else {
                xv = reinterpret_cast<const float*>(x)[i];
                b = __float_as_uint(xv) & 0x7FFFFFFFu;
            }
            uint32_t s;
            q[i] = (uint8_t)quant_one<FMT>(xv, scale, &s);
            sat += s;
            am32 = umax(am32, b);
        }
    }

    if constexpr (AMAX || SAT) {
        __shared__ uint32_t red[32];
        __shared__ unsigned long long red64[32];
        uint32_t bits = umax(am32, BF16 ? fold_u16x2_to_f32bits(am16) : 0u);
        if constexpr (AMAX) bits = block_max_u32(bits, red);
        unsigned long long total = 0;
        if constexpr (SAT) total = block_sum_u64((unsigned long long)sat, red64);
        if (threadIdx.x == 0) {
            if constexpr (AMAX) part_amax[blockIdx.x] = bits;
            if constexpr (SAT) part_sat[blockIdx.x] = total;
        }
    }
}

// Element-at-a-time path for pointers that are not 16-byte aligned.
template <int FMT, bool BF16>
__global__ void __launch_bounds__(kThreads)
quantize_scalar_kernel(const uint8_t* __restrict__ x, uint8_t* __restrict__ q, int64_t n, const float* scale_ptr,
                       uint32_t* __restrict__ part_amax, unsigned long long* __restrict__ part_sat) {
    pdl_begin();
    const float scale = *scale_ptr;
    uint32_t am = 0, sat = 0;
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n; i += (int64_t)gridDim.x * kThreads) {
        float xv;
        uint32_t b;
        if constexpr (BF16) {
            uint16_t h = reinterpret_cast<const uint16_t*>(x)[i];
            xv = __uint_as_float((uint32_t)h << 16);
            b = (uint32_t)(h & 0x7FFFu) << 16;
        } else {
            xv = reinterpret_cast<const float*>(x)[i];
            b = __float_as_uint(xv) & 0x7FFFFFFFu;
        }
        uint32_t s;
        q[i] = (uint8_t)quant_one<FMT>(xv, scale, &s);
        sat += s;
        am = umax(am, b);
    }
    if (part_amax != nullptr || part_sat != nullptr) {
        __shared__ uint32_t red[32];
        __shared__ unsigned long long red64[32];
        const uint32_t bits = block_max_u32(am, red);
        const unsigned long long total = block_sum_u64((unsigned long long)sat, red64);
        if (threadIdx.x == 0) {
            if (part_amax) part_amax[blockIdx.x] = bits;
            if (part_sat) part_sat[blockIdx.x] = total;
        }
    }
}

template <int FMT, bool BF16>
fp8_status_t launch_vec(bool amax, bool satc, unsigned grid, cudaStream_t st, const uint8_t* x, uint8_t* q, int64_t n,
                        const float* scale, uint32_t* pa, unsigned long long* ps) {
    const char* w = "fp8_quantize";
    const dim3 g(grid), b(kThreads);
    const CurArgs none;
    if (amax && satc) return launch(w, quantize_vec_kernel<FMT, BF16, true, true>, g, b, st, x, q, n, scale, pa, ps, none);
    if (amax) return launch(w, quantize_vec_kernel<FMT, BF16, true, false>, g, b, st, x, q, n, scale, pa, ps, none);
    if (satc) return launch(w, quantize_vec_kernel<FMT, BF16, false, true>, g, b, st, x, q, n, scale, pa, ps, none);
    return launch(w, quantize_vec_kernel<FMT, BF16, false, false>, g, b, st, x, q, n, scale, pa, ps, none);
}

// The cast, with per-CTA partials when reducing; *nparts receives their count.
fp8_status_t enqueue_cast(const uint8_t* x, bool bf16, int64_t n, int fmt, const float* scale, uint8_t* q,
                          Workspace* ws, bool amax, bool satc, cudaStream_t st, int* nparts) {
    const bool reduce = amax || satc;
    uint32_t* pa = reduce ? ws->amax : nullptr;
    unsigned long long* ps = reduce ? ws->sat : nullptr;
    if (aligned16(x) && aligned16(q)) {
        const int64_t per_cta = bf16 ? VecCfg<true>::kItemsPerCta : VecCfg<false>::kItemsPerCta;
        int64_t grid = (n / (bf16 ? 8 : 4) + per_cta - 1) / per_cta;
        const int64_t cap = reduce ? kMaxPartials : 0x7FFFFFFF;
        if (grid > cap) grid = cap;
        if (grid < 1) grid = 1;
        *nparts = (int)(reduce ? grid : 0);
        const unsigned g = (unsigned)grid;
        if (fmt == FP8_E4M3)
            return bf16 ? launch_vec<kE4M3, true>(amax, satc, g, st, x, q, n, scale, pa, ps)
                        : launch_vec<kE4M3, false>(amax, satc, g, st, x, q, n, scale, pa, ps);
        return bf16 ? launch_vec<kE5M2, true>(amax, satc, g, st, x, q, n, scale, pa, ps)
                    : launch_vec<kE5M2, false>(amax, satc, g, st, x, q, n, scale, pa, ps);
    }
    int64_t grid = (n + kThreads - 1) / kThreads;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    *nparts = (int)(reduce ? grid : 0);
    const dim3 g((unsigned)grid), b(kThreads);
    const char* w = "fp8_quantize";
    if (fmt == FP8_E4M3)
        return bf16 ? launch(w, quantize_scalar_kernel<kE4M3, true>, g, b, st, x, q, n, scale, pa, ps)
                    : launch(w, quantize_scalar_kernel<kE4M3, false>, g, b, st, x, q, n, scale, pa, ps);
    return bf16 ? launch(w, quantize_scalar_kernel<kE5M2, true>, g, b, st, x, q, n, scale, pa, ps)
                : launch(w, quantize_scalar_kernel<kE5M2, false>, g, b, st, x, q, n, scale, pa, ps);
}

}  // namespace
}  // namespace fp8q

using namespace fp8q;

extern "C" fp8_status_t fp8_quantize(const void* x, fp8_dtype_t dtype, int64_t n, fp8_format_t fmt,
                                     const float* scale, uint8_t* q_out, float* amax_out,
                                     unsigned long long* sat_count_out, void* stream) {
    if (!valid_dtype(dtype)) return fail(FP8_ERR_INVALID_ARG, "fp8_quantize: unknown dtype %d", (int)dtype);
    if (!valid_fmt(fmt)) return fail(FP8_ERR_INVALID_ARG, "fp8_quantize: unknown format %d", (int)fmt);
    if (n < 0) return fail(FP8_ERR_INVALID_ARG, "fp8_quantize: n < 0");
    if (scale == nullptr) return fail(FP8_ERR_INVALID_ARG, "fp8_quantize: scale is NULL");
    if (n > 0 && (x == nullptr || q_out == nullptr))
        return fail(FP8_ERR_INVALID_ARG, "fp8_quantize: x / q_out is NULL");
    const int es = dtype_size(dtype);
    if (reinterpret_cast<uintptr_t>(x) % es) return fail(FP8_ERR_INVALID_ARG, "fp8_quantize: x not element-aligned");

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool reduce = amax_out != nullptr || sat_count_out != nullptr;
    if (n == 0 && !reduce) return FP8_OK;
    Workspace* ws = nullptr;
    if (reduce) {
        fp8_status_t s;
        ws = stream_workspace(st, &s);
        if (!ws) return s;
    }
    int nparts = 0;
    fp8_status_t s = enqueue_cast(static_cast<const uint8_t*>(x), dtype == FP8_DT_BF16, n, (int)fmt, scale, q_out, ws,
                                  amax_out != nullptr, sat_count_out != nullptr, st, &nparts);
    if (s != FP8_OK || !reduce) return s;
    FinalizeArgs fa;
    fa.part_amax = amax_out ? ws->amax : nullptr;
    fa.part_sat = sat_count_out ? ws->sat : nullptr;
    fa.nparts = nparts;
    fa.amax_out = amax_out;
    fa.sat_out = sat_count_out;
    fa.fmt = (int)fmt;
    return launch_finalize(fa, st);
}

extern "C" fp8_status_t fp8_quantize_delayed(const void* x, fp8_dtype_t dtype, int64_t n, fp8_format_t fmt,
                                             float* scale, float* scale_inv, uint8_t* q_out, float* amax_history,
                                             int history_len, int64_t step, fp8_amax_algo_t algo, int margin,
                                             float* amax_out, unsigned long long* sat_count_out, void* stream) {
    const char* fn = "fp8_quantize_delayed";
    if (!valid_dtype(dtype)) return fail(FP8_ERR_INVALID_ARG, "%s: unknown dtype %d", fn, (int)dtype);
    if (!valid_fmt(fmt)) return fail(FP8_ERR_INVALID_ARG, "%s: unknown format %d", fn, (int)fmt);
    if (n < 0) return fail(FP8_ERR_INVALID_ARG, "%s: n < 0", fn);
    if (scale == nullptr || scale_inv == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: scale / scale_inv is NULL", fn);
    if (n > 0 && (x == nullptr || q_out == nullptr)) return fail(FP8_ERR_INVALID_ARG, "%s: x / q_out is NULL", fn);
    if (amax_history == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: amax_history is NULL", fn);
    if (history_len < 1 || history_len > 65536) return fail(FP8_ERR_INVALID_ARG, "%s: history_len must be in [1, 65536]", fn);
    if (step < 0) return fail(FP8_ERR_INVALID_ARG, "%s: step < 0", fn);
    if (algo != FP8_AMAX_MAX && algo != FP8_AMAX_MOST_RECENT) return fail(FP8_ERR_INVALID_ARG, "%s: unknown algo %d", fn, (int)algo);
    if (!valid_margin(margin)) return fail(FP8_ERR_INVALID_ARG, "%s: margin out of [-126, 126]", fn);
    const int es = dtype_size(dtype);
    if (reinterpret_cast<uintptr_t>(x) % es) return fail(FP8_ERR_INVALID_ARG, "%s: x not element-aligned", fn);

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    fp8_status_t s;
    Workspace* ws = stream_workspace(st, &s);
    if (!ws) return s;
    int nparts = 0;
    s = enqueue_cast(static_cast<const uint8_t*>(x), dtype == FP8_DT_BF16, n, (int)fmt, scale, q_out, ws, true,
                     sat_count_out != nullptr, st, &nparts);
    if (s != FP8_OK) return s;
    // The finalize runs after the cast has completed, so it may overwrite the
    // scale the cast read.
    FinalizeArgs fa;
    fa.part_amax = ws->amax;
    fa.part_sat = sat_count_out ? ws->sat : nullptr;
    fa.nparts = nparts;
    fa.amax_out = amax_out;
    fa.sat_out = sat_count_out;
    fa.scale_out = scale;
    fa.scale_inv_out = scale_inv;
    fa.fmt = (int)fmt;
    fa.margin = margin;
    fa.hist = amax_history;
    fa.hist_len = history_len;
    fa.slot = (int)(step % history_len);
    fa.algo = (int)algo;
    return launch_finalize(fa, st);
}

extern "C" fp8_status_t fp8_quantize_current(const void* x, fp8_dtype_t dtype, int64_t n, fp8_format_t fmt,
                                             int margin, uint8_t* q_out, float* amax_out, float* scale_out,
                                             float* scale_inv_out, void* stream) {
    const char* fn = "fp8_quantize_current";
    if (!valid_dtype(dtype)) return fail(FP8_ERR_INVALID_ARG, "%s: unknown dtype %d", fn, (int)dtype);
    if (!valid_fmt(fmt)) return fail(FP8_ERR_INVALID_ARG, "%s: unknown format %d", fn, (int)fmt);
    if (!valid_margin(margin)) return fail(FP8_ERR_INVALID_ARG, "%s: margin out of [-126, 126]", fn);
    if (n < 0) return fail(FP8_ERR_INVALID_ARG, "%s: n < 0", fn);
    if (n > 0 && (x == nullptr || q_out == nullptr)) return fail(FP8_ERR_INVALID_ARG, "%s: x / q_out is NULL", fn);
    if (reinterpret_cast<uintptr_t>(x) % dtype_size(dtype)) return fail(FP8_ERR_INVALID_ARG, "%s: x not element-aligned", fn);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    fp8_status_t s;
    Workspace* ws = stream_workspace(st, &s);
    if (!ws) return s;
    const bool bf16 = dtype == FP8_DT_BF16;
    if (n == 0 || !aligned16(x) || !aligned16(q_out)) {
        // amax + finalize, then the element-wise cast with that scale
        float* a = amax_out ? amax_out : &ws->scratch[0];
        float* sc = scale_out ? scale_out : &ws->scratch[1];
        float* si = scale_inv_out ? scale_inv_out : &ws->scratch[2];
        s = fp8_amax(x, dtype, n, a, fmt, margin, sc, si, stream);
        if (s != FP8_OK || n == 0) return s;
        return fp8_quantize(x, dtype, n, fmt, sc, q_out, nullptr, nullptr, stream);
    }
    int nparts = 0;
    s = enqueue_amax_partials(x, dtype, n, ws, st, &nparts);
    if (s != FP8_OK) return s;
    if (nparts > kCastReducesUpTo) {
        // Large tensor: every cast CTA reading every partial would cost more
        // than the one-CTA finalize it saves, so finalize, then the plain cast.
        FinalizeArgs fa;
        fa.part_amax = ws->amax;
        fa.nparts = nparts;
        fa.amax_out = amax_out;
        fa.scale_out = scale_out ? scale_out : &ws->scratch[1];
        fa.scale_inv_out = scale_inv_out ? scale_inv_out : &ws->scratch[2];
        fa.fmt = (int)fmt;
        fa.margin = margin;
        s = launch_finalize(fa, st);
        if (s != FP8_OK) return s;
        return enqueue_cast(static_cast<const uint8_t*>(x), bf16, n, (int)fmt, fa.scale_out, q_out, ws, false, false,
                            st, &nparts);
    }
    CurArgs cur;
    cur.part = ws->amax;
    cur.nparts = nparts;
    cur.margin = margin;
    cur.amax_out = amax_out;
    cur.scale_out = scale_out;
    cur.scale_inv_out = scale_inv_out;
    const int64_t per_cta = bf16 ? VecCfg<true>::kItemsPerCta : VecCfg<false>::kItemsPerCta;
    int64_t grid = (n / (bf16 ? 8 : 4) + per_cta - 1) / per_cta;
    if (grid > 0x7FFFFFFF) grid = 0x7FFFFFFF;
    if (grid < 1) grid = 1;
    const uint8_t* xp = static_cast<const uint8_t*>(x);
    const dim3 g((unsigned)grid), b(kThreads);
    const float* no_scale = nullptr;
    uint32_t* no_pa = nullptr;
    unsigned long long* no_ps = nullptr;
    if (fmt == FP8_E4M3)
        return bf16 ? launch(fn, quantize_vec_kernel<kE4M3, true, false, false, true>, g, b, st, xp, q_out, n, no_scale,
                             no_pa, no_ps, cur)
                    : launch(fn, quantize_vec_kernel<kE4M3, false, false, false, true>, g, b, st, xp, q_out, n,
                             no_scale, no_pa, no_ps, cur);
    return bf16 ? launch(fn, quantize_vec_kernel<kE5M2, true, false, false, true>, g, b, st, xp, q_out, n, no_scale,
                         no_pa, no_ps, cur)
                : launch(fn, quantize_vec_kernel<kE5M2, false, false, false, true>, g, b, st, xp, q_out, n, no_scale,
                         no_pa, no_ps, cur);
}
