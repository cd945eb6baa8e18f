// quantize.cu -- per-tensor scaled cast BF16/FP32 -> E4M3FN/E5M2 with an
// optional fused amax (the delayed recipe records it) and saturation count.
//
// "Megatron FP8" §4 (x * scale, clamp to +-FP8_MAX), §2 (E4M3FN saturates,
// E5M2 keeps Inf), §6 (cast_to_fp8 feeding the FP8 GEMM), §24 (overflow
// counts per layer).
//
// HBM-bound: each thread moves 16 elements per unit (two 16-byte BF16 loads or
// four 16-byte fp32 loads in, one 16-byte code store out) and keeps 8 loads in
// flight; one CTA per fixed chunk of 16384 (BF16) / 8192 (fp32) elements.
#include "fp8q_device.cuh"
#include "fp8q_host.h"

namespace fp8q {
namespace {

constexpr int kThreads = 256;

// 16-element units per thread: every thread issues all its 16-byte loads
// (8 for BF16, 8 for fp32) before converting, and each CTA owns one fixed
// chunk of 256 * kUnits units; the hardware scheduler balances the CTAs.
template <bool BF16> struct VecCfg {
    static constexpr int kUnits = BF16 ? 4 : 2;
    static constexpr int kLoads = BF16 ? 2 : 4;  // 16-byte loads per unit
    static constexpr int64_t kUnitsPerCta = (int64_t)kThreads * kUnits;
};

// The delayed recipe's history update ("Megatron FP8" §5, update_fp8_meta):
// write this step's amax into slot step % len, take the window maximum
// (NaN-propagating) or the slot, and overwrite scale / scale_inv with the
// scale of the next step.  The window maximum is max(this amax, the maximum
// of the other len - 1 entries); CTAs b < ceil(len / blockDim) each reduce
// grid-strided slices of those entries before they arrive, folding an order-preserving
// key into the workspace, so the last CTA only combines scalars.  Every CTA
// has read the old scale before it arrives, so the overwrite races with
// nothing, and no CTA reads the history slot that the last CTA writes.
struct DelayedArgs {
    float* hist;
    int len;
    int slot;
    int algo;
    float* scale;
    float* scale_inv;
};

// Unsigned key with the order of the float values (NaN handled apart).
__device__ __forceinline__ uint32_t f32_order_key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float f32_from_order_key(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

template <int FMT>
__device__ __forceinline__ void delayed_finish(Workspace* ws, uint32_t cta_amax_bits, unsigned long long cta_sat,
                                               const FinishArgs& fa, const DelayedArgs& da) {
    __shared__ uint32_t s_key[32];
    const unsigned cta = blockIdx.x;
    uint32_t key = 0;
    int nan = 0;
    const bool scans = da.algo == FP8_AMAX_MAX && (int64_t)cta * blockDim.x < da.len;
    if (scans) {
        // grid-strided, so that a grid smaller than the history still covers it
        for (int64_t i = (int64_t)cta * blockDim.x + threadIdx.x; i < da.len;
             i += (int64_t)gridDim.x * blockDim.x) {
            if (i == da.slot) continue;
            const float v = da.hist[i];
            if (isnan(v)) nan = 1;
            else key = umax(key, f32_order_key(v));
        }
        nan = __syncthreads_or(nan);
        key = __reduce_max_sync(0xFFFFFFFFu, key);
        if ((threadIdx.x & 31) == 0) s_key[threadIdx.x >> 5] = key;
        __syncthreads();
        key = (threadIdx.x < (blockDim.x >> 5)) ? s_key[threadIdx.x] : 0u;
        key = __reduce_max_sync(0xFFFFFFFFu, key);
    }
    if (threadIdx.x != 0) return;
    if (scans) {
        if (key) atomicMax(&ws->hist_key, key);
        if (nan) atomicOr(&ws->hist_nan, 1u);
    }
    if (cta_amax_bits) atomicMax(&ws->amax_bits, cta_amax_bits);
    if (cta_sat) atomicAdd(&ws->sat, cta_sat);
    __threadfence();
    if (atomicAdd(&ws->done, 1u) != gridDim.x * gridDim.y * gridDim.z - 1) return;
    __threadfence();
    uint32_t bits = atomicExch(&ws->amax_bits, 0u);
    const unsigned long long sat = atomicExch(&ws->sat, 0ull);
    const uint32_t hkey = atomicExch(&ws->hist_key, 0u);
    const uint32_t hnan = atomicExch(&ws->hist_nan, 0u);
    atomicExch(&ws->done, 0u);
    if (bits > 0x7F800000u) bits = 0x7FC00000u;  // canonical NaN
    const float amax = __uint_as_float(bits);
    if (fa.amax_out) *fa.amax_out = amax;
    if (fa.sat_out) *fa.sat_out = sat;
    da.hist[da.slot] = amax;
    float eff = amax;
    if (da.algo == FP8_AMAX_MAX) {
        if (hnan || isnan(amax)) eff = __uint_as_float(0x7FC00000u);
        else if (hkey) eff = fmaxf(amax, f32_from_order_key(hkey));
    }
    float sc, si;
    scale_from_amax<FMT>(eff, fa.margin, &sc, &si);
    *da.scale = sc;
    *da.scale_inv = si;
}

// At most 48 registers, so that 5 CTAs (1280 threads, 160 KB of loads in
// flight) fit on an SM whichever reductions are fused in.
template <int FMT, bool BF16, bool AMAX, bool SAT, bool DELAYED = false>
__global__ void __launch_bounds__(kThreads, 5)
quantize_vec_kernel(const uint8_t* __restrict__ x, uint8_t* __restrict__ q, int64_t n,
                    const float* scale_ptr, Workspace* ws, FinishArgs fa, DelayedArgs da = DelayedArgs{}) {
    using C = VecCfg<BF16>;
    const int64_t nunits = n / 16;
    // Chunks run in reverse order with evict_first loads: after an amax pass
    // over x (current scaling) the end of x is the part still in L2.
    const int64_t chunk = (int64_t)(gridDim.x - 1 - blockIdx.x);
    const int64_t ubase = chunk * C::kUnitsPerCta + threadIdx.x;
    const uint64_t pol = l2_policy_evict_first();
    uint4 v[C::kUnits][C::kLoads];
#pragma unroll
    for (int k = 0; k < C::kUnits; ++k) {
        const int64_t u = ubase + (int64_t)k * kThreads;
        if (u < nunits) {
#pragma unroll
            for (int h = 0; h < C::kLoads; ++h) v[k][h] = ldg_stream_hint(x + u * (BF16 ? 32 : 64) + h * 16, pol);
        }
    }
    const float scale = *scale_ptr;  // plain load: the delayed variant rewrites it at the end
    uint32_t am16 = 0;  // BF16: u16x2 max of |x|
    uint32_t am32 = 0;  // fp32 bits max of |x|
    uint32_t sat = 0;
#pragma unroll
    for (int k = 0; k < C::kUnits; ++k) {
        const int64_t u = ubase + (int64_t)k * kThreads;
        if (u >= nunits) break;
        if constexpr (BF16) {
            Codes8 c[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t m;
                c[h] = cvt_bf16x8<FMT>(v[k][h], scale, &m);
                if (chunk_needs_fixup<FMT, SAT>(fold_u16x2_to_f32bits(m), scale))
                    sat += fixup_bf16x8<FMT>(v[k][h], scale, &c[h]);
                if constexpr (AMAX) am16 = max_u16x2(am16, m);
            }
            stg_stream(q + u * 16, make_uint4(c[0].lo, c[0].hi, c[1].lo, c[1].hi));
        } else {
            uint32_t w[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                float4 f = make_float4(__uint_as_float(v[k][h].x), __uint_as_float(v[k][h].y),
                                       __uint_as_float(v[k][h].z), __uint_as_float(v[k][h].w));
                uint32_t m;
                w[h] = cvt_f32x4<FMT>(f, scale, &m);
                if (chunk_needs_fixup<FMT, SAT>(m, scale)) sat += fixup_f32x4<FMT>(f, scale, &w[h]);
                if constexpr (AMAX) am32 = umax(am32, m);
            }
            stg_stream(q + u * 16, make_uint4(w[0], w[1], w[2], w[3]));
        }
    }

    // Tail (< 16 elements): the CTA of the last chunk.
    if (chunk == gridDim.x - 1) {
        for (int64_t i = nunits * 16 + threadIdx.x; i < n; i += kThreads) {
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

    if constexpr (AMAX || SAT || DELAYED) {
        __shared__ uint32_t red[32];
        __shared__ unsigned long long red64[32];
        uint32_t bits = umax(am32, BF16 ? fold_u16x2_to_f32bits(am16) : 0u);
        bits = block_max_u32(bits, red);
        unsigned long long total = SAT ? block_sum_u64((unsigned long long)sat, red64) : 0ull;
        if constexpr (DELAYED) delayed_finish<FMT>(ws, bits, total, fa, da);
        else grid_finish(ws, bits, total, fa);
    }
}

// Element-at-a-time path for pointers that are not 16-byte aligned.
template <int FMT, bool BF16, bool DELAYED = false>
__global__ void __launch_bounds__(kThreads)
quantize_scalar_kernel(const uint8_t* __restrict__ x, uint8_t* __restrict__ q, int64_t n,
                       const float* scale_ptr, Workspace* ws, FinishArgs fa, int reduce,
                       DelayedArgs da = DelayedArgs{}) {
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
    if (reduce || DELAYED) {
        __shared__ uint32_t red[32];
        __shared__ unsigned long long red64[32];
        uint32_t bits = block_max_u32(am, red);
        unsigned long long total = block_sum_u64((unsigned long long)sat, red64);
        if constexpr (DELAYED) delayed_finish<FMT>(ws, bits, total, fa, da);
        else grid_finish(ws, bits, total, fa);
    }
}

template <int FMT, bool BF16>
void launch_vec(bool amax, bool satc, unsigned grid, cudaStream_t st, const uint8_t* x, uint8_t* q, int64_t n,
                const float* scale, Workspace* ws, const FinishArgs& fa) {
    if (amax && satc) quantize_vec_kernel<FMT, BF16, true, true><<<grid, kThreads, 0, st>>>(x, q, n, scale, ws, fa);
    else if (amax) quantize_vec_kernel<FMT, BF16, true, false><<<grid, kThreads, 0, st>>>(x, q, n, scale, ws, fa);
    else if (satc) quantize_vec_kernel<FMT, BF16, false, true><<<grid, kThreads, 0, st>>>(x, q, n, scale, ws, fa);
    else quantize_vec_kernel<FMT, BF16, false, false><<<grid, kThreads, 0, st>>>(x, q, n, scale, ws, fa);
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
    FinishArgs fa{amax_out, nullptr, nullptr, sat_count_out, (int)fmt, 0};
    const uint8_t* xp = static_cast<const uint8_t*>(x);
    const bool bf16 = dtype == FP8_DT_BF16;

    if (aligned16(x) && aligned16(q_out)) {
        const int64_t units = n / 16;
        const int64_t per_cta = bf16 ? VecCfg<true>::kUnitsPerCta : VecCfg<false>::kUnitsPerCta;
        int64_t grid = (units + per_cta - 1) / per_cta;
        if (grid < 1) grid = 1;
        if (grid > 0x7FFFFFFF) return fail(FP8_ERR_UNSUPPORTED, "fp8_quantize: n too large");
        const bool am = amax_out != nullptr, sc = sat_count_out != nullptr;
        if (fmt == FP8_E4M3) {
            if (bf16) launch_vec<kE4M3, true>(am, sc, (unsigned)grid, st, xp, q_out, n, scale, ws, fa);
            else launch_vec<kE4M3, false>(am, sc, (unsigned)grid, st, xp, q_out, n, scale, ws, fa);
        } else {
            if (bf16) launch_vec<kE5M2, true>(am, sc, (unsigned)grid, st, xp, q_out, n, scale, ws, fa);
            else launch_vec<kE5M2, false>(am, sc, (unsigned)grid, st, xp, q_out, n, scale, ws, fa);
        }
    } else {
        int64_t grid = (n + kThreads - 1) / kThreads;
        const int64_t cap = (int64_t)sm_count() * 8;
        if (grid > cap) grid = cap;
        if (grid < 1) grid = 1;
        const int r = reduce ? 1 : 0;
        if (fmt == FP8_E4M3) {
            if (bf16) quantize_scalar_kernel<kE4M3, true><<<(unsigned)grid, kThreads, 0, st>>>(xp, q_out, n, scale, ws, fa, r);
            else quantize_scalar_kernel<kE4M3, false><<<(unsigned)grid, kThreads, 0, st>>>(xp, q_out, n, scale, ws, fa, r);
        } else {
            if (bf16) quantize_scalar_kernel<kE5M2, true><<<(unsigned)grid, kThreads, 0, st>>>(xp, q_out, n, scale, ws, fa, r);
            else quantize_scalar_kernel<kE5M2, false><<<(unsigned)grid, kThreads, 0, st>>>(xp, q_out, n, scale, ws, fa, r);
        }
    }
    return after_launch("fp8_quantize");
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
    FinishArgs fa{amax_out, nullptr, nullptr, sat_count_out, (int)fmt, margin};
    DelayedArgs da{amax_history, history_len, (int)(step % history_len), (int)algo, scale, scale_inv};
    const uint8_t* xp = static_cast<const uint8_t*>(x);
    const bool bf16 = dtype == FP8_DT_BF16, sc = sat_count_out != nullptr;
    if (aligned16(x) && aligned16(q_out)) {
        const int64_t per_cta = bf16 ? VecCfg<true>::kUnitsPerCta : VecCfg<false>::kUnitsPerCta;
        int64_t grid = (n / 16 + per_cta - 1) / per_cta;
        if (grid < 1) grid = 1;
        if (grid > 0x7FFFFFFF) return fail(FP8_ERR_UNSUPPORTED, "%s: n too large", fn);
        const unsigned g = (unsigned)grid;
#define FP8Q_LAUNCH_DELAYED(F, B)                                                                                  \
    do {                                                                                                           \
        if (sc) quantize_vec_kernel<F, B, true, true, true><<<g, kThreads, 0, st>>>(xp, q_out, n, scale, ws, fa, da); \
        else quantize_vec_kernel<F, B, true, false, true><<<g, kThreads, 0, st>>>(xp, q_out, n, scale, ws, fa, da);  \
    } while (0)
        if (fmt == FP8_E4M3) {
            if (bf16) FP8Q_LAUNCH_DELAYED(kE4M3, true);
            else FP8Q_LAUNCH_DELAYED(kE4M3, false);
        } else {
            if (bf16) FP8Q_LAUNCH_DELAYED(kE5M2, true);
            else FP8Q_LAUNCH_DELAYED(kE5M2, false);
        }
#undef FP8Q_LAUNCH_DELAYED
    } else {
        int64_t grid = (n + kThreads - 1) / kThreads;
        const int64_t cap = (int64_t)sm_count() * 8;
        if (grid > cap) grid = cap;
        if (grid < 1) grid = 1;
        const unsigned g = (unsigned)grid;
        if (fmt == FP8_E4M3) {
            if (bf16) quantize_scalar_kernel<kE4M3, true, true><<<g, kThreads, 0, st>>>(xp, q_out, n, scale, ws, fa, 1, da);
            else quantize_scalar_kernel<kE4M3, false, true><<<g, kThreads, 0, st>>>(xp, q_out, n, scale, ws, fa, 1, da);
        } else {
            if (bf16) quantize_scalar_kernel<kE5M2, true, true><<<g, kThreads, 0, st>>>(xp, q_out, n, scale, ws, fa, 1, da);
            else quantize_scalar_kernel<kE5M2, false, true><<<g, kThreads, 0, st>>>(xp, q_out, n, scale, ws, fa, 1, da);
        }
    }
    return after_launch(fn);
}
