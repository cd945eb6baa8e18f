// quantize.cu -- per-tensor scaled cast BF16/FP32 -> E4M3FN/E5M2 with an
// optional fused amax (the delayed recipe records it) and saturation count.
//
// "Megatron FP8" §4 (x * scale, clamp to +-FP8_MAX), §2 (E4M3FN saturates,
// E5M2 keeps Inf), §6 (cast_to_fp8 feeding the FP8 GEMM), §24 (overflow
// counts per layer).
//
// HBM-bound: each thread moves 16 elements per unit (two 16-byte BF16 loads or
// four 16-byte fp32 loads in, one 16-byte code store out), two units in
// flight; grid-stride over a grid of 8 CTAs per SM.
#include "fp8q_device.cuh"
#include "fp8q_host.h"

namespace fp8q {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 2;  // 16-element units in flight per thread

template <int FMT, bool BF16, bool AMAX, bool SAT>
__global__ void __launch_bounds__(kThreads)
quantize_vec_kernel(const uint8_t* __restrict__ x, uint8_t* __restrict__ q, int64_t n,
                    const float* __restrict__ scale_ptr, Workspace* ws, FinishArgs fa) {
    const float scale = __ldg(scale_ptr);
    const int64_t nunits = n / 16;
    uint32_t am16 = 0;  // BF16: u16x2 max of |x|
    uint32_t am32 = 0;  // fp32 bits max of |x|
    uint32_t sat = 0;

    const int64_t step = (int64_t)gridDim.x * kThreads * kUnroll;
    for (int64_t base = (int64_t)blockIdx.x * kThreads * kUnroll + threadIdx.x; base < nunits; base += step) {
        if constexpr (BF16) {
            uint4 v[kUnroll][2];
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                const int64_t u = base + (int64_t)k * kThreads;
                if (u < nunits) {
                    v[k][0] = ldg_stream(x + u * 32);
                    v[k][1] = ldg_stream(x + u * 32 + 16);
                }
            }
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                const int64_t u = base + (int64_t)k * kThreads;
                if (u >= nunits) break;
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
            }
        } else {
            uint4 v[kUnroll][4];
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                const int64_t u = base + (int64_t)k * kThreads;
                if (u < nunits) {
#pragma unroll
                    for (int h = 0; h < 4; ++h) v[k][h] = ldg_stream(x + u * 64 + h * 16);
                }
            }
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                const int64_t u = base + (int64_t)k * kThreads;
                if (u >= nunits) break;
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
    }

    // Tail (< 16 elements): block 0.
    if (blockIdx.x == 0) {
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

    if constexpr (AMAX || SAT) {
        __shared__ uint32_t red[32];
        __shared__ unsigned long long red64[32];
        uint32_t bits = umax(am32, BF16 ? fold_u16x2_to_f32bits(am16) : 0u);
        bits = block_max_u32(bits, red);
        unsigned long long total = SAT ? block_sum_u64((unsigned long long)sat, red64) : 0ull;
        grid_finish(ws, bits, total, fa);
    }
}

// Element-at-a-time path for pointers that are not 16-byte aligned.
template <int FMT, bool BF16>
__global__ void __launch_bounds__(kThreads)
quantize_scalar_kernel(const uint8_t* __restrict__ x, uint8_t* __restrict__ q, int64_t n,
                       const float* __restrict__ scale_ptr, Workspace* ws, FinishArgs fa, int reduce) {
    const float scale = __ldg(scale_ptr);
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
    if (reduce) {
        __shared__ uint32_t red[32];
        __shared__ unsigned long long red64[32];
        uint32_t bits = block_max_u32(am, red);
        unsigned long long total = block_sum_u64((unsigned long long)sat, red64);
        grid_finish(ws, bits, total, fa);
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
        int64_t grid = (units + (int64_t)kThreads * kUnroll - 1) / ((int64_t)kThreads * kUnroll);
        const int64_t cap = (int64_t)sm_count() * 8;
        if (grid > cap) grid = cap;
        if (grid < 1) grid = 1;
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
