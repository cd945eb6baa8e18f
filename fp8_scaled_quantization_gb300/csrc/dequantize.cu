// dequantize.cu -- y = decode(q) * scale_inv (one fp32 multiply), stored as
// BF16 (round to nearest even) or fp32.
//
// "Megatron FP8" §4 (scale_inv = 1/s cached so dequantize is one element
// multiply), §23 (reconstructed = fp8 value * scale); "Low Precision Training
// and Rollout", "Implementation Notes" (FP8 weights dequantized to BF16).
//
// Decoding is exact: E4M3 pairs go through cvt.rn.f16x2.e4m3x2 (every E4M3FN
// value is a binary16 value); an E5M2 code is the upper byte of a binary16.
// Both paths work in items of one 16-byte output piece per thread (8 codes
// for BF16, 4 for fp32), so every warp store covers 512 contiguous bytes.
// Per-tensor: one chunk of 256 x 16 items per CTA.  Block-scaled: grid.y walks
// rows, the scale of each item read from the block grid.
#include "fp8q_device.cuh"
#include "fp8q_host.h"

namespace fp8q {
namespace {

constexpr int kThreads = 256;

// 4 codes (one word) -> 4 products in fp32.
template <int FMT>
__device__ __forceinline__ void decode4(uint32_t w, float si, float* o) {
    const uint32_t h01 = fp8x2_to_f16x2<FMT>(w & 0xFFFFu);
    const uint32_t h23 = fp8x2_to_f16x2<FMT>(w >> 16);
    o[0] = __fmul_rn(f16_lo_to_f32(h01), si);
    o[1] = __fmul_rn(f16_hi_to_f32(h01), si);
    o[2] = __fmul_rn(f16_lo_to_f32(h23), si);
    o[3] = __fmul_rn(f16_hi_to_f32(h23), si);
}

template <int FMT, bool OUT_BF16>
__device__ __forceinline__ void dequant_one(uint8_t code, float si, uint8_t* y, int64_t e) {
    float f[4];
    decode4<FMT>(code, si, f);
    if constexpr (OUT_BF16) reinterpret_cast<uint16_t*>(y)[e] = (uint16_t)(f32x2_to_bf16x2(f[0], 0.0f) & 0xFFFFu);
    else reinterpret_cast<float*>(y)[e] = f[0];
}

// Per-tensor path: each item is the codes of one 16-byte output piece (8 codes
// for BF16, 4 for fp32), so a warp's store covers 512 contiguous bytes and its
// load 256 / 128 contiguous bytes; 16 items in flight per thread, one chunk of
// 256 * 16 items per CTA.  (Two 16-byte stores per thread at a 32-byte stride,
// each filling half of every sector it touches, measured 26% slower.)
constexpr int kItems = 16;

template <int FMT, bool OUT_BF16>
__global__ void __launch_bounds__(kThreads)
dequant_tensor_kernel(const uint8_t* __restrict__ q, int64_t n, const float* __restrict__ scale_inv,
                      uint8_t* __restrict__ y) {
    pdl_begin();
    constexpr int kCodes = OUT_BF16 ? 8 : 4;
    const int64_t nitems = n / kCodes;
    const int64_t ibase = (int64_t)blockIdx.x * kThreads * kItems + threadIdx.x;
    uint32_t c[kItems][kCodes / 4];
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
        const int64_t i = ibase + (int64_t)k * kThreads;
        if (i < nitems) {
            if constexpr (OUT_BF16) {
                const uint2 v = __ldcs(reinterpret_cast<const uint2*>(q) + i);
                c[k][0] = v.x;
                c[k][kCodes / 4 - 1] = v.y;
            } else {
                c[k][0] = __ldcs(reinterpret_cast<const unsigned int*>(q) + i);
            }
        }
    }
    const float si = __ldg(scale_inv);
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
        const int64_t i = ibase + (int64_t)k * kThreads;
        if (i >= nitems) continue;
        if constexpr (OUT_BF16) {
            float a[4], b[4];
            decode4<FMT>(c[k][0], si, a);
            decode4<FMT>(c[k][kCodes / 4 - 1], si, b);
            stg_evict_first(y + i * 16, make_uint4(f32x2_to_bf16x2(a[0], a[1]), f32x2_to_bf16x2(a[2], a[3]),
                                              f32x2_to_bf16x2(b[0], b[1]), f32x2_to_bf16x2(b[2], b[3])));
        } else {
            float a[4];
            decode4<FMT>(c[k][0], si, a);
            stg_evict_first(y + i * 16, make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]),
                                              __float_as_uint(a[3])));
        }
    }
    if (blockIdx.x == gridDim.x - 1)
        for (int64_t e = nitems * kCodes + threadIdx.x; e < n; e += kThreads) dequant_one<FMT, OUT_BF16>(q[e], si, y, e);
}

// Any layout: grid.y walks rows, threads walk columns.  `vec` selects 16-code
// chunks (cols % 16 == 0, aligned pointers); otherwise one element per thread.
// br == 0 means a per-tensor scale; block columns are always 128 wide.
template <int FMT, bool OUT_BF16>
__global__ void __launch_bounds__(kThreads)
dequant_rows_kernel(const uint8_t* __restrict__ q, int64_t rows, int64_t cols, const float* __restrict__ scale_inv,
                    int br, int64_t nbc, uint8_t* __restrict__ y, int vec) {
    pdl_begin();
    for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
        const float* srow = br > 0 ? scale_inv + (br == 1 ? r : (r >> 7)) * nbc : scale_inv;
        if (vec) {  // items of one 16-byte output piece, as in dequant_tensor_kernel
            constexpr int kCodes = OUT_BF16 ? 8 : 4;
            const int64_t nit = cols / kCodes;
            for (int64_t it = (int64_t)blockIdx.x * kThreads + threadIdx.x; it < nit; it += (int64_t)gridDim.x * kThreads) {
                const int64_t c = it * kCodes;
                const float si = __ldg(br > 0 ? srow + (c >> 7) : srow);
                const int64_t e = r * cols + c;
                float a[4];
                if constexpr (OUT_BF16) {
                    const uint2 v = __ldcs(reinterpret_cast<const uint2*>(q + e));
                    float b[4];
                    decode4<FMT>(v.x, si, a);
                    decode4<FMT>(v.y, si, b);
                    stg_evict_first(y + e * 2, make_uint4(f32x2_to_bf16x2(a[0], a[1]), f32x2_to_bf16x2(a[2], a[3]),
                                                     f32x2_to_bf16x2(b[0], b[1]), f32x2_to_bf16x2(b[2], b[3])));
                } else {
                    decode4<FMT>(__ldcs(reinterpret_cast<const unsigned int*>(q + e)), si, a);
                    stg_evict_first(y + e * 4, make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]),
                                                     __float_as_uint(a[3])));
                }
            }
        } else {
            for (int64_t c = (int64_t)blockIdx.x * kThreads + threadIdx.x; c < cols; c += (int64_t)gridDim.x * kThreads) {
                const float si = __ldg(br > 0 ? srow + (c >> 7) : srow);
                const int64_t e = r * cols + c;
                dequant_one<FMT, OUT_BF16>(q[e], si, y, e);
            }
        }
    }
}

template <int FMT, bool OUT_BF16>
fp8_status_t launch_deq(const uint8_t* q, int64_t rows, int64_t cols, const float* si, int br, int bc, uint8_t* y,
                        cudaStream_t st) {
    const char* w = "fp8_dequantize";
    const int64_t n = rows * cols;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (br == 0 && aligned16(q) && aligned16(y)) {
        const int64_t nitems = n / (OUT_BF16 ? 8 : 4);
        int64_t grid = (nitems + (int64_t)kThreads * kItems - 1) / ((int64_t)kThreads * kItems);
        if (grid < 1) grid = 1;
        return launch(w, dequant_tensor_kernel<FMT, OUT_BF16>, dim3((unsigned)grid), dim3(kThreads), st, q, n, si, y);
    }
    const int vec = aligned16(q) && aligned16(y) && cols % 16 == 0;
    const int64_t per_row = vec ? cols / (OUT_BF16 ? 8 : 4) : cols;
    int64_t gx = (per_row + kThreads - 1) / kThreads;
    if (gx < 1) gx = 1;
    if (gx > cap) gx = cap;
    int64_t gy = rows < 65535 ? rows : 65535;
    if (gy < 1) gy = 1;
    const int64_t nbc = bc > 0 ? (cols + bc - 1) / bc : 0;
    return launch(w, dequant_rows_kernel<FMT, OUT_BF16>, dim3((unsigned)gx, (unsigned)gy), dim3(kThreads), st, q, rows,
                  cols, si, br, nbc, y, vec);
}

}  // namespace
}  // namespace fp8q

using namespace fp8q;

extern "C" fp8_status_t fp8_dequantize(const uint8_t* q, fp8_format_t fmt, int64_t rows, int64_t cols,
                                       const float* scale_inv, int block_rows, int block_cols, void* y,
                                       fp8_dtype_t out_dtype, void* stream) {
    const char* fn = "fp8_dequantize";
    if (!valid_fmt(fmt)) return fail(FP8_ERR_INVALID_ARG, "%s: unknown format %d", fn, (int)fmt);
    if (!valid_dtype(out_dtype)) return fail(FP8_ERR_INVALID_ARG, "%s: unknown out_dtype %d", fn, (int)out_dtype);
    if (rows < 0 || cols < 0) return fail(FP8_ERR_INVALID_ARG, "%s: negative shape", fn);
    const bool per_tensor = block_rows == 0 && block_cols == 0;
    if (!per_tensor && !((block_rows == 128 && block_cols == 128) || (block_rows == 1 && block_cols == 128)))
        return fail(FP8_ERR_UNSUPPORTED, "%s: block shape %dx%d (supported: 0x0, 128x128, 1x128)", fn, block_rows,
                    block_cols);
    if (rows == 0 || cols == 0) return FP8_OK;
    if (q == nullptr || y == nullptr || scale_inv == nullptr)
        return fail(FP8_ERR_INVALID_ARG, "%s: q / y / scale_inv is NULL", fn);
    if (reinterpret_cast<uintptr_t>(y) % dtype_size(out_dtype)) return fail(FP8_ERR_INVALID_ARG, "%s: y not element-aligned", fn);
    if (reinterpret_cast<uintptr_t>(scale_inv) % 4) return fail(FP8_ERR_INVALID_ARG, "%s: scale_inv not 4-byte aligned", fn);

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* yp = static_cast<uint8_t*>(y);
    const bool bf16 = out_dtype == FP8_DT_BF16;
    if (fmt == FP8_E4M3)
        return bf16 ? launch_deq<kE4M3, true>(q, rows, cols, scale_inv, block_rows, block_cols, yp, st)
                    : launch_deq<kE4M3, false>(q, rows, cols, scale_inv, block_rows, block_cols, yp, st);
    return bf16 ? launch_deq<kE5M2, true>(q, rows, cols, scale_inv, block_rows, block_cols, yp, st)
                : launch_deq<kE5M2, false>(q, rows, cols, scale_inv, block_rows, block_cols, yp, st);
}
