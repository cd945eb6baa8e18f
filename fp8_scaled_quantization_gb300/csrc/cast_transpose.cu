// cast_transpose.cu -- one read of x, two FP8 copies under one scale: the
// rowwise codes q_row[r, c] and the columnwise (transposed) codes
// q_col[c, r] == q_row[r, c].
//
// "Megatron FP8" §6: the weight-gradient GEMM consumes transpose(dy_fp8);
// "[Pytorch][Common] Hybrid quantization #2817": Hopper-style FP8 GEMMs need
// a physically transposed columnwise copy (columnwise_source = original).
//
// One CTA (256 threads) per 128 x 128 tile.
//   Load:   16-byte loads of x; each 8-element chunk is converted to 8 codes
//           in registers (so shared memory holds bytes, not BF16), written
//           rowwise to global memory (full 128-byte lines per warp) and
//           stored into a 16 KB shared tile.  Tile words are XOR-swizzled on
//           bits 2-4 by (row / 16) % 8 so the transposed reads are free of
//           bank conflicts.
//   Store:  each thread reads a 16-row x 4-column block of codes as sixteen
//           32-bit words, transposes 4 x 4 byte blocks with byte permutes and
//           writes four 16-byte pieces of q_col; the 8 lanes sharing a column
//           cover one full 128-byte line.
// Edge tiles (and shapes / pointers that do not meet the vector rules) take
// a guarded element path inside the same kernel.
#include "fp8q_device.cuh"
#include "fp8q_host.h"

namespace fp8q {
namespace {

constexpr int kTile = 128;
constexpr int kThreads = 256;

__device__ __forceinline__ int swz(int row) { return ((row >> 4) & 7) << 2; }

// 4 x 4 byte transpose: in a[k] byte j is (row k, col j); out b[j] byte k.
__device__ __forceinline__ void transpose4x4(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t& b0,
                                             uint32_t& b1, uint32_t& b2, uint32_t& b3) {
    const uint32_t t0 = __byte_perm(a0, a1, 0x5140);  // a0.0 a1.0 a0.1 a1.1
    const uint32_t t1 = __byte_perm(a0, a1, 0x7362);  // a0.2 a1.2 a0.3 a1.3
    const uint32_t t2 = __byte_perm(a2, a3, 0x5140);
    const uint32_t t3 = __byte_perm(a2, a3, 0x7362);
    b0 = __byte_perm(t0, t2, 0x5410);
    b1 = __byte_perm(t0, t2, 0x7632);
    b2 = __byte_perm(t1, t3, 0x5410);
    b3 = __byte_perm(t1, t3, 0x7632);
}

// Where the columnwise codes come from ("[Pytorch][Common] Hybrid quantization
// #2817", columnwise_source): kSame -- the rowwise codes themselves (one format
// and scale); kOriginal -- x, in the columnwise format and scale;
// kRowDequant -- the BF16 dequantized rowwise value.
constexpr int kSame = 0, kOriginal = 1, kRowDequant = 2;

// 8 rowwise codes -> 8 BF16 values: RNE_bf16(fl32(decode(code) * scale_inv)).
template <int FMT>
__device__ __forceinline__ uint4 dequant8_bf16(uint32_t lo, uint32_t hi, float si) {
    const uint32_t w[2] = {lo, hi};
    uint32_t out[4];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const uint32_t h01 = fp8x2_to_f16x2<FMT>(w[i] & 0xFFFFu), h23 = fp8x2_to_f16x2<FMT>(w[i] >> 16);
        const float2 p01 = fmul2_rn(f16_lo_to_f32(h01), f16_hi_to_f32(h01), si);
        const float2 p23 = fmul2_rn(f16_lo_to_f32(h23), f16_hi_to_f32(h23), si);
        out[2 * i] = f32x2_to_bf16x2(p01.x, p01.y);
        out[2 * i + 1] = f32x2_to_bf16x2(p23.x, p23.y);
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
}

// Columnwise codes of 8 BF16 values (with the exact slow path for Inf / NaN).
template <int FMT_COL>
__device__ __forceinline__ Codes8 col_codes_bf16x8(uint4 v, float scale) {
    uint32_t m;
    Codes8 c = cvt_bf16x8<FMT_COL>(v, scale, &m);
    if (chunk_needs_fixup<FMT_COL, false>(fold_u16x2_to_f32bits(m), scale)) fixup_bf16x8<FMT_COL>(v, scale, &c);
    return c;
}

template <int FMT, bool BF16, bool AMAX, int FMT_COL = FMT, int SRC = kSame>
__global__ void __launch_bounds__(kThreads, 4)
cast_transpose_kernel(const uint8_t* __restrict__ x, int64_t rows, int64_t cols, const float* __restrict__ scale_ptr,
                      uint8_t* __restrict__ q_row, uint8_t* __restrict__ q_col, int vec_ok,
                      uint32_t* __restrict__ part_amax, const float* __restrict__ scale_col_ptr) {
    pdl_begin();
    __shared__ __align__(16) uint32_t tile[kTile * kTile / 4];
    const float scale = __ldg(scale_ptr);
    const float scale_col = SRC == kSame ? scale : __ldg(scale_col_ptr);
    const float scale_inv_row = SRC == kRowDequant ? __fdiv_rn(1.0f, scale) : 1.0f;
    // Tiles run in reverse order with evict_first loads: after an amax pass over
    // x (current scaling) the end of x is the part still in L2.  One tile per
    // CTA, except with the fused amax, whose grid is capped at the workspace's
    // partial slots and walks the tiles with a stride.
    const uint64_t pol = l2_policy_evict_first();
    const int t = threadIdx.x;
    uint32_t am = 0;  // fp32 bits of max |x| seen by this thread
    const int64_t gx = (cols + kTile - 1) / kTile, ntiles = gx * ((rows + kTile - 1) / kTile);
    for (int64_t tl = blockIdx.x; tl < ntiles; tl += gridDim.x) {
    const int64_t rev = ntiles - 1 - tl;
    const int64_t r0 = rev / gx * kTile, c0 = rev % gx * kTile;
    const bool full = vec_ok && r0 + kTile <= rows && c0 + kTile <= cols;
    if (full) {
        if constexpr (BF16) {
            // 16 threads per 256-byte row, 16 rows per pass, 8 passes.
            const int cc = t & 15, rsub = t >> 4;
            const uint8_t* src = x + ((r0 + rsub) * cols + c0 + cc * 8) * 2;
            uint4 v[8];
#pragma unroll
            for (int p = 0; p < 8; ++p) v[p] = ldg_stream_hint(src + (int64_t)p * 16 * cols * 2, pol);
            uint32_t m16 = 0;
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                uint32_t m;
                Codes8 c = cvt_bf16x8<FMT>(v[p], scale, &m);
                if (chunk_needs_fixup<FMT, false>(fold_u16x2_to_f32bits(m), scale)) fixup_bf16x8<FMT>(v[p], scale, &c);
                if constexpr (AMAX) m16 = max_u16x2(m16, m);
                const int r = p * 16 + rsub;
                if (q_row) stg_stream(q_row + (r0 + r) * cols + c0 + cc * 8, make_uint2(c.lo, c.hi));
                Codes8 cc8 = c;
                if constexpr (SRC == kOriginal) cc8 = col_codes_bf16x8<FMT_COL>(v[p], scale_col);
                if constexpr (SRC == kRowDequant)
                    cc8 = col_codes_bf16x8<FMT_COL>(dequant8_bf16<FMT>(c.lo, c.hi, scale_inv_row), scale_col);
                *reinterpret_cast<uint2*>(&tile[r * 32 + ((cc * 2) ^ (p << 2))]) = make_uint2(cc8.lo, cc8.hi);
            }
            if constexpr (AMAX) am = umax(am, fold_u16x2_to_f32bits(m16));
        } else {
            // 32 threads per 512-byte row, 8 rows per pass, 16 passes in two halves.
            const int lane = t & 31, rsub = t >> 5;
            const uint8_t* src = x + ((r0 + rsub) * cols + c0 + lane * 4) * 4;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint4 v[8];
#pragma unroll
                for (int p = 0; p < 8; ++p) v[p] = ldg_stream_hint(src + (int64_t)(half * 8 + p) * 8 * cols * 4, pol);
#pragma unroll
                for (int p = 0; p < 8; ++p) {
                    float4 f = make_float4(__uint_as_float(v[p].x), __uint_as_float(v[p].y), __uint_as_float(v[p].z),
                                           __uint_as_float(v[p].w));
                    uint32_t m;
                    uint32_t w = cvt_f32x4<FMT>(f, scale, &m);
                    if (chunk_needs_fixup<FMT, false>(m, scale)) fixup_f32x4<FMT>(f, scale, &w);
                    if constexpr (AMAX) am = umax(am, m);
                    const int r = (half * 8 + p) * 8 + rsub;
                    if (q_row) *reinterpret_cast<uint32_t*>(q_row + (r0 + r) * cols + c0 + lane * 4) = w;
                    uint32_t wc = w;
                    if constexpr (SRC == kOriginal) {
                        uint32_t m2;
                        wc = cvt_f32x4<FMT_COL>(f, scale_col, &m2);
                        if (chunk_needs_fixup<FMT_COL, false>(m2, scale_col)) fixup_f32x4<FMT_COL>(f, scale_col, &wc);
                    }
                    if constexpr (SRC == kRowDequant) {
                        const uint4 d = dequant8_bf16<FMT>(w, 0u, scale_inv_row);  // 4 values in d.x, d.y
                        const float4 g = make_float4(bf16lo(d.x), bf16hi(d.x), bf16lo(d.y), bf16hi(d.y));
                        uint32_t m2;
                        wc = cvt_f32x4<FMT_COL>(g, scale_col, &m2);
                        if (chunk_needs_fixup<FMT_COL, false>(m2, scale_col)) fixup_f32x4<FMT_COL>(g, scale_col, &wc);
                    }
                    tile[r * 32 + (lane ^ swz(r))] = wc;
                }
            }
        }
        __syncthreads();
        if (q_col) {
            const int warp = t >> 5, lane = t & 31;
            const int cg = warp * 4 + (lane >> 3);  // 4-column group (word index)
            const int rc = lane & 7;                // 16-row chunk
            uint32_t out[4][4];                     // [column j][row quad i]
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int rb = rc * 16 + i * 4;
                const int sw = rc << 2;  // == swz(rb + k) for k < 4
                const uint32_t a0 = tile[(rb + 0) * 32 + (cg ^ sw)];
                const uint32_t a1 = tile[(rb + 1) * 32 + (cg ^ sw)];
                const uint32_t a2 = tile[(rb + 2) * 32 + (cg ^ sw)];
                const uint32_t a3 = tile[(rb + 3) * 32 + (cg ^ sw)];
                transpose4x4(a0, a1, a2, a3, out[0][i], out[1][i], out[2][i], out[3][i]);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
                stg_stream(q_col + (c0 + cg * 4 + j) * rows + r0 + rc * 16,
                           make_uint4(out[j][0], out[j][1], out[j][2], out[j][3]));
        }
    } else {
        // Guarded element path: bytes in the tile, no swizzle.
        uint8_t* tb = reinterpret_cast<uint8_t*>(tile);
        for (int i = t; i < kTile * kTile; i += kThreads) {
            const int r = i >> 7, c = i & (kTile - 1);
            if (r0 + r < rows && c0 + c < cols) {
                const int64_t e = (r0 + r) * cols + c0 + c;
                float xv;
                uint32_t b;
                if constexpr (BF16) {
                    uint16_t h = reinterpret_cast<const uint16_t*>(x)[e];
                    xv = __uint_as_float((uint32_t)h << 16);
                    b = (uint32_t)(h & 0x7FFFu) << 16;
                } else {
                    xv = reinterpret_cast<const float*>(x)[e];
                    b = __float_as_uint(xv) & 0x7FFFFFFFu;
                }
                uint32_t s;
                const uint8_t code = (uint8_t)quant_one<FMT>(xv, scale, &s);
                am = umax(am, b);
                if (q_row) q_row[e] = code;
                uint8_t ccode = code;
                if constexpr (SRC == kOriginal) ccode = (uint8_t)quant_one<FMT_COL>(xv, scale_col, &s);
                if constexpr (SRC == kRowDequant) {
                    const uint4 d = dequant8_bf16<FMT>(code, 0u, scale_inv_row);
                    ccode = (uint8_t)quant_one<FMT_COL>(bf16lo(d.x), scale_col, &s);
                }
                tb[r * kTile + c] = ccode;
            }
        }
        __syncthreads();
        if (q_col) {
            for (int i = t; i < kTile * kTile; i += kThreads) {
                const int c = i >> 7, r = i & (kTile - 1);
                if (r0 + r < rows && c0 + c < cols) q_col[(c0 + c) * rows + r0 + r] = tb[r * kTile + c];
            }
        }
    }
    __syncthreads();  // the shared tile is rewritten by the next tile of this CTA
    }

    if constexpr (AMAX) {
        __shared__ uint32_t red[32];
        const uint32_t bits = block_max_u32(am, red);
        if (threadIdx.x == 0) part_amax[blockIdx.x] = bits;
    }
}

template <int FMT, bool BF16>
fp8_status_t launch_ct(bool amax, dim3 grid, cudaStream_t st, const uint8_t* x, int64_t rows, int64_t cols,
                       const float* scale, uint8_t* q_row, uint8_t* q_col, int vec_ok, uint32_t* pa) {
    const char* w = "fp8_quantize_cast_transpose";
    if (amax)
        return launch(w, cast_transpose_kernel<FMT, BF16, true>, grid, dim3(kThreads), st, x, rows, cols, scale, q_row,
                      q_col, vec_ok, pa, static_cast<const float*>(nullptr));
    return launch(w, cast_transpose_kernel<FMT, BF16, false>, grid, dim3(kThreads), st, x, rows, cols, scale, q_row,
                  q_col, vec_ok, pa, static_cast<const float*>(nullptr));
}

}  // namespace
}  // namespace fp8q

using namespace fp8q;

extern "C" fp8_status_t fp8_quantize_cast_transpose(const void* x, fp8_dtype_t dtype, int64_t rows, int64_t cols,
                                                    fp8_format_t fmt, const float* scale, uint8_t* q_row,
                                                    uint8_t* q_col, float* amax_out, void* stream) {
    const char* fn = "fp8_quantize_cast_transpose";
    if (!valid_dtype(dtype)) return fail(FP8_ERR_INVALID_ARG, "%s: unknown dtype %d", fn, (int)dtype);
    if (!valid_fmt(fmt)) return fail(FP8_ERR_INVALID_ARG, "%s: unknown format %d", fn, (int)fmt);
    if (rows < 0 || cols < 0) return fail(FP8_ERR_INVALID_ARG, "%s: negative shape", fn);
    if (scale == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: scale is NULL", fn);
    const int64_t n = rows * cols;
    if (n > 0 && q_row == nullptr && q_col == nullptr)
        return fail(FP8_ERR_INVALID_ARG, "%s: q_row and q_col are both NULL", fn);
    if (n > 0 && x == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: x is NULL", fn);
    if (reinterpret_cast<uintptr_t>(x) % dtype_size(dtype)) return fail(FP8_ERR_INVALID_ARG, "%s: x not element-aligned", fn);
    const int64_t ntiles = ((cols + kTile - 1) / kTile) * ((rows + kTile - 1) / kTile);

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Workspace* ws = nullptr;
    if (amax_out) {
        fp8_status_t s;
        ws = stream_workspace(st, &s);
        if (!ws) return s;
    }
    if (n == 0 && !amax_out) return FP8_OK;
    // One CTA per tile; with the fused amax at most one CTA per partial slot
    // (n == 0: one CTA with nothing to do but report amax 0).
    int64_t g = ntiles;
    if (amax_out && g > kMaxPartials) g = kMaxPartials;
    if (g > 0x7FFFFFFF) g = 0x7FFFFFFF;
    if (g < 1) g = 1;
    const dim3 grid((unsigned)g);
    const int vec_ok = aligned16(x) && (q_row == nullptr || aligned16(q_row)) && (q_col == nullptr || aligned16(q_col)) &&
                       cols % 16 == 0 && rows % 16 == 0;
    const uint8_t* xp = static_cast<const uint8_t*>(x);
    const bool bf16 = dtype == FP8_DT_BF16, am = amax_out != nullptr;
    uint32_t* pa = am ? ws->amax : nullptr;
    fp8_status_t s;
    if (fmt == FP8_E4M3)
        s = bf16 ? launch_ct<kE4M3, true>(am, grid, st, xp, rows, cols, scale, q_row, q_col, vec_ok, pa)
                 : launch_ct<kE4M3, false>(am, grid, st, xp, rows, cols, scale, q_row, q_col, vec_ok, pa);
    else
        s = bf16 ? launch_ct<kE5M2, true>(am, grid, st, xp, rows, cols, scale, q_row, q_col, vec_ok, pa)
                 : launch_ct<kE5M2, false>(am, grid, st, xp, rows, cols, scale, q_row, q_col, vec_ok, pa);
    if (s != FP8_OK || !am) return s;
    FinalizeArgs fa;
    fa.part_amax = ws->amax;
    fa.nparts = (int)grid.x;
    fa.amax_out = amax_out;
    fa.fmt = (int)fmt;
    return launch_finalize(fa, st);
}

extern "C" fp8_status_t fp8_quantize_hybrid(const void* x, fp8_dtype_t dtype, int64_t rows, int64_t cols,
                                            fp8_format_t fmt_row, const float* scale_row, uint8_t* q_row,
                                            fp8_format_t fmt_col, const float* scale_col, uint8_t* q_col,
                                            fp8_columnwise_source_t source, void* stream) {
    const char* fn = "fp8_quantize_hybrid";
    if (!valid_dtype(dtype)) return fail(FP8_ERR_INVALID_ARG, "%s: unknown dtype %d", fn, (int)dtype);
    if (!valid_fmt(fmt_row) || !valid_fmt(fmt_col)) return fail(FP8_ERR_INVALID_ARG, "%s: unknown format", fn);
    if (source != FP8_COLUMNWISE_FROM_ORIGINAL && source != FP8_COLUMNWISE_FROM_ROWWISE_DEQUANTIZED)
        return fail(FP8_ERR_INVALID_ARG, "%s: unknown columnwise source %d", fn, (int)source);
    if (rows < 0 || cols < 0) return fail(FP8_ERR_INVALID_ARG, "%s: negative shape", fn);
    if (scale_row == nullptr || scale_col == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: scale is NULL", fn);
    const int64_t n = rows * cols;
    if (n == 0) return FP8_OK;
    if (x == nullptr || q_row == nullptr || q_col == nullptr)
        return fail(FP8_ERR_INVALID_ARG, "%s: x / q_row / q_col is NULL", fn);
    if (reinterpret_cast<uintptr_t>(x) % dtype_size(dtype)) return fail(FP8_ERR_INVALID_ARG, "%s: x not element-aligned", fn);
    int64_t g = ((cols + kTile - 1) / kTile) * ((rows + kTile - 1) / kTile);
    if (g > 0x7FFFFFFF) g = 0x7FFFFFFF;
    const int vec_ok = aligned16(x) && aligned16(q_row) && aligned16(q_col) && cols % 16 == 0 && rows % 16 == 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint8_t* xp = static_cast<const uint8_t*>(x);
    const dim3 grid((unsigned)g), block(kThreads);
    uint32_t* none = nullptr;
    const bool deq = source == FP8_COLUMNWISE_FROM_ROWWISE_DEQUANTIZED;
#define FP8Q_HYB(FR, FC, B)                                                                                           \
    (deq ? launch(fn, cast_transpose_kernel<FR, B, false, FC, kRowDequant>, grid, block, st, xp, rows, cols, scale_row, \
                  q_row, q_col, vec_ok, none, scale_col)                                                              \
         : launch(fn, cast_transpose_kernel<FR, B, false, FC, kOriginal>, grid, block, st, xp, rows, cols, scale_row,   \
                  q_row, q_col, vec_ok, none, scale_col))
    const bool bf16 = dtype == FP8_DT_BF16;
    if (fmt_row == FP8_E4M3 && fmt_col == FP8_E4M3) return bf16 ? FP8Q_HYB(kE4M3, kE4M3, true) : FP8Q_HYB(kE4M3, kE4M3, false);
    if (fmt_row == FP8_E4M3) return bf16 ? FP8Q_HYB(kE4M3, kE5M2, true) : FP8Q_HYB(kE4M3, kE5M2, false);
    if (fmt_col == FP8_E4M3) return bf16 ? FP8Q_HYB(kE5M2, kE4M3, true) : FP8Q_HYB(kE5M2, kE4M3, false);
    return bf16 ? FP8Q_HYB(kE5M2, kE5M2, true) : FP8Q_HYB(kE5M2, kE5M2, false);
#undef FP8Q_HYB
}
