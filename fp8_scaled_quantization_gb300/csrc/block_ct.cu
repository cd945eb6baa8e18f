// block_ct.cu -- blockwise cast + transpose: one read of x gives rowwise codes
// with one fp32 scale per 1 x 128 row tile and columnwise codes (written
// transposed) with one fp32 scale per 128 x 1 column tile.
//
// "[Pytorch][Common] Hybrid quantization #2817": the backward GEMM consumes a
// columnwise copy (Float8Blockwise sub-storage, columnwise_source = original);
// "Low Precision Training and Rollout": FP32 block scales, the stored factor
// being the inverse scale.  The columnwise copy is exactly the 1 x 128
// blockwise quantization of x^T, so q_col[c, r] and scale_inv_col[c, r / 128]
// follow the same scale rule (margin 0) as the rowwise copy.
//
// Fast path (BF16, rows % 128 == 0, cols % 128 == 0, 16-byte aligned): one CTA
// per 128 x 128 tile; each thread holds 8 rows x 8 columns of x in registers.
//   rows:    the 16 lanes sharing a row reduce its 1 x 128 amax by shuffles,
//            two rows per 32-bit word (u16x2); 8 lanes each derive one row's
//            scale and shuffle it.
//   columns: each thread folds its 8 rows per column pair (u16x2), a 16 x 64
//            shared table completes the 128-row reduction, 64 threads derive
//            two column scales each; two rows of a column share its scale, so
//            one two-lane multiply and one two-value cvt give both codes; the
//            codes go through a swizzled byte-transpose tile (16-byte stores,
//            full lines).
//   Scales come from block_scale_bf16 (exact tables, no division); the
//   element-exact fixup runs only for a row or tile holding Inf / NaN.
#include "fp8q_device.cuh"
#include "fp8q_host.h"

namespace fp8q {
namespace {

constexpr int kTile = 128;
constexpr int kThreads = 256;

__device__ __forceinline__ void transpose4x4_b(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t& b0,
                                               uint32_t& b1, uint32_t& b2, uint32_t& b3) {
    const uint32_t t0 = __byte_perm(a0, a1, 0x5140);
    const uint32_t t1 = __byte_perm(a0, a1, 0x7362);
    const uint32_t t2 = __byte_perm(a2, a3, 0x5140);
    const uint32_t t3 = __byte_perm(a2, a3, 0x7362);
    b0 = __byte_perm(t0, t2, 0x5410);
    b1 = __byte_perm(t0, t2, 0x7632);
    b2 = __byte_perm(t1, t3, 0x5410);
    b3 = __byte_perm(t1, t3, 0x7632);
}

// At most 64 registers: 4 CTAs (1024 threads) per SM.
template <int FMT>
__global__ void __launch_bounds__(kThreads, 4)
block_ct_kernel(const uint8_t* __restrict__ x, int64_t rows, int64_t cols, uint8_t* __restrict__ q_row,
                float* __restrict__ si_row, uint8_t* __restrict__ q_col, float* __restrict__ si_col) {
    const uint32_t tword = table_word<FMT>(threadIdx.x);
    pdl_begin();
    __shared__ __align__(16) uint32_t tile[kTile * kTile / 4];  // columnwise codes, swizzled
    __shared__ uint32_t tab[256];
    __shared__ __align__(16) uint32_t colmax2[16][kTile / 2];    // per row group: column-pair maxima (u16x2)
    __shared__ float colscale[kTile];
    const int64_t nbr_row = cols / 128, nbr_col = rows / 128;
    const int64_t r0 = (int64_t)blockIdx.x / nbr_row * kTile, c0 = (int64_t)blockIdx.x % nbr_row * kTile;
    const int t = threadIdx.x, lane = t & 31, cc = t & 15, rsub = t >> 4;

    uint4 v[8];  // v[p]: row p * 16 + rsub, columns cc * 8 .. cc * 8 + 7
#pragma unroll
    for (int p = 0; p < 8; ++p) v[p] = ldg_stream(x + ((r0 + p * 16 + rsub) * cols + c0 + cc * 8) * 2);
    tab[t] = tword;
    __syncthreads();

    // ---- rowwise 1 x 128 tiles: the half-warp of 16 lanes holds one row per p.
    // Rows p = 2j and 2j + 1 share a word (low / high 16 bits of their |x| bit
    // patterns), so one u16x2 shuffle-max reduction serves two rows.
    uint32_t rm2[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint4 a = v[2 * j], b = v[2 * j + 1];
        const uint32_t ma = max_u16x2(max_u16x2(abs_bf16x2(a.x), abs_bf16x2(a.y)),
                                      max_u16x2(abs_bf16x2(a.z), abs_bf16x2(a.w)));
        const uint32_t mb = max_u16x2(max_u16x2(abs_bf16x2(b.x), abs_bf16x2(b.y)),
                                      max_u16x2(abs_bf16x2(b.z), abs_bf16x2(b.w)));
        uint32_t w = max_u16x2(__byte_perm(ma, mb, 0x5410), __byte_perm(ma, mb, 0x7632));
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) w = max_u16x2(w, __shfl_xor_sync(0xFFFFFFFFu, w, o));
        rm2[j] = w;
    }
    uint32_t mine2 = rm2[0];
#pragma unroll
    for (int j = 1; j < 4; ++j) mine2 = (cc >> 1) == j ? rm2[j] : mine2;
    float rs, rsi;  // lane cc < 8: the scale of row p = cc
    block_scale_bf16<FMT>(tab, (cc & 1) ? (mine2 & 0xFFFF0000u) : (mine2 << 16), &rs, &rsi);
    if (q_row != nullptr && cc < 8) si_row[(r0 + cc * 16 + rsub) * nbr_row + (c0 >> 7)] = rsi;

    // ---- column partial maxima over this thread's 8 rows (column pairs as u16x2)
    if (q_col != nullptr) {
        uint4 cm = make_uint4(0u, 0u, 0u, 0u);  // columns (2k, 2k + 1) of the thread's 8 in word k
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            cm.x = max_u16x2(cm.x, abs_bf16x2(v[p].x));
            cm.y = max_u16x2(cm.y, abs_bf16x2(v[p].y));
            cm.z = max_u16x2(cm.z, abs_bf16x2(v[p].z));
            cm.w = max_u16x2(cm.w, abs_bf16x2(v[p].w));
        }
        *reinterpret_cast<uint4*>(&colmax2[rsub][cc * 4]) = cm;
    }

    // ---- rowwise codes; the element-exact fixup only for a row holding Inf / NaN
    if (q_row != nullptr) {
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            const float scale = __shfl_sync(0xFFFFFFFFu, rs, (lane & 16) | p);
            const uint32_t rmax = (p & 1) ? (rm2[p >> 1] & 0xFFFF0000u) : (rm2[p >> 1] << 16);
            Codes8 c = cvt_bf16x8_nomax<FMT>(v[p], scale);
            if (rmax >= 0x7F800000u) fixup_bf16x8<FMT>(v[p], scale, &c);
            stg_stream(q_row + (r0 + p * 16 + rsub) * cols + c0 + cc * 8, make_uint2(c.lo, c.hi));
        }
    }
    if (q_col == nullptr) return;

    // ---- column scales, two columns per thread; `special`: some column of the
    // tile holds Inf / NaN
    __syncthreads();
    uint32_t cb2 = 0;
    if (t < kTile / 2) {
#pragma unroll
        for (int g = 0; g < 16; ++g) cb2 = max_u16x2(cb2, colmax2[g][t]);
        float s0, si0, s1, si1;
        block_scale_bf16<FMT>(tab, cb2 << 16, &s0, &si0);
        block_scale_bf16<FMT>(tab, cb2 & 0xFFFF0000u, &s1, &si1);
        *reinterpret_cast<float2*>(&colscale[2 * t]) = make_float2(s0, s1);
        si_col[(c0 + 2 * t) * nbr_col + (r0 >> 7)] = si0;
        si_col[(c0 + 2 * t + 1) * nbr_col + (r0 >> 7)] = si1;
    }
    const int special = __syncthreads_or(t < kTile / 2 && ((cb2 & 0xFFFFu) >= 0x7F80u || cb2 >= 0x7F800000u));

    // ---- columnwise codes into the swizzled tile, then transposed 16-byte stores.
    // Rows p and p + 1 of one column share its scale, so one two-lane multiply
    // and one two-value cvt give both codes; byte permutes then form each
    // row's 4-byte words.  With no Inf / NaN in a column, |x * scale| <= its
    // amax * scale, so the round-to-nearest-even saturating cvt is the exact
    // per-element rule.
    float cs[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) cs[j] = colscale[cc * 8 + j];
    if (!special) {
#pragma unroll
        for (int p = 0; p < 8; p += 2) {
            const uint32_t a[4] = {v[p].x, v[p].y, v[p].z, v[p].w};
            const uint32_t bq[4] = {v[p + 1].x, v[p + 1].y, v[p + 1].z, v[p + 1].w};
            uint32_t pr[4];  // pr[h]: bytes (row p, col 2h), (row p+1, col 2h), (row p, col 2h+1), (row p+1, col 2h+1)
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const float2 l = fmul2_rn(bf16lo(a[h]), bf16lo(bq[h]), cs[2 * h]);
                const float2 u = fmul2_rn(bf16hi(a[h]), bf16hi(bq[h]), cs[2 * h + 1]);
                pr[h] = __byte_perm(cvt2<FMT>(l.x, l.y), cvt2<FMT>(u.x, u.y), 0x5410);
            }
            const uint32_t lo0 = __byte_perm(pr[0], pr[1], 0x6420), lo1 = __byte_perm(pr[0], pr[1], 0x7531);
            const uint32_t hi0 = __byte_perm(pr[2], pr[3], 0x6420), hi1 = __byte_perm(pr[2], pr[3], 0x7531);
            const int r = p * 16 + rsub;
            *reinterpret_cast<uint2*>(&tile[r * 32 + ((cc * 2) ^ (p << 2))]) = make_uint2(lo0, hi0);
            *reinterpret_cast<uint2*>(&tile[(r + 16) * 32 + ((cc * 2) ^ ((p + 1) << 2))]) = make_uint2(lo1, hi1);
        }
    } else {
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            const uint32_t w[4] = {v[p].x, v[p].y, v[p].z, v[p].w};
            uint32_t code[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint32_t sat;
                code[j] = quant_one<FMT>((j & 1) ? bf16hi(w[j >> 1]) : bf16lo(w[j >> 1]), cs[j], &sat);
            }
            const uint32_t lo = code[0] | (code[1] << 8) | (code[2] << 16) | (code[3] << 24);
            const uint32_t hi = code[4] | (code[5] << 8) | (code[6] << 16) | (code[7] << 24);
            const int r = p * 16 + rsub;
            *reinterpret_cast<uint2*>(&tile[r * 32 + ((cc * 2) ^ (p << 2))]) = make_uint2(lo, hi);
        }
    }
    __syncthreads();
    {
        const int warp = t >> 5;
        const int cg = warp * 4 + (lane >> 3);
        const int rc = lane & 7;
        uint32_t out[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int rb = rc * 16 + i * 4;
            const int sw = rc << 2;
            transpose4x4_b(tile[(rb + 0) * 32 + (cg ^ sw)], tile[(rb + 1) * 32 + (cg ^ sw)],
                           tile[(rb + 2) * 32 + (cg ^ sw)], tile[(rb + 3) * 32 + (cg ^ sw)], out[0][i], out[1][i],
                           out[2][i], out[3][i]);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
            stg_stream(q_col + (c0 + cg * 4 + j) * rows + r0 + rc * 16,
                       make_uint4(out[j][0], out[j][1], out[j][2], out[j][3]));
    }
}

// Guarded path: one half-warp per 128-element tile along a line (rowwise:
// a row of x; columnwise: a column of x, written as a row of q_col).
template <int FMT, bool BF16>
__global__ void __launch_bounds__(kThreads)
line128_guarded_kernel(const uint8_t* __restrict__ x, int64_t nlines, int64_t len, int64_t line_stride,
                       int64_t elem_stride, uint8_t* __restrict__ q, float* __restrict__ si) {
    pdl_begin();
    const int t = threadIdx.x, hw = t >> 4, l16 = t & 15;
    const int64_t nb = (len + 127) / 128, ntiles = nlines * nb;
    for (int64_t tile0 = (int64_t)blockIdx.x * 16; tile0 < ntiles; tile0 += (int64_t)gridDim.x * 16) {
        const int64_t tl = tile0 + hw;
        const bool live = tl < ntiles;
        const int64_t line = live ? tl / nb : 0, b = live ? tl % nb : 0;
        const int64_t i0 = b * 128, i1 = i0 + 128 < len ? i0 + 128 : len;
        uint32_t am = 0;
        if (live)
            for (int64_t i = i0 + l16; i < i1; i += 16) {
                const int64_t e = line * line_stride + i * elem_stride;
                const uint32_t bits = BF16 ? (uint32_t)(reinterpret_cast<const uint16_t*>(x)[e] & 0x7FFFu) << 16
                                           : (reinterpret_cast<const uint32_t*>(x)[e] & 0x7FFFFFFFu);
                am = umax(am, bits);
            }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) am = umax(am, __shfl_xor_sync(0xFFFFFFFFu, am, o));
        float sc, s_inv;
        scale_from_amax<FMT>(__uint_as_float(am), 0, &sc, &s_inv);
        if (!live) continue;
        if (l16 == 0) si[line * nb + b] = s_inv;
        for (int64_t i = i0 + l16; i < i1; i += 16) {
            const int64_t e = line * line_stride + i * elem_stride;
            const float xv = BF16 ? __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(x)[e] << 16)
                                  : reinterpret_cast<const float*>(x)[e];
            uint32_t sat;
            q[line * len + i] = (uint8_t)quant_one<FMT>(xv, sc, &sat);
        }
    }
}

template <int FMT>
fp8_status_t launch_bct(const uint8_t* x, bool bf16, int64_t rows, int64_t cols, uint8_t* q_row, float* si_row,
                        uint8_t* q_col, float* si_col, cudaStream_t st) {
    const char* w = "fp8_quantize_block_cast_transpose";
    const bool fast = bf16 && rows % kTile == 0 && cols % kTile == 0 && aligned16(x) && (!q_row || aligned16(q_row)) &&
                      (!q_col || aligned16(q_col)) && (rows / kTile) * (cols / kTile) <= 0x7FFFFFFF;
    if (fast)
        return launch(w, block_ct_kernel<FMT>, dim3((unsigned)((rows / kTile) * (cols / kTile))), dim3(kThreads), st, x,
                      rows, cols, q_row, si_row, q_col, si_col);
    const int64_t cap = (int64_t)sm_count() * 8;
    const int64_t one = 1;
    if (q_row) {
        int64_t g = (rows * ((cols + 127) / 128) + 15) / 16;
        g = g < 1 ? 1 : (g > cap ? cap : g);
        fp8_status_t s = bf16 ? launch(w, line128_guarded_kernel<FMT, true>, dim3((unsigned)g), dim3(kThreads), st, x,
                                       rows, cols, cols, one, q_row, si_row)
                              : launch(w, line128_guarded_kernel<FMT, false>, dim3((unsigned)g), dim3(kThreads), st, x,
                                       rows, cols, cols, one, q_row, si_row);
        if (s != FP8_OK) return s;
    }
    if (q_col) {
        int64_t g = (cols * ((rows + 127) / 128) + 15) / 16;
        g = g < 1 ? 1 : (g > cap ? cap : g);
        return bf16 ? launch(w, line128_guarded_kernel<FMT, true>, dim3((unsigned)g), dim3(kThreads), st, x, cols, rows,
                             one, cols, q_col, si_col)
                    : launch(w, line128_guarded_kernel<FMT, false>, dim3((unsigned)g), dim3(kThreads), st, x, cols,
                             rows, one, cols, q_col, si_col);
    }
    return FP8_OK;
}

}  // namespace
}  // namespace fp8q

using namespace fp8q;

extern "C" fp8_status_t fp8_quantize_block_cast_transpose(const void* x, fp8_dtype_t dtype, int64_t rows,
                                                          int64_t cols, fp8_format_t fmt, uint8_t* q_row,
                                                          float* scale_inv_row, uint8_t* q_col, float* scale_inv_col,
                                                          void* stream) {
    const char* fn = "fp8_quantize_block_cast_transpose";
    if (!valid_dtype(dtype)) return fail(FP8_ERR_INVALID_ARG, "%s: unknown dtype %d", fn, (int)dtype);
    if (!valid_fmt(fmt)) return fail(FP8_ERR_INVALID_ARG, "%s: unknown format %d", fn, (int)fmt);
    if (rows < 0 || cols < 0) return fail(FP8_ERR_INVALID_ARG, "%s: negative shape", fn);
    if ((q_row == nullptr) != (scale_inv_row == nullptr) || (q_col == nullptr) != (scale_inv_col == nullptr))
        return fail(FP8_ERR_INVALID_ARG, "%s: each direction needs both its codes and its scales", fn);
    if (rows == 0 || cols == 0) return FP8_OK;
    if (x == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: x is NULL", fn);
    if (q_row == nullptr && q_col == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: no output requested", fn);
    if (reinterpret_cast<uintptr_t>(x) % dtype_size(dtype)) return fail(FP8_ERR_INVALID_ARG, "%s: x not element-aligned", fn);
    if ((scale_inv_row && reinterpret_cast<uintptr_t>(scale_inv_row) % 4) ||
        (scale_inv_col && reinterpret_cast<uintptr_t>(scale_inv_col) % 4))
        return fail(FP8_ERR_INVALID_ARG, "%s: scale_inv not 4-byte aligned", fn);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint8_t* xp = static_cast<const uint8_t*>(x);
    const bool bf16 = dtype == FP8_DT_BF16;
    if (fmt == FP8_E4M3) return launch_bct<kE4M3>(xp, bf16, rows, cols, q_row, scale_inv_row, q_col, scale_inv_col, st);
    return launch_bct<kE5M2>(xp, bf16, rows, cols, q_row, scale_inv_row, q_col, scale_inv_col, st);
}
