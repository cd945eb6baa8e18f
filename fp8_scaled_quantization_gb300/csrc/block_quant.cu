// block_quant.cu -- block-scaled quantize with one fp32 scale per 128 x 128
// block or per 1 x 128 row tile; the stored factor is scale_inv.
//
// "Low Precision Training and Rollout": 128 x 128 block FP8 ("BF16 Training
// with FP8 Rollout"), FP32 block scales ("FP8 Quick Start"), the inverse
// scale stored per block ("MXFP8 (Blackwell only)", weight_scale_inv).  The
// 1 x 128 tile is the activation-side Float8Blockwise shape of
// "[Pytorch][Common] Hybrid quantization #2817".
//
// Single pass over x: a block is held in registers while its amax is reduced,
// then converted with that block's scale (3 bytes of HBM traffic per element
// plus 4 bytes per block).
//   128 x 128: one CTA of 256 threads per block, 64 elements per thread.
//   1 x 128:   one half-warp per tile, 8 elements per lane, eight tiles in
//              flight per half-warp; the eight scales are computed one per
//              lane and shuffled back.
// Block scales of BF16 data come from block_scale_bf16 (exact tables, no
// division); the element-exact fixup runs only in blocks whose amax is Inf /
// NaN, decided once per block from the amax already reduced.
#include "fp8q_device.cuh"
#include "fp8q_host.h"

namespace fp8q {
namespace {

constexpr int kThreads = 256;

// --------------------------------------------------------------- 128 x 128

template <int FMT, bool BF16>
__global__ void __launch_bounds__(kThreads)
block128_kernel(const uint8_t* __restrict__ x, int64_t rows, int64_t cols, uint8_t* __restrict__ q,
                float* __restrict__ scale_inv, int64_t nbc, int vec_ok) {
    const uint32_t tword = BF16 ? table_word<FMT>(threadIdx.x) : 0u;
    pdl_begin();
    __shared__ uint32_t red[32];
    __shared__ float s_scale;
    __shared__ uint32_t tab[256];
    const int64_t bid = blockIdx.x;  // block (bid / nbc, bid % nbc) of the row-major block grid
    const int64_t r0 = bid / nbc * 128, c0 = bid % nbc * 128;
    const int t = threadIdx.x;
    const bool full = vec_ok && r0 + 128 <= rows && c0 + 128 <= cols;

    if (full && BF16) {
        const int cc = t & 15, rsub = t >> 4;
        const uint8_t* src = x + ((r0 + rsub) * cols + c0 + cc * 8) * 2;
        uint4 v[8];
#pragma unroll
        for (int p = 0; p < 8; ++p) v[p] = ldg_stream(src + (int64_t)p * 16 * cols * 2);
        tab[t] = tword;  // visible to thread 0 after block_max_u32's barriers
        uint32_t m16 = 0;
#pragma unroll
        for (int p = 0; p < 8; ++p)
            m16 = max_u16x2(m16, max_u16x2(max_u16x2(abs_bf16x2(v[p].x), abs_bf16x2(v[p].y)),
                                           max_u16x2(abs_bf16x2(v[p].z), abs_bf16x2(v[p].w))));
        const uint32_t bits = block_max_u32(fold_u16x2_to_f32bits(m16), red);
        if (t == 0) {
            float sc, si;  // a NaN amax (bits above Inf) gets scale 1 from the scale rule
            block_scale_bf16<FMT>(tab, bits, &sc, &si);
            s_scale = sc;
            scale_inv[bid] = si;
        }
        __syncthreads();
        const float scale = s_scale;
        const bool special = bits >= 0x7F800000u;  // the block holds Inf / NaN: element-exact codes
        uint8_t* dst = q + (r0 + rsub) * cols + c0 + cc * 8;
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            Codes8 c = cvt_bf16x8_nomax<FMT>(v[p], scale);
            if (special) fixup_bf16x8<FMT>(v[p], scale, &c);
            stg_stream(dst + (int64_t)p * 16 * cols, make_uint2(c.lo, c.hi));
        }
        return;
    }

    // Guarded element path (edges, fp32 input, unaligned): two sweeps over the
    // block, the second one re-reading x through the cache.
    const int64_t rn = rows - r0 < 128 ? rows - r0 : 128, cn = cols - c0 < 128 ? cols - c0 : 128;
    uint32_t am = 0;
    for (int i = t; i < 128 * 128; i += kThreads) {
        const int r = i >> 7, c = i & 127;
        if (r < rn && c < cn) {
            const int64_t e = (r0 + r) * cols + c0 + c;
            uint32_t b = BF16 ? (uint32_t)(reinterpret_cast<const uint16_t*>(x)[e] & 0x7FFFu) << 16
                              : (reinterpret_cast<const uint32_t*>(x)[e] & 0x7FFFFFFFu);
            am = umax(am, b);
        }
    }
    const uint32_t bits = block_max_u32(am, red);
    if (t == 0) {
        float sc, si;
        scale_from_amax<FMT>(__uint_as_float(bits), 0, &sc, &si);
        s_scale = sc;
        scale_inv[bid] = si;
    }
    __syncthreads();
    const float scale = s_scale;
    for (int i = t; i < 128 * 128; i += kThreads) {
        const int r = i >> 7, c = i & 127;
        if (r < rn && c < cn) {
            const int64_t e = (r0 + r) * cols + c0 + c;
            const float xv = BF16 ? __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(x)[e] << 16)
                                  : reinterpret_cast<const float*>(x)[e];
            uint32_t s;
            q[e] = (uint8_t)quant_one<FMT>(xv, scale, &s);
        }
    }
}

// ------------------------------------------------------------------ 1 x 128

constexpr int kTilesInFlight = 8;  // per half-warp: 8 independent 16-byte loads per lane

// Fast path: cols % 128 == 0, x and q 16-byte aligned, BF16 input; the tiles
// are then the consecutive 128-element segments of the flat array.
template <int FMT>
__global__ void __launch_bounds__(kThreads)
row128_bf16_kernel(const uint8_t* __restrict__ x, int64_t ntiles, uint8_t* __restrict__ q,
                   float* __restrict__ scale_inv) {
    __shared__ uint32_t tab[256];
    const uint32_t tword = table_word<FMT>(threadIdx.x);
    pdl_begin();
    const int t = threadIdx.x;
    const int hw = t >> 4, l16 = t & 15;
    const int lane = t & 31;
    bool tab_ready = false;
    constexpr int kTilesPerCta = (kThreads / 16) * kTilesInFlight;
    for (int64_t base = (int64_t)blockIdx.x * kTilesPerCta; base < ntiles; base += (int64_t)gridDim.x * kTilesPerCta) {
        uint4 v[kTilesInFlight];
#pragma unroll
        for (int k = 0; k < kTilesInFlight; ++k) {
            const int64_t tile = base + k * 16 + hw;
            v[k] = tile < ntiles ? ldg_stream(x + tile * 256 + l16 * 16) : make_uint4(0, 0, 0, 0);
        }
        if (!tab_ready) {  // first chunk (every thread of the CTA walks the same chunks)
            tab[t] = tword;
            __syncthreads();
            tab_ready = true;
        }
        // Tile amax: two tiles per 32-bit word (tile 2j in the low half, 2j + 1
        // in the high half, each the top 16 bits of its |x| bit pattern), so one
        // u16x2 shuffle-max reduction over the half-warp serves two tiles.
        uint32_t amx2[kTilesInFlight / 2];
#pragma unroll
        for (int j = 0; j < kTilesInFlight / 2; ++j) {
            const uint4 a = v[2 * j], b = v[2 * j + 1];
            const uint32_t ma = max_u16x2(max_u16x2(abs_bf16x2(a.x), abs_bf16x2(a.y)),
                                          max_u16x2(abs_bf16x2(a.z), abs_bf16x2(a.w)));
            const uint32_t mb = max_u16x2(max_u16x2(abs_bf16x2(b.x), abs_bf16x2(b.y)),
                                          max_u16x2(abs_bf16x2(b.z), abs_bf16x2(b.w)));
            // low halves of ma / mb in one word, high halves in another: the max
            // of the two words is (amax of tile 2j, amax of tile 2j + 1)
            uint32_t w = max_u16x2(__byte_perm(ma, mb, 0x5410), __byte_perm(ma, mb, 0x7632));
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) w = max_u16x2(w, __shfl_xor_sync(0xFFFFFFFFu, w, o));
            amx2[j] = w;
        }
        // Lane l16 < kTilesInFlight of each half-warp derives the scale of tile k = l16.
        uint32_t mine2 = amx2[0];
#pragma unroll
        for (int j = 1; j < kTilesInFlight / 2; ++j) mine2 = (l16 >> 1) == j ? amx2[j] : mine2;
        const uint32_t mine = (l16 & 1) ? (mine2 & 0xFFFF0000u) : (mine2 << 16);
        float sc, si;
        block_scale_bf16<FMT>(tab, mine, &sc, &si);
        if (l16 < kTilesInFlight) {
            const int64_t tile = base + l16 * 16 + hw;
            if (tile < ntiles) scale_inv[tile] = si;
        }
#pragma unroll
        for (int k = 0; k < kTilesInFlight; ++k) {
            const float scale = __shfl_sync(0xFFFFFFFFu, sc, (lane & 16) | k);
            const int64_t tile = base + k * 16 + hw;
            if (tile >= ntiles) continue;
            const uint32_t tmax = (k & 1) ? (amx2[k >> 1] & 0xFFFF0000u) : (amx2[k >> 1] << 16);
            Codes8 c = cvt_bf16x8_nomax<FMT>(v[k], scale);
            if (tmax >= 0x7F800000u) fixup_bf16x8<FMT>(v[k], scale, &c);  // the tile holds Inf / NaN
            stg_stream(q + tile * 128 + l16 * 8, make_uint2(c.lo, c.hi));
        }
    }
}

// Guarded path: one half-warp per (row, 128-column tile), any shape / dtype.
template <int FMT, bool BF16>
__global__ void __launch_bounds__(kThreads)
row128_guarded_kernel(const uint8_t* __restrict__ x, int64_t rows, int64_t cols, int64_t nbc,
                      uint8_t* __restrict__ q, float* __restrict__ scale_inv) {
    pdl_begin();
    const int t = threadIdx.x, hw = t >> 4, l16 = t & 15;
    const int64_t ntiles = rows * nbc;
    for (int64_t tile0 = (int64_t)blockIdx.x * 16; tile0 < ntiles; tile0 += (int64_t)gridDim.x * 16) {
        const int64_t tile = tile0 + hw;
        const bool live = tile < ntiles;
        const int64_t r = live ? tile / nbc : 0, j = live ? tile % nbc : 0;
        const int64_t cbeg = j * 128, cend = cbeg + 128 < cols ? cbeg + 128 : cols;
        uint32_t am = 0;
        if (live)
            for (int64_t c = cbeg + l16; c < cend; c += 16) {
                const int64_t e = r * cols + c;
                uint32_t b = BF16 ? (uint32_t)(reinterpret_cast<const uint16_t*>(x)[e] & 0x7FFFu) << 16
                                  : (reinterpret_cast<const uint32_t*>(x)[e] & 0x7FFFFFFFu);
                am = umax(am, b);
            }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) am = umax(am, __shfl_xor_sync(0xFFFFFFFFu, am, o));
        float sc, si;
        scale_from_amax<FMT>(__uint_as_float(am), 0, &sc, &si);
        if (!live) continue;
        if (l16 == 0) scale_inv[tile] = si;
        for (int64_t c = cbeg + l16; c < cend; c += 16) {
            const int64_t e = r * cols + c;
            const float xv = BF16 ? __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(x)[e] << 16)
                                  : reinterpret_cast<const float*>(x)[e];
            uint32_t s;
            q[e] = (uint8_t)quant_one<FMT>(xv, sc, &s);
        }
    }
}

template <int FMT>
fp8_status_t launch_block(const uint8_t* x, bool bf16, int64_t rows, int64_t cols, int br, uint8_t* q, float* si,
                          cudaStream_t st) {
    const char* w = "fp8_quantize_block";
    const int64_t nbc = (cols + 127) / 128;
    if (br == 128) {
        const int64_t nbr = (rows + 127) / 128;
        const int vec_ok = aligned16(x) && aligned16(q) && cols % 16 == 0;
        const dim3 grid((unsigned)(nbc * nbr));
        if (bf16) return launch(w, block128_kernel<FMT, true>, grid, dim3(kThreads), st, x, rows, cols, q, si, nbc, vec_ok);
        return launch(w, block128_kernel<FMT, false>, grid, dim3(kThreads), st, x, rows, cols, q, si, nbc, vec_ok);
    }
    const int64_t cap = (int64_t)sm_count() * 8;
    if (bf16 && cols % 128 == 0 && aligned16(x) && aligned16(q)) {
        // one chunk of kTilesPerCta tiles per CTA (the loop in the kernel runs once)
        const int64_t ntiles = rows * nbc;
        constexpr int kTilesPerCta = (kThreads / 16) * kTilesInFlight;
        const int64_t grid = (ntiles + kTilesPerCta - 1) / kTilesPerCta;
        return launch(w, row128_bf16_kernel<FMT>, dim3((unsigned)grid), dim3(kThreads), st, x, ntiles, q, si);
    }
    int64_t grid = (rows * nbc + 15) / 16;
    if (grid > cap) grid = cap;
    if (bf16) return launch(w, row128_guarded_kernel<FMT, true>, dim3((unsigned)grid), dim3(kThreads), st, x, rows, cols, nbc, q, si);
    return launch(w, row128_guarded_kernel<FMT, false>, dim3((unsigned)grid), dim3(kThreads), st, x, rows, cols, nbc, q, si);
}

}  // namespace
}  // namespace fp8q

using namespace fp8q;

extern "C" fp8_status_t fp8_quantize_block(const void* x, fp8_dtype_t dtype, int64_t rows, int64_t cols, int block_rows,
                                           int block_cols, fp8_format_t fmt, uint8_t* q_out, float* scale_inv_out,
                                           void* stream) {
    const char* fn = "fp8_quantize_block";
    if (!valid_dtype(dtype)) return fail(FP8_ERR_INVALID_ARG, "%s: unknown dtype %d", fn, (int)dtype);
    if (!valid_fmt(fmt)) return fail(FP8_ERR_INVALID_ARG, "%s: unknown format %d", fn, (int)fmt);
    if (rows < 0 || cols < 0) return fail(FP8_ERR_INVALID_ARG, "%s: negative shape", fn);
    if (!((block_rows == 128 && block_cols == 128) || (block_rows == 1 && block_cols == 128)))
        return fail(FP8_ERR_UNSUPPORTED, "%s: block shape %dx%d (supported: 128x128, 1x128)", fn, block_rows, block_cols);
    if (rows == 0 || cols == 0) return FP8_OK;
    if (x == nullptr || q_out == nullptr || scale_inv_out == nullptr)
        return fail(FP8_ERR_INVALID_ARG, "%s: x / q_out / scale_inv_out is NULL", fn);
    if (reinterpret_cast<uintptr_t>(x) % dtype_size(dtype)) return fail(FP8_ERR_INVALID_ARG, "%s: x not element-aligned", fn);
    if (reinterpret_cast<uintptr_t>(scale_inv_out) % 4) return fail(FP8_ERR_INVALID_ARG, "%s: scale_inv_out not 4-byte aligned", fn);
    if (block_rows == 128 && ((rows + 127) / 128) * ((cols + 127) / 128) > 0x7FFFFFFFLL)
        return fail(FP8_ERR_UNSUPPORTED, "%s: too many blocks", fn);
    if (rows * ((cols + 127) / 128) / 16 > 0x7FFFFFFFLL) return fail(FP8_ERR_UNSUPPORTED, "%s: too many tiles", fn);

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint8_t* xp = static_cast<const uint8_t*>(x);
    const bool bf16 = dtype == FP8_DT_BF16;
    if (fmt == FP8_E4M3) return launch_block<kE4M3>(xp, bf16, rows, cols, block_rows, q_out, scale_inv_out, st);
    return launch_block<kE5M2>(xp, bf16, rows, cols, block_rows, q_out, scale_inv_out, st);
}
