// mx_quant.cu -- MXFP8: FP8 codes with one E8M0 (power-of-two) scale per 32
// consecutive elements, rowwise (1 x 32 blocks) and columnwise (32 x 1 blocks,
// written transposed), MX dequantize, and the lossless re-blocking of 128 x 128
// power-of-two block scales into 1 x 32 E8M0 scales.
//
// "Megatron FP8" §10 and §16: 32 consecutive elements share one E8M0 scale
// (8 exponent bits, no mantissa, no sign, 2^-127 .. 2^127, the OCP MX format);
// "Low Precision Training and Rollout", "MXFP8 (Blackwell only)": E4M3 values
// with UE8M0 scales per 32-element group, and [128,128] block-FP8 scales
// rescaled to [1,32] without dequantizing when they are powers of two.
//
// Scale rule (OCP MX, the reading the library takes): shared_exp =
// floor(log2(block amax)) - emax_elem (8 for E4M3, 15 for E5M2), clamped to
// [-127, 127]; an all-zero block takes -127; a block holding Inf or NaN gets
// the NaN scale 0xFF and NaN codes.  floor(log2(amax)) is the exponent field
// of the fp32 amax, so no division is needed; codes are
// cvt.rn.satfinite(fl32(x * 2^-shared_exp)).
#include <type_traits>

#include "fp8q_device.cuh"
#include "fp8q_host.h"

namespace fp8q {
namespace {

constexpr int kThreads = 256;
// 128 x 128 tile of up to four 32-row sub-tiles (the fast path needs rows % 32
// == 0): 4 row blocks per row and up to 4 column blocks per column.
constexpr int kTileR = 128, kTileC = 128, kSubR = 32;

template <int FMT> struct MxEmax;
template <> struct MxEmax<kE4M3> { static constexpr int kE = 8; };
template <> struct MxEmax<kE5M2> { static constexpr int kE = 15; };

// E8M0 code of a finite, non-negative amax (fp32 bits).
template <int FMT>
__device__ __forceinline__ uint32_t mx_scale_code(uint32_t amax_bits) {
    const int e = (int)(amax_bits >> 23);  // biased exponent; 0 for zero / subnormal amax
    int se = e - 127 - MxEmax<FMT>::kE;
    if (e == 0 || se < -127) se = -127;
    return (uint32_t)(se + 127);
}

// 2^-shared_exp from the code (exact; -shared_exp lies in [-119, 127]).
__device__ __forceinline__ float mx_multiplier(uint32_t code) { return exp2i(127 - (int)code); }

// One block's worth of 8 BF16 values -> 8 codes with the block's multiplier.
template <int FMT>
__device__ __forceinline__ uint2 mx_codes8(uint4 v, float m) {
    const Codes8 c = cvt_bf16x8_nomax<FMT>(v, m);
    return make_uint2(c.lo, c.hi);
}

// Fast path: rows % 32 == 0, cols % 128 == 0, BF16, 16-byte aligned pointers.
// Row pass: thread t takes 16 bytes (8 elements) of rows t / 16 + 16 p, p = 0..7
// (the sub-tiles inside the tensor); the 4 lanes of a 32-element row block
// reduce its amax by shuffles.  The BF16 tile is staged in shared memory as
// 16-byte chunks, chunk k of row r at position k ^ ((r / 16) % 8), so that the
// row stores (8 lanes x 16 bytes of one row) and the column reads (8 lanes on 8
// row groups, same chunk) both hit 32 distinct banks.  Column pass: a thread
// owns the column pair 2 cp, +1 and the 16 rows 16 g .. +15 (twice, cp and
// cp + 32); it reads one 32-bit word (two columns) per row, lanes g and g ^ 1
// hold the two halves of a 32-row column block and combine its amax with one
// shuffle, and each lane stores 16 codes per column: 8 lanes write a column's
// 128 contiguous bytes, as the cast-transpose does.
__device__ __forceinline__ int mx_chunk(int row, int chunk) { return chunk ^ ((row >> 4) & 7); }

template <int FMT>
__device__ __forceinline__ void mx_block_codes(uint32_t bits, uint4 lo, uint4 hi, uint4* codes, uint32_t* code) {
    if (bits >= 0x7F800000u) {
        *code = 0xFFu;
        *codes = make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
    } else {
        *code = mx_scale_code<FMT>(bits);
        const float m = mx_multiplier(*code);
        const uint2 a = mx_codes8<FMT>(lo, m), b = mx_codes8<FMT>(hi, m);
        *codes = make_uint4(a.x, a.y, b.x, b.y);
    }
}

// NARROW (rows, cols < 2^24): addresses are per-tile 64-bit bases plus 32-bit
// offsets inside the tile, which saves the 64-bit multiply-adds of every access.
// 48 registers: 5 CTAs (1280 threads) per SM, 160 KB of tiles in shared memory.
template <int FMT, bool NARROW>
__global__ void __launch_bounds__(kThreads, 5)
mx_tile_kernel(const uint8_t* __restrict__ x, int64_t rows, int64_t cols, uint8_t* __restrict__ q_row,
               uint8_t* __restrict__ s_row, uint8_t* __restrict__ q_col, uint8_t* __restrict__ s_col) {
    using Off = typename std::conditional<NARROW, uint32_t, int64_t>::type;
    pdl_begin();
    constexpr int kLoads = kTileR / 16;
    __shared__ __align__(16) uint4 tile[kTileR * kTileC / 8];  // 128 rows x 16 chunks of 8 BF16
    const int64_t gx = cols / kTileC;  // tile (blockIdx.x / gx, blockIdx.x % gx)
    const int64_t r0 = (int64_t)blockIdx.x / gx * kTileR, c0 = (int64_t)blockIdx.x % gx * kTileC;
    const int vrows = (int)min((int64_t)kTileR, rows - r0);  // a multiple of 32
    const int t = threadIdx.x, lane = t & 31;
    const int cc = t & 15, rsub = t >> 4;  // 16 threads per 256-byte row
    const Off ocols = (Off)cols, orows = (Off)rows;
    const Off nbr = (Off)(cols / 32), ncb = (Off)(rows / 32);
    const uint8_t* xt = x + (r0 * cols + c0) * 2;  // this tile's corner in each array
    uint8_t* qr = q_row ? q_row + r0 * cols + c0 : nullptr;
    uint8_t* sr = s_row ? s_row + r0 * (cols / 32) + (c0 >> 5) : nullptr;
    uint8_t* qc = q_col ? q_col + c0 * rows + r0 : nullptr;
    uint8_t* sc = s_col ? s_col + c0 * (rows / 32) + (r0 >> 5) : nullptr;
    uint4 v[kLoads];
#pragma unroll
    for (int p = 0; p < kLoads; ++p)
        if (p * 16 < vrows) v[p] = ldg_stream(xt + ((Off)(p * 16 + rsub) * ocols + (Off)(cc * 8)) * 2);
    // Row blocks: rows p = 2j and 2j + 1 share a word (low / high 16 bits of
    // their |x| bit patterns), so one u16x2 shuffle-max over the 4 lanes of a
    // 32-element block serves both rows.  vrows is a multiple of 32, so the
    // rows of a pair are both inside the tensor or both outside.
    // Stage the tile for the column pass first, so that the barrier does not
    // wait for the other warps' row passes.
    if (q_col) {
#pragma unroll
        for (int p = 0; p < kLoads; ++p) {
            if (p * 16 >= vrows) break;  // uniform over the CTA
            const int r = p * 16 + rsub;
            tile[r * 16 + mx_chunk(r, cc)] = v[p];
        }
        __syncthreads();
    }
    uint32_t rb2[kLoads / 2] = {};
    if (q_row) {
#pragma unroll
        for (int j = 0; j < kLoads / 2; ++j) {
            if (2 * j * 16 >= vrows) break;  // uniform over the CTA
            const uint4 a = v[2 * j], b = v[2 * j + 1];
            const uint32_t ma = max_u16x2(max_u16x2(abs_bf16x2(a.x), abs_bf16x2(a.y)),
                                          max_u16x2(abs_bf16x2(a.z), abs_bf16x2(a.w)));
            const uint32_t mb = max_u16x2(max_u16x2(abs_bf16x2(b.x), abs_bf16x2(b.y)),
                                          max_u16x2(abs_bf16x2(b.z), abs_bf16x2(b.w)));
            uint32_t w = max_u16x2(__byte_perm(ma, mb, 0x5410), __byte_perm(ma, mb, 0x7632));
            w = max_u16x2(w, __shfl_xor_sync(0xFFFFFFFFu, w, 1));
            w = max_u16x2(w, __shfl_xor_sync(0xFFFFFFFFu, w, 2));  // 4 lanes = one 32-element block
            rb2[j] = w;
        }
    }
#pragma unroll
    for (int p = 0; p < kLoads; ++p) {
        if (p * 16 >= vrows) break;  // uniform over the CTA
        const int r = p * 16 + rsub;
        if (q_row) {
            const uint32_t bits = (p & 1) ? (rb2[p >> 1] & 0xFFFF0000u) : (rb2[p >> 1] << 16);
            uint2 codes;
            uint32_t code;
            if (bits >= 0x7F800000u) {
                code = 0xFFu;
                codes = make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);
            } else {
                code = mx_scale_code<FMT>(bits);
                codes = mx_codes8<FMT>(v[p], mx_multiplier(code));
            }
            stg_stream(qr + ((Off)r * ocols + (Off)(cc * 8)), codes);
            if ((lane & 3) == 0) sr[(Off)r * nbr + (Off)(cc >> 2)] = (uint8_t)code;
        }
    }
    if (!q_col) return;
    const uint32_t* tw = reinterpret_cast<const uint32_t*>(tile);
    const int g = t & 7;  // rows 16 g .. 16 g + 15
    const bool live = g * 16 < vrows;  // lanes g and g ^ 1 agree (vrows % 32 == 0)
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int cp = (t >> 3) + 32 * u;  // columns 2 cp, 2 cp + 1
        // rows 16 g .. 16 g + 15 all have (row / 16) % 8 == g, so one chunk swizzle
        const uint32_t* wcol = tw + g * 16 * 64 + mx_chunk(g * 16, cp >> 2) * 4 + (cp & 3);
        uint32_t w[16];  // w[i]: row 16 g + i, columns 2 cp (low half) and 2 cp + 1 (high half)
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = wcol[i * 64];
        // Both columns' |x| maxima at once (u16x2), then the other half of the
        // 32-row block from lane g ^ 1.
        uint32_t m2 = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) m2 = max_u16x2(m2, abs_bf16x2(w[i]));
        m2 = max_u16x2(m2, __shfl_xor_sync(0xFFFFFFFFu, m2, 1));
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const uint32_t bits = j ? (m2 & 0xFFFF0000u) : (m2 << 16);  // column 2 cp + j
            uint4 codes;
            uint32_t code;
            if (bits >= 0x7F800000u) {
                code = 0xFFu;
                codes = make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
            } else {
                code = mx_scale_code<FMT>(bits);
                const float mul = mx_multiplier(code);
                uint32_t c4[4];  // codes of rows 4 i .. 4 i + 3
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 f = j ? fmul2_rn(bf16hi(w[4 * i]), bf16hi(w[4 * i + 1]), mul)
                                       : fmul2_rn(bf16lo(w[4 * i]), bf16lo(w[4 * i + 1]), mul);
                    const float2 g = j ? fmul2_rn(bf16hi(w[4 * i + 2]), bf16hi(w[4 * i + 3]), mul)
                                       : fmul2_rn(bf16lo(w[4 * i + 2]), bf16lo(w[4 * i + 3]), mul);
                    c4[i] = cvt4<FMT>(f.x, f.y, g.x, g.y);
                }
                codes = make_uint4(c4[0], c4[1], c4[2], c4[3]);
            }
            const Off c = (Off)(2 * cp + j);  // column inside the tile
            if (live) {
                stg_stream(qc + (c * orows + (Off)(g * 16)), codes);
                if ((g & 1) == 0) sc[c * ncb + (Off)(g >> 1)] = (uint8_t)code;
            }
        }
    }
}

// Guarded path for any shape / dtype / alignment: one thread per block.
template <int FMT, bool BF16>
__device__ __forceinline__ float mx_load(const uint8_t* x, int64_t e) {
    if constexpr (BF16) return __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(x)[e] << 16);
    else return reinterpret_cast<const float*>(x)[e];
}

// Blocks of 32 consecutive elements along a line; `stride` is the distance
// between the block's consecutive elements in x, `nlines` lines of `len`
// elements.  Output codes go to q[line * len + i], scales to s[line * nb + b].
template <int FMT, bool BF16>
__global__ void __launch_bounds__(kThreads)
mx_guarded_kernel(const uint8_t* __restrict__ x, int64_t nlines, int64_t len, int64_t line_stride,
                  int64_t elem_stride, uint8_t* __restrict__ q, uint8_t* __restrict__ s) {
    pdl_begin();
    const int64_t nb = (len + 31) / 32;
    for (int64_t task = (int64_t)blockIdx.x * kThreads + threadIdx.x; task < nlines * nb;
         task += (int64_t)gridDim.x * kThreads) {
        const int64_t line = task / nb, b = task % nb;
        const int64_t i0 = b * 32, i1 = i0 + 32 < len ? i0 + 32 : len;
        uint32_t bits = 0;
        for (int64_t i = i0; i < i1; ++i)
            bits = umax(bits, __float_as_uint(mx_load<FMT, BF16>(x, line * line_stride + i * elem_stride)) & 0x7FFFFFFFu);
        uint32_t code = bits >= 0x7F800000u ? 0xFFu : mx_scale_code<FMT>(bits);
        const float mul = mx_multiplier(code);
        for (int64_t i = i0; i < i1; ++i) {
            uint32_t c = kNaNCode;
            if (code != 0xFFu) {
                uint32_t sat;
                c = quant_one<FMT>(mx_load<FMT, BF16>(x, line * line_stride + i * elem_stride), mul, &sat);
            }
            q[line * len + i] = (uint8_t)c;
        }
        s[line * nb + b] = (uint8_t)code;
    }
}

// MX dequantize (rowwise layout [rows, cols], scales [rows, ceil(cols / 32)]).
template <int FMT, bool OUT_BF16>
__global__ void __launch_bounds__(kThreads)
mx_dequant_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ s, int64_t rows, int64_t cols,
                  uint8_t* __restrict__ y) {
    pdl_begin();
    const int64_t nb = (cols + 31) / 32;
    const int64_t n = rows * cols;
    for (int64_t e = (int64_t)blockIdx.x * kThreads + threadIdx.x; e < n; e += (int64_t)gridDim.x * kThreads) {
        const int64_t r = e / cols, c = e % cols;
        const uint32_t code = s[r * nb + c / 32];
        const uint32_t h2 = fp8x2_to_f16x2<FMT>(q[e]);
        // 2^(code - 127): code 0 is the fp32 subnormal 2^-127; a NaN scale (0xFF) makes the block NaN
        const float m = code == 0xFFu ? __uint_as_float(0x7FFFFFFFu)
                                      : (code == 0u ? __uint_as_float(0x00400000u) : exp2i((int)code - 127));
        const float out = __fmul_rn(f16_lo_to_f32(h2), m);
        if constexpr (OUT_BF16) reinterpret_cast<uint16_t*>(y)[e] = (uint16_t)(f32x2_to_bf16x2(out, 0.0f) & 0xFFFFu);
        else reinterpret_cast<float*>(y)[e] = isnan(out) ? __uint_as_float(0x7FFFFFFFu) : out;
    }
}

// Fast MX dequantize: cols % 32 == 0 and 16-byte aligned q / y, so the block of
// flat element e is e / 32.  Each item is the codes of one 16-byte output
// piece (8 codes for BF16, 4 for fp32; always inside one 32-element block), so
// every warp store covers 512 contiguous bytes; 16 items in flight per thread,
// each item's E8M0 byte loaded together with its codes.
template <int FMT, bool OUT_BF16>
__global__ void __launch_bounds__(kThreads, 4)
mx_dequant_vec_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ s, int64_t n,
                      uint8_t* __restrict__ y) {
    pdl_begin();
    constexpr int kI = 16, kCodes = OUT_BF16 ? 8 : 4, kPerBlock = 32 / kCodes;
    const int64_t nitems = n / kCodes;
    const int64_t ib = (int64_t)blockIdx.x * kThreads * kI + threadIdx.x;
    uint32_t c[kI][kCodes / 4];
    uint32_t code[kI];
#pragma unroll
    for (int k = 0; k < kI; ++k) {
        const int64_t i = ib + (int64_t)k * kThreads;
        if (i < nitems) {
            if constexpr (OUT_BF16) {
                const uint2 v = __ldcs(reinterpret_cast<const uint2*>(q) + i);
                c[k][0] = v.x;
                c[k][kCodes / 4 - 1] = v.y;
            } else {
                c[k][0] = __ldcs(reinterpret_cast<const unsigned int*>(q) + i);
            }
            code[k] = s[i / kPerBlock];
        }
    }
#pragma unroll
    for (int k = 0; k < kI; ++k) {
        const int64_t i = ib + (int64_t)k * kThreads;
        if (i >= nitems) continue;
        const float m = code[k] == 0xFFu ? __uint_as_float(0x7FFFFFFFu)
                                         : (code[k] == 0u ? __uint_as_float(0x00400000u) : exp2i((int)code[k] - 127));
        float f[kCodes];
#pragma unroll
        for (int w = 0; w < kCodes / 4; ++w) {
            const uint32_t h01 = fp8x2_to_f16x2<FMT>(c[k][w] & 0xFFFFu), h23 = fp8x2_to_f16x2<FMT>(c[k][w] >> 16);
            f[4 * w + 0] = __fmul_rn(f16_lo_to_f32(h01), m);
            f[4 * w + 1] = __fmul_rn(f16_hi_to_f32(h01), m);
            f[4 * w + 2] = __fmul_rn(f16_lo_to_f32(h23), m);
            f[4 * w + 3] = __fmul_rn(f16_hi_to_f32(h23), m);
        }
        if constexpr (OUT_BF16) {
            stg_evict_first(y + i * 16, make_uint4(f32x2_to_bf16x2(f[0], f[1]), f32x2_to_bf16x2(f[2], f[3]),
                                              f32x2_to_bf16x2(f[4], f[5]), f32x2_to_bf16x2(f[6], f[7])));
        } else {
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) o[j] = isnan(f[j]) ? 0x7FFFFFFFu : __float_as_uint(f[j]);
            stg_evict_first(y + i * 16, make_uint4(o[0], o[1], o[2], o[3]));
        }
    }
}

// 128 x 128 scale_inv -> 1 x 32 E8M0 codes; counts blocks whose scale_inv is
// not a power of two in [2^-127, 2^127] (they get 0xFF).
__global__ void __launch_bounds__(kThreads)
block128_to_mx_kernel(const float* __restrict__ si, int64_t rows, int64_t cols, uint8_t* __restrict__ out,
                      unsigned long long* bad) {
    pdl_begin();
    const int64_t nb32 = (cols + 31) / 32, nbc128 = (cols + 127) / 128;
    const int64_t n = rows * nb32;
    for (int64_t k = (int64_t)blockIdx.x * kThreads + threadIdx.x; k < n; k += (int64_t)gridDim.x * kThreads) {
        const int64_t r = k / nb32, b = k % nb32;
        const uint32_t u = __float_as_uint(si[(r >> 7) * nbc128 + ((b * 32) >> 7)]);
        uint32_t code = 0xFFu;
        const uint32_t e = u >> 23, mant = u & 0x7FFFFFu;
        if (!(u & 0x80000000u) && e >= 1 && e <= 254 && mant == 0) code = e;          // 2^(e-127), e in [1, 254]
        else if (u == 0x00400000u) code = 0;                                           // 2^-127 (subnormal)
        out[k] = (uint8_t)code;
        // count each 128 x 128 block once: at its first row and first 1 x 32 block
        if (code == 0xFFu && bad && (r & 127) == 0 && ((b * 32) & 127) == 0) atomicAdd(bad, 1ull);
    }
}

template <int FMT>
fp8_status_t launch_mx(const uint8_t* x, bool bf16, int64_t rows, int64_t cols, uint8_t* q_row, uint8_t* s_row,
                       uint8_t* q_col, uint8_t* s_col, cudaStream_t st) {
    const char* w = "fp8_quantize_mx";
    const bool fast = bf16 && rows % kSubR == 0 && cols % kTileC == 0 && aligned16(x) &&
                      (!q_row || aligned16(q_row)) && (!q_col || aligned16(q_col)) &&
                      ((rows + kTileR - 1) / kTileR) * (cols / kTileC) <= 0x7FFFFFFF;
    if (fast) {
        const dim3 grid((unsigned)(((rows + kTileR - 1) / kTileR) * (cols / kTileC)));
        if (rows < (1 << 24) && cols < (1 << 24))
            return launch(w, mx_tile_kernel<FMT, true>, grid, dim3(kThreads), st, x, rows, cols, q_row, s_row, q_col,
                          s_col);
        return launch(w, mx_tile_kernel<FMT, false>, grid, dim3(kThreads), st, x, rows, cols, q_row, s_row, q_col,
                      s_col);
    }
    const int64_t cap = (int64_t)sm_count() * 8;
    if (q_row) {
        int64_t g = (rows * ((cols + 31) / 32) + kThreads - 1) / kThreads;
        g = g < 1 ? 1 : (g > cap ? cap : g);
        const int64_t one = 1;
        fp8_status_t s = bf16 ? launch(w, mx_guarded_kernel<FMT, true>, dim3((unsigned)g), dim3(kThreads), st, x, rows,
                                       cols, cols, one, q_row, s_row)
                              : launch(w, mx_guarded_kernel<FMT, false>, dim3((unsigned)g), dim3(kThreads), st, x, rows,
                                       cols, cols, one, q_row, s_row);
        if (s != FP8_OK) return s;
    }
    if (q_col) {
        int64_t g = (cols * ((rows + 31) / 32) + kThreads - 1) / kThreads;
        g = g < 1 ? 1 : (g > cap ? cap : g);
        const int64_t one = 1;
        return bf16 ? launch(w, mx_guarded_kernel<FMT, true>, dim3((unsigned)g), dim3(kThreads), st, x, cols, rows, one,
                             cols, q_col, s_col)
                    : launch(w, mx_guarded_kernel<FMT, false>, dim3((unsigned)g), dim3(kThreads), st, x, cols, rows,
                             one, cols, q_col, s_col);
    }
    return FP8_OK;
}

}  // namespace
}  // namespace fp8q

using namespace fp8q;

extern "C" fp8_status_t fp8_quantize_mx(const void* x, fp8_dtype_t dtype, int64_t rows, int64_t cols,
                                        fp8_format_t fmt, uint8_t* q_row, uint8_t* scale_row, uint8_t* q_col,
                                        uint8_t* scale_col, void* stream) {
    const char* fn = "fp8_quantize_mx";
    if (!valid_dtype(dtype)) return fail(FP8_ERR_INVALID_ARG, "%s: unknown dtype %d", fn, (int)dtype);
    if (!valid_fmt(fmt)) return fail(FP8_ERR_INVALID_ARG, "%s: unknown format %d", fn, (int)fmt);
    if (rows < 0 || cols < 0) return fail(FP8_ERR_INVALID_ARG, "%s: negative shape", fn);
    if ((q_row == nullptr) != (scale_row == nullptr) || (q_col == nullptr) != (scale_col == nullptr))
        return fail(FP8_ERR_INVALID_ARG, "%s: each direction needs both its codes and its scales", fn);
    if (rows == 0 || cols == 0) return FP8_OK;
    if (x == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: x is NULL", fn);
    if (q_row == nullptr && q_col == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: no output requested", fn);
    if (reinterpret_cast<uintptr_t>(x) % dtype_size(dtype)) return fail(FP8_ERR_INVALID_ARG, "%s: x not element-aligned", fn);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint8_t* xp = static_cast<const uint8_t*>(x);
    const bool bf16 = dtype == FP8_DT_BF16;
    if (fmt == FP8_E4M3) return launch_mx<kE4M3>(xp, bf16, rows, cols, q_row, scale_row, q_col, scale_col, st);
    return launch_mx<kE5M2>(xp, bf16, rows, cols, q_row, scale_row, q_col, scale_col, st);
}

extern "C" fp8_status_t fp8_dequantize_mx(const uint8_t* q, const uint8_t* scales, fp8_format_t fmt, int64_t rows,
                                          int64_t cols, void* y, fp8_dtype_t out_dtype, void* stream) {
    const char* fn = "fp8_dequantize_mx";
    if (!valid_fmt(fmt)) return fail(FP8_ERR_INVALID_ARG, "%s: unknown format %d", fn, (int)fmt);
    if (!valid_dtype(out_dtype)) return fail(FP8_ERR_INVALID_ARG, "%s: unknown out_dtype %d", fn, (int)out_dtype);
    if (rows < 0 || cols < 0) return fail(FP8_ERR_INVALID_ARG, "%s: negative shape", fn);
    if (rows == 0 || cols == 0) return FP8_OK;
    if (q == nullptr || scales == nullptr || y == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: NULL pointer", fn);
    if (reinterpret_cast<uintptr_t>(y) % dtype_size(out_dtype)) return fail(FP8_ERR_INVALID_ARG, "%s: y not element-aligned", fn);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int64_t g = (rows * cols + kThreads - 1) / kThreads;
    const int64_t cap = (int64_t)sm_count() * 8;
    g = g > cap ? cap : g;
    uint8_t* yp = static_cast<uint8_t*>(y);
    const bool bf16 = out_dtype == FP8_DT_BF16;
    if (cols % 32 == 0 && aligned16(q) && aligned16(y)) {
        const int64_t n = rows * cols;
        const int64_t nitems = n / (bf16 ? 8 : 4);
        const dim3 vg((unsigned)((nitems + kThreads * 16 - 1) / (kThreads * 16))), vb(kThreads);
        if (fmt == FP8_E4M3)
            return bf16 ? launch(fn, mx_dequant_vec_kernel<kE4M3, true>, vg, vb, st, q, scales, n, yp)
                        : launch(fn, mx_dequant_vec_kernel<kE4M3, false>, vg, vb, st, q, scales, n, yp);
        return bf16 ? launch(fn, mx_dequant_vec_kernel<kE5M2, true>, vg, vb, st, q, scales, n, yp)
                    : launch(fn, mx_dequant_vec_kernel<kE5M2, false>, vg, vb, st, q, scales, n, yp);
    }
    const dim3 grid((unsigned)g), block(kThreads);
    if (fmt == FP8_E4M3)
        return bf16 ? launch(fn, mx_dequant_kernel<kE4M3, true>, grid, block, st, q, scales, rows, cols, yp)
                    : launch(fn, mx_dequant_kernel<kE4M3, false>, grid, block, st, q, scales, rows, cols, yp);
    return bf16 ? launch(fn, mx_dequant_kernel<kE5M2, true>, grid, block, st, q, scales, rows, cols, yp)
                : launch(fn, mx_dequant_kernel<kE5M2, false>, grid, block, st, q, scales, rows, cols, yp);
}

extern "C" fp8_status_t fp8_block128_scales_to_mx(const float* scale_inv, int64_t rows, int64_t cols,
                                                  uint8_t* mx_scales, unsigned long long* bad_blocks_out,
                                                  void* stream) {
    const char* fn = "fp8_block128_scales_to_mx";
    if (rows < 0 || cols < 0) return fail(FP8_ERR_INVALID_ARG, "%s: negative shape", fn);
    const bool empty = rows == 0 || cols == 0;
    if (!empty && (scale_inv == nullptr || mx_scales == nullptr)) return fail(FP8_ERR_INVALID_ARG, "%s: NULL pointer", fn);
    if (!empty && reinterpret_cast<uintptr_t>(scale_inv) % 4)
        return fail(FP8_ERR_INVALID_ARG, "%s: scale_inv not 4-byte aligned", fn);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (bad_blocks_out) {  // overwritten, also for an empty shape
        cudaError_t e = cudaMemsetAsync(bad_blocks_out, 0, sizeof(unsigned long long), st);
        if (e != cudaSuccess) return cuda_status(e, "fp8_block128_scales_to_mx: cudaMemsetAsync");
    }
    if (empty) return FP8_OK;
    int64_t g = (rows * ((cols + 31) / 32) + kThreads - 1) / kThreads;
    const int64_t cap = (int64_t)sm_count() * 8;
    g = g < 1 ? 1 : (g > cap ? cap : g);
    return launch(fn, block128_to_mx_kernel, dim3((unsigned)g), dim3(kThreads), st, scale_inv, rows, cols, mx_scales,
                  bad_blocks_out);
}
