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
// Fast path (BF16, rows % 128 == 0, cols % 128 == 0, 16-byte aligned): a
// persistent kernel, one CTA per SM.  One thread streams 128 x 128 tiles of x
// into a ring of shared-memory stages with 2-D tensor-map bulk copies (TMA,
// one 32 KB copy per tile), each stage guarded by mbarriers; two groups of 256
// threads take the tiles in turn, so that reads stay in flight while the
// groups reduce and convert.  Each thread of a group holds 8 rows x 8 columns:
//   rows:    the 16 lanes sharing a row reduce its 1 x 128 amax by shuffles,
//            two rows per 32-bit word (u16x2); 8 lanes each derive one row's
//            scale and shuffle it.
//   columns: each thread folds its 8 rows per column pair (u16x2), a shuffle
//            adds the other half-warp's 8, an 8 x 64 shared table the other
//            warps'; four threads per column pair finish it and two derive the
//            pair's scales.
//   codes:   each BF16 pair is unpacked once for both directions; two-lane
//            multiplies and two-value cvts give the rowwise codes (stored
//            directly, one 128-byte line per half-warp) and the columnwise
//            codes, which go through a swizzled byte-transpose tile (16-byte
//            stores, full lines).
//   Scales come from block_scale_bf16 (exact tables, no division); a tile
//   holding Inf / NaN takes the element-exact path.
#include "fp8q_device.cuh"
#include "fp8q_host.h"
#include "fp8q_pipeline.cuh"

namespace fp8q {
namespace {

constexpr int kTile = 128;
constexpr int kThreads = 256;
// The pipelined kernel: consumer groups of 256 threads and ring stages (a
// multiple of the groups); 2 x 4 measured fastest among 1 x 6, 2 x 4 and 3 x 3.
constexpr int kGroups = 2, kStages = 4;

// a * sa and b * sb in one packed two-lane multiply (round to nearest even).
__device__ __forceinline__ float2 fmul2_rn_pair(float a, float b, float sa, float sb) {
    unsigned long long r;
    asm("{\n\t.reg .b64 x, y;\n\t"
        "mov.b64 x, {%1, %2};\n\t"
        "mov.b64 y, {%3, %4};\n\t"
        "mul.rn.f32x2 %0, x, y;\n\t}"
        : "=l"(r)
        : "r"(__float_as_uint(a)), "r"(__float_as_uint(b)), "r"(__float_as_uint(sa)), "r"(__float_as_uint(sb)));
    return make_float2(__uint_as_float((uint32_t)r), __uint_as_float((uint32_t)(r >> 32)));
}

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

// Eight codes of one row of x, column j with scale c[j], every special case
// spelled out: the path of a tile holding Inf / NaN (out of line, so that it
// costs the common path no registers).
template <int FMT>
__device__ __noinline__ uint2 codes8_exact(uint4 v, float4 c_lo, float4 c_hi) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    const float c[8] = {c_lo.x, c_lo.y, c_lo.z, c_lo.w, c_hi.x, c_hi.y, c_hi.z, c_hi.w};
    uint2 r = make_uint2(0u, 0u);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t sat;
        const uint32_t code = quant_one<FMT>((j & 1) ? bf16hi(w[j >> 1]) : bf16lo(w[j >> 1]), c[j], &sat);
        if (j < 4) r.x |= code << (8 * j);
        else r.y |= code << (8 * (j - 4));
    }
    return r;
}

// Shared memory of one 256-thread group working on a tile.
struct TileSmem {
    uint32_t tile[kTile * kTile / 4];  // columnwise codes, swizzled
    uint32_t colmax2[8][68];           // per warp (16 rows): column-pair maxima (u16x2); padded rows
    float colscale[kTile];
};

// Rowwise codes of row p of the thread (8 values) with scale `scale`; the
// element-exact fixup when the row holds Inf / NaN.
template <int FMT>
__device__ __forceinline__ uint2 row_codes(uint4 v, float scale, uint32_t rmax) {
    Codes8 c = cvt_bf16x8_nomax<FMT>(v, scale);
    if (rmax >= 0x7F800000u) fixup_bf16x8<FMT>(v, scale, &c);
    return make_uint2(c.lo, c.hi);
}

// Both directions of one 128 x 128 tile whose values are in v (thread tg of
// the group: v[p] = row p * 16 + tg / 16, columns (tg % 16) * 8 .. + 7).  The
// group's 256 threads synchronise on hardware barrier `bar`.  ROWS / COLS: the
// rowwise / columnwise outputs are requested (a one-direction form skips the
// other direction's reductions and products).
template <int FMT, bool ROWS, bool COLS>
__device__ __forceinline__ void bct_tile(const uint4 (&v)[8], const uint32_t* tab, TileSmem& ts, int bar, int tg,
                                         int64_t r0, int64_t c0, int64_t rows, int64_t cols, uint8_t* q_row,
                                         float* si_row, uint8_t* q_col, float* si_col) {
    const int lane = tg & 31, warp = tg >> 5, cc = tg & 15, rsub = tg >> 4;
    const int64_t nbr_row = cols / kTile, nbr_col = rows / kTile;

    // ---- rowwise 1 x 128 tiles: the half-warp of 16 lanes holds one row per p.
    // Rows p = 2j and 2j + 1 share a word (low / high 16 bits of their |x| bit
    // patterns), so one u16x2 shuffle-max reduction serves two rows.
    uint32_t rm2[4] = {0u, 0u, 0u, 0u};
    float rs = 1.0f, rsi = 1.0f;  // lane cc < 8: the scale of row p = cc
    if (ROWS) {
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
        // rm2[cc / 2] as a tree of selects: written as a loop of compares the
        // compiler turns it into an indexed read of rm2 kept in local memory.
        const uint32_t m01 = (cc & 2) ? rm2[1] : rm2[0], m23 = (cc & 2) ? rm2[3] : rm2[2];
        const uint32_t mine2 = (cc & 4) ? m23 : m01;
        block_scale_bf16<FMT>(tab, (cc & 1) ? (mine2 & 0xFFFF0000u) : (mine2 << 16), &rs, &rsi);
        if (cc < 8) si_row[(r0 + cc * 16 + rsub) * nbr_row + (c0 >> 7)] = rsi;
    }

    if (!COLS) {  // rowwise codes only
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            const float scale = __shfl_sync(0xFFFFFFFFu, rs, (lane & 16) | p);
            const uint32_t rmax = (p & 1) ? (rm2[p >> 1] & 0xFFFF0000u) : (rm2[p >> 1] << 16);
            stg_stream(q_row + (r0 + p * 16 + rsub) * cols + c0 + cc * 8, row_codes<FMT>(v[p], scale, rmax));
        }
        return;
    }

    // ---- column maxima: over the thread's 8 rows, the warp's 16 (a shuffle
    // with the other half-warp), then the 8 warps through shared memory.
    {
        uint4 cm = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            cm.x = max_u16x2(cm.x, abs_bf16x2(v[p].x));
            cm.y = max_u16x2(cm.y, abs_bf16x2(v[p].y));
            cm.z = max_u16x2(cm.z, abs_bf16x2(v[p].z));
            cm.w = max_u16x2(cm.w, abs_bf16x2(v[p].w));
        }
        cm.x = max_u16x2(cm.x, __shfl_xor_sync(0xFFFFFFFFu, cm.x, 16));
        cm.y = max_u16x2(cm.y, __shfl_xor_sync(0xFFFFFFFFu, cm.y, 16));
        cm.z = max_u16x2(cm.z, __shfl_xor_sync(0xFFFFFFFFu, cm.z, 16));
        cm.w = max_u16x2(cm.w, __shfl_xor_sync(0xFFFFFFFFu, cm.w, 16));
        if (lane < 16) *reinterpret_cast<uint4*>(&ts.colmax2[warp][cc * 4]) = cm;
    }
    group_sync(bar, 256);

    // ---- column scales: four threads per column pair cp, each folding two of
    // the eight warp maxima; threads qq = 0 / 1 derive the scale of column
    // 2 cp / 2 cp + 1.  `special`: some column of the tile holds Inf / NaN.
    {
        const int cp = tg >> 2, qq = tg & 3;
        uint32_t m2 = max_u16x2(ts.colmax2[2 * qq][cp], ts.colmax2[2 * qq + 1][cp]);
        m2 = max_u16x2(m2, __shfl_xor_sync(0xFFFFFFFFu, m2, 1));
        m2 = max_u16x2(m2, __shfl_xor_sync(0xFFFFFFFFu, m2, 2));
        if (qq < 2) {
            float sc, sci;
            block_scale_bf16<FMT>(tab, qq ? (m2 & 0xFFFF0000u) : (m2 << 16), &sc, &sci);
            ts.colscale[2 * cp + qq] = sc;
            si_col[(c0 + 2 * cp + qq) * nbr_col + (r0 >> 7)] = sci;
        }
        if (group_sync_or(bar, 256, (m2 & 0xFFFFu) >= 0x7F80u || m2 >= 0x7F800000u)) {
            // ---- a tile with Inf / NaN in some column: every element exactly
            float cs[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) cs[j] = ts.colscale[cc * 8 + j];
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                const float scale = __shfl_sync(0xFFFFFFFFu, rs, (lane & 16) | p);
                const uint32_t rmax = (p & 1) ? (rm2[p >> 1] & 0xFFFF0000u) : (rm2[p >> 1] << 16);
                if (ROWS)
                    stg_stream(q_row + (r0 + p * 16 + rsub) * cols + c0 + cc * 8, row_codes<FMT>(v[p], scale, rmax));
                const uint2 c = codes8_exact<FMT>(v[p], make_float4(cs[0], cs[1], cs[2], cs[3]),
                                                  make_float4(cs[4], cs[5], cs[6], cs[7]));
                const int r = p * 16 + rsub;
                *reinterpret_cast<uint2*>(&ts.tile[r * 32 + ((cc * 2) ^ (p << 2))]) = c;
            }
            goto transpose;
        }
    }

    // ---- both code sets from one unpacking of each BF16 pair.  For rows p and
    // p + 1 and columns (2h, 2h + 1) of the thread: the rowwise products take
    // the row's scale, the columnwise ones the columns' pair of scales; with
    // no Inf / NaN in a column, |x * scale| <= its amax * scale, so the
    // round-to-nearest-even saturating cvt is the exact per-element rule.  The
    // columnwise bytes of the two rows are interleaved per column and go
    // through the swizzled byte-transpose tile (16-byte stores, full lines).
    {
        const float4 csl = *reinterpret_cast<const float4*>(&ts.colscale[cc * 8]);
        const float4 csh = *reinterpret_cast<const float4*>(&ts.colscale[cc * 8 + 4]);
        const float cs[8] = {csl.x, csl.y, csl.z, csl.w, csh.x, csh.y, csh.z, csh.w};
#pragma unroll
        for (int p = 0; p < 8; p += 2) {
            const float sa = __shfl_sync(0xFFFFFFFFu, rs, (lane & 16) | p);
            const float sb = __shfl_sync(0xFFFFFFFFu, rs, (lane & 16) | (p + 1));
            const uint32_t a[4] = {v[p].x, v[p].y, v[p].z, v[p].w};
            const uint32_t b[4] = {v[p + 1].x, v[p + 1].y, v[p + 1].z, v[p + 1].w};
            uint32_t ra[4], rb[4], pr[4];  // ra / rb: row p / p + 1, columns 2h, 2h + 1 (16 bits)
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const float alo = bf16lo(a[h]), ahi = bf16hi(a[h]), blo = bf16lo(b[h]), bhi = bf16hi(b[h]);
                if (ROWS) {
                    const float2 xa = fmul2_rn(alo, ahi, sa), xb = fmul2_rn(blo, bhi, sb);
                    ra[h] = cvt2<FMT>(xa.x, xa.y);
                    rb[h] = cvt2<FMT>(xb.x, xb.y);
                }
                const float2 ya = fmul2_rn_pair(alo, ahi, cs[2 * h], cs[2 * h + 1]);
                const float2 yb = fmul2_rn_pair(blo, bhi, cs[2 * h], cs[2 * h + 1]);
                // bytes (row p, col 2h), (row p+1, col 2h), (row p, col 2h+1), (row p+1, col 2h+1)
                pr[h] = __byte_perm(cvt2<FMT>(ya.x, ya.y), cvt2<FMT>(yb.x, yb.y), 0x5140);
            }
            if (ROWS) {
                uint2 ca = make_uint2(__byte_perm(ra[0], ra[1], 0x5410), __byte_perm(ra[2], ra[3], 0x5410));
                uint2 cb = make_uint2(__byte_perm(rb[0], rb[1], 0x5410), __byte_perm(rb[2], rb[3], 0x5410));
                const uint32_t rmaxa = rm2[p >> 1] << 16, rmaxb = rm2[p >> 1] & 0xFFFF0000u;
                if (rmaxa >= 0x7F800000u) ca = row_codes<FMT>(v[p], sa, rmaxa);
                if (rmaxb >= 0x7F800000u) cb = row_codes<FMT>(v[p + 1], sb, rmaxb);
                stg_stream(q_row + (r0 + p * 16 + rsub) * cols + c0 + cc * 8, ca);
                stg_stream(q_row + (r0 + (p + 1) * 16 + rsub) * cols + c0 + cc * 8, cb);
            }
            const uint32_t lo0 = __byte_perm(pr[0], pr[1], 0x6420), lo1 = __byte_perm(pr[0], pr[1], 0x7531);
            const uint32_t hi0 = __byte_perm(pr[2], pr[3], 0x6420), hi1 = __byte_perm(pr[2], pr[3], 0x7531);
            const int r = p * 16 + rsub;
            *reinterpret_cast<uint2*>(&ts.tile[r * 32 + ((cc * 2) ^ (p << 2))]) = make_uint2(lo0, hi0);
            *reinterpret_cast<uint2*>(&ts.tile[(r + 16) * 32 + ((cc * 2) ^ ((p + 1) << 2))]) = make_uint2(lo1, hi1);
        }
    }

transpose:
    group_sync(bar, 256);
    {
        const int cg = warp * 4 + (lane >> 3);
        const int rc = lane & 7;
        uint32_t out[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int rb = rc * 16 + i * 4;
            const int sw = rc << 2;
            transpose4x4_b(ts.tile[(rb + 0) * 32 + (cg ^ sw)], ts.tile[(rb + 1) * 32 + (cg ^ sw)],
                           ts.tile[(rb + 2) * 32 + (cg ^ sw)], ts.tile[(rb + 3) * 32 + (cg ^ sw)], out[0][i],
                           out[1][i], out[2][i], out[3][i]);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
            stg_stream(q_col + (c0 + cg * 4 + j) * rows + r0 + rc * 16,
                       make_uint4(out[j][0], out[j][1], out[j][2], out[j][3]));
    }
}

// Test hook (fp8_test_drop_tile_copy): the copying thread of every CTA skips
// the copy of its tile number g_drop_tile, so that the waits on that stage
// expire; -1 (the default) skips none.
__device__ int g_drop_tile = -1;

// Shared memory of the pipelined kernel: S stages of one 128 x 128 BF16 tile
// (32 KB, rows of 256 bytes), NG group areas, the scale tables, the barriers.
template <int NG, int S>
struct BctLayout {
    static constexpr int kStage = kTile * kTile * 2;
    static constexpr int kGroups = S * kStage;
    static constexpr int kTab = kGroups + NG * (int)sizeof(TileSmem);
    static constexpr int kBars = kTab + 256 * 4;
    static constexpr int kBytes = kBars + 2 * S * 8;
};

// Persistent, one CTA per SM: lane 0 of warp NG * 8 copies tile i =
// blockIdx.x + k * gridDim.x (k = 0, 1, ...) into stage k % S with one tensor
// copy; the NG groups of 256 threads take the tiles in turn (group k % NG),
// read their values from the stage into registers, release it and finish the
// tile.  A wait that times out is counted and skips the rest of that thread's
// waits (the group keeps its barrier pattern, its later tiles are garbage, and
// a warp whose first lane timed out releases no more stages, so that no copy
// is ever issued into a stage with one still in flight); every thread ends.
// Registers: 17 warps per SM leave at most 96 per thread.
template <int FMT, int NG, int S, bool ROWS, bool COLS>
__global__ void __maxnreg__(ROWS ? 88 : 96)
block_ct_pipe_kernel(const __grid_constant__ CUtensorMap xmap, int64_t rows, int64_t cols, uint8_t* __restrict__ q_row,
                     float* __restrict__ si_row, uint8_t* __restrict__ q_col, float* __restrict__ si_col) {
    // Stage k % S is consumed by group k % NG; with S a multiple of NG every
    // stage belongs to one group, which has finished tile k - S (phase k / S - 1
    // of the stage's `full` barrier) before it waits for tile k (phase k / S).
    // Otherwise a group could wait for parity (k / S) & 1 while another group's
    // tile k - S is still in flight, a parity that try_wait reports as complete.
    static_assert(S % NG == 0, "each ring stage must belong to one consumer group");
    using L = BctLayout<NG, S>;
    extern __shared__ __align__(128) uint8_t smem[];
    uint32_t* tab = reinterpret_cast<uint32_t*>(smem + L::kTab);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBars);
    uint64_t* empty = full + S;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    if (t < 256) tab[t] = table_word<FMT>(t);
    if (t == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 8);  // one arrival per warp of the consuming group
        }
        mbar_init_fence();
    }
    __syncthreads();
    pdl_begin();
    // tile counts fit 31 bits (checked by the launcher)
    const uint32_t nbr_row = (uint32_t)(cols / kTile), ntiles = nbr_row * (uint32_t)(rows / kTile);
    const uint32_t n_my = ntiles > blockIdx.x ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;

    if (warp == NG * 8) {  // producer: one thread issues the tile copies
        if (lane != 0) return;
        const int drop = g_drop_tile;
        uint32_t k = 0;
        for (; k < n_my; ++k) {
            const uint32_t s = k % S;
            if (k >= S && !mbar_wait(&empty[s], ((k / S) & 1u) ^ 1u)) {
                atomicAdd(&g_wait_timeouts, 1ull);
                break;
            }
            if ((int)k == drop) continue;
            const uint32_t tile = blockIdx.x + k * gridDim.x;
            mbar_arrive_expect_tx(&full[s], L::kStage);
            tma_load_2d(smem + s * L::kStage, &xmap, (int)(tile % nbr_row) * kTile, (int)(tile / nbr_row) * kTile,
                        &full[s]);
        }
        // the CTA's shared memory must outlive every copy issued into it
        for (uint32_t j = k > S ? k - S : 0; j < k; ++j)
            if (!mbar_wait(&full[j % S], (j / S) & 1u)) atomicAdd(&g_wait_timeouts, 1ull);
        return;
    }

    const int g = warp >> 3, tg = t & 255, rsub = tg >> 4, cc = tg & 15;
    TileSmem& ts = reinterpret_cast<TileSmem*>(smem + L::kGroups)[g];
    bool live = true;
    for (uint32_t k = g; k < n_my; k += NG) {
        const uint32_t s = k % S;
        if (live && !mbar_wait(&full[s], (k / S) & 1u)) {
            live = false;
            atomicAdd(&g_wait_timeouts, 1ull);
        }
        const uint8_t* stage = smem + s * L::kStage + rsub * (kTile * 2) + cc * 16;
        uint4 v[8];
#pragma unroll
        for (int p = 0; p < 8; ++p) v[p] = *reinterpret_cast<const uint4*>(stage + p * 16 * (kTile * 2));
        __syncwarp();
        if (lane == 0 && live) mbar_arrive(&empty[s]);  // never release a stage whose copy may be in flight
        const uint32_t tile = blockIdx.x + k * gridDim.x;
        const int64_t r0 = (int64_t)(tile / nbr_row) * kTile, c0 = (int64_t)(tile % nbr_row) * kTile;
        bct_tile<FMT, ROWS, COLS>(v, tab, ts, 1 + g, tg, r0, c0, rows, cols, q_row, si_row, q_col, si_col);
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
                      (!q_col || aligned16(q_col)) && (rows / kTile) * (cols / kTile) <= 0x7FFFFFFF &&
                      rows <= 0x7FFFFFFF && cols <= 0x7FFFFFFF;
    if (fast) {
        constexpr int NG = kGroups, S = kStages;
        CUtensorMap xmap;
        const fp8_status_t es = encode_tile_map_u16(&xmap, x, rows, cols, kTile, kTile);
        if (es != FP8_OK) return es;
        const int64_t ntiles = (rows / kTile) * (cols / kTile);
        const int64_t grid = ntiles < sm_count() ? ntiles : sm_count();
        auto kernel = q_row == nullptr   ? block_ct_pipe_kernel<FMT, NG, S, false, true>
                      : q_col == nullptr ? block_ct_pipe_kernel<FMT, NG, S, true, false>
                                         : block_ct_pipe_kernel<FMT, NG, S, true, true>;
        return launch_smem(w, kernel, dim3((unsigned)grid), dim3(NG * 256 + 32), (size_t)BctLayout<NG, S>::kBytes, st,
                           xmap, rows, cols, q_row, si_row, q_col, si_col);
    }
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
    if (reinterpret_cast<uintptr_t>(x) % dtype_size(dtype))
        return fail(FP8_ERR_INVALID_ARG, "%s: x not element-aligned", fn);
    if ((scale_inv_row && reinterpret_cast<uintptr_t>(scale_inv_row) % 4) ||
        (scale_inv_col && reinterpret_cast<uintptr_t>(scale_inv_col) % 4))
        return fail(FP8_ERR_INVALID_ARG, "%s: scale_inv not 4-byte aligned", fn);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint8_t* xp = static_cast<const uint8_t*>(x);
    const bool bf16 = dtype == FP8_DT_BF16;
    if (fmt == FP8_E4M3) return launch_bct<kE4M3>(xp, bf16, rows, cols, q_row, scale_inv_row, q_col, scale_inv_col, st);
    return launch_bct<kE5M2>(xp, bf16, rows, cols, q_row, scale_inv_row, q_col, scale_inv_col, st);
}

namespace fp8q {
fp8_status_t block_ct_wait_timeouts(unsigned long long* count) {
    return cuda_status(cudaMemcpyFromSymbol(count, g_wait_timeouts, sizeof *count), "fp8_wait_timeouts");
}
}  // namespace fp8q

extern "C" fp8_status_t fp8_test_drop_tile_copy(int tile) {
    return cuda_status(cudaMemcpyToSymbol(g_drop_tile, &tile, sizeof tile), "fp8_test_drop_tile_copy");
}
