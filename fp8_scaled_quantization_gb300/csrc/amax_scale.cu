// amax_scale.cu -- amax reduction, the finalize kernel that turns per-CTA
// partials into amax / saturation totals / scales, and the delayed-scaling
// history update.
//
// amax ("Megatron FP8" §4: a dedicated reduction kernel producing an fp32
// scalar; §10: current scaling scans the tensor before the cast).  |x| of
// BF16 is its bit pattern with the sign cleared; for non-negative floats the
// unsigned order of the bits is the numeric order and NaN patterns sort above
// Inf, so an unsigned 16-bit max (two lanes per 32-bit word) is an exact,
// order-free, NaN-propagating amax.  Each CTA stores its maximum in its own
// workspace slot; the finalize kernel (one CTA, launched right after with
// programmatic dependent launch) reduces the slots and derives the scale.
//
// Delayed update ("Megatron FP8" §5, update_fp8_meta): write the new amax into
// slot step % len, take the window maximum (or the slot, for most_recent) and
// derive scale / scale_inv for the next cast.  Used both stand-alone
// (fp8_update_scale_delayed) and as the finalize of fp8_quantize_delayed.
#include "fp8q_device.cuh"
#include "fp8q_host.h"

namespace fp8q {
namespace {

constexpr int kThreads = 256;
// 12 16-byte loads in flight per thread (one chunk of 256 * 12 loads per CTA)
// at 4 CTAs per SM: 192 KB of reads in flight per SM, without spills.
constexpr int kLoads = 12;
constexpr int kFinThreads = 1024;

// x is 16-byte aligned here; `n` counts elements of width 2 (BF16) or 4 from x.
// CTA b reduces chunks b, b + grid, ... (one chunk unless the tensor needs
// more chunks than there are partial slots).
template <bool BF16>
__global__ void __launch_bounds__(kThreads, 4)
amax_kernel(const uint8_t* __restrict__ head, int head_n, const uint8_t* __restrict__ x, int64_t n,
            uint32_t* __restrict__ part_amax) {
    pdl_begin();
    constexpr int kPer = BF16 ? 8 : 4;  // elements per 16-byte chunk
    const int64_t nchunks = n / kPer;
    const int64_t per_cta = (int64_t)kThreads * kLoads;
    uint32_t acc = 0;  // BF16: u16x2 lanes; fp32: f32 bits
    for (int64_t base = (int64_t)blockIdx.x * per_cta + threadIdx.x; base < nchunks; base += (int64_t)gridDim.x * per_cta) {
        uint4 v[kLoads];
#pragma unroll
        for (int k = 0; k < kLoads; ++k) {
            const int64_t c = base + (int64_t)k * kThreads;
            v[k] = c < nchunks ? ldg_stream(x + c * 16) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int k = 0; k < kLoads; ++k) {
            if constexpr (BF16) {
                acc = max_u16x2(acc, max_u16x2(max_u16x2(abs_bf16x2(v[k].x), abs_bf16x2(v[k].y)),
                                               max_u16x2(abs_bf16x2(v[k].z), abs_bf16x2(v[k].w))));
            } else {
                acc = umax(acc, umax(umax(v[k].x & 0x7FFFFFFFu, v[k].y & 0x7FFFFFFFu),
                                     umax(v[k].z & 0x7FFFFFFFu, v[k].w & 0x7FFFFFFFu)));
            }
        }
    }
    uint32_t bits = BF16 ? fold_u16x2_to_f32bits(acc) : acc;

    // Elements before the first 16-byte boundary and after the last chunk.
    if (blockIdx.x == 0) {
        const int64_t tail_start = nchunks * kPer;
        const int64_t tail_n = n - tail_start;
        for (int64_t i = threadIdx.x; i < head_n + tail_n; i += kThreads) {
            const uint8_t* p = i < head_n ? head + i * (BF16 ? 2 : 4) : x + (tail_start + (i - head_n)) * (BF16 ? 2 : 4);
            uint32_t b = BF16 ? ((uint32_t)(*reinterpret_cast<const uint16_t*>(p) & 0x7FFFu) << 16)
                              : (*reinterpret_cast<const uint32_t*>(p) & 0x7FFFFFFFu);
            bits = umax(bits, b);
        }
    }

    __shared__ uint32_t red[32];
    bits = block_max_u32(bits, red);
    if (threadIdx.x == 0) part_amax[blockIdx.x] = bits;
}

// NaN-propagating maximum of hist[0..len) by the whole CTA (hist already
// holds this step's amax in its slot); valid in every thread.
__device__ __forceinline__ float window_max(const float* hist, int len) {
    __shared__ float red[32];
    float m = -INFINITY;
    int saw_nan = 0;
    for (int i = threadIdx.x; i < len; i += blockDim.x) {
        const float v = hist[i];
        if (isnan(v)) saw_nan = 1;
        else m = fmaxf(m, v);
    }
    saw_nan = __syncthreads_or(saw_nan);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = m;
    __syncthreads();
    m = lane < (int)(blockDim.x >> 5) ? red[lane] : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    return saw_nan ? __uint_as_float(0x7FC00000u) : m;
}

// One CTA: reduce the partials of the previous launch and write the results.
// Every load is issued up front (at most kFinLoads partials per thread and the
// history entries other than this step's slot) and one block reduction
// combines the amax maximum, the saturation sum and the window maximum of the
// old entries; the window maximum with the new amax is then the maximum of
// the two (NaN if either holds a NaN), which equals the maximum of the window
// after the slot write.
constexpr int kFinLoads = kMaxPartials / kFinThreads;

template <int FMT>
__global__ void __launch_bounds__(kFinThreads)
finalize_kernel(const uint32_t* __restrict__ part_amax, const unsigned long long* __restrict__ part_sat, int nparts,
                float* amax_out, unsigned long long* sat_out, float* scale_out, float* scale_inv_out, int margin,
                float* hist, int hist_len, int slot, int algo) {
    pdl_begin();
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    uint32_t a[kFinLoads];
    unsigned long long c[kFinLoads];
#pragma unroll
    for (int k = 0; k < kFinLoads; ++k) {
        const int i = t + k * kFinThreads;
        a[k] = (part_amax != nullptr && i < nparts) ? part_amax[i] : 0u;
        c[k] = (part_sat != nullptr && i < nparts) ? part_sat[i] : 0ull;
    }
    const bool window = hist != nullptr && algo == FP8_AMAX_MAX;
    float hm = -INFINITY;
    int nan = 0;
    if (window)
        for (int i = t; i < hist_len; i += kFinThreads) {
            if (i == slot) continue;
            const float v = hist[i];
            if (isnan(v)) nan = 1;
            else hm = fmaxf(hm, v);
        }
    uint32_t bits = 0;
    unsigned long long sat = 0;
#pragma unroll
    for (int k = 0; k < kFinLoads; ++k) {
        bits = umax(bits, a[k]);
        sat += c[k];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        bits = umax(bits, __shfl_xor_sync(0xFFFFFFFFu, bits, o));
        sat += __shfl_xor_sync(0xFFFFFFFFu, sat, o);
        hm = fmaxf(hm, __shfl_xor_sync(0xFFFFFFFFu, hm, o));
        nan |= __shfl_xor_sync(0xFFFFFFFFu, nan, o);
    }
    __shared__ uint32_t s_bits[32];
    __shared__ unsigned long long s_sat[32];
    __shared__ float s_hm[32];
    __shared__ int s_nan[32];
    if (lane == 0) {
        s_bits[warp] = bits;
        s_sat[warp] = sat;
        s_hm[warp] = hm;
        s_nan[warp] = nan;
    }
    __syncthreads();
    if (warp != 0) return;
    constexpr int kWarps = kFinThreads / 32;
    bits = lane < kWarps ? s_bits[lane] : 0u;
    sat = lane < kWarps ? s_sat[lane] : 0ull;
    hm = lane < kWarps ? s_hm[lane] : -INFINITY;
    nan = lane < kWarps ? s_nan[lane] : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        bits = umax(bits, __shfl_xor_sync(0xFFFFFFFFu, bits, o));
        sat += __shfl_xor_sync(0xFFFFFFFFu, sat, o);
        hm = fmaxf(hm, __shfl_xor_sync(0xFFFFFFFFu, hm, o));
        nan |= __shfl_xor_sync(0xFFFFFFFFu, nan, o);
    }
    if (lane != 0) return;
    if (bits > 0x7F800000u) bits = 0x7FC00000u;  // canonical NaN
    const float amax = __uint_as_float(bits);
    if (amax_out) *amax_out = amax;
    if (sat_out) *sat_out = sat;
    float eff = amax;
    if (hist != nullptr) {
        hist[slot] = amax;
        if (window) eff = (nan || isnan(amax)) ? __uint_as_float(0x7FC00000u) : fmaxf(hm, amax);
    }
    if (scale_out != nullptr) {
        float s, si;
        scale_from_amax<FMT>(eff, margin, &s, &si);
        *scale_out = s;
        *scale_inv_out = si;
    }
}

template <int FMT>
__global__ void __launch_bounds__(1024)
update_delayed_kernel(float* hist, int len, int slot, const float* new_amax, int algo, int margin,
                      float* scale_out, float* scale_inv_out) {
    pdl_begin();
    if (new_amax != nullptr && threadIdx.x == 0) hist[slot] = *new_amax;
    __syncthreads();  // the slot write is visible to the whole CTA
    const float eff = algo == FP8_AMAX_MOST_RECENT ? hist[slot] : window_max(hist, len);
    if (threadIdx.x == 0) {
        float s, si;
        scale_from_amax<FMT>(eff, margin, &s, &si);
        *scale_out = s;
        *scale_inv_out = si;
    }
}

}  // namespace

fp8_status_t launch_finalize(const FinalizeArgs& a, cudaStream_t st) {
    if (a.fmt == FP8_E4M3)
        return launch("finalize", finalize_kernel<kE4M3>, dim3(1), dim3(kFinThreads), st, a.part_amax, a.part_sat,
                      a.nparts, a.amax_out, a.sat_out, a.scale_out, a.scale_inv_out, a.margin, a.hist, a.hist_len,
                      a.slot, a.algo);
    return launch("finalize", finalize_kernel<kE5M2>, dim3(1), dim3(kFinThreads), st, a.part_amax, a.part_sat,
                  a.nparts, a.amax_out, a.sat_out, a.scale_out, a.scale_inv_out, a.margin, a.hist, a.hist_len, a.slot,
                  a.algo);
}

fp8_status_t enqueue_amax_partials(const void* x, fp8_dtype_t dtype, int64_t n, Workspace* ws, cudaStream_t st,
                                   int* nparts) {
    const int es = dtype_size(dtype);
    // Peel elements up to the first 16-byte boundary.
    const uint8_t* p = static_cast<const uint8_t*>(x);
    int64_t head = p ? (int64_t)(((16u - (reinterpret_cast<uintptr_t>(p) & 15u)) & 15u) / es) : 0;
    if (head > n) head = n;
    const uint8_t* body = p ? p + head * es : p;
    const int64_t body_n = n - head;

    const int per = dtype == FP8_DT_BF16 ? 8 : 4;
    const int64_t chunks = body_n / per;
    int64_t grid = (chunks + (int64_t)kThreads * kLoads - 1) / ((int64_t)kThreads * kLoads);
    if (grid < 1) grid = 1;
    if (grid > kMaxPartials) grid = kMaxPartials;
    *nparts = (int)grid;
    if (dtype == FP8_DT_BF16)
        return launch("fp8_amax", amax_kernel<true>, dim3((unsigned)grid), dim3(kThreads), st, p, (int)head, body,
                      body_n, ws->amax);
    return launch("fp8_amax", amax_kernel<false>, dim3((unsigned)grid), dim3(kThreads), st, p, (int)head, body, body_n,
                  ws->amax);
}

}  // namespace fp8q

using namespace fp8q;

extern "C" fp8_status_t fp8_amax(const void* x, fp8_dtype_t dtype, int64_t n, float* amax_out,
                                 fp8_format_t fmt, int margin, float* scale_out, float* scale_inv_out,
                                 void* stream) {
    if (!valid_dtype(dtype)) return fail(FP8_ERR_INVALID_ARG, "fp8_amax: unknown dtype %d", (int)dtype);
    if (n < 0) return fail(FP8_ERR_INVALID_ARG, "fp8_amax: n < 0");
    if (n > 0 && x == nullptr) return fail(FP8_ERR_INVALID_ARG, "fp8_amax: x is NULL");
    if (amax_out == nullptr) return fail(FP8_ERR_INVALID_ARG, "fp8_amax: amax_out is NULL");
    if ((scale_out == nullptr) != (scale_inv_out == nullptr))
        return fail(FP8_ERR_INVALID_ARG, "fp8_amax: scale_out and scale_inv_out must both be set or both NULL");
    if (scale_out && !valid_fmt(fmt)) return fail(FP8_ERR_INVALID_ARG, "fp8_amax: unknown format %d", (int)fmt);
    if (scale_out && !valid_margin(margin)) return fail(FP8_ERR_INVALID_ARG, "fp8_amax: margin out of [-126, 126]");
    const int es = dtype_size(dtype);
    if (reinterpret_cast<uintptr_t>(x) % es) return fail(FP8_ERR_INVALID_ARG, "fp8_amax: x not element-aligned");

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    fp8_status_t s;
    Workspace* ws = stream_workspace(st, &s);
    if (!ws) return s;
    int nparts = 0;
    s = enqueue_amax_partials(x, dtype, n, ws, st, &nparts);
    if (s != FP8_OK) return s;
    FinalizeArgs fa;
    fa.part_amax = ws->amax;
    fa.nparts = nparts;
    fa.amax_out = amax_out;
    fa.scale_out = scale_out;
    fa.scale_inv_out = scale_inv_out;
    fa.fmt = (int)fmt;
    fa.margin = margin;
    return launch_finalize(fa, st);
}

extern "C" fp8_status_t fp8_update_scale_delayed(float* amax_history, int history_len, int64_t step,
                                                 const float* new_amax, fp8_amax_algo_t algo,
                                                 fp8_format_t fmt, int margin, float* scale_out,
                                                 float* scale_inv_out, void* stream) {
    if (amax_history == nullptr) return fail(FP8_ERR_INVALID_ARG, "fp8_update_scale_delayed: amax_history is NULL");
    if (history_len < 1 || history_len > 65536)
        return fail(FP8_ERR_INVALID_ARG, "fp8_update_scale_delayed: history_len must be in [1, 65536]");
    if (step < 0) return fail(FP8_ERR_INVALID_ARG, "fp8_update_scale_delayed: step < 0");
    if (algo != FP8_AMAX_MAX && algo != FP8_AMAX_MOST_RECENT)
        return fail(FP8_ERR_INVALID_ARG, "fp8_update_scale_delayed: unknown algo %d", (int)algo);
    if (!valid_fmt(fmt)) return fail(FP8_ERR_INVALID_ARG, "fp8_update_scale_delayed: unknown format %d", (int)fmt);
    if (!valid_margin(margin)) return fail(FP8_ERR_INVALID_ARG, "fp8_update_scale_delayed: margin out of [-126, 126]");
    if (scale_out == nullptr || scale_inv_out == nullptr)
        return fail(FP8_ERR_INVALID_ARG, "fp8_update_scale_delayed: scale_out / scale_inv_out is NULL");

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int slot = (int)(step % history_len);
    const int threads = history_len >= 1024 ? 1024 : (history_len >= 256 ? 256 : 32);
    if (fmt == FP8_E4M3)
        return launch("fp8_update_scale_delayed", update_delayed_kernel<kE4M3>, dim3(1), dim3(threads), st,
                      amax_history, history_len, slot, new_amax, (int)algo, margin, scale_out, scale_inv_out);
    return launch("fp8_update_scale_delayed", update_delayed_kernel<kE5M2>, dim3(1), dim3(threads), st, amax_history,
                  history_len, slot, new_amax, (int)algo, margin, scale_out, scale_inv_out);
}
