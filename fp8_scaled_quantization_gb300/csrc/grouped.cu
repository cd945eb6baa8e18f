// grouped.cu -- many tensors in one launch: per-tensor amax with current
// scale, and per-tensor scaled casts, over a table of tensors passed by value
// in the kernel parameters.
//
// "Megatron FP8" §21: every expert of an MoE layer keeps its own FP8 scaling
// state (per-tensor amax and scale, no synchronisation between experts); §24:
// the scaling overhead (amax and scale computation) should stay a small share
// of the step.  Issuing one launch for all tensors instead of two or three per
// tensor removes the per-launch ramp and tail that dominate small tensors.
//
// Work is split into fixed chunks (16384 BF16 / 8192 fp32 elements for the
// cast, a multiple of 2048 16-byte loads for amax); CTA b finds its tensor by
// binary search over the table's chunk offsets.  Reductions store one partial
// per CTA; the grouped finalize runs one CTA per tensor over that tensor's
// partials.
#include "fp8q_device.cuh"
#include "fp8q_host.h"

namespace fp8q {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxGroup = 128;

struct GroupTable {
    const uint8_t* x[kMaxGroup];
    uint8_t* q[kMaxGroup];
    int64_t n[kMaxGroup];
    int64_t chunk_begin[kMaxGroup + 1];  // prefix sums of per-tensor chunk counts
    int count;
};

__device__ __forceinline__ int find_tensor(const GroupTable& t, int64_t chunk) {
    int lo = 0, hi = t.count - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (t.chunk_begin[mid] <= chunk) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// amax: one chunk of `reps` x 2048 16-byte loads per CTA (reps > 1 only when
// the group needs more chunks than there are partial slots); x pointers
// 16-byte aligned.
template <bool BF16>
__global__ void __launch_bounds__(kThreads)
grouped_amax_kernel(const __grid_constant__ GroupTable t, int reps, uint32_t* __restrict__ part_amax) {
    pdl_begin();
    constexpr int kPer = BF16 ? 8 : 4;
    const int64_t chunk = blockIdx.x;
    const int i = find_tensor(t, chunk);
    const int64_t local = chunk - t.chunk_begin[i];
    const uint8_t* x = t.x[i];
    const int64_t n = t.n[i], nl = n / kPer;  // 16-byte loads of tensor i
    uint32_t acc = 0;
    for (int r = 0; r < reps; ++r) {
        const int64_t base = (local * reps + r) * kThreads * 8 + threadIdx.x;
        if (base >= nl) break;
        uint4 v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int64_t c = base + (int64_t)k * kThreads;
            v[k] = c < nl ? ldg_stream(x + c * 16) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
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
    if (local == 0) {  // elements after the last full 16-byte load of tensor i
        for (int64_t e = nl * kPer + threadIdx.x; e < n; e += kThreads) {
            const uint32_t b = BF16 ? (uint32_t)(reinterpret_cast<const uint16_t*>(x)[e] & 0x7FFFu) << 16
                                    : (reinterpret_cast<const uint32_t*>(x)[e] & 0x7FFFFFFFu);
            bits = umax(bits, b);
        }
    }
    __shared__ uint32_t red[32];
    bits = block_max_u32(bits, red);
    if (threadIdx.x == 0) part_amax[chunk] = bits;
}

// One CTA per tensor: reduce its partials, write amax / scale / scale_inv.
template <int FMT>
__global__ void __launch_bounds__(kThreads)
grouped_finalize_kernel(const __grid_constant__ GroupTable t, const uint32_t* __restrict__ part_amax,
                        float* amax_out, float* scale_out, float* scale_inv_out, int margin) {
    pdl_begin();
    const int i = blockIdx.x;
    uint32_t bits = 0;
    for (int64_t c = t.chunk_begin[i] + threadIdx.x; c < t.chunk_begin[i + 1]; c += kThreads)
        bits = umax(bits, part_amax[c]);
    __shared__ uint32_t red[32];
    bits = block_max_u32(bits, red);
    if (threadIdx.x != 0) return;
    if (bits > 0x7F800000u) bits = 0x7FC00000u;
    const float amax = __uint_as_float(bits);
    if (amax_out) amax_out[i] = amax;
    if (scale_out) {
        float s, si;
        scale_from_amax<FMT>(amax, margin, &s, &si);
        scale_out[i] = s;
        scale_inv_out[i] = si;
    }
}

// Cast: one chunk of 8 items of one 16-byte load (8 BF16 / 4 fp32 elements)
// per thread per CTA -- a warp loads 512 contiguous bytes -- tensor i scaled by
// scale[i]; x and q pointers 16-byte aligned.
template <int FMT, bool BF16>
__global__ void __launch_bounds__(kThreads, 5)
grouped_quantize_kernel(const __grid_constant__ GroupTable t, const float* __restrict__ scales) {
    pdl_begin();
    constexpr int kItems = 8, kPer = BF16 ? 8 : 4;
    const int64_t chunk = blockIdx.x;
    const int i = find_tensor(t, chunk);
    const int64_t local = chunk - t.chunk_begin[i];
    const uint8_t* x = t.x[i];
    uint8_t* q = t.q[i];
    const int64_t n = t.n[i], nitems = n / kPer;
    const float scale = scales[i];
    const int64_t ib = local * kThreads * kItems + threadIdx.x;
    uint4 v[kItems];
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
        const int64_t it = ib + (int64_t)k * kThreads;
        if (it < nitems) v[k] = ldg_stream(x + it * 16);
    }
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
        const int64_t it = ib + (int64_t)k * kThreads;
        if (it >= nitems) break;
        if constexpr (BF16) {
            uint32_t m;
            Codes8 cd = cvt_bf16x8<FMT>(v[k], scale, &m);
            if (chunk_needs_fixup<FMT, false>(fold_u16x2_to_f32bits(m), scale)) fixup_bf16x8<FMT>(v[k], scale, &cd);
            stg_stream(q + it * 8, make_uint2(cd.lo, cd.hi));
        } else {
            const float4 f = make_float4(__uint_as_float(v[k].x), __uint_as_float(v[k].y), __uint_as_float(v[k].z),
                                         __uint_as_float(v[k].w));
            uint32_t m;
            uint32_t w = cvt_f32x4<FMT>(f, scale, &m);
            if (chunk_needs_fixup<FMT, false>(m, scale)) fixup_f32x4<FMT>(f, scale, &w);
            __stcs(reinterpret_cast<unsigned int*>(q + it * 4), w);
        }
    }
    if (local == 0) {  // elements after the last full item of tensor i
        for (int64_t e = nitems * kPer + threadIdx.x; e < n; e += kThreads) {
            const float xv = BF16 ? __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(x)[e] << 16)
                                  : reinterpret_cast<const float*>(x)[e];
            uint32_t s;
            q[e] = (uint8_t)quant_one<FMT>(xv, scale, &s);
        }
    }
}

// Fill the table; chunk sizes in elements.  Returns false (message set) on a
// bad entry.
bool fill_table(GroupTable* t, int count, const void* const* xs, uint8_t* const* qs, const int64_t* ns,
                int64_t chunk_elems, const char* fn, fp8_status_t* st) {
    t->count = count;
    t->chunk_begin[0] = 0;
    for (int i = 0; i < count; ++i) {
        if (ns[i] < 0) { *st = fail(FP8_ERR_INVALID_ARG, "%s: tensor %d has n < 0", fn, i); return false; }
        if (ns[i] > 0 && xs[i] == nullptr) { *st = fail(FP8_ERR_INVALID_ARG, "%s: tensor %d x is NULL", fn, i); return false; }
        if (ns[i] > 0 && !aligned16(xs[i]))
            { *st = fail(FP8_ERR_UNSUPPORTED, "%s: tensor %d x is not 16-byte aligned", fn, i); return false; }
        if (qs) {
            if (ns[i] > 0 && qs[i] == nullptr) { *st = fail(FP8_ERR_INVALID_ARG, "%s: tensor %d q is NULL", fn, i); return false; }
            if (ns[i] > 0 && !aligned16(qs[i]))
                { *st = fail(FP8_ERR_UNSUPPORTED, "%s: tensor %d q is not 16-byte aligned", fn, i); return false; }
            t->q[i] = qs[i];
        }
        t->x[i] = static_cast<const uint8_t*>(xs[i]);
        t->n[i] = ns[i];
        int64_t chunks = (ns[i] + chunk_elems - 1) / chunk_elems;
        if (chunks < 1) chunks = 1;  // every tensor owns a chunk, so its partial / tail is written
        t->chunk_begin[i + 1] = t->chunk_begin[i] + chunks;
    }
    if (t->chunk_begin[count] > 0x7FFFFFFF) { *st = fail(FP8_ERR_UNSUPPORTED, "%s: too many chunks", fn); return false; }
    return true;
}

}  // namespace
}  // namespace fp8q

using namespace fp8q;

extern "C" fp8_status_t fp8_amax_grouped(int count, const void* const* xs, const int64_t* ns, fp8_dtype_t dtype,
                                         float* amax_out, fp8_format_t fmt, int margin, float* scale_out,
                                         float* scale_inv_out, void* stream) {
    const char* fn = "fp8_amax_grouped";
    if (count < 1 || count > kMaxGroup) return fail(FP8_ERR_INVALID_ARG, "%s: count must be in [1, %d]", fn, kMaxGroup);
    if (xs == nullptr || ns == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: xs / ns is NULL", fn);
    if (!valid_dtype(dtype)) return fail(FP8_ERR_INVALID_ARG, "%s: unknown dtype %d", fn, (int)dtype);
    if (amax_out == nullptr && scale_out == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: no output requested", fn);
    if ((scale_out == nullptr) != (scale_inv_out == nullptr))
        return fail(FP8_ERR_INVALID_ARG, "%s: scale_out and scale_inv_out must both be set or both NULL", fn);
    if (scale_out && !valid_fmt(fmt)) return fail(FP8_ERR_INVALID_ARG, "%s: unknown format %d", fn, (int)fmt);
    if (scale_out && !valid_margin(margin)) return fail(FP8_ERR_INVALID_ARG, "%s: margin out of [-126, 126]", fn);
    const bool bf16 = dtype == FP8_DT_BF16;
    GroupTable t;
    fp8_status_t s = FP8_OK;
    const int64_t base_elems = (int64_t)kThreads * 8 * (bf16 ? 8 : 4);  // one chunk of 2048 16-byte loads
    if (!fill_table(&t, count, xs, nullptr, ns, base_elems, fn, &s)) return s;
    // Every tensor rounds its chunk count up, so with chunks of reps base
    // chunks the group needs at most total / reps + count of them.
    int64_t reps = 1;
    if (t.chunk_begin[count] > kMaxPartials) {
        reps = (t.chunk_begin[count] + (kMaxPartials - count) - 1) / (kMaxPartials - count);
        if (reps > 0x7FFFFFFF) return fail(FP8_ERR_UNSUPPORTED, "%s: group too large", fn);
        if (!fill_table(&t, count, xs, nullptr, ns, base_elems * reps, fn, &s)) return s;
        if (t.chunk_begin[count] > kMaxPartials) return fail(FP8_ERR_UNSUPPORTED, "%s: group too large", fn);
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Workspace* ws = stream_workspace(st, &s);
    if (!ws) return s;
    const dim3 grid((unsigned)t.chunk_begin[count]), block(kThreads);
    const int r = (int)reps;
    s = bf16 ? launch(fn, grouped_amax_kernel<true>, grid, block, st, t, r, ws->amax)
             : launch(fn, grouped_amax_kernel<false>, grid, block, st, t, r, ws->amax);
    if (s != FP8_OK) return s;
    if (fmt == FP8_E5M2)
        return launch(fn, grouped_finalize_kernel<kE5M2>, dim3(count), block, st, t, (const uint32_t*)ws->amax, amax_out,
                      scale_out, scale_inv_out, margin);
    return launch(fn, grouped_finalize_kernel<kE4M3>, dim3(count), block, st, t, (const uint32_t*)ws->amax, amax_out,
                  scale_out, scale_inv_out, margin);
}

extern "C" fp8_status_t fp8_quantize_grouped(int count, const void* const* xs, const int64_t* ns, fp8_dtype_t dtype,
                                             fp8_format_t fmt, const float* scales, uint8_t* const* qs, void* stream) {
    const char* fn = "fp8_quantize_grouped";
    if (count < 1 || count > kMaxGroup) return fail(FP8_ERR_INVALID_ARG, "%s: count must be in [1, %d]", fn, kMaxGroup);
    if (xs == nullptr || ns == nullptr || qs == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: xs / ns / qs is NULL", fn);
    if (!valid_dtype(dtype)) return fail(FP8_ERR_INVALID_ARG, "%s: unknown dtype %d", fn, (int)dtype);
    if (!valid_fmt(fmt)) return fail(FP8_ERR_INVALID_ARG, "%s: unknown format %d", fn, (int)fmt);
    if (scales == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: scales is NULL", fn);
    const bool bf16 = dtype == FP8_DT_BF16;
    GroupTable t;
    fp8_status_t s = FP8_OK;
    if (!fill_table(&t, count, xs, qs, ns, (int64_t)kThreads * 8 * (bf16 ? 8 : 4), fn, &s)) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const dim3 grid((unsigned)t.chunk_begin[count]), block(kThreads);
    if (fmt == FP8_E4M3)
        return bf16 ? launch(fn, grouped_quantize_kernel<kE4M3, true>, grid, block, st, t, scales)
                    : launch(fn, grouped_quantize_kernel<kE4M3, false>, grid, block, st, t, scales);
    return bf16 ? launch(fn, grouped_quantize_kernel<kE5M2, true>, grid, block, st, t, scales)
                : launch(fn, grouped_quantize_kernel<kE5M2, false>, grid, block, st, t, scales);
}
