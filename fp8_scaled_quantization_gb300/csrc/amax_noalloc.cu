// amax_noalloc.cu -- fp8_amax_noalloc: the amax reduction with fused
// current-scale finalize, for callers that must not allocate device memory.
//
// Some callers cannot let a library call cudaMalloc: code that runs while a
// stream is captured under the global capture mode (where the allocation is
// an illegal call), engines and plugins that own a fixed memory budget and
// hand out only the buffers they planned, and allocator-managed frameworks
// that forbid raw device allocations behind their back.  fp8_amax keeps a
// small workspace per (device, stream) that it allocates on first use; this
// variant keeps its scratch in a file-scope device array instead, so it never
// allocates.
//
// The scratch (kScratchWords 32-bit words, 16.25 KB) lives for the whole
// process on every GPU that loads the library.  Word 0 is the CTA arrival
// counter; words 64 .. 64 + kMaxCtas - 1 hold one partial maximum per CTA.
// Each CTA reduces a fixed slice of kSliceElems elements, so the scratch
// bounds the input: n <= kMaxCtas * kSliceElems = 2^28 elements.
#include <map>
#include <mutex>

#include "fp8q_device.cuh"
#include "fp8q_host.h"

namespace fp8q {
namespace {

constexpr int kMaxCtas = 4096;
constexpr int64_t kSliceElems = 65536;
constexpr int kPartialBase = 64;  // partials start one 256-byte line after the counter
constexpr int kScratchWords = kPartialBase + kMaxCtas;
constexpr int kNaThreads = 256;

static __device__ __align__(256) unsigned int g_amax_scratch[kScratchWords];

template <bool BF16>
__device__ __forceinline__ uint32_t abs_bits_at(const uint8_t* x, int64_t i) {
    if constexpr (BF16) return (uint32_t)(reinterpret_cast<const uint16_t*>(x)[i] & 0x7FFFu) << 16;
    else return reinterpret_cast<const uint32_t*>(x)[i] & 0x7FFFFFFFu;
}

// One CTA per slice [blockIdx.x * kSliceElems, +kSliceElems) of x.
template <bool BF16>
__global__ void __launch_bounds__(kNaThreads)
amax_noalloc_kernel(const uint8_t* __restrict__ x, int64_t n, int vec, unsigned int* scratch, FinishArgs fa) {
    constexpr int kPer = BF16 ? 8 : 4;  // elements per 16-byte chunk
    const int64_t e0 = (int64_t)blockIdx.x * kSliceElems;
    const int64_t e1 = e0 + kSliceElems < n ? e0 + kSliceElems : n;
    uint32_t bits = 0;
    if (vec) {
        // x is 16-byte aligned and so is every slice start.
        const int64_t c0 = e0 / kPer, c1 = e1 / kPer;
        uint32_t acc = 0;
        for (int64_t c = c0 + threadIdx.x; c < c1; c += kNaThreads * 8) {
            uint4 v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int64_t cc = c + (int64_t)k * kNaThreads;
                v[k] = cc < c1 ? ldg_stream(x + cc * 16) : make_uint4(0, 0, 0, 0);
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
        bits = BF16 ? fold_u16x2_to_f32bits(acc) : acc;
        for (int64_t i = c1 * kPer + threadIdx.x; i < e1; i += kNaThreads) bits = umax(bits, abs_bits_at<BF16>(x, i));
    } else {
        for (int64_t i = e0 + threadIdx.x; i < e1; i += kNaThreads) bits = umax(bits, abs_bits_at<BF16>(x, i));
    }

    __shared__ uint32_t red[32];
    __shared__ int is_last;
    bits = block_max_u32(bits, red);
    if (threadIdx.x == 0) {
        scratch[kPartialBase + blockIdx.x] = bits;
        __threadfence();
        is_last = atomicAdd(&scratch[0], 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    uint32_t m = 0;
    for (unsigned i = threadIdx.x; i < gridDim.x; i += kNaThreads) m = umax(m, __ldcg(&scratch[kPartialBase + i]));
    m = block_max_u32(m, red);
    if (threadIdx.x == 0) {
        scratch[0] = 0u;  // leave the counter cleared for the next call
        if (m > 0x7F800000u) m = 0x7FC00000u;  // canonical NaN
        const float amax = __uint_as_float(m);
        *fa.amax_out = amax;
        if (fa.scale_out) {
            float si;
            const float s = scale_from_amax_rt(fa.fmt, amax, fa.margin, &si);
            *fa.scale_out = s;
            *fa.scale_inv_out = si;
        }
    }
}

std::mutex g_na_mu;
std::map<int, unsigned int*> g_na_scratch;  // device -> address of g_amax_scratch

// Device address of the scratch on the current device, looked up once per
// device (the first call on a device does this set-up).
fp8_status_t scratch_address(unsigned int** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e, "fp8_amax_noalloc: cudaGetDevice");
    std::lock_guard<std::mutex> lk(g_na_mu);
    auto it = g_na_scratch.find(dev);
    if (it != g_na_scratch.end()) {
        *out = it->second;
        return FP8_OK;
    }
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_amax_scratch);
    if (e != cudaSuccess) return cuda_status(e, "fp8_amax_noalloc: cudaGetSymbolAddress(scratch)");
    g_na_scratch[dev] = static_cast<unsigned int*>(p);
    *out = static_cast<unsigned int*>(p);
    return FP8_OK;
}

}  // namespace
}  // namespace fp8q

using namespace fp8q;

extern "C" fp8_status_t fp8_amax_noalloc(const void* x, fp8_dtype_t dtype, int64_t n, float* amax_out,
                                         fp8_format_t fmt, int margin, float* scale_out, float* scale_inv_out,
                                         void* stream) {
    const char* fn = "fp8_amax_noalloc";
    if (!valid_dtype(dtype)) return fail(FP8_ERR_INVALID_ARG, "%s: unknown dtype %d", fn, (int)dtype);
    if (n < 0) return fail(FP8_ERR_INVALID_ARG, "%s: n < 0", fn);
    if (n > (int64_t)kMaxCtas * kSliceElems)
        return fail(FP8_ERR_UNSUPPORTED, "%s: n = %lld exceeds the fixed scratch capacity of %lld elements", fn,
                    (long long)n, (long long)kMaxCtas * kSliceElems);
    if (n > 0 && x == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: x is NULL", fn);
    if (amax_out == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: amax_out is NULL", fn);
    if ((scale_out == nullptr) != (scale_inv_out == nullptr))
        return fail(FP8_ERR_INVALID_ARG, "%s: scale_out and scale_inv_out must both be set or both NULL", fn);
    if (scale_out && !valid_fmt(fmt)) return fail(FP8_ERR_INVALID_ARG, "%s: unknown format %d", fn, (int)fmt);
    if (scale_out && !valid_margin(margin)) return fail(FP8_ERR_INVALID_ARG, "%s: margin out of [-126, 126]", fn);
    if (reinterpret_cast<uintptr_t>(x) % dtype_size(dtype)) return fail(FP8_ERR_INVALID_ARG, "%s: x not element-aligned", fn);

    unsigned int* scratch = nullptr;
    fp8_status_t s = scratch_address(&scratch);
    if (s != FP8_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // The arrival counter must start at zero; clear it on the stream in case an
    // earlier launch did not finish.
    cudaError_t e = cudaMemsetAsync(scratch, 0, sizeof(unsigned int), st);
    if (e != cudaSuccess) return cuda_status(e, "fp8_amax_noalloc: cudaMemsetAsync(counter)");
    int64_t grid = (n + kSliceElems - 1) / kSliceElems;
    if (grid < 1) grid = 1;
    const int vec = aligned16(x);
    FinishArgs fa{amax_out, scale_out, scale_inv_out, nullptr, (int)fmt, margin};
    const uint8_t* xp = static_cast<const uint8_t*>(x);
    if (dtype == FP8_DT_BF16)
        amax_noalloc_kernel<true><<<(unsigned)grid, kNaThreads, 0, st>>>(xp, n, vec, scratch, fa);
    else
        amax_noalloc_kernel<false><<<(unsigned)grid, kNaThreads, 0, st>>>(xp, n, vec, scratch, fa);
    return after_launch(fn);
}
