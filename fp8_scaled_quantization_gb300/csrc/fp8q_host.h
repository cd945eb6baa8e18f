// fp8q_host.h -- host-side helpers shared by the C-ABI entry points.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "fp8q.h"

namespace fp8q {

struct Workspace;

// Record `msg` as the calling thread's last error and return `st`.
fp8_status_t fail(fp8_status_t st, const char* fmt, ...);

// FP8_OK, or FP8_ERR_CUDA with the runtime's text when `e` is an error.
fp8_status_t cuda_status(cudaError_t e, const char* what);

// Check the launch just made (cudaGetLastError) and count it.
fp8_status_t after_launch(const char* kernel);

// Number of SMs of the current device (cached per device).
int sm_count();

// Tensor map of a row-major [rows, cols] array of 16-bit elements at `base`
// (16-byte aligned, cols * 2 a multiple of 16, rows and cols at most 2^32),
// read in boxes of box_rows x box_cols elements into packed shared-memory rows
// (no swizzle).  Elements outside the array read as zero.  The encoder is the
// driver's, reached through the runtime.
fp8_status_t encode_tile_map_u16(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_rows,
                                 int box_cols);

// The wait-timeout counter of the pipelined kernels' translation unit on the
// current device (no synchronisation: call after the device is idle).
fp8_status_t block_ct_wait_timeouts(unsigned long long* count);

// Workspace of (current device, stream) for per-CTA partials; nullptr on
// failure (the error message is set).
Workspace* stream_workspace(cudaStream_t stream, fp8_status_t* st);

// Launch `kernel` on `st` with `smem` bytes of dynamic shared memory and
// programmatic stream serialization allowed (the kernel starts with
// pdl_begin()), then check and count the launch.
template <typename... KArgs, typename... Args>
fp8_status_t launch_smem(const char* what, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                         cudaStream_t st, Args... args) {
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return cuda_status(e, what);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
    if (e != cudaSuccess) return cuda_status(e, what);
    return after_launch(what);
}

// The same without dynamic shared memory.
template <typename... KArgs, typename... Args>
fp8_status_t launch(const char* what, void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t st,
                    Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
    if (e != cudaSuccess) return cuda_status(e, what);
    return after_launch(what);
}

// What the one-CTA finalize kernel does with the partials of `nparts` CTAs:
// amax (NaN-canonical) and saturation totals, the current scale from the amax,
// or -- when hist is set -- the delayed update (hist[slot] = amax, scale from
// the window) written to scale_out / scale_inv_out.
struct FinalizeArgs {
    const uint32_t* part_amax = nullptr;
    const unsigned long long* part_sat = nullptr;
    int nparts = 0;
    float* amax_out = nullptr;
    unsigned long long* sat_out = nullptr;
    float* scale_out = nullptr;
    float* scale_inv_out = nullptr;
    int fmt = FP8_E4M3;
    int margin = 0;
    float* hist = nullptr;
    int hist_len = 0;
    int slot = 0;
    int algo = FP8_AMAX_MAX;
};
fp8_status_t launch_finalize(const FinalizeArgs& fa, cudaStream_t st);

// The amax kernel alone: one partial max |x| (fp32 bits) per CTA into
// ws->amax; *nparts receives their count.  x element-aligned, n >= 0.
fp8_status_t enqueue_amax_partials(const void* x, fp8_dtype_t dtype, int64_t n, Workspace* ws, cudaStream_t st,
                                   int* nparts);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool valid_fmt(int f) { return f == FP8_E4M3 || f == FP8_E5M2; }
inline bool valid_dtype(int d) { return d == FP8_DT_BF16 || d == FP8_DT_FP32; }
inline bool valid_margin(int m) { return m >= -126 && m <= 126; }
inline int dtype_size(int d) { return d == FP8_DT_BF16 ? 2 : 4; }

}  // namespace fp8q
