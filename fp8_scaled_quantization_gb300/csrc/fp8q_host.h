// fp8q_host.h -- host-side helpers shared by the C-ABI entry points.
#pragma once

#include <cstdint>
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

// Zero-initialised 64-byte workspace of (current device, stream); nullptr on
// failure (the error message is set).
Workspace* stream_workspace(cudaStream_t stream, fp8_status_t* st);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool valid_fmt(int f) { return f == FP8_E4M3 || f == FP8_E5M2; }
inline bool valid_dtype(int d) { return d == FP8_DT_BF16 || d == FP8_DT_FP32; }
inline bool valid_margin(int m) { return m >= -126 && m <= 126; }
inline int dtype_size(int d) { return d == FP8_DT_BF16 ? 2 : 4; }

}  // namespace fp8q
