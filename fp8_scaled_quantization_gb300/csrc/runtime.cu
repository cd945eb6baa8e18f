// runtime.cu -- status strings, per-thread error text, launch counting, SM
// count cache and the per-(device, stream) reduction workspace.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <map>
#include <mutex>
#include <utility>

#include <cudaTypedefs.h>

#include "fp8q_device.cuh"
#include "fp8q_host.h"

namespace fp8q {

namespace {
thread_local char g_last_error[512] = "";
std::atomic<unsigned long long> g_launches{0};

std::mutex g_mu;
std::map<int, int> g_sm_count;                                 // device -> SMs
std::map<std::pair<int, uintptr_t>, Workspace*> g_workspaces;  // (device, stream) -> ws
}  // namespace

fp8_status_t fail(fp8_status_t st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return st;
}

fp8_status_t cuda_status(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return FP8_OK;
    return fail(FP8_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

fp8_status_t after_launch(const char* kernel) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_status(e, kernel);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return FP8_OK;
}

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_sm_count.find(dev);
    if (it != g_sm_count.end()) return it->second;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    g_sm_count[dev] = n;
    return n;
}

fp8_status_t encode_tile_map_u16(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_rows,
                                 int box_cols) {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (encode == nullptr) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
            cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
            if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
                return fail(FP8_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
            encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
    }
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    const cuuint32_t elem_strides[2] = {1, 1};
    const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), dims, strides, box,
                              elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(FP8_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return FP8_OK;
}

Workspace* stream_workspace(cudaStream_t stream, fp8_status_t* st) {
    *st = FP8_OK;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        *st = cuda_status(e, "cudaGetDevice");
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    auto key = std::make_pair(dev, reinterpret_cast<uintptr_t>(stream));
    auto it = g_workspaces.find(key);
    if (it != g_workspaces.end()) return it->second;
    // First use on this stream.  Relax the thread's capture mode so that the
    // allocation is legal while a stream is being captured.  The partial slots
    // need no initial value: a launch writes every slot its finalize reads.
    cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
    cudaThreadExchangeStreamCaptureMode(&mode);
    void* p = nullptr;
    e = cudaMalloc(&p, sizeof(Workspace));
    cudaThreadExchangeStreamCaptureMode(&mode);
    if (e != cudaSuccess) {
        *st = cuda_status(e, "cudaMalloc(workspace)");
        return nullptr;
    }
    auto* ws = static_cast<Workspace*>(p);
    g_workspaces[key] = ws;
    return ws;
}

}  // namespace fp8q

extern "C" {

const char* fp8_status_string(fp8_status_t status) {
    switch (status) {
        case FP8_OK: return "FP8_OK";
        case FP8_ERR_INVALID_ARG: return "FP8_ERR_INVALID_ARG";
        case FP8_ERR_UNSUPPORTED: return "FP8_ERR_UNSUPPORTED";
        case FP8_ERR_CUDA: return "FP8_ERR_CUDA";
    }
    return "FP8_ERR_UNKNOWN";
}

const char* fp8_last_error_message(void) { return fp8q::g_last_error; }

int fp8_version(void) { return (FP8Q_VERSION_MAJOR << 16) | FP8Q_VERSION_MINOR; }

unsigned long long fp8_launch_count(void) { return fp8q::g_launches.load(std::memory_order_relaxed); }

fp8_status_t fp8_wait_timeouts(unsigned long long* count) {
    using namespace fp8q;
    if (count == nullptr) return fail(FP8_ERR_INVALID_ARG, "fp8_wait_timeouts: count is NULL");
    fp8_status_t st = cuda_status(cudaDeviceSynchronize(), "fp8_wait_timeouts");
    if (st == FP8_OK) st = block_ct_wait_timeouts(count);
    return st;
}

fp8_status_t fp8_release_stream_workspace(void* stream) {
    using namespace fp8q;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e, "fp8_release_stream_workspace: cudaGetDevice");
    Workspace* ws = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_workspaces.find(std::make_pair(dev, reinterpret_cast<uintptr_t>(stream)));
        if (it == g_workspaces.end()) return FP8_OK;  // nothing was allocated for this stream
        ws = it->second;
        g_workspaces.erase(it);
    }
    // The stream's queued work may still use the workspace.
    e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) e = cudaFree(ws);
    return cuda_status(e, "fp8_release_stream_workspace");
}

}  // extern "C"
