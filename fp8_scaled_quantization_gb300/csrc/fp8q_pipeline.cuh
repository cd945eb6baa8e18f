// fp8q_pipeline.cuh -- tile pipelines of the sm_103a kernels: mbarriers,
// 2-D tensor-map bulk copies (TMA) into shared memory, bounded waits and named
// barriers for groups of warps.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fp8q {

// Waits of this translation unit's pipelines that gave up (each unit that
// includes this header has its own counter and a host reader for it).
static __device__ unsigned long long g_wait_timeouts;

// Tile pipelines: one producer thread copies input tiles into a ring of
// shared memory stages with the bulk-copy (TMA) engine, each stage guarded by two
// mbarriers -- `full` completes when the stage's bytes have landed, `empty`
// when its consumers have read it -- so that reads of the next tiles stay in
// flight while consumer warps work on the current one.

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t arrivals) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(arrivals) : "memory");
}

// Makes initialised mbarriers visible to the bulk-copy engine.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                     smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Waits for the phase of `bar` with the given parity to complete; gives up
// after about two seconds of %globaltimer (a copy that never lands) and
// returns false.  A cap on the number of polls bounds the wait even if the
// timer did not advance.
constexpr uint64_t kMbarWaitLimitNs = 2000000000ull;
constexpr uint32_t kMbarWaitMaxPolls = 1u << 24;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 0; i < kMbarWaitMaxPolls; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > kMbarWaitLimitNs) return false;
    }
    return false;
}

// The box of tensor map `map` at element coordinates (x, y) -- x innermost,
// x * element size a multiple of 16 bytes -- into shared `dst` (16-byte
// aligned, rows packed) by the bulk-copy engine; completion is counted on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// Barrier `id` (1..15) among `n` threads of the CTA (a multiple of 32).
__device__ __forceinline__ void group_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// The same, returning whether `pred` is true in any of the n threads.
__device__ __forceinline__ bool group_sync_or(int id, int n, bool pred) {
    uint32_t any;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.or.pred p, %2, %3, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(any)
        : "r"((uint32_t)pred), "r"(id), "r"(n)
        : "memory");
    return any != 0;
}

}  // namespace fp8q
