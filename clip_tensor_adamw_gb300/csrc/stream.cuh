// Device helpers shared by the streaming kernels (adamw.cu, norm.cu, sgd.cu, scale.cu): 32- and 16-byte streaming
// accesses, binary16 widening, programmatic dependent launch, the gradient factor read, L2 prefetch, the search in a
// pack's table, and the persistent grids' work queue.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "plan.h"

namespace mica {
namespace {

// ------------------------------------------------------------------------------------------------------------------
// memory access
// ------------------------------------------------------------------------------------------------------------------

// 32 bytes, not kept in L1, first to leave L2 (each byte is used once)
__device__ __forceinline__ void ld8_stream(const float* p, float (&a)[8]) {
    asm volatile("ld.global.L1::no_allocate.L2::evict_first.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=f"(a[0]), "=f"(a[1]), "=f"(a[2]), "=f"(a[3]), "=f"(a[4]), "=f"(a[5]), "=f"(a[6]), "=f"(a[7])
                 : "l"(p));
}
__device__ __forceinline__ void st8(float* p, const float (&a)[8]) {
    asm volatile("st.global.cs.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "f"(a[0]), "f"(a[1]), "f"(a[2]),
                 "f"(a[3]), "f"(a[4]), "f"(a[5]), "f"(a[6]), "f"(a[7])
                 : "memory");
}
__device__ __forceinline__ uint4 ld16_stream(const void* p) {
    uint4 r;
    asm volatile("ld.global.cs.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}
__device__ __forceinline__ void st16(void* p, uint4 x) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(x.x), "r"(x.y), "r"(x.z), "r"(x.w)
                 : "memory");
}

// eight binary16 values (16 bytes) -> float32 (exact)
__device__ __forceinline__ void h8_to(const uint4& x, float (&a)[8]) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
        a[2 * k] = f.x;
        a[2 * k + 1] = f.y;
    }
}

// ------------------------------------------------------------------------------------------------------------------
// programmatic dependent launch
// ------------------------------------------------------------------------------------------------------------------

// Lets the kernel queued after this one start launching (it still waits for this one before using its results).
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Waits until the kernel queued before this one has completed and its writes are visible (returns at once when this
// kernel was not launched as a programmatic dependent).
__device__ __forceinline__ void wait_prerequisite() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// The gradient factor, read once per thread right before its first update (after the prerequisite has finished).
struct Factor {
    const float* src;
    float value;
    bool ready;
    __device__ __forceinline__ float get() {
        if (!ready) {
            wait_prerequisite();
            value = src ? __ldcg(src) : 1.0f;
            ready = true;
        }
        return value;
    }
};

// A step to skip: the caller asked to skip steps whose norm was not finite (kSkip), and the factor is not > 0 (a
// NaN norm gives a NaN factor, an infinite one a zero factor). Without kSkip the test compiles away.
template <bool kSkip>
__device__ __forceinline__ bool skip_step(float f) { return kSkip && !(f > 0.0f); }

// Asks L2 to fetch `bytes` (a multiple of 16) from `p` (16-byte aligned), without waiting for them.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// In a pack's table (non-decreasing first octets of its tensors): the last j in [j, count) with pre[j] <= q, given
// pre[j] <= q already.
__device__ __forceinline__ int32_t pack_search(const int32_t* __restrict__ pre, int32_t j, int32_t count, int32_t q) {
    int32_t hi = count - 1;
    while (j < hi) {
        const int32_t mid = (j + hi + 1) >> 1;
        if (__ldg(pre + mid) <= q) j = mid;
        else hi = mid - 1;
    }
    return j;
}

// A persistent grid's work queue: q[0] counts the items handed out, q[1] the CTAs that have finished. Each CTA's
// thread 0 takes items one at a time (the next one while the CTA works on the current one); the CTA that finishes
// last resets both counters for the launch that uses this queue next. Launches that may overlap (a programmatic
// dependent starts before its predecessor ends) are given different queues.
__device__ __forceinline__ int32_t queue_take(unsigned int* q) { return (int32_t)atomicAdd(q, 1u); }

__device__ __forceinline__ void queue_finish(unsigned int* q) {
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(q + 1, 1u) == gridDim.x - 1) {
            q[0] = 0u;
            q[1] = 0u;
        }
    }
}

}  // namespace
}  // namespace mica
