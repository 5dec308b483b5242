// ScaleTensors ("Mica 7.7 ...", section "The whole model in one call"): each element of each listed tensor times one
// factor, float32 or binary16 (widened, multiplied, rounded back to nearest-even), one CTA per work item, launched as
// a programmatic dependent of the kernel queued before it.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "plan.h"
#include "stream.cuh"

namespace mica {
namespace {

constexpr int kUnrollScale = 2;  // octets in flight per thread and round in ScaleTensors

// ------------------------------------------------------------------------------------------------------------------
// ScaleTensors
// ------------------------------------------------------------------------------------------------------------------

template <Dtype T>
__device__ __forceinline__ void scale_range(const TensorRec& r, int64_t ob, int64_t oe, int lane, int stride,
                                            float f) {
    constexpr int U = kUnrollScale;
    const int64_t full = r.n / kOct;
    const int64_t vend = r.vec ? (oe < full ? oe : full) : ob;
    for (int64_t o0 = ob + lane; o0 < vend; o0 += (int64_t)stride * U) {
        float X[U][8];
        uint4 H[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t o = o0 + (int64_t)u * stride;
            if (o < vend) {
                if constexpr (T == kF16) H[u] = ld16_stream(reinterpret_cast<const __half*>(r.w) + kOct * o);
                else ld8_stream(r.w + kOct * o, X[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t o = o0 + (int64_t)u * stride;
            if (o < vend) {
                if constexpr (T == kF16) h8_to(H[u], X[u]);
#pragma unroll
                for (int j = 0; j < 8; ++j) X[u][j] = __fmul_rn(X[u][j], f);
                if constexpr (T == kF16) {
                    uint32_t h[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const __half2 p = __floats2half2_rn(X[u][2 * k], X[u][2 * k + 1]);
                        h[k] = *reinterpret_cast<const uint32_t*>(&p);
                    }
                    st16(reinterpret_cast<__half*>(r.w) + kOct * o, make_uint4(h[0], h[1], h[2], h[3]));
                } else {
                    st8(r.w + kOct * o, X[u]);
                }
            }
        }
    }
    // elements not covered by vectors: the partial last octet, or everything when unaligned
    const int64_t eb = (vend > ob ? vend : ob) * kOct;
    const int64_t ee = r.n < oe * kOct ? r.n : oe * kOct;
    for (int64_t i = eb + lane; i < ee; i += stride) {
        if constexpr (T == kF16) {
            __half* p = reinterpret_cast<__half*>(r.w) + i;
            *p = __float2half_rn(__fmul_rn(__half2float(*p), f));
        } else {
            r.w[i] = __fmul_rn(r.w[i], f);
        }
    }
}

template <Dtype T>
__global__ void __launch_bounds__(kThreads) scale_kernel(const TensorRec* __restrict__ recs,
                                                         const WorkItem* __restrict__ items, int32_t num_items,
                                                         int32_t item_octs, float factor,
                                                         const float* __restrict__ d_factor) {
    wait_prerequisite();  // the kernel queued before may still be writing these tensors or the factor
    allow_dependents();   // the kernel queued next may launch (it waits for this one before touching its data)
    const float f = d_factor ? __ldcg(d_factor) : factor;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int32_t it = blockIdx.x; it < num_items; it += gridDim.x) {
        const WorkItem item = items[it];
        if (item.count == 1) {
            const TensorRec r = recs[item.t];
            const int64_t no = (r.n + kOct - 1) / kOct;
            scale_range<T>(r, item.o0, item.o0 + item_octs < no ? item.o0 + item_octs : no, threadIdx.x, kThreads,
                           f);
        } else {
            for (int j = warp; j < item.count; j += kWarps) {
                const TensorRec r = recs[item.t + j];
                scale_range<T>(r, 0, (r.n + kOct - 1) / kOct, lane, 32, f);
            }
        }
    }
}

}  // namespace

int launch_scale(const TensorRec* recs, const WorkItem* items, int32_t num_items, int32_t item_octs, Dtype dt,
                 float factor, const float* d_factor, void* stream) {
    if (num_items <= 0) return (int)cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_items);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];  // a programmatic dependent of the kernel queued before (as the other kernels are)
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = (dt == kF16)
                              ? cudaLaunchKernelEx(&cfg, scale_kernel<kF16>, recs, items, num_items, item_octs, factor,
                                                   d_factor)
                              : cudaLaunchKernelEx(&cfg, scale_kernel<kF32>, recs, items, num_items, item_octs, factor,
                                                   d_factor);
    count_launches(1);
    return (int)(e != cudaSuccess ? e : cudaGetLastError());
}

}  // namespace mica
