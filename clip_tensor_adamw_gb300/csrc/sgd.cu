// SGD and SGD with momentum over a tensor list in one launch, with the clip factor folded in: BendTorch "main.bend",
// section "Optimizers", whose two plain optimizers are w + (-lr) g and, with a momentum buffer b, b = b mu + g then
// w + (-lr) b (PyTorch's SGD without weight decay, dampening or Nesterov). The gradient entering either is
// gh = g * f, f the factor of the joint-norm clip (and of the loss-scale unscale), read from device memory.
//
// Same work items and access scheme as the AdamW kernel: a persistent grid whose CTAs take the items (a slice of a
// large tensor, or a pack of small tensors whose octets the threads share out) one at a time from a queue, 32-byte
// streaming loads and stores, L2 prefetch two rounds ahead on the slices, and a programmatic-dependent launch whose
// CTAs only ask L2 for their first item before the norm has finished. Every float operation is a separate correctly
// rounded intrinsic, in the page's order, so the result is bit-identical to the same step on the CPU.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "plan.h"
#include "stream.cuh"

namespace mica {
namespace {

// One octet in registers: w, the gradient g (already widened to float32) and, with kMomentum, the buffer b.
template <bool kMomentum>
__device__ __forceinline__ void sgd8(float (&w)[8], const float (&g)[8], float (&b)[8], const SgdScalars& s,
                                     float f) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float gh = __fmul_rn(g[j], f);
        if constexpr (kMomentum) {
            b[j] = __fadd_rn(__fmul_rn(b[j], s.mu), gh);
            w[j] = __fadd_rn(w[j], __fmul_rn(s.neg_lr, b[j]));
        } else {
            w[j] = __fadd_rn(w[j], __fmul_rn(s.neg_lr, gh));
        }
    }
}

// One octet element by element (an unaligned tensor, or a tensor's last, partial octet): elements past n are
// neither read nor written.
template <Dtype G, bool kMomentum, bool kSkip>
__device__ __noinline__ void sgd_oct_elements(const TensorRec& r, int64_t o, const SgdScalars& s, Factor& fac) {
    const int64_t i0 = o * kOct;
    const int64_t left = r.n - i0;
    const int cnt = left < kOct ? (int)left : kOct;
    float w[8], g[8], b[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        w[j] = g[j] = b[j] = 0.f;
        if (j < cnt) {
            w[j] = r.w[i0 + j];
            g[j] = (G == kF16) ? __half2float(static_cast<const __half*>(r.g)[i0 + j])
                               : static_cast<const float*>(r.g)[i0 + j];
            if constexpr (kMomentum) b[j] = static_cast<const float*>(r.m)[i0 + j];
        }
    }
    const float f = fac.get();
    const bool skip = skip_step<kSkip>(f);
    if (!skip) sgd8<kMomentum>(w, g, b, s, f);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if (j < cnt) {
            if (!skip) {
                r.w[i0 + j] = w[j];
                if constexpr (kMomentum) static_cast<float*>(r.m)[i0 + j] = b[j];
            }
            if (s.zero_grad) {
                if (G == kF16) static_cast<__half*>(r.g)[i0 + j] = __ushort_as_half(0);
                else static_cast<float*>(r.g)[i0 + j] = 0.f;
            }
        }
    }
}

// The streams of octets [a, b) of tensor r into L2 (whole octets of an aligned tensor).
template <Dtype G, bool kMomentum>
__device__ __forceinline__ void sgd_prefetch(const TensorRec& r, int64_t a, int64_t b) {
    constexpr int kGb = (G == kF16) ? 16 : 32;
    const uint32_t n = (uint32_t)(b - a);
    prefetch_l2(reinterpret_cast<const char*>(r.w) + a * 32, n * 32);
    prefetch_l2(static_cast<const char*>(r.g) + a * kGb, n * kGb);
    if constexpr (kMomentum) prefetch_l2(static_cast<const char*>(r.m) + a * 32, n * 32);
}

// One whole octet of a tensor whose bases are aligned for the vectors.
template <Dtype G, bool kMomentum, bool kSkip>
__device__ __forceinline__ void sgd_vec_octet(const TensorRec& r, int64_t o, const SgdScalars& s, Factor& fac) {
    float w[8], g[8], b[8];
    uint4 gh;
    ld8_stream(r.w + kOct * o, w);
    if constexpr (G == kF16) gh = ld16_stream(static_cast<const __half*>(r.g) + kOct * o);
    else ld8_stream(static_cast<const float*>(r.g) + kOct * o, g);
    if constexpr (kMomentum) ld8_stream(static_cast<const float*>(r.m) + kOct * o, b);
    const float f = fac.get();
    if (!skip_step<kSkip>(f)) {
        if constexpr (G == kF16) h8_to(gh, g);
        sgd8<kMomentum>(w, g, b, s, f);
        st8(r.w + kOct * o, w);
        if constexpr (kMomentum) st8(static_cast<float*>(r.m) + kOct * o, b);
    }
    if (s.zero_grad) {
        if constexpr (G == kF16) {
            st16(static_cast<__half*>(r.g) + kOct * o, make_uint4(0u, 0u, 0u, 0u));
        } else {
            const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            st8(static_cast<float*>(r.g) + kOct * o, z);
        }
    }
}

// Octets [ob, oe) of one tensor: octet ob + lane first, then every `stride`-th; with `prefetch` (a whole CTA on one
// slice) thread 0 asks L2 for the rounds one and two ahead.
template <Dtype G, bool kMomentum, bool kSkip>
__device__ __forceinline__ void sgd_range(const TensorRec& r, int64_t ob, int64_t oe, int lane, int stride,
                                          const SgdScalars& s, Factor& fac, bool prefetch = false) {
    const int64_t full = r.n / kOct;
    if (r.vec) {
        const int64_t vend = oe < full ? oe : full;
        if (prefetch && lane == 0 && ob + stride < vend)
            sgd_prefetch<G, kMomentum>(r, ob + stride, ob + 2 * stride < vend ? ob + 2 * stride : vend);
        for (int64_t o = ob + lane; o < vend; o += stride) {
            if (prefetch && lane == 0 && o + 2 * stride < vend)
                sgd_prefetch<G, kMomentum>(r, o + 2 * stride, o + 3 * stride < vend ? o + 3 * stride : vend);
            sgd_vec_octet<G, kMomentum, kSkip>(r, o, s, fac);
        }
        if (full < oe && full >= ob && lane == (int)((full - ob) % stride))
            sgd_oct_elements<G, kMomentum, kSkip>(r, full, s, fac);
    } else {
        for (int64_t o = ob + lane; o < oe; o += stride) sgd_oct_elements<G, kMomentum, kSkip>(r, o, s, fac);
    }
}

// A pack of small tensors, its octets spread over the CTA's threads, whole octets first (as the AdamW kernel's
// packs).
template <Dtype G, bool kMomentum, bool kSkip>
__device__ __forceinline__ void sgd_pack(const TensorRec* __restrict__ recs, const WorkItem& item,
                                         const int32_t* __restrict__ pack_pre, const SgdScalars& s, Factor& fac) {
    const int32_t* pre_w = pack_pre + item.o0;
    const int32_t* pre_e = pre_w + item.count + 1;
    for (int32_t i = threadIdx.x; i < item.count; i += kThreads) {  // the pack into L2 first, one tensor a thread
        const TensorRec r = recs[item.t + i];
        if (r.vec && r.n >= kOct) sgd_prefetch<G, kMomentum>(r, 0, r.n / kOct);
    }
    const int32_t total_w = __ldg(pre_w + item.count);
    const int32_t total = total_w + __ldg(pre_e + item.count);
    int32_t jw = 0, je = 0;
    for (int32_t q = threadIdx.x; q < total; q += kThreads) {
        if (q < total_w) {
            jw = pack_search(pre_w, jw, item.count, q);
            const TensorRec r = recs[item.t + jw];
            sgd_vec_octet<G, kMomentum, kSkip>(r, q - __ldg(pre_w + jw), s, fac);
        } else {
            const int32_t qe = q - total_w;
            je = pack_search(pre_e, je, item.count, qe);
            const TensorRec r = recs[item.t + je];
            sgd_oct_elements<G, kMomentum, kSkip>(r, (r.vec ? r.n / kOct : 0) + (qe - __ldg(pre_e + je)), s, fac);
        }
    }
}

// L2 prefetch of one item's whole octets: the slice's, or every tensor of the pack (one tensor a thread).
template <Dtype G, bool kMomentum>
__device__ __forceinline__ void sgd_prefetch_item(const TensorRec* __restrict__ recs, const WorkItem& item,
                                                  int32_t item_octs) {
    if (item.count == 1) {
        if (threadIdx.x == 0) {
            const TensorRec r = recs[item.t];
            const int64_t full = r.n / kOct;
            const int64_t oe = item.o0 + item_octs < full ? item.o0 + item_octs : full;
            if (r.vec && oe > item.o0) sgd_prefetch<G, kMomentum>(r, item.o0, oe);
        }
    } else {
        for (int32_t i = threadIdx.x; i < item.count; i += kThreads) {
            const TensorRec r = recs[item.t + i];
            if (r.vec && r.n >= kOct) sgd_prefetch<G, kMomentum>(r, 0, r.n / kOct);
        }
    }
}

// A persistent grid taking the items from `queue` (or, with no queue, one CTA per item), as the AdamW kernel does.
template <Dtype G, bool kMomentum, bool kSkip>
__global__ void __launch_bounds__(kThreads, 3) sgd_kernel(const TensorRec* __restrict__ recs,
                                                          const WorkItem* __restrict__ items, int32_t num_items,
                                                          int32_t item_octs, const int32_t* __restrict__ pack_pre,
                                                          unsigned int* queue, SgdScalars s,
                                                          const float* __restrict__ d_factor) {
    allow_dependents();
    Factor fac{d_factor, 1.0f, false};
    __shared__ int32_t s_item[2];
    const bool persistent = queue != nullptr;  // else one CTA per item: item blockIdx.x
    if (threadIdx.x == 0) s_item[0] = persistent ? queue_take(queue) : (int32_t)blockIdx.x;
    __syncthreads();
    // only an L2 prefetch before the wait for the kernel queued before (as in the AdamW kernel)
    if (s_item[0] < num_items) sgd_prefetch_item<G, kMomentum>(recs, items[num_items - 1 - s_item[0]], item_octs);
    fac.get();
    int32_t cur = 0;
    for (int32_t k = s_item[0]; k < num_items; k = s_item[cur]) {
        if (threadIdx.x == 0) s_item[cur ^ 1] = persistent ? queue_take(queue) : num_items;
        const WorkItem item = items[num_items - 1 - k];
        if (item.count == 1) {
            const TensorRec r = recs[item.t];
            const int64_t no = (r.n + kOct - 1) / kOct;
            const int64_t oe = item.o0 + item_octs < no ? item.o0 + item_octs : no;
            sgd_range<G, kMomentum, kSkip>(r, item.o0, oe, threadIdx.x, kThreads, s, fac, true);
        } else {
            sgd_pack<G, kMomentum, kSkip>(recs, item, pack_pre, s, fac);
        }
        __syncthreads();
        cur ^= 1;
    }
    if (persistent) queue_finish(queue);
}

template <Dtype G, bool kMomentum, bool kSkip>
cudaError_t launch_sgd_t(const UpdateLaunch& u, const SgdScalars& s, const float* d_factor, cudaStream_t st) {
    static const int per_sm = [] {  // CTAs of this instantiation that fit on one SM (found once, thread-safely)
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, sgd_kernel<G, kMomentum, kSkip>, kThreads, 0) !=
                cudaSuccess ||
            n <= 0) {
            cudaGetLastError();
            n = 1;
        }
        return n;
    }();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(u.queue ? persistent_grid(u.num_items, per_sm, u.sms) : u.num_items);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, sgd_kernel<G, kMomentum, kSkip>, u.recs, u.items, u.num_items, u.item_octs,
                              u.pack_pre, u.queue, s, d_factor);
}

template <Dtype G>
cudaError_t launch_sgd_g(const UpdateLaunch& u, bool momentum, bool skip, const SgdScalars& s, const float* d_factor,
                         cudaStream_t st) {
    if (momentum)
        return skip ? launch_sgd_t<G, true, true>(u, s, d_factor, st)
                    : launch_sgd_t<G, true, false>(u, s, d_factor, st);
    return skip ? launch_sgd_t<G, false, true>(u, s, d_factor, st) : launch_sgd_t<G, false, false>(u, s, d_factor, st);
}

}  // namespace

int launch_sgd(const UpdateLaunch& u, Dtype gdt, bool momentum, bool skip, const SgdScalars& s,
               const float* d_factor, void* stream) {
    if (u.num_items <= 0) return (int)cudaSuccess;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const cudaError_t e = (gdt == kF16) ? launch_sgd_g<kF16>(u, momentum, skip, s, d_factor, st)
                                        : launch_sgd_g<kF32>(u, momentum, skip, s, d_factor, st);
    count_launches(1);
    return (int)(e != cudaSuccess ? e : cudaGetLastError());
}

}  // namespace mica
