// The multi-tensor AdamW update for sm_103a (and the Adam family's options: coupled L2, skip of a non-finite step,
// parameter groups), over float32, packed BF16 or packed-m / float32-v moments. It streams HBM with no data reuse, so
// it is built for bandwidth: a persistent grid fed by a work queue, 32-byte vector accesses (sm_100's 256-bit loads
// and stores) that coalesce across a warp, evict-first cache hints, L2 prefetch ahead of the loads, and a launch as
// a programmatic dependent of the norm, so that its CTAs are resident and have asked L2 for their first data by the
// time the norm finishes.
//
// Per-element arithmetic follows BendTorch "main.bend", section "Optimizers" (adam.cuh): every float32 operation a
// separate correctly rounded intrinsic, in the order that section gives, so the update is bit-identical to the same
// step on the CPU.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "adam.cuh"
#include "plan.h"
#include "stream.cuh"

namespace mica {
namespace {

// A persistent grid (as many CTAs as fit on the GPU at once) taking the work items one at a time from `queue` (or,
// with no queue, one CTA per item), in reverse order (the norm reads them forwards, so the gradient it read last may
// still be in L2 when this kernel starts). Without kGrouped the scalars are read straight from the kernel's
// parameters; with it each tensor's group picks its own (the parameter array is indexed in place).
template <Dtype G, Dtype M, bool kCoupled, bool kSkip, bool kGrouped>
__global__ void __launch_bounds__(kThreads, 3) adamw_kernel(const TensorRec* __restrict__ recs,
                                                            const WorkItem* __restrict__ items, int32_t num_items,
                                                            int32_t item_octs,
                                                            const int32_t* __restrict__ pack_pre,
                                                            unsigned int* queue, StepScalars s,
                                                            const __grid_constant__ GroupScalars gs,
                                                            const float* __restrict__ d_factor) {
    allow_dependents();  // the next step's norm may launch and set up while this kernel's last CTAs run
    Factor fac{d_factor, 1.0f, false};
    __shared__ int32_t s_item[2];
    const bool persistent = queue != nullptr;  // else one CTA per item: item blockIdx.x
    if (threadIdx.x == 0) s_item[0] = persistent ? queue_take(queue) : (int32_t)blockIdx.x;
    __syncthreads();
    // Until the kernel queued before this one has finished, its writes to these tensors may still be on their way:
    // the CTA only asks L2 for its first item's data (L2 keeps global memory coherent, so a prefetch cannot return
    // stale data to a later load), and every load of w, g, m and v follows the wait.
    if (s_item[0] < num_items) prefetch_item<G, M>(recs, items[num_items - 1 - s_item[0]], item_octs);
    fac.get();
    adamw_item_loop<G, M, kCoupled, kSkip, kGrouped>(recs, items, num_items, item_octs, pack_pre, queue, s, gs, fac,
                                                     s_item);
    if (persistent) queue_finish(queue);
}

// The AdamW launch options: each selects a kernel instantiation, so that the common step compiles without the
// others' tests.
struct AdamwLaunch {
    const WorkItem* items;
    const TensorRec* recs;
    const int32_t* pack_pre;
    unsigned int* queue;
    int32_t num_items, item_octs, sms;
    cudaStream_t st;
    const StepScalars* s;
    const GroupScalars* groups;  // nullptr: one group
    const float* d_factor;
};

template <Dtype G, Dtype M, bool kCoupled, bool kSkip, bool kGrouped>
cudaError_t launch_adamw_t(const AdamwLaunch& a) {
    static const int per_sm = [] {  // CTAs of this instantiation that fit on one SM (found once, thread-safely)
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, adamw_kernel<G, M, kCoupled, kSkip, kGrouped>, kThreads,
                                                          0) != cudaSuccess ||
            n <= 0) {
            cudaGetLastError();
            n = 1;
        }
        return n;
    }();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.queue ? persistent_grid(a.num_items, per_sm, a.sms) : a.num_items);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = a.st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const GroupScalars gs = a.groups ? *a.groups : GroupScalars{};
    return cudaLaunchKernelEx(&cfg, adamw_kernel<G, M, kCoupled, kSkip, kGrouped>, a.recs, a.items, a.num_items,
                              a.item_octs, a.pack_pre, a.queue, *a.s, gs, a.d_factor);
}

template <Dtype G, Dtype M, bool kCoupled, bool kSkip>
cudaError_t launch_adamw_g(const AdamwLaunch& a) {
    return a.groups ? launch_adamw_t<G, M, kCoupled, kSkip, true>(a) : launch_adamw_t<G, M, kCoupled, kSkip, false>(a);
}

template <Dtype G, Dtype M>
cudaError_t launch_adamw_c(bool coupled, const AdamwLaunch& a) {
    if (a.s->skip_nonfinite)
        return coupled ? launch_adamw_g<G, M, true, true>(a) : launch_adamw_g<G, M, false, true>(a);
    return coupled ? launch_adamw_g<G, M, true, false>(a) : launch_adamw_g<G, M, false, false>(a);
}

template <Dtype G>
cudaError_t launch_adamw_m(Dtype mdt, bool coupled, const AdamwLaunch& a) {
    if (mdt == kBF16x2) return launch_adamw_c<G, kBF16x2>(coupled, a);
    if (mdt == kBF16x2M) return launch_adamw_c<G, kBF16x2M>(coupled, a);
    return launch_adamw_c<G, kF32>(coupled, a);
}

}  // namespace

int launch_adamw(const UpdateLaunch& u, Dtype gdt, Dtype mdt, bool coupled, const StepScalars& s,
                 const GroupScalars* groups, const float* d_factor, void* stream) {
    if (u.num_items <= 0) return (int)cudaSuccess;
    const AdamwLaunch a{u.items, u.recs, u.pack_pre, u.queue, u.num_items, u.item_octs, u.sms,
                        static_cast<cudaStream_t>(stream), &s, groups, d_factor};
    const cudaError_t e = (gdt == kF16) ? launch_adamw_m<kF16>(mdt, coupled, a) : launch_adamw_m<kF32>(mdt, coupled, a);
    count_launches(1);
    return (int)(e != cudaSuccess ? e : cudaGetLastError());
}

// Both norm kernels are launched as programmatic dependents of the kernel queued before them: they may start and
// set up while it finishes, and wait for it (griddepcontrol.wait) before reading any gradient.
}  // namespace mica
