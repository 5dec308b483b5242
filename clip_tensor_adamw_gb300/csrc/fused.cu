// ClipGradNorms and AdamWSteps in one cooperative launch ("Mica 7.7 ...", section "Values that stay on the card": the
// norm is measured, decided and applied on the card). Phase 1: each CTA sums the squares of its equal chunk of the
// gradient, asking L2 to keep the lines it loads; the CTAs then meet at one bounded grid-wide wait; every CTA sums
// the partials in the same fixed order, so all hold the same norm and clip factor (CTA 0 writes both to device
// memory); phase 2 is the AdamW update over the work queue, whose gradient reads
// then find the lines phase 1 left in L2 instead of reading them from HBM a second time. While it waits, a CTA has
// already taken its first work item and asked L2 for its data.
//
// The grid is one wave (3 CTAs of 256 threads per SM) launched cooperatively, so every CTA is resident and the wait
// can end. The wait gives up after a bounded number of polls, sets the status word and returns, as the pipeline
// waits of the norm kernels do.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "adam.cuh"
#include "normsum.cuh"
#include "plan.h"
#include "stream.cuh"

namespace mica {
namespace {

// OR-ed by a kernel whose grid-wide wait gave up (its results are not valid); read and cleared by the host.
__device__ unsigned int g_fused_status;
enum : unsigned int { kStatusGridWait = 8u, kStatusGridSelfTest = 16u };
constexpr uint32_t kMaxGridPolls = 1u << 24;  // polls (each followed by a sleep of ~128 ns) before a wait gives up

// The two words of a grid-wide wait, for the self-test (the launches' own live in their list's table).
__device__ unsigned int g_selftest_bar[2];

__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int* p) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Every CTA of the grid waits here until all `nblocks` have arrived. bar[0] counts this round's arrivals and bar[1]
// the rounds completed: the last CTA to arrive clears bar[0] and advances bar[1], which the others poll. A CTA's
// writes before the wait are visible to every CTA after it. Returns false (in every thread of the CTA) if the
// wait gave up after max_polls polls.
__device__ bool grid_wait(unsigned int* bar, unsigned int nblocks, uint32_t max_polls, int* s_ok) {
    __syncthreads();
    if (threadIdx.x == 0) {
        bool ok = true;
        const unsigned int round = ld_acquire_gpu(bar + 1);
        __threadfence();
        if (atomicAdd(bar, 1u) == nblocks - 1) {
            atomicExch(bar, 0u);
            __threadfence();
            atomicAdd(bar + 1, 1u);
        } else {
            for (uint32_t i = 0; ld_acquire_gpu(bar + 1) == round; ++i) {
                if (i >= max_polls) {
                    ok = false;
                    break;
                }
                __nanosleep(128);
            }
        }
        *s_ok = ok ? 1 : 0;
    }
    __syncthreads();
    return *s_ok != 0;
}

struct FusedParams {
    ChunkTable ct;            // the gradient in ct.grid equal chunks, one per CTA (the register-streaming layout)
    double* partials;         // ct.grid entries
    unsigned int* bar;        // the grid-wide wait's two words (zero before the first launch)
    UpdateLaunch u;           // the update's tables and its work queue
    float max_norm, inv_scale;
    float* d_norm;            // may be null
    float* d_factor;
};

template <Dtype G, Dtype M, bool kCoupled, bool kSkip, int kMode>
__global__ void __launch_bounds__(kThreads, 3) clip_adamw_kernel(const __grid_constant__ FusedParams p,
                                                                 StepScalars s) {
    __shared__ StagedSpan sp;
    __shared__ double red[kWarps];
    __shared__ int32_t s_item[2];
    __shared__ int s_ok;
    __shared__ float s_factor;
    const int t = threadIdx.x;

    // phase 1: this CTA's share of the joint norm; the gradient lines stay in L2 for phase 2
    const double mine = direct_chunk_share<G, kMode, true>(p.ct, (int32_t)blockIdx.x, (int32_t)gridDim.x,
                                                           p.inv_scale, sp);
    const double part = block_sum(mine, red);
    if (t == 0) {
        p.partials[blockIdx.x] = part;
        s_item[0] = queue_take(p.u.queue);  // the first work item, so that its data can be on its way meanwhile
    }
    __syncthreads();
    if (s_item[0] < p.u.num_items)
        prefetch_item<G, M>(p.u.recs, p.u.items[p.u.num_items - 1 - s_item[0]], p.u.item_octs);
    if (!grid_wait(p.bar, gridDim.x, kMaxGridPolls, &s_ok)) {
        if (t == 0) atomicOr(&g_fused_status, kStatusGridWait);
        return;
    }

    // the norm and the factor, from every CTA's partial in the same order, so every CTA gets the same bits
    const double S = sum_partials(p.partials, (int32_t)gridDim.x, red);
    if (t == 0) {
        float norm, factor;
        norm_and_factor(S, p.max_norm, p.inv_scale, &norm, &factor);
        s_factor = factor;
        if (blockIdx.x == 0) {
            if (p.d_norm) *p.d_norm = norm;
            *p.d_factor = factor;
        }
    }
    __syncthreads();

    // phase 2: the update
    Factor fac{nullptr, s_factor, true};
    const GroupScalars none{};
    adamw_item_loop<G, M, kCoupled, kSkip, false>(p.u.recs, p.u.items, p.u.num_items, p.u.item_octs, p.u.pack_pre,
                                                  p.u.queue, s, none, fac, s_item);
    queue_finish(p.u.queue);
}

// The grid-wide wait's failure path, on purpose: one CTA waits for a second one that is never launched, gives up
// after `polls` polls and reports it in the status word, as a launch whose CTAs were not all resident would.
__global__ void __launch_bounds__(32) grid_wait_selftest_kernel(uint32_t polls) {
    __shared__ int s_ok;
    if (threadIdx.x == 0) {
        g_selftest_bar[0] = 0u;
        g_selftest_bar[1] = 0u;
        __threadfence();
    }
    if (!grid_wait(g_selftest_bar, 2u, polls, &s_ok) && threadIdx.x == 0) atomicOr(&g_fused_status, kStatusGridSelfTest);
}

template <Dtype G, Dtype M, bool kCoupled, bool kSkip, int kMode>
cudaError_t launch_fused_t(const FusedParams& p, const StepScalars& s, int32_t grid, cudaStream_t st) {
    static const int per_sm = [] {  // CTAs of this instantiation that fit on one SM (found once, thread-safely)
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, clip_adamw_kernel<G, M, kCoupled, kSkip, kMode>,
                                                          kThreads, 0) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        return n;
    }();
    if (per_sm * p.u.sms < grid) return cudaErrorCooperativeLaunchTooLarge;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, clip_adamw_kernel<G, M, kCoupled, kSkip, kMode>, p, s);
}

template <Dtype G, Dtype M, bool kCoupled, bool kSkip>
cudaError_t launch_fused_mode(const FusedParams& p, const StepScalars& s, int32_t grid, cudaStream_t st) {
    // binary16 times a power of two in [2^-102, 2^111]: every product is an exact normal float32
    int ex = 0;
    const bool pow2 = std::frexp(p.inv_scale, &ex) == 0.5f && p.inv_scale >= 0x1p-102f && p.inv_scale <= 0x1p111f;
    if constexpr (G == kF16) {
        if (pow2) return launch_fused_t<G, M, kCoupled, kSkip, kSumHalfPow2>(p, s, grid, st);
        return launch_fused_t<G, M, kCoupled, kSkip, kSumScaled>(p, s, grid, st);
    } else {
        if (p.inv_scale != 1.0f) return launch_fused_t<G, M, kCoupled, kSkip, kSumScaled>(p, s, grid, st);
        return launch_fused_t<G, M, kCoupled, kSkip, kSumUnscaled>(p, s, grid, st);
    }
}

template <Dtype G, Dtype M>
cudaError_t launch_fused_opts(bool coupled, bool skip, const FusedParams& p, const StepScalars& s, int32_t grid,
                              cudaStream_t st) {
    if (skip)
        return coupled ? launch_fused_mode<G, M, true, true>(p, s, grid, st)
                       : launch_fused_mode<G, M, false, true>(p, s, grid, st);
    return coupled ? launch_fused_mode<G, M, true, false>(p, s, grid, st)
                   : launch_fused_mode<G, M, false, false>(p, s, grid, st);
}

template <Dtype G>
cudaError_t launch_fused_m(Dtype mdt, bool coupled, bool skip, const FusedParams& p, const StepScalars& s,
                           int32_t grid, cudaStream_t st) {
    if (mdt == kBF16x2) return launch_fused_opts<G, kBF16x2>(coupled, skip, p, s, grid, st);
    if (mdt == kBF16x2M) return launch_fused_opts<G, kBF16x2M>(coupled, skip, p, s, grid, st);
    return launch_fused_opts<G, kF32>(coupled, skip, p, s, grid, st);
}

}  // namespace

int launch_clip_adamw(const ChunkTable& ct, double* partials, unsigned int* bar, const UpdateLaunch& u, Dtype gdt,
                      Dtype mdt, bool coupled, const StepScalars& s, float max_norm, float inv_scale, float* d_norm,
                      float* d_factor, void* stream) {
    FusedParams p{};
    p.ct = ct;
    p.partials = partials;
    p.bar = bar;
    p.u = u;
    p.max_norm = max_norm;
    p.inv_scale = inv_scale;
    p.d_norm = d_norm;
    p.d_factor = d_factor;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool skip = s.skip_nonfinite != 0;
    if (!u.queue) return (int)cudaErrorInvalidValue;  // the update's items come from the work queue
    const cudaError_t e = (gdt == kF16) ? launch_fused_m<kF16>(mdt, coupled, skip, p, s, ct.grid, st)
                                        : launch_fused_m<kF32>(mdt, coupled, skip, p, s, ct.grid, st);
    if (e == cudaErrorCooperativeLaunchTooLarge) return (int)e;  // nothing was queued: the caller may fall back
    count_launches(1);
    return (int)(e != cudaSuccess ? e : cudaGetLastError());
}

int launch_grid_wait_selftest(uint32_t polls, void* stream) {
    grid_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(polls);
    count_launches(1);
    return (int)cudaGetLastError();
}

int read_fused_status(unsigned int* status) {
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_fused_status, sizeof v);
    if (e != cudaSuccess) return (int)e;
    if (v) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_fused_status, &zero, sizeof zero);
    }
    *status = v;
    return (int)e;
}

}  // namespace mica
