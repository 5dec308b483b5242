// The joint L2 norm of a gradient list and its clip factor for sm_103a ("Mica 7.7 ...", section "The whole model in
// one call": ClipGradNorms), in one launch: equal contiguous chunks of the list's octets per CTA (a TMA pipeline for
// lists of large tensors, register streaming for lists of small ones), squares summed exactly to about twice
// float32's precision, and a fixed-order finalize by the CTA that finishes last. Also the device status word of the
// bounded pipeline waits, and the self-test of their failure path.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "normsum.cuh"
#include "plan.h"
#include "stream.cuh"

namespace mica {
namespace {

// The joint norm for lists of many small tensors: CTA b sums its equal contiguous chunk (direct_chunk_share); the
// rest is as in norm_tma_kernel. kKeepL2: the gradient's loads ask L2 to keep the lines (see launch_norm).
template <Dtype G, int kMode, bool kKeepL2>
__global__ void __launch_bounds__(kThreads, kNormDirectCtasPerSm) norm_direct_kernel(ChunkTable ct, float inv_scale,
                                                                        double* __restrict__ partials,
                                                                        unsigned int* ticket, float max_norm,
                                                                        float* d_norm, float* d_factor,
                                                                        double* d_sumsq) {
    __shared__ double red[kWarps];
    __shared__ int last;
    __shared__ StagedSpan sp;
    const int t = threadIdx.x;
    wait_prerequisite();  // the kernel queued before may still be writing the gradients (zero_grad)
    allow_dependents();   // the kernel queued next may launch from here (as in the TMA kernel)
    const double mine = direct_chunk_share<G, kMode, kKeepL2>(ct, (int32_t)blockIdx.x, ct.grid, inv_scale, sp);

    const double part = block_sum(mine, red);
    if (t == 0) {
        partials[blockIdx.x] = part;
        __threadfence();  // the partial is visible before the ticket says so
        last = (atomicAdd(ticket, 1u) == (unsigned int)(ct.grid - 1));
    }
    __syncthreads();
    if (last) {  // every other CTA's partial is written: sum them all, in order
        __threadfence();
        finalize_norm(partials, ct.grid, max_norm, inv_scale, d_norm, d_factor, d_sumsq, red);
        if (t == 0) *ticket = 0u;  // ready for the next launch on this list
    }
}

// ------------------------------------------------------------------------------------------------------------------
// TMA bulk copies and mbarriers
// ------------------------------------------------------------------------------------------------------------------

// Set (OR-ed) by a kernel whose pipeline wait gave up; read and cleared by the host (read_device_status).
__device__ unsigned int g_mica_status;

constexpr uint32_t kMaxPolls = 1u << 22;  // try_wait rounds before a wait gives up (each round may suspend a while)

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Waits until the barrier's phase of parity `parity` has completed; false if it has not after kMaxPolls rounds.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t max_polls = kMaxPolls) {
    const uint32_t addr = smem_u32(bar);
    for (uint32_t i = 0; i < max_polls; ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(addr), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}
// `bytes` (a multiple of 16) from global to shared memory, both 16-byte aligned, completing on `bar`.
__device__ __forceinline__ void bulk_copy_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(smem_dst)),
                 "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}
// The same with an L2 cache policy (an evict-last policy from l2_keep_policy keeps the lines for a later reader).
__device__ __forceinline__ void bulk_copy_g2s_hint(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar,
                                                   uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(smem_u32(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// ------------------------------------------------------------------------------------------------------------------
// the joint norm: a TMA pipeline over equal contiguous chunks
// ------------------------------------------------------------------------------------------------------------------

// Each CTA streams its chunk of the list's octets through kNormStages shared-memory stages of 512 octets. One
// producer warp (its lane 0) walks the chunk and, per stage, issues one bulk copy per run of whole octets of an
// aligned tensor (a stage may cross tensor boundaries), completing on the stage's `full` barrier; the 8 consumer
// warps wait on it, thread t takes the stage's octets t and t + 256 (from shared memory, or element by element from
// global memory for a tensor's partial last octet or an unaligned tensor), then each warp arrives on the stage's
// `empty` barrier so the producer may refill it. The bytes in flight (up to 3 stages x 16 KB per CTA, 3 CTAs per
// SM) cost shared memory, not registers; two octets per thread and stage halve the per-stage bookkeeping. Three
// stages measured best on GB300 in the whole step (GPT-2 small 0.5929 ms against 0.5978 with four and 0.5949 with
// two; packed moments 0.4541 against 0.4592 and 0.4557), though GPT-2 XL's step is 0.2% slower than with four.
constexpr int kNormStages = 3;
constexpr int kNormStageOcts = 2 * kThreads;
constexpr int kNormThreads = kThreads + 32;

template <Dtype G>
__host__ __device__ constexpr int norm_stage_bytes() { return kNormStageOcts * ((G == kF16) ? 16 : 32); }

template <Dtype G>
size_t norm_smem_bytes() { return (size_t)kNormStages * norm_stage_bytes<G>(); }

enum : unsigned int { kStatusNormProducer = 1u, kStatusNormConsumer = 2u, kStatusSelfTest = 4u };

// The bounded wait's failure path, on purpose: one thread waits `polls` rounds on a barrier that nothing arrives at,
// gives up and reports it in the status word, as a pipeline kernel whose copies never landed would.
__global__ void __launch_bounds__(32) wait_selftest_kernel(uint32_t polls) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
    }
    __syncwarp();
    if (threadIdx.x == 0 && !mbar_wait(&bar, 0, polls)) atomicOr(&g_mica_status, kStatusSelfTest);
}

template <Dtype G, int kMode, bool kKeepL2>
__global__ void __launch_bounds__(kNormThreads, kNormTmaCtasPerSm) norm_tma_kernel(ChunkTable ct, float inv_scale,
                                                                            double* __restrict__ partials,
                                                                            unsigned int* ticket, float max_norm,
                                                                            float* d_norm, float* d_factor, double* d_sumsq) {
    constexpr int S = kNormStages;
    constexpr int kOctBytes = (G == kF16) ? 16 : 32;
    constexpr int kStageBytes = norm_stage_bytes<G>();
    extern __shared__ __align__(128) unsigned char stages[];
    __shared__ __align__(8) uint64_t full[S];
    __shared__ __align__(8) uint64_t empty[S];
    __shared__ double red[kWarps + 1];
    __shared__ int last;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int64_t c0 = ct.total_octs * blockIdx.x / ct.grid;
    const int64_t c1 = ct.total_octs * (blockIdx.x + 1) / ct.grid;
    const int32_t k0 = ct.first[blockIdx.x];
    const int64_t nstage = (c1 - c0 + kNormStageOcts - 1) / kNormStageOcts;
    if (t == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);          // the producer's arrive (with the stage's byte count)
            mbar_init(&empty[s], kWarps);    // one arrive per consumer warp
        }
        mbar_fence_init();
    }
    __syncthreads();
    wait_prerequisite();  // the kernel queued before may still be writing the gradients (zero_grad)
    // The kernel queued next (the update) may launch from here, once every kernel before the norm has finished: so
    // at most the norm and the update are in flight at once, and the update's early CTAs do not take room on the SMs
    // from a kernel that is still running.
    allow_dependents();

    double mine = 0.0;
    if (warp == kWarps) {
        // ---- producer ----
        if (lane == 0) {
            const uint64_t keep = kKeepL2 ? l2_keep_policy() : 0;
            Cursor pc;
            pc.init(ct, k0);
            bool ok = true;
            int64_t i = 0;
            int slot = 0;
            uint32_t round = 0;  // how many times the ring has wrapped
            for (; i < nstage; ++i) {
                if (round > 0 && !mbar_wait(&empty[slot], (round - 1) & 1u)) {
                    ok = false;
                    break;
                }
                const int64_t a = c0 + i * kNormStageOcts;
                const int64_t b = a + kNormStageOcts < c1 ? a + kNormStageOcts : c1;
                unsigned char* stage = stages + (size_t)slot * kStageBytes;
                // the runs of whole octets of aligned tensors in [a, b): counted first, then copied
                for (int pass = 0; pass < 2; ++pass) {
                    Cursor c = pc;
                    uint32_t bytes = 0;
                    for (int64_t o = a; o < b;) {
                        c.advance(ct, o);
                        const int64_t seg_end = b < c.hi ? b : c.hi;
                        const int64_t whole_end = c.lo + c.full < seg_end ? c.lo + c.full : seg_end;
                        if (c.vec && whole_end > o) {
                            const uint32_t nb = (uint32_t)(whole_end - o) * kOctBytes;
                            if (pass == 1)
                                if constexpr (kKeepL2)
                                    bulk_copy_g2s_hint(stage + (o - a) * kOctBytes, c.base + (o - c.lo) * kOctBytes,
                                                       nb, &full[slot], keep);
                                else
                                    bulk_copy_g2s(stage + (o - a) * kOctBytes, c.base + (o - c.lo) * kOctBytes, nb,
                                                  &full[slot]);
                            bytes += nb;
                        }
                        o = seg_end;
                    }
                    if (pass == 0) {
                        mbar_arrive_expect_tx(&full[slot], bytes);
                    } else {
                        pc = c;
                    }
                }
                if (++slot == S) {
                    slot = 0;
                    ++round;
                }
            }
            // every copy this CTA issued has landed before it may exit: wait for each slot's last use
            const int64_t from = i > S ? i - S : 0;
            for (int64_t j = from; j < i; ++j) mbar_wait(&full[j % S], (uint32_t)((j / S) & 1));
            if (!ok) atomicOr(&g_mica_status, kStatusNormProducer);
        }
    } else {
        // ---- consumers ----
        SumSq acc{{0.f, 0.f}, {0.f, 0.f}, 0.f};
        Cursor cc;
        cc.init(ct, k0);
        bool ok = true;
        int slot = 0;
        uint32_t phase = 0;
        // octet o of the list, at position pos of the current stage
        auto read_octet = [&](int64_t o, int pos, float (&x)[8]) {
            if (o < c1) {
                cc.advance(ct, o);
                const int64_t local = o - cc.lo;
                if (cc.vec && local < cc.full) {
                    const unsigned char* src = stages + (size_t)slot * kStageBytes + (size_t)pos * kOctBytes;
                    if constexpr (G == kF16) {
                        h8_to(*reinterpret_cast<const uint4*>(src), x);
                    } else {
                        // the octet's two halves, lanes whose bit 2 is set reading the upper half first: each
                        // 16-byte read of the warp then covers all 32 banks four times, not half of them eight
                        const int h = (lane >> 2) & 1;
                        const float4 p = *reinterpret_cast<const float4*>(src + 16 * h);
                        const float4 q = *reinterpret_cast<const float4*>(src + 16 * (h ^ 1));
                        const float4 lo4 = h ? q : p, hi4 = h ? p : q;
                        x[0] = lo4.x; x[1] = lo4.y; x[2] = lo4.z; x[3] = lo4.w;
                        x[4] = hi4.x; x[5] = hi4.y; x[6] = hi4.z; x[7] = hi4.w;
                    }
                } else {  // a tensor's partial last octet, or an unaligned tensor
                    load_elements<G>(cc, local, x);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) x[j] = 0.0f;
            }
        };
        for (int64_t i = 0; i < nstage; ++i) {
            if (!mbar_wait(&full[slot], phase)) {
                ok = false;
                break;
            }
            const int64_t a = c0 + i * kNormStageOcts;
            float x0[8], x1[8];
            read_octet(a + t, t, x0);
            read_octet(a + t + kThreads, t + kThreads, x1);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);  // this warp is done reading the stage
            acc.add8<kMode>(x0, inv_scale);
            acc.add8<kMode>(x1, inv_scale);
            if (++slot == S) {
                slot = 0;
                phase ^= 1u;
            }
        }
        mine = share_total<G, kMode>(acc, ct, k0, c0, c1, inv_scale);
        if (!ok) atomicOr(&g_mica_status, kStatusNormConsumer);
    }

    const double part = block_sum(mine, red);
    if (t == 0) {
        partials[blockIdx.x] = part;
        __threadfence();  // the partial is visible before the ticket says so
        last = (atomicAdd(ticket, 1u) == (unsigned int)(ct.grid - 1));
    }
    __syncthreads();
    if (last) {  // every other CTA's partial is written: sum them all, in order
        __threadfence();
        finalize_norm(partials, ct.grid, max_norm, inv_scale, d_norm, d_factor, d_sumsq, red);
        if (t == 0) *ticket = 0u;  // ready for the next launch on this list
    }
}

}  // namespace

template <Dtype G, int kMode, bool kKeepL2>
cudaError_t launch_norm_t(const ChunkTable& ct, cudaStream_t st, float inv_scale, double* partials,
                          unsigned int* ticket, float max_norm, float* d_norm, float* d_factor, double* d_sumsq) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ct.grid > 0 ? ct.grid : 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (ct.direct) {
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = 0;
        return cudaLaunchKernelEx(&cfg, norm_direct_kernel<G, kMode, kKeepL2>, ct, inv_scale, partials, ticket,
                                  max_norm, d_norm, d_factor, d_sumsq);
    }
    const size_t smem = norm_smem_bytes<G>();
    cudaError_t e = cudaFuncSetAttribute(norm_tma_kernel<G, kMode, kKeepL2>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cfg.blockDim = dim3(kNormThreads);
    cfg.dynamicSmemBytes = smem;
    return cudaLaunchKernelEx(&cfg, norm_tma_kernel<G, kMode, kKeepL2>, ct, inv_scale, partials, ticket, max_norm,
                              d_norm, d_factor, d_sumsq);
}

template <Dtype G, int kMode>
cudaError_t launch_norm_k(bool keep_l2, const ChunkTable& ct, cudaStream_t st, float inv_scale, double* partials,
                          unsigned int* ticket, float max_norm, float* d_norm, float* d_factor, double* d_sumsq) {
    return keep_l2 ? launch_norm_t<G, kMode, true>(ct, st, inv_scale, partials, ticket, max_norm, d_norm, d_factor,
                                                   d_sumsq)
                   : launch_norm_t<G, kMode, false>(ct, st, inv_scale, partials, ticket, max_norm, d_norm, d_factor,
                                                    d_sumsq);
}

// The norm and factor of rank-ordered partial square sums: one thread adds parts[0], parts[1], ... in double.
static __global__ void __launch_bounds__(32) factor_from_sumsq_kernel(const double* __restrict__ parts, int32_t count,
                                                               float max_norm, float inv_scale, float* d_norm,
                                                               float* d_factor) {
    if (threadIdx.x != 0) return;
    double S = 0.0;
    for (int32_t i = 0; i < count; ++i) S += __ldcg(parts + i);
    float norm, factor;
    norm_and_factor(S, max_norm, inv_scale, &norm, &factor);
    if (d_norm) *d_norm = norm;
    *d_factor = factor;
}

int launch_norm(const ChunkTable& ct, Dtype gdt, float inv_scale, double* partials, unsigned int* ticket,
                float max_norm, float* d_norm, float* d_factor, double* d_sumsq, bool keep_l2, void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool scaled = inv_scale != 1.0f;  // an unscaled list skips the multiply (x * 1 is x)
    // binary16 times a power of two in [2^-102, 2^111]: every product is an exact normal float32
    int ex = 0;
    const bool pow2 = std::frexp(inv_scale, &ex) == 0.5f && inv_scale >= 0x1p-102f && inv_scale <= 0x1p111f;
    cudaError_t e;
    if (gdt == kF16 && pow2)
        e = launch_norm_k<kF16, kSumHalfPow2>(keep_l2, ct, st, inv_scale, partials, ticket, max_norm, d_norm,
                                              d_factor, d_sumsq);
    else if (gdt == kF16)
        e = launch_norm_k<kF16, kSumScaled>(keep_l2, ct, st, inv_scale, partials, ticket, max_norm, d_norm, d_factor,
                                            d_sumsq);
    else if (scaled)
        e = launch_norm_k<kF32, kSumScaled>(keep_l2, ct, st, inv_scale, partials, ticket, max_norm, d_norm, d_factor,
                                            d_sumsq);
    else
        e = launch_norm_k<kF32, kSumUnscaled>(keep_l2, ct, st, inv_scale, partials, ticket, max_norm, d_norm,
                                              d_factor, d_sumsq);
    count_launches(1);
    return (int)e;
}

int launch_factor_from_sumsq(const double* parts, int32_t count, float max_norm, float inv_scale, float* d_norm,
                             float* d_factor, void* stream) {
    factor_from_sumsq_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(parts, count, max_norm, inv_scale,
                                                                             d_norm, d_factor);
    count_launches(1);
    return (int)cudaGetLastError();
}

int launch_wait_selftest(uint32_t polls, void* stream) {
    wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(polls);
    count_launches(1);
    return (int)cudaGetLastError();
}

int read_device_status(unsigned int* status) {
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_mica_status, sizeof v);
    if (e != cudaSuccess) return (int)e;
    if (v) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_mica_status, &zero, sizeof zero);
    }
    *status = v;
    return (int)e;
}

}  // namespace mica
