// The joint L2 norm of a gradient list and its clip factor for sm_103a ("Mica 7.7 ...", section "The whole model in
// one call": ClipGradNorms), in one launch: equal contiguous chunks of the list's octets per CTA (a TMA pipeline for
// lists of large tensors, register streaming for lists of small ones), squares summed exactly to about twice
// float32's precision, and a fixed-order finalize by the CTA that finishes last. Also the device status word of the
// bounded pipeline waits, and the self-test of their failure path.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "plan.h"
#include "stream.cuh"

namespace mica {
namespace {

// ------------------------------------------------------------------------------------------------------------------
// the joint norm: per-item partial square sums, finalized by the CTA that finishes last
// ------------------------------------------------------------------------------------------------------------------

// x^2 summed to about twice float32's precision: each square is split exactly into p + e (p = x*x rounded, e its
// rounding error from an FMA) and p is added to the running hi by Knuth's two-sum, whose exact error joins e in lo.
// The two halves of a float2 are two independent (hi, lo) chains (even and odd elements), advanced together by
// sm_100's packed float32x2 instructions, each half rounded exactly as the scalar operation would be. This is exact
// up to the float32 rounding of lo while every |x| lies in [2^-50, 2^50): squares then stay below 2^100 (no
// overflow) and every e is a normal float32. Elements below 2^-50 in a share whose largest |x| is at least 2^-50
// lose at most 2^-150 each, a relative 2^-44 of that share's sum; any other share (a value at or above 2^50, an
// infinity or NaN, or nothing but values below 2^-50) is summed again in double by the caller.
__device__ __forceinline__ float2 neg2(float2 v) { return make_float2(-v.x, -v.y); }

// How a kernel sums the squares of x = g * inv_scale: kSumUnscaled (inv_scale is 1), kSumScaled (each x formed in
// float32), or kSumHalfPow2 (binary16 g and a power-of-two inv_scale for which every g * inv_scale is an exact
// normal float32: g^2 then has at most 22 significant bits and lies in [2^-48, 2^32], so each square is exact in
// float32 and needs neither the error term nor the range check; the sum of g^2 is scaled by inv_scale^2 at the end,
// exactly).
enum : int { kSumUnscaled = 0, kSumScaled = 1, kSumHalfPow2 = 2 };

struct SumSq {
    float2 hi, lo;
    float mx;  // the largest |x| seen (NaNs are ignored here and show up in hi instead)
    __device__ __forceinline__ void add2(float2 x) {
        mx = fmaxf(mx, fmaxf(fabsf(x.x), fabsf(x.y)));
        const float2 p = __fmul2_rn(x, x);
        const float2 e = __ffma2_rn(x, x, neg2(p));
        const float2 s = __fadd2_rn(hi, p);
        const float2 bp = __fadd2_rn(s, neg2(hi));
        const float2 err = __fadd2_rn(__fadd2_rn(hi, neg2(__fadd2_rn(s, neg2(bp)))), __fadd2_rn(p, neg2(bp)));
        hi = s;
        lo = __fadd2_rn(lo, __fadd2_rn(err, e));
    }
    // the same for a pair whose squares are exact in float32 (no rounding error term) and whose |x| need no check
    __device__ __forceinline__ void add2_exact_squares(float2 x) {
        const float2 p = __fmul2_rn(x, x);
        const float2 s = __fadd2_rn(hi, p);
        const float2 bp = __fadd2_rn(s, neg2(hi));
        const float2 err = __fadd2_rn(__fadd2_rn(hi, neg2(__fadd2_rn(s, neg2(bp)))), __fadd2_rn(p, neg2(bp)));
        hi = s;
        lo = __fadd2_rn(lo, err);
    }
    template <int kMode>
    __device__ __forceinline__ void add8(const float (&x)[8], float inv_scale) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float2 v = make_float2(x[2 * j], x[2 * j + 1]);
            if constexpr (kMode == kSumScaled) v = __fmul2_rn(v, make_float2(inv_scale, inv_scale));
            if constexpr (kMode == kSumHalfPow2) add2_exact_squares(v);
            else add2(v);
        }
    }
    __device__ __forceinline__ double total() const {
        return ((double)hi.x + (double)lo.x) + ((double)hi.y + (double)lo.y);
    }
    template <int kMode>
    __device__ __forceinline__ bool exact(double t) const {
        if constexpr (kMode == kSumHalfPow2) return t < 0x1p100;  // false for an infinity or a NaN
        return mx < 0x1p50f && !(mx < 0x1p-50f && mx > 0.0f) && t < 0x1p100;
    }
};

// Follows the list's octet space forwards: which tensor holds octet o, where that tensor's octets start, and its
// gradient base, length and vector flag. Octets only move forwards, so each tensor boundary is crossed once.
struct Cursor {
    int32_t k;
    int64_t lo, hi;
    const char* base;
    int64_t n;
    int64_t full;  // octets of the tensor with all eight elements
    int32_t vec;
    __device__ __forceinline__ void load(const ChunkTable& ct) {
        const TensorRec& r = ct.recs[k];
        base = static_cast<const char*>(r.g);
        n = r.n;
        full = r.n / kOct;
        vec = r.vec;
    }
    __device__ __forceinline__ void init(const ChunkTable& ct, int32_t k0) {
        k = k0;
        if (ct.T > 0) {
            lo = __ldg(ct.prefix + k0);
            hi = __ldg(ct.prefix + k0 + 1);
            load(ct);
        } else {  // an empty list: no octet is ever asked for
            lo = hi = 0;
            base = nullptr;
            n = 0;
            full = 0;
            vec = 0;
        }
    }
    __device__ __forceinline__ void advance(const ChunkTable& ct, int64_t o) {
        if (o < hi) return;
        do {
            ++k;
            lo = hi;
            hi = __ldg(ct.prefix + k + 1);
        } while (o >= hi);
        load(ct);
    }
};

// The elements of octet `local` of the cursor's tensor one by one (zeros past its end).
template <Dtype G>
__device__ __forceinline__ void load_elements(const Cursor& c, int64_t local, float (&x)[8]) {
    const int64_t i0 = local * kOct;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if (i0 + j < c.n) {
            x[j] = (G == kF16) ? __half2float(reinterpret_cast<const __half*>(c.base)[i0 + j])
                               : reinterpret_cast<const float*>(c.base)[i0 + j];
        } else {
            x[j] = 0.0f;
        }
    }
}

// Sum of one double per thread over the CTA, in a fixed order (a butterfly within each warp, then the warps in
// order). Valid in thread 0. Ends with a barrier, so `red` may be reused at once.
__device__ __forceinline__ double block_sum(double x, double* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if (lane == 0) red[warp] = x;
    __syncthreads();
    double t = 0.0;
    if (threadIdx.x == 0)
        for (int k = 0; k < nw; ++k) t += red[k];
    __syncthreads();
    return t;
}

// S = the partials summed in a fixed order (thread i takes i, i + 256, ... then block_sum); norm = f32(sqrt(S));
// factor = inv_scale * min(1, max_norm / (norm + 1e-6)) with PyTorch's clip_grad_norm_ rounding (every step in
// float32) and a NaN passed through.
__device__ void finalize_norm(const double* partials, int32_t num, float max_norm, float inv_scale, float* d_norm,
                              float* d_factor, double* red) {
    double acc = 0.0;
    for (int32_t i = threadIdx.x; i < num; i += blockDim.x) acc += __ldcg(partials + i);
    const double S = block_sum(acc, red);
    if (threadIdx.x == 0) {
        const float norm = __double2float_rn(__dsqrt_rn(S));
        const float coef = __fdiv_rn(max_norm, __fadd_rn(norm, 1e-6f));
        const float clip = (coef > 1.0f) ? 1.0f : coef;
        if (d_norm) *d_norm = norm;
        *d_factor = __fmul_rn(inv_scale, clip);
    }
}

// This thread's octets c0 + t, c0 + t + 256, ... below c1, squared and summed in double: the rare chunks the
// float32 pairs cannot hold exactly.
template <Dtype G>
__device__ __noinline__ double sumsq_chunk_double(const ChunkTable& ct, int32_t k0, int64_t c0, int64_t c1,
                                                  float inv_scale) {
    Cursor c;
    c.init(ct, k0);
    double t = 0.0;
    for (int64_t o = c0 + threadIdx.x; o < c1; o += kThreads) {
        c.advance(ct, o);
        float x[8];
        load_elements<G>(c, o - c.lo, x);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const double xd = (double)__fmul_rn(x[j], inv_scale);
            t = __fma_rn(xd, xd, t);
        }
    }
    return t;
}

// This thread's share of the sum of squares of the unscaled gradient, from its accumulator: in kSumHalfPow2 the
// squares of the binary16 values themselves were summed, and the power-of-two scale is applied here (exactly). A
// share the float32 pairs could not hold exactly is summed again in double.
template <Dtype G, int kMode>
__device__ __forceinline__ double share_total(const SumSq& acc, const ChunkTable& ct, int32_t k0, int64_t c0,
                                              int64_t c1, float inv_scale) {
    const double t = acc.total();
    if (!acc.exact<kMode>(t)) return sumsq_chunk_double<G>(ct, k0, c0, c1, kMode == kSumUnscaled ? 1.0f : inv_scale);
    if constexpr (kMode == kSumHalfPow2) return t * ((double)inv_scale * (double)inv_scale);
    return t;
}

// Up to kStaged consecutive tensors of a chunk, staged in shared memory: tensor i holds the list's octets
// [lo[i], lo[i + 1]), its gradient starts at base[i] and has n[i] elements, vec[i] says whether it is aligned for
// the vector loads.
constexpr int kStaged = 256;
struct StagedSpan {
    int64_t lo[kStaged + 1];
    const char* base[kStaged];
    int64_t n[kStaged];
    int32_t vec[kStaged];
};

// One gradient octet as loaded, before it is used: binary16 as its 4 words, float32 as its 8 values. Fetching the
// four octets of a round first and widening them afterwards keeps all four loads in flight at once.
template <Dtype G>
struct RawOctet;
template <>
struct RawOctet<kF16> {
    uint4 h;
};
template <>
struct RawOctet<kF32> {
    float x[8];
};

// Gradient octet `local` of staged tensor j (zeros past its end): one 32-byte load (16 for binary16) when whole and
// aligned, else element by element.
template <Dtype G>
__device__ __forceinline__ void fetch_staged_octet(const StagedSpan& sp, int32_t j, int64_t local, RawOctet<G>& r) {
    const char* base = sp.base[j];
    const int64_t n = sp.n[j];
    if (sp.vec[j] && local < n / kOct) {
        if constexpr (G == kF16) {
            asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(r.h.x), "=r"(r.h.y), "=r"(r.h.z), "=r"(r.h.w)
                         : "l"(base + local * 16));
        } else {
            asm volatile("ld.global.L1::no_allocate.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                         : "=f"(r.x[0]), "=f"(r.x[1]), "=f"(r.x[2]), "=f"(r.x[3]), "=f"(r.x[4]), "=f"(r.x[5]),
                           "=f"(r.x[6]), "=f"(r.x[7])
                         : "l"(base + local * 32));
        }
    } else {
        const int64_t i0 = local * kOct;
        if constexpr (G == kF16) {
            const uint16_t* p = reinterpret_cast<const uint16_t*>(base) + i0;
            uint32_t hv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) hv[e] = (i0 + e < n) ? p[e] : 0u;
            r.h = make_uint4(hv[0] | (hv[1] << 16), hv[2] | (hv[3] << 16), hv[4] | (hv[5] << 16),
                             hv[6] | (hv[7] << 16));
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) r.x[e] = (i0 + e < n) ? reinterpret_cast<const float*>(base)[i0 + e] : 0.0f;
        }
    }
}

template <Dtype G>
__device__ __forceinline__ void zero_octet(RawOctet<G>& r) {
    if constexpr (G == kF16) {
        r.h = make_uint4(0u, 0u, 0u, 0u);
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) r.x[e] = 0.0f;
    }
}

// The octet's values as float32 (binary16 widened exactly).
template <Dtype G>
__device__ __forceinline__ void widen_octet(const RawOctet<G>& r, float (&x)[8]) {
    if constexpr (G == kF16) {
        h8_to(r.h, x);
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = r.x[e];
    }
}

// The joint norm for lists of many small tensors, where a stage of the TMA pipeline would cross several tensors:
// CTA b streams its equal, contiguous chunk of the list's octets straight into registers. The CTA stages the
// chunk's tensors (their octet ranges, bases, sizes) in shared memory up to kStaged at a time; thread t takes the
// staged span's octets c + t, c + t + 256, ..., four at a time (eight for binary16), all their loads in flight
// before any is widened and summed, finding each octet's tensor by walking the staged table forwards. The rest is as in norm_tma_kernel.
template <Dtype G, int kMode>
__global__ void __launch_bounds__(kThreads, kNormDirectCtasPerSm) norm_direct_kernel(ChunkTable ct, float inv_scale,
                                                                        double* __restrict__ partials,
                                                                        unsigned int* ticket, float max_norm,
                                                                        float* d_norm, float* d_factor) {
    __shared__ double red[kWarps];
    __shared__ int last;
    __shared__ StagedSpan sp;
    const int t = threadIdx.x;
    const int64_t c0 = ct.total_octs * blockIdx.x / ct.grid;
    const int64_t c1 = ct.total_octs * (blockIdx.x + 1) / ct.grid;
    const int32_t k0 = ct.first[blockIdx.x];

    SumSq acc{{0.f, 0.f}, {0.f, 0.f}, 0.f};
    wait_prerequisite();  // the kernel queued before may still be writing the gradients (zero_grad)
    allow_dependents();   // the kernel queued next may launch from here (as in the TMA kernel)
    int32_t k = k0;
    int64_t ob = c0;
    while (ob < c1) {
        // stage tensors k .. k + cnt - 1 (ob lies in the first of them)
        const int32_t cnt = ct.T - k < kStaged ? ct.T - k : kStaged;
        __syncthreads();  // every thread is done with the previous span
        for (int i = t; i <= cnt; i += kThreads) sp.lo[i] = __ldg(ct.prefix + k + i);
        for (int i = t; i < cnt; i += kThreads) {
            const TensorRec& r = ct.recs[k + i];
            sp.base[i] = static_cast<const char*>(r.g);
            sp.n[i] = r.n;
            sp.vec[i] = r.vec;
        }
        __syncthreads();
        const int64_t oe = sp.lo[cnt] < c1 ? sp.lo[cnt] : c1;
        int32_t j = 0;
        constexpr int U = (G == kF16) ? 8 : 4;  // octets in flight per thread (a binary16 octet is 4 registers)
        for (int64_t o = ob + t; o < oe; o += U * kThreads) {
            RawOctet<G> raw[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t q = o + (int64_t)u * kThreads;
                if (q < oe) {
                    while (q >= sp.lo[j + 1]) ++j;
                    fetch_staged_octet<G>(sp, j, q - sp.lo[j], raw[u]);
                } else {
                    zero_octet<G>(raw[u]);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float x[8];
                widen_octet<G>(raw[u], x);
                acc.add8<kMode>(x, inv_scale);
            }
        }
        ob = oe;
        k += cnt;
    }
    double mine = share_total<G, kMode>(acc, ct, k0, c0, c1, inv_scale);

    const double part = block_sum(mine, red);
    if (t == 0) {
        partials[blockIdx.x] = part;
        __threadfence();  // the partial is visible before the ticket says so
        last = (atomicAdd(ticket, 1u) == (unsigned int)(ct.grid - 1));
    }
    __syncthreads();
    if (last) {  // every other CTA's partial is written: sum them all, in order
        __threadfence();
        finalize_norm(partials, ct.grid, max_norm, inv_scale, d_norm, d_factor, red);
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

// ------------------------------------------------------------------------------------------------------------------
// the joint norm: a TMA pipeline over equal contiguous chunks
// ------------------------------------------------------------------------------------------------------------------

// Each CTA streams its chunk of the list's octets through kNormStages shared-memory stages of 512 octets. One
// producer warp (its lane 0) walks the chunk and, per stage, issues one bulk copy per run of whole octets of an
// aligned tensor (a stage may cross tensor boundaries), completing on the stage's `full` barrier; the 8 consumer
// warps wait on it, thread t takes the stage's octets t and t + 256 (from shared memory, or element by element from
// global memory for a tensor's partial last octet or an unaligned tensor), then each warp arrives on the stage's
// `empty` barrier so the producer may refill it. The bytes in flight (up to 4 stages x 16 KB per CTA, 3 CTAs per
// SM) cost shared memory, not registers; two octets per thread and stage halve the per-stage bookkeeping.
constexpr int kNormStages = 4;
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

template <Dtype G, int kMode>
__global__ void __launch_bounds__(kNormThreads, kNormTmaCtasPerSm) norm_tma_kernel(ChunkTable ct, float inv_scale,
                                                                            double* __restrict__ partials,
                                                                            unsigned int* ticket, float max_norm,
                                                                            float* d_norm, float* d_factor) {
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
        finalize_norm(partials, ct.grid, max_norm, inv_scale, d_norm, d_factor, red);
        if (t == 0) *ticket = 0u;  // ready for the next launch on this list
    }
}

}  // namespace

template <Dtype G, int kMode>
cudaError_t launch_norm_t(const ChunkTable& ct, cudaStream_t st, float inv_scale, double* partials,
                          unsigned int* ticket, float max_norm, float* d_norm, float* d_factor) {
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
        return cudaLaunchKernelEx(&cfg, norm_direct_kernel<G, kMode>, ct, inv_scale, partials, ticket, max_norm,
                                  d_norm, d_factor);
    }
    const size_t smem = norm_smem_bytes<G>();
    cudaError_t e = cudaFuncSetAttribute(norm_tma_kernel<G, kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    cfg.blockDim = dim3(kNormThreads);
    cfg.dynamicSmemBytes = smem;
    return cudaLaunchKernelEx(&cfg, norm_tma_kernel<G, kMode>, ct, inv_scale, partials, ticket, max_norm, d_norm,
                              d_factor);
}

int launch_norm(const ChunkTable& ct, Dtype gdt, float inv_scale, double* partials, unsigned int* ticket,
                float max_norm, float* d_norm, float* d_factor, void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool scaled = inv_scale != 1.0f;  // an unscaled list skips the multiply (x * 1 is x)
    // binary16 times a power of two in [2^-102, 2^111]: every product is an exact normal float32
    int ex = 0;
    const bool pow2 = std::frexp(inv_scale, &ex) == 0.5f && inv_scale >= 0x1p-102f && inv_scale <= 0x1p111f;
    cudaError_t e;
    if (gdt == kF16 && pow2)
        e = launch_norm_t<kF16, kSumHalfPow2>(ct, st, inv_scale, partials, ticket, max_norm, d_norm, d_factor);
    else if (gdt == kF16)
        e = launch_norm_t<kF16, kSumScaled>(ct, st, inv_scale, partials, ticket, max_norm, d_norm, d_factor);
    else if (scaled)
        e = launch_norm_t<kF32, kSumScaled>(ct, st, inv_scale, partials, ticket, max_norm, d_norm, d_factor);
    else
        e = launch_norm_t<kF32, kSumUnscaled>(ct, st, inv_scale, partials, ticket, max_norm, d_norm, d_factor);
    count_launches(1);
    return (int)e;
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
