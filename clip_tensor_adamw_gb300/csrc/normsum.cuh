// Device code of the joint norm's sums shared by the kernels that compute it (norm.cu: the norm alone; fused.cu:
// the norm and the update in one cooperative launch): the exact sum of squares in float32 pairs, the walk over the
// list's octet space, the fixed-order reductions and finalize (the clip factor), and the register-streaming chunk
// sum for lists of small tensors.
#pragma once

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

// The partials summed in a fixed order (thread i takes i, i + B, ... then block_sum); valid in thread 0.
__device__ __forceinline__ double sum_partials(const double* partials, int32_t num, double* red) {
    double acc = 0.0;
    for (int32_t i = threadIdx.x; i < num; i += blockDim.x) acc += __ldcg(partials + i);
    return block_sum(acc, red);
}

// norm = f32(sqrt(S)); factor = inv_scale * min(1, max_norm / (norm + 1e-6)) with PyTorch's clip_grad_norm_
// rounding (every step in float32) and a NaN passed through.
__device__ __forceinline__ void norm_and_factor(double S, float max_norm, float inv_scale, float* norm_out,
                                                float* factor_out) {
    const float norm = __double2float_rn(__dsqrt_rn(S));
    const float coef = __fdiv_rn(max_norm, __fadd_rn(norm, 1e-6f));
    const float clip = (coef > 1.0f) ? 1.0f : coef;
    *norm_out = norm;
    *factor_out = __fmul_rn(inv_scale, clip);
}

// The finalize of a norm launch: the partials summed in a fixed order; the square sum itself written to d_sumsq
// when that is not null, and norm and factor to d_norm and d_factor when those are not null.
__device__ void finalize_norm(const double* partials, int32_t num, float max_norm, float inv_scale, float* d_norm,
                              float* d_factor, double* d_sumsq, double* red) {
    const double S = sum_partials(partials, num, red);
    if (threadIdx.x == 0) {
        float norm, factor;
        norm_and_factor(S, max_norm, inv_scale, &norm, &factor);
        if (d_norm) *d_norm = norm;
        if (d_factor) *d_factor = factor;
        if (d_sumsq) *d_sumsq = S;
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
static_assert((kThreads & (kThreads - 1)) == 0, "a thread's octets are found with a mask of kThreads - 1");
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
// With kKeepL2 the vector loads carry the L2 cache policy `keep` (an evict-last policy from l2_keep_policy), for a
// gradient that is read again soon.
__device__ __forceinline__ uint64_t l2_keep_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

template <Dtype G, bool kKeepL2 = false>
__device__ __forceinline__ void fetch_staged_octet(const StagedSpan& sp, int32_t j, int64_t local, RawOctet<G>& r,
                                                   uint64_t keep = 0) {
    const char* base = sp.base[j];
    const int64_t n = sp.n[j];
    if (sp.vec[j] && local < n / kOct) {
        if constexpr (G == kF16 && kKeepL2) {
            asm volatile("ld.global.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                         : "=r"(r.h.x), "=r"(r.h.y), "=r"(r.h.z), "=r"(r.h.w)
                         : "l"(base + local * 16), "l"(keep));
        } else if constexpr (G == kF16) {
            asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(r.h.x), "=r"(r.h.y), "=r"(r.h.z), "=r"(r.h.w)
                         : "l"(base + local * 16));
        } else if constexpr (kKeepL2) {
            asm volatile("ld.global.L1::no_allocate.L2::cache_hint.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8], %9;"
                         : "=f"(r.x[0]), "=f"(r.x[1]), "=f"(r.x[2]), "=f"(r.x[3]), "=f"(r.x[4]), "=f"(r.x[5]),
                           "=f"(r.x[6]), "=f"(r.x[7])
                         : "l"(base + local * 32), "l"(keep));
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

// This thread's share of the sum of squares of chunk b of `grid` equal contiguous chunks of the list's octets, for
// lists of many small tensors, where a stage of the TMA pipeline would cross several tensors: the CTA streams the
// chunk straight into registers, staging the chunk's tensors (their octet ranges, bases, sizes) in `sp` up to
// kStaged at a time; thread t takes the chunk's octets c0 + t, c0 + t + 256, ... (in every staged span, those of
// them that lie in it: the same octets that its double-precision re-sum in share_total takes, however many spans
// the chunk has), four at a time (eight for binary16), all their loads in flight before any is widened and summed,
// finding each octet's tensor by walking the staged table forwards. Every thread of the CTA calls it (it meets the
// others at barriers).
template <Dtype G, int kMode, bool kKeepL2 = false>
__device__ __forceinline__ double direct_chunk_share(const ChunkTable& ct, int32_t b, int32_t grid, float inv_scale,
                                                     StagedSpan& sp) {
    const int t = threadIdx.x;
    const int64_t c0 = ct.total_octs * b / grid;
    const int64_t c1 = ct.total_octs * (b + 1) / grid;
    const int32_t k0 = ct.first[b];
    SumSq acc{{0.f, 0.f}, {0.f, 0.f}, 0.f};
    const uint64_t keep = kKeepL2 ? l2_keep_policy() : 0;
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
        // this thread's first octet of the span: the first at or after ob that is c0 + t plus a multiple of 256
        const int64_t first = ob + ((t - (int32_t)((ob - c0) & (kThreads - 1))) & (kThreads - 1));
        for (int64_t o = first; o < oe; o += U * kThreads) {
            RawOctet<G> raw[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t q = o + (int64_t)u * kThreads;
                if (q < oe) {
                    while (q >= sp.lo[j + 1]) ++j;
                    fetch_staged_octet<G, kKeepL2>(sp, j, q - sp.lo[j], raw[u], keep);
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
    return share_total<G, kMode>(acc, ct, k0, c0, c1, inv_scale);
}

}  // namespace
}  // namespace mica
