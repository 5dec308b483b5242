// The hot path's kernels for sm_103a: the joint-norm partials and their fixed-order finalize, the multi-tensor AdamW
// update, and ScaleTensors. All three are streams over HBM with no data reuse, so they are built for bandwidth:
// 16-byte vector accesses that coalesce across a warp, several quads in flight per thread, evict-first cache hints,
// and enough CTAs per SM to keep ~100 KB of loads outstanding on each of the 152 SMs.
//
// Per-element arithmetic follows BendTorch "main.bend", section "Optimizers": every float32 operation is a separate
// correctly rounded intrinsic (__fmul_rn, __fadd_rn, __fdiv_rn, __fsqrt_rn), which the compiler never fuses into an
// FMA, in the order that section gives; so the update is bit-identical to the same step on the CPU.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "plan.h"

namespace mica {
namespace {

constexpr int kUnrollAdam = 2;   // quads each thread keeps in flight per round (AdamW: 4 streams)
constexpr int kUnrollNorm = 8;   // (norm: the gradient only)
constexpr int kUnrollScale = 4;  // (scale: one stream)

// ------------------------------------------------------------------------------------------------------------------
// memory access: streaming (evict-first) 16- and 8-byte vectors
// ------------------------------------------------------------------------------------------------------------------

__device__ __forceinline__ float4 ld_f4(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ void st_f4(float* p, float4 x) { __stcs(reinterpret_cast<float4*>(p), x); }
__device__ __forceinline__ uint2 ld_u2(const void* p) { return __ldcs(reinterpret_cast<const uint2*>(p)); }
__device__ __forceinline__ void st_u2(void* p, uint2 x) { __stcs(reinterpret_cast<uint2*>(p), x); }

__device__ __forceinline__ void f4_to(const float4& x, float (&a)[4]) {
    a[0] = x.x; a[1] = x.y; a[2] = x.z; a[3] = x.w;
}
__device__ __forceinline__ float4 f4_of(const float (&a)[4]) { return make_float4(a[0], a[1], a[2], a[3]); }

// four binary16 values (8 bytes) -> float32 (exact)
__device__ __forceinline__ void h4_to(const uint2& x, float (&a)[4]) {
    __half2 lo = *reinterpret_cast<const __half2*>(&x.x);
    __half2 hi = *reinterpret_cast<const __half2*>(&x.y);
    float2 l = __half22float2(lo), h = __half22float2(hi);
    a[0] = l.x; a[1] = l.y; a[2] = h.x; a[3] = h.y;
}

// ------------------------------------------------------------------------------------------------------------------
// packed BF16 (BendTorch "main.bend", "AdamW over packed BF16 moments"): element 2k is the low half of word k
// ------------------------------------------------------------------------------------------------------------------

__device__ __forceinline__ float bf16_lo(uint32_t word) { return __uint_as_float(word << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t word) { return __uint_as_float(word & 0xFFFF0000u); }

// Two float32 -> one word, each rounded to nearest-even by the hardware conversion; a NaN is stored as 0xFFFF.
__device__ __forceinline__ uint32_t pack_bf16x2(float even, float odd) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(odd), "f"(even));  // first source -> high half
    if (even != even) r |= 0x0000FFFFu;
    if (odd != odd) r |= 0xFFFF0000u;
    return r;
}

// ------------------------------------------------------------------------------------------------------------------
// AdamW on one quad, in registers
// ------------------------------------------------------------------------------------------------------------------

// m, v hold the moments read (float32, or the exact widening of the stored BF16); on return they hold the new
// moments as the weight update reads them (rounded through BF16 when kPacked), and pm, pv the packed words to store.
template <bool kPacked>
__device__ __forceinline__ void adam_quad(float (&w)[4], const float (&g)[4], float (&m)[4], float (&v)[4],
                                          uint32_t (&pm)[2], uint32_t (&pv)[2], const StepScalars& s, float f) {
    float wdec[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float gh = __fmul_rn(g[j], f);
        wdec[j] = __fmul_rn(w[j], s.dec);
        m[j] = __fadd_rn(m[j], __fmul_rn(s.c1, __fsub_rn(gh, m[j])));
        v[j] = __fadd_rn(__fmul_rn(v[j], s.b2), __fmul_rn(__fmul_rn(s.c2, gh), gh));
    }
    if constexpr (kPacked) {
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            pm[p] = pack_bf16x2(m[2 * p], m[2 * p + 1]);
            pv[p] = pack_bf16x2(v[2 * p], v[2 * p + 1]);
            m[2 * p] = bf16_lo(pm[p]);
            m[2 * p + 1] = bf16_hi(pm[p]);
            v[2 * p] = bf16_lo(pv[p]);
            v[2 * p + 1] = bf16_hi(pv[p]);
        }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float denom = __fadd_rn(__fdiv_rn(__fsqrt_rn(v[j]), s.bc2), s.eps);
        w[j] = __fadd_rn(wdec[j], __fdiv_rn(__fmul_rn(s.neg_step, m[j]), denom));
    }
}

// One quad element by element: for bases not 16-byte aligned and for a tensor's last, partial quad. Elements past n
// are neither read nor written, nor is the high half of a last packed word that holds no element.
template <Dtype G, Dtype M>
__device__ void adam_quad_elements(const TensorRec& r, int64_t q, const StepScalars& s, float f) {
    const int64_t i0 = q * 4;
    const int64_t left = r.n - i0;
    const int cnt = left < 4 ? (int)left : 4;
    float w[4] = {0.f, 0.f, 0.f, 0.f}, g[4] = {0.f, 0.f, 0.f, 0.f};
    float m[4] = {0.f, 0.f, 0.f, 0.f}, v[4] = {0.f, 0.f, 0.f, 0.f};
    uint32_t om[2] = {0u, 0u}, ov[2] = {0u, 0u}, pm[2], pv[2];
    for (int j = 0; j < cnt; ++j) {
        w[j] = r.w[i0 + j];
        g[j] = (G == kF16) ? __half2float(static_cast<const __half*>(r.g)[i0 + j]) : static_cast<const float*>(r.g)[i0 + j];
    }
    if constexpr (M == kBF16x2) {
        for (int p = 0; p < 2; ++p) {
            if (2 * p < cnt) {
                om[p] = static_cast<const uint32_t*>(r.m)[2 * q + p];
                ov[p] = static_cast<const uint32_t*>(r.v)[2 * q + p];
                m[2 * p] = bf16_lo(om[p]);
                m[2 * p + 1] = bf16_hi(om[p]);
                v[2 * p] = bf16_lo(ov[p]);
                v[2 * p + 1] = bf16_hi(ov[p]);
            }
        }
    } else {
        for (int j = 0; j < cnt; ++j) {
            m[j] = static_cast<const float*>(r.m)[i0 + j];
            v[j] = static_cast<const float*>(r.v)[i0 + j];
        }
    }
    adam_quad<M == kBF16x2>(w, g, m, v, pm, pv, s, f);
    for (int j = 0; j < cnt; ++j) {
        r.w[i0 + j] = w[j];
        if (s.zero_grad) {
            if (G == kF16) static_cast<__half*>(r.g)[i0 + j] = __ushort_as_half(0);
            else static_cast<float*>(r.g)[i0 + j] = 0.f;
        }
    }
    if constexpr (M == kBF16x2) {
        for (int p = 0; p < 2; ++p) {
            if (2 * p < cnt) {
                uint32_t nm = pm[p], nv = pv[p];
                if (2 * p + 1 >= cnt) {  // the word's high half holds no element: keep it as it was
                    nm = (nm & 0x0000FFFFu) | (om[p] & 0xFFFF0000u);
                    nv = (nv & 0x0000FFFFu) | (ov[p] & 0xFFFF0000u);
                }
                static_cast<uint32_t*>(r.m)[2 * q + p] = nm;
                static_cast<uint32_t*>(r.v)[2 * q + p] = nv;
            }
        }
    } else {
        for (int j = 0; j < cnt; ++j) {
            static_cast<float*>(r.m)[i0 + j] = m[j];
            static_cast<float*>(r.v)[i0 + j] = v[j];
        }
    }
}

// Quads [qb, qe) of one tensor, quad qb + lane first, then every `stride`-th.
template <Dtype G, Dtype M>
__device__ __forceinline__ void adam_range(const TensorRec& r, int64_t qb, int64_t qe, int lane, int stride,
                                           const StepScalars& s, float f) {
    const int64_t full = r.n >> 2;  // quads with all four elements
    if (r.vec) {
        const int64_t vend = min(qe, full);
        for (int64_t q0 = qb + lane; q0 < vend; q0 += (int64_t)stride * kUnrollAdam) {
            float4 W[kUnrollAdam], Gf[kUnrollAdam], Mf[kUnrollAdam], Vf[kUnrollAdam];
            uint2 Gh[kUnrollAdam], Mp[kUnrollAdam], Vp[kUnrollAdam];
#pragma unroll
            for (int u = 0; u < kUnrollAdam; ++u) {
                const int64_t q = q0 + (int64_t)u * stride;
                if (q < vend) {
                    W[u] = ld_f4(r.w + 4 * q);
                    if constexpr (G == kF16) Gh[u] = ld_u2(static_cast<const __half*>(r.g) + 4 * q);
                    else Gf[u] = ld_f4(static_cast<const float*>(r.g) + 4 * q);
                    if constexpr (M == kBF16x2) {
                        Mp[u] = ld_u2(static_cast<const uint32_t*>(r.m) + 2 * q);
                        Vp[u] = ld_u2(static_cast<const uint32_t*>(r.v) + 2 * q);
                    } else {
                        Mf[u] = ld_f4(static_cast<const float*>(r.m) + 4 * q);
                        Vf[u] = ld_f4(static_cast<const float*>(r.v) + 4 * q);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kUnrollAdam; ++u) {
                const int64_t q = q0 + (int64_t)u * stride;
                if (q < vend) {
                    float w[4], g[4], m[4], v[4];
                    uint32_t pm[2], pv[2];
                    f4_to(W[u], w);
                    if constexpr (G == kF16) h4_to(Gh[u], g);
                    else f4_to(Gf[u], g);
                    if constexpr (M == kBF16x2) {
                        m[0] = bf16_lo(Mp[u].x); m[1] = bf16_hi(Mp[u].x);
                        m[2] = bf16_lo(Mp[u].y); m[3] = bf16_hi(Mp[u].y);
                        v[0] = bf16_lo(Vp[u].x); v[1] = bf16_hi(Vp[u].x);
                        v[2] = bf16_lo(Vp[u].y); v[3] = bf16_hi(Vp[u].y);
                    } else {
                        f4_to(Mf[u], m);
                        f4_to(Vf[u], v);
                    }
                    adam_quad<M == kBF16x2>(w, g, m, v, pm, pv, s, f);
                    st_f4(r.w + 4 * q, f4_of(w));
                    if constexpr (M == kBF16x2) {
                        st_u2(static_cast<uint32_t*>(r.m) + 2 * q, make_uint2(pm[0], pm[1]));
                        st_u2(static_cast<uint32_t*>(r.v) + 2 * q, make_uint2(pv[0], pv[1]));
                    } else {
                        st_f4(static_cast<float*>(r.m) + 4 * q, f4_of(m));
                        st_f4(static_cast<float*>(r.v) + 4 * q, f4_of(v));
                    }
                    if (s.zero_grad) {
                        if constexpr (G == kF16) st_u2(static_cast<__half*>(r.g) + 4 * q, make_uint2(0u, 0u));
                        else st_f4(static_cast<float*>(r.g) + 4 * q, make_float4(0.f, 0.f, 0.f, 0.f));
                    }
                }
            }
        }
        // the last, partial quad (n % 4 != 0), when it lies in this range
        if (full < qe && full >= qb && lane == (int)((full - qb) % stride)) adam_quad_elements<G, M>(r, full, s, f);
    } else {
        for (int64_t q = qb + lane; q < qe; q += stride) adam_quad_elements<G, M>(r, q, s, f);
    }
}

template <Dtype G, Dtype M>
__global__ void __launch_bounds__(kThreads, 2) adamw_kernel(const TensorRec* __restrict__ recs,
                                                         const WorkItem* __restrict__ items, int32_t num_items,
                                                         int32_t item_quads, StepScalars s,
                                                         const float* __restrict__ d_factor) {
    const float f = d_factor ? __ldg(d_factor) : 1.0f;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int32_t it = blockIdx.x; it < num_items; it += gridDim.x) {
        const WorkItem item = items[it];
        if (item.count == 1) {
            const TensorRec r = recs[item.t];
            const int64_t nq = (r.n + 3) >> 2;
            adam_range<G, M>(r, item.q0, min(item.q0 + (int64_t)item_quads, nq), threadIdx.x, kThreads, s, f);
        } else {
            for (int k = warp; k < item.count; k += kWarps) {
                const TensorRec r = recs[item.t + k];
                adam_range<G, M>(r, 0, (r.n + 3) >> 2, lane, 32, s, f);
            }
        }
    }
}

// ------------------------------------------------------------------------------------------------------------------
// joint norm: per-item partial square sums, then one fixed-order finalize
// ------------------------------------------------------------------------------------------------------------------

// Adds x^2 to the pair (hi, lo) without loss: the product's rounding error comes from an FMA and the sum's from
// Knuth's two-sum, so hi + lo carries the running sum to about twice float32's precision. This holds while
// 2^-50 <= |x| < 2^50 (the product error then stays a normal float32 and sums cannot overflow); a zero adds nothing;
// anything else (tiny, huge, infinite, NaN) is squared and summed in double in `ext`.
__device__ __forceinline__ void add_square(float x, float& hi, float& lo, double& ext) {
    const uint32_t ex = (__float_as_uint(x) >> 23) & 0xFFu;
    if ((ex - 77u) < 100u) {
        const float p = __fmul_rn(x, x);
        const float e = __fmaf_rn(x, x, -p);
        const float s = __fadd_rn(hi, p);
        const float bp = __fsub_rn(s, hi);
        const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(p, bp));
        hi = s;
        lo = __fadd_rn(lo, __fadd_rn(err, e));
    } else if (x != 0.0f) {
        const double xd = (double)x;
        ext = __fma_rn(xd, xd, ext);
    }
}

template <Dtype G>
__device__ __forceinline__ void sumsq_range(const TensorRec& r, int64_t qb, int64_t qe, int lane, int stride,
                                            float inv_scale, float& hi, float& lo, double& ext) {
    const int64_t full = r.n >> 2;
    if (r.vec) {
        const int64_t vend = min(qe, full);
        for (int64_t q0 = qb + lane; q0 < vend; q0 += (int64_t)stride * kUnrollNorm) {
            float4 Gf[kUnrollNorm];
            uint2 Gh[kUnrollNorm];
#pragma unroll
            for (int u = 0; u < kUnrollNorm; ++u) {
                const int64_t q = q0 + (int64_t)u * stride;
                if (q < vend) {
                    if constexpr (G == kF16) Gh[u] = ld_u2(static_cast<const __half*>(r.g) + 4 * q);
                    else Gf[u] = ld_f4(static_cast<const float*>(r.g) + 4 * q);
                }
            }
#pragma unroll
            for (int u = 0; u < kUnrollNorm; ++u) {
                const int64_t q = q0 + (int64_t)u * stride;
                if (q < vend) {
                    float g[4];
                    if constexpr (G == kF16) h4_to(Gh[u], g);
                    else f4_to(Gf[u], g);
#pragma unroll
                    for (int j = 0; j < 4; ++j) add_square(__fmul_rn(g[j], inv_scale), hi, lo, ext);
                }
            }
        }
        if (full < qe && full >= qb && lane == (int)((full - qb) % stride)) {
            for (int64_t i = full * 4; i < r.n; ++i) {
                const float g = (G == kF16) ? __half2float(static_cast<const __half*>(r.g)[i])
                                            : static_cast<const float*>(r.g)[i];
                add_square(__fmul_rn(g, inv_scale), hi, lo, ext);
            }
        }
    } else {
        for (int64_t q = qb + lane; q < qe; q += stride) {
            const int64_t end = min(r.n, 4 * q + 4);
            for (int64_t i = 4 * q; i < end; ++i) {
                const float g = (G == kF16) ? __half2float(static_cast<const __half*>(r.g)[i])
                                            : static_cast<const float*>(r.g)[i];
                add_square(__fmul_rn(g, inv_scale), hi, lo, ext);
            }
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

template <Dtype G>
__global__ void __launch_bounds__(kThreads) norm_partials_kernel(const TensorRec* __restrict__ recs,
                                                                 const WorkItem* __restrict__ items,
                                                                 int32_t num_items, int32_t item_quads,
                                                                 float inv_scale, double* __restrict__ partials) {
    __shared__ double red[kWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int32_t it = blockIdx.x; it < num_items; it += gridDim.x) {
        const WorkItem item = items[it];
        float hi = 0.f, lo = 0.f;
        double ext = 0.0;
        if (item.count == 1) {
            const TensorRec r = recs[item.t];
            const int64_t nq = (r.n + 3) >> 2;
            sumsq_range<G>(r, item.q0, min(item.q0 + (int64_t)item_quads, nq), threadIdx.x, kThreads, inv_scale,
                           hi, lo, ext);
        } else {
            for (int k = warp; k < item.count; k += kWarps) {
                const TensorRec r = recs[item.t + k];
                sumsq_range<G>(r, 0, (r.n + 3) >> 2, lane, 32, inv_scale, hi, lo, ext);
            }
        }
        const double t = block_sum(((double)hi + (double)lo) + ext, red);
        if (threadIdx.x == 0) partials[it] = t;
    }
}

constexpr int kFinalizeThreads = 1024;

// S = the partials summed in a fixed order; norm = f32(sqrt(S)); factor = inv_scale * min(1, max_norm / (norm +
// 1e-6)) with PyTorch's clip_grad_norm_ rounding (every step in float32) and a NaN passed through.
__global__ void __launch_bounds__(kFinalizeThreads) norm_finalize_kernel(const double* __restrict__ partials,
                                                                         int32_t num, float max_norm,
                                                                         float inv_scale, float* d_norm,
                                                                         float* d_factor) {
    __shared__ double red[kFinalizeThreads / 32];
    double acc = 0.0;
    for (int32_t i = threadIdx.x; i < num; i += kFinalizeThreads) acc += partials[i];
    const double S = block_sum(acc, red);
    if (threadIdx.x == 0) {
        const float norm = __double2float_rn(__dsqrt_rn(S));
        const float coef = __fdiv_rn(max_norm, __fadd_rn(norm, 1e-6f));
        const float clip = (coef > 1.0f) ? 1.0f : coef;
        if (d_norm) *d_norm = norm;
        *d_factor = __fmul_rn(inv_scale, clip);
    }
}

// ------------------------------------------------------------------------------------------------------------------
// ScaleTensors
// ------------------------------------------------------------------------------------------------------------------

template <Dtype T>
__device__ __forceinline__ void scale_range(const TensorRec& r, int64_t qb, int64_t qe, int lane, int stride,
                                            float f) {
    const int64_t full = r.n >> 2;
    const int64_t vend = r.vec ? min(qe, full) : qb;
    for (int64_t q0 = qb + lane; q0 < vend; q0 += (int64_t)stride * kUnrollScale) {
        float4 X[kUnrollScale];
        uint2 H[kUnrollScale];
#pragma unroll
        for (int u = 0; u < kUnrollScale; ++u) {
            const int64_t q = q0 + (int64_t)u * stride;
            if (q < vend) {
                if constexpr (T == kF16) H[u] = ld_u2(reinterpret_cast<const __half*>(r.w) + 4 * q);
                else X[u] = ld_f4(r.w + 4 * q);
            }
        }
#pragma unroll
        for (int u = 0; u < kUnrollScale; ++u) {
            const int64_t q = q0 + (int64_t)u * stride;
            if (q < vend) {
                float a[4];
                if constexpr (T == kF16) h4_to(H[u], a);
                else f4_to(X[u], a);
#pragma unroll
                for (int j = 0; j < 4; ++j) a[j] = __fmul_rn(a[j], f);
                if constexpr (T == kF16) {
                    __half2 lo = __floats2half2_rn(a[0], a[1]), hi = __floats2half2_rn(a[2], a[3]);
                    st_u2(reinterpret_cast<__half*>(r.w) + 4 * q,
                          make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi)));
                } else {
                    st_f4(r.w + 4 * q, f4_of(a));
                }
            }
        }
    }
    // elements not covered by vectors: the partial last quad, or everything when unaligned
    const int64_t eb = (vend > qb ? vend : qb) * 4, ee = min(r.n, qe * 4);
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
                                                         int32_t item_quads, float factor,
                                                         const float* __restrict__ d_factor) {
    const float f = d_factor ? __ldg(d_factor) : factor;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int32_t it = blockIdx.x; it < num_items; it += gridDim.x) {
        const WorkItem item = items[it];
        if (item.count == 1) {
            const TensorRec r = recs[item.t];
            const int64_t nq = (r.n + 3) >> 2;
            scale_range<T>(r, item.q0, min(item.q0 + (int64_t)item_quads, nq), threadIdx.x, kThreads, f);
        } else {
            for (int k = warp; k < item.count; k += kWarps) {
                const TensorRec r = recs[item.t + k];
                scale_range<T>(r, 0, (r.n + 3) >> 2, lane, 32, f);
            }
        }
    }
}

int grid_for(int32_t num_items) { return num_items; }

}  // namespace

// ------------------------------------------------------------------------------------------------------------------
// launchers
// ------------------------------------------------------------------------------------------------------------------

int launch_adamw(const TensorRec* recs, const WorkItem* items, int32_t num_items, int32_t item_quads, Dtype gdt,
                 Dtype mdt, const StepScalars& s, const float* d_factor, void* stream) {
    if (num_items <= 0) return (int)cudaSuccess;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const dim3 grid(grid_for(num_items)), block(kThreads);
    if (gdt == kF32 && mdt == kF32)
        adamw_kernel<kF32, kF32><<<grid, block, 0, st>>>(recs, items, num_items, item_quads, s, d_factor);
    else if (gdt == kF32 && mdt == kBF16x2)
        adamw_kernel<kF32, kBF16x2><<<grid, block, 0, st>>>(recs, items, num_items, item_quads, s, d_factor);
    else if (gdt == kF16 && mdt == kF32)
        adamw_kernel<kF16, kF32><<<grid, block, 0, st>>>(recs, items, num_items, item_quads, s, d_factor);
    else
        adamw_kernel<kF16, kBF16x2><<<grid, block, 0, st>>>(recs, items, num_items, item_quads, s, d_factor);
    count_launches(1);
    return (int)cudaGetLastError();
}

int launch_norm(const TensorRec* recs, const WorkItem* items, int32_t num_items, int32_t item_quads, Dtype gdt,
                float inv_scale, double* partials, float max_norm, float* d_norm, float* d_factor, void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (num_items > 0) {
        const dim3 grid(grid_for(num_items)), block(kThreads);
        if (gdt == kF16)
            norm_partials_kernel<kF16><<<grid, block, 0, st>>>(recs, items, num_items, item_quads, inv_scale,
                                                               partials);
        else
            norm_partials_kernel<kF32><<<grid, block, 0, st>>>(recs, items, num_items, item_quads, inv_scale,
                                                               partials);
        count_launches(1);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return (int)e;
    }
    norm_finalize_kernel<<<1, kFinalizeThreads, 0, st>>>(partials, num_items, max_norm, inv_scale, d_norm, d_factor);
    count_launches(1);
    return (int)cudaGetLastError();
}

int launch_scale(const TensorRec* recs, const WorkItem* items, int32_t num_items, int32_t item_quads, Dtype dt,
                 float factor, const float* d_factor, void* stream) {
    if (num_items <= 0) return (int)cudaSuccess;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const dim3 grid(grid_for(num_items)), block(kThreads);
    if (dt == kF16)
        scale_kernel<kF16><<<grid, block, 0, st>>>(recs, items, num_items, item_quads, factor, d_factor);
    else
        scale_kernel<kF32><<<grid, block, 0, st>>>(recs, items, num_items, item_quads, factor, d_factor);
    count_launches(1);
    return (int)cudaGetLastError();
}

}  // namespace mica
