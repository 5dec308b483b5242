// The gradient's last write fused with ClipGradNorms, for sm_103a: when a gradient has several contributions (a
// weight read by more than one step of the recorded model, or micro-batches summed), its last write is an add, and
// this kernel makes that add and measures the joint norm of the list it leaves in one pass. The norm then reads the
// values it has just written from registers, not from HBM a second time.
//
// The add: an operand read by several recorded steps gets the sum of what each hands it ("Mica 7.7", section
// "Values that stay on the card": the tape walks the steps backwards and hands each operand its gradient). float32
// cells add in float32; binary16 cells are widened, added in float32 and rounded back to nearest-even, which is the
// correctly rounded binary16 sum (float32 carries at least 2 x 11 + 2 significant bits). The norm is ClipGradNorms's
// ("Mica 7.7", sections "The whole model in one call" and "Values that stay on the card") over the result: the
// exact float32-pair square sums of normsum.cuh, one partial per CTA, the fixed-order finalize by the CTA that
// finishes last.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "normsum.cuh"
#include "plan.h"
#include "stream.cuh"

namespace mica {
namespace {

// Up to kStaged consecutive tensors of a chunk, staged in shared memory: tensor i holds the list's octets
// [lo[i], lo[i + 1]), its gradient starts at g[i] and its addend at a[i], it has n[i] elements, and vec[i] says
// whether both are aligned for the vector accesses.
struct AccSpan {
    int64_t lo[kStaged + 1];
    char* g[kStaged];
    const char* a[kStaged];
    int64_t n[kStaged];
    int32_t vec[kStaged];
};

// Octets in flight per thread and round: 2 float32 octets (g and a: 32 registers), 4 binary16 ones.
template <Dtype G>
__host__ __device__ constexpr int acc_round() { return G == kF16 ? 4 : 2; }

// Plain loads (both streams are read once here; g's lines are written right after, a's are not used again).
template <Dtype G>
__device__ __forceinline__ void load_vec(const char* p, RawOctet<G>& r) {
    if constexpr (G == kF16) {
        asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(r.h.x), "=r"(r.h.y), "=r"(r.h.z), "=r"(r.h.w)
                     : "l"(p));
    } else {
        asm volatile("ld.global.L1::no_allocate.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=f"(r.x[0]), "=f"(r.x[1]), "=f"(r.x[2]), "=f"(r.x[3]), "=f"(r.x[4]), "=f"(r.x[5]),
                       "=f"(r.x[6]), "=f"(r.x[7])
                     : "l"(p));
    }
}

// The new gradient octet back to `p`; with kKeepL2 the store carries the L2 policy `keep` (evict-last), so that the
// update that follows finds a gradient that fits in L2 there.
template <Dtype G, bool kKeepL2>
__device__ __forceinline__ void store_vec(char* p, const RawOctet<G>& r, uint64_t keep) {
    if constexpr (G == kF16 && kKeepL2) {
        asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "r"(r.h.x), "r"(r.h.y),
                     "r"(r.h.z), "r"(r.h.w), "l"(keep)
                     : "memory");
    } else if constexpr (G == kF16) {
        asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(r.h.x), "r"(r.h.y), "r"(r.h.z),
                     "r"(r.h.w)
                     : "memory");
    } else if constexpr (kKeepL2) {
        asm volatile("st.global.L2::cache_hint.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8}, %9;" ::"l"(p), "f"(r.x[0]),
                     "f"(r.x[1]), "f"(r.x[2]), "f"(r.x[3]), "f"(r.x[4]), "f"(r.x[5]), "f"(r.x[6]), "f"(r.x[7]),
                     "l"(keep)
                     : "memory");
    } else {
        asm volatile("st.global.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "f"(r.x[0]), "f"(r.x[1]),
                     "f"(r.x[2]), "f"(r.x[3]), "f"(r.x[4]), "f"(r.x[5]), "f"(r.x[6]), "f"(r.x[7])
                     : "memory");
    }
}

// One binary16 pair plus another, each half widened, added in float32 and rounded back to nearest-even.
__device__ __forceinline__ uint32_t add_half2(uint32_t x, uint32_t y) {
    __half2 hx, hy;
    memcpy(&hx, &x, 4);
    memcpy(&hy, &y, 4);
    const float2 fx = __half22float2(hx), fy = __half22float2(hy);
    const __half2 r = __floats2half2_rn(__fadd_rn(fx.x, fy.x), __fadd_rn(fx.y, fy.y));
    uint32_t out;
    memcpy(&out, &r, 4);
    return out;
}

// g + a over one octet held in registers; the result replaces g.
template <Dtype G>
__device__ __forceinline__ void add_octet(RawOctet<G>& g, const RawOctet<G>& a) {
    if constexpr (G == kF16) {
        g.h = make_uint4(add_half2(g.h.x, a.h.x), add_half2(g.h.y, a.h.y), add_half2(g.h.z, a.h.z),
                         add_half2(g.h.w, a.h.w));
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) g.x[e] = __fadd_rn(g.x[e], a.x[e]);
    }
}

// Octet `local` of a tensor element by element (a partial last octet, or a tensor not aligned for the vectors): the
// sums of its elements below n (at most 8) written back, and returned as float32 in x (zeros past the end).
template <Dtype G>
__device__ __noinline__ void add_octet_elements(char* g, const char* a, int64_t n, int64_t local, float (&x)[8]) {
    const int64_t i0 = local * kOct;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        x[e] = 0.0f;
        if (i0 + e < n) {
            if constexpr (G == kF16) {
                __half* gp = reinterpret_cast<__half*>(g) + i0 + e;
                const __half s = __float2half_rn(
                    __fadd_rn(__half2float(*gp), __half2float(reinterpret_cast<const __half*>(a)[i0 + e])));
                *gp = s;
                x[e] = __half2float(s);
            } else {
                float* gp = reinterpret_cast<float*>(g) + i0 + e;
                const float s = __fadd_rn(*gp, reinterpret_cast<const float*>(a)[i0 + e]);
                *gp = s;
                x[e] = s;
            }
        }
    }
}

// This thread's share of the square sum of chunk b's new gradient, after writing it: the chunk's tensors are staged
// in `sp` up to kStaged at a time; thread t takes the chunk's octets c0 + t + 256 k (in every staged span those of
// them that lie in it, which is also what share_total's double-precision re-sum takes), acc_round<G>() at a time
// with all their loads in flight, adds, stores and sums the squares of what it stored.
template <Dtype G, int kMode, bool kKeepL2>
__device__ __forceinline__ double accumulate_chunk_share(const ChunkTable& ct, int32_t b, float inv_scale,
                                                         AccSpan& sp) {
    constexpr int U = acc_round<G>();
    constexpr int kOctBytes = (G == kF16) ? 16 : 32;
    const int t = threadIdx.x;
    const int64_t c0 = ct.total_octs * b / ct.grid;
    const int64_t c1 = ct.total_octs * (b + 1) / ct.grid;
    const int32_t k0 = ct.first[b];
    SumSq acc{{0.f, 0.f}, {0.f, 0.f}, 0.f};
    const uint64_t keep = kKeepL2 ? l2_keep_policy() : 0;
    int32_t k = k0;
    int64_t ob = c0;
    while (ob < c1) {
        const int32_t cnt = ct.T - k < kStaged ? ct.T - k : kStaged;
        __syncthreads();  // every thread is done with the previous span
        for (int i = t; i <= cnt; i += kThreads) sp.lo[i] = __ldg(ct.prefix + k + i);
        for (int i = t; i < cnt; i += kThreads) {
            const TensorRec& r = ct.recs[k + i];
            sp.g[i] = static_cast<char*>(r.g);
            sp.a[i] = static_cast<const char*>(r.m);
            sp.n[i] = r.n;
            sp.vec[i] = r.vec;
        }
        __syncthreads();
        const int64_t oe = sp.lo[cnt] < c1 ? sp.lo[cnt] : c1;
        int32_t j = 0;
        const int64_t first = ob + ((t - (int32_t)((ob - c0) & (kThreads - 1))) & (kThreads - 1));
        for (int64_t o = first; o < oe; o += U * kThreads) {
            RawOctet<G> gr[U], ar[U];
            int32_t ju[U];     // the octet's staged tensor, or -1 past the span
            bool whole[U];     // a whole octet of an aligned tensor: vector accesses
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t q = o + (int64_t)u * kThreads;
                ju[u] = -1;
                whole[u] = false;
                if (q < oe) {
                    while (q >= sp.lo[j + 1]) ++j;
                    ju[u] = j;
                    const int64_t local = q - sp.lo[j];
                    whole[u] = sp.vec[j] && local < sp.n[j] / kOct;
                    if (whole[u]) {
                        load_vec<G>(sp.g[j] + local * kOctBytes, gr[u]);
                        load_vec<G>(sp.a[j] + local * kOctBytes, ar[u]);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (ju[u] < 0) continue;
                const int32_t jj = ju[u];
                const int64_t local = o + (int64_t)u * kThreads - sp.lo[jj];
                float x[8];
                if (whole[u]) {
                    add_octet<G>(gr[u], ar[u]);
                    store_vec<G, kKeepL2>(sp.g[jj] + local * kOctBytes, gr[u], keep);
                    widen_octet<G>(gr[u], x);
                } else {
                    add_octet_elements<G>(sp.g[jj], sp.a[jj], sp.n[jj], local, x);
                }
                acc.add8<kMode>(x, inv_scale);
            }
        }
        ob = oe;
        k += cnt;
    }
    return share_total<G, kMode>(acc, ct, k0, c0, c1, inv_scale);
}

template <Dtype G, int kMode, bool kKeepL2>
__global__ void __launch_bounds__(kThreads, kAccCtasPerSm) accumulate_norm_kernel(ChunkTable ct, float inv_scale,
                                                                           double* __restrict__ partials,
                                                                           unsigned int* ticket, float max_norm,
                                                                           float* d_norm, float* d_factor,
                                                                           double* d_sumsq) {
    __shared__ double red[kWarps];
    __shared__ int last;
    __shared__ AccSpan sp;
    const int t = threadIdx.x;
    wait_prerequisite();  // the kernel queued before may still be writing g or a
    allow_dependents();   // the update queued next may launch and ask L2 for its first data (L2 stays coherent)
    const double mine = accumulate_chunk_share<G, kMode, kKeepL2>(ct, (int32_t)blockIdx.x, inv_scale, sp);
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

template <Dtype G, int kMode, bool kKeepL2>
cudaError_t launch_acc_t(const ChunkTable& ct, cudaStream_t st, float inv_scale, double* partials,
                         unsigned int* ticket, float max_norm, float* d_norm, float* d_factor, double* d_sumsq) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ct.grid > 0 ? ct.grid : 1);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, accumulate_norm_kernel<G, kMode, kKeepL2>, ct, inv_scale, partials, ticket,
                              max_norm, d_norm, d_factor, d_sumsq);
}

template <Dtype G, int kMode>
cudaError_t launch_acc_k(bool keep_l2, const ChunkTable& ct, cudaStream_t st, float inv_scale, double* partials,
                         unsigned int* ticket, float max_norm, float* d_norm, float* d_factor, double* d_sumsq) {
    return keep_l2 ? launch_acc_t<G, kMode, true>(ct, st, inv_scale, partials, ticket, max_norm, d_norm, d_factor,
                                                  d_sumsq)
                   : launch_acc_t<G, kMode, false>(ct, st, inv_scale, partials, ticket, max_norm, d_norm, d_factor,
                                                   d_sumsq);
}

}  // namespace

int launch_accumulate_norm(const ChunkTable& ct, Dtype gdt, float inv_scale, double* partials, unsigned int* ticket,
                           float max_norm, float* d_norm, float* d_factor, double* d_sumsq, bool keep_l2,
                           void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool scaled = inv_scale != 1.0f;
    int ex = 0;  // binary16 times a power of two in [2^-102, 2^111]: every product is an exact normal float32
    const bool pow2 = std::frexp(inv_scale, &ex) == 0.5f && inv_scale >= 0x1p-102f && inv_scale <= 0x1p111f;
    cudaError_t e;
    if (gdt == kF16 && pow2)
        e = launch_acc_k<kF16, kSumHalfPow2>(keep_l2, ct, st, inv_scale, partials, ticket, max_norm, d_norm, d_factor,
                                              d_sumsq);
    else if (gdt == kF16)
        e = launch_acc_k<kF16, kSumScaled>(keep_l2, ct, st, inv_scale, partials, ticket, max_norm, d_norm, d_factor,
                                              d_sumsq);
    else if (scaled)
        e = launch_acc_k<kF32, kSumScaled>(keep_l2, ct, st, inv_scale, partials, ticket, max_norm, d_norm, d_factor,
                                              d_sumsq);
    else
        e = launch_acc_k<kF32, kSumUnscaled>(keep_l2, ct, st, inv_scale, partials, ticket, max_norm, d_norm, d_factor,
                                              d_sumsq);
    count_launches(1);
    return (int)e;
}

}  // namespace mica
