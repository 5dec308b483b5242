// Device code of the AdamW update shared by the kernels that run it (adamw.cu: the update alone; fused.cu: the
// norm and the update in one cooperative launch): packed BF16 moments, the per-octet update in registers, the
// slice and pack walks, L2 prefetch of an item, and the persistent grids' item loop.
//
// Per-element arithmetic follows BendTorch "main.bend", section "Optimizers": every float32 operation is a separate
// correctly rounded intrinsic (__fmul_rn, __fadd_rn, __fdiv_rn, __fsqrt_rn), which the compiler never fuses into an
// FMA, in the order that section gives; so the update is bit-identical to the same step on the CPU.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "plan.h"
#include "stream.cuh"

namespace mica {
namespace {

// ------------------------------------------------------------------------------------------------------------------
// packed BF16 (BendTorch "main.bend", "AdamW over packed BF16 moments"): element 2k is the low half of word k
// ------------------------------------------------------------------------------------------------------------------

__device__ __forceinline__ float bf16_lo(uint32_t word) { return __uint_as_float(word << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t word) { return __uint_as_float(word & 0xFFFF0000u); }

__device__ __forceinline__ void bf8_to(const uint4& x, float (&a)[8]) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        a[2 * k] = bf16_lo(w[k]);
        a[2 * k + 1] = bf16_hi(w[k]);
    }
}

// Two float32 -> one word, each rounded to nearest-even by the hardware conversion; a NaN is stored as 0xFFFF.
__device__ __forceinline__ uint32_t pack_bf16x2(float even, float odd) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(odd), "f"(even));  // first source -> high half
    if (even != even) r |= 0x0000FFFFu;
    if (odd != odd) r |= 0xFFFF0000u;
    return r;
}

// ------------------------------------------------------------------------------------------------------------------
// AdamW on one octet, in registers
// ------------------------------------------------------------------------------------------------------------------

// Which moments a moment type stores as packed BF16 words, and the bytes of one octet of each.
template <Dtype M>
struct MomentLayout {
    static constexpr bool kMPacked = (M == kBF16x2 || M == kBF16x2M);
    static constexpr bool kVPacked = (M == kBF16x2);
    static constexpr int kMb = kMPacked ? 16 : 32;
    static constexpr int kVb = kVPacked ? 16 : 32;
};

// m, v hold the moments read (float32, or the exact widening of the stored BF16); on return they hold the new
// moments as the weight update reads them (rounded through BF16 where stored packed), and pm, pv the packed words to
// store. kCoupled is Adam's coupled L2 form (g + w * wd, no decoupled decay).
template <Dtype M, bool kCoupled>
__device__ __forceinline__ void adam8(float (&w)[8], const float (&g)[8], float (&m)[8], float (&v)[8],
                                      uint32_t (&pm)[4], uint32_t (&pv)[4], const StepScalars& s, float f) {
    using L = MomentLayout<M>;
    float wdec[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float gh = __fmul_rn(g[j], f);
        if constexpr (kCoupled) {
            gh = __fadd_rn(gh, __fmul_rn(w[j], s.wd));
            wdec[j] = w[j];
        } else {
            wdec[j] = __fmul_rn(w[j], s.dec);
        }
        m[j] = __fadd_rn(m[j], __fmul_rn(s.c1, __fsub_rn(gh, m[j])));
        v[j] = __fadd_rn(__fmul_rn(v[j], s.b2), __fmul_rn(__fmul_rn(s.c2, gh), gh));
    }
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        if constexpr (L::kMPacked) {
            pm[p] = pack_bf16x2(m[2 * p], m[2 * p + 1]);
            m[2 * p] = bf16_lo(pm[p]);
            m[2 * p + 1] = bf16_hi(pm[p]);
        }
        if constexpr (L::kVPacked) {
            pv[p] = pack_bf16x2(v[2 * p], v[2 * p + 1]);
            v[2 * p] = bf16_lo(pv[p]);
            v[2 * p + 1] = bf16_hi(pv[p]);
        }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float denom = __fadd_rn(__fdiv_rn(__fsqrt_rn(v[j]), s.bc2), s.eps);
        w[j] = __fadd_rn(wdec[j], __fdiv_rn(__fmul_rn(s.neg_step, m[j]), denom));
    }
}

// One packed-moment octet's 4 words, element by element (words past the tensor's last element are not read).
__device__ __forceinline__ void load_words(const void* base, int64_t o, int cnt, uint32_t (&word)[4],
                                           float (&x)[8]) {
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        if (2 * p < cnt) {
            word[p] = static_cast<const uint32_t*>(base)[4 * o + p];
            x[2 * p] = bf16_lo(word[p]);
            x[2 * p + 1] = bf16_hi(word[p]);
        }
    }
}

// ... and back: the high half of a word that holds no element keeps what it held.
__device__ __forceinline__ void store_words(void* base, int64_t o, int cnt, const uint32_t (&old)[4],
                                            const uint32_t (&word)[4]) {
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        if (2 * p < cnt) {
            uint32_t x = word[p];
            if (2 * p + 1 >= cnt) x = (x & 0x0000FFFFu) | (old[p] & 0xFFFF0000u);
            static_cast<uint32_t*>(base)[4 * o + p] = x;
        }
    }
}

// One octet element by element: for bases not aligned for the vectors, and for a tensor's last, partial octet.
// Elements past n are neither read nor written, nor is the high half of a last packed word that holds no element.
template <Dtype G, Dtype M, bool kCoupled, bool kSkip>
__device__ __noinline__ void adam_oct_elements(const TensorRec& r, int64_t o, const StepScalars& s, Factor& fac) {
    using L = MomentLayout<M>;
    const int64_t i0 = o * kOct;
    const int64_t left = r.n - i0;
    const int cnt = left < kOct ? (int)left : kOct;
    float w[8], g[8], m[8], v[8];
    uint32_t om[4], ov[4], pm[4], pv[4];
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = g[j] = m[j] = v[j] = 0.f;
#pragma unroll
    for (int p = 0; p < 4; ++p) om[p] = ov[p] = pm[p] = pv[p] = 0u;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if (j < cnt) {
            w[j] = r.w[i0 + j];
            g[j] = (G == kF16) ? __half2float(static_cast<const __half*>(r.g)[i0 + j])
                               : static_cast<const float*>(r.g)[i0 + j];
            if constexpr (!L::kMPacked) m[j] = static_cast<const float*>(r.m)[i0 + j];
            if constexpr (!L::kVPacked) v[j] = static_cast<const float*>(r.v)[i0 + j];
        }
    }
    if constexpr (L::kMPacked) load_words(r.m, o, cnt, om, m);
    if constexpr (L::kVPacked) load_words(r.v, o, cnt, ov, v);
    const float f = fac.get();
    const bool skip = skip_step<kSkip>(f);
    if (!skip) adam8<M, kCoupled>(w, g, m, v, pm, pv, s, f);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if (j < cnt) {
            if (!skip) {
                r.w[i0 + j] = w[j];
                if constexpr (!L::kMPacked) static_cast<float*>(r.m)[i0 + j] = m[j];
                if constexpr (!L::kVPacked) static_cast<float*>(r.v)[i0 + j] = v[j];
            }
            if (s.zero_grad) {
                if (G == kF16) static_cast<__half*>(r.g)[i0 + j] = __ushort_as_half(0);
                else static_cast<float*>(r.g)[i0 + j] = 0.f;
            }
        }
    }
    if (!skip) {
        if constexpr (L::kMPacked) store_words(r.m, o, cnt, om, pm);
        if constexpr (L::kVPacked) store_words(r.v, o, cnt, ov, pv);
    }
}

// The four streams of octets [a, b) of tensor r into L2 (a < b, whole octets of an aligned tensor).
template <Dtype G, Dtype M>
__device__ __forceinline__ void prefetch_octets(const TensorRec& r, int64_t a, int64_t b) {
    using L = MomentLayout<M>;
    constexpr int kGb = (G == kF16) ? 16 : 32;
    const uint32_t n = (uint32_t)(b - a);
    prefetch_l2(reinterpret_cast<const char*>(r.w) + a * 32, n * 32);
    prefetch_l2(static_cast<const char*>(r.g) + a * kGb, n * kGb);
    prefetch_l2(static_cast<const char*>(r.m) + a * L::kMb, n * L::kMb);
    prefetch_l2(static_cast<const char*>(r.v) + a * L::kVb, n * L::kVb);
}

// One whole octet of a tensor whose bases are aligned for the vectors: 256-bit loads (128-bit for binary16 g and
// packed moments), the update in registers, 256-bit streaming stores.
template <Dtype G, Dtype M, bool kCoupled, bool kSkip>
__device__ __forceinline__ void adam_vec_octet(const TensorRec& r, int64_t o, const StepScalars& s, Factor& fac) {
    using L = MomentLayout<M>;
    float w[8], g[8], m[8], v[8];
    uint4 gh, mp, vp;
    ld8_stream(r.w + kOct * o, w);
    if constexpr (G == kF16) gh = ld16_stream(static_cast<const __half*>(r.g) + kOct * o);
    else ld8_stream(static_cast<const float*>(r.g) + kOct * o, g);
    if constexpr (L::kMPacked) mp = ld16_stream(static_cast<const uint32_t*>(r.m) + 4 * o);
    else ld8_stream(static_cast<const float*>(r.m) + kOct * o, m);
    if constexpr (L::kVPacked) vp = ld16_stream(static_cast<const uint32_t*>(r.v) + 4 * o);
    else ld8_stream(static_cast<const float*>(r.v) + kOct * o, v);
    const float f = fac.get();
    if (!skip_step<kSkip>(f)) {
        uint32_t pm[4], pv[4];
        if constexpr (G == kF16) h8_to(gh, g);
        if constexpr (L::kMPacked) bf8_to(mp, m);
        if constexpr (L::kVPacked) bf8_to(vp, v);
        adam8<M, kCoupled>(w, g, m, v, pm, pv, s, f);
        st8(r.w + kOct * o, w);
        if constexpr (L::kMPacked) st16(static_cast<uint32_t*>(r.m) + 4 * o, make_uint4(pm[0], pm[1], pm[2], pm[3]));
        else st8(static_cast<float*>(r.m) + kOct * o, m);
        if constexpr (L::kVPacked) st16(static_cast<uint32_t*>(r.v) + 4 * o, make_uint4(pv[0], pv[1], pv[2], pv[3]));
        else st8(static_cast<float*>(r.v) + kOct * o, v);
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

// Octets [ob, oe) of one tensor: octet ob + lane first, then every `stride`-th. With `prefetch` (a whole CTA on
// one slice: lane is the thread index and stride the CTA size) thread 0 asks L2 for the rounds one and two ahead,
// so that the other threads' loads of those rounds find their data in L2 rather than waiting on DRAM, and, at the
// slice's second-to-last round, for the first round of `nx`, the slice the CTA takes next.
// The item a CTA takes after the current one, whose first round of octets (when it is a slice) the CTA's thread 0
// asks L2 for while the CTA works on the current slice's last round, as it does for the current slice's own rounds.
struct NextSlice {
    const TensorRec* recs;
    const WorkItem* item;  // null: none, or no prefetch of the next item
};

template <Dtype G, Dtype M>
__device__ __noinline__ void prefetch_next_round(const NextSlice& nx, int32_t round) {
    const WorkItem it = *nx.item;
    if (it.count != 1) return;
    const TensorRec r = nx.recs[it.t];
    const int64_t full = r.n / kOct;
    const int64_t oe = it.o0 + round < full ? it.o0 + round : full;
    if (r.vec && oe > it.o0) prefetch_octets<G, M>(r, it.o0, oe);
}

template <Dtype G, Dtype M, bool kCoupled, bool kSkip>
__device__ __forceinline__ void adam_range(const TensorRec& r, int64_t ob, int64_t oe, int lane, int stride,
                                           const StepScalars& s, Factor& fac, bool prefetch = false,
                                           NextSlice nx = NextSlice{nullptr, nullptr}) {
    using L = MomentLayout<M>;
    const int64_t full = r.n / kOct;  // octets with all eight elements
    if (r.vec) {
        const int64_t vend = oe < full ? oe : full;
        const int64_t round = stride;
        if (prefetch && lane == 0 && ob + round < vend)
            prefetch_octets<G, M>(r, ob + round, ob + 2 * round < vend ? ob + 2 * round : vend);
        for (int64_t o = ob + lane; o < vend; o += round) {
            if (prefetch && lane == 0) {
                if (o + 2 * round < vend) {
                    prefetch_octets<G, M>(r, o + 2 * round, o + 3 * round < vend ? o + 3 * round : vend);
                } else if (nx.item && o + round < vend) {  // the second-to-last round: the next slice's first
                    prefetch_next_round<G, M>(nx, (int32_t)round);
                }
            }
            adam_vec_octet<G, M, kCoupled, kSkip>(r, o, s, fac);
        }
        // the last, partial octet (n % 8 != 0), when it lies in this range
        if (full < oe && full >= ob && lane == (int)((full - ob) % stride))
            adam_oct_elements<G, M, kCoupled, kSkip>(r, full, s, fac);
    } else {
        for (int64_t o = ob + lane; o < oe; o += stride) adam_oct_elements<G, M, kCoupled, kSkip>(r, o, s, fac);
    }
}

// The scalars of tensor r: with kGrouped its group's neg_step, dec and wd replace those of s (the rest is shared).
template <bool kGrouped>
__device__ __forceinline__ StepScalars group_scalars(const StepScalars& s, const GroupScalars& gs,
                                                     const TensorRec& r) {
    StepScalars x = s;
    if constexpr (kGrouped) {
        x.neg_step = gs.neg_step[r.group];
        x.dec = gs.dec[r.group];
        x.wd = gs.wd[r.group];
    }
    return x;
}

// A pack of small tensors (t .. t+count-1, whole): their octets are spread over the CTA's threads, thread i taking
// pack octets i, i + 256, ..., so that every thread has work however small the tensors are. The pack numbers the
// whole octets of its aligned tensors first, then the octets taken element by element (see the pack table in
// plan.h), so that the two kinds seldom share a warp; a thread finds its octet's tensor by binary search from the
// last one it found. The CTA first asks L2 for the pack's whole octets.
template <Dtype G, Dtype M, bool kCoupled, bool kSkip, bool kGrouped>
__device__ __forceinline__ void adam_pack(const TensorRec* __restrict__ recs, const WorkItem& item,
                                          const int32_t* __restrict__ pack_pre, const StepScalars& s,
                                          const GroupScalars& gs, Factor& fac) {
    const int32_t* pre_w = pack_pre + item.o0;        // whole octets: count + 1 entries
    const int32_t* pre_e = pre_w + item.count + 1;   // the others: count + 1 entries
    for (int32_t i = threadIdx.x; i < item.count; i += kThreads) {
        const TensorRec r = recs[item.t + i];
        if (r.vec && r.n >= kOct) prefetch_octets<G, M>(r, 0, r.n / kOct);
    }
    const int32_t total_w = __ldg(pre_w + item.count);
    const int32_t total = total_w + __ldg(pre_e + item.count);
    int32_t jw = 0, je = 0;
    for (int32_t q = threadIdx.x; q < total; q += kThreads) {
        const bool whole = q < total_w;
        int64_t o;
        TensorRec r;
        if (whole) {
            jw = pack_search(pre_w, jw, item.count, q);
            r = recs[item.t + jw];
            o = q - __ldg(pre_w + jw);
        } else {
            const int32_t qe = q - total_w;
            je = pack_search(pre_e, je, item.count, qe);
            r = recs[item.t + je];
            o = (r.vec ? r.n / kOct : 0) + (qe - __ldg(pre_e + je));
        }
        if constexpr (kGrouped) {
            const StepScalars x = group_scalars<kGrouped>(s, gs, r);
            if (whole) adam_vec_octet<G, M, kCoupled, kSkip>(r, o, x, fac);
            else adam_oct_elements<G, M, kCoupled, kSkip>(r, o, x, fac);
        } else {
            if (whole) adam_vec_octet<G, M, kCoupled, kSkip>(r, o, s, fac);
            else adam_oct_elements<G, M, kCoupled, kSkip>(r, o, s, fac);
        }
    }
}

// L2 prefetch of one item's whole octets: the slice's, or every tensor of the pack (one tensor a thread).
template <Dtype G, Dtype M>
__device__ __forceinline__ void prefetch_item(const TensorRec* __restrict__ recs, const WorkItem& item,
                                              int32_t item_octs) {
    if (item.count == 1) {
        if (threadIdx.x == 0) {
            const TensorRec r = recs[item.t];
            const int64_t full = r.n / kOct;
            const int64_t oe = item.o0 + item_octs < full ? item.o0 + item_octs : full;
            if (r.vec && oe > item.o0) prefetch_octets<G, M>(r, item.o0, oe);
        }
    } else {
        for (int32_t i = threadIdx.x; i < item.count; i += kThreads) {
            const TensorRec r = recs[item.t + i];
            if (r.vec && r.n >= kOct) prefetch_octets<G, M>(r, 0, r.n / kOct);
        }
    }
}

// The items of a persistent grid (or, with no queue, the CTA's one item), the first index already in s_item[0]:
// taken one at a time from the end of the item array (the norm reads the list forwards, so the gradient it read
// last may still be in L2), thread 0 taking the next index while the CTA works on the current item (and, with both
// moments packed, asking L2 for that item's first round before the current slice ends). Without
// kGrouped the scalars come straight from s; with it each tensor's group picks its own from gs.
template <Dtype G, Dtype M, bool kCoupled, bool kSkip, bool kGrouped>
__device__ __forceinline__ void adamw_item_loop(const TensorRec* __restrict__ recs, const WorkItem* __restrict__ items,
                                                int32_t num_items, int32_t item_octs,
                                                const int32_t* __restrict__ pack_pre, unsigned int* queue,
                                                const StepScalars& s, const GroupScalars& gs, Factor& fac,
                                                int32_t* s_item) {
    const bool persistent = queue != nullptr;
    int32_t cur = 0;
    for (int32_t k = s_item[0]; k < num_items; k = s_item[cur]) {
        NextSlice nx{recs, nullptr};
        if (threadIdx.x == 0) {
            const int32_t nk = persistent ? queue_take(queue) : num_items;
            s_item[cur ^ 1] = nk;
            // measured on GB300: with both moments packed (160-byte octets) the next slice's first round is asked
            // for early (GPT-2 small's step 0.465 -> 0.458 ms, GPT-2 XL's 5.41 -> 5.32 ms); with float32 moments
            // (224-byte octets) the extra data in L2 made the step slower, and with m packed alone it changed nothing
            if (MomentLayout<M>::kVPacked && nk < num_items) nx.item = items + (num_items - 1 - nk);
        }
        const WorkItem item = items[num_items - 1 - k];
        if (item.count == 1) {
            const TensorRec r = recs[item.t];
            const int64_t no = (r.n + kOct - 1) / kOct;
            const int64_t oe = item.o0 + item_octs < no ? item.o0 + item_octs : no;
            if constexpr (kGrouped) {
                const StepScalars x = group_scalars<kGrouped>(s, gs, r);
                adam_range<G, M, kCoupled, kSkip>(r, item.o0, oe, threadIdx.x, kThreads, x, fac, true, nx);
            } else {
                adam_range<G, M, kCoupled, kSkip>(r, item.o0, oe, threadIdx.x, kThreads, s, fac, true, nx);
            }
        } else {
            adam_pack<G, M, kCoupled, kSkip, kGrouped>(recs, item, pack_pre, s, gs, fac);
        }
        __syncthreads();  // the next item's index is in s_item[cur ^ 1]; this one's slot may be reused
        cur ^= 1;
    }
}

}  // namespace
}  // namespace mica
