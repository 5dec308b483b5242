// Internal layout shared by the host plan builder (plan.cpp) and the kernels (kernels.cu).
//
// A call's tensor list becomes one device table:
//   TensorRec[T]   the four base pointers and the element count of every tensor;
//   WorkItem[I]    the units of work one CTA takes at a time;
//   double[I]      (norm plans only) one partial square sum per work item.
//
// Work items are counted in quads (4 consecutive elements, one 16-byte float32 vector). A large tensor is cut into
// slices of `item_quads` quads; runs of consecutive small tensors (each at most item_quads / 2 quads) are packed
// into one item whose tensors the CTA's warps share out. Every element belongs to exactly one item, so each element
// is read and written by exactly one thread per launch and the results do not depend on how items are scheduled.
#pragma once

#include <cstdint>

namespace mica {

constexpr int kThreads = 256;  // threads per CTA of every streaming kernel
constexpr int kWarps = kThreads / 32;

struct TensorRec {
    float* w;      // weights (AdamW) / the tensor itself (scale) / unused (norm)
    void* g;       // gradient (AdamW, norm)
    void* m;       // first moment
    void* v;       // second moment
    int64_t n;     // elements
    int32_t vec;   // 1 when every base pointer is 16-byte aligned (the quad-vector path); 0: element path
    int32_t pad;
};
static_assert(sizeof(TensorRec) == 48, "TensorRec layout");

struct WorkItem {
    int32_t t;      // first tensor
    int32_t count;  // 1: quads [q0, min(q0 + item_quads, ceil(n/4))) of tensor t; > 1: tensors t .. t+count-1 whole
    int64_t q0;     // first quad of a slice (0 for a pack)
};
static_assert(sizeof(WorkItem) == 16, "WorkItem layout");

// The step's float32 scalars, each computed in double on the host and rounded once.
struct StepScalars {
    float c1;        // 1 - beta1
    float b2;        // beta2
    float c2;        // 1 - beta2
    float neg_step;  // -(lr / (1 - beta1^t))
    float bc2;       // sqrt(1 - beta2^t)
    float dec;       // 1 - lr * weight_decay
    float eps;       // eps
    int32_t zero_grad;
};

enum Dtype : int32_t { kF32 = 0, kF16 = 1, kBF16x2 = 2 };

// Kernel launchers (kernels.cu). Each returns the cudaError_t of its launch as an int.
int launch_adamw(const TensorRec* recs, const WorkItem* items, int32_t num_items, int32_t item_quads, Dtype gdt,
                 Dtype mdt, const StepScalars& s, const float* d_factor, void* stream);
int launch_norm(const TensorRec* recs, const WorkItem* items, int32_t num_items, int32_t item_quads, Dtype gdt,
                float inv_scale, double* partials, float max_norm, float* d_norm, float* d_factor, void* stream);
int launch_scale(const TensorRec* recs, const WorkItem* items, int32_t num_items, int32_t item_quads, Dtype dt,
                 float factor, const float* d_factor, void* stream);

// kernels queued so far (incremented by the launchers)
void count_launches(uint64_t k);

}  // namespace mica
