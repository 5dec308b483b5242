// Internal layout shared by the host side (api.cpp: validation, tables, launches) and the kernels (adamw.cu,
// norm.cu, sgd.cu, scale.cu).
//
// A call's tensor list becomes one device table:
//   TensorRec[T]   the four base pointers and the element count of every tensor;
//   WorkItem[I]    the units of work one CTA takes at a time;
// and a norm's list instead becomes
//   TensorRec[T], int64 prefix[T + 1], int32 first[G], double partials[G] and a 32-bit ticket counter
// (see ChunkTable).
//
// Work items are counted in octets (8 consecutive elements: one 32-byte float32 vector, one 16-byte vector of
// binary16 values or of 4 packed BF16 words). A large tensor is cut into slices of `item_octs` octets; runs of
// consecutive small tensors (each at most min(512, item_octs) octets, at most min(1536, 3 item_octs) octets a pack)
// are packed into one item whose octets the CTA's threads share out one by one (the list's pack table holds, per
// pack, the first pack octet of each of its tensors and the pack's total; ScaleTensors instead gives each warp whole
// tensors). Every element belongs to exactly one item, so each element is read and written by exactly one thread per
// launch and the results do not depend on how items are scheduled.
#pragma once

#include <cstdint>

namespace mica {

constexpr int kThreads = 256;  // threads per CTA of every streaming kernel
constexpr int kWarps = kThreads / 32;
constexpr int kOct = 8;        // elements per vector unit

struct TensorRec {
    float* w;      // weights (AdamW, SGD) / the tensor itself (scale) / unused (norm)
    void* g;       // gradient (AdamW, SGD, norm)
    void* m;       // first moment (AdamW) / momentum buffer (SGD with momentum)
    void* v;       // second moment
    int64_t n;     // elements
    int32_t vec;   // 1 when every base pointer is aligned for its octet vector (32 B for float32 streams, 16 B for
                   // binary16 and packed streams): the vector path; 0: the element path
    int32_t group; // AdamW over parameter groups: the tensor's group (0 otherwise)
};
static_assert(sizeof(TensorRec) == 48, "TensorRec layout");

struct WorkItem {
    int32_t t;      // first tensor
    int32_t count;  // 1: octets [o0, min(o0 + item_octs, ceil(n/8))) of tensor t; > 1: tensors t .. t+count-1 whole
    int64_t o0;     // a slice: its first octet; a pack: where its count + 1 entries start in the pack table
};
static_assert(sizeof(WorkItem) == 16, "WorkItem layout");

// A list walked as contiguous chunks of its octet space (the norm's layout): tensor k holds the list's octets
// [prefix[k], prefix[k+1]); CTA b of `grid` takes octets [total*b/grid, total*(b+1)/grid), starting in tensor
// first[b]. Every CTA gets the same number of octets whatever the tensors' sizes.
struct ChunkTable {
    const TensorRec* recs;
    const int64_t* prefix;  // T + 1 entries
    const int32_t* first;   // grid entries
    int32_t T;
    int32_t grid;
    int64_t total_octs;
    int32_t direct;         // 1: the register-streaming kernel (many small tensors); 0: the TMA pipeline
    int32_t pad;
};

// The norm's launch shape. Lists whose tensors average under 512 octets (4,096 elements) are streamed straight into
// registers, one wave of 4 CTAs of 256 threads per SM; others go through the TMA pipeline, 3 CTAs of 288 threads per
// SM, in one wave per 1.5 MB of gradient that a CTA of a single wave would stream (at most 8 waves): equal chunks do
// not take equal times (the 456 CTAs of one wave over GPT-2 XL's 6.2 GB gradient finished between 0.65 and 0.96 ms
// on GB300), and the CTAs of later waves go to whichever SMs free up first, while each wave costs a few
// microseconds of start-up per CTA. Either way no more than one CTA per 256 octets (and at least one, and at most
// max_grid). `oct_bytes`: the bytes of one gradient octet (32 for float32, 16 for binary16).
constexpr int kNormDirectCtasPerSm = 4;
constexpr int kNormTmaCtasPerSm = 3;
constexpr int kNormTmaMaxWaves = 8;
constexpr int64_t kNormWaveBytes = 1536 * 1024;
inline void choose_norm_shape(int64_t total_octs, int64_t nonempty_tensors, int oct_bytes, int sms,
                              int32_t max_grid, int32_t* grid, int32_t* direct) {
    *direct = (nonempty_tensors > 0 && total_octs < 512 * nonempty_tensors) ? 1 : 0;
    int64_t g = (int64_t)(*direct ? kNormDirectCtasPerSm : kNormTmaCtasPerSm) * (sms > 0 ? sms : 1);
    if (!*direct) {
        int64_t waves = total_octs * oct_bytes / g / kNormWaveBytes;
        waves = waves < 1 ? 1 : (waves > kNormTmaMaxWaves ? kNormTmaMaxWaves : waves);
        g *= waves;
    }
    const int64_t want = total_octs > 256 ? (total_octs + 255) / 256 : 1;
    if (g > want) g = want;
    if (g > max_grid) g = max_grid;
    *grid = (int32_t)(g > 0 ? g : 1);
}

// The step's float32 scalars, each computed in double on the host and rounded once.
struct StepScalars {
    float c1;        // 1 - beta1
    float b2;        // beta2
    float c2;        // 1 - beta2
    float neg_step;  // -(lr / (1 - beta1^t))
    float bc2;       // sqrt(1 - beta2^t)
    float dec;       // 1 - lr * weight_decay (AdamW's decoupled decay)
    float eps;       // eps
    float wd;        // weight_decay (Adam's coupled L2 term)
    int32_t zero_grad;
    int32_t skip_nonfinite;  // leave w, m, v as they are when the factor is not > 0
};

// Parameter groups (PyTorch's param_groups): per group, the scalars that depend on its lr and weight decay. The
// other scalars are the same for every group.
constexpr int kMaxGroups = 8;
struct GroupScalars {
    float neg_step[kMaxGroups];
    float dec[kMaxGroups];
    float wd[kMaxGroups];
};

// SGD and SGD with momentum, float32 scalars rounded once from the host's doubles.
struct SgdScalars {
    float neg_lr;    // -lr
    float mu;        // momentum
    int32_t zero_grad;
    int32_t pad;
};

// kBF16x2M (moments only): m packed as kBF16x2, v float32
enum Dtype : int32_t { kF32 = 0, kF16 = 1, kBF16x2 = 2, kBF16x2M = 3 };

// The tables of an update launch (AdamW, SGD): a persistent grid of at most `sms` x (CTAs that fit on an SM) takes
// the items from `queue` (two counters, zero before the launch, left zero by it; launches that may overlap need
// different queues), or, with `queue` null, one CTA per item.
struct UpdateLaunch {
    const TensorRec* recs;
    const WorkItem* items;
    const int32_t* pack_pre;
    unsigned int* queue;
    int32_t num_items;
    int32_t item_octs;
    int32_t sms;
};

// The grid of a persistent update launch.
inline int32_t persistent_grid(int32_t num_items, int per_sm, int sms) {
    const int64_t cap = (int64_t)(per_sm > 0 ? per_sm : 1) * (sms > 0 ? sms : 1);
    return (int32_t)(num_items < cap ? num_items : cap);
}

// Kernel launchers (adamw.cu, sgd.cu, norm.cu, scale.cu). Each returns the cudaError_t of its launch as an int.
// AdamW (or, with `coupled`, Adam with the coupled L2 term) over every item. It is launched as a programmatic
// dependent of the kernel queued before it: it may start while that kernel finishes and ask L2 for its first item's
// data, but reads w, g, m, v and d_factor only once that kernel has completed. With `groups`, tensor k takes
// neg_step, dec and wd from entry recs[k].group of it instead of from s.
int launch_adamw(const UpdateLaunch& u, Dtype gdt, Dtype mdt, bool coupled, const StepScalars& s,
                 const GroupScalars* groups, const float* d_factor, void* stream);
// SGD (momentum false) or SGD with momentum over every item, launched as AdamW is. `skip`: leave w (and the
// buffer) as they are when the factor is not > 0.
int launch_sgd(const UpdateLaunch& u, Dtype gdt, bool momentum, bool skip, const SgdScalars& s,
               const float* d_factor, void* stream);
// The joint norm in one launch of ct.grid CTAs: one partial square sum per CTA into `partials` (ct.grid doubles),
// and the CTA that finishes last sums them in a fixed order and writes norm and factor. `ticket` must be 0 before
// the launch; the kernel leaves it 0.
// d_norm, d_factor and d_sumsq (the square sum itself, in double) are each written when not null. keep_l2: the
// gradient's loads (and bulk copies) carry an evict-last L2 policy, so that the update that follows reads the
// gradient from L2 (for gradients that fit in it, see kKeepL2MaxGradBytes).
int launch_norm(const ChunkTable& ct, Dtype gdt, float inv_scale, double* partials, unsigned int* ticket,
                float max_norm, float* d_norm, float* d_factor, double* d_sumsq, bool keep_l2, void* stream);
// Norm and factor from `count` partial square sums (one per rank of a sharded list), added in index order in double;
// one thread of one CTA.
int launch_factor_from_sumsq(const double* parts, int32_t count, float max_norm, float inv_scale, float* d_norm,
                             float* d_factor, void* stream);
// Gradient bytes up to which the norm asks L2 to keep the gradient for the update (GB300 has 126 MB of L2; the
// update's own streams pass through it with evict-first hints). Larger gradients would only push the update's
// other streams out.
constexpr int64_t kKeepL2MaxGradBytes = (int64_t)96 << 20;
int launch_scale(const TensorRec* recs, const WorkItem* items, int32_t num_items, int32_t item_octs, Dtype dt,
                 float factor, const float* d_factor, void* stream);

// The gradient's last write fused with the norm (accnorm.cu): for every tensor k of ct, g += a (g in recs[k].g, the
// addend in recs[k].m, each sum rounded to the gradient's type), and the joint norm and factor of the result, as
// launch_norm computes them (one partial per CTA into `partials`, the CTA that finishes last writing d_norm,
// d_factor and d_sumsq, each when not null). ct is laid out as for the register-streaming norm, with ct.grid CTAs from
// choose_accumulate_grid. keep_l2: the new gradient's stores carry an evict-last L2 policy (for gradients that fit
// in L2, which the update reads next).
int launch_accumulate_norm(const ChunkTable& ct, Dtype gdt, float inv_scale, double* partials, unsigned int* ticket,
                           float max_norm, float* d_norm, float* d_factor, double* d_sumsq, bool keep_l2,
                           void* stream);
constexpr int kAccCtasPerSm = 4;
// kAccCtasPerSm CTAs per SM in one wave per 192 KB of gradient that a CTA of a single wave would take, from 2 to 8
// waves (measured on GB300: the loss-scaled list's 76 MB best in 2 waves, GPT-2 small's 498 MB in 4, GPT-2 XL's
// 6.2 GB in 8), no more than one CTA per 256 octets and at least one. `oct_bytes`: one gradient octet's bytes.
constexpr int64_t kAccWaveBytes = 192 * 1024;
inline int32_t choose_accumulate_grid(int64_t total_octs, int oct_bytes, int sms) {
    const int64_t wave = (int64_t)kAccCtasPerSm * (sms > 0 ? sms : 1);
    int64_t waves = total_octs * oct_bytes / wave / kAccWaveBytes;
    waves = waves < 2 ? 2 : (waves > 8 ? 8 : waves);
    const int64_t g = wave * waves;
    const int64_t want = total_octs > 256 ? (total_octs + 255) / 256 : 1;
    return (int32_t)(g < want ? g : want);
}

// The norm and the AdamW update in one cooperative launch of ct.grid CTAs (fused.cu): CTA b sums the squares of
// chunk b of ct (the register-streaming layout, ct.first holding ct.grid entries) into partials[b]; the CTAs meet
// at a bounded grid-wide wait on `bar` (two words, zero before the first launch, left ready by each); every CTA then
// computes norm and factor from the partials in a fixed order (CTA 0 writes them to d_norm, when not null, and
// d_factor), and the grid runs the update's items from u's queue (not null) with that factor. Returns
// cudaErrorCooperativeLaunchTooLarge, having queued nothing, when ct.grid CTAs of the instantiation cannot all be
// resident at once.
int launch_clip_adamw(const ChunkTable& ct, double* partials, unsigned int* bar, const UpdateLaunch& u, Dtype gdt,
                      Dtype mdt, bool coupled, const StepScalars& s, float max_norm, float inv_scale, float* d_norm,
                      float* d_factor, void* stream);
constexpr int kFusedCtasPerSm = 3;

// One CTA whose bounded mbarrier wait runs out after `polls` rounds (nothing arrives) and sets the status word.
int launch_wait_selftest(uint32_t polls, void* stream);
// One CTA whose grid-wide wait for a second CTA (never launched) runs out after `polls` polls and sets the fused
// kernels' status word.
int launch_grid_wait_selftest(uint32_t polls, void* stream);

// The device's pipeline status word: nonzero when a kernel's bounded wait on a shared-memory barrier gave up (the
// kernel then stopped early and its results are not valid). Reads it (synchronously) and clears it.
int read_device_status(unsigned int* status);
// The same for the fused kernels' grid-wide waits.
int read_fused_status(unsigned int* status);

// kernels queued so far (incremented by the launchers)
void count_launches(uint64_t k);

// sets the calling thread's one-line error detail (what mica_last_error_detail returns)
void set_error_detail(const char* msg);

}  // namespace mica
