/*
 * mica_optim: the clip + AdamW optimizer step on one GB300 (sm_103a), as a C ABI.
 *
 * Three verbs, named for those of the Mica 7.7 release note ("Mica 7.7: a training step on the card, in every float
 * type", section "The whole model in one call"):
 *
 *   mica_scale_tensors    ScaleTensors: each element of each listed tensor times one factor (a float16 step's
 *                         unscale).
 *   mica_clip_grad_norms  ClipGradNorms: the joint L2 norm of every listed gradient and the clip factor, both left
 *                         in device memory ("Values that stay on the card"); the gradients are not rewritten.
 *   mica_adamw_steps      AdamWSteps: AdamW over every (w, g, m, v) group in one launch, each group updated exactly
 *                         as a single-group step would update it.
 *
 * and, over the same lists, the other optimizer steps of BendTorch "main.bend", section "Optimizers":
 *
 *   mica_adamw_steps_grouped  AdamWSteps over a list split into parameter groups (PyTorch's param_groups) with
 *                             their own lr and weight decay, still one launch.
 *   mica_sgd_steps            SGD, and SGD with momentum, over every (w, g[, buf]) group in one launch.
 *
 * and mica_accumulate_clip_grad_norms, ClipGradNorms fused into the gradient's last write when that write is an
 * add (a gradient with several contributions), so that the norm reads no gradient a second time.
 *
 * The per-element arithmetic is BendTorch "main.bend", section "Optimizers" (AdamW in PyTorch's order of operations;
 * the part "AdamW over packed BF16 moments (CAdamWBF16)" for packed moments), with PyTorch's scalars:
 *   step = lr / (1 - beta1^t), bc2 = sqrt(1 - beta2^t), decay w *= 1 - lr*wd,
 * each computed in double on the host and rounded once to float32.
 *
 * Conventions shared by every entry point:
 *   - Pointer arrays (`w`, `g`, `m`, `v`, `t`) are HOST arrays of DEVICE pointers; `n` is a host array of element
 *     counts. The library reads them during the call only and keeps no reference to the host arrays.
 *   - Every tensor buffer belongs to the caller and must be device memory of the current CUDA device. The library
 *     never allocates per call; it allocates once, per distinct tensor list, a small device table (tensor records,
 *     work items and, for the norms, one double per CTA), kept until mica_release_cache().
 *   - Work is queued on `stream` (a cudaStream_t; NULL is the legacy default stream) and returns at once. Calls that
 *     share a tensor list must be ordered on one stream: they share that list's cached table.
 *   - Validation happens on the host before anything is queued; a call that returns an error has queued nothing.
 *     A fault of earlier queued work surfaces as MICA_ERR_CUDA from a later call or from mica_sync(). With the
 *     environment variable MICA_SYNC_DEBUG=1 every call waits for its own kernels, so a fault is reported by the
 *     call that caused it.
 *   - Two more environment variables tune the update kernels and never change a result: MICA_ITEM_OCTS (a power of
 *     two from 16 to 2^20, read when a list's table is built) replaces the octets per work item, and
 *     MICA_UPDATE_GRID=items (read at each call) runs one CTA per work item instead of the persistent grid.
 *   - A tensor with n[i] == 0 is skipped and its pointers may be NULL. T == 0 is allowed.
 *   - mica_last_error_detail() gives a one-line description of the last error on the calling thread.
 */
#ifndef MICA_OPTIM_H
#define MICA_OPTIM_H

#include <stdint.h>

#if defined(__GNUC__)
#define MICA_API __attribute__((visibility("default")))
#else
#define MICA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MICA_OK = 0,
    MICA_ERR_NULL = 1,     /* a required pointer (array, tensor with n > 0, output, hp) is NULL */
    MICA_ERR_COUNT = 2,    /* T < 0 or T > MICA_MAX_TENSORS, or some n[i] < 0 */
    MICA_ERR_DTYPE = 3,    /* an element type the call does not take */
    MICA_ERR_HYPER = 4,    /* lr, eps, weight_decay, step, max_norm, inv_scale or factor out of range / not finite */
    MICA_ERR_BETA = 5,     /* beta1 or beta2 outside [0, 1), or NaN */
    MICA_ERR_OVERLAP = 6,  /* two buffers the call writes (or one it writes and one it reads) overlap */
    MICA_ERR_DEVICE = 7,   /* no usable CUDA device */
    MICA_ERR_ADDRESS = 8,  /* a pointer is not device memory of the current device, is not aligned to its element,
                              or its extent runs past the end of its allocation */
    MICA_ERR_CUDA = 9,     /* a CUDA call failed, including a fault of earlier queued work */
    MICA_ERR_NOMEM = 10,   /* the per-list device table could not be allocated */
    MICA_ERR_CAPTURE = 11  /* the call was refused because `stream` is capturing work into a CUDA graph (only
                              mica_clip_grad_norms_noalloc refuses this; see there) */
} mica_status;

/* Element types.
 *   MICA_F32       float32.
 *   MICA_F16       IEEE binary16 (gradients, and tensors of mica_scale_tensors).
 *   MICA_BF16X2    packed BF16 moments: a tensor of n elements is ceil(n/2) uint32 words; element 2k is the low 16
 *                  bits of word k and element 2k+1 the high 16 bits (BendTorch "main.bend", section "The layer
 *                  protocol", the PTree comment). Rounding into it is to nearest, ties to even; a NaN is stored as
 *                  0xFFFF. For odd n the high half of the last word is never written.
 *   MICA_BF16X2_M  moments only: m packed as MICA_BF16X2, v float32 (the same page's CAdamWBF16 with v16 false). */
typedef enum { MICA_F32 = 0, MICA_F16 = 1, MICA_BF16X2 = 2, MICA_BF16X2_M = 3 } mica_dtype;

/* mica_adamw_hp.flags */
#define MICA_STEP_SKIP_NONFINITE 1u /* leave w, m and v as they are when the factor read from d_factor is not > 0:
                                       the norm of the unscaled gradient was NaN or infinite (a float16 step that
                                       overflowed; the caller then lowers its loss scale). The gradient is still
                                       zeroed when zero_grad asks for it. */
#define MICA_STEP_COUPLED_L2 2u     /* Adam with the coupled L2 term instead of AdamW's decoupled decay: the
                                       gradient becomes g * f + w * weight_decay and w is not decayed (BendTorch
                                       "main.bend", section "Optimizers": the Adam case of its Adam family). */

#define MICA_MAX_TENSORS (1 << 24)
#define MICA_MAX_GROUPS 8 /* parameter groups of one mica_adamw_steps_grouped call */

/* One AdamW step's hyperparameters. */
typedef struct {
    double lr;            /* finite, >= 0 */
    double beta1;         /* [0, 1) */
    double beta2;         /* [0, 1) */
    double eps;           /* finite, >= 0 */
    double weight_decay;  /* finite, >= 0; decoupled: w *= 1 - lr * weight_decay */
    int64_t step;         /* t, 1-based: the count of steps including this one (>= 1) */
    int32_t zero_grad;    /* nonzero: the gradient is written back as zeros (BendTorch "main.bend", section "The layer
                             protocol": a step hands the gradient back zeroed) */
    uint32_t flags;       /* MICA_STEP_* bits; others must be 0 */
} mica_adamw_hp;

/*
 * ScaleTensors. For every tensor k and element i < n[k]:  t[k][i] = t[k][i] * f, in place, where f = *d_factor when
 * d_factor is not NULL (a device float32, read by the kernel) and f = factor otherwise. float16 cells are widened to
 * float32, multiplied, and rounded back to nearest-even. dt: MICA_F32 or MICA_F16.
 * Source: "Mica 7.7 ...", section "The whole model in one call" (ScaleTensors).
 * Errors: NULL / COUNT / DTYPE / HYPER (host factor not finite when d_factor is NULL) / ADDRESS / OVERLAP (two
 * tensors overlap) / DEVICE / CUDA / NOMEM.
 */
MICA_API mica_status mica_scale_tensors(void* const* t, const int64_t* n, int32_t T, mica_dtype dt, float factor,
                               const float* d_factor, void* stream);

/*
 * ClipGradNorms, with the unscale folded in. Reads g[k][i] (gdt MICA_F32 or MICA_F16) for every tensor k and
 * element i < n[k], and writes two device float32 scalars:
 *   *d_norm   = the joint L2 norm of x = f32(g * inv_scale) over every element of every tensor: the squares are
 *               formed exactly and summed in double precision in a fixed order, the square root taken in double
 *               and rounded to float32;
 *   *d_factor = inv_scale * min(1, max_norm / (norm + 1e-6)) in float32 (PyTorch's clip_grad_norm_ coefficient; a
 *               NaN norm gives a NaN factor), the one factor mica_adamw_steps multiplies every gradient by.
 * Neither is copied to the host. d_norm may be NULL (not written); d_factor may not. The gradients are only read.
 * max_norm: > 0, not NaN (infinity means never clip). inv_scale: finite, > 0 (1 when the loss is not scaled).
 * Sources: "Mica 7.7 ...", sections "The whole model in one call" and "Values that stay on the card"; BendTorch
 * "main.bend", section "Losses over arrays" (a running float32 sum of many squares drifts).
 * Errors: NULL / COUNT / DTYPE / HYPER / ADDRESS / DEVICE / CUDA / NOMEM.
 */
MICA_API mica_status mica_clip_grad_norms(const void* const* g, const int64_t* n, int32_t T, mica_dtype gdt, float max_norm,
                                 float inv_scale, float* d_norm, float* d_factor, void* stream);

/*
 * AccumulateClipGradNorms: a gradient's last write, when it has several contributions, fused with ClipGradNorms.
 * An operand that several recorded steps read gets the sum of what each hands it ("Mica 7.7 ...", section "Values
 * that stay on the card": the tape walks the steps backwards and hands each operand its gradient), so the last
 * write to such a gradient (a weight read twice, or micro-batches summed) is an add; this call makes that add and
 * measures the joint norm of the result in one pass, so the norm costs no second read of the gradient.
 * For every tensor k and element i < n[k]:
 *   g[k][i] = g[k][i] + a[k][i], in place, rounded once to the gradient type: float32 cells add in float32;
 *             float16 cells are widened, added in float32 and rounded back to nearest-even (the correctly rounded
 *             float16 sum); a NaN sum is stored as a NaN (payload unspecified);
 * then *d_norm and *d_factor exactly as mica_clip_grad_norms computes them over the updated g (same sums, same
 * rounding, same handling of NaN and infinity). a[k] is only read. gdt (MICA_F32 or MICA_F16) is the type of both.
 * Layout and ownership as mica_clip_grad_norms; every g[k] and a[k] must be disjoint from every other buffer of
 * the call (MICA_ERR_OVERLAP otherwise, also when d_norm or d_factor lies inside one). Like the norm, it allocates
 * one device table per distinct list (g, a and n), kept until mica_release_cache().
 * Sources: "Mica 7.7 ...", sections "The whole model in one call" (ClipGradNorms) and "Values that stay on the
 * card" (the tape).
 * Errors: NULL / COUNT / DTYPE / HYPER / ADDRESS / OVERLAP / DEVICE / CUDA / NOMEM.
 */
MICA_API mica_status mica_accumulate_clip_grad_norms(void* const* g, const void* const* a, const int64_t* n, int32_t T,
                                                     mica_dtype gdt, float max_norm, float inv_scale, float* d_norm,
                                                     float* d_factor, void* stream);

/*
 * mica_accumulate_grad_sumsq: the same add over one rank's part of a sharded list, fused with that part's square sum
 * (the sharded step's counterpart of mica_accumulate_clip_grad_norms, as mica_grad_sumsq is mica_clip_grad_norms's):
 * g[k] += a[k] exactly as mica_accumulate_clip_grad_norms adds, then *d_sumsq (a device double) = the sum over the
 * list of x^2, x = f32(g * inv_scale), of the updated g, summed exactly as mica_grad_sumsq sums it. The ranks' sums
 * then go to mica_clip_factor_from_sumsq.
 * Sources: as mica_accumulate_clip_grad_norms and mica_grad_sumsq.
 * Errors: NULL / COUNT / DTYPE / HYPER (inv_scale) / ADDRESS / OVERLAP (also d_sumsq inside a gradient or an
 * addend) / DEVICE / CUDA / NOMEM.
 */
MICA_API mica_status mica_accumulate_grad_sumsq(void* const* g, const void* const* a, const int64_t* n, int32_t T,
                                                mica_dtype gdt, float inv_scale, double* d_sumsq, void* stream);

/*
 * The joint norm of a list sharded over several GPUs (each rank holding a contiguous part of the parameters, as a
 * ZeRO-style partition does), in two calls around one exchange that the caller makes (an all-gather of one double
 * per rank): ClipGradNorms's joint norm ("Mica 7.7 ...", section "The whole model in one call") is that of every
 * gradient of every rank, so each rank sums its own part and the sums are added in rank order.
 *
 * mica_grad_sumsq: writes *d_sumsq (a device double) = the sum over the list of x^2, x = f32(g * inv_scale), summed
 * exactly as mica_clip_grad_norms sums it (the same kernel and work split; an empty list gives 0).
 * Errors: NULL / COUNT / DTYPE / HYPER (inv_scale) / ADDRESS / OVERLAP (d_sumsq inside a gradient) / DEVICE / CUDA /
 * NOMEM.
 */
MICA_API mica_status mica_grad_sumsq(const void* const* g, const int64_t* n, int32_t T, mica_dtype gdt, float inv_scale,
                                     double* d_sumsq, void* stream);

/*
 * mica_clip_factor_from_sumsq: from `count` per-rank square sums d_parts[0 .. count-1] (device doubles, in rank
 * order), S = d_parts[0] + d_parts[1] + ... in double, in that order, and then, as mica_clip_grad_norms:
 * *d_norm = f32(sqrt(S)) (when d_norm is not NULL) and *d_factor = inv_scale * min(1, max_norm / (norm + 1e-6)). Every
 * rank that passes the same d_parts gets the same bits. 1 <= count <= 65536.
 * Errors: NULL / COUNT / HYPER / ADDRESS / DEVICE / CUDA.
 */
MICA_API mica_status mica_clip_factor_from_sumsq(const double* d_parts, int32_t count, float max_norm, float inv_scale,
                                                 float* d_norm, float* d_factor, void* stream);

/*
 * AdamWSteps. For every group k and element i < n[k], in float32, each operation rounded on its own:
 *   gh = g * f                          f = *d_factor (device float32) or 1 when d_factor is NULL
 *   w' = w * (1 - lr*wd)
 *   m  = m + (1 - beta1) * (gh - m)
 *   v  = v * beta2 + ((1 - beta2) * gh) * gh
 *   [mdt == MICA_BF16X2: m and v rounded to BF16, stored, and read back exactly]
 *   w  = w' + (-step * m) / (sqrt(v) / bc2 + eps)
 *   g  = 0                              when hp->zero_grad
 * w: float32 [n]; g: gdt (MICA_F32 or MICA_F16) [n]; m, v: float32 [n] or packed words [ceil(n/2)] (mdt
 * MICA_F32, MICA_BF16X2, or MICA_BF16X2_M for packed m and float32 v). hp->flags selects Adam's coupled L2 form and
 * the skip of a step whose norm was not finite (MICA_STEP_*).
 * All in place. The results are bit-identical to stepping each group alone, and to the same step on the CPU.
 * Sources: "Mica 7.7 ...", section "The whole model in one call" (AdamWSteps); BendTorch "main.bend", section
 * "Optimizers" (the per-element order) and its part "AdamW over packed BF16 moments (CAdamWBF16)".
 * Errors: NULL / COUNT / DTYPE / HYPER / BETA / ADDRESS / OVERLAP / DEVICE / CUDA / NOMEM.
 */
MICA_API mica_status mica_adamw_steps(float* const* w, void* const* g, void* const* m, void* const* v, const int64_t* n,
                             int32_t T, mica_dtype gdt, mica_dtype mdt, const mica_adamw_hp* hp,
                             const float* d_factor, void* stream);

/*
 * AdamWSteps over parameter groups (PyTorch's param_groups, e.g. weight decay on the matrices and none on biases and
 * norm gains): tensor k is stepped exactly as mica_adamw_steps would step it with hyperparameters hp[group[k]], all
 * tensors in one launch. group: a host array of T indices in [0, num_groups); hp: num_groups entries, which may
 * differ only in lr and weight_decay (beta1, beta2, eps, step, zero_grad and flags must equal hp[0]'s, else
 * MICA_ERR_HYPER). 1 <= num_groups <= MICA_MAX_GROUPS (else MICA_ERR_COUNT). The group array is part of the list's
 * identity: its cached table records each tensor's group. The pages' optimizer takes one weight decay for every
 * tensor (the section "Optimizers" of BendTorch "main.bend"); the groups are this library's addition, for the
 * usual split of a transformer's parameters.
 * Errors: those of mica_adamw_steps, and COUNT for a group index or num_groups out of range.
 */
MICA_API mica_status mica_adamw_steps_grouped(float* const* w, void* const* g, void* const* m, void* const* v,
                                              const int64_t* n, int32_t T, mica_dtype gdt, mica_dtype mdt,
                                              const int32_t* group, const mica_adamw_hp* hp, int32_t num_groups,
                                              const float* d_factor, void* stream);

/*
 * One whole step of the hot path: ClipGradNorms followed by AdamWSteps on the same list, with the results of
 *   mica_clip_grad_norms(g, n, T, gdt, max_norm, inv_scale, d_norm, d_factor, stream);
 *   mica_adamw_steps(w, g, m, v, n, T, gdt, mdt, hp, d_factor, stream);
 * (the same arguments, checks and errors as those two calls, and the same results: the update bit for bit given
 * the factor; the norm within its rounding, see below). Source: "Mica 7.7 ...", sections "The whole model in one
 * call" (ClipGradNorms then AdamWSteps) and "Values that stay on the card" (the norm measured, decided and applied on
 * the card, never copied to the host).
 *
 * By default the two run as those two launches, the update a programmatic dependent of the norm; for a gradient
 * of at most 96 MB the norm's loads ask L2 to keep the gradient (an evict-last policy), so that the update reads it
 * from L2 rather than HBM (mica_clip_grad_norms does the same). With MICA_FUSED=1 (read at each call) they run as
 * ONE cooperative launch instead: each CTA sums its chunk of the gradient, keeping the lines in L2, the CTAs meet at
 * one grid-wide wait, every CTA derives the same norm and factor from the partial sums in a fixed order, and the
 * update follows in the same kernel. That launch's partial sums are grouped by its own CTAs, so its norm may differ
 * from mica_clip_grad_norms's in the last bit when the exact sum lies within ~1e-13 of a float32 rounding boundary
 * (both are within the norm's 1e-5 of the exact value). On GB300 it is the slower of the two (a cooperative launch
 * cannot overlap the steps around it). Its grid-wide wait is bounded: if it gives up (only a GPU that did not keep
 * the launch's CTAs resident could make it), the kernel stops, mica_sync() reports MICA_ERR_CUDA and the list's
 * cached table must be released (mica_release_cache) before it is used again.
 * Errors: those of mica_clip_grad_norms and mica_adamw_steps.
 */
MICA_API mica_status mica_clip_adamw_step(float* const* w, void* const* g, void* const* m, void* const* v,
                                          const int64_t* n, int32_t T, mica_dtype gdt, mica_dtype mdt,
                                          const mica_adamw_hp* hp, float max_norm, float inv_scale, float* d_norm,
                                          float* d_factor, void* stream);

/* One SGD step's hyperparameters. */
typedef struct {
    double lr;          /* finite, >= 0 */
    double momentum;    /* finite, >= 0; must be 0 when buf is NULL */
    int32_t zero_grad;  /* nonzero: the gradient is written back as zeros */
    uint32_t flags;     /* MICA_STEP_SKIP_NONFINITE or 0 */
} mica_sgd_hp;

/*
 * SGD and SGD with momentum (BendTorch "main.bend", section "Optimizers": its SGD and Momentum cases, which are
 * PyTorch's SGD without weight decay, dampening or Nesterov). For every tensor k and element i < n[k], in float32,
 * each operation rounded on its own:
 *   gh = g * f                    f = *d_factor (device float32) or 1 when d_factor is NULL
 *   buf == NULL:   w = w + (-lr) * gh
 *   buf != NULL:   b = buf * momentum + gh;  buf = b;  w = w + (-lr) * b
 *   g  = 0                        when hp->zero_grad
 * w: float32 [n]; g: gdt (MICA_F32 or MICA_F16) [n]; buf: NULL, or a host array of T device pointers to float32
 * momentum buffers [n] (zeros before the first step: b = g then, as PyTorch's first step sets it). lr and momentum
 * are rounded once to float32. With MICA_STEP_SKIP_NONFINITE, w and buf are left as they are when the factor is not
 * > 0. In place, one launch; bit-identical to the same step on the CPU.
 * Errors: NULL / COUNT / DTYPE / HYPER / ADDRESS / OVERLAP / DEVICE / CUDA / NOMEM.
 */
MICA_API mica_status mica_sgd_steps(float* const* w, void* const* g, float* const* buf, const int64_t* n, int32_t T,
                                    mica_dtype gdt, const mica_sgd_hp* hp, const float* d_factor, void* stream);

/*
 * ClipGradNorms for callers that cannot let a library allocate device memory: a runtime that reserves its whole
 * device-memory budget at start-up and treats any later cudaMalloc as a failure, a caller whose memory is all held
 * by another allocator, or a loop that cannot afford cudaMalloc's implicit synchronisation. The method's pages have
 * no counterpart to this entry point; it is an addition of this library.
 *
 * Arguments, results and errors are those of mica_clip_grad_norms (same kernel and arithmetic; the same bits too,
 * unless a list of more than about 2 GB of gradient asks for more than 1,024 CTAs, which this entry point caps, so
 * that its partial sums are grouped differently: the norm then agrees to ~1e-13 relative). The difference is where
 * the scratch lives: instead of a per-list table allocated on first use, every call copies its tables into one
 * fixed device array of this library (930,304 bytes, held by every GPU that loads the library until the process
 * exits) and launches on `stream`. The call allocates nothing: no cudaMalloc, no cudaFree, no host heap.
 *   - Limit: at most 16,384 tensors (MICA_ERR_COUNT beyond, with a detail naming the limit).
 *   - Every call checks every gradient as a table build of mica_clip_grad_norms does (device memory of the current
 *     device, n elements inside its allocation, else MICA_ERR_ADDRESS), and uploads its tables: its host cost grows
 *     linearly with T (two driver queries per tensor and up to 1 MB copied from host memory).
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress) with that device
 *     current, and keeps it; make that first call before any stream capture. mica_release_cache() forgets the
 *     address, so that the next call looks it up again: call mica_release_cache() after a cudaDeviceReset before
 *     using this entry point again.
 *   - The tables are copied from a host buffer that every call reuses, so a call on a stream that is capturing a
 *     CUDA graph is refused with MICA_ERR_CAPTURE before anything is queued (the capture is left intact).
 *   - The array is shared by every call and keeps the last call's contents; each call rewrites what it reads, so
 *     calls ordered on one stream are safe, while calls that overlap on the GPU (other streams, other threads'
 *     streams) race on it.
 *   - The host side of concurrent calls is serialised (one static staging buffer).
 */
MICA_API mica_status mica_clip_grad_norms_noalloc(const void* const* g, const int64_t* n, int32_t T, mica_dtype gdt,
                                                  float max_norm, float inv_scale, float* d_norm, float* d_factor,
                                                  void* stream);

/* Waits for `stream` and reports a fault of any work queued on it (MICA_OK or MICA_ERR_CUDA). It also reads and clears
 * the device's pipeline status word: every wait of a kernel on its shared-memory barriers is bounded, and a wait
 * that gives up (which only a broken memory system could cause) stops that kernel early and is reported here as
 * MICA_ERR_CUDA, with its results not valid. */
MICA_API mica_status mica_sync(void* stream);

/*
 * Self-test of the failure path above, which the method's pages have no counterpart to: queues on `stream` one
 * one-warp kernel whose bounded mbarrier wait runs out after `polls` polling rounds (1 <= polls <= 2^20, else
 * MICA_ERR_HYPER) because nothing ever arrives at the barrier; the kernel then ORs 0x4 into the status word and
 * returns. The next mica_sync(stream) reports MICA_ERR_CUDA ("... gave up (status 0x4)"), the one after it MICA_OK,
 * and the context stays usable. Nothing faults, traps or hangs.
 */
MICA_API mica_status mica_selftest_wait_timeout(uint32_t polls, void* stream);

/*
 * Self-test of the fused launch's grid-wide wait (mica_clip_adamw_step), which the method's pages have no
 * counterpart to: queues on `stream` one one-CTA kernel that waits for a second CTA that is never launched; its
 * bounded wait gives up after `polls` polls (1 <= polls <= 2^20, else MICA_ERR_HYPER; each poll sleeps ~128 ns or
 * more) and ORs 0x10 into the fused kernels' status word. The next mica_sync(stream) reports MICA_ERR_CUDA
 * ("... grid-wide wait gave up (status 0x10)"), the one after it MICA_OK, and the context stays usable. Nothing
 * faults, traps or hangs.
 */
MICA_API mica_status mica_selftest_grid_wait_timeout(uint32_t polls, void* stream);

/* Waits for the current device, then frees every cached per-list device table (but those a call in progress on
 * another thread holds, which stay cached). Returns MICA_OK or MICA_ERR_CUDA. The cache holds at most 1,024 tables;
 * a new table beyond that first frees, the same way, every table no call in progress holds. */
MICA_API mica_status mica_release_cache(void);

/* A static, human-readable name for a status. */
MICA_API const char* mica_status_string(mica_status s);

/* One line describing the last error returned on the calling thread ("" if none); valid until the thread's next
 * call into the library. */
MICA_API const char* mica_last_error_detail(void);

/* How many kernels this library has queued since it was loaded, over all threads. */
MICA_API uint64_t mica_launch_count(void);

/* The work items an update call (AdamWSteps, SGD) cuts a list into, for inspection and tests; no device is used and
 * nothing is cached. The list is n[T] (element counts) and vec[T] (nonzero where a tensor's buffers are aligned for
 * the vector path: 32 bytes for float32 streams, 16 for binary16 and packed ones). item_octs is the octets (8
 * elements) per slice of a large tensor, a power of two from 16 to 2^20, or 0 for what an AdamW call with float32
 * moments chooses on a GPU of `sms` SMs (`*used_item_octs` gets the value used; it may be NULL).
 * Output, in array order (the kernels take the items from the end of the array): item i as three int64 values in
 * items[3i .. 3i+2]: its first tensor t, its tensor count c, and o0. A slice has c == 1; it covers octets
 * [o0, min(o0 + item_octs, ceil(n[t]/8))) of tensor t. A pack has c > 1; it covers tensors t .. t+c-1 whole, and its
 * row of the pack table starts at pack[o0]: c + 1 running counts of the tensors' whole octets (those of vec
 * tensors' first floor(n/8) octets), then c + 1 running counts of their other octets. Up to max_items items and
 * max_pack table entries are written; *num_items and *pack_len get the full counts either way.
 * Errors: MICA_ERR_NULL (num_items, pack_len, n or vec NULL where needed, or an output NULL with a nonzero
 * capacity), MICA_ERR_COUNT (T, an n[i], item_octs, sms or a capacity out of range). This is a description of this
 * library's own scheduling, with no counterpart in the method's pages. */
MICA_API mica_status mica_work_items(const int64_t* n, const int32_t* vec, int32_t T, int32_t item_octs, int32_t sms,
                                     int64_t* items, int32_t max_items, int32_t* pack, int32_t max_pack,
                                     int32_t* num_items, int32_t* pack_len, int32_t* used_item_octs);

/* The ABI version of this header: 5 (4 had neither mica_accumulate_clip_grad_norms nor mica_accumulate_grad_sumsq; 3 had none of mica_clip_adamw_step,
 * mica_grad_sumsq, mica_clip_factor_from_sumsq, mica_selftest_grid_wait_timeout and MICA_ERR_CAPTURE; 2 had no
 * mica_work_items; 1 had neither mica_adamw_steps_grouped nor mica_sgd_steps). */
MICA_API int32_t mica_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MICA_OPTIM_H */
