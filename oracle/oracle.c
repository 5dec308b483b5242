/*
 * Oracle for the clip + AdamW optimizer step: plain, single-threaded and slow on purpose.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's CPU-baseline leg load this file's
 * library. The product library does not call, link or include it, and it includes nothing of the product's: the
 * dtype codes, the scalars and every conversion below are written out here on their own.
 *
 * Pages it follows (title, then section):
 *   [MICA]  "Mica 7.7: a training step on the card, in every float type", sections "The whole model in one call"
 *           and "Values that stay on the card": ClipGradNorms caps the joint L2 norm of every listed gradient;
 *           AdamWSteps updates each (w, g, m, v) group exactly as a single-group AdamWStep would; ScaleTensors
 *           scales each element of each listed tensor by a single factor (a float16 step's unscale).
 *   [OPT]   BendTorch "main.bend", section "Optimizers": AdamW element by element in PyTorch's order of
 *           operations, the gradient written back as zero, c1 = 1 - b1 and c2 = 1 - b2 taken as constants of
 *           their own; the same section's plain SGD (w + (-lr) g) and SGD with momentum (b = b mu + g,
 *           w + (-lr) b), both as PyTorch's SGD without weight decay, dampening or Nesterov.
 *   [BF16]  BendTorch "main.bend", section "Optimizers", part "AdamW over packed BF16 moments (CAdamWBF16)": BF16
 *           rounding to nearest-even with NaN -> 0xFFFF, element 2k in the low half of word k, and the weight update
 *           reading the rounded moments.
 *   [LAYOUT] BendTorch "main.bend", section "The layer protocol" (the PTree comment): ceil(n/2) words per packed
 *           buffer, zero-initialised (BF16 0x0000 is +0.0).
 *   [SUM]   BendTorch "main.bend", section "Losses over arrays": a running F32 sum of many squares drifts, so the
 *           joint norm here is summed in double over exactly formed squares.
 *   [PREC]  "Precision and numerics", section "bf16 regions": rounding to nearest-even is the one cast.
 *   [TAPE]  "Mica 7.7", section "Values that stay on the card": the tape walks the recorded steps backwards and
 *           hands each operand its gradient; an operand read by more than one step gets the sum of what each
 *           step hands it (the chain rule), so the last write to such a gradient is an element-wise add.
 *
 * Readings where the pages leave a step open (each is listed in the design notes):
 *   - The step's scalars are PyTorch's: every one is computed in double and rounded once to float32 (c1, c2, b2,
 *     step = lr / (1 - b1^t), bc2 = sqrt(1 - b2^t), the decay 1 - lr*wd, eps).
 *   - The joint norm is that of the unscaled gradient x = f32(g * inv_scale); its square sum is taken in double
 *     (each f32 square is exact there), its square root in double, and the result rounded to float32.
 *   - The clip coefficient is PyTorch's clip_grad_norm_: f32(max_norm) / f32(norm + f32(1e-6)), clamped at 1 with
 *     a NaN passed through. The unscale and the clip fold into one factor f32(inv_scale * clip) that multiplies g
 *     inside the update; the gradient is never rewritten by the clip.
 *   - Parameter groups (PyTorch's param_groups: a list split into groups with their own lr and weight decay, e.g.
 *     no decay on biases and norm gains) step every tensor exactly as a call over its group alone would.
 *   - A gradient's last write when it has several contributions (a weight read twice, micro-batches summed) is
 *     g + a rounded once to the gradient's type, as PyTorch's add_ does: float32 cells add in float32; binary16
 *     cells are widened, added in float32 and rounded back to nearest-even (float32 holds at least 2 * 11 + 2
 *     significant bits, so this is the correctly rounded binary16 sum). The norm fused into that write is the
 *     norm of the list after the add.
 *
 * Build with -O2 -ffp-contract=off and without -ffast-math: every float operation below rounds on its own, with no
 * fused multiply-add, exactly in the order written.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* element types, the oracle's own codes; ORA_BF16X2_M (moments only): m packed, v float32 */
enum { ORA_F32 = 0, ORA_F16 = 1, ORA_BF16X2 = 2, ORA_BF16X2_M = 3 };

/* ------------------------------------------------------------------------------------------------------------ */
/* bit casts                                                                                                    */
/* ------------------------------------------------------------------------------------------------------------ */

static uint32_t bits_of(float x) {
    uint32_t u;
    memcpy(&u, &x, 4);
    return u;
}

static float float_of(uint32_t u) {
    float x;
    memcpy(&x, &u, 4);
    return x;
}

/* ------------------------------------------------------------------------------------------------------------ */
/* BF16 [BF16], [PREC]                                                                                           */
/* ------------------------------------------------------------------------------------------------------------ */

/* float32 bits -> BF16 bits, nearest-even. Adding 0x7FFF plus the lowest bit that survives the shift rounds the
 * dropped 16 bits to nearest with ties going to the even kept value; a carry out of the mantissa moves into the
 * exponent, so the largest finite values round up to infinity as nearest-even says. Any NaN becomes 0xFFFF. */
uint16_t ora_bf16_from_bits(uint32_t u) {
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0xFFFFu;
    uint32_t keep_lsb = (u >> 16) & 1u;
    return (uint16_t)((u + 0x7FFFu + keep_lsb) >> 16);
}

uint16_t ora_bf16_from_f32(float x) { return ora_bf16_from_bits(bits_of(x)); }

/* BF16 bits -> float32: the 16 bits are the top half of the float32, so the widening is exact. */
float ora_f32_from_bf16(uint16_t h) { return float_of((uint32_t)h << 16); }

/* ------------------------------------------------------------------------------------------------------------ */
/* IEEE binary16 (the loss-scaled gradient and ScaleTensors on float16 tensors), from the format's definition      */
/* ------------------------------------------------------------------------------------------------------------ */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
float ora_f32_from_f16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    float mag;
    if (e == 0x1F) {
        mag = f ? NAN : INFINITY;
    } else if (e == 0) {
        mag = ldexpf((float)f, -24);             /* subnormal: f * 2^-24 */
    } else {
        mag = ldexpf((float)(f | 0x400), e - 25); /* (1024 + f) * 2^(e - 15 - 10) */
    }
    return sign ? -mag : mag;
}

/* float32 -> binary16, round to nearest, ties to even. */
uint16_t ora_f16_from_f32(float x) {
    uint32_t u = bits_of(x);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t a = u & 0x7FFFFFFFu;
    if (a > 0x7F800000u) return (uint16_t)(sign | 0x7E00u);  /* NaN stays NaN */
    if (a == 0x7F800000u) return (uint16_t)(sign | 0x7C00u); /* infinity */
    int e32 = (int)(a >> 23);
    if (e32 == 0) return sign;                 /* float32 subnormals are far below binary16's smallest half-ulp */
    uint32_t mant = (a & 0x7FFFFFu) | 0x800000u; /* 24-bit significand */
    int e16 = e32 - 127 + 15;                   /* biased binary16 exponent of the same binade */
    int shift;                                  /* significand bits dropped */
    uint32_t base;                              /* what the kept significand adds to */
    if (e16 >= 1) {
        shift = 13;
        base = (uint32_t)e16 << 10;             /* the hidden bit of `mant >> 13` (0x400) adds one more to e16 */
        base -= 0x400u;
    } else {
        shift = 13 + (1 - e16);                 /* subnormal result: scale down to units of 2^-24 */
        if (shift > 25) return sign;            /* below half the smallest subnormal: rounds to zero */
        base = 0;
    }
    uint32_t kept = mant >> shift;
    uint32_t rem = mant & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (kept & 1u))) kept += 1u;
    uint32_t r = base + kept;                   /* a carry walks into the exponent, up to 0x7C00 = infinity */
    if (r >= 0x7C00u) r = 0x7C00u;
    return (uint16_t)(sign | r);
}

/* The conversions above over arrays, one element at a time (for the exhaustive checks of the test suite). */
void ora_bf16_from_bits_array(const uint32_t* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = ora_bf16_from_bits(in[i]);
}

void ora_f32_from_bf16_array(const uint16_t* in, float* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = ora_f32_from_bf16(in[i]);
}

void ora_f32_from_f16_array(const uint16_t* in, float* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = ora_f32_from_f16(in[i]);
}

void ora_f16_from_f32_array(const float* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = ora_f16_from_f32(in[i]);
}

/* ------------------------------------------------------------------------------------------------------------ */
/* the step's scalars [OPT]                                                                                       */
/* ------------------------------------------------------------------------------------------------------------ */

typedef struct {
    float c1;   /* 1 - b1, the lerp weight */
    float b2;   /* b2 */
    float c2;   /* 1 - b2 */
    float step; /* lr / (1 - b1^t) */
    float bc2;  /* sqrt(1 - b2^t) */
    float dec;  /* 1 - lr * wd, AdamW's decoupled decay */
    float eps;  /* eps */
    float wd;   /* wd, for Adam's coupled L2 form (g + wd * w) */
} ora_scalars;

/* Every scalar in double, then rounded once to float32, as PyTorch's Python-float scalars are. t is 1-based. */
void ora_step_scalars(double lr, double b1, double b2, double eps, double wd, int64_t t, ora_scalars* s) {
    double tt = (double)t;
    s->c1 = (float)(1.0 - b1);
    s->b2 = (float)b2;
    s->c2 = (float)(1.0 - b2);
    s->step = (float)(lr / (1.0 - pow(b1, tt)));
    s->bc2 = (float)sqrt(1.0 - pow(b2, tt));
    s->dec = (float)(1.0 - lr * wd);
    s->eps = (float)eps;
    s->wd = (float)wd;
}

/* ------------------------------------------------------------------------------------------------------------ */
/* joint norm and clip factor [MICA], [SUM]                                                                       */
/* ------------------------------------------------------------------------------------------------------------ */

static float grad_at(const void* g, int gdt, int64_t i) {
    if (gdt == ORA_F16) return ora_f32_from_f16(((const uint16_t*)g)[i]);
    return ((const float*)g)[i];
}

/* Sum over every tensor (in list order) and every element (in order) of x^2, x = f32(g * inv_scale). Each square
 * of a float32 is exact in double; the running sum is in double. */
double ora_sum_squares(const void* const* g, const int64_t* n, int32_t T, int32_t gdt, float inv_scale) {
    double S = 0.0;
    for (int32_t k = 0; k < T; ++k) {
        for (int64_t i = 0; i < n[k]; ++i) {
            float x = grad_at(g[k], gdt, i) * inv_scale;
            double xd = (double)x;
            S = S + xd * xd;
        }
    }
    return S;
}

/* The joint L2 norm, rounded to float32 from its double square root. */
float ora_norm_from_sum(double S) { return (float)sqrt(S); }

/* PyTorch's clip_grad_norm_ coefficient, clamped at 1 (a NaN norm gives a NaN coefficient), then times the
 * unscale: the one factor every gradient element is multiplied by in the update. */
float ora_clip_factor(float norm, float max_norm, float inv_scale) {
    float denom = norm + 1e-6f;
    float coef = max_norm / denom;
    float clip = (coef > 1.0f) ? 1.0f : coef;
    return inv_scale * clip;
}

/* ------------------------------------------------------------------------------------------------------------ */
/* AdamW, one group [OPT], [BF16]                                                                                */
/* ------------------------------------------------------------------------------------------------------------ */

/* the half of packed word `word` that holds element i: even i the low 16 bits, odd i the high 16 bits */
static uint16_t half_of(uint32_t word, int64_t i) {
    return (uint16_t)((i & 1) ? (word >> 16) : (word & 0xFFFFu));
}

static uint32_t with_half(uint32_t word, int64_t i, uint16_t h) {
    if (i & 1) return (word & 0x0000FFFFu) | ((uint32_t)h << 16);
    return (word & 0xFFFF0000u) | (uint32_t)h;
}

/* One group: n elements of the float32 weight w, its gradient g (float32 or binary16), and the two moments m and
 * v (float32, or packed BF16 words, ceil(n/2) of them; or, for ORA_BF16X2_M, m packed and v float32 - the page's
 * CAdamWBF16 with v16 false). decoupled != 0 is AdamW (w *= 1 - lr*wd); decoupled == 0
 * is Adam's coupled L2 (g += wd * w), the other case the page's Adam family holds. Element by element, each float
 * operation rounded on its own, in this order:
 *   gh = g * factor                        (unscale and clip, folded)
 *   [Adam: gh = gh + w * wd]
 *   wd' = w * dec                          [AdamW; Adam: wd' = w]
 *   m = m + c1 * (gh - m)
 *   v = v * b2 + (c2 * gh) * gh
 *   [packed: m and v rounded to BF16 and read back]
 *   w = wd' + ((-step) * m) / (sqrt(v) / bc2 + eps)
 *   g = 0                                  (when zero_grad)
 * With packed moments, m and v live in separate halves of their words; an odd n leaves the high half of the last
 * word as it was. */
void ora_adam_group(float* w, void* g, void* m, void* v, int64_t n, int32_t gdt, int32_t mdt,
                    const ora_scalars* s, float factor, int32_t zero_grad, int32_t decoupled) {
    float neg_step = -s->step;
    for (int64_t i = 0; i < n; ++i) {
        float gh = grad_at(g, gdt, i) * factor;
        float wi = w[i];
        if (!decoupled) gh = gh + wi * s->wd;
        float wdec = decoupled ? wi * s->dec : wi;

        const int m_packed = (mdt == ORA_BF16X2 || mdt == ORA_BF16X2_M);
        const int v_packed = (mdt == ORA_BF16X2);
        float mi = m_packed ? ora_f32_from_bf16(half_of(((uint32_t*)m)[i >> 1], i)) : ((float*)m)[i];
        float vi = v_packed ? ora_f32_from_bf16(half_of(((uint32_t*)v)[i >> 1], i)) : ((float*)v)[i];

        float m_new = mi + s->c1 * (gh - mi);
        float v_new = vi * s->b2 + (s->c2 * gh) * gh;

        /* a packed moment is rounded to BF16 and stored; the weight reads the stored, rounded value */
        if (m_packed) {
            uint16_t hm = ora_bf16_from_f32(m_new);
            ((uint32_t*)m)[i >> 1] = with_half(((uint32_t*)m)[i >> 1], i, hm);
            m_new = ora_f32_from_bf16(hm);
        } else {
            ((float*)m)[i] = m_new;
        }
        if (v_packed) {
            uint16_t hv = ora_bf16_from_f32(v_new);
            ((uint32_t*)v)[i >> 1] = with_half(((uint32_t*)v)[i >> 1], i, hv);
            v_new = ora_f32_from_bf16(hv);
        } else {
            ((float*)v)[i] = v_new;
        }

        float denom = sqrtf(v_new) / s->bc2 + s->eps;
        w[i] = wdec + (neg_step * m_new) / denom;

        if (zero_grad) {
            if (gdt == ORA_F16) ((uint16_t*)g)[i] = 0;
            else ((float*)g)[i] = 0.0f;
        }
    }
}

/* ------------------------------------------------------------------------------------------------------------ */
/* the three verbs over a list [MICA]                                                                            */
/* ------------------------------------------------------------------------------------------------------------ */

/* AdamWSteps: every group in list order, each exactly as it would be stepped alone. */
void ora_adamw_steps(float* const* w, void* const* g, void* const* m, void* const* v, const int64_t* n, int32_t T,
                     int32_t gdt, int32_t mdt, const ora_scalars* s, float factor, int32_t zero_grad) {
    for (int32_t k = 0; k < T; ++k)
        ora_adam_group(w[k], g[k], m[k], v[k], n[k], gdt, mdt, s, factor, zero_grad, 1);
}

/* Adam with the coupled L2 term, over a list. */
void ora_adam_l2_steps(float* const* w, void* const* g, void* const* m, void* const* v, const int64_t* n, int32_t T,
                       int32_t gdt, int32_t mdt, const ora_scalars* s, float factor, int32_t zero_grad) {
    for (int32_t k = 0; k < T; ++k)
        ora_adam_group(w[k], g[k], m[k], v[k], n[k], gdt, mdt, s, factor, zero_grad, 0);
}

/* The Adam family over a list with the step's options: bit 1 of `flags` picks Adam's coupled L2 form over AdamW's
 * decoupled decay; bit 0 skips the update when the factor is not > 0 - the joint norm was NaN (factor NaN) or
 * infinite (factor 0), the overflow a loss-scaled float16 step checks for before stepping - in which case only the
 * gradient is zeroed (when zero_grad). */
void ora_adam_steps_flags(float* const* w, void* const* g, void* const* m, void* const* v, const int64_t* n,
                          int32_t T, int32_t gdt, int32_t mdt, const ora_scalars* s, float factor, int32_t zero_grad,
                          uint32_t flags) {
    const int skip = (flags & 1u) && !(factor > 0.0f);
    const int decoupled = !(flags & 2u);
    for (int32_t k = 0; k < T; ++k) {
        if (!skip) {
            ora_adam_group(w[k], g[k], m[k], v[k], n[k], gdt, mdt, s, factor, zero_grad, decoupled);
        } else if (zero_grad) {
            for (int64_t i = 0; i < n[k]; ++i) {
                if (gdt == ORA_F16) ((uint16_t*)g[k])[i] = 0;
                else ((float*)g[k])[i] = 0.0f;
            }
        }
    }
}

/* The Adam family over a list split into parameter groups: tensor k steps with the scalars s[group[k]] (group ==
 * NULL: every tensor in group 0), and the options of `flags` as in ora_adam_steps_flags. */
void ora_adam_steps_grouped(float* const* w, void* const* g, void* const* m, void* const* v, const int64_t* n,
                            int32_t T, int32_t gdt, int32_t mdt, const int32_t* group, const ora_scalars* s,
                            float factor, int32_t zero_grad, uint32_t flags) {
    for (int32_t k = 0; k < T; ++k) {
        const ora_scalars* sk = group ? &s[group[k]] : &s[0];
        ora_adam_steps_flags(&w[k], &g[k], &m[k], &v[k], &n[k], 1, gdt, mdt, sk, factor, zero_grad, flags);
    }
}

/* ------------------------------------------------------------------------------------------------------------ */
/* SGD and SGD with momentum [OPT]                                                                                */
/* ------------------------------------------------------------------------------------------------------------ */

/* One group of the page's two plain optimizers, with PyTorch's SGD arithmetic (no weight decay, dampening or
 * Nesterov). lr and mu arrive as float32. Element by element, each float operation rounded on its own:
 *   gh = g * factor                        (unscale and clip, folded)
 *   buf == NULL (SGD):       w = w + (-lr) * gh
 *   buf != NULL (momentum):  b = b * mu + gh;  w = w + (-lr) * b;  buf = b
 *   g = 0                                  (when zero_grad) */
void ora_sgd_group(float* w, void* g, float* buf, int64_t n, int32_t gdt, float lr, float mu, float factor,
                   int32_t zero_grad) {
    float neg_lr = -lr;
    for (int64_t i = 0; i < n; ++i) {
        float gh = grad_at(g, gdt, i) * factor;
        if (buf) {
            float b = buf[i] * mu + gh;
            buf[i] = b;
            w[i] = w[i] + neg_lr * b;
        } else {
            w[i] = w[i] + neg_lr * gh;
        }
        if (zero_grad) {
            if (gdt == ORA_F16) ((uint16_t*)g)[i] = 0;
            else ((float*)g)[i] = 0.0f;
        }
    }
}

/* SGD (buf == NULL) or SGD with momentum over a list; lr and mu are rounded once to float32, as PyTorch passes its
 * Python-float scalars to float32 arithmetic. Bit 0 of `flags` skips the update when the factor is not > 0, as in
 * ora_adam_steps_flags (only the gradient is then zeroed, when zero_grad). */
void ora_sgd_steps(float* const* w, void* const* g, float* const* buf, const int64_t* n, int32_t T, int32_t gdt,
                   double lr, double mu, float factor, int32_t zero_grad, uint32_t flags) {
    const int skipped = (flags & 1u) && !(factor > 0.0f);
    for (int32_t k = 0; k < T; ++k) {
        if (!skipped) {
            ora_sgd_group(w[k], g[k], buf ? buf[k] : 0, n[k], gdt, (float)lr, (float)mu, factor, zero_grad);
        } else if (zero_grad) {
            for (int64_t i = 0; i < n[k]; ++i) {
                if (gdt == ORA_F16) ((uint16_t*)g[k])[i] = 0;
                else ((float*)g[k])[i] = 0.0f;
            }
        }
    }
}

/* ClipGradNorms: the joint norm and the folded factor of one list. */
void ora_clip_grad_norms(const void* const* g, const int64_t* n, int32_t T, int32_t gdt, float max_norm,
                         float inv_scale, float* norm_out, float* factor_out, double* sumsq_out) {
    double S = ora_sum_squares(g, n, T, gdt, inv_scale);
    float norm = ora_norm_from_sum(S);
    if (sumsq_out) *sumsq_out = S;
    *norm_out = norm;
    *factor_out = ora_clip_factor(norm, max_norm, inv_scale);
}

/* ScaleTensors: every cell times one factor, in place; binary16 cells are widened, multiplied in float32 and
 * rounded back to nearest-even. */
void ora_scale_tensors(void* const* t, const int64_t* n, int32_t T, int32_t dt, float factor) {
    for (int32_t k = 0; k < T; ++k) {
        for (int64_t i = 0; i < n[k]; ++i) {
            if (dt == ORA_F16) {
                uint16_t* p = (uint16_t*)t[k];
                p[i] = ora_f16_from_f32(ora_f32_from_f16(p[i]) * factor);
            } else {
                float* p = (float*)t[k];
                p[i] = p[i] * factor;
            }
        }
    }
}

/* ------------------------------------------------------------------------------------------------------------ */
/* the gradient's last write, an add, with the joint norm of its result [TAPE], [MICA], [SUM]                      */
/* ------------------------------------------------------------------------------------------------------------ */

/* Every cell of every listed gradient plus the same cell of its addend, in place. */
void ora_accumulate_grads(void* const* g, const void* const* a, const int64_t* n, int32_t T, int32_t gdt) {
    for (int32_t k = 0; k < T; ++k) {
        for (int64_t i = 0; i < n[k]; ++i) {
            if (gdt == ORA_F16) {
                uint16_t* p = (uint16_t*)g[k];
                const uint16_t* q = (const uint16_t*)a[k];
                p[i] = ora_f16_from_f32(ora_f32_from_f16(p[i]) + ora_f32_from_f16(q[i]));
            } else {
                float* p = (float*)g[k];
                const float* q = (const float*)a[k];
                p[i] = p[i] + q[i];
            }
        }
    }
}

/* The add, then ClipGradNorms over the list it leaves: what one pass over g and a computes. */
void ora_accumulate_clip_grad_norms(void* const* g, const void* const* a, const int64_t* n, int32_t T, int32_t gdt,
                                    float max_norm, float inv_scale, float* norm_out, float* factor_out) {
    ora_accumulate_grads(g, a, n, T, gdt);
    ora_clip_grad_norms((const void* const*)g, n, T, gdt, max_norm, inv_scale, norm_out, factor_out, 0);
}

/* The whole step of the hot path: the joint norm and its factor, then AdamW over every group. */
void ora_clip_adamw_step(float* const* w, void* const* g, void* const* m, void* const* v, const int64_t* n,
                         int32_t T, int32_t gdt, int32_t mdt, const ora_scalars* s, float max_norm, float inv_scale,
                         int32_t zero_grad, float* norm_out, float* factor_out) {
    float norm, factor;
    ora_clip_grad_norms((const void* const*)g, n, T, gdt, max_norm, inv_scale, &norm, &factor, 0);
    ora_adamw_steps(w, g, m, v, n, T, gdt, mdt, s, factor, zero_grad);
    *norm_out = norm;
    *factor_out = factor;
}
