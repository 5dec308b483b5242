"""Plant one plausible mistake at a time in a copy of the oracle (on the CPU) and require the pins to catch it.

Each mutation is a textual replacement in a temporary copy of ``oracle/oracle.c``; the copy is compiled with the
oracle's own flags and every pin is run against it. Every mutation keeps the oracle's memory accesses in bounds
(a mistake that wrote past an array would corrupt this test process instead of being caught by a pin). A mutation that no pin catches would mean the pins cannot tell
that mistake from the page's arithmetic.
"""
import os
import shutil

import pytest

import oracle
import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTATIONS = {
    "decay_dropped": ("float wdec = decoupled ? wi * s->dec : wi;", "float wdec = wi;"),
    "step_sign": ("float neg_step = -s->step;", "float neg_step = s->step;"),
    "c1_c2_swapped_in_m": ("mi + s->c1 * (gh - mi)", "mi + s->c2 * (gh - mi)"),
    "b1_in_bc2": ("s->bc2 = (float)sqrt(1.0 - pow(b2, tt));", "s->bc2 = (float)sqrt(1.0 - pow(b1, tt));"),
    "no_bias_correction1": ("s->step = (float)(lr / (1.0 - pow(b1, tt)));", "s->step = (float)lr;"),
    "eps_inside_sqrt": ("sqrtf(v_new) / s->bc2 + s->eps", "sqrtf(v_new + s->eps) / s->bc2"),
    "v_linear_in_g": ("(s->c2 * gh) * gh", "(s->c2 * gh)"),
    "w_reads_unrounded_m": ("m_new = ora_f32_from_bf16(hm);", ";"),
    "w_reads_unrounded_v": ("v_new = ora_f32_from_bf16(hv);", ";"),
    "bf16_truncates": ("return (uint16_t)((u + 0x7FFFu + keep_lsb) >> 16);", "return (uint16_t)(u >> 16);"),
    "bf16_ties_up": ("return (uint16_t)((u + 0x7FFFu + keep_lsb) >> 16);",
                     "return (uint16_t)((u + 0x8000u) >> 16);"),
    "bf16_nan_canonical": ("if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0xFFFFu;",
                           "if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0u;"),
    "halves_swapped": ("return (uint16_t)((i & 1) ? (word >> 16) : (word & 0xFFFFu));",
                       "return (uint16_t)((i & 1) ? (word & 0xFFFFu) : (word >> 16));"),
    "norm_ignores_unscale": ("float x = grad_at(g[k], gdt, i) * inv_scale;", "float x = grad_at(g[k], gdt, i);"),
    "norm_summed_in_f32": ("double S = 0.0;\n    for (int32_t k = 0; k < T; ++k) {",
                           "float S = 0.0f;\n    for (int32_t k = 0; k < T; ++k) {"),
    "clip_not_clamped": ("float clip = (coef > 1.0f) ? 1.0f : coef;", "float clip = coef;"),
    "clip_eps_dropped": ("float denom = norm + 1e-6f;", "float denom = norm;"),
    "c2_taken_in_f32": ("s->c2 = (float)(1.0 - b2);", "s->c2 = 1.0f - (float)b2;"),
    "zero_grad_ignored": ("w[i] = wdec + (neg_step * m_new) / denom;\n\n        if (zero_grad) {\n",
                          "w[i] = wdec + (neg_step * m_new) / denom;\n\n        if (0) {\n"),
    "sgd_zero_grad_ignored": ("w[i] = w[i] + neg_lr * gh;\n        }\n        if (zero_grad) {",
                              "w[i] = w[i] + neg_lr * gh;\n        }\n        if (0) {"),
    "f16_exponent_bias": ("mag = ldexpf((float)(f | 0x400), e - 25);", "mag = ldexpf((float)(f | 0x400), e - 24);"),
    "f16_round_down": ("if (rem > half || (rem == half && (kept & 1u))) kept += 1u;", ";"),
    "scale_ignores_factor": ("p[i] = p[i] * factor;", "p[i] = p[i];"),
    "packed_m_rounds_v_too": ("const int v_packed = (mdt == ORA_BF16X2);",
                              "const int v_packed = (mdt == ORA_BF16X2 || mdt == ORA_BF16X2_M);"),
    "skip_ignored": ("const int skip = (flags & 1u) && !(factor > 0.0f);", "const int skip = 0;"),
    "skip_on_finite": ("const int skip = (flags & 1u) && !(factor > 0.0f);", "const int skip = (flags & 1u);"),
    "groups_ignored": ("const ora_scalars* sk = group ? &s[group[k]] : &s[0];", "const ora_scalars* sk = &s[0];"),
    "sgd_sign": ("float neg_lr = -lr;", "float neg_lr = lr;"),
    "sgd_momentum_dropped": ("float b = buf[i] * mu + gh;", "float b = gh;"),
    "sgd_momentum_not_decayed": ("float b = buf[i] * mu + gh;", "float b = buf[i] + gh;"),
    "sgd_w_reads_gradient": ("w[i] = w[i] + neg_lr * b;", "w[i] = w[i] + neg_lr * gh;"),
    "sgd_buffer_not_stored": ("buf[i] = b;", ";"),
    "sgd_ignores_factor": ("float gh = grad_at(g, gdt, i) * factor;\n        if (buf) {",
                           "float gh = grad_at(g, gdt, i);\n        if (buf) {"),
    "sgd_skip_ignored": ("const int skipped = (flags & 1u) && !(factor > 0.0f);", "const int skipped = 0;"),
    # orders of the per-element arithmetic and of the scalars that a reader could take for the page's
    "lerp_as_weighted_sum": ("float m_new = mi + s->c1 * (gh - mi);",
                             "float m_new = (1.0f - s->c1) * mi + s->c1 * gh;"),
    "v_groups_gh_squared": ("float v_new = vi * s->b2 + (s->c2 * gh) * gh;",
                            "float v_new = vi * s->b2 + s->c2 * (gh * gh);"),
    "w_divides_m_first": ("w[i] = wdec + (neg_step * m_new) / denom;", "w[i] = wdec + neg_step * (m_new / denom);"),
    "bc2_inside_sqrt": ("float denom = sqrtf(v_new) / s->bc2 + s->eps;",
                        "float denom = sqrtf(v_new / (s->bc2 * s->bc2)) + s->eps;"),
    "eps_before_bc2": ("float denom = sqrtf(v_new) / s->bc2 + s->eps;",
                       "float denom = (sqrtf(v_new) + s->eps) / s->bc2;"),
    "decay_after_update": ("w[i] = wdec + (neg_step * m_new) / denom;",
                           "w[i] = (wi + (neg_step * m_new) / denom) * (decoupled ? s->dec : 1.0f);"),
    "step_in_f32": ("s->step = (float)(lr / (1.0 - pow(b1, tt)));",
                    "s->step = (float)lr / (float)(1.0 - pow(b1, tt));"),
    "bc2_in_f32": ("s->bc2 = (float)sqrt(1.0 - pow(b2, tt));", "s->bc2 = sqrtf((float)(1.0 - pow(b2, tt)));"),
    "decay_in_f32": ("s->dec = (float)(1.0 - lr * wd);", "s->dec = 1.0f - (float)lr * (float)wd;"),
    # the gradient's last write (an add) and the norm fused into it
    "accumulate_f16_rounds_down": ("p[i] = ora_f16_from_f32(ora_f32_from_f16(p[i]) + ora_f32_from_f16(q[i]));",
                                   "p[i] = ora_f16_from_f32(nextafterf(ora_f32_from_f16(p[i]) + ora_f32_from_f16(q[i]), 0.0f));"),
    "accumulate_f32_ignores_addend": ("p[i] = p[i] + q[i];", "p[i] = p[i];"),
    "accumulate_subtracts": ("p[i] = p[i] + q[i];", "p[i] = p[i] - q[i];"),
    "accumulate_norm_before_add": ("    ora_accumulate_grads(g, a, n, T, gdt);\n    ora_clip_grad_norms((const void* const*)g, n, T, gdt, max_norm, inv_scale, norm_out, factor_out, 0);",
                                   "    ora_clip_grad_norms((const void* const*)g, n, T, gdt, max_norm, inv_scale, norm_out, factor_out, 0);\n    ora_accumulate_grads(g, a, n, T, gdt);"),
    "odd_tail_clobbered": ("if (i & 1) return (word & 0x0000FFFFu) | ((uint32_t)h << 16);\n    return (word & 0xFFFF0000u) | (uint32_t)h;",
                           "if (i & 1) return (word & 0x0000FFFFu) | ((uint32_t)h << 16);\n    return (uint32_t)h;"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation {name}: the text to replace is not in oracle.c exactly once"
    mutant_c = tmp_path / "mutant.c"
    mutant_c.write_text(src.replace(old, new))
    lib = oracle.build(str(mutant_c), str(tmp_path / f"libmutant_{name}.so"))
    o = oracle.Oracle(lib)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(o)
        except AssertionError:
            caught.append(pin.__name__)
        except (FloatingPointError, OverflowError, ValueError, ZeroDivisionError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name}"
