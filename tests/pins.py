"""Pins for the oracle: checks against facts that do not come from the oracle itself.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises ``AssertionError`` when the oracle disagrees with the fact it
is pinned to. ``test_oracle_pins.py`` runs them on the oracle; ``test_oracle_mutations.py`` runs them on copies of
the oracle with one plausible mistake planted each and requires every planted mistake to fail at least one pin.

What the pins hold the oracle to (no pin re-types the oracle's own formula):

* library routines: PyTorch's CPU ``torch.optim.AdamW`` / ``torch.optim.Adam`` (also with two param_groups),
  ``torch.optim.SGD`` (plain and with momentum), ``GradScaler`` and ``clip_grad_norm_``, PyTorch's
  float32 -> bfloat16 conversion, numpy's binary16 conversions and float32 add, Python's exactly rounded
  ``math.fsum``;
* closed forms: the first step from zero moments, a constant gradient over many steps (also for SGD and momentum in
  dyadic values, where every operation is exact), norms of all-ones and Pythagorean vectors, and the b1 = b2 = eps = 0 step whose weight update is lr * m / sqrt(v) of rounded moments;
* the pages' printed values (``tests/golden/printed_values.txt``): the F32 rounding of 1 - 0.999 and the BF16 codes
  of NaN and zero;
* invariants: one call over a list equals one call per group; zero_grad zeroes exactly the gradient; a factor of
  exactly inv_scale below the clip threshold.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

import oracle
from oracle import Hyper, unpack_bf16

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def f32_ulp(x) -> np.ndarray:
    x = np.abs(np.asarray(x, np.float32))
    return np.spacing(x).astype(np.float64)


def bf16_rne_reference(bits: np.ndarray) -> np.ndarray:
    """BF16 bits of float32 bit patterns by the definition of round-to-nearest-even, in float64: take the two BF16
    neighbours of |x| (truncation toward zero, and that plus one BF16 ulp of the binade, with an unbounded exponent
    so that past the largest finite value it is 2^128, which encodes as infinity), pick the nearer, and on a tie the
    one with an even last bit. NaN inputs give 0xFFFF (the pages' convention); infinities stay infinities."""
    u = np.asarray(bits, np.uint32)
    with np.errstate(invalid="ignore", over="ignore"):
        ax = (u & 0x7FFFFFFF).view(np.float32).astype(np.float64)
        lo = (u >> 16).astype(np.uint32)                      # truncated toward zero, sign kept
        mag_lo = ((lo & 0x7FFF) << 16).astype(np.uint32).view(np.float32).astype(np.float64)
        e = ((u >> 23) & 0xFF).astype(np.int64)
        ulp = np.where(e == 0, 2.0 ** -133, np.exp2((e - 134).astype(np.float64)))
        d_lo = ax - mag_lo
        d_hi = (mag_lo + ulp) - ax
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((lo & 1) == 1))
    out = np.where(pick_hi, lo + 1, lo).astype(np.uint32)
    special = ((u >> 23) & 0xFF) == 0xFF
    out[special] = lo[special]                                # infinities keep their code
    out[np.isnan(ax)] = 0xFFFF
    return out.astype(np.uint16)


def edge_f32_bits(rng: np.random.Generator, n_random: int = 1 << 18) -> np.ndarray:
    """Random float32 bit patterns plus every pattern within 2 of each BF16 rounding boundary of a sample of
    exponents, the signed zeros, infinities, NaNs and the largest finite values."""
    r = rng.integers(0, 1 << 32, size=n_random, dtype=np.uint64).astype(np.uint32)
    tops = rng.integers(0, 1 << 16, size=4096, dtype=np.uint64).astype(np.uint32) << 16
    offs = np.array([0x7FFE, 0x7FFF, 0x8000, 0x8001, 0x8002, 0, 1, 0xFFFF], np.uint32)
    edges = (tops[:, None] + offs[None, :]).ravel()
    special = np.array([0, 0x80000000, 0x7F800000, 0xFF800000, 0x7FC00000, 0xFFC00000, 0x7F800001, 0x7F7FFFFF,
                        0xFF7FFFFF, 0x7F7F8000, 0x7F7F7FFF, 0x00000001, 0x00008000, 0x00018000, 0x3F808000,
                        0x3F818000], np.uint32)
    return np.concatenate([r, edges, special])


# ------------------------------------------------------------------------------------------------------------------
# BF16
# ------------------------------------------------------------------------------------------------------------------

def pin_bf16_rounding(o: oracle.Oracle) -> None:
    """Nearest-even by definition, and PyTorch's float32 -> bfloat16 conversion on every non-NaN input."""
    bits = edge_f32_bits(_rng(1))
    got = o.bf16_from_f32_bits(bits)
    np.testing.assert_array_equal(got, bf16_rne_reference(bits))
    x = torch.from_numpy(bits.view(np.float32).copy())
    keep = ~torch.isnan(x)
    lib = x[keep].to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(got[keep.numpy()], lib)


def pin_bf16_printed(o: oracle.Oracle) -> None:
    """The pages' codes: NaN -> 0xFFFF, and BF16 0x0000 is +0.0."""
    vals = read_golden("printed_values.txt")
    nan_bits = np.array([0x7FC00000, 0xFFC00000, 0x7F800001, 0xFFFFFFFF], np.uint32)
    assert (o.bf16_from_f32_bits(nan_bits) == int(vals["bf16_of_nan"], 16)).all()
    z = o.f32_from_bf16(np.array([int(vals["bf16_zero_bits"], 16)], np.uint16))[0]
    assert z == 0.0 and not np.signbit(z)
    # widening is exact: every non-NaN BF16 pattern survives a round trip
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    back = o.bf16_from_f32_bits(o.f32_from_bf16(h).view(np.uint32))
    isnan = ((h & 0x7F80) == 0x7F80) & ((h & 0x7F) != 0)
    np.testing.assert_array_equal(back[~isnan], h[~isnan])


# ------------------------------------------------------------------------------------------------------------------
# binary16
# ------------------------------------------------------------------------------------------------------------------

def pin_f16(o: oracle.Oracle) -> None:
    """binary16 <-> float32 against numpy's conversions (every binary16; float32 near every binary16 midpoint)."""
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = o.f32_from_f16_bits(h)
    ref = h.view(np.float16).astype(np.float32)
    same = (got.view(np.uint32) == ref.view(np.uint32)) | (np.isnan(got) & np.isnan(ref))
    assert same.all()
    fin = np.isfinite(ref)
    vals = np.sort(np.unique(ref[fin].astype(np.float64)))
    mids = ((vals[1:] + vals[:-1]) / 2).astype(np.float32)
    around = (mids.view(np.uint32)[:, None].astype(np.int64) + np.arange(-2, 3)[None, :]).ravel()
    around = around[(around >= 0) & (around < (1 << 32))].astype(np.uint32)
    x = np.concatenate([around, edge_f32_bits(_rng(2), 1 << 16)]).view(np.float32)
    got16 = o.f16_bits_from_f32(x)
    with np.errstate(over="ignore", invalid="ignore"):
        ref16 = x.astype(np.float16).view(np.uint16)
    both_nan = np.isnan(x)
    np.testing.assert_array_equal(got16[~both_nan], ref16[~both_nan])
    assert np.isnan(got16[both_nan].view(np.float16)).all()


# ------------------------------------------------------------------------------------------------------------------
# the joint norm and the clip factor
# ------------------------------------------------------------------------------------------------------------------

def _exact_sumsq(grads, inv_scale: float) -> float:
    """sum of x^2, x = f32(g * inv_scale), exactly rounded (every float32 square is exact in float64)."""
    terms = []
    for g in grads:
        x = (g.astype(np.float32) * np.float32(inv_scale)).astype(np.float64)
        terms.append(x * x)
    return math.fsum(np.concatenate(terms).tolist()) if terms else 0.0


def pin_norm_fsum(o: oracle.Oracle) -> None:
    """Square sum within n * 2^-53 (relative) of the exactly rounded sum; norm = the float32 of its square root
    to within one float32 ulp. A float32 running sum is far outside this (the pages print ~1e-4 off for 295k
    squares)."""
    rng = _rng(3)
    grads = [rng.normal(0, 1e-3, size=n).astype(np.float32) for n in (295_000, 1, 7, 4097)]
    for inv in (1.0, 2.0 ** -16):
        S = o.sum_squares(grads, inv)
        ref = _exact_sumsq(grads, inv)
        n = sum(g.size for g in grads)
        assert abs(S - ref) <= n * 2.0 ** -53 * ref, (S, ref)
        norm, _, _ = o.clip_grad_norms(grads, 1.0, inv)
        assert abs(float(norm) - math.sqrt(ref)) <= f32_ulp(np.float32(math.sqrt(ref))), (norm, math.sqrt(ref))
    # float16 gradients: the norm of f32(h) * inv_scale
    h = (rng.normal(0, 1e-4, size=10_000) * 65536).astype(np.float16)
    S = o.sum_squares([h], 2.0 ** -16)
    ref = _exact_sumsq([h.astype(np.float32)], 2.0 ** -16)
    assert abs(S - ref) <= 1e4 * 2.0 ** -53 * ref


def pin_norm_closed_forms(o: oracle.Oracle) -> None:
    """All-ones of k^2 elements has norm k; (3, 4) * 2^j has norm 5 * 2^j; an empty list has norm 0."""
    for k in (1, 3, 64, 1000):
        norm, _, _ = o.clip_grad_norms([np.ones(k * k, np.float32)], 1e9)
        assert norm == np.float32(k)
    for j in (-20, 0, 10):
        g = [np.array([3.0 * 2.0 ** j], np.float32), np.array([4.0 * 2.0 ** j], np.float32)]
        norm, _, _ = o.clip_grad_norms(g, 1e9)
        assert norm == np.float32(5.0 * 2.0 ** j)
    norm, factor, S = o.clip_grad_norms([], 1.0)
    assert norm == 0.0 and S == 0.0 and factor == 1.0


def pin_clip_factor(o: oracle.Oracle) -> None:
    """PyTorch's clip_grad_norm_ coefficient: exactly 1 (so the factor is exactly inv_scale) at or below
    max_norm - 1e-6; max_norm / (norm + 1e-6) above it; NaN passes through; an infinite norm gives 0."""
    for inv in (1.0, 2.0 ** -16):
        assert o.clip_factor(0.5, 1.0, inv) == np.float32(inv)
        assert o.clip_factor(0.0, 1.0, inv) == np.float32(inv)
        f = o.clip_factor(4.0, 1.0, inv)
        assert f == np.float32(inv) * (np.float32(1.0) / (np.float32(4.0) + np.float32(1e-6)))
    assert np.isnan(o.clip_factor(np.nan, 1.0, 1.0))
    assert o.clip_factor(np.inf, 1.0, 1.0) == 0.0
    # library: torch's clip coefficient on the same norm
    rng = _rng(4)
    for _ in range(20):
        gs = [torch.from_numpy(rng.normal(0, rng.uniform(1e-4, 1e-1), size=n).astype(np.float32))
              for n in (300, 17, 1024)]
        ps = [torch.nn.Parameter(torch.zeros_like(g)) for g in gs]
        for p, g in zip(ps, gs):
            p.grad = g.clone()
        max_norm = float(rng.uniform(0.05, 2.0))
        total = torch.nn.utils.clip_grad_norm_(ps, max_norm, foreach=False)
        norm, factor, _ = o.clip_grad_norms([g.numpy() for g in gs], max_norm)
        assert abs(float(norm) - float(total)) <= 2e-6 * float(total)
        clipped = ps[0].grad[0] / gs[0][0] if gs[0][0] != 0 else None
        if clipped is not None:
            assert abs(float(clipped) - float(factor)) <= 4e-6 * float(factor) + 1e-30


# ------------------------------------------------------------------------------------------------------------------
# AdamW
# ------------------------------------------------------------------------------------------------------------------

HP0 = dict(lr=6e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)


def _torch_run(ws, gs_per_step, hp: dict, max_norm: float, inv_scale: float, adam_l2: bool = False):
    """PyTorch's own single-tensor (foreach=False, fused=False) AdamW on CPU float32, gradients unscaled and clipped
    by clip_grad_norm_ first. Returns weights, exp_avg, exp_avg_sq and the norms."""
    ps = [torch.nn.Parameter(torch.from_numpy(w.copy())) for w in ws]
    cls = torch.optim.Adam if adam_l2 else torch.optim.AdamW
    opt = cls(ps, lr=hp["lr"], betas=(hp["beta1"], hp["beta2"]), eps=hp["eps"], weight_decay=hp["weight_decay"],
              foreach=False, fused=False)
    norms = []
    for gs in gs_per_step:
        for p, g in zip(ps, gs):
            p.grad = torch.from_numpy(g.astype(np.float32)) * inv_scale
        norms.append(float(torch.nn.utils.clip_grad_norm_(ps, max_norm, foreach=False)))
        opt.step()
    st = [opt.state[p] for p in ps]
    return ([p.detach().numpy().copy() for p in ps], [s["exp_avg"].numpy().copy() for s in st],
            [s["exp_avg_sq"].numpy().copy() for s in st], norms)


def _close(a, b, rtol, atol):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    bad = ~(np.abs(a - b) <= atol + rtol * np.abs(b))
    assert not bad.any(), f"{bad.sum()} of {bad.size} differ; worst {np.max(np.abs(a - b)[bad])}"


def pin_torch_adamw(o: oracle.Oracle, adam_l2: bool = False) -> None:
    """Six steps of clip + AdamW (float32 moments) against PyTorch's CPU optimizer, with float32 and with
    loss-scaled float16 gradients."""
    rng = _rng(5 if not adam_l2 else 6)
    sizes = [37, 1, 512, 130]
    for gkind in ("f32", "f16"):
        ws = [rng.normal(0, 0.02, size=n).astype(np.float32) for n in sizes]
        steps = []
        for t in range(6):
            if gkind == "f16":
                steps.append([(rng.normal(0, 1e-3, size=n) * 65536).astype(np.float16) for n in sizes])
            else:
                steps.append([(rng.normal(0, 0.05 if t % 2 else 1e-3, size=n)).astype(np.float32) for n in sizes])
        inv = 2.0 ** -16 if gkind == "f16" else 1.0
        max_norm = 0.3
        tw, tm, tv, tn = _torch_run(ws, steps, HP0, max_norm, inv, adam_l2)
        w = [x.copy() for x in ws]
        m = [np.zeros(n, np.float32) for n in sizes]
        v = [np.zeros(n, np.float32) for n in sizes]
        for t, gs in enumerate(steps, start=1):
            gs = [g.copy() for g in gs]
            norm, factor, _ = o.clip_grad_norms(gs, max_norm, inv)
            assert abs(float(norm) - tn[t - 1]) <= 2e-6 * tn[t - 1]
            o.adamw_steps(w, gs, m, v, Hyper(step=t, **HP0), factor=factor, decoupled=not adam_l2)
        for k in range(len(sizes)):
            _close(w[k], tw[k], 1e-6, 1e-7)
            # moments: relative to the tensor's scale (a moment near a sign change has few significant bits left)
            _close(m[k], tm[k], 2e-5, 1e-5 * np.abs(tm[k]).max())
            _close(v[k], tv[k], 2e-5, 1e-5 * np.abs(tv[k]).max())


def pin_torch_adam_l2(o: oracle.Oracle) -> None:
    """Adam's coupled L2 form (g += wd * w) against PyTorch's Adam(weight_decay=wd)."""
    pin_torch_adamw(o, adam_l2=True)


def pin_first_step_closed_form(o: oracle.Oracle) -> None:
    """From m = v = 0 the first step moves w to w * (1 - lr*wd) - lr * g / (|g| + eps) (bias corrections cancel the
    (1 - b) factors), up to float32 rounding; the moments are (1 - b1) g and (1 - b2) g^2."""
    rng = _rng(7)
    g = np.concatenate([rng.normal(0, 1e-3, size=200), [1e-3, -1e-3, 0.0, 1e-12, -5.0, 3e-9]]).astype(np.float32)
    w0 = rng.normal(0, 0.02, size=g.size).astype(np.float32)
    for packed in (False, True):
        w = w0.copy()
        if packed:
            m = np.zeros((g.size + 1) // 2, np.uint32)
            v = np.zeros_like(m)
        else:
            m = np.zeros(g.size, np.float32)
            v = np.zeros(g.size, np.float32)
        hp = dict(HP0)
        o.adamw_steps([w], [g.copy()], [m], [v], Hyper(step=1, **hp))
        gd = g.astype(np.float64)
        upd = hp["lr"] * gd / (np.abs(gd) + hp["eps"])
        ref = w0.astype(np.float64) * (1 - hp["lr"] * hp["weight_decay"]) - upd
        rel = 2.0 ** -7 if packed else 4e-6  # packed moments carry BF16's 8-bit precision into the update
        _close(w, ref, 0, 2 * f32_ulp(w0) + rel * np.abs(upd) + 1e-12)
        mm = unpack_bf16(m, g.size) if packed else m
        vv = unpack_bf16(v, g.size) if packed else v
        mrel = 2.0 ** -8 if packed else 2e-7
        _close(mm, 0.1 * gd, mrel, 1e-30)
        _close(vv, 0.05 * gd * gd, mrel * 2, 1e-30)


def pin_constant_gradient(o: oracle.Oracle) -> None:
    """wd = 0, a constant gradient: m_t = (1 - b1^t) g and v_t = (1 - b2^t) g^2, so every step moves w by
    lr * g / (|g| + eps) and after t steps w = w0 - t * lr * g / (|g| + eps)."""
    rng = _rng(8)
    g = rng.normal(0, 1e-2, size=300).astype(np.float32)
    w0 = rng.normal(0, 0.02, size=g.size).astype(np.float32)
    hp = dict(HP0, weight_decay=0.0)
    w = w0.copy()
    m = np.zeros(g.size, np.float32)
    v = np.zeros(g.size, np.float32)
    T = 10
    for t in range(1, T + 1):
        o.adamw_steps([w], [g.copy()], [m], [v], Hyper(step=t, **hp))
    gd = g.astype(np.float64)
    ref = w0.astype(np.float64) - T * hp["lr"] * gd / (np.abs(gd) + hp["eps"])
    _close(w, ref, 0, T * (2 * f32_ulp(w0) + 1e-5 * hp["lr"]))
    _close(m, (1 - 0.9 ** T) * gd, 1e-5, 1e-30)
    _close(v, (1 - 0.95 ** T) * gd * gd, 1e-5, 1e-30)


def pin_packed_reads_rounded_moments(o: oracle.Oracle) -> None:
    """b1 = b2 = 0, eps = 0, t = 1: m = g and v = g*g, stored as BF16; the weight then moves by exactly
    lr * bf16(g) / sqrt(bf16(g*g)), the rounded moments (PyTorch's bfloat16 conversion rounds them here). The
    unrounded moments would give lr * sign(g), off by up to 2^-8 relative."""
    rng = _rng(9)
    g = rng.uniform(0.5, 2.0, size=257).astype(np.float32) * rng.choice([-1, 1], size=257).astype(np.float32)
    w0 = np.zeros(g.size, np.float32)
    w = w0.copy()
    m = np.zeros((g.size + 1) // 2, np.uint32)
    v = np.zeros_like(m)
    hp = Hyper(lr=1e-3, beta1=0.0, beta2=0.0, eps=0.0, weight_decay=0.0, step=1)
    o.adamw_steps([w], [g.copy()], [m], [v], hp)
    tg = torch.from_numpy(g)
    mr = tg.to(torch.bfloat16).to(torch.float64)
    vr = (tg * tg).to(torch.bfloat16).to(torch.float64)
    ref = (-1e-3 * mr / vr.sqrt()).numpy()
    _close(w, ref, 4 * 2.0 ** -24, 0)
    # the layout: element 2k in the low half of word k
    lo = (m & 0xFFFF).astype(np.uint16)
    hi = (m >> 16).astype(np.uint16)
    want = tg.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(lo, want[0::2])
    np.testing.assert_array_equal(hi[:-1], want[1::2])
    assert hi[-1] == 0  # odd n: the unused high half keeps its zero


def pin_odd_tail_untouched(o: oracle.Oracle) -> None:
    """With an odd n the high half of the last packed word is never written."""
    for n in (1, 3, 9):
        g = np.full(n, 1e-3, np.float32)
        w = np.zeros(n, np.float32)
        m = np.zeros((n + 1) // 2, np.uint32)
        v = np.zeros_like(m)
        m[-1] |= np.uint32(0xABCD0000)
        v[-1] |= np.uint32(0x12340000)
        o.adamw_steps([w], [g], [m], [v], Hyper(step=1, **HP0))
        assert (m[-1] >> 16) == 0xABCD and (v[-1] >> 16) == 0x1234


def pin_zero_grad(o: oracle.Oracle) -> None:
    """zero_grad writes the gradient as zeros and changes nothing else; without it the gradient is untouched."""
    rng = _rng(10)
    for gkind in (np.float32, np.float16):
        g = rng.normal(0, 1e-3, size=33).astype(gkind)
        outs = []
        for zg in (False, True):
            w = np.ones(33, np.float32)
            m = np.zeros(33, np.float32)
            v = np.zeros(33, np.float32)
            gg = g.copy()
            o.adamw_steps([w], [gg], [m], [v], Hyper(step=1, **HP0), zero_grad=zg)
            outs.append((w, m, v))
            if zg:
                assert (gg.view(np.uint16 if gkind == np.float16 else np.uint32) == 0).all()
            else:
                np.testing.assert_array_equal(gg, g)
        for a, b in zip(outs[0], outs[1]):
            np.testing.assert_array_equal(a, b)


def pin_list_equals_groups(o: oracle.Oracle) -> None:
    """One call over a list updates each group exactly as a call on that group alone (the multi-tensor verb's
    contract), and the list's order changes nothing."""
    rng = _rng(11)
    sizes = [5, 64, 1, 100]
    for packed in (False, True):
        ws = [rng.normal(0, 0.02, size=n).astype(np.float32) for n in sizes]
        gs = [rng.normal(0, 1e-2, size=n).astype(np.float32) for n in sizes]

        def zeros(n):
            return np.zeros((n + 1) // 2, np.uint32) if packed else np.zeros(n, np.float32)
        hp = Hyper(step=3, **HP0)
        a = ([w.copy() for w in ws], [g.copy() for g in gs], [zeros(n) for n in sizes], [zeros(n) for n in sizes])
        o.adamw_steps(*a, hp, factor=0.7)
        for k in range(len(sizes)):
            b = ([ws[k].copy()], [gs[k].copy()], [zeros(sizes[k])], [zeros(sizes[k])])
            o.adamw_steps(*b, hp, factor=0.7)
            for x, y in zip(a, b):
                np.testing.assert_array_equal(x[k], y[0])
        perm = [2, 0, 3, 1]
        c = ([ws[k].copy() for k in perm], [gs[k].copy() for k in perm], [zeros(sizes[k]) for k in perm],
             [zeros(sizes[k]) for k in perm])
        o.adamw_steps(*c, hp, factor=0.7)
        for j, k in enumerate(perm):
            for x, y in zip(a, c):
                np.testing.assert_array_equal(x[k], y[j])


def pin_scale_tensors(o: oracle.Oracle) -> None:
    """ScaleTensors: float32 cells times the factor (numpy's float32 product); binary16 cells widened, multiplied
    and rounded back to nearest-even (numpy's conversions)."""
    rng = _rng(12)
    t32 = [rng.normal(0, 1, size=n).astype(np.float32) for n in (3, 1000)]
    want = [x * np.float32(0.37) for x in t32]
    o.scale_tensors(t32, 0.37)
    for a, b in zip(t32, want):
        np.testing.assert_array_equal(a, b)
    t16 = [(rng.normal(0, 1e3, size=n)).astype(np.float16) for n in (5, 999)]
    want16 = [(x.astype(np.float32) * np.float32(2.0 ** -16 * 3)).astype(np.float16) for x in t16]
    o.scale_tensors(t16, 2.0 ** -16 * 3)
    for a, b in zip(t16, want16):
        np.testing.assert_array_equal(a.view(np.uint16), b.view(np.uint16))


def pin_accumulate(o: oracle.Oracle) -> None:
    """The gradient's last write, g + a rounded once to the gradient's type: float32 cells against numpy's float32
    add (random bit patterns and the edge cases: zeros, infinities, NaNs, subnormals, the largest values);
    binary16 cells against the exact sum (exact in float64 for two binary16 values) rounded to binary16 by numpy's
    float64 -> float16 conversion, on random bit-pattern pairs and on every pair of a set of edge values."""
    rng = _rng(31)
    x = edge_f32_bits(rng, 1 << 16).view(np.float32)
    y = rng.permutation(edge_f32_bits(rng, 1 << 16)).view(np.float32)[: x.size]
    g, a = [x.copy(), x[:7].copy()], [y.copy(), y[:7].copy()]
    o.accumulate_grads(g, a)
    with np.errstate(over="ignore", invalid="ignore"):
        want = x + y
    for got, w in ((g[0], want), (g[1], want[:7])):
        nan = np.isnan(w)
        np.testing.assert_array_equal(got.view(np.uint32)[~nan], w.view(np.uint32)[~nan])
        assert np.isnan(got[nan]).all()
    edge16 = np.array([0x0000, 0x8000, 0x0001, 0x8001, 0x03FF, 0x0400, 0x3C00, 0xBC00, 0x3C01, 0x7BFF, 0xFBFF,
                       0x7C00, 0xFC00, 0x7E00, 0x5800, 0x1400, 0x6BFF, 0xEBFF, 0x0200], np.uint16)
    ex, ey = np.meshgrid(edge16, edge16)
    hx = np.concatenate([rng.integers(0, 1 << 16, size=1 << 18).astype(np.uint16), ex.ravel()])
    hy = np.concatenate([rng.integers(0, 1 << 16, size=1 << 18).astype(np.uint16), ey.ravel()])
    g16, a16 = [hx.view(np.float16).copy()], [hy.view(np.float16).copy()]
    o.accumulate_grads(g16, a16)
    with np.errstate(over="ignore", invalid="ignore"):
        exact = hx.view(np.float16).astype(np.float64) + hy.view(np.float16).astype(np.float64)
        want16 = exact.astype(np.float16)
    nan = np.isnan(exact)
    np.testing.assert_array_equal(g16[0].view(np.uint16)[~nan], want16.view(np.uint16)[~nan])
    assert np.isnan(g16[0][nan]).all()
    # the norm fused into the write is that of the list the add leaves
    grads = [rng.normal(0, 1e-3, size=n).astype(np.float32) for n in (50_000, 3)]
    adds = [rng.normal(0, 1e-3, size=gr.size).astype(np.float32) for gr in grads]
    sums = [gr + ad for gr, ad in zip(grads, adds)]
    norm, factor = o.accumulate_clip_grad_norms(grads, adds, 0.01)
    for gr, sm in zip(grads, sums):
        np.testing.assert_array_equal(gr, sm)
    ref = math.sqrt(_exact_sumsq(sums, 1.0))
    assert abs(float(norm) - ref) <= f32_ulp(np.float32(ref)), (norm, ref)
    assert factor == np.float32(np.float32(0.01) / (norm + np.float32(1e-6)))


def pin_packed_m_float_v(o: oracle.Oracle) -> None:
    """m packed, v float32 (the page's CAdamWBF16 with v16 false). With b1 = b2 = eps = 0 and t = 1, m = bf16(g)
    and v = g*g unrounded, so the weight moves by exactly lr * bf16(g) / sqrt(g*g) (PyTorch's bfloat16 rounding
    for m). Rounding v too, or leaving m unrounded, moves it by up to 2^-8 relative more. From zero moments with the
    usual betas, the first step's moments are (1-b1) g within BF16 and (1-b2) g^2 within float32 rounding."""
    rng = _rng(13)
    g = rng.uniform(0.5, 2.0, size=301).astype(np.float32) * rng.choice([-1, 1], size=301).astype(np.float32)
    w = np.zeros(g.size, np.float32)
    m = np.zeros((g.size + 1) // 2, np.uint32)
    v = np.zeros(g.size, np.float32)
    o.adamw_steps([w], [g.copy()], [m], [v], Hyper(lr=1e-3, beta1=0.0, beta2=0.0, eps=0.0, weight_decay=0.0, step=1))
    tg = torch.from_numpy(g)
    mr = tg.to(torch.bfloat16).to(torch.float64)
    vv = (tg * tg).to(torch.float64)
    _close(w, (-1e-3 * mr / vv.sqrt()).numpy(), 4 * 2.0 ** -24, 0)
    _close(v, vv.numpy(), 2.0 ** -24, 0)
    g2 = rng.normal(0, 1e-3, size=257).astype(np.float32)
    w0 = rng.normal(0, 0.02, size=g2.size).astype(np.float32)
    w = w0.copy()
    m = np.zeros((g2.size + 1) // 2, np.uint32)
    v = np.zeros(g2.size, np.float32)
    o.adamw_steps([w], [g2.copy()], [m], [v], Hyper(step=1, **HP0))
    gd = g2.astype(np.float64)
    _close(unpack_bf16(m, g2.size), 0.1 * gd, 2.0 ** -8, 1e-30)
    _close(v, 0.05 * gd * gd, 4 * 2.0 ** -24, 1e-30)
    upd = HP0["lr"] * gd / (np.abs(gd) + HP0["eps"])
    _close(w, w0.astype(np.float64) * (1 - HP0["lr"] * HP0["weight_decay"]) - upd, 0,
           2 * f32_ulp(w0) + 2.0 ** -7 * np.abs(upd) + 1e-12)


def pin_skip_nonfinite_vs_gradscaler(o: oracle.Oracle) -> None:
    """A loss-scaled step whose gradient overflowed is skipped, as PyTorch's GradScaler skips optimizer.step(): the
    parameters and moments stay as they were; the next, finite step is the normal AdamW step on the unscaled
    gradient. (GradScaler does not clip, so max_norm is infinite here; t counts only the steps taken.)"""
    rng = _rng(14)
    n = 64
    w0 = rng.normal(0, 0.02, size=n).astype(np.float32)
    grads = [rng.normal(0, 1e-2, size=n).astype(np.float32) for _ in range(2)]
    grads[0][5] = np.inf
    scale = 1024.0
    p = torch.nn.Parameter(torch.from_numpy(w0.copy()))
    opt = torch.optim.AdamW([p], lr=HP0["lr"], betas=(HP0["beta1"], HP0["beta2"]), eps=HP0["eps"],
                            weight_decay=HP0["weight_decay"], foreach=False, fused=False)
    scaler = torch.amp.GradScaler("cpu", init_scale=scale, growth_interval=1000)
    scales = []
    for gnp in grads:
        scales.append(scaler.get_scale())
        opt.zero_grad()
        scaler.scale((p * torch.from_numpy(gnp)).sum()).backward()  # the gradient is g * scale
        scaler.step(opt)
        scaler.update()
    w = w0.copy()
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    t = 0
    for gnp, sc in zip(grads, scales):
        g_scaled = (gnp.astype(np.float64) * sc).astype(np.float32)
        inv = 1.0 / sc
        norm, factor, _ = o.clip_grad_norms([g_scaled], np.inf, inv)
        taken = bool(factor > 0)
        o.adamw_steps([w], [g_scaled.copy()], [m], [v], Hyper(step=t + 1, **HP0), factor=factor, zero_grad=True,
                      skip_nonfinite=True)
        if taken:
            t += 1
        else:
            np.testing.assert_array_equal(w, w0)
            assert not m.any() and not v.any()
    assert t == 1
    _close(w, p.detach().numpy(), 1e-6, 1e-7)
    st = opt.state[p]
    _close(m, st["exp_avg"].numpy(), 2e-5, 1e-12)
    _close(v, st["exp_avg_sq"].numpy(), 2e-5, 1e-16)


# ------------------------------------------------------------------------------------------------------------------
# parameter groups
# ------------------------------------------------------------------------------------------------------------------

def pin_torch_adamw_param_groups(o: oracle.Oracle) -> None:
    """Five steps of clip + AdamW over two parameter groups (matrices: lr 6e-4, weight decay 0.1; vectors: lr 3e-4,
    no decay) against PyTorch's CPU AdamW given the same two param_groups."""
    rng = _rng(15)
    sizes = [(24, 16), (16,), (16, 40), (40,), (7,)]
    ns = [int(np.prod(s)) for s in sizes]
    group = [0 if len(s) == 2 else 1 for s in sizes]
    hps = [dict(HP0), dict(HP0, lr=3e-4, weight_decay=0.0)]
    ws = [rng.normal(0, 0.02, size=n).astype(np.float32) for n in ns]
    steps = [[rng.normal(0, 0.05, size=n).astype(np.float32) for n in ns] for _ in range(5)]
    ps = [torch.nn.Parameter(torch.from_numpy(w.copy())) for w in ws]
    opt = torch.optim.AdamW(
        [{"params": [p for p, gr in zip(ps, group) if gr == j], "lr": hps[j]["lr"],
          "weight_decay": hps[j]["weight_decay"]} for j in range(2)],
        betas=(HP0["beta1"], HP0["beta2"]), eps=HP0["eps"], foreach=False, fused=False)
    max_norm = 0.5
    for gs in steps:
        for p, g in zip(ps, gs):
            p.grad = torch.from_numpy(g.copy())
        torch.nn.utils.clip_grad_norm_(ps, max_norm, foreach=False)
        opt.step()
    w = [x.copy() for x in ws]
    m = [np.zeros(n, np.float32) for n in ns]
    v = [np.zeros(n, np.float32) for n in ns]
    for t, gs in enumerate(steps, start=1):
        gs = [g.copy() for g in gs]
        _, factor, _ = o.clip_grad_norms(gs, max_norm)
        o.adamw_steps_grouped(w, gs, m, v, group, [Hyper(step=t, **hp) for hp in hps], factor=factor)
    for k, p in enumerate(ps):
        _close(w[k], p.detach().numpy(), 1e-6, 1e-7)
        st = opt.state[p]
        _close(m[k], st["exp_avg"].numpy(), 2e-5, 1e-5 * np.abs(st["exp_avg"].numpy()).max())
        _close(v[k], st["exp_avg_sq"].numpy(), 2e-5, 1e-5 * np.abs(st["exp_avg_sq"].numpy()).max())


# ------------------------------------------------------------------------------------------------------------------
# SGD and SGD with momentum
# ------------------------------------------------------------------------------------------------------------------

def _torch_sgd(ws, gs_per_step, lr, momentum, max_norm, inv_scale, factors=None):
    """PyTorch's CPU SGD (foreach=False). With ``factors`` each step's gradient is handed over already multiplied by
    that step's factor (float32 product) and not clipped; otherwise it is unscaled and clipped by clip_grad_norm_."""
    ps = [torch.nn.Parameter(torch.from_numpy(w.copy())) for w in ws]
    opt = torch.optim.SGD(ps, lr=lr, momentum=momentum, foreach=False)
    for t, gs in enumerate(gs_per_step):
        for p, g in zip(ps, gs):
            if factors is None:
                p.grad = torch.from_numpy(g.astype(np.float32)) * inv_scale
            else:
                p.grad = torch.from_numpy(g.astype(np.float32) * np.float32(factors[t]))
        if factors is None:
            torch.nn.utils.clip_grad_norm_(ps, max_norm, foreach=False)
        opt.step()
    bufs = [opt.state[p].get("momentum_buffer") for p in ps]
    return [p.detach().numpy().copy() for p in ps], [None if b is None else b.numpy().copy() for b in bufs]


def pin_torch_sgd(o: oracle.Oracle) -> None:
    """Six steps of SGD, and of SGD with momentum 0.9, against PyTorch's CPU SGD, with float32 and with loss-scaled
    float16 gradients. Given the same folded factor, the momentum buffers agree exactly and the weights to a few
    float32 ulps (PyTorch's w + (-lr) b may round once, as a fused multiply-add, where the page rounds twice). The
    whole clip + step agrees within float32 rounding with clip_grad_norm_ (whose coefficient PyTorch takes as
    max_norm * (1 / d), one ulp away from the quotient at times)."""
    rng = _rng(16)
    sizes = [33, 1, 300, 64]
    for gkind in ("f32", "f16"):
        for mom in (0.0, 0.9):
            ws = [rng.normal(0, 0.02, size=n).astype(np.float32) for n in sizes]
            steps = []
            for t in range(6):
                if gkind == "f16":
                    steps.append([(rng.normal(0, 1e-3, size=n) * 65536).astype(np.float16) for n in sizes])
                else:
                    steps.append([rng.normal(0, 0.05 if t % 2 else 1e-3, size=n).astype(np.float32) for n in sizes])
            inv = 2.0 ** -16 if gkind == "f16" else 1.0
            factors = [o.clip_grad_norms([g.copy() for g in gs], 0.3, inv)[1] for gs in steps]
            tw, tb = _torch_sgd(ws, steps, 0.05, mom, 0.3, inv, factors=factors)
            cw, cb = _torch_sgd(ws, steps, 0.05, mom, 0.3, inv)
            w = [x.copy() for x in ws]
            bufs = [np.zeros(n, np.float32) for n in sizes] if mom else None
            for gs, f in zip(steps, factors):
                o.sgd_steps(w, [g.copy() for g in gs], bufs, 0.05, mom, factor=f)
            w2 = [x.copy() for x in ws]
            bufs2 = [np.zeros(n, np.float32) for n in sizes] if mom else None
            for gs in steps:
                o.clip_sgd_step(w2, [g.copy() for g in gs], bufs2, 0.05, mom, 0.3, inv)
            for k in range(len(sizes)):
                _close(w[k], tw[k], 8 * 2.0 ** -24, 1e-9)
                # the coefficient's ulp reaches the weights through up to ~60 lr-sized updates: 1e-6 of their sum
                _close(w2[k], cw[k], 8 * 2.0 ** -24, 2e-8)
                if mom:
                    np.testing.assert_array_equal(bufs[k], tb[k])
                    # relative to the tensor's scale: b * mu + gh may cancel to a value with few significant bits
                    _close(bufs2[k], cb[k], 8 * 2.0 ** -24, 1e-6 * np.abs(cb[k]).max())


def pin_sgd_dyadic_closed_form(o: oracle.Oracle) -> None:
    """Dyadic values, where every float32 operation is exact: a constant gradient g, lr = 1/8, momentum 1/2 and a
    folded factor of 1/2 give b_t = gh (2 - 2^(1-t)) and w_t = w_0 - lr gh sum_j (2 - 2^(1-j)) with gh = g/2;
    plain SGD gives w_t = w_0 - t lr gh."""
    g = np.array([0.25, -0.5, 1.0, 0.0, -2.0], np.float32)
    w0 = np.array([1.0, -1.0, 0.5, 2.0, 0.0], np.float32)
    lr, mu, factor = 0.125, 0.5, 0.5
    gh = g.astype(np.float64) * factor
    for mom in (False, True):
        w = w0.copy()
        b = np.zeros(g.size, np.float32) if mom else None
        for t in range(1, 7):
            gg = g.copy()
            o.sgd_steps([w], [gg], None if b is None else [b], lr, mu if mom else 0.0, factor=factor, zero_grad=True)
            assert not gg.any()
            if mom:
                bt = gh * (2.0 - 2.0 ** (1 - t))
                np.testing.assert_array_equal(b, bt.astype(np.float32))
                acc = sum(2.0 - 2.0 ** (1 - j) for j in range(1, t + 1))
            else:
                acc = float(t)
            np.testing.assert_array_equal(w, (w0.astype(np.float64) - lr * gh * acc).astype(np.float32))


def pin_sgd_skip_vs_gradscaler(o: oracle.Oracle) -> None:
    """SGD with momentum under PyTorch's GradScaler: the step whose scaled gradient overflowed is skipped (w and the
    momentum buffer unchanged), the next one taken on the unscaled gradient."""
    rng = _rng(17)
    n = 48
    w0 = rng.normal(0, 0.02, size=n).astype(np.float32)
    grads = [rng.normal(0, 1e-2, size=n).astype(np.float32) for _ in range(3)]
    grads[1][7] = np.inf
    p = torch.nn.Parameter(torch.from_numpy(w0.copy()))
    opt = torch.optim.SGD([p], lr=0.1, momentum=0.9, foreach=False)
    scaler = torch.amp.GradScaler("cpu", init_scale=512.0, growth_interval=1000)
    scales = []
    for gnp in grads:
        scales.append(scaler.get_scale())
        opt.zero_grad()
        scaler.scale((p * torch.from_numpy(gnp)).sum()).backward()
        scaler.step(opt)
        scaler.update()
    w = w0.copy()
    b = np.zeros(n, np.float32)
    for j, (gnp, sc) in enumerate(zip(grads, scales)):
        g_scaled = (gnp.astype(np.float64) * sc).astype(np.float32)
        w_before, b_before = w.copy(), b.copy()
        o.clip_sgd_step([w], [g_scaled], [b], 0.1, 0.9, np.inf, 1.0 / sc, zero_grad=True, skip_nonfinite=True)
        if j == 1:
            np.testing.assert_array_equal(w, w_before)
            np.testing.assert_array_equal(b, b_before)
    _close(w, p.detach().numpy(), 8 * 2.0 ** -24, 1e-9)
    np.testing.assert_array_equal(b, opt.state[p]["momentum_buffer"].numpy())


def read_golden(name: str) -> dict:
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(None, 1)
            out[k] = v
    return out


def pin_printed_beta_rounding(o: oracle.Oracle) -> None:
    """The pages print that b2 = 0.999 reads 0.99900001287 in F32 and that 1 - b2 taken in F32 is 1.3e-5 too small;
    the oracle's c2 must be 1 - b2 taken in double and rounded once (the value PyTorch uses)."""
    vals = read_golden("printed_values.txt")
    b2f = np.float32(0.999)
    assert f"{float(b2f):.11f}" == vals["f32_of_0.999"]
    s = o.scalars(Hyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0, step=1))
    f32_route = np.float32(1.0) - b2f
    rel = (float(s["c2"]) - float(f32_route)) / float(s["c2"])
    printed = float(vals["rel_shortfall_1_minus_b2_in_f32"])
    assert abs(rel - printed) <= 0.05e-5, (rel, printed)  # agrees to the two digits printed
    assert s["c2"] == np.float32(0.001)


def pin_adamw_op_order(o: oracle.Oracle) -> None:
    """Single elements worked out by hand in the pages' order, one float32 operation per line
    (``tests/golden/adamw_op_order.txt``, each line re-derived exactly by ``golden_steps``): the oracle must end on
    the derivations' bits for w, m and v. Each element is one where a plausible other order (the weighted-sum
    moment, c2 (gh gh), (-step) (m / denom), bc2 inside the root, eps before the division, the decay after the
    update, or step, bc2 or dec taken in float32) rounds differently, so this pins the order to the bit."""
    import golden_steps
    for case in golden_steps.read_cases():
        x = {k: np.array([b], np.uint32).view(np.float32) for k, b in case.inputs.items()}
        w, g = x["w"].copy(), x["g"].copy()
        if case.moments == "bf16x2":
            assert (case.inputs["m"] & 0xFFFF) == 0 and (case.inputs["v"] & 0xFFFF) == 0, case.name
            m = np.array([case.inputs["m"] >> 16], np.uint32)
            v = np.array([case.inputs["v"] >> 16], np.uint32)
        else:
            m, v = x["m"].copy(), x["v"].copy()
        o.adamw_steps([w], [g], [m], [v], Hyper(**case.hp), factor=x["factor"][0])
        want = {k: case.bits[name] for k, name in case.output.items()}
        assert int(w.view(np.uint32)[0]) == want["w"], (case.name, "w", hex(int(w.view(np.uint32)[0])))
        if case.moments == "bf16x2":
            got_m, got_v = int(m[0]) & 0xFFFF, int(v[0]) & 0xFFFF
            assert got_m == want["m"] >> 16 and got_v == want["v"] >> 16, (case.name, hex(got_m), hex(got_v))
            assert (int(m[0]) >> 16) == 0 and (int(v[0]) >> 16) == 0, case.name  # n = 1: the high half untouched
        else:
            assert int(m.view(np.uint32)[0]) == want["m"], (case.name, "m")
            assert int(v.view(np.uint32)[0]) == want["v"], (case.name, "v")


ALL_PINS = [
    pin_bf16_rounding, pin_bf16_printed, pin_f16, pin_norm_fsum, pin_norm_closed_forms, pin_clip_factor,
    pin_torch_adamw, pin_torch_adam_l2, pin_first_step_closed_form, pin_constant_gradient,
    pin_packed_reads_rounded_moments, pin_odd_tail_untouched, pin_zero_grad, pin_list_equals_groups,
    pin_scale_tensors, pin_printed_beta_rounding, pin_packed_m_float_v, pin_skip_nonfinite_vs_gradscaler,
    pin_torch_adamw_param_groups, pin_torch_sgd, pin_sgd_dyadic_closed_form, pin_sgd_skip_vs_gradscaler,
    pin_adamw_op_order, pin_accumulate,
]
