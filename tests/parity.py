"""Shared machinery of the GPU parity tests: run the step through the C ABI (via the binding) and through the oracle
on the same seeded inputs, and compare them element by element.

Tolerances (the optimizer-step benchmark's):
* joint norm: relative 1e-5;
* weights and float32 moments: |gpu - oracle| <= 1e-6 * |oracle| + 1e-7;
* packed BF16 moments: bit-exact, or one BF16 ulp apart where the float32 values before rounding differ; with the
  same factor on both sides, every packed word identical (a NaN moment must carry the pages' code 0xFFFF).
The kernels are written to be bit-identical to the oracle, so on top of those tolerances every test also requires
identical bits wherever both sides used the same clip factor (the factor is a float32; the two sides compute it
from square sums that agree to ~1e-13, so in practice it always has the same bits).
"""
from __future__ import annotations

import numpy as np
import torch

import clip_tensor_adamw_gb300 as mica
import oracle
import workloads

NORM_RTOL = 1e-5


def f32_close(a: np.ndarray, b: np.ndarray, what: str) -> None:
    a64, b64 = a.astype(np.float64), b.astype(np.float64)
    same_nan = np.isnan(a64) & np.isnan(b64)
    same_inf = np.isinf(a64) & np.isinf(b64) & (np.sign(a64) == np.sign(b64))
    ok = same_nan | same_inf | (np.abs(a64 - b64) <= 1e-6 * np.abs(b64) + 1e-7)
    if not ok.all():
        i = np.nonzero(~ok)[0][:5]
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} outside tolerance; e.g. idx {i.tolist()} "
                             f"gpu {a[i].tolist()} oracle {b[i].tolist()}")


def bf16_within_one_ulp(a_words: np.ndarray, b_words: np.ndarray, n: int, what: str) -> np.ndarray:
    """Returns the mask of elements whose BF16 codes differ (each by at most one ulp, else it raises)."""
    a = np.empty(2 * a_words.size, np.int64)
    b = np.empty(2 * b_words.size, np.int64)
    a[0::2], a[1::2] = a_words & 0xFFFF, a_words >> 16
    b[0::2], b[1::2] = b_words & 0xFFFF, b_words >> 16
    a, b = a[:n], b[:n]

    def ordered(h):  # BF16 codes on one monotone integer line
        return np.where(h & 0x8000, -(h & 0x7FFF), h)
    nan_a = ((a & 0x7F80) == 0x7F80) & ((a & 0x7F) != 0)
    nan_b = ((b & 0x7F80) == 0x7F80) & ((b & 0x7F) != 0)
    diff = np.abs(ordered(a) - ordered(b))
    bad = (diff > 1) & ~(nan_a & nan_b)
    if bad.any():
        i = np.nonzero(bad)[0][:5]
        raise AssertionError(f"{what}: {int(bad.sum())} BF16 values more than one ulp apart; idx {i.tolist()}")
    return (diff != 0) & ~(nan_a & nan_b)


def exact(a: np.ndarray, b: np.ndarray, what: str) -> None:
    """Identical bits. For float arrays two NaNs count as equal whatever their payloads (the pages fix no float32
    NaN code, and the CPU and the GPU make different ones); integer arrays (packed BF16 words) must match bit for
    bit, NaN codes included."""
    bits = {2: np.uint16, 4: np.uint32}[a.dtype.itemsize]
    au, bu = a.view(bits), b.view(bits)
    neq = au != bu
    if a.dtype.kind == "f":
        neq &= ~(np.isnan(a) & np.isnan(b))
    if neq.any():
        diff = np.nonzero(neq)[0]
        raise AssertionError(f"{what}: {diff.size} of {a.size} differ in bits; first idx {diff[:5].tolist()}")


def check_norm(g_norm, o_norm, t) -> None:
    """The device norm against the oracle's: relative 1e-5, or the same NaN / infinity."""
    g, o = float(g_norm), float(o_norm)
    if np.isfinite(o):
        assert abs(g - o) <= NORM_RTOL * abs(o), (t, g, o)
    else:
        assert (np.isnan(g) and np.isnan(o)) or g == o, (t, g, o)


def hp_of(wl: workloads.Workload, t: int) -> oracle.Hyper:
    return oracle.Hyper(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps, weight_decay=wl.weight_decay, step=t)


def gpu_step(st: workloads.State, lists, t: int, zero_grad: bool = False, max_norm: float | None = None,
             norm_out=None, factor_out=None, coupled_l2: bool = False, skip_nonfinite: bool = False,
             fused: bool = False):
    """One clip + AdamW step of the hot path on the device, through the binding: one C-ABI call each for the norm
    and the update, or (``fused``) the one call of mica_clip_adamw_step."""
    wl = st.wl
    W, G, M, V = lists
    if fused:
        return mica.mica_clip_adamw_step(W, G, M, V, max_norm=wl.max_norm if max_norm is None else max_norm,
                                         inv_scale=wl.inv_scale, lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2,
                                         eps=wl.eps, weight_decay=wl.weight_decay, step=t, zero_grad=zero_grad,
                                         norm_out=norm_out, factor_out=factor_out, coupled_l2=coupled_l2,
                                         skip_nonfinite=skip_nonfinite)
    norm, factor = mica.mica_clip_grad_norms(G, wl.max_norm if max_norm is None else max_norm, wl.inv_scale,
                                             norm_out=norm_out, factor_out=factor_out)
    mica.mica_adamw_steps(W, G, M, V, lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps,
                          weight_decay=wl.weight_decay, step=t, zero_grad=zero_grad, factor=factor,
                          coupled_l2=coupled_l2, skip_nonfinite=skip_nonfinite)
    return norm, factor


def tensor_lists(st: workloads.State):
    W = mica.TensorList(st.w)
    return W, mica.TensorList(st.g), mica.TensorList(st.m, W.counts), mica.TensorList(st.v, W.counts)


def compare_state(st: workloads.State, host, same_factor: bool, tag: str) -> None:
    """Compare the device state with the oracle's host lists ``host`` = (w, g, m, v)."""
    gw, gg, gm, gv = workloads.host_lists(st)
    ow, og, om, ov = host
    for k, n in enumerate(st.sizes):
        if n == 0:
            continue
        f32_close(gw[k], ow[k], f"{tag} w[{k}]")
        if same_factor:
            exact(gw[k], ow[k], f"{tag} w[{k}] bits")
            exact(gg[k], og[k], f"{tag} g[{k}] bits")
        for name, gx, ox, packed in (("m", gm[k], om[k], st.m_packed), ("v", gv[k], ov[k], st.packed)):
            if packed:
                bf16_within_one_ulp(gx, ox, n, f"{tag} {name}[{k}]")
                if same_factor:
                    # the same factor: every packed word identical, NaN codes included (a NaN moment is stored as
                    # the pages' 0xFFFF, not as a canonical NaN)
                    exact(gx, ox, f"{tag} packed {name}[{k}] words")
            else:
                f32_close(gx, ox, f"{tag} {name}[{k}]")
                if same_factor:
                    exact(gx, ox, f"{tag} {name}[{k}] bits")


def run_parity(wl: workloads.Workload, sizes=None, steps: int | None = None, zero_grad: bool = False,
               seed: int | None = None, ora: oracle.Oracle | None = None, check_every_step: bool = True,
               grad_hook=None, coupled_l2: bool = False, skip_nonfinite: bool = False, fused: bool = False) -> dict:
    """Both sides from the same initial state for ``steps`` steps, each step's gradient drawn on the device and
    copied to the oracle. Compares the norm every step and the state every step (or only at the end)."""
    ora = ora or oracle.Oracle()
    steps = wl.steps if steps is None else steps
    st = workloads.make_state(wl, "cuda", sizes=sizes, seed=seed)
    lists = tensor_lists(st)
    host = workloads.host_lists(st)
    norms = []
    same_all = True
    for t in range(1, steps + 1):
        workloads.fill_grad(st, t, seed=seed)
        if grad_hook is not None:
            grad_hook(st, t)
        host_g = [x.detach().cpu().numpy().copy() for x in st.g]  # this step's gradient, for the oracle
        host = (host[0], host_g, host[2], host[3])
        d_norm, d_factor = gpu_step(st, lists, t, zero_grad=zero_grad, coupled_l2=coupled_l2,
                                    skip_nonfinite=skip_nonfinite, fused=fused)
        o_norm, o_factor = ora.clip_adamw_step(*host, hp_of(wl, t), wl.max_norm, wl.inv_scale, zero_grad=zero_grad,
                                               decoupled=not coupled_l2, skip_nonfinite=skip_nonfinite)
        torch.cuda.synchronize()
        g_norm = np.float32(d_norm.item())
        g_factor = np.float32(d_factor.item())
        check_norm(g_norm, o_norm, t)
        same = g_factor.view(np.uint32) == o_factor.view(np.uint32)
        same_all &= bool(same)
        norms.append((float(g_norm), float(o_norm), float(g_factor), float(o_factor)))
        if check_every_step or t == steps:
            compare_state(st, host, bool(same), f"{wl.name} step {t}")
    mica.mica_sync()  # raises if a kernel's bounded pipeline wait gave up
    return {"norms": norms, "same_factor_every_step": same_all, "state": st}


# ------------------------------------------------------------------------------------------------------------------
# AdamW over parameter groups; SGD and SGD with momentum
# ------------------------------------------------------------------------------------------------------------------

def decay_groups(shapes) -> list[int]:
    """The usual split of a transformer's parameters: matrices (group 0) decay, vectors (group 1) do not."""
    return [0 if len(s) >= 2 else 1 for s in shapes]


def group_hps(wl: workloads.Workload) -> list[dict]:
    return [dict(lr=wl.lr, weight_decay=wl.weight_decay), dict(lr=wl.lr / 2, weight_decay=0.0)]


def run_parity_groups(wl: workloads.Workload, group, sizes=None, steps: int | None = None, zero_grad: bool = False,
                      ora: oracle.Oracle | None = None, check_every_step: bool = True) -> dict:
    """As run_parity, with the update split into parameter groups (``group[k]`` the group of tensor k)."""
    ora = ora or oracle.Oracle()
    steps = wl.steps if steps is None else steps
    st = workloads.make_state(wl, "cuda", sizes=sizes)
    W, G, M, V = tensor_lists(st)
    gi = mica.GroupIndex(group)
    hps = group_hps(wl)
    host = workloads.host_lists(st)
    same_all = True
    for t in range(1, steps + 1):
        workloads.fill_grad(st, t)
        host = (host[0], [x.copy() for x in workloads.host_lists(st)[1]], host[2], host[3])
        d_norm, d_factor = mica.mica_clip_grad_norms(G, wl.max_norm, wl.inv_scale)
        mica.mica_adamw_steps_grouped(W, G, M, V, gi, hps, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps, step=t,
                                      zero_grad=zero_grad, factor=d_factor)
        o_norm, o_factor, _ = ora.clip_grad_norms(host[1], wl.max_norm, wl.inv_scale)
        ohps = [oracle.Hyper(lr=h["lr"], beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps, weight_decay=h["weight_decay"],
                             step=t) for h in hps]
        ora.adamw_steps_grouped(*host, group, ohps, factor=o_factor, zero_grad=zero_grad)
        torch.cuda.synchronize()
        check_norm(np.float32(d_norm.item()), o_norm, t)
        same = np.float32(d_factor.item()).view(np.uint32) == o_factor.view(np.uint32)
        same_all &= bool(same)
        if check_every_step or t == steps:
            compare_state(st, host, bool(same), f"{wl.name} groups step {t}")
    mica.mica_sync()
    return {"same_factor_every_step": same_all, "state": st}


SGD_LR = 0.1


def run_parity_sgd(wl: workloads.Workload, momentum: float, sizes=None, steps: int | None = None,
                   zero_grad: bool = False, skip_nonfinite: bool = False, grad_hook=None,
                   ora: oracle.Oracle | None = None, check_every_step: bool = True) -> dict:
    """Clip + SGD (momentum 0: no buffers) or clip + SGD with momentum, the momentum buffers being the workload's
    float32 first-moment buffers (zeros), against the oracle, element by element every step."""
    assert wl.moments == "f32"
    ora = ora or oracle.Oracle()
    steps = wl.steps if steps is None else steps
    st = workloads.make_state(wl, "cuda", sizes=sizes)
    W, G, M, _ = tensor_lists(st)
    B = M if momentum else None
    hw, _, hb, _ = workloads.host_lists(st)
    same_all = True
    for t in range(1, steps + 1):
        workloads.fill_grad(st, t)
        if grad_hook is not None:
            grad_hook(st, t)
        hg = [x.copy() for x in workloads.host_lists(st)[1]]
        d_norm, d_factor = mica.mica_clip_grad_norms(G, wl.max_norm, wl.inv_scale)
        mica.mica_sgd_steps(W, G, B, lr=SGD_LR, momentum=momentum, zero_grad=zero_grad, factor=d_factor,
                            skip_nonfinite=skip_nonfinite)
        o_norm, o_factor = ora.clip_sgd_step(hw, hg, hb if momentum else None, SGD_LR, momentum, wl.max_norm,
                                             wl.inv_scale, zero_grad=zero_grad, skip_nonfinite=skip_nonfinite)
        torch.cuda.synchronize()
        check_norm(np.float32(d_norm.item()), o_norm, t)
        same = np.float32(d_factor.item()).view(np.uint32) == o_factor.view(np.uint32)
        same_all &= bool(same)
        if check_every_step or t == steps:
            gw, gg, gb, _ = workloads.host_lists(st)
            tag = f"{wl.name} sgd(mu={momentum}) step {t}"
            for k, n in enumerate(st.sizes):
                if n == 0:
                    continue
                f32_close(gw[k], hw[k], f"{tag} w[{k}]")
                if momentum:
                    f32_close(gb[k], hb[k], f"{tag} buf[{k}]")
                if same:
                    exact(gw[k], hw[k], f"{tag} w[{k}] bits")
                    exact(gg[k], hg[k], f"{tag} g[{k}] bits")
                    if momentum:
                        exact(gb[k], hb[k], f"{tag} buf[{k}] bits")
    mica.mica_sync()
    return {"same_factor_every_step": same_all, "state": st}
