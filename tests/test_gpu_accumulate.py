"""mica_accumulate_clip_grad_norms against the oracle: the gradient's last write as an add (g += a, each sum rounded
to the gradient's type) fused with ClipGradNorms ("Mica 7.7", sections "Values that stay on the card" and "The
whole model in one call").

The added gradient must be the oracle's bit for bit (two NaNs count as equal: the pages fix no NaN payload), the
norm within relative 1e-5, and the factor the oracle's bits. Lists: the tiny workload, GPT-2-shaped lists with
ragged tails, the loss-scaled list's small tensors (binary16, unscaled inside the norm), tensors not aligned for the
vector accesses, special values, a list whose chunks span several staged runs of 256 tensors, GPT-2 small at full
size, and three accumulate-then-update steps against the oracle's.
"""
import numpy as np
import pytest
import torch

import clip_tensor_adamw_gb300 as mica
import parity
import workloads

pytestmark = pytest.mark.gpu

W = workloads.WORKLOADS
OVERLAP = 6


def _gpt_sizes():
    return [int(np.prod(s)) for s in workloads._gpt2_shapes(90, 2, 1003, 67)] + [1, 7, 4097]


def _addend(st: workloads.State, seed: int) -> torch.Tensor:
    """A second contribution to every gradient, drawn like the gradient itself, as one flat buffer laid out as g."""
    other = workloads.make_state(st.wl, st.device, sizes=st.sizes)
    workloads.fill_grad(other, 1, seed=seed)
    return other


def _check(ora, st, add_st, max_norm=None, inv_scale=None):
    wl = st.wl
    max_norm = wl.max_norm if max_norm is None else max_norm
    inv_scale = wl.inv_scale if inv_scale is None else inv_scale
    _, g, _, _ = workloads.host_lists(st)
    _, a, _, _ = workloads.host_lists(add_st)
    o_norm, o_factor = ora.accumulate_clip_grad_norms(g, a, max_norm, inv_scale)
    norm, factor = mica.mica_accumulate_clip_grad_norms(st.g, add_st.g, max_norm, inv_scale)
    torch.cuda.synchronize()
    _, got, _, _ = workloads.host_lists(st)
    for k, (x, y) in enumerate(zip(got, g)):
        parity.exact(x, y, f"g[{k}]")
    parity.check_norm(norm.item(), o_norm, 0)
    if np.isfinite(o_norm):
        assert np.float32(factor.item()).view(np.uint32) == o_factor.view(np.uint32)
    return norm, factor


@pytest.mark.parametrize("name,sizes", [("tiny", None), ("gpt2_small", "gpt"), ("gpt2_small_bf16", "gpt"),
                                        ("fp16_scaled", "small")])
def test_accumulate_parity(ora, name, sizes):
    wl = W[name]
    if sizes == "gpt":
        sizes = _gpt_sizes()
    elif sizes == "small":
        sizes = list(wl.sizes[:300]) + [1, 7, 4097, 3 * 768]
    st = workloads.make_state(wl, "cuda", sizes=sizes)
    workloads.fill_grad(st, 1)
    _check(ora, st, _addend(st, 77))


def test_accumulate_repeated_calls(ora):
    """The same list three times (the cached table and its ticket reused): each call against the oracle."""
    wl = W["gpt2_small"]
    st = workloads.make_state(wl, "cuda", sizes=_gpt_sizes())
    workloads.fill_grad(st, 1)
    add = _addend(st, 78)
    for _ in range(3):
        _check(ora, st, add)


@pytest.mark.parametrize("gdt", [torch.float32, torch.float16])
def test_accumulate_unaligned_tensors(ora, gdt):
    """Tensors that start one element past a vector boundary take the element path; ragged lengths."""
    rng = np.random.Generator(np.random.PCG64(9))
    sizes = [1, 5, 8, 9, 31, 257, 4099, 20000]
    g_host, a_host, g_dev, a_dev = [], [], [], []
    for n in sizes:
        x = rng.normal(0, 3.0, size=n + 1).astype(np.float32)
        y = rng.normal(0, 3.0, size=n + 1).astype(np.float32)
        gx = torch.from_numpy(x).to(gdt).cuda()[1:]
        ay = torch.from_numpy(y).to(gdt).cuda()[1:]
        g_dev.append(gx)
        a_dev.append(ay)
        g_host.append(gx.cpu().numpy().copy())
        a_host.append(ay.cpu().numpy().copy())
    o_norm, o_factor = ora.accumulate_clip_grad_norms(g_host, a_host, 1.0)
    norm, factor = mica.mica_accumulate_clip_grad_norms(g_dev, a_dev, 1.0)
    torch.cuda.synchronize()
    for k, (x, y) in enumerate(zip(g_dev, g_host)):
        parity.exact(x.cpu().numpy(), y, f"g[{k}]")
    parity.check_norm(norm.item(), o_norm, 0)
    assert np.float32(factor.item()).view(np.uint32) == o_factor.view(np.uint32)


@pytest.mark.parametrize("values", [[float("nan")], [float("inf")], [-float("inf"), 1.0], [1e30, -1e30],
                                    [3e38, 3e38]],
                         ids=["nan", "inf", "neg_inf", "huge", "sum_overflows"])
@pytest.mark.parametrize("gdt", ["f32", "f16"])
def test_accumulate_special_values(ora, values, gdt):
    wl = W["gpt2_small"] if gdt == "f32" else W["fp16_scaled"]
    st = workloads.make_state(wl, "cuda", sizes=[4096, 333, 64])
    workloads.fill_grad(st, 1)
    add = _addend(st, 79)
    big = 6e4 if gdt == "f16" else None  # binary16: 6e4 + 6e4 overflows to infinity
    vals = [big if (big and v == 3e38) else v for v in values]
    for j, v in enumerate(vals):
        st.g[1][j] = v
        add.g[1][j] = v
    _check(ora, st, add)


def test_accumulate_empty_lists(ora):
    f = torch.zeros(1, device="cuda")
    norm, factor = mica.mica_accumulate_clip_grad_norms([], [], 1.0, 0.25, factor_out=f)
    torch.cuda.synchronize()
    assert norm.item() == 0.0 and factor.item() == 0.25
    e = [torch.empty(0, device="cuda") for _ in range(3)]
    norm, factor = mica.mica_accumulate_clip_grad_norms(e, [torch.empty(0, device="cuda") for _ in range(3)], 1.0)
    torch.cuda.synchronize()
    assert norm.item() == 0.0 and factor.item() == 1.0


def test_accumulate_over_many_staged_spans(ora):
    """4,096 tensors, three of four empty: each CTA's chunk spans four staged runs of 256 tensors, an infinity
    planted in the first octet of a later run (see test_gpu_norm_spans.py)."""
    from test_gpu_norm_spans import spanning_list
    g_host, g_dev, _ = spanning_list([float("inf")], [64])
    a_host, a_dev, _ = spanning_list([], [])
    o_norm, o_factor = ora.accumulate_clip_grad_norms(g_host, a_host, 1.0)
    norm, factor = mica.mica_accumulate_clip_grad_norms(g_dev, a_dev, 1.0)
    torch.cuda.synchronize()
    assert np.isinf(o_norm) and np.isinf(norm.item()) and factor.item() == 0.0 == float(o_factor)
    for k, (x, y) in enumerate(zip(g_dev, g_host)):
        parity.exact(x.cpu().numpy(), y, f"g[{k}]")


def test_accumulate_refuses_overlap():
    g = torch.zeros(1024, device="cuda")
    f = torch.zeros(1, device="cuda")
    L = mica.lib()
    for a in (g, g[8:]):  # the gradient as its own addend, or an addend overlapping it
        G, A = mica.TensorList([g[:512]]), mica.TensorList([a[:512]])
        st = L.mica_accumulate_clip_grad_norms(G.ptrs, A.ptrs, G.n, 1, 0, 1.0, 1.0, None, f.data_ptr(), None)
        assert st == OVERLAP, st
    G, A = mica.TensorList([g[:512]]), mica.TensorList([g[512:]])
    st = L.mica_accumulate_clip_grad_norms(G.ptrs, A.ptrs, G.n, 1, 0, 1.0, 1.0, None, g[600:].data_ptr(), None)
    assert st == OVERLAP, st  # d_factor inside an addend


def test_accumulate_gpt2_small_full_size(ora):
    """All 124,439,808 elements of GPT-2 small: every added gradient element against the oracle, and the norm."""
    wl = W["gpt2_small"]
    st = workloads.make_state(wl, "cuda")
    workloads.fill_grad(st, 1)
    add = _addend(st, 80)
    _check(ora, st, add)
    del st, add
    mica.mica_release_cache()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["gpt2_small_bf16", "fp16_scaled"])
def test_accumulate_then_update_three_steps(ora, name):
    """Three steps of (g = g_1 + g_2 with the fused norm, then AdamWSteps with its factor) against the oracle's
    same steps: the update's w, m and v identical bits."""
    wl = W[name]
    sizes = _gpt_sizes() if name != "fp16_scaled" else list(wl.sizes[:200]) + [7, 4097]
    st = workloads.make_state(wl, "cuda", sizes=sizes)
    w, _, m, v = workloads.host_lists(st)
    for t in (1, 2, 3):
        workloads.fill_grad(st, t)
        add = _addend(st, 100 + t)
        _, g, _, _ = workloads.host_lists(st)
        _, a, _, _ = workloads.host_lists(add)
        o_norm, o_factor = ora.accumulate_clip_grad_norms(g, a, wl.max_norm, wl.inv_scale)
        ora.adamw_steps(w, g, m, v, parity.hp_of(wl, t), factor=o_factor)
        norm, factor = mica.mica_accumulate_clip_grad_norms(st.g, add.g, wl.max_norm, wl.inv_scale)
        mica.mica_adamw_steps(st.w, st.g, st.m, st.v, lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps,
                              weight_decay=wl.weight_decay, step=t, factor=factor)
        torch.cuda.synchronize()
        parity.check_norm(norm.item(), o_norm, t)
        assert np.float32(factor.item()).view(np.uint32) == o_factor.view(np.uint32)
        gw, gg, gm, gv = workloads.host_lists(st)
        for k in range(len(sizes)):
            parity.exact(gg[k], g[k], f"g[{k}] t={t}")
            parity.exact(gw[k], w[k], f"w[{k}] t={t}")
            parity.exact(gm[k], m[k], f"m[{k}] t={t}")
            parity.exact(gv[k], v[k], f"v[{k}] t={t}")


@pytest.mark.parametrize("gdt,inv_scale", [("f32", 1.0), ("f32", 0.3), ("f16", 2.0 ** -16), ("f16", 0.3)],
                         ids=["f32_unscaled", "f32_scaled", "f16_pow2", "f16_scaled"])
def test_accumulate_every_unscale_mode(ora, gdt, inv_scale):
    """Each of the kernel's ways to sum the squares (float32 unscaled or scaled, binary16 with a power-of-two or any
    other unscale) against the oracle, on a GPT-2-shaped list with ragged tails."""
    wl = W["gpt2_small"] if gdt == "f32" else W["fp16_scaled"]
    st = workloads.make_state(wl, "cuda", sizes=_gpt_sizes())
    workloads.fill_grad(st, 1)
    _check(ora, st, _addend(st, 81), max_norm=1.0, inv_scale=inv_scale)


def test_accumulate_f16_list_larger_than_l2(ora):
    """A binary16 gradient of 120 MB (more than the 96 MB below which the stores ask L2 to keep the lines): every
    added element against the oracle, and the norm."""
    wl = W["fp16_scaled"]
    st = workloads.make_state(wl, "cuda", sizes=[768 * 3072] * 26 + [4097])
    workloads.fill_grad(st, 1)
    assert st.g_flat.numel() * 2 > 96 << 20
    _check(ora, st, _addend(st, 82))
    del st
    mica.mica_release_cache()
    torch.cuda.empty_cache()
