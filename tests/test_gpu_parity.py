"""The CUDA path (through the C ABI) against the oracle, element by element, on the same seeded inputs.

Small cases span many work items and ragged tails and run 10 consecutive steps compared after every step; the
full-size workloads run in the launch configuration the benchmark times (the same cached tables, item sizes and
grids), compared in full (GPT-2 small, the loss-scaled list, GPT-2 XL)."""
import dataclasses
import os

import numpy as np
import pytest
import torch

import clip_tensor_adamw_gb300 as mica
import oracle
import parity
import workloads

pytestmark = pytest.mark.gpu

W = workloads.WORKLOADS


def small_gpt2_sizes(d=90, layers=2, vocab=1003, ctx=67):
    return [int(np.prod(s)) for s in workloads._gpt2_shapes(d, layers, vocab, ctx)]


RAGGED = [1, 2, 3, 5, 7, 9, 31, 33, 1025, 4097, 16385, 65537, 262147]


@pytest.fixture(scope="module")
def ora():
    return oracle.Oracle()


def test_tiny_ten_steps(ora):
    r = parity.run_parity(W["tiny"], ora=ora)
    assert r["same_factor_every_step"]


@pytest.mark.parametrize("name", ["gpt2_small", "gpt2_small_bf16", "gpt2_xl"])
@pytest.mark.parametrize("zero_grad", [False, True])
def test_small_gpt2_lists(ora, name, zero_grad):
    r = parity.run_parity(W[name], sizes=small_gpt2_sizes(), ora=ora, zero_grad=zero_grad)
    assert r["same_factor_every_step"]


@pytest.mark.parametrize("name", ["gpt2_small", "gpt2_small_bf16", "fp16_scaled"])
def test_ragged_sizes(ora, name):
    r = parity.run_parity(W[name], sizes=RAGGED, ora=ora)
    assert r["same_factor_every_step"]


@pytest.mark.parametrize("name", ["gpt2_small", "fp16_scaled"])
def test_many_tiny_tensors(ora, name):
    """30,000 tensors of 0 to 9 elements (a tenth of them empty): the norm's chunks each span more tensors than it
    stages in shared memory at once, and every AdamW pack holds hundreds of tensors, empty ones among them."""
    rng = np.random.Generator(np.random.PCG64(77))
    sizes = [int(x) for x in rng.integers(0, 10, size=30_000)]
    r = parity.run_parity(W[name], sizes=sizes, ora=ora, steps=3, zero_grad=True)
    assert r["same_factor_every_step"]


def test_loss_scaled_small(ora):
    sizes = list(W["fp16_scaled"].sizes[:700]) + [768 * 3072]
    r = parity.run_parity(W["fp16_scaled"], sizes=sizes, ora=ora, zero_grad=True)
    assert r["same_factor_every_step"]


def test_fp16_grads_packed_moments(ora):
    wl = dataclasses.replace(W["fp16_scaled"], name="fp16_packed", moments="bf16x2")
    r = parity.run_parity(wl, sizes=RAGGED + [3000, 70000], ora=ora)
    assert r["same_factor_every_step"]


def test_empty_tensors_and_list(ora):
    sizes = [0, 5, 0, 0, 4096, 0, 3]
    r = parity.run_parity(W["gpt2_small_bf16"], sizes=sizes, ora=ora, steps=3)
    assert r["same_factor_every_step"]
    # an empty list: norm 0, factor exactly inv_scale, nothing else happens
    norm, factor = mica.mica_clip_grad_norms([], 1.0, 0.25)
    torch.cuda.synchronize()
    assert norm.item() == 0.0 and factor.item() == 0.25
    mica.mica_adamw_steps([], [], [], [], lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, step=1)


@pytest.mark.parametrize("grad", ["f32", "f16"])
def test_packed_m_float_v(ora, grad):
    """m packed, v float32 (the moment type of the page's CAdamWBF16 with v16 false)."""
    base = W["fp16_scaled"] if grad == "f16" else W["gpt2_small_bf16"]
    wl = dataclasses.replace(base, name=f"packed_m_{grad}", moments="bf16x2_m")
    r = parity.run_parity(wl, sizes=small_gpt2_sizes() + RAGGED, ora=ora, zero_grad=True)
    assert r["same_factor_every_step"]


@pytest.mark.parametrize("name", ["gpt2_small", "gpt2_small_bf16", "fp16_scaled"])
def test_adam_coupled_l2(ora, name):
    """Adam with the coupled L2 term (the page's Adam case) instead of AdamW's decoupled decay."""
    r = parity.run_parity(W[name], sizes=small_gpt2_sizes() + RAGGED, ora=ora, coupled_l2=True)
    assert r["same_factor_every_step"]


@pytest.mark.parametrize("bad", [float("inf"), float("nan")], ids=["inf", "nan"])
@pytest.mark.parametrize("name", ["gpt2_small_bf16", "fp16_scaled"])
def test_skip_step_with_nonfinite_gradient(ora, name, bad):
    """A step whose gradient overflowed (its norm is not finite) leaves w, m and v as they were; the steps before
    and after it are normal; zero_grad still zeroes the gradient."""
    r = parity.run_parity(W[name], sizes=[4096, 333, 70000, 9], ora=ora, steps=4, zero_grad=True,
                          skip_nonfinite=True, grad_hook=_plant([bad]))
    g_norm, o_norm, g_factor, o_factor = r["norms"][1]
    assert not (np.float32(g_factor) > 0) and not (np.float32(o_factor) > 0)


def _misaligned_state(wl, sizes, off):
    """Tensors placed `off` elements (or packed words) past a 16-byte boundary: the element-by-element path."""
    st = workloads.make_state(wl, "cuda", sizes=[n + 8 for n in sizes])
    packed = st.packed
    st.w = [t[off:off + n] for t, n in zip(st.w, sizes)]
    st.g = [t[off:off + n] for t, n in zip(st.g, sizes)]
    words = [(n + 1) // 2 if packed else n for n in sizes]
    st.m = [t[off:off + k] for t, k in zip(st.m, words)]
    st.v = [t[off:off + k] for t, k in zip(st.v, words)]
    st.sizes = list(sizes)
    return st


@pytest.mark.parametrize("name", ["gpt2_small", "gpt2_small_bf16", "fp16_scaled"])
def test_unaligned_pointers(ora, name):
    wl = W[name]
    st = _misaligned_state(wl, [3, 17, 1000, 5001], off=1)
    lists = parity.tensor_lists(st)
    host = workloads.host_lists(st)
    for t in range(1, 4):
        for g in st.g:
            g.copy_(torch.randn(g.numel(), device="cuda", generator=workloads._gen("cuda", 100 + t)).to(g.dtype)
                    * (1e-3 if g.dtype == torch.float32 else 6.0))
        host = (host[0], [x.copy() for x in workloads.host_lists(st)[1]], host[2], host[3])
        _, d_factor = parity.gpu_step(st, lists, t)
        _, o_factor = ora.clip_adamw_step(*host, parity.hp_of(wl, t), wl.max_norm, wl.inv_scale)
        torch.cuda.synchronize()
        same = np.float32(d_factor.item()).view(np.uint32) == o_factor.view(np.uint32)
        parity.compare_state(st, host, bool(same), f"unaligned {name} step {t}")


def _plant(values):
    def hook(st, t):
        if t == 2:
            flat = st.g[1]
            k = min(len(values), flat.numel())
            flat[:k] = torch.tensor(values[:k], dtype=flat.dtype, device=flat.device)
    return hook


@pytest.mark.parametrize("values", [[float("nan")], [float("inf")], [-float("inf"), 1.0],
                                    [1e30, -1e30, 3e-39, 1e-45], [3e38, 3e38]],
                         ids=["nan", "inf", "neg_inf", "huge_and_subnormal", "near_max"])
@pytest.mark.parametrize("name", ["gpt2_small", "gpt2_small_bf16"])
def test_special_gradient_values(ora, name, values):
    r = parity.run_parity(W[name], sizes=[4096, 333, 64], ora=ora, steps=3, grad_hook=_plant(values))
    assert len(r["norms"]) == 3
    if values[0] in (float("inf"), -float("inf")) and W[name].moments == "bf16x2":
        # an infinite norm gives a zero factor, so the planted element's moments become NaN (inf * 0): the device
        # stores them as the pages' BF16 NaN code 0xFFFF (BendTorch "main.bend", part "AdamW over packed BF16
        # moments (CAdamWBF16)")
        st = r["state"]
        _, _, gm, gv = workloads.host_lists(st)
        assert int(gm[1][0]) & 0xFFFF == 0xFFFF and int(gv[1][0]) & 0xFFFF == 0xFFFF, (hex(int(gm[1][0])),
                                                                                      hex(int(gv[1][0])))


def test_no_clip_moments_overflow_to_bf16_infinity(ora):
    wl = dataclasses.replace(W["gpt2_small_bf16"], max_norm=float("inf"))
    r = parity.run_parity(wl, sizes=[64, 9], ora=ora, steps=2, grad_hook=_plant([1e30, -2e35, 3e38]))
    assert len(r["norms"]) == 2


def test_list_call_equals_per_group_calls():
    wl = W["gpt2_small_bf16"]
    sizes = small_gpt2_sizes()
    a = workloads.make_state(wl, "cuda", sizes=sizes)
    b = workloads.make_state(wl, "cuda", sizes=sizes)
    for st in (a, b):
        workloads.fill_grad(st, 1)
    factor = torch.tensor([0.37], device="cuda")
    kw = dict(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps, weight_decay=wl.weight_decay, step=1,
              factor=factor)
    mica.mica_adamw_steps(a.w, a.g, a.m, a.v, **kw)
    for k in range(len(sizes)):
        mica.mica_adamw_steps(b.w[k:k + 1], b.g[k:k + 1], b.m[k:k + 1], b.v[k:k + 1], **kw)
    torch.cuda.synchronize()
    for x, y in ((a.w_flat, b.w_flat), (a.m_flat, b.m_flat), (a.v_flat, b.v_flat)):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))


def test_deterministic_bits():
    wl = W["gpt2_small_bf16"]
    out = []
    for _ in range(2):
        st = workloads.make_state(wl, "cuda", sizes=small_gpt2_sizes())
        lists = parity.tensor_lists(st)
        norms = []
        for t in range(1, 4):
            workloads.fill_grad(st, t)
            n, _ = parity.gpu_step(st, lists, t)
            norms.append(n.item())
        out.append((norms, st.w_flat.clone(), st.m_flat.clone(), st.v_flat.clone()))
    assert out[0][0] == out[1][0]
    for x, y in zip(out[0][1:], out[1][1:]):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))


def test_padding_between_tensors_untouched():
    """Guard bands: the bytes between tensors in the flat buffers (and past the last) never change."""
    wl = W["gpt2_small_bf16"]
    sizes = RAGGED
    st = workloads.make_state(wl, "cuda", sizes=sizes)
    sentinel = {}
    for name in ("w_flat", "g_flat", "m_flat", "v_flat"):
        flat = getattr(st, name)
        mask = torch.ones(flat.numel(), dtype=torch.bool, device="cuda")
        for view in getattr(st, name[0]):
            if view.numel():
                start = (view.data_ptr() - flat.data_ptr()) // flat.element_size()
                mask[start:start + view.numel()] = False
        as_int = flat.view(torch.int16) if flat.element_size() == 2 else flat.view(torch.int32)
        bits = torch.randint(-2**15, 2**15, (flat.numel(),), device="cuda").to(as_int.dtype)
        as_int[mask] = bits[mask]
        sentinel[name] = (mask, as_int[mask].clone())
    lists = parity.tensor_lists(st)
    for t in range(1, 3):
        workloads.fill_grad(st, t)
        for name in ("g_flat",):  # fill_grad writes the whole flat gradient: restore the guard bands
            mask, vals = sentinel[name]
            flat = getattr(st, name)
            (flat.view(torch.int16) if flat.element_size() == 2 else flat.view(torch.int32))[mask] = vals
        parity.gpu_step(st, lists, t, zero_grad=True)
    torch.cuda.synchronize()
    for name, (mask, vals) in sentinel.items():
        flat = getattr(st, name)
        as_int = flat.view(torch.int16) if flat.element_size() == 2 else flat.view(torch.int32)
        assert torch.equal(as_int[mask], vals), f"{name}: a guard band changed"


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16])
def test_scale_tensors(ora, dtype):
    gen = workloads._gen("cuda", 7)
    ts = [torch.randn(n, device="cuda", generator=gen).mul(300.0).to(dtype) for n in RAGGED]
    ts[3][0] = float("nan")
    ts[4][1] = float("inf")
    host = [t.cpu().numpy().copy() for t in ts]
    mica.mica_scale_tensors(ts, 0.3)
    ora.scale_tensors(host, 0.3)
    dev_factor = torch.tensor([2.0 ** -16], device="cuda")
    mica.mica_scale_tensors(ts, 123.0, d_factor=dev_factor)  # the device factor wins over the host one
    ora.scale_tensors(host, 2.0 ** -16)
    torch.cuda.synchronize()
    for k, t in enumerate(ts):
        parity.exact(t.cpu().numpy(), host[k], f"scale {dtype} [{k}]")


# ------------------------------------------------------------------------------------------------------------------
# AdamW over parameter groups; SGD and SGD with momentum
# ------------------------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["gpt2_small", "gpt2_small_bf16", "fp16_scaled"])
def test_param_groups(ora, name):
    """Matrices with decay, vectors without and at half the lr, in one launch, against the oracle's per-group step."""
    if name == "fp16_scaled":
        shapes = list(W[name].shapes[:700]) + [(768, 3072)] * 2
    else:
        shapes = workloads._gpt2_shapes(90, 2, 1003, 67)
    sizes = [int(np.prod(s)) for s in shapes]
    r = parity.run_parity_groups(W[name], parity.decay_groups(shapes), sizes=sizes, ora=ora, zero_grad=True)
    assert r["same_factor_every_step"]


def test_param_groups_ragged_and_many(ora):
    """Eight groups (the most one call takes) assigned round-robin over ragged sizes."""
    group = [k % 8 for k in range(len(RAGGED))]
    wl = W["gpt2_small_bf16"]
    st_hps = [dict(lr=wl.lr * (1 + j) / 8, weight_decay=0.02 * j) for j in range(8)]
    orig = parity.group_hps
    parity.group_hps = lambda _wl: st_hps
    try:
        r = parity.run_parity_groups(wl, group, sizes=RAGGED, ora=ora)
    finally:
        parity.group_hps = orig
    assert r["same_factor_every_step"]


def test_param_groups_index_checked_on_cached_list():
    """A list first stepped with two groups, then called with one group: refused, not run with a missing group."""
    wl = W["tiny"]
    st = workloads.make_state(wl, "cuda")
    Wl, G, M, V = parity.tensor_lists(st)
    gi = mica.GroupIndex([0, 1, 0, 1])
    kw = dict(beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps, step=1)
    mica.mica_adamw_steps_grouped(Wl, G, M, V, gi, parity.group_hps(wl), **kw)
    with pytest.raises(mica.MicaError, match="MICA_ERR_COUNT"):
        mica.mica_adamw_steps_grouped(Wl, G, M, V, gi, parity.group_hps(wl)[:1], **kw)
    mica.mica_sync()


@pytest.mark.parametrize("momentum", [0.0, 0.9])
@pytest.mark.parametrize("name,sizes", [("tiny", None), ("gpt2_small", "small"), ("gpt2_small", "ragged"),
                                        ("fp16_scaled", "scaled")])
def test_sgd(ora, name, sizes, momentum):
    sz = {None: None, "small": small_gpt2_sizes(), "ragged": RAGGED,
          "scaled": list(W["fp16_scaled"].sizes[:700]) + [768 * 3072]}[sizes]
    r = parity.run_parity_sgd(W[name], momentum, sizes=sz, ora=ora, zero_grad=(sizes == "ragged"))
    assert r["same_factor_every_step"]


@pytest.mark.parametrize("momentum", [0.0, 0.9])
def test_sgd_full_size(ora, momentum):
    r = parity.run_parity_sgd(W["gpt2_small"], momentum, ora=ora, steps=4, check_every_step=False)
    assert r["same_factor_every_step"]


def test_sgd_skip_step_with_nonfinite_gradient(ora):
    def poison(st, t):
        if t == 2:
            st.g[4].view(-1)[5] = float("inf")  # tensor 4 holds 7 elements
    r = parity.run_parity_sgd(W["fp16_scaled"], 0.9, sizes=RAGGED, ora=ora, steps=4, zero_grad=True,
                              skip_nonfinite=True, grad_hook=poison)
    assert r["same_factor_every_step"]


def test_sgd_unaligned(ora):
    """Tensors one element past a 16-byte boundary take the element path."""
    wl = W["gpt2_small"]
    st = _misaligned_state(wl, [1, 7, 9, 1000, 4099], off=1)
    for t in range(1, 4):
        for g in st.g:
            g.copy_(torch.randn(g.numel(), device="cuda", generator=workloads._gen("cuda", 200 + t)) * 0.05)
        hw, hg, hb, _ = workloads.host_lists(st) if t == 1 else (hw, workloads.host_lists(st)[1], hb, None)
        d_norm, d_factor = mica.mica_clip_grad_norms(st.g, wl.max_norm)
        mica.mica_sgd_steps(st.w, st.g, st.m, lr=parity.SGD_LR, momentum=0.9, factor=d_factor)
        _, o_factor = ora.clip_sgd_step(hw, hg, hb, parity.SGD_LR, 0.9, wl.max_norm)
        torch.cuda.synchronize()
        assert np.float32(d_factor.item()) == o_factor
        gw, _, gb, _ = workloads.host_lists(st)
        for k in range(len(st.sizes)):
            parity.exact(gw[k], hw[k], f"step {t} w[{k}]")
            parity.exact(gb[k], hb[k], f"step {t} buf[{k}]")
    mica.mica_sync()


# ------------------------------------------------------------------------------------------------------------------
# the full-size workloads, in the benchmark's launch configuration
# ------------------------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["gpt2_small", "gpt2_small_bf16", "fp16_scaled"])
def test_full_size_ten_steps(ora, name):
    r = parity.run_parity(W[name], ora=ora, check_every_step=False)
    assert r["same_factor_every_step"]
    if name != "fp16_scaled":  # the clip fires on these two (expected norms ~11 and ~112)
        assert all(g > 1.0 for g, _, _, _ in r["norms"])


def test_gpt2_xl_full_two_steps(ora):
    """GPT-2 XL (1,557,611,200 parameters in 580 tensors, packed BF16 moments) in the benchmark's launch
    configuration: two consecutive steps through the one-step entry point, the norm and every element of w, g, m and
    v compared with the oracle after each step."""
    r = parity.run_parity(W["gpt2_xl"], ora=ora, steps=2, fused=True)
    assert r["same_factor_every_step"]
    assert all(g > 1.0 for g, _, _, _ in r["norms"])  # the clip fires (expected norm ~3.9)
    del r
    torch.cuda.empty_cache()


# ------------------------------------------------------------------------------------------------------------------
# the per-list table cache
# ------------------------------------------------------------------------------------------------------------------

def test_table_cache_eviction_and_release(ora):
    """More distinct lists than the cache holds (it is then emptied and refilled), and mica_release_cache between
    steps: every step's norm and update still match the oracle."""
    wl = W["tiny"]
    st = workloads.make_state(wl, "cuda")
    workloads.fill_grad(st, 1)
    host_g = workloads.host_lists(st)[1]
    factor = torch.empty(1, device="cuda")
    norm = torch.empty(1, device="cuda")
    # 1,100 distinct one-tensor lists (views at different offsets of the first gradient): each gets its own table
    g0 = st.g[0]
    for i in range(1100):
        view = g0[i:i + 64]
        mica.mica_clip_grad_norms([view], 1e9, 1.0, norm_out=norm, factor_out=factor)
        if i % 250 == 0 or i == 1099:
            o_norm, _, _ = ora.clip_grad_norms([host_g[0][i:i + 64].copy()], 1e9)
            torch.cuda.synchronize()
            parity.check_norm(np.float32(norm.item()), o_norm, i)
    mica.mica_release_cache()
    # a full step after the release rebuilds its tables and still matches
    r = parity.run_parity(wl, steps=2, ora=ora)
    assert r["same_factor_every_step"]
    mica.mica_sync()


# ------------------------------------------------------------------------------------------------------------------
# resume, and the synchronous debug tier
# ------------------------------------------------------------------------------------------------------------------

def test_resume_from_saved_state():
    """The optimizer's state is the caller's buffers and the step count: saving w, m, v to the host after step 3,
    restoring them into new buffers and going on from t = 4 gives the same bits as six uninterrupted steps."""
    wl = W["gpt2_small_bf16"]
    sizes = small_gpt2_sizes()
    a = workloads.make_state(wl, "cuda", sizes=sizes)
    la = parity.tensor_lists(a)
    for t in range(1, 7):
        workloads.fill_grad(a, t)
        parity.gpu_step(a, la, t)
    b = workloads.make_state(wl, "cuda", sizes=sizes)
    lb = parity.tensor_lists(b)
    for t in range(1, 4):
        workloads.fill_grad(b, t)
        parity.gpu_step(b, lb, t)
    torch.cuda.synchronize()
    saved = [x.cpu().clone() for x in (b.w_flat, b.m_flat, b.v_flat)]
    c = workloads.make_state(wl, "cuda", sizes=sizes, seed=12345)  # other buffers, other initial values
    for dst, src in zip((c.w_flat, c.m_flat, c.v_flat), saved):
        dst.copy_(src)
    lc = parity.tensor_lists(c)
    for t in range(4, 7):
        workloads.fill_grad(c, t, seed=wl.seed)
        parity.gpu_step(c, lc, t)
    torch.cuda.synchronize()
    for x, y in ((a.w_flat, c.w_flat), (a.m_flat, c.m_flat), (a.v_flat, c.v_flat)):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    mica.mica_sync()


def test_sync_debug_tier(tmp_path):
    """With MICA_SYNC_DEBUG=1 every call waits for its own kernels; a step still matches the oracle."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = ("import sys; sys.path[:0] = [%r, %r]; import parity, workloads; "
            "r = parity.run_parity(workloads.WORKLOADS['tiny'], steps=2); "
            "assert r['same_factor_every_step']; print('ok')" % (root, os.path.join(root, "tests")))
    env = dict(os.environ, MICA_SYNC_DEBUG="1")
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0 and "ok" in out.stdout, out.stderr[-2000:]


@pytest.mark.parametrize("env", [{"MICA_ITEM_OCTS": "16"},
                                 {"MICA_ITEM_OCTS": "64", "MICA_UPDATE_GRID": "items"},
                                 {"MICA_UPDATE_GRID": "items"}],
                         ids=["items_16", "items_64_one_cta_each", "one_cta_each"])
def test_item_size_and_grid_overrides(env):
    """The tuning overrides change how a list is cut into work items (MICA_ITEM_OCTS: octets per slice, and with it
    which tensors are packed) and how the update grid takes them (MICA_UPDATE_GRID=items: one CTA per item instead
    of the persistent queue); every element still matches the oracle, for AdamW (float32, packed BF16, binary16
    gradients) and SGD with momentum."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = ("import sys; sys.path[:0] = [%r, %r]; import parity, workloads\n"
            "R = %r\n"
            "for name in ('gpt2_small', 'gpt2_small_bf16', 'fp16_scaled'):\n"
            "    parity.run_parity(workloads.WORKLOADS[name], sizes=R + R[::-1], steps=3)\n"
            "parity.run_parity_sgd(workloads.WORKLOADS['gpt2_small'], 0.9, sizes=R, steps=3)\n"
            "print('ok')\n" % (root, os.path.join(root, "tests"), RAGGED))
    out = subprocess.run([sys.executable, "-c", code], env=dict(os.environ, **env), capture_output=True, text=True,
                         timeout=600)
    assert out.returncode == 0 and "ok" in out.stdout, out.stderr[-2000:]
