"""mica_clip_adamw_step, ClipGradNorms and AdamWSteps as one step, against the oracle element by element.

By default the step is the two launches of the separate entry points (the norm keeping a gradient that fits in L2
there for the update); with MICA_FUSED=1 it is one cooperative launch (the norm's chunks, a bounded grid-wide wait,
the update reading the gradient from L2). Both paths are compared with the oracle on the same seeded inputs, after
every step, and with each other."""
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
RAGGED = [1, 2, 3, 5, 7, 9, 31, 33, 1025, 4097, 16385, 65537, 262147]


@pytest.fixture(scope="module")
def ora():
    return oracle.Oracle()


@pytest.fixture
def fused_env(monkeypatch):
    """MICA_FUSED set for one test (the library reads it at each call)."""
    def set_(value):
        if value is None:
            monkeypatch.delenv("MICA_FUSED", raising=False)
        else:
            monkeypatch.setenv("MICA_FUSED", value)
    return set_


def small_gpt2_sizes(d=90, layers=2, vocab=1003, ctx=67):
    return [int(np.prod(s)) for s in workloads._gpt2_shapes(d, layers, vocab, ctx)]


@pytest.mark.parametrize("mode", ["1", None], ids=["cooperative", "two_launches"])
@pytest.mark.parametrize("name", ["tiny", "gpt2_small", "gpt2_small_bf16", "fp16_scaled"])
def test_fused_small_lists_ten_steps(ora, fused_env, name, mode):
    """Ten steps through the one-step entry point, each path, compared after every step."""
    fused_env(mode)
    wl = W[name]
    sizes = None if name == "tiny" else (small_gpt2_sizes() + RAGGED if name != "fp16_scaled"
                                         else list(wl.sizes[:700]) + [768 * 3072] + RAGGED)
    r = parity.run_parity(wl, sizes=sizes, ora=ora, fused=True)
    assert r["same_factor_every_step"]


@pytest.mark.parametrize("moments", ["bf16x2_m", "f32"])
def test_fused_options(ora, fused_env, moments):
    """The cooperative launch with packed m and float32 v, Adam's coupled L2 form, zero_grad."""
    fused_env("1")
    wl = dataclasses.replace(W["fp16_scaled"], name=f"fused_{moments}", moments=moments)
    sizes = list(wl.sizes[:300]) + RAGGED
    r = parity.run_parity(wl, sizes=sizes, ora=ora, zero_grad=True, coupled_l2=(moments == "f32"), fused=True,
                          steps=4)
    assert r["same_factor_every_step"]


@pytest.mark.parametrize("bad", [float("inf"), float("nan")], ids=["inf", "nan"])
def test_fused_skip_step_with_nonfinite_gradient(ora, fused_env, bad):
    """In the cooperative launch, a step whose norm is not finite leaves w, m, v as they were (the steps around it
    are normal)."""
    fused_env("1")

    def plant(st, t):
        if t == 2:
            st.g[1][:1] = torch.tensor([bad], dtype=st.g[1].dtype, device="cuda")
    r = parity.run_parity(W["fp16_scaled"], sizes=[4096, 333, 70000, 9], ora=ora, steps=4, zero_grad=True,
                          skip_nonfinite=True, grad_hook=plant, fused=True)
    assert not (np.float32(r["norms"][1][2]) > 0)


def test_fused_and_two_launches_agree(fused_env):
    """The same list stepped by the fused launch and by the two launches gives the same bits whenever the two norms
    are the same float32 (they are summed in different groupings), three steps in a row."""
    wl = W["fp16_scaled"]
    sizes = list(wl.sizes[:2000]) + [768 * 3072, 5001]
    out = {}
    for mode in ("1", "0"):
        fused_env(mode)
        st = workloads.make_state(wl, "cuda", sizes=sizes)
        lists = parity.tensor_lists(st)
        norms = []
        for t in range(1, 4):
            workloads.fill_grad(st, t)
            n, _ = parity.gpu_step(st, lists, t, fused=True)
            norms.append(np.float32(n.item()))
        torch.cuda.synchronize()
        out[mode] = (norms, st.w_flat.clone(), st.m_flat.clone(), st.v_flat.clone())
    fused_env(None)
    if [x.view(np.uint32) for x in out["1"][0]] == [x.view(np.uint32) for x in out["0"][0]]:
        for a, b in zip(out["1"][1:], out["0"][1:]):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    else:
        for a, b in zip(out["1"][0], out["0"][0]):
            assert abs(float(a) - float(b)) <= 1e-6 * abs(float(b))


@pytest.mark.parametrize("mode", ["1", None], ids=["cooperative", "two_launches"])
def test_fused_full_size_loss_scaled_ten_steps(ora, fused_env, mode):
    """The loss-scaled list of 10,012 tensors (a 76 MB binary16 gradient, which the norm keeps in L2) through the
    one-step entry point, each path, over ten steps against the oracle."""
    fused_env(mode)
    r = parity.run_parity(W["fp16_scaled"], ora=ora, check_every_step=False, fused=True)
    assert r["same_factor_every_step"]


def test_fused_launch_on_a_large_list(ora, fused_env):
    """The cooperative launch on a list whose gradient (100 MB of float32) is larger than the norm keeps in L2:
    still correct, the gradient then read from HBM twice."""
    fused_env("1")
    wl = W["gpt2_small"]
    sizes = [25_000_000, 999, 4097]
    r = parity.run_parity(wl, sizes=sizes, ora=ora, steps=2, fused=True, check_every_step=False)
    assert r["same_factor_every_step"]


def test_fused_empty_list():
    norm, factor = mica.mica_clip_adamw_step([], [], [], [], max_norm=1.0, inv_scale=0.25, lr=1e-3, beta1=0.9,
                                             beta2=0.95, eps=1e-8, weight_decay=0.1, step=1)
    torch.cuda.synchronize()
    assert norm.item() == 0.0 and factor.item() == 0.25


def test_grid_wait_selftest(ora, fused_env):
    """The grid-wide wait's failure path: a wait that runs out sets the status word, the next mica_sync reports it
    (once), and a cooperative step right after still matches the oracle bit for bit."""
    fused_env("1")
    mica.mica_selftest_grid_wait_timeout(64)
    with pytest.raises(mica.MicaError, match="grid-wide wait gave up"):
        mica.mica_sync()
    mica.mica_sync()
    r = parity.run_parity(W["tiny"], ora=ora, steps=2, fused=True)
    assert r["same_factor_every_step"]
