"""Seeded random configurations of the whole step against the oracle, element by element: random tensor lists
(empty, tiny, ragged, large, misaligned), gradient and moment types, zero_grad, the Adam family's options and
parameter groups, and the SGD steps. Each configuration runs three steps from its own seed and must match the oracle
bit for bit wherever the two sides' clip factors agree (they agree unless the norm sits on a float32 rounding
boundary)."""
import dataclasses

import numpy as np
import pytest
import torch

import clip_tensor_adamw_gb300 as mica
import oracle
import parity
import workloads

pytestmark = pytest.mark.gpu

N_CASES = 64


def _config(i: int):
    rng = np.random.Generator(np.random.PCG64(1000 + i))
    T = int(rng.integers(1, 60))
    kind = rng.choice(["tiny", "mixed", "large"])
    if kind == "tiny":
        sizes = rng.integers(0, 40, size=T)
    elif kind == "mixed":
        sizes = np.exp(rng.uniform(0, np.log(20000), size=T)).astype(int)
    else:
        sizes = rng.integers(1, 300000, size=min(T, 6))
    sizes = [int(x) for x in sizes]
    grad = rng.choice(["f32", "f16"])
    moments = rng.choice(["f32", "bf16x2", "bf16x2_m"])
    opt = rng.choice(["adamw", "adam_l2", "groups", "sgd", "momentum"], p=[0.3, 0.15, 0.25, 0.15, 0.15])
    if opt in ("sgd", "momentum"):
        moments = "f32"
    wl = dataclasses.replace(
        workloads.WORKLOADS["fp16_scaled" if grad == "f16" else "gpt2_small"], name=f"fuzz{i}", moments=str(moments),
        g_std=float(rng.choice([1e-4, 1e-2, 1.0])), spike_p=0.0 if grad == "f16" else float(rng.choice([0.0, 0.01])),
        spike_mult=100.0, max_norm=float(rng.choice([0.1, 1.0, 1e9])), seed=int(rng.integers(0, 1 << 30)))
    return dict(wl=wl, sizes=sizes, opt=str(opt), zero_grad=bool(rng.integers(0, 2)),
                skip=bool(rng.integers(0, 2)), ngroups=int(rng.integers(1, 9)), seed=int(rng.integers(0, 1 << 30)))


@pytest.fixture(scope="module")
def ora():
    return oracle.Oracle()


@pytest.mark.parametrize("i", range(N_CASES))
def test_fuzz(ora, i):
    c = _config(i)
    wl, sizes, opt = c["wl"], c["sizes"], c["opt"]
    if opt in ("sgd", "momentum"):
        r = parity.run_parity_sgd(wl, 0.9 if opt == "momentum" else 0.0, sizes=sizes, steps=3, ora=ora,
                                  zero_grad=c["zero_grad"], skip_nonfinite=c["skip"])
    elif opt == "groups":
        group = [int(k) % c["ngroups"] for k in np.random.Generator(np.random.PCG64(c["seed"])).permutation(len(sizes))]
        hps = [dict(lr=wl.lr * (j + 1) / c["ngroups"], weight_decay=0.05 * j) for j in range(c["ngroups"])]
        orig = parity.group_hps
        parity.group_hps = lambda _wl: hps
        try:
            r = parity.run_parity_groups(wl, group, sizes=sizes, steps=3, ora=ora, zero_grad=c["zero_grad"])
        finally:
            parity.group_hps = orig
    else:
        r = parity.run_parity(wl, sizes=sizes, steps=3, ora=ora, zero_grad=c["zero_grad"],
                              coupled_l2=(opt == "adam_l2"), skip_nonfinite=c["skip"])
    assert r["same_factor_every_step"]
