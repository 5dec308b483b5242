"""The seeded synthetic inputs: the five workloads' shapes and parameter counts, their shared hyperparameters, the
bucket layout of their buffers, and the determinism of their draws (CPU only)."""
import numpy as np
import pytest
import torch

import workloads

W = workloads.WORKLOADS


def test_parameter_counts_and_tensor_counts():
    assert (len(W["tiny"].sizes), W["tiny"].params) == (4, 739_200)
    assert (len(W["gpt2_small"].sizes), W["gpt2_small"].params) == (148, 124_439_808)
    assert W["gpt2_small_bf16"].shapes == W["gpt2_small"].shapes
    assert (len(W["gpt2_xl"].sizes), W["gpt2_xl"].params) == (580, 1_557_611_200)
    c4 = W["fp16_scaled"]
    assert (len(c4.sizes), c4.params) == (10_012, 37_981_154)
    assert c4.shapes[-12:] == ((768, 3072),) * 12
    small = np.array(c4.sizes[:10_000])
    assert small.min() >= 64 and small.max() < 4096


def test_gpt2_small_shapes():
    s = W["gpt2_small"].shapes
    assert s[0] == (50257, 768) and s[1] == (1024, 768) and s[-2:] == ((768,), (768,))
    block = s[2:14]
    assert block == ((768,), (768,), (768, 2304), (2304,), (768, 768), (768,), (768,), (768,), (768, 3072), (3072,),
                     (3072, 768), (768,))
    assert all(s[2 + 12 * k:14 + 12 * k] == block for k in range(12))


def test_dtypes_and_hyperparameters():
    kinds = {n: (w.grad_dtype, w.moments) for n, w in W.items()}
    assert kinds == {"tiny": ("f32", "f32"), "gpt2_small": ("f32", "f32"), "gpt2_small_bf16": ("f32", "bf16x2"),
                     "fp16_scaled": ("f16", "f32"), "gpt2_xl": ("f32", "bf16x2")}
    for w in W.values():
        assert (w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.max_norm, w.steps, w.seed) == \
            (6e-4, 0.9, 0.95, 1e-8, 0.1, 1.0, 10, 0)
    assert W["fp16_scaled"].inv_scale == 2.0 ** -16
    assert W["gpt2_small_bf16"].spike_p == 0.01 and W["gpt2_small_bf16"].spike_mult == 100.0


@pytest.mark.parametrize("name", ["tiny", "gpt2_small_bf16", "fp16_scaled"])
def test_bucket_layout(name):
    """Each tensor a view into one flat buffer per stream, at a 256-byte-aligned offset; m and v zero; packed
    moments hold ceil(n/2) words."""
    wl = W[name]
    sizes = wl.sizes if name == "tiny" else [1, 7, 9, 4097, 33, 0, 3]
    st = workloads.make_state(wl, "cpu", sizes=sizes)
    for views, flat in ((st.w, st.w_flat), (st.g, st.g_flat), (st.m, st.m_flat), (st.v, st.v_flat)):
        for x in views:
            if x.numel():  # an empty view has no address of its own
                assert (x.data_ptr() - flat.data_ptr()) % workloads.ALIGN_BYTES == 0
    for n, m, v in zip(sizes, st.m, st.v):
        assert m.numel() == ((n + 1) // 2 if st.m_packed else n)
        assert v.numel() == ((n + 1) // 2 if st.packed else n)
    assert not st.m_flat.any() and not st.v_flat.any() and not st.g_flat.any()


def test_draws_are_seeded():
    wl = W["tiny"]
    a, b = workloads.make_state(wl, "cpu"), workloads.make_state(wl, "cpu")
    assert torch.equal(a.w_flat, b.w_flat)
    workloads.fill_grad(a, 3)
    workloads.fill_grad(b, 3)
    assert torch.equal(a.g_flat, b.g_flat)
    g3 = a.g_flat.clone()
    workloads.fill_grad(a, 4)
    assert not torch.equal(a.g_flat, g3)
    assert abs(float(a.w_flat[:a.sizes[0]].std()) - wl.w_std) < 0.1 * wl.w_std


def test_loss_scaled_gradient_is_binary16():
    wl = W["fp16_scaled"]
    st = workloads.make_state(wl, "cpu", sizes=[100_000])
    workloads.fill_grad(st, 1)
    g = st.g_flat[:100_000].float()
    assert st.g_flat.dtype == torch.float16
    assert abs(float(g.std()) - wl.g_std * wl.loss_scale) < 0.05 * wl.g_std * wl.loss_scale
