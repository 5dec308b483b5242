"""One tensor of more than 2^31 elements (2^31 + 13) between two small ones, through the C ABI, against the oracle.

Element indices past 2^31, byte offsets past 2^32, a work item per 512 octets of it (over half a million), and a
ragged last octet of 5 elements. The norm is checked against the oracle's norm of the whole gradient; the update
(AdamW with float32 or loss-scaled binary16 gradients, SGD with momentum) on sampled elements: every element of the
small tensors, and of the large one a random sample plus the elements around 2^29, 2^30 and 2^31 and its end.
The update is elementwise, so the oracle steps the sampled elements as one list of their own, with its own factor.
Each case holds about 35 GB on the device and copies the gradient (up to 8.6 GB) to the host once per step."""
import numpy as np
import pytest
import torch

import clip_tensor_adamw_gb300 as mica
import oracle
import parity
import workloads

pytestmark = pytest.mark.gpu

BIG = 2 ** 31 + 13
SIZES = [1000, BIG, 37]


@pytest.fixture(scope="module")
def ora():
    return oracle.Oracle()


def _picks(sizes, rng):
    """Per tensor, the sorted element indices the update is checked on."""
    out = []
    for n in sizes:
        if n <= 4096:
            out.append(np.arange(n, dtype=np.int64))
            continue
        edges = [np.arange(0, 64)]
        for b in (2 ** 29, 2 ** 30, 2 ** 31):
            if b < n:
                edges.append(np.arange(b - 64, min(b + 64, n)))
        edges.append(np.arange(n - 64, n))
        sel = np.concatenate([rng.integers(0, n, size=100_000)] + edges)
        out.append(np.unique(sel))
    return out


def _gather(tensors, picks):
    return np.concatenate([t[torch.from_numpy(sel).to(t.device)].cpu().numpy() for t, sel in zip(tensors, picks)])


def _host_grads(st):
    """The whole gradient on the host, one numpy view per tensor (one copy of the flat buffer)."""
    flat = st.g_flat.cpu().numpy()
    es = flat.dtype.itemsize
    return [flat[(x.data_ptr() - st.g_flat.data_ptr()) // es:][:x.numel()] for x in st.g]


@pytest.mark.parametrize("name,opt", [("gpt2_small", "adamw"), ("fp16_scaled", "adamw"),
                                      ("gpt2_small", "sgd_momentum")])
def test_one_tensor_past_2e31_elements(ora, name, opt):
    wl = workloads.WORKLOADS[name]
    st = workloads.make_state(wl, "cuda", sizes=SIZES)
    try:
        W, G, M, V = parity.tensor_lists(st)
        picks = _picks(st.sizes, np.random.Generator(np.random.PCG64(2024)))
        w_s, m_s, v_s = _gather(st.w, picks), _gather(st.m, picks), _gather(st.v, picks)
        for t in (1, 2):
            zero_grad = t == 2
            workloads.fill_grad(st, t)
            hg = _host_grads(st)
            o_norm, o_factor, _ = ora.clip_grad_norms(hg, wl.max_norm, wl.inv_scale)
            del hg
            g_s = _gather(st.g, picks)
            if opt == "adamw":
                ora.adamw_steps([w_s], [g_s], [m_s], [v_s], parity.hp_of(wl, t), factor=o_factor)
            else:
                ora.sgd_steps([w_s], [g_s], [m_s], parity.SGD_LR, 0.9, factor=o_factor)
            d_norm, d_factor = mica.mica_clip_grad_norms(G, wl.max_norm, wl.inv_scale)
            if opt == "adamw":
                mica.mica_adamw_steps(W, G, M, V, lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps,
                                      weight_decay=wl.weight_decay, step=t, zero_grad=zero_grad, factor=d_factor)
            else:
                mica.mica_sgd_steps(W, G, M, lr=parity.SGD_LR, momentum=0.9, zero_grad=zero_grad, factor=d_factor)
            torch.cuda.synchronize()
            parity.check_norm(np.float32(d_norm.item()), o_norm, t)
            assert float(o_norm) > wl.max_norm or name == "fp16_scaled"  # the clip fires on the float32 list
            same = np.float32(d_factor.item()).view(np.uint32) == o_factor.view(np.uint32)
            tag = f"{name} {opt} 2^31+13 step {t}"
            gw, gm = _gather(st.w, picks), _gather(st.m, picks)
            parity.f32_close(gw, w_s, f"{tag} w")
            parity.f32_close(gm, m_s, f"{tag} m")
            if opt == "adamw":
                gv = _gather(st.v, picks)
                parity.f32_close(gv, v_s, f"{tag} v")
            if same:
                parity.exact(gw, w_s, f"{tag} w bits")
                parity.exact(gm, m_s, f"{tag} m bits")
                if opt == "adamw":
                    parity.exact(gv, v_s, f"{tag} v bits")
            gg = _gather(st.g, picks)
            if zero_grad:
                assert not gg.any(), f"{tag}: gradient not zeroed"
            else:
                parity.exact(gg, g_s, f"{tag} g untouched")
    finally:
        del st
        torch.cuda.empty_cache()
