"""The sharded step's GPU entry points (mica_grad_sumsq, mica_clip_factor_from_sumsq) on one GPU: the list split as
a data-parallel job of N ranks would split it, each part's square sum on the device, the factor from the sums in
rank order, and each part's update, against the oracle's step of the whole list. The ranks run one after another
in this one process (no rank waits on another); the exchange between real ranks is the caller's all-gather."""
import numpy as np
import pytest
import torch

import clip_tensor_adamw_gb300 as mica
import oracle
import parity
import workloads
from clip_tensor_adamw_gb300.shard import piece_views, shard_pieces

pytestmark = pytest.mark.gpu

W = workloads.WORKLOADS


def small_gpt2_sizes(d=90, layers=2, vocab=1003, ctx=67):
    return [int(np.prod(s)) for s in workloads._gpt2_shapes(d, layers, vocab, ctx)]


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("name", ["gpt2_small", "gpt2_small_bf16", "fp16_scaled"])
def test_sharded_step_matches_the_oracle(name, world):
    wl = W[name]
    sizes = small_gpt2_sizes() + [1, 7, 4097] if name != "fp16_scaled" else list(wl.sizes[:500]) + [768 * 3072]
    ora = oracle.Oracle()
    st = workloads.make_state(wl, "cuda", sizes=sizes)
    host = workloads.host_lists(st)
    ranks = []
    for r in range(world):
        pieces = shard_pieces(sizes, world, r)
        ranks.append(dict(W=mica.TensorList(piece_views(st.w, pieces)), G=mica.TensorList(piece_views(st.g, pieces)),
                          M=mica.TensorList(piece_views(st.m, pieces, st.m_packed), [b - a for _, a, b in pieces]),
                          V=mica.TensorList(piece_views(st.v, pieces, st.packed), [b - a for _, a, b in pieces])))
    parts = torch.zeros(world, dtype=torch.float64, device="cuda")
    for t in (1, 2, 3):
        workloads.fill_grad(st, t)
        host = (host[0], [x.detach().cpu().numpy().copy() for x in st.g], host[2], host[3])
        for r, lists in enumerate(ranks):
            mica.mica_grad_sumsq(lists["G"], wl.inv_scale, out=parts[r:r + 1])
        d_norm, d_factor = mica.mica_clip_factor_from_sumsq(parts, wl.max_norm, wl.inv_scale)
        for lists in ranks:
            mica.mica_adamw_steps(lists["W"], lists["G"], lists["M"], lists["V"], lr=wl.lr, beta1=wl.beta1,
                                  beta2=wl.beta2, eps=wl.eps, weight_decay=wl.weight_decay, step=t, factor=d_factor)
        o_norm, o_factor = ora.clip_adamw_step(*host, parity.hp_of(wl, t), wl.max_norm, wl.inv_scale)
        torch.cuda.synchronize()
        parity.check_norm(np.float32(d_norm.item()), o_norm, t)
        # each rank's sum is that of its part, exactly as the norm sums it
        o_parts = [ora.sum_squares([host[1][k][a:b] for k, a, b in shard_pieces(sizes, world, r)] or
                                   [np.zeros(0, host[1][0].dtype)], wl.inv_scale) for r in range(world)]
        np.testing.assert_allclose(parts.cpu().numpy(), o_parts, rtol=1e-12)
        same = np.float32(d_factor.item()).view(np.uint32) == o_factor.view(np.uint32)
        parity.compare_state(st, host, bool(same), f"{name} sharded x{world} step {t}")
    mica.mica_sync()


def test_factor_from_sumsq_rank_order_and_validation():
    """The factor from given sums: S added in index order, then PyTorch's clip rounding; bad arguments refused."""
    parts = torch.tensor([9.0, 16.0], dtype=torch.float64, device="cuda")  # S = 25: norm 5
    norm, factor = mica.mica_clip_factor_from_sumsq(parts, 1.0, 0.5)
    torch.cuda.synchronize()
    assert norm.item() == 5.0
    ora = oracle.Oracle()
    assert np.float32(factor.item()) == ora.clip_factor(np.float32(5.0), 1.0, 0.5)
    L = mica.lib()
    for count in (0, -1, (1 << 16) + 1):  # COUNT
        assert L.mica_clip_factor_from_sumsq(parts.data_ptr(), count, 1.0, 1.0, None, factor.data_ptr(), None) == 2
    assert L.mica_clip_factor_from_sumsq(None, 2, 1.0, 1.0, None, factor.data_ptr(), None) == 1  # NULL
    with pytest.raises(mica.MicaError, match="HYPER"):
        mica.mica_clip_factor_from_sumsq(parts, 0.0, 1.0)


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("name", ["gpt2_small", "fp16_scaled"])
def test_sharded_accumulate_matches_the_whole_list(ora, name, world):
    """The sharded form of the norm fused into the gradient's last write: each rank's g += a with its part's square
    sum (mica_accumulate_grad_sumsq), the factor from the sums in rank order, against the oracle's add and norm of
    the whole list; every added element bit-exact, each rank's sum that of its part."""
    wl = W[name]
    sizes = small_gpt2_sizes() + [1, 7, 4097] if name != "fp16_scaled" else list(wl.sizes[:500]) + [768 * 3072]
    st = workloads.make_state(wl, "cuda", sizes=sizes)
    add = workloads.make_state(wl, "cuda", sizes=sizes)
    workloads.fill_grad(st, 1)
    workloads.fill_grad(add, 1, seed=91)
    g_host = [x.detach().cpu().numpy().copy() for x in st.g]
    a_host = [x.detach().cpu().numpy().copy() for x in add.g]
    parts = torch.zeros(world, dtype=torch.float64, device="cuda")
    for r in range(world):
        pieces = shard_pieces(sizes, world, r)
        mica.mica_accumulate_grad_sumsq(piece_views(st.g, pieces), piece_views(add.g, pieces), wl.inv_scale,
                                        out=parts[r:r + 1])
    d_norm, d_factor = mica.mica_clip_factor_from_sumsq(parts, wl.max_norm, wl.inv_scale)
    o_norm, o_factor = ora.accumulate_clip_grad_norms(g_host, a_host, wl.max_norm, wl.inv_scale)
    torch.cuda.synchronize()
    for k, x in enumerate(st.g):
        parity.exact(x.detach().cpu().numpy(), g_host[k], f"g[{k}]")
    parity.check_norm(np.float32(d_norm.item()), o_norm, 0)
    assert np.float32(d_factor.item()).view(np.uint32) == o_factor.view(np.uint32)
    o_parts = [ora.sum_squares([g_host[k][a:b] for k, a, b in shard_pieces(sizes, world, r)] or
                               [np.zeros(0, g_host[0].dtype)], wl.inv_scale) for r in range(world)]
    np.testing.assert_allclose(parts.cpu().numpy(), o_parts, rtol=1e-12)
