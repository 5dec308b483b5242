"""The sharded step on the CPU: the list split over the ranks of a data-parallel job, each rank's square sum, one
exchange (an all-gather of one double per rank over gloo), the factor from the sums in rank order, and each rank's
update of its own part, against the same step of the whole list in one process. The per-rank arithmetic here is the
oracle's (no GPU on this host); the GPU path of the same split is in test_gpu_shard.py."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from clip_tensor_adamw_gb300.shard import OCT, shard_pieces  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("world", [1, 2, 3, 4, 7, 16])
def test_pieces_cover_every_element_once(world):
    rng = np.random.Generator(np.random.PCG64(world))
    for trial in range(20):
        sizes = [int(x) for x in rng.integers(0, 5000, size=int(rng.integers(1, 40)))]
        if trial == 0:
            sizes = [0, 1, 7, 9, 0, 16385]
        seen = [np.zeros(n, np.int32) for n in sizes]
        for r in range(world):
            for k, a, b in shard_pieces(sizes, world, r):
                assert 0 <= a < b <= sizes[k]
                assert a % OCT == 0  # every piece starts at a whole octet of its tensor
                seen[k][a:b] += 1
        assert all((s == 1).all() for s in seen), sizes


def test_pieces_are_balanced():
    sizes = [50257 * 768, 1024 * 768] + [768 * 2304, 2304, 768 * 768, 768] * 12
    total = sum(sizes)
    for world in (2, 4, 8):
        counts = [sum(b - a for _, a, b in shard_pieces(sizes, world, r)) for r in range(world)]
        assert sum(counts) == total
        assert max(counts) - min(counts) <= 2 * OCT * world


def _rank_step(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import oracle
    import workloads
    from clip_tensor_adamw_gb300.shard import shard_pieces
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ora = oracle.Oracle()
        wl = workloads.WORKLOADS["gpt2_small_bf16"]
        sizes = [int(np.prod(s)) for s in workloads._gpt2_shapes(90, 2, 1003, 67)] + [1, 7, 4097]
        st = workloads.make_state(wl, "cpu", sizes=sizes)
        w, _, m, v = workloads.host_lists(st)
        pieces = shard_pieces(sizes, world, rank)
        results = []
        for t in (1, 2, 3):
            workloads.fill_grad(st, t)
            g = workloads.host_lists(st)[1]
            gp = [g[k][a:b] for k, a, b in pieces]
            # this rank's square sum, then the exchange and the rank-ordered sum
            mine = torch.tensor([ora.sum_squares(gp, wl.inv_scale) if gp else 0.0], dtype=torch.float64)
            parts = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
            dist.all_gather(parts, mine)
            S = 0.0
            for p in parts:
                S += float(p.item())
            norm = np.float32(np.sqrt(S))
            factor = ora.clip_factor(norm, wl.max_norm, wl.inv_scale)
            # this rank's update of its own pieces (packed moments: whole words, a piece starts at an even element)
            for k, a, b in pieces:
                wk, gk = w[k][a:b], g[k][a:b].copy()
                mk, vk = m[k][a // 2:(b + 1) // 2], v[k][a // 2:(b + 1) // 2]
                ws, ms, vs = wk.copy(), mk.copy(), vk.copy()
                ora.adamw_steps([ws], [gk], [ms], [vs], oracle.Hyper(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2,
                                                                      eps=wl.eps, weight_decay=wl.weight_decay,
                                                                      step=t), factor=factor)
                wk[:], mk[:], vk[:] = ws, ms, vs
            results.append((float(norm), int(factor.view(np.uint32))))
        out[rank] = (results, pieces, [x.copy() for x in w], [x.copy() for x in m], [x.copy() for x in v])
    finally:
        dist.destroy_process_group()


def test_two_rank_sharded_step_equals_the_whole_list():
    """Both ranks derive the single-process factor's bits, and the two ranks' parts together are the single-process
    step bit for bit, over three steps."""
    import oracle
    import workloads
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank_step, args=(world, port, out), nprocs=world, join=True)
    # the whole list in one process
    ora = oracle.Oracle()
    wl = workloads.WORKLOADS["gpt2_small_bf16"]
    sizes = [int(np.prod(s)) for s in workloads._gpt2_shapes(90, 2, 1003, 67)] + [1, 7, 4097]
    st = workloads.make_state(wl, "cpu", sizes=sizes)
    w, _, m, v = workloads.host_lists(st)
    want = []
    for t in (1, 2, 3):
        workloads.fill_grad(st, t)
        g = workloads.host_lists(st)[1]
        norm, factor = ora.clip_adamw_step(w, g, m, v, oracle.Hyper(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2,
                                                                     eps=wl.eps, weight_decay=wl.weight_decay,
                                                                     step=t), wl.max_norm, wl.inv_scale)
        want.append((float(norm), int(factor.view(np.uint32))))
    assert out[0][0] == out[1][0] == want
    for rank in range(world):
        _, pieces, rw, rm, rv = out[rank]
        for k, a, b in pieces:
            assert np.array_equal(rw[k][a:b].view(np.uint32), w[k][a:b].view(np.uint32))
            assert np.array_equal(rm[k][a // 2:(b + 1) // 2], m[k][a // 2:(b + 1) // 2])
            assert np.array_equal(rv[k][a // 2:(b + 1) // 2], v[k][a // 2:(b + 1) // 2])


def _rank_accumulate(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import oracle
    from clip_tensor_adamw_gb300.shard import shard_pieces
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ora = oracle.Oracle()
        g, a, sizes = _accumulate_inputs()
        pieces = shard_pieces(sizes, world, rank)
        gp = [g[k][x:y].copy() for k, x, y in pieces]
        ap = [a[k][x:y].copy() for k, x, y in pieces]
        ora.accumulate_grads(gp, ap)  # this rank's part of the gradients' last write ...
        mine = torch.tensor([ora.sum_squares(gp, 1.0) if gp else 0.0], dtype=torch.float64)  # ... and its sum
        parts = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(parts, mine)
        S = 0.0
        for p in parts:
            S += float(p.item())
        norm = np.float32(np.sqrt(S))
        factor = ora.clip_factor(norm, 1.0, 1.0)
        out[rank] = (float(norm), int(factor.view(np.uint32)), pieces, gp)
    finally:
        dist.destroy_process_group()


def _accumulate_inputs():
    rng = np.random.Generator(np.random.PCG64(17))
    sizes = [5000, 1, 0, 777, 64, 9, 40000]
    g = [rng.normal(0, 0.05, size=n).astype(np.float32) for n in sizes]
    a = [rng.normal(0, 0.05, size=n).astype(np.float32) for n in sizes]
    return g, a, sizes


def test_two_rank_sharded_accumulate_equals_the_whole_list():
    """The sharded form of the norm fused into the gradients' last write, with the oracle's arithmetic on each rank:
    every rank's part of g + a, the rank-ordered sum of the parts' square sums, and the factor, equal to the
    single-process add and norm of the whole list."""
    import oracle
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank_accumulate, args=(world, port, out), nprocs=world, join=True)
    g, a, sizes = _accumulate_inputs()
    norm, factor = oracle.Oracle().accumulate_clip_grad_norms(g, a, 1.0)
    assert out[0][:2] == out[1][:2] == (float(norm), int(factor.view(np.uint32)))
    for rank in range(world):
        _, _, pieces, gp = out[rank]
        for (k, x, y), part in zip(pieces, gp):
            assert np.array_equal(part.view(np.uint32), g[k][x:y].view(np.uint32))
