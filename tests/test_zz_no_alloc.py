"""mica_clip_grad_norms_noalloc, the norm entry point that allocates nothing, against mica_clip_grad_norms and the
oracle.

Callers that cannot let a library allocate device memory (a runtime that has reserved its whole budget, memory
held by another allocator, a loop that cannot afford cudaMalloc's synchronisation) use this entry point; it keeps its
scratch in a fixed-size device array of the library. This file is collected last so that a run stopping at the
first failure has already run every other test; it passes alone and after the others.
"""
import ctypes

import numpy as np
import pytest
import torch

import clip_tensor_adamw_gb300 as mica
import oracle
import workloads

pytestmark = pytest.mark.gpu

NORM_RTOL = 1e-5
OK, COUNT, ADDRESS, CAPTURE = 0, 2, 8, 11


def _noalloc():
    L = mica.lib()
    fn = L.mica_clip_grad_norms_noalloc
    fn.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int64), ctypes.c_int32, ctypes.c_int32, ctypes.c_float,
                   ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


def _detail():
    return mica.lib().mica_last_error_detail().decode()


def _call(fn, grads, max_norm, inv_scale, gdt, stream=None):
    lst = mica.TensorList(grads)
    norm = torch.full((1,), -1.0, device="cuda")
    factor = torch.full((1,), -1.0, device="cuda")
    st = torch.cuda.current_stream().cuda_stream if stream is None else stream
    status = fn(lst.ptrs, lst.n, lst.T, gdt, max_norm, inv_scale, norm.data_ptr(), factor.data_ptr(), st)
    assert status == OK, _detail()
    return norm, factor


def _bits(x: torch.Tensor) -> int:
    return int(np.float32(x.item()).view(np.uint32))


def _lists():
    """A loss-scaled list of small tensors (the register-streaming kernel) and a GPT-2-like list (the TMA one),
    each with a ragged tail."""
    fp16 = workloads.WORKLOADS["fp16_scaled"]
    gpt = workloads.WORKLOADS["gpt2_small_bf16"]
    gpt_sizes = [int(np.prod(s)) for s in workloads._gpt2_shapes(90, 2, 1003, 67)]
    return [(fp16, list(fp16.sizes[:300]) + [1, 7, 4097]), (gpt, gpt_sizes + [1, 7, 4097])]


@pytest.mark.parametrize("case", [0, 1], ids=["small_tensors", "gpt2_like"])
def test_noalloc_matches_allocating_entry_point_and_oracle(case):
    """Two calls in a row on different gradients: the same norm and factor bits as the allocating entry point (the
    list is small enough that both take the same work split), and the oracle's norm and factor."""
    fn = _noalloc()
    ora = oracle.Oracle()
    wl, sizes = _lists()[case]
    st = workloads.make_state(wl, "cuda", sizes=sizes)
    gdt = 1 if wl.grad_dtype == "f16" else 0
    for t in (1, 2):
        workloads.fill_grad(st, t)
        n_ref, f_ref = mica.mica_clip_grad_norms(st.g, wl.max_norm, wl.inv_scale)
        n_na, f_na = _call(fn, st.g, wl.max_norm, wl.inv_scale, gdt)
        torch.cuda.synchronize()
        assert _bits(n_na) == _bits(n_ref) and _bits(f_na) == _bits(f_ref), (t, n_na.item(), n_ref.item())
        o_norm, o_factor, _ = ora.clip_grad_norms(workloads.host_lists(st)[1], wl.max_norm, wl.inv_scale)
        assert abs(n_na.item() - float(o_norm)) <= NORM_RTOL * float(o_norm), (t, n_na.item(), o_norm)
        if _bits(n_na) == int(o_norm.view(np.uint32)):  # the same norm gives the same factor, bit for bit
            assert _bits(f_na) == int(o_factor.view(np.uint32)), (t, f_na.item(), o_factor)
        else:
            assert abs(f_na.item() - float(o_factor)) <= NORM_RTOL * float(o_factor)


def test_noalloc_large_list_beyond_the_allocating_split():
    """A list of 600 M float32 elements: more work units than the scratch has room for at the allocating entry
    point's split, so this entry point splits it coarser. The norm still agrees with the allocating entry point and
    the oracle to 1e-5."""
    fn = _noalloc()
    ora = oracle.Oracle()
    sizes = [250_000_000, 199_999_993, 150_000_007]
    gen = torch.Generator(device="cuda")
    gen.manual_seed(11)
    grads = [torch.randn(n, device="cuda", generator=gen) * 1e-3 for n in sizes]
    n_ref, f_ref = mica.mica_clip_grad_norms(grads, 1.0, 1.0)
    n_na, f_na = _call(fn, grads, 1.0, 1.0, 0)
    torch.cuda.synchronize()
    o_norm, o_factor, _ = ora.clip_grad_norms([g.cpu().numpy() for g in grads], 1.0, 1.0)
    for got in (n_na.item(), n_ref.item()):
        assert abs(got - float(o_norm)) <= NORM_RTOL * float(o_norm), (got, o_norm)
    assert abs(f_na.item() - float(o_factor)) <= NORM_RTOL * float(o_factor)
    del grads
    mica.mica_release_cache()
    torch.cuda.empty_cache()


def test_noalloc_tensor_limit_and_empty_lists():
    fn = _noalloc()
    f = torch.zeros(1, device="cuda")
    nrm = torch.zeros(1, device="cuda")
    g = torch.ones(8, device="cuda")
    # 16,384 tensors is the limit: accepted; 16,385: refused with a detail naming the limit
    for T, want in ((16384, OK), (16385, COUNT)):
        ptrs = (ctypes.c_void_p * T)(*([g.data_ptr()] * T))
        n = (ctypes.c_int64 * T)(*([8] * T))
        status = fn(ptrs, n, T, 0, 1e9, 1.0, nrm.data_ptr(), f.data_ptr(), None)
        assert status == want, (T, status, _detail())
        if want == COUNT:
            assert "16384" in _detail()
    torch.cuda.synchronize()
    assert nrm.item() == pytest.approx(float(np.sqrt(16384 * 8)), rel=1e-6)
    # tensors that are all empty: norm 0 and factor exactly inv_scale (as for an empty list)
    T = 5
    ptrs = (ctypes.c_void_p * T)(*([None] * T))
    n = (ctypes.c_int64 * T)(*([0] * T))
    assert fn(ptrs, n, T, 0, 1.0, 0.25, nrm.data_ptr(), f.data_ptr(), None) == OK, _detail()
    torch.cuda.synchronize()
    assert nrm.item() == 0.0 and f.item() == 0.25


def test_noalloc_rejects_a_gradient_past_its_allocation():
    """An element count that runs past the end of the gradient's allocation is refused on the host."""
    fn = _noalloc()
    g = torch.zeros(1000, device="cuda")
    f = torch.zeros(1, device="cuda")
    ptrs = (ctypes.c_void_p * 1)(g.data_ptr())
    n = (ctypes.c_int64 * 1)(1 << 33)  # 32 GB of float32: past any allocation that holds 1000 elements
    assert fn(ptrs, n, 1, 0, 1.0, 1.0, None, f.data_ptr(), None) == ADDRESS
    assert "past the end" in _detail()


def test_noalloc_refuses_a_capturing_stream():
    """A stream that is capturing a CUDA graph is refused before anything is queued, and the capture stays valid
    (the graph holds the caller's own work and replays it)."""
    fn = _noalloc()
    g = torch.randn(4096, device="cuda")
    lst = mica.TensorList([g])
    f = torch.zeros(1, device="cuda")
    x = torch.zeros(4, device="cuda")
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        status = fn(lst.ptrs, lst.n, lst.T, 0, 1.0, 1.0, None, f.data_ptr(), torch.cuda.current_stream().cuda_stream)
        x.add_(1.0)
    assert status == CAPTURE, _detail()
    assert "capturing" in _detail()
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(x, torch.full((4,), 2.0, device="cuda"))  # captured work runs only when replayed: twice
    assert f.item() == 0.0  # the refused call queued nothing


def test_noalloc_after_release_cache():
    """mica_release_cache() also drops the scratch's cached device address; the next call looks it up again and
    gives the same bits."""
    fn = _noalloc()
    wl, sizes = _lists()[0]
    st = workloads.make_state(wl, "cuda", sizes=sizes)
    workloads.fill_grad(st, 3)
    a = _call(fn, st.g, wl.max_norm, wl.inv_scale, 1)
    mica.mica_release_cache()
    b = _call(fn, st.g, wl.max_norm, wl.inv_scale, 1)
    torch.cuda.synchronize()
    assert _bits(a[0]) == _bits(b[0]) and _bits(a[1]) == _bits(b[1])


@pytest.mark.parametrize("values,at", [([float("inf")], [64]), ([1e30, -3e25], [64, 130])], ids=["inf", "two_huge"])
def test_noalloc_norm_over_many_staged_spans(ora, values, at):
    """The list of 4,096 tensors whose register-norm chunks span four staged runs of 256 tensors each, a value that
    the float32 pairs cannot hold planted in a later span (see test_gpu_norm_spans.py): the same norm as the oracle
    and the same bits as the allocating entry point."""
    from test_gpu_norm_spans import spanning_list
    host, dev, _ = spanning_list(values, at)
    o_norm, o_factor, _ = ora.clip_grad_norms(host, 1.0)
    norm, factor = _call(_noalloc(), dev, 1.0, 1.0, 0)
    a_norm, a_factor = mica.mica_clip_grad_norms(dev, 1.0, 1.0)
    torch.cuda.synchronize()
    assert _bits(norm) == _bits(a_norm) and _bits(factor) == _bits(a_factor)
    if np.isinf(o_norm):
        assert np.isinf(norm.item()) and factor.item() == 0.0
    else:
        assert abs(norm.item() - float(o_norm)) <= NORM_RTOL * float(o_norm)
        assert np.float32(factor.item()).view(np.uint32) == o_factor.view(np.uint32)
