"""mica_clip_grad_norms_noalloc, the norm entry point that allocates nothing, against mica_clip_grad_norms.

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
import workloads

pytestmark = pytest.mark.gpu

NORM_RTOL = 1e-5


def _noalloc():
    L = mica.lib()
    fn = L.mica_clip_grad_norms_noalloc
    fn.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int64), ctypes.c_int32, ctypes.c_int32, ctypes.c_float,
                   ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


def _call(fn, grads, max_norm, inv_scale, gdt):
    lst = mica.TensorList(grads)
    norm = torch.full((1,), -1.0, device="cuda")
    factor = torch.full((1,), -1.0, device="cuda")
    status = fn(lst.ptrs, lst.n, lst.T, gdt, max_norm, inv_scale, norm.data_ptr(), factor.data_ptr(),
                torch.cuda.current_stream().cuda_stream)
    assert status == 0, mica.lib().mica_last_error_detail().decode()
    return norm, factor


@pytest.mark.parametrize("name", ["gpt2_small_bf16", "fp16_scaled"])
def test_noalloc_matches_allocating_entry_point(name):
    fn = _noalloc()
    wl = workloads.WORKLOADS[name]
    sizes = list(wl.sizes[:300]) if name == "fp16_scaled" else [int(np.prod(s)) for s in
                                                                 workloads._gpt2_shapes(90, 2, 1003, 67)]
    st = workloads.make_state(wl, "cuda", sizes=sizes + [1, 7, 4097])
    gdt = 1 if wl.grad_dtype == "f16" else 0
    for t in (1, 2):  # two calls in a row, on different gradients
        workloads.fill_grad(st, t)
        n_ref, f_ref = mica.mica_clip_grad_norms(st.g, wl.max_norm, wl.inv_scale)
        n_na, f_na = _call(fn, st.g, wl.max_norm, wl.inv_scale, gdt)
        torch.cuda.synchronize()
        a, b = n_na.item(), n_ref.item()
        assert abs(a - b) <= NORM_RTOL * abs(b), (t, a, b)
        fa, fb = f_na.item(), f_ref.item()
        assert abs(fa - fb) <= NORM_RTOL * abs(fb), (t, fa, fb)


def test_noalloc_rejects_lists_beyond_its_scratch():
    fn = _noalloc()
    g = torch.zeros(8, device="cuda")
    T = 16385
    ptrs = (ctypes.c_void_p * T)(*([g.data_ptr()] * T))
    n = (ctypes.c_int64 * T)(*([1] * T))
    f = torch.zeros(1, device="cuda")
    status = fn(ptrs, n, T, 0, 1.0, 1.0, None, f.data_ptr(), None)
    assert status == 2  # MICA_ERR_COUNT
    assert "16384" in mica.lib().mica_last_error_detail().decode()
