"""The C ABI without a GPU: the library loads, exports every entry point its header declares, and rejects bad
arguments on the host, before anything reaches a device, with the documented status codes."""
import ctypes
import glob
import math
import os
import re

import pytest

import clip_tensor_adamw_gb300 as mica
from clip_tensor_adamw_gb300.mica import _HP, _SgdHP

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, NULL, COUNT, DTYPE, HYPER, BETA, OVERLAP, DEVICE, ADDRESS, CUDA, NOMEM = range(11)


def declared_symbols():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names += re.findall(r"MICA_API\s+[\w\s\*]+?\b(mica_\w+)\s*\(", text)
    return sorted(set(names))


def test_exports_every_declared_symbol():
    L = mica.lib()
    names = declared_symbols()
    assert len(names) >= 9
    for name in names:
        assert hasattr(L, name), name
    assert L.mica_abi_version() == 5


def test_status_strings():
    L = mica.lib()
    for code, name in enumerate(mica.mica.STATUS):
        assert L.mica_status_string(code).decode() == name


def _arr(ctype, vals):
    return (ctype * max(1, len(vals)))(*vals)


def _hp(**kw):
    d = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, step=1, zero_grad=0, flags=0)
    d.update(kw)
    return _HP(**d)


def adamw(T=1, n=(4,), ptrs=0x1000, gdt=0, mdt=0, hp=None, null_arrays=False):
    L = mica.lib()
    P = _arr(ctypes.c_void_p, [ptrs] * T)
    N = _arr(ctypes.c_int64, list(n)[:T])
    arrays = [None] * 4 if null_arrays else [P, P, P, P]
    hp_ref = ctypes.byref(hp) if hp is not None else None
    return L.mica_adamw_steps(*arrays, N, T, gdt, mdt, hp_ref, None, None)


def test_adamw_host_validation():
    assert adamw(hp=None) == NULL
    assert adamw(hp=_hp(), gdt=2) == DTYPE
    assert adamw(hp=_hp(), mdt=1) == DTYPE
    assert adamw(hp=_hp(), mdt=4) == DTYPE
    for bad in (dict(lr=math.nan), dict(lr=-1.0), dict(lr=math.inf), dict(eps=-1e-8), dict(eps=math.inf),
                dict(weight_decay=-0.1), dict(step=0), dict(step=-3), dict(flags=4), dict(flags=0x80000000)):
        assert adamw(hp=_hp(**bad)) == HYPER, bad
    for bad in (dict(beta1=1.0), dict(beta1=-0.1), dict(beta2=math.nan), dict(beta2=1.5)):
        assert adamw(hp=_hp(**bad)) == BETA, bad
    assert adamw(T=-1, hp=_hp()) == COUNT
    assert adamw(T=1, n=(-5,), hp=_hp()) == COUNT
    assert adamw(T=1, hp=_hp(), null_arrays=True) == NULL
    assert adamw(T=1, ptrs=0, hp=_hp()) == NULL            # a NULL tensor with n > 0
    assert adamw(T=1, n=(0,), ptrs=0, hp=_hp()) == OK       # empty tensors may be NULL: nothing to do
    assert adamw(T=0, hp=_hp()) == OK


def grouped(T=2, n=(4, 4), ptrs=0x1000, group=(0, 1), hps=None, num_groups=None, null_group=False):
    L = mica.lib()
    P = _arr(ctypes.c_void_p, [ptrs] * T)
    N = _arr(ctypes.c_int64, list(n)[:T])
    hps = [_hp(), _hp(lr=5e-4, weight_decay=0.0)] if hps is None else hps
    H = (_HP * len(hps))(*hps)
    G = None if null_group else _arr(ctypes.c_int32, list(group)[:T])
    ng = len(hps) if num_groups is None else num_groups
    return L.mica_adamw_steps_grouped(P, P, P, P, N, T, 0, 0, G, H, ng, None, None)


def test_grouped_host_validation():
    assert grouped(num_groups=0) == COUNT
    assert grouped(num_groups=9) == COUNT
    assert grouped(null_group=True) == NULL
    assert grouped(group=(0, 2)) == COUNT                   # index past num_groups
    assert grouped(group=(-1, 0)) == COUNT
    for field, val, want in (("beta1", 0.8, HYPER), ("beta2", 0.9, HYPER), ("eps", 1e-6, HYPER), ("step", 2, HYPER),
                             ("zero_grad", 1, HYPER), ("flags", 1, HYPER), ("lr", -1.0, HYPER),
                             ("weight_decay", math.nan, HYPER), ("beta1", 1.0, BETA)):
        assert grouped(hps=[_hp(), _hp(**{field: val})]) == want, field
    assert grouped(T=0) == OK
    assert grouped(n=(0, 0), ptrs=0) == OK


def sgd(T=1, n=(4,), ptrs=0x1000, gdt=0, hp=None, with_buf=True, null_arrays=False):
    L = mica.lib()
    P = _arr(ctypes.c_void_p, [ptrs] * T)
    N = _arr(ctypes.c_int64, list(n)[:T])
    hp_ref = ctypes.byref(hp) if hp is not None else None
    arrays = [None, None] if null_arrays else [P, P]
    return L.mica_sgd_steps(*arrays, P if with_buf else None, N, T, gdt, hp_ref, None, None)


def _sgd_hp(**kw):
    d = dict(lr=0.1, momentum=0.9, zero_grad=0, flags=0)
    d.update(kw)
    return _SgdHP(**d)


def test_sgd_host_validation():
    assert sgd(hp=None) == NULL
    assert sgd(hp=_sgd_hp(), gdt=2) == DTYPE
    for bad in (dict(lr=math.nan), dict(lr=-0.1), dict(momentum=-0.5), dict(momentum=math.inf), dict(flags=2),
                dict(flags=4)):
        assert sgd(hp=_sgd_hp(**bad)) == HYPER, bad
    assert sgd(hp=_sgd_hp(momentum=0.9), with_buf=False) == NULL   # momentum needs its buffers
    assert sgd(T=-1, hp=_sgd_hp()) == COUNT
    assert sgd(hp=_sgd_hp(), null_arrays=True) == NULL
    assert sgd(ptrs=0, hp=_sgd_hp()) == NULL
    assert sgd(T=0, hp=_sgd_hp()) == OK
    assert sgd(n=(0,), ptrs=0, hp=_sgd_hp(momentum=0.0), with_buf=False) == OK


def test_adamw_needs_device_memory():
    """A well-formed call with pointers that are not device memory never launches: without a GPU it reports no
    device, with one it reports the address."""
    import torch
    status = adamw(hp=_hp())
    assert status == (ADDRESS if torch.cuda.is_available() else DEVICE)
    assert mica.lib().mica_last_error_detail().decode()


def test_clip_host_validation():
    L = mica.lib()
    G = _arr(ctypes.c_void_p, [0x1000])
    N = _arr(ctypes.c_int64, [4])
    f = ctypes.c_void_p(0x2000)
    assert L.mica_clip_grad_norms(G, N, 1, 0, 1.0, 1.0, None, None, None) == NULL
    assert L.mica_clip_grad_norms(G, N, 1, 2, 1.0, 1.0, None, f, None) == DTYPE
    for mx, inv in ((0.0, 1.0), (-1.0, 1.0), (math.nan, 1.0), (1.0, 0.0), (1.0, math.inf), (1.0, -2.0)):
        assert L.mica_clip_grad_norms(G, N, 1, 0, mx, inv, None, f, None) == HYPER, (mx, inv)
    assert L.mica_clip_grad_norms(G, N, -2, 0, 1.0, 1.0, None, f, None) == COUNT


def test_accumulate_host_validation():
    """The fused add + norm checks its arguments on the host before anything is queued."""
    L = mica.lib()
    G = _arr(ctypes.c_void_p, [0x1000])
    A = _arr(ctypes.c_void_p, [0x3000])
    N = _arr(ctypes.c_int64, [4])
    f = ctypes.c_void_p(0x2000)
    acc = L.mica_accumulate_clip_grad_norms
    assert acc(G, A, N, 1, 0, 1.0, 1.0, None, None, None) == NULL         # no d_factor
    assert acc(G, None, N, 1, 0, 1.0, 1.0, None, f, None) == NULL         # no addend array
    assert acc(G, A, N, 1, 3, 1.0, 1.0, None, f, None) == DTYPE           # packed words are not gradients
    for mx, inv in ((0.0, 1.0), (math.nan, 1.0), (1.0, 0.0), (1.0, math.inf)):
        assert acc(G, A, N, 1, 0, mx, inv, None, f, None) == HYPER, (mx, inv)
    assert acc(G, A, N, -1, 0, 1.0, 1.0, None, f, None) == COUNT
    assert acc(G, A, _arr(ctypes.c_int64, [-4]), 1, 0, 1.0, 1.0, None, f, None) == COUNT
    nullA = _arr(ctypes.c_void_p, [None])
    assert acc(G, nullA, N, 1, 0, 1.0, 1.0, None, f, None) == NULL        # a NULL addend with n > 0
    assert acc(G, A, N, 1, 0, 1.0, 1.0, None, f, None) in (ADDRESS, DEVICE)  # host addresses: refused
    assert mica.lib().mica_last_error_detail().decode()
    sq = L.mica_accumulate_grad_sumsq
    assert sq(G, A, N, 1, 0, 1.0, None, None) == NULL                      # no d_sumsq
    assert sq(G, None, N, 1, 0, 1.0, f, None) == NULL
    assert sq(G, A, N, 1, 2, 1.0, f, None) == DTYPE
    for inv in (0.0, -1.0, math.inf, math.nan):
        assert sq(G, A, N, 1, 0, inv, f, None) == HYPER, inv
    assert sq(G, A, N, -3, 0, 1.0, f, None) == COUNT
    assert sq(G, A, N, 1, 0, 1.0, f, None) in (ADDRESS, DEVICE)


def test_clip_adamw_step_host_validation():
    """The fused step checks the norm's arguments and the update's, on the host, before anything is queued."""
    L = mica.lib()
    P = _arr(ctypes.c_void_p, [0x1000])
    N = _arr(ctypes.c_int64, [4])
    f = ctypes.c_void_p(0x2000)

    def step(hp=None, gdt=0, mdt=0, mx=1.0, inv=1.0, factor=f, T=1, n=N):
        hp_ref = ctypes.byref(hp) if hp is not None else None
        return L.mica_clip_adamw_step(P, P, P, P, n, T, gdt, mdt, hp_ref, mx, inv, None, factor, None)
    assert step(hp=_hp(), factor=None) == NULL
    assert step(hp=None) == NULL
    assert step(hp=_hp(), gdt=2) == DTYPE
    assert step(hp=_hp(), mdt=1) == DTYPE
    for mx, inv in ((0.0, 1.0), (math.nan, 1.0), (1.0, 0.0), (1.0, math.inf)):
        assert step(hp=_hp(), mx=mx, inv=inv) == HYPER, (mx, inv)
    assert step(hp=_hp(lr=-1.0)) == HYPER
    assert step(hp=_hp(beta2=1.0)) == BETA
    assert step(hp=_hp(), T=-1) == COUNT
    assert step(hp=_hp(), n=_arr(ctypes.c_int64, [-4])) == COUNT


def test_scale_host_validation():
    L = mica.lib()
    t = _arr(ctypes.c_void_p, [0x1000])
    N = _arr(ctypes.c_int64, [4])
    assert L.mica_scale_tensors(t, N, 1, 2, 1.0, None, None) == DTYPE
    assert L.mica_scale_tensors(t, N, 1, 0, math.inf, None, None) == HYPER
    assert L.mica_scale_tensors(t, N, 1, 0, math.nan, None, None) == HYPER
    assert L.mica_scale_tensors(None, N, 1, 0, 1.0, None, None) == NULL
    assert L.mica_scale_tensors(t, N, 0, 0, 1.0, None, None) == OK


def test_selftest_host_validation():
    L = mica.lib()
    for fn in (L.mica_selftest_wait_timeout, L.mica_selftest_grid_wait_timeout):
        assert fn(0, None) == HYPER
        assert fn((1 << 20) + 1, None) == HYPER


def test_no_kernels_without_a_device():
    import torch
    if torch.cuda.is_available():
        pytest.skip("counts launches only on a host without a GPU")
    assert mica.mica_launch_count() == 0


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    from clip_tensor_adamw_gb300 import mica as m
    monkeypatch.setattr(m, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(m, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        m.lib()


def test_binding_checks_each_list_dtype_once():
    """The binding refuses, before any call, a list that mixes dtypes (it passes one dtype for the whole list to
    the library) and weights or momentum buffers that are not float32."""
    import torch
    with pytest.raises(TypeError, match="mixes dtypes"):
        mica.TensorList([torch.zeros(4), torch.zeros(4, dtype=torch.float16)])
    L = mica.TensorList([torch.zeros(4), torch.zeros(8)])
    assert L.dtype == torch.float32 and L.total == 12
    assert mica.TensorList([]).dtype is None
    half = [torch.zeros(8, dtype=torch.float16)]
    f32 = [torch.zeros(8)]
    kw = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, step=1)
    with pytest.raises(TypeError, match="float32"):
        mica.mica_adamw_steps(half, f32, f32, f32, **kw)
    with pytest.raises(TypeError, match="float32"):
        mica.mica_sgd_steps(f32, f32, half, lr=0.1, momentum=0.9)
    with pytest.raises(TypeError, match="dtype"):
        mica.mica_accumulate_clip_grad_norms(f32, half, 1.0)
