"""Python face of the CPU oracle for the clip + AdamW optimizer step.

TEST INFRASTRUCTURE. Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg (and its
``--impl reference`` arm) import this package. The product library never imports, loads or calls it, and this
package imports nothing of the product's.

The arithmetic lives in ``oracle.c`` (plain C, one thread, ``-O2 -ffp-contract=off``); this module only compiles it,
loads it with ctypes and passes numpy arrays in and out. Which page and section each function follows is written
beside each C function. Arrays are host numpy arrays:

* float32 tensors: ``np.float32``;
* binary16 gradients: ``np.float16`` (passed as their bits);
* packed BF16 moments: ``np.uint32`` of ``ceil(n/2)`` words, element 2k in the low half of word k.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F32, F16, BF16X2, BF16X2_M = 0, 1, 2, 3
SKIP_NONFINITE, COUPLED_L2 = 1, 2
CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-shared", "-fPIC"]


def build(src: str = _SRC, out: str = _LIB, extra: list[str] | None = None) -> str:
    """Compile ``oracle.c`` into a shared library with gcc; returns its path."""
    cmd = ["gcc", *CFLAGS, *(extra or []), "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


class _Scalars(ctypes.Structure):
    _fields_ = [(k, ctypes.c_float) for k in ("c1", "b2", "c2", "step", "bc2", "dec", "eps", "wd")]


_P = ctypes.c_void_p
_I64P = ctypes.POINTER(ctypes.c_int64)


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    lib.ora_bf16_from_bits.argtypes = [ctypes.c_uint32]
    lib.ora_bf16_from_bits.restype = ctypes.c_uint16
    lib.ora_f32_from_bf16.argtypes = [ctypes.c_uint16]
    lib.ora_f32_from_bf16.restype = ctypes.c_float
    lib.ora_f32_from_f16.argtypes = [ctypes.c_uint16]
    lib.ora_f32_from_f16.restype = ctypes.c_float
    lib.ora_f16_from_f32.argtypes = [ctypes.c_float]
    lib.ora_f16_from_f32.restype = ctypes.c_uint16
    for name in ("ora_bf16_from_bits_array", "ora_f32_from_bf16_array", "ora_f32_from_f16_array",
                 "ora_f16_from_f32_array"):
        fn = getattr(lib, name)
        fn.argtypes = [_P, _P, ctypes.c_int64]
        fn.restype = None
    lib.ora_step_scalars.argtypes = [ctypes.c_double] * 5 + [ctypes.c_int64, ctypes.POINTER(_Scalars)]
    lib.ora_step_scalars.restype = None
    lib.ora_sum_squares.argtypes = [_P, _I64P, ctypes.c_int32, ctypes.c_int32, ctypes.c_float]
    lib.ora_sum_squares.restype = ctypes.c_double
    lib.ora_norm_from_sum.argtypes = [ctypes.c_double]
    lib.ora_norm_from_sum.restype = ctypes.c_float
    lib.ora_clip_factor.argtypes = [ctypes.c_float] * 3
    lib.ora_clip_factor.restype = ctypes.c_float
    lib.ora_adam_group.argtypes = [_P, _P, _P, _P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                   ctypes.POINTER(_Scalars), ctypes.c_float, ctypes.c_int32, ctypes.c_int32]
    lib.ora_adam_group.restype = None
    for name in ("ora_adamw_steps", "ora_adam_l2_steps"):
        fn = getattr(lib, name)
        fn.argtypes = [_P, _P, _P, _P, _I64P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                       ctypes.POINTER(_Scalars), ctypes.c_float, ctypes.c_int32]
        fn.restype = None
    lib.ora_adam_steps_flags.argtypes = [_P, _P, _P, _P, _I64P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                         ctypes.POINTER(_Scalars), ctypes.c_float, ctypes.c_int32, ctypes.c_uint32]
    lib.ora_adam_steps_flags.restype = None
    lib.ora_adam_steps_grouped.argtypes = [_P, _P, _P, _P, _I64P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                           _P, ctypes.POINTER(_Scalars), ctypes.c_float, ctypes.c_int32,
                                           ctypes.c_uint32]
    lib.ora_adam_steps_grouped.restype = None
    lib.ora_sgd_steps.argtypes = [_P, _P, _P, _I64P, ctypes.c_int32, ctypes.c_int32, ctypes.c_double,
                                  ctypes.c_double, ctypes.c_float, ctypes.c_int32, ctypes.c_uint32]
    lib.ora_sgd_steps.restype = None
    lib.ora_clip_grad_norms.argtypes = [_P, _I64P, ctypes.c_int32, ctypes.c_int32, ctypes.c_float, ctypes.c_float,
                                        ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_float),
                                        ctypes.POINTER(ctypes.c_double)]
    lib.ora_clip_grad_norms.restype = None
    lib.ora_scale_tensors.argtypes = [_P, _I64P, ctypes.c_int32, ctypes.c_int32, ctypes.c_float]
    lib.ora_scale_tensors.restype = None
    lib.ora_accumulate_grads.argtypes = [_P, _P, _I64P, ctypes.c_int32, ctypes.c_int32]
    lib.ora_accumulate_grads.restype = None
    lib.ora_accumulate_clip_grad_norms.argtypes = [_P, _P, _I64P, ctypes.c_int32, ctypes.c_int32, ctypes.c_float,
                                                   ctypes.c_float, ctypes.POINTER(ctypes.c_float),
                                                   ctypes.POINTER(ctypes.c_float)]
    lib.ora_accumulate_clip_grad_norms.restype = None
    return lib


_lib_cache: dict[str, ctypes.CDLL] = {}


def load(path: str = _LIB) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library at ``path``."""
    if path not in _lib_cache:
        if path == _LIB and (not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)):
            build()
        _lib_cache[path] = _declare(ctypes.CDLL(path))
    return _lib_cache[path]


@dataclass(frozen=True)
class Hyper:
    """One AdamW step's hyperparameters; ``step`` is the 1-based t."""
    lr: float
    beta1: float
    beta2: float
    eps: float
    weight_decay: float
    step: int


def _ptrs(arrays) -> ctypes.Array:
    arr = (ctypes.c_void_p * max(1, len(arrays)))()
    for i, a in enumerate(arrays):
        arr[i] = a.ctypes.data if a.size else None
    return arr


def _sizes(ns) -> ctypes.Array:
    arr = (ctypes.c_int64 * max(1, len(ns)))()
    for i, k in enumerate(ns):
        arr[i] = int(k)
    return arr


def _gdt(g: np.ndarray) -> int:
    if g.dtype == np.float32:
        return F32
    if g.dtype == np.float16:
        return F16
    raise TypeError(f"gradient dtype {g.dtype} is neither float32 nor float16")


def _mdt(m: np.ndarray, v: np.ndarray | None = None) -> int:
    if m.dtype == np.float32:
        return F32
    if m.dtype == np.uint32:
        return BF16X2_M if v is not None and v.dtype == np.float32 else BF16X2
    raise TypeError(f"moment dtype {m.dtype} is neither float32 nor packed uint32")


class Oracle:
    """The oracle's functions bound to one compiled copy of ``oracle.c`` (the default, or a test's variant)."""

    def __init__(self, path: str = _LIB):
        self.lib = load(path)

    # ---- element conversions ----
    def _map(self, fn, x: np.ndarray, in_dtype, out_dtype) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=in_dtype)
        out = np.empty(x.shape, out_dtype)
        fn(x.ctypes.data, out.ctypes.data, x.size)
        return out

    def bf16_from_f32_bits(self, u: np.ndarray) -> np.ndarray:
        """float32 bit patterns -> BF16 bit patterns (nearest-even, NaN -> 0xFFFF)."""
        return self._map(self.lib.ora_bf16_from_bits_array, u, np.uint32, np.uint16)

    def f32_from_bf16(self, h: np.ndarray) -> np.ndarray:
        return self._map(self.lib.ora_f32_from_bf16_array, h, np.uint16, np.float32)

    def f32_from_f16_bits(self, h: np.ndarray) -> np.ndarray:
        return self._map(self.lib.ora_f32_from_f16_array, h, np.uint16, np.float32)

    def f16_bits_from_f32(self, x: np.ndarray) -> np.ndarray:
        return self._map(self.lib.ora_f16_from_f32_array, x, np.float32, np.uint16)

    def scalars(self, hp: Hyper) -> dict:
        s = _Scalars()
        self.lib.ora_step_scalars(hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, hp.step, ctypes.byref(s))
        return {k: np.float32(getattr(s, k)) for k, _ in _Scalars._fields_}

    def _scalars_struct(self, hp: Hyper) -> _Scalars:
        s = _Scalars()
        self.lib.ora_step_scalars(hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, hp.step, ctypes.byref(s))
        return s

    # ---- ClipGradNorms ----
    def sum_squares(self, grads, inv_scale: float = 1.0) -> float:
        gdt = _gdt(grads[0]) if grads else F32
        return self.lib.ora_sum_squares(_ptrs(grads), _sizes([g.size for g in grads]), len(grads), gdt,
                                        np.float32(inv_scale))

    def clip_grad_norms(self, grads, max_norm: float, inv_scale: float = 1.0):
        """Returns ``(norm, factor, sum_of_squares)``: float32, float32, float64."""
        gdt = _gdt(grads[0]) if grads else F32
        norm, factor, S = ctypes.c_float(), ctypes.c_float(), ctypes.c_double()
        self.lib.ora_clip_grad_norms(_ptrs(grads), _sizes([g.size for g in grads]), len(grads), gdt,
                                     np.float32(max_norm), np.float32(inv_scale), ctypes.byref(norm),
                                     ctypes.byref(factor), ctypes.byref(S))
        return np.float32(norm.value), np.float32(factor.value), S.value

    def clip_factor(self, norm: float, max_norm: float, inv_scale: float = 1.0) -> np.float32:
        return np.float32(self.lib.ora_clip_factor(np.float32(norm), np.float32(max_norm), np.float32(inv_scale)))

    # ---- AdamWSteps ----
    def adamw_steps(self, ws, gs, ms, vs, hp: Hyper, factor: float = 1.0, zero_grad: bool = False,
                    decoupled: bool = True, skip_nonfinite: bool = False) -> None:
        """In place over the lists; ``decoupled=False`` is Adam with the coupled L2 term; ``skip_nonfinite`` leaves
        w, m, v as they are when the factor is not > 0. Packed m with float32 v is the BF16X2_M moment type."""
        T = len(ws)
        if T == 0:
            return
        gdt, mdt = _gdt(gs[0]), _mdt(ms[0], vs[0])
        for w, g, m, v in zip(ws, gs, ms, vs):
            assert w.dtype == np.float32 and w.flags.c_contiguous and g.size == w.size
            half = (w.size + 1) // 2
            assert m.size == (half if mdt in (BF16X2, BF16X2_M) else w.size)
            assert v.size == (half if mdt == BF16X2 else w.size)
        s = self._scalars_struct(hp)
        if skip_nonfinite:
            flags = SKIP_NONFINITE | (0 if decoupled else COUPLED_L2)
            self.lib.ora_adam_steps_flags(_ptrs(ws), _ptrs(gs), _ptrs(ms), _ptrs(vs), _sizes([w.size for w in ws]), T,
                                          gdt, mdt, ctypes.byref(s), np.float32(factor), int(bool(zero_grad)), flags)
            return
        fn = self.lib.ora_adamw_steps if decoupled else self.lib.ora_adam_l2_steps
        fn(_ptrs(ws), _ptrs(gs), _ptrs(ms), _ptrs(vs), _sizes([w.size for w in ws]), T, gdt, mdt, ctypes.byref(s),
           np.float32(factor), int(bool(zero_grad)))

    def adamw_steps_grouped(self, ws, gs, ms, vs, group, hps, factor: float = 1.0, zero_grad: bool = False,
                            decoupled: bool = True, skip_nonfinite: bool = False) -> None:
        """As ``adamw_steps`` over a list split into parameter groups: tensor k steps with ``hps[group[k]]``."""
        T = len(ws)
        if T == 0:
            return
        assert len(group) == T and all(0 <= int(x) < len(hps) for x in group)
        gdt, mdt = _gdt(gs[0]), _mdt(ms[0], vs[0])
        for w, g, m, v in zip(ws, gs, ms, vs):
            assert w.dtype == np.float32 and w.flags.c_contiguous and g.size == w.size
            half = (w.size + 1) // 2
            assert m.size == (half if mdt in (BF16X2, BF16X2_M) else w.size)
            assert v.size == (half if mdt == BF16X2 else w.size)
        ss = (_Scalars * len(hps))(*[self._scalars_struct(hp) for hp in hps])
        grp = np.ascontiguousarray(group, dtype=np.int32)
        flags = (SKIP_NONFINITE if skip_nonfinite else 0) | (0 if decoupled else COUPLED_L2)
        self.lib.ora_adam_steps_grouped(_ptrs(ws), _ptrs(gs), _ptrs(ms), _ptrs(vs), _sizes([w.size for w in ws]), T,
                                        gdt, mdt, grp.ctypes.data, ss, np.float32(factor), int(bool(zero_grad)),
                                        flags)

    # ---- SGD and SGD with momentum ----
    def sgd_steps(self, ws, gs, bufs, lr: float, momentum: float = 0.0, factor: float = 1.0,
                  zero_grad: bool = False, skip_nonfinite: bool = False) -> None:
        """In place; ``bufs`` None is plain SGD, else one float32 momentum buffer per tensor."""
        T = len(ws)
        if T == 0:
            return
        gdt = _gdt(gs[0])
        for k, (w, g) in enumerate(zip(ws, gs)):
            assert w.dtype == np.float32 and w.flags.c_contiguous and g.size == w.size
            if bufs is not None:
                assert bufs[k].dtype == np.float32 and bufs[k].size == w.size
        self.lib.ora_sgd_steps(_ptrs(ws), _ptrs(gs), None if bufs is None else _ptrs(bufs),
                               _sizes([w.size for w in ws]), T, gdt, float(lr), float(momentum), np.float32(factor),
                               int(bool(zero_grad)), SKIP_NONFINITE if skip_nonfinite else 0)

    def clip_sgd_step(self, ws, gs, bufs, lr: float, momentum: float, max_norm: float, inv_scale: float = 1.0,
                      zero_grad: bool = False, skip_nonfinite: bool = False):
        """Norm, clip factor, then SGD (or SGD with momentum) over every tensor. Returns ``(norm, factor)``."""
        norm, factor, _ = self.clip_grad_norms(gs, max_norm, inv_scale)
        self.sgd_steps(ws, gs, bufs, lr, momentum, factor=factor, zero_grad=zero_grad, skip_nonfinite=skip_nonfinite)
        return norm, factor

    # ---- ScaleTensors ----
    def scale_tensors(self, ts, factor: float) -> None:
        if not ts:
            return
        dt = _gdt(ts[0])
        self.lib.ora_scale_tensors(_ptrs(ts), _sizes([t.size for t in ts]), len(ts), dt, np.float32(factor))

    # ---- the gradient's last write (an add) with the norm of its result ----
    def accumulate_grads(self, gs, adds) -> None:
        """gs[k] += adds[k] in place, each sum rounded to the gradients' type."""
        if not gs:
            return
        dt = _gdt(gs[0])
        assert all(a.dtype == g.dtype and a.size == g.size for g, a in zip(gs, adds))
        self.lib.ora_accumulate_grads(_ptrs(gs), _ptrs(adds), _sizes([g.size for g in gs]), len(gs), dt)

    def accumulate_clip_grad_norms(self, gs, adds, max_norm: float, inv_scale: float = 1.0):
        """gs[k] += adds[k], then the joint norm and factor of the result. Returns ``(norm, factor)``."""
        gdt = _gdt(gs[0]) if gs else F32
        assert all(a.dtype == g.dtype and a.size == g.size for g, a in zip(gs, adds))
        norm, factor = ctypes.c_float(), ctypes.c_float()
        self.lib.ora_accumulate_clip_grad_norms(_ptrs(gs), _ptrs(adds), _sizes([g.size for g in gs]), len(gs), gdt,
                                                np.float32(max_norm), np.float32(inv_scale), ctypes.byref(norm),
                                                ctypes.byref(factor))
        return np.float32(norm.value), np.float32(factor.value)

    # ---- the whole hot path ----
    def clip_adamw_step(self, ws, gs, ms, vs, hp: Hyper, max_norm: float, inv_scale: float = 1.0,
                        zero_grad: bool = False, decoupled: bool = True, skip_nonfinite: bool = False):
        """Norm, clip factor, then the Adam-family update over every group. Returns ``(norm, factor)``."""
        norm, factor, _ = self.clip_grad_norms(gs, max_norm, inv_scale)
        self.adamw_steps(ws, gs, ms, vs, hp, factor=factor, zero_grad=zero_grad, decoupled=decoupled,
                         skip_nonfinite=skip_nonfinite)
        return norm, factor


def packed_words(n: int) -> int:
    """Words of a packed BF16 buffer of n elements: ceil(n/2)."""
    return (n + 1) // 2


def unpack_bf16(words: np.ndarray, n: int) -> np.ndarray:
    """Packed words -> float32 values of the n elements (exact widening; element 2k low half of word k)."""
    w = np.asarray(words, np.uint32)
    halves = np.empty(2 * w.size, np.uint32)
    halves[0::2] = w & 0xFFFF
    halves[1::2] = w >> 16
    return (halves[:n] << 16).view(np.float32)
