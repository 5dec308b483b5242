"""Python binding of libmica_optim.so: the entry points of the C ABI (include/mica_optim.h), taking torch tensors.

This module only marshals arguments: it collects data pointers, element counts, the current CUDA stream and the
hyperparameters into the C call, and turns a non-OK status into an exception. Every element of the step is read and
written by the library's kernels; there is no fallback when the library is missing or the call fails.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# the library this package builds; MICA_LIB names another build of the same ABI instead
LIB_PATH = os.environ.get("MICA_LIB") or os.path.join(_PKG, "libmica_optim.so")

MICA_F32, MICA_F16, MICA_BF16X2, MICA_BF16X2_M = 0, 1, 2, 3
MICA_STEP_SKIP_NONFINITE, MICA_STEP_COUPLED_L2 = 1, 2
STATUS = ["MICA_OK", "MICA_ERR_NULL", "MICA_ERR_COUNT", "MICA_ERR_DTYPE", "MICA_ERR_HYPER", "MICA_ERR_BETA",
          "MICA_ERR_OVERLAP", "MICA_ERR_DEVICE", "MICA_ERR_ADDRESS", "MICA_ERR_CUDA", "MICA_ERR_NOMEM",
          "MICA_ERR_CAPTURE"]


class MicaError(RuntimeError):
    """A non-OK status from the library; ``status`` is its name, the message the library's one-line detail."""

    def __init__(self, status: int, detail: str):
        self.status = STATUS[status] if 0 <= status < len(STATUS) else f"status {status}"
        super().__init__(f"{self.status}: {detail}")


MICA_MAX_GROUPS = 8


class _SgdHP(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("momentum", ctypes.c_double), ("zero_grad", ctypes.c_int32),
                ("flags", ctypes.c_uint32)]


class _HP(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("eps", ctypes.c_double), ("weight_decay", ctypes.c_double), ("step", ctypes.c_int64),
                ("zero_grad", ctypes.c_int32), ("flags", ctypes.c_uint32)]


_P = ctypes.c_void_p
_I64P = ctypes.POINTER(ctypes.c_int64)
_lib: ctypes.CDLL | None = None


def lib() -> ctypes.CDLL:
    """The loaded library. Raises if it has not been built: nothing here runs without it."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m clip_tensor_adamw_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        L.mica_scale_tensors.argtypes = [_P, _I64P, ctypes.c_int32, ctypes.c_int32, ctypes.c_float, _P, _P]
        L.mica_clip_grad_norms.argtypes = [_P, _I64P, ctypes.c_int32, ctypes.c_int32, ctypes.c_float,
                                           ctypes.c_float, _P, _P, _P]
        L.mica_adamw_steps.argtypes = [_P, _P, _P, _P, _I64P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                       ctypes.POINTER(_HP), _P, _P]
        L.mica_adamw_steps_grouped.argtypes = [_P, _P, _P, _P, _I64P, ctypes.c_int32, ctypes.c_int32,
                                               ctypes.c_int32, _P, ctypes.POINTER(_HP), ctypes.c_int32, _P, _P]
        L.mica_sgd_steps.argtypes = [_P, _P, _P, _I64P, ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(_SgdHP),
                                     _P, _P]
        L.mica_clip_adamw_step.argtypes = [_P, _P, _P, _P, _I64P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                           ctypes.POINTER(_HP), ctypes.c_float, ctypes.c_float, _P, _P, _P]
        L.mica_grad_sumsq.argtypes = [_P, _I64P, ctypes.c_int32, ctypes.c_int32, ctypes.c_float, _P, _P]
        L.mica_accumulate_clip_grad_norms.argtypes = [_P, _P, _I64P, ctypes.c_int32, ctypes.c_int32, ctypes.c_float,
                                                      ctypes.c_float, _P, _P, _P]
        L.mica_accumulate_grad_sumsq.argtypes = [_P, _P, _I64P, ctypes.c_int32, ctypes.c_int32, ctypes.c_float, _P, _P]
        L.mica_clip_factor_from_sumsq.argtypes = [_P, ctypes.c_int32, ctypes.c_float, ctypes.c_float, _P, _P, _P]
        for f in ("mica_scale_tensors", "mica_clip_grad_norms", "mica_adamw_steps", "mica_adamw_steps_grouped",
                  "mica_sgd_steps", "mica_clip_adamw_step", "mica_grad_sumsq", "mica_clip_factor_from_sumsq",
                  "mica_accumulate_clip_grad_norms", "mica_accumulate_grad_sumsq", "mica_sync", "mica_release_cache"):
            getattr(L, f).restype = ctypes.c_int
        for f in ("mica_selftest_wait_timeout", "mica_selftest_grid_wait_timeout"):
            getattr(L, f).argtypes = [ctypes.c_uint32, _P]
            getattr(L, f).restype = ctypes.c_int
        L.mica_sync.argtypes = [_P]
        L.mica_release_cache.argtypes = []
        L.mica_status_string.argtypes = [ctypes.c_int]
        L.mica_status_string.restype = ctypes.c_char_p
        L.mica_last_error_detail.argtypes = []
        L.mica_last_error_detail.restype = ctypes.c_char_p
        L.mica_launch_count.argtypes = []
        L.mica_launch_count.restype = ctypes.c_uint64
        L.mica_abi_version.argtypes = []
        L.mica_abi_version.restype = ctypes.c_int32
        _I32P = ctypes.POINTER(ctypes.c_int32)
        L.mica_work_items.argtypes = [_I64P, _I32P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _I64P,
                                      ctypes.c_int32, _I32P, ctypes.c_int32, _I32P, _I32P, _I32P]
        L.mica_work_items.restype = ctypes.c_int
        _lib = L
    return _lib


def _check(status: int) -> None:
    if status != 0:
        raise MicaError(status, lib().mica_last_error_detail().decode())


class TensorList:
    """The pointer and size arrays of a list of tensors, built once and reusable across calls (the tensors must stay
    alive and in place). Element counts are those of the tensors, or ``sizes`` when given (packed moments hold
    ceil(n/2) words for n elements, so their list carries the elements' counts). Every tensor of a list must have
    the same dtype (checked here, once, so that a call reads one dtype for the whole list)."""

    def __init__(self, tensors: Sequence[torch.Tensor], sizes: Sequence[int] | None = None):
        self.tensors = list(tensors)
        T = len(self.tensors)
        self.T = T
        self.ptrs = (ctypes.c_void_p * max(T, 1))()
        for i, t in enumerate(self.tensors):
            if not t.is_contiguous():
                raise ValueError(f"tensor {i} is not contiguous")
            self.ptrs[i] = t.data_ptr() if t.numel() else None
        counts = [t.numel() for t in self.tensors] if sizes is None else list(sizes)
        self.n = (ctypes.c_int64 * max(T, 1))(*counts)
        self.counts = counts
        self.total = sum(counts)
        dtypes = {t.dtype for t in self.tensors}
        if len(dtypes) > 1:
            raise TypeError(f"a tensor list mixes dtypes {sorted(str(d) for d in dtypes)}")
        self.dtype = dtypes.pop() if dtypes else None


def _as_list(x, sizes=None) -> TensorList:
    return x if isinstance(x, TensorList) else TensorList(x, sizes)


def _dtype_code(L: TensorList, what: str) -> int:
    """The ABI dtype of a list's tensors (float32 for an empty list)."""
    if L.dtype is None or L.dtype == torch.float32:
        return MICA_F32
    if L.dtype == torch.float16:
        return MICA_F16
    if L.dtype == torch.int32 or str(L.dtype) == "torch.uint32":  # packed BF16 words
        return MICA_BF16X2
    raise TypeError(f"{what}: unsupported dtype {L.dtype}")


def _weights(W: TensorList) -> None:
    if W.dtype is not None and W.dtype != torch.float32:
        raise TypeError(f"w: the weights must be float32, not {W.dtype}")


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: torch.Tensor | None):
    return None if t is None else t.data_ptr()


def mica_scale_tensors(tensors, factor: float = 1.0, d_factor: torch.Tensor | None = None, stream=None) -> None:
    """ScaleTensors: every cell of every tensor times ``factor`` (or the device scalar ``d_factor``), in place."""
    L = _as_list(tensors)
    dt = _dtype_code(L, "tensors")
    _check(lib().mica_scale_tensors(L.ptrs, L.n, L.T, dt, float(factor), _ptr(d_factor), _stream(stream)))


def mica_clip_grad_norms(grads, max_norm: float, inv_scale: float = 1.0, norm_out: torch.Tensor | None = None,
                         factor_out: torch.Tensor | None = None, stream=None):
    """ClipGradNorms: the joint norm of the unscaled gradients and the folded clip factor, as two one-element
    float32 device tensors (``norm_out`` / ``factor_out`` when given). Nothing is copied to the host."""
    L = _as_list(grads)
    dev = L.tensors[0].device if L.T else torch.device("cuda", torch.cuda.current_device())
    if norm_out is None:
        norm_out = torch.empty(1, dtype=torch.float32, device=dev)
    if factor_out is None:
        factor_out = torch.empty(1, dtype=torch.float32, device=dev)
    gdt = _dtype_code(L, "grads")
    _check(lib().mica_clip_grad_norms(L.ptrs, L.n, L.T, gdt, float(max_norm), float(inv_scale), _ptr(norm_out),
                                      _ptr(factor_out), _stream(stream)))
    return norm_out, factor_out


def mica_accumulate_clip_grad_norms(grads, addends, max_norm: float, inv_scale: float = 1.0,
                                    norm_out: torch.Tensor | None = None, factor_out: torch.Tensor | None = None,
                                    stream=None):
    """The gradients' last write as an add, fused with ClipGradNorms: ``grads[k] += addends[k]`` in place (each sum
    rounded to the gradients' type), then the joint norm and clip factor of the result, in one pass over the list.
    Returns the device (norm, factor) as ``mica_clip_grad_norms`` does."""
    G = _as_list(grads)
    A = _as_list(addends)
    if A.T != G.T or A.total != G.total:  # the call passes the gradients' counts for both lists
        raise ValueError("addends must match the gradients tensor for tensor")
    if G.T and A.dtype != G.dtype:
        raise TypeError("addends must have the gradients' dtype")
    dev = G.tensors[0].device if G.T else torch.device("cuda", torch.cuda.current_device())
    if norm_out is None:
        norm_out = torch.empty(1, dtype=torch.float32, device=dev)
    if factor_out is None:
        factor_out = torch.empty(1, dtype=torch.float32, device=dev)
    gdt = _dtype_code(G, "grads")
    _check(lib().mica_accumulate_clip_grad_norms(G.ptrs, A.ptrs, G.n, G.T, gdt, float(max_norm), float(inv_scale),
                                                 _ptr(norm_out), _ptr(factor_out), _stream(stream)))
    return norm_out, factor_out


def mica_accumulate_grad_sumsq(grads, addends, inv_scale: float = 1.0, out: torch.Tensor | None = None,
                               stream=None) -> torch.Tensor:
    """``grads[k] += addends[k]`` in place, then the sum of squares of the unscaled result, exactly as the norm sums
    it, as a one-element float64 device tensor (``out`` when given): one rank's share of a sharded list's joint
    norm, with the add fused into its pass."""
    G = _as_list(grads)
    A = _as_list(addends)
    if A.T != G.T or A.total != G.total:  # the call passes the gradients' counts for both lists
        raise ValueError("addends must match the gradients tensor for tensor")
    if G.T and A.dtype != G.dtype:
        raise TypeError("addends must have the gradients' dtype")
    dev = G.tensors[0].device if G.T else torch.device("cuda", torch.cuda.current_device())
    if out is None:
        out = torch.empty(1, dtype=torch.float64, device=dev)
    gdt = _dtype_code(G, "grads")
    _check(lib().mica_accumulate_grad_sumsq(G.ptrs, A.ptrs, G.n, G.T, gdt, float(inv_scale), _ptr(out),
                                            _stream(stream)))
    return out


def mica_grad_sumsq(grads, inv_scale: float = 1.0, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The sum of squares of the unscaled gradients, exactly as the norm sums it, as a one-element float64 device
    tensor (``out`` when given): one rank's share of a sharded list's joint norm."""
    L = _as_list(grads)
    dev = L.tensors[0].device if L.T else torch.device("cuda", torch.cuda.current_device())
    if out is None:
        out = torch.empty(1, dtype=torch.float64, device=dev)
    gdt = _dtype_code(L, "grads")
    _check(lib().mica_grad_sumsq(L.ptrs, L.n, L.T, gdt, float(inv_scale), _ptr(out), _stream(stream)))
    return out


def mica_clip_factor_from_sumsq(parts: torch.Tensor, max_norm: float, inv_scale: float = 1.0,
                                norm_out: torch.Tensor | None = None, factor_out: torch.Tensor | None = None,
                                stream=None):
    """Norm and clip factor from the ranks' square sums ``parts`` (a float64 device tensor, in rank order), added
    in that order: every rank passing the same parts gets the same bits. Returns the device (norm, factor)."""
    if parts.dtype != torch.float64 or not parts.is_contiguous():
        raise TypeError("parts must be a contiguous float64 tensor")
    if norm_out is None:
        norm_out = torch.empty(1, dtype=torch.float32, device=parts.device)
    if factor_out is None:
        factor_out = torch.empty(1, dtype=torch.float32, device=parts.device)
    _check(lib().mica_clip_factor_from_sumsq(_ptr(parts), parts.numel(), float(max_norm), float(inv_scale),
                                             _ptr(norm_out), _ptr(factor_out), _stream(stream)))
    return norm_out, factor_out


@dataclass
class AdamWHyper:
    lr: float
    beta1: float
    beta2: float
    eps: float
    weight_decay: float


def mica_adamw_steps(w, g, m, v, *, lr: float, beta1: float, beta2: float, eps: float, weight_decay: float,
                     step: int, zero_grad: bool = False, factor: torch.Tensor | None = None, stream=None,
                     skip_nonfinite: bool = False, coupled_l2: bool = False) -> None:
    """AdamWSteps over every group in one launch, in place. ``m`` and ``v`` are float32 tensors of the weights'
    shapes, or int32 tensors of ceil(n/2) packed BF16 words (packed m with float32 v is allowed); ``factor`` is the
    device scalar from mica_clip_grad_norms (None: 1). ``skip_nonfinite`` leaves w, m, v as they are when the factor
    is not > 0 (the norm was not finite); ``coupled_l2`` is Adam's coupled L2 form instead of AdamW's decay."""
    W = _as_list(w)
    _weights(W)
    sizes = W.counts
    G = _as_list(g)
    M = _as_list(m, sizes)
    V = _as_list(v, sizes)
    if not (W.T == G.T == M.T == V.T):
        raise ValueError("w, g, m and v must list the same number of tensors")
    gdt = _dtype_code(G, "g")
    mdt = _dtype_code(M, "m")
    if mdt == MICA_BF16X2 and V.T and _dtype_code(V, "v") == MICA_F32:
        mdt = MICA_BF16X2_M
    flags = (MICA_STEP_SKIP_NONFINITE if skip_nonfinite else 0) | (MICA_STEP_COUPLED_L2 if coupled_l2 else 0)
    hp = _HP(float(lr), float(beta1), float(beta2), float(eps), float(weight_decay), int(step), int(bool(zero_grad)),
             flags)
    _check(lib().mica_adamw_steps(W.ptrs, G.ptrs, M.ptrs, V.ptrs, W.n, W.T, gdt, mdt, ctypes.byref(hp), _ptr(factor),
                                  _stream(stream)))


def mica_clip_adamw_step(w, g, m, v, *, max_norm: float, inv_scale: float = 1.0, lr: float, beta1: float,
                         beta2: float, eps: float, weight_decay: float, step: int, zero_grad: bool = False,
                         norm_out: torch.Tensor | None = None, factor_out: torch.Tensor | None = None, stream=None,
                         skip_nonfinite: bool = False, coupled_l2: bool = False):
    """One whole step: ClipGradNorms then AdamWSteps on the same list (one cooperative launch when the gradient
    fits in L2). Arguments as mica_clip_grad_norms and mica_adamw_steps; returns the device (norm, factor)."""
    W = _as_list(w)
    _weights(W)
    sizes = W.counts
    G = _as_list(g)
    M = _as_list(m, sizes)
    V = _as_list(v, sizes)
    if not (W.T == G.T == M.T == V.T):
        raise ValueError("w, g, m and v must list the same number of tensors")
    dev = G.tensors[0].device if G.T else torch.device("cuda", torch.cuda.current_device())
    if norm_out is None:
        norm_out = torch.empty(1, dtype=torch.float32, device=dev)
    if factor_out is None:
        factor_out = torch.empty(1, dtype=torch.float32, device=dev)
    gdt = _dtype_code(G, "g")
    mdt = _dtype_code(M, "m")
    if mdt == MICA_BF16X2 and V.T and _dtype_code(V, "v") == MICA_F32:
        mdt = MICA_BF16X2_M
    flags = (MICA_STEP_SKIP_NONFINITE if skip_nonfinite else 0) | (MICA_STEP_COUPLED_L2 if coupled_l2 else 0)
    hp = _HP(float(lr), float(beta1), float(beta2), float(eps), float(weight_decay), int(step), int(bool(zero_grad)),
             flags)
    _check(lib().mica_clip_adamw_step(W.ptrs, G.ptrs, M.ptrs, V.ptrs, W.n, W.T, gdt, mdt, ctypes.byref(hp),
                                      float(max_norm), float(inv_scale), _ptr(norm_out), _ptr(factor_out),
                                      _stream(stream)))
    return norm_out, factor_out


class GroupIndex:
    """The per-tensor group indices of mica_adamw_steps_grouped as a host int32 array, built once and reusable."""

    def __init__(self, group: Sequence[int]):
        self.values = [int(x) for x in group]
        self.arr = (ctypes.c_int32 * max(len(self.values), 1))(*self.values)


def mica_adamw_steps_grouped(w, g, m, v, group, groups: Sequence[dict], *, beta1: float, beta2: float, eps: float,
                             step: int, zero_grad: bool = False, factor: torch.Tensor | None = None, stream=None,
                             skip_nonfinite: bool = False, coupled_l2: bool = False) -> None:
    """AdamWSteps over parameter groups in one launch: tensor k is stepped with ``groups[group[k]]``, a dict with
    ``lr`` and ``weight_decay`` (the other hyperparameters are shared). ``group`` is a sequence of ints or a
    GroupIndex; the rest is as mica_adamw_steps."""
    W = _as_list(w)
    _weights(W)
    sizes = W.counts
    G = _as_list(g)
    M = _as_list(m, sizes)
    V = _as_list(v, sizes)
    if not (W.T == G.T == M.T == V.T):
        raise ValueError("w, g, m and v must list the same number of tensors")
    gi = group if isinstance(group, GroupIndex) else GroupIndex(group)
    if len(gi.values) != W.T:
        raise ValueError("group must hold one index per tensor")
    gdt = _dtype_code(G, "g")
    mdt = _dtype_code(M, "m")
    if mdt == MICA_BF16X2 and V.T and _dtype_code(V, "v") == MICA_F32:
        mdt = MICA_BF16X2_M
    flags = (MICA_STEP_SKIP_NONFINITE if skip_nonfinite else 0) | (MICA_STEP_COUPLED_L2 if coupled_l2 else 0)
    hps = (_HP * max(len(groups), 1))(*[
        _HP(float(gr["lr"]), float(beta1), float(beta2), float(eps), float(gr["weight_decay"]), int(step),
            int(bool(zero_grad)), flags) for gr in groups])
    _check(lib().mica_adamw_steps_grouped(W.ptrs, G.ptrs, M.ptrs, V.ptrs, W.n, W.T, gdt, mdt, gi.arr, hps,
                                          len(groups), _ptr(factor), _stream(stream)))


def mica_sgd_steps(w, g, buf=None, *, lr: float, momentum: float = 0.0, zero_grad: bool = False,
                   factor: torch.Tensor | None = None, stream=None, skip_nonfinite: bool = False) -> None:
    """SGD (``buf`` None) or SGD with momentum (one float32 buffer per tensor, zeros before the first step) over
    every tensor in one launch, in place; ``factor`` is the device scalar from mica_clip_grad_norms (None: 1)."""
    W = _as_list(w)
    _weights(W)
    G = _as_list(g)
    B = None if buf is None else _as_list(buf)
    if W.T != G.T or (B is not None and B.T != W.T):
        raise ValueError("w, g (and buf) must list the same number of tensors")
    if B is not None and B.dtype not in (None, torch.float32):
        raise TypeError(f"buf: the momentum buffers must be float32, not {B.dtype}")
    gdt = _dtype_code(G, "g")
    hp = _SgdHP(float(lr), float(momentum), int(bool(zero_grad)), MICA_STEP_SKIP_NONFINITE if skip_nonfinite else 0)
    _check(lib().mica_sgd_steps(W.ptrs, G.ptrs, None if B is None else B.ptrs, W.n, W.T, gdt, ctypes.byref(hp),
                                _ptr(factor), _stream(stream)))


def mica_work_items(sizes: Sequence[int], vec: Sequence[bool] | None = None, item_octs: int = 0, sms: int = 152):
    """The work items an update call cuts a list of ``sizes`` into (no device used): ``(items, pack, item_octs)``
    with items a list of (first tensor, tensor count, o0) in array order (the kernels take them from the end),
    pack the pack table, and the octets per slice used. ``vec``: which tensors take the vector path (default all)."""
    T = len(sizes)
    n = (ctypes.c_int64 * max(T, 1))(*[int(x) for x in sizes])
    v = (ctypes.c_int32 * max(T, 1))(*[1 if x else 0 for x in (vec if vec is not None else [True] * T)])
    num, plen, used = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _check(lib().mica_work_items(n, v, T, int(item_octs), int(sms), None, 0, None, 0, ctypes.byref(num),
                                 ctypes.byref(plen), ctypes.byref(used)))
    items = (ctypes.c_int64 * max(3 * num.value, 1))()
    pack = (ctypes.c_int32 * max(plen.value, 1))()
    _check(lib().mica_work_items(n, v, T, int(item_octs), int(sms), items, num.value, pack, plen.value,
                                 ctypes.byref(num), ctypes.byref(plen), ctypes.byref(used)))
    out = [(items[3 * i], items[3 * i + 1], items[3 * i + 2]) for i in range(num.value)]
    return out, list(pack[:plen.value]), used.value


def mica_sync(stream=None) -> None:
    _check(lib().mica_sync(_stream(stream)))


def mica_selftest_wait_timeout(polls: int = 16, stream=None) -> None:
    """Queues the self-test kernel whose bounded wait runs out; the next mica_sync raises MicaError (MICA_ERR_CUDA)."""
    _check(lib().mica_selftest_wait_timeout(int(polls), _stream(stream)))


def mica_selftest_grid_wait_timeout(polls: int = 16, stream=None) -> None:
    """Queues the self-test kernel whose grid-wide wait runs out; the next mica_sync raises MicaError."""
    _check(lib().mica_selftest_grid_wait_timeout(int(polls), _stream(stream)))


def mica_release_cache() -> None:
    _check(lib().mica_release_cache())


def mica_launch_count() -> int:
    return int(lib().mica_launch_count())
