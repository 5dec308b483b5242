"""Seeded synthetic inputs for the clip + AdamW step: parameter lists, gradients and zeroed moments.

This module holds random numbers and shapes only, none of the step's arithmetic. The oracle's tests, the GPU parity
tests, ``smoke()`` and ``bench.py`` all draw their inputs from here, so both sides of every comparison see the same
seeded values.

The five workloads (shapes and distributions as the optimizer-step benchmark states them; "N(0, s)" is a normal
with standard deviation s):

* ``tiny``: 4 float32 tensors [384,384], [384], [384,1536], [1536]; w ~ N(0, 0.02), g ~ N(0, 1e-2).
* ``gpt2_small``: GPT-2 small's 148 tensors (124,439,808 parameters), float32 moments, g ~ N(0, 1e-3).
* ``gpt2_small_bf16``: the same list with packed BF16 moments; g ~ N(0, 1e-3), each entry independently multiplied
  by 100 with probability 0.01, so that the clip fires.
* ``fp16_scaled``: 10,000 tensors of floor(exp(U(ln 64, ln 4096))) elements plus 12 of 768x3072; float16 gradients
  fp16(N(0, 1e-4) * 65536) (nearest-even), unscaled by 1/65536 inside the step; float32 moments.
* ``gpt2_xl``: GPT-2 XL's 580 tensors (1,557,611,200 parameters: d 1600, 48 layers, vocabulary 50257, context 1024),
  packed BF16 moments, g ~ N(0, 1e-4).

Every workload uses lr 6e-4, betas (0.9, 0.95), eps 1e-8, weight decay 0.1, clip 1.0 and starts from m = v = 0.

Buffers are laid out the way a training framework's parameter and gradient buckets are: one flat allocation per
stream, each tensor at an offset rounded up to 256 bytes, the tensors being views into it.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

ALIGN_BYTES = 256


@dataclass(frozen=True)
class Workload:
    name: str
    shapes: tuple
    grad_dtype: str = "f32"        # "f32" or "f16"
    moments: str = "f32"           # "f32", "bf16x2" (two BF16 per uint32 word) or "bf16x2_m" (m packed, v f32)
    w_std: float = 0.02
    g_std: float = 1e-3
    spike_p: float = 0.0           # probability that a gradient entry is multiplied by spike_mult
    spike_mult: float = 1.0
    loss_scale: float = 1.0        # float16 gradients are drawn as N(0, g_std) * loss_scale
    lr: float = 6e-4
    beta1: float = 0.9
    beta2: float = 0.95
    eps: float = 1e-8
    weight_decay: float = 0.1
    max_norm: float = 1.0
    steps: int = 10
    seed: int = 0

    @property
    def sizes(self) -> list[int]:
        return [int(np.prod(s)) for s in self.shapes]

    @property
    def params(self) -> int:
        return sum(self.sizes)

    @property
    def inv_scale(self) -> float:
        return 1.0 / self.loss_scale


def _gpt2_shapes(d: int, layers: int, vocab: int = 50257, ctx: int = 1024) -> tuple:
    shapes = [(vocab, d), (ctx, d)]
    for _ in range(layers):
        shapes += [(d,), (d,),                  # ln_1 weight, bias
                   (d, 3 * d), (3 * d,),        # c_attn
                   (d, d), (d,),                # attention c_proj
                   (d,), (d,),                  # ln_2 weight, bias
                   (d, 4 * d), (4 * d,),        # mlp c_fc
                   (4 * d, d), (d,)]            # mlp c_proj
    shapes += [(d,), (d,)]                      # ln_f
    return tuple(shapes)


def _loss_scaled_shapes(seed: int = 0) -> tuple:
    rng = np.random.Generator(np.random.PCG64(seed))
    u = rng.uniform(math.log(64.0), math.log(4096.0), size=10_000)
    small = [(int(math.floor(math.exp(x))),) for x in u]
    return tuple(small + [(768, 3072)] * 12)


WORKLOADS = {
    "tiny": Workload("tiny", ((384, 384), (384,), (384, 1536), (1536,)), g_std=1e-2),
    "gpt2_small": Workload("gpt2_small", _gpt2_shapes(768, 12), g_std=1e-3),
    "gpt2_small_bf16": Workload("gpt2_small_bf16", _gpt2_shapes(768, 12), moments="bf16x2", g_std=1e-3,
                                spike_p=0.01, spike_mult=100.0),
    "fp16_scaled": Workload("fp16_scaled", _loss_scaled_shapes(), grad_dtype="f16", g_std=1e-4,
                            loss_scale=65536.0),
    "gpt2_xl": Workload("gpt2_xl", _gpt2_shapes(1600, 48), moments="bf16x2", g_std=1e-4),
}


def _padded(n: int, elem_bytes: int) -> int:
    per = ALIGN_BYTES // elem_bytes
    return (n + per - 1) // per * per


def _layout(sizes, elem_bytes: int, packed: bool = False):
    """Offsets (in elements, or words when packed) of each tensor in its flat buffer, and the buffer's length."""
    offs, cur = [], 0
    for n in sizes:
        cnt = (n + 1) // 2 if packed else n
        offs.append(cur)
        cur += _padded(cnt, elem_bytes)
    return offs, max(cur, 1)


def _gen(device, seed: int) -> torch.Generator:
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed) & 0x7FFF_FFFF_FFFF_FFFF)
    return gen


def _mix(*xs: int) -> int:
    """A seed for one stream of one step, from the workload seed and small integers."""
    h = 0x9E3779B97F4A7C15
    for x in xs:
        h = ((h ^ (int(x) & 0xFFFFFFFFFFFFFFFF)) * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
        h ^= h >> 31
    return h & 0x7FFF_FFFF_FFFF_FFFF


@dataclass
class State:
    """A workload's buffers on one device: flat allocations and per-tensor views into them."""
    wl: Workload
    device: torch.device
    sizes: list
    w_flat: torch.Tensor
    g_flat: torch.Tensor
    m_flat: torch.Tensor
    v_flat: torch.Tensor
    w: list = field(default_factory=list)
    g: list = field(default_factory=list)
    m: list = field(default_factory=list)
    v: list = field(default_factory=list)

    @property
    def packed(self) -> bool:
        """Both moments packed."""
        return self.wl.moments == "bf16x2"

    @property
    def m_packed(self) -> bool:
        return self.wl.moments in ("bf16x2", "bf16x2_m")


def make_state(wl: Workload, device="cpu", sizes=None, seed: int | None = None) -> State:
    """Allocate a workload's buffers on ``device``: w drawn from N(0, w_std), m = v = 0, g = 0 (see ``fill_grad``).

    ``sizes`` overrides the workload's tensor sizes (for small parity cases with the same distributions)."""
    device = torch.device(device)
    sizes = list(wl.sizes if sizes is None else sizes)
    seed = wl.seed if seed is None else seed
    packed = wl.moments == "bf16x2"
    w_off, w_len = _layout(sizes, 4)
    g_es = 2 if wl.grad_dtype == "f16" else 4
    g_off, g_len = _layout(sizes, g_es)
    m_packed = wl.moments in ("bf16x2", "bf16x2_m")
    m_off, m_len = _layout(sizes, 4, packed=m_packed)
    v_off, v_len = _layout(sizes, 4, packed=packed)
    gdt = torch.float16 if wl.grad_dtype == "f16" else torch.float32
    mdt = torch.int32 if m_packed else torch.float32  # packed words are stored in int32 tensors (uint32 bits)
    vdt = torch.int32 if packed else torch.float32

    w_flat = torch.empty(w_len, dtype=torch.float32, device=device)
    w_flat.normal_(0.0, wl.w_std, generator=_gen(device, _mix(seed, 0xA)))
    g_flat = torch.zeros(g_len, dtype=gdt, device=device)
    m_flat = torch.zeros(m_len, dtype=mdt, device=device)
    v_flat = torch.zeros(v_len, dtype=vdt, device=device)
    st = State(wl, device, sizes, w_flat, g_flat, m_flat, v_flat)
    for n, wo, go, mo, vo in zip(sizes, w_off, g_off, m_off, v_off):
        st.w.append(w_flat[wo:wo + n])
        st.g.append(g_flat[go:go + n])
        st.m.append(m_flat[mo:mo + ((n + 1) // 2 if m_packed else n)])
        st.v.append(v_flat[vo:vo + ((n + 1) // 2 if packed else n)])
    return st


def fill_grad(st: State, t: int, seed: int | None = None) -> None:
    """Write step t's gradient into ``st.g`` (one draw over the flat buffer, seeded by (seed, t))."""
    wl = st.wl
    seed = wl.seed if seed is None else seed
    gen = _gen(st.device, _mix(seed, 0xB, t))
    n = st.g_flat.numel()
    if wl.grad_dtype == "f16":
        x = torch.randn(n, dtype=torch.float32, device=st.device, generator=gen)
        x.mul_(wl.g_std * wl.loss_scale)
        st.g_flat.copy_(x)  # float32 -> float16, nearest-even
        return
    st.g_flat.normal_(0.0, wl.g_std, generator=gen)
    if wl.spike_p > 0.0:
        u = torch.rand(n, dtype=torch.float32, device=st.device, generator=_gen(st.device, _mix(seed, 0xC, t)))
        st.g_flat.mul_(torch.where(u < wl.spike_p, wl.spike_mult, 1.0))


def host_lists(st: State):
    """numpy copies of the per-tensor views, in the dtypes the oracle takes (packed words as uint32)."""
    def conv(t: torch.Tensor) -> np.ndarray:
        a = t.detach().cpu().numpy()
        return a.view(np.uint32) if a.dtype == np.int32 else a.copy()
    return ([conv(x) for x in st.w], [conv(x) for x in st.g], [conv(x) for x in st.m], [conv(x) for x in st.v])
