"""The register-streaming norm on lists whose CTA chunks span more than 256 tensors.

That kernel stages the records of 256 tensors at a time in shared memory. A thread whose float32-pair sum cannot
hold its share exactly (an infinity, a NaN, a value of 2^50 or more) sums the share again in double; both passes
must take the same octets of the chunk however many staged spans it has. The list here has 4,096 tensors, three of
every four empty and the fourth one octet long: the norm's 4 CTAs each take 256 octets over 1,024 tensors, four
spans, and the value planted in the first octet of a later span is summed by the thread whose re-sum covers it.
Against the oracle (ClipGradNorms, "Mica 7.7", section "The whole model in one call").
"""
import numpy as np
import pytest
import torch

import clip_tensor_adamw_gb300 as mica

pytestmark = pytest.mark.gpu

NORM_RTOL = 1e-5


def spanning_list(values, at):
    """4,096 float32 tensors (every fourth of 8 elements, the others empty), g ~ N(0, 1e-3), and `values` written
    from element 0 of the non-empty tensors numbered `at` (one value each)."""
    rng = np.random.Generator(np.random.PCG64(5))
    sizes = [8 if k % 4 == 3 else 0 for k in range(4096)]
    host = [rng.normal(0, 1e-3, size=n).astype(np.float32) for n in sizes]
    nonempty = [k for k, n in enumerate(sizes) if n]
    for v, j in zip(values, at):
        host[nonempty[j]][0] = v
    flat = torch.from_numpy(np.concatenate(host)).cuda()
    dev, off = [], 0
    for n in sizes:
        dev.append(flat[off:off + n] if n else torch.empty(0, device="cuda"))
        off += n
    return host, dev, flat


CASES = [([float("inf")], [64]), ([float("nan")], [64]), ([-float("inf")], [200]), ([1e30], [64]),
         ([1e30, -3e25], [64, 130]), ([2.0 ** 60], [255])]


@pytest.mark.parametrize("values,at", CASES, ids=["inf", "nan", "neg_inf_late", "huge", "two_huge", "pow2_60_last"])
@pytest.mark.parametrize("inv_scale", [1.0, 0.5])
def test_norm_over_many_staged_spans(ora, values, at, inv_scale):
    host, dev, _ = spanning_list(values, at)
    o_norm, o_factor, _ = ora.clip_grad_norms(host, 1.0, inv_scale)
    norm, factor = mica.mica_clip_grad_norms(dev, 1.0, inv_scale)
    torch.cuda.synchronize()
    g_norm, g_factor = np.float32(norm.item()), np.float32(factor.item())
    if np.isnan(o_norm):
        assert np.isnan(g_norm) and np.isnan(g_factor)
    elif np.isinf(o_norm):
        assert np.isinf(g_norm) and g_factor == o_factor == 0.0
    else:
        assert abs(float(g_norm) - float(o_norm)) <= NORM_RTOL * float(o_norm), (g_norm, o_norm)
        assert g_factor.view(np.uint32) == o_factor.view(np.uint32), (g_factor, o_factor)


def test_finite_norm_over_many_staged_spans(ora):
    """No planted value: every share is summed in float32 pairs, across four spans per CTA."""
    host, dev, _ = spanning_list([], [])
    o_norm, o_factor, _ = ora.clip_grad_norms(host, 1e-3)
    norm, factor = mica.mica_clip_grad_norms(dev, 1e-3)
    torch.cuda.synchronize()
    assert abs(norm.item() - float(o_norm)) <= NORM_RTOL * float(o_norm)
    assert np.float32(factor.item()).view(np.uint32) == o_factor.view(np.uint32)
