"""The step captured once into a CUDA graph and replayed: the library's calls are stream work only (once a list's
table exists), so a captured clip + AdamW step replays with the same results as the oracle's step, and a replayed
step takes its parameters' new values from device memory each time."""
import numpy as np
import pytest
import torch

import clip_tensor_adamw_gb300 as mica
import parity
import workloads

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("entry", ["separate", "one_step"])
def test_captured_step_replays(ora, entry, monkeypatch):
    """The norm and the update captured as two calls, or as the one call of mica_clip_adamw_step (its default
    path: the same two launches)."""
    monkeypatch.delenv("MICA_FUSED", raising=False)
    wl = workloads.WORKLOADS["gpt2_small"]
    sizes = [int(np.prod(s)) for s in workloads._gpt2_shapes(90, 2, 1003, 67)]
    st = workloads.make_state(wl, "cuda", sizes=sizes)
    W, G, M, V = parity.tensor_lists(st)
    norm = torch.empty(1, device="cuda")
    factor = torch.empty(1, device="cuda")
    t_fixed = 5  # the step count is a host scalar, captured with the graph
    kw = dict(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps, weight_decay=wl.weight_decay, step=t_fixed,
              factor=factor)
    # tables built (and the scalar outputs checked) outside the capture
    workloads.fill_grad(st, 1)
    host = workloads.host_lists(st)
    mica.mica_clip_grad_norms(G, wl.max_norm, wl.inv_scale, norm_out=norm, factor_out=factor)
    mica.mica_adamw_steps(W, G, M, V, **kw)
    if entry == "one_step":  # its scalar-output check (norm and factor together) also happens once, outside
        mica.mica_clip_adamw_step(W, G, M, V, max_norm=wl.max_norm, inv_scale=wl.inv_scale, norm_out=norm,
                                  factor_out=factor, **{k: v for k, v in kw.items() if k != "factor"})
        ora.clip_adamw_step(*host, parity.hp_of(wl, t_fixed), wl.max_norm, wl.inv_scale)
    hp = parity.hp_of(wl, t_fixed)
    ora.clip_adamw_step(*host, hp, wl.max_norm, wl.inv_scale)
    torch.cuda.synchronize()

    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        graph.capture_begin()
        if entry == "separate":
            mica.mica_clip_grad_norms(G, wl.max_norm, wl.inv_scale, norm_out=norm, factor_out=factor, stream=stream)
            mica.mica_adamw_steps(W, G, M, V, stream=stream, **kw)
        else:
            one = {k: v for k, v in kw.items() if k != "factor"}
            mica.mica_clip_adamw_step(W, G, M, V, max_norm=wl.max_norm, inv_scale=wl.inv_scale, norm_out=norm,
                                      factor_out=factor, stream=stream, **one)
        graph.capture_end()
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()
    for t in range(2, 6):
        workloads.fill_grad(st, t)
        g_host = [x.copy() for x in workloads.host_lists(st)[1]]
        host = (host[0], g_host, host[2], host[3])
        graph.replay()
        o_norm, o_factor = ora.clip_adamw_step(*host, hp, wl.max_norm, wl.inv_scale)
        torch.cuda.synchronize()
        assert abs(norm.item() - float(o_norm)) <= parity.NORM_RTOL * float(o_norm)
        same = np.float32(factor.item()).view(np.uint32) == o_factor.view(np.uint32)
        parity.compare_state(st, host, bool(same), f"graph replay {t}")
    mica.mica_sync()
