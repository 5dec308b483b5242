"""The library's cache of per-list device tables: it holds at most 1,024 tables and, when full, frees those that no
call in progress holds. mica_clip_adamw_step looks up its update's table and then its norm's; with the cache one
table short of full, the norm's new table makes it evict while the call still holds the update's, which must
survive: the step is checked against the oracle bit for bit, and the cache keeps working afterwards."""
import numpy as np
import pytest
import torch

import clip_tensor_adamw_gb300 as mica
import parity
import workloads

pytestmark = pytest.mark.gpu

MAX_TABLES = 1024


def _fill_cache(count, buf, f):
    """`count` distinct one-tensor lists, one new table each."""
    for i in range(count):
        mica.mica_clip_grad_norms([buf[8 * i:8 * i + 8]], 1.0, factor_out=f)


@pytest.mark.parametrize("fused", ["0", "1"])
def test_eviction_keeps_the_tables_a_call_holds(ora, fused, monkeypatch):
    monkeypatch.setenv("MICA_FUSED", fused)
    wl = workloads.WORKLOADS["gpt2_small_bf16"]
    sizes = [4096, 333, 64, 7]
    st = workloads.make_state(wl, "cuda", sizes=sizes)
    W, G = mica.TensorList(st.w), mica.TensorList(st.g)
    M, V = mica.TensorList(st.m, W.counts), mica.TensorList(st.v, W.counts)
    buf = torch.ones(8 * MAX_TABLES, device="cuda")
    f = torch.zeros(1, device="cuda")
    kw = dict(max_norm=wl.max_norm, inv_scale=wl.inv_scale, lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps,
              weight_decay=wl.weight_decay)
    host = workloads.host_lists(st)
    mica.mica_release_cache()
    for t in (1, 2):
        workloads.fill_grad(st, t)
        host = (host[0], [x.detach().cpu().numpy().copy() for x in st.g], host[2], host[3])
        if t == 1:
            _fill_cache(MAX_TABLES - 1, buf, f)  # the step's update table is the 1,024th; its norm's evicts
        norm, factor = mica.mica_clip_adamw_step(W, G, M, V, step=t, **kw)
        o_norm, o_factor = ora.clip_adamw_step(*host, parity.hp_of(wl, t), wl.max_norm, wl.inv_scale)
        torch.cuda.synchronize()
        parity.check_norm(np.float32(norm.item()), o_norm, t)
        same = np.float32(factor.item()).view(np.uint32) == o_factor.view(np.uint32)
        parity.compare_state(st, host, bool(same), f"after eviction, step {t}")
    # the evicted lists still work (their tables are built again)
    _fill_cache(3, buf, f)
    torch.cuda.synchronize()
    assert f.item() == pytest.approx(1.0 / (np.sqrt(8.0) + 1e-6), rel=1e-6)
    mica.mica_release_cache()
