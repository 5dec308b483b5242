"""Failure detection without a GPU fault: a kernel's bounded wait that runs out is reported by mica_sync, once, and
the context stays usable (the self-test kernel waits on a barrier that nothing arrives at)."""
import time

import pytest
import torch

import clip_tensor_adamw_gb300 as mica
import parity
import workloads

pytestmark = pytest.mark.gpu

OK, HYPER, CUDA = 0, 4, 9


def test_bounded_wait_runs_out_and_is_reported():
    L = mica.lib()
    stream = torch.cuda.current_stream().cuda_stream
    assert L.mica_sync(stream) == OK  # nothing pending
    t0 = time.perf_counter()
    assert L.mica_selftest_wait_timeout(16, stream) == OK
    assert L.mica_sync(stream) == CUDA
    elapsed = time.perf_counter() - t0
    detail = L.mica_last_error_detail().decode()
    assert "gave up" in detail and "0x4" in detail, detail
    assert L.mica_sync(stream) == OK  # read once, then cleared
    mica.mica_selftest_wait_timeout(16)
    with pytest.raises(mica.MicaError, match="MICA_ERR_CUDA"):
        mica.mica_sync()
    mica.mica_sync()
    print(f"16 polls gave up after {elapsed * 1e3:.2f} ms")
    # the context still works: a clip + AdamW step still matches the oracle bit for bit
    r = parity.run_parity(workloads.WORKLOADS["tiny"], steps=2)
    assert r["same_factor_every_step"]


def test_selftest_arguments_checked_on_the_host():
    L = mica.lib()
    assert L.mica_selftest_wait_timeout(0, None) == HYPER
    assert L.mica_selftest_wait_timeout((1 << 20) + 1, None) == HYPER
