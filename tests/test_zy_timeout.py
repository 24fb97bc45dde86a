"""Failure detection without a GPU fault: a device-side wait that runs out.

PLSH_FAULT=stall makes the tensor-core kernel's scheduler publish no work
item, so every other warp waits on an mbarrier that nothing will complete.
Each wait gives up after the library's wait limit (shortened here), the
kernel records the timeout in the device error flag and exits with no copy
or MMA in flight; the host reads PLSH_ERR_TIMEOUT at the next
plsh_stream_status, and the next call on the same context works.
"""
import numpy as np
import pytest
import torch

import positional_lsh_approximation_gb300 as plsh
from positional_lsh_approximation_gb300.inputs import Workload, make_qkv

pytestmark = pytest.mark.gpu


def test_stalled_kernel_reports_timeout_and_context_recovers(monkeypatch):
    plsh.build()
    w = Workload("timeout", 1, 2, 1, 512, 128, "bf16", True, 6, (2.0, 40.0), qkv_seed=77)
    Q, K, V = make_qkv(w)
    q, k, v = (torch.from_numpy(x).to(torch.bfloat16).cuda() for x in (Q, K, V))
    bins = plsh.sample_bins(w.n, w.sigmas(), w.s, seed=5)
    ref = plsh.alibi_attn(q, k, v, bins, True)
    plsh.stream_status()

    plsh.set_wait_limit_ns(20_000_000)         # 20 ms per wait
    try:
        monkeypatch.setenv("PLSH_FAULT", "stall")
        out = torch.zeros_like(ref)
        plsh.alibi_attn(q, k, v, bins, True, out=out)
        with pytest.raises(plsh.PlshError) as err:
            plsh.stream_status()
        assert err.value.status == plsh.PLSH_ERR_TIMEOUT
        # the flag was cleared by the report
        plsh.stream_status()
    finally:
        monkeypatch.delenv("PLSH_FAULT", raising=False)
        plsh.set_wait_limit_ns(0)

    again = plsh.alibi_attn(q, k, v, bins, True)
    plsh.stream_status()
    assert torch.equal(again, ref)
    bins.free()


def test_injected_allocation_failure_is_reported(monkeypatch):
    plsh.build()
    sigma = np.array([3.0, 30.0])
    monkeypatch.setenv("PLSH_FAULT", "oom")
    with pytest.raises(plsh.PlshError) as err:
        plsh.sample_bins(1000, sigma, 4, seed=1)
    assert err.value.status == plsh.PLSH_ERR_NOMEM
    monkeypatch.delenv("PLSH_FAULT")
    bins = plsh.sample_bins(1000, sigma, 4, seed=1)
    assert bins.shape() == (1000, 2, 4)
    bins.free()
