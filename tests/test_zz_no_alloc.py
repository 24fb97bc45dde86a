"""The allocation-free attention entry point agrees with plsh_alibi_attn.

Collected last on purpose: if it fails, a run that stops at the first failure
has already run every other test.  Calls go through the C ABI with ctypes;
the reference is the ordinary entry point on the same inputs and bins.
"""
import ctypes

import numpy as np
import pytest
import torch

import positional_lsh_approximation_gb300 as plsh
from positional_lsh_approximation_gb300.inputs import WORKLOADS, make_qkv

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-3, 1e-2   # the bf16 tolerance of the parity tests


def _desc(t):
    B, H, n, d = t.shape
    return plsh._Tensor(t.data_ptr(), plsh.PLSH_BF16, B, H, n, d)


def _call(fn, q, k, v, bins, causal, out):
    tq, tk, tv, to = _desc(q), _desc(k), _desc(v), _desc(out)
    st = fn(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv), bins.handle,
            int(causal), ctypes.byref(to), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == plsh.PLSH_OK, plsh.load().plsh_last_error().decode()


@pytest.mark.parametrize("name,n", [("mistral", 2048), ("scout", 4096)])
def test_noalloc_matches_attn_twice(name, n):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    plsh.build()
    lib = plsh.load()
    w = WORKLOADS[name].with_(n=n)
    Q, K, V = make_qkv(w)
    q, k, v = (torch.from_numpy(x).to(torch.bfloat16).cuda() for x in (Q, K, V))
    bins = plsh.sample_bins(w.n, w.sigmas(), w.s, w.hash_seed)
    ref = torch.empty_like(q)
    _call(lib.plsh_alibi_attn, q, k, v, bins, w.causal, ref)
    plsh.stream_status()
    refd = ref.float().cpu().numpy()
    for _ in range(2):
        out = torch.full_like(q, float("nan"))
        _call(lib.plsh_alibi_attn_noalloc, q, k, v, bins, w.causal, out)
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        assert not np.isnan(got).any()
        assert np.all(np.abs(got - refd) <= ATOL + RTOL * np.abs(refd))


def test_noalloc_rejects_oversized_requests():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = plsh.load()
    # 65536 work items is the limit: 2 heads x 2 * 65536 row tiles exceed it
    n = 128 * 65537
    T = plsh._Tensor
    q = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    big = T(q.data_ptr(), plsh.PLSH_BF16, 1, 2, n, 128)
    bins = plsh.sample_bins(n, [4.0, 4.0], 2, 0)
    st = lib.plsh_alibi_attn_noalloc(ctypes.byref(big), ctypes.byref(big), ctypes.byref(big),
                                     bins.handle, 1, ctypes.byref(big), None)
    assert st == plsh.PLSH_ERR_UNSUPPORTED
    assert b"work items" in lib.plsh_last_error()


def test_noalloc_timeout_is_reported_and_next_call_agrees(monkeypatch):
    """A device-side wait of the allocation-free path that runs out is kept in
    the fixed array's error word (the call itself cannot see it) and reported
    by plsh_noalloc_status, which clears it; plsh_set_wait_limit_ns applies to
    this path, and the next call agrees with plsh_alibi_attn."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = plsh.load()
    w = WORKLOADS["mistral"].with_(n=1024)
    Q, K, V = make_qkv(w)
    q, k, v = (torch.from_numpy(x).to(torch.bfloat16).cuda() for x in (Q, K, V))
    bins = plsh.sample_bins(w.n, w.sigmas(), w.s, w.hash_seed)
    ref = torch.empty_like(q)
    _call(lib.plsh_alibi_attn, q, k, v, bins, w.causal, ref)
    plsh.stream_status()
    plsh.noalloc_status()                       # nothing pending
    plsh.set_wait_limit_ns(20_000_000)         # 20 ms per wait
    try:
        monkeypatch.setenv("PLSH_FAULT", "stall")
        out = torch.zeros_like(q)
        _call(lib.plsh_alibi_attn_noalloc, q, k, v, bins, w.causal, out)
        with pytest.raises(plsh.PlshError) as err:
            plsh.noalloc_status()
        assert err.value.status == plsh.PLSH_ERR_TIMEOUT
        plsh.noalloc_status()                   # cleared by the report
        plsh.stream_status()                    # the library's own flag is untouched
    finally:
        monkeypatch.delenv("PLSH_FAULT", raising=False)
        plsh.set_wait_limit_ns(0)
    again = torch.full_like(q, float("nan"))
    _call(lib.plsh_alibi_attn_noalloc, q, k, v, bins, w.causal, again)
    plsh.noalloc_status()
    refd = ref.float().cpu().numpy()
    got = again.float().cpu().numpy()
    assert np.all(np.abs(got - refd) <= ATOL + RTOL * np.abs(refd))
    bins.free()
