"""GPU checks of plsh_alibi_attn_backward against the oracle's gradients.
fp32 inputs: 1e-4 relative to the largest gradient entry; bf16 inputs: the
gradients are rounded to bf16, 1e-2 of that scale.  bf16 with d = 128 and
s <= 16 runs on the tensor cores (P and dS in bf16), everything else on the
CUDA cores."""
import numpy as np
import pytest
import torch

import oracle
import positional_lsh_approximation_gb300 as plsh
from positional_lsh_approximation_gb300.inputs import Workload, make_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    plsh.build()
    plsh.load()


CASES = [
    # name, B, Hq, Hkv, n, d, dtype, causal, s, sigma
    ("f32_causal_gqa", 2, 4, 2, 260, 128, "f32", True, 5, (0.7, 3.0, 20.0, 90.0)),
    ("f32_noncausal", 1, 2, 1, 300, 64, "f32", False, 6, (2.0, 40.0)),
    ("bf16_causal", 1, 4, 2, 400, 128, "bf16", True, 10, (1.2, 6.0, 40.0, 300.0)),
    ("bf16_noncausal_d64", 1, 2, 2, 333, 64, "bf16", False, 4, (5.0, 60.0)),
    # tensor-core path: several key tiles, ragged tails, GQA, s = 16
    ("tc_noncausal", 2, 4, 1, 520, 128, "bf16", False, 6, (3.0, 25.0, 150.0, 900.0)),
    ("tc_causal_gqa4", 1, 8, 2, 1000, 128, "bf16", True, 10,
     (1.2, 6.0, 40.0, 300.0, 2.0, 9.0, 70.0, 500.0)),
    ("tc_causal_s16", 1, 2, 1, 700, 128, "bf16", True, 16, (4.0, 120.0)),
    ("tc_one_tile", 1, 2, 2, 100, 128, "bf16", True, 3, (2.0, 1e4)),
    # every register-slot variant of the kernel (s <= 4, 8, 10, 12, 16), and
    # sigma far below one position, where many bins of a key end on one row
    ("tc_noncausal_s3", 1, 2, 2, 260, 128, "bf16", False, 3, (1.5, 30.0)),
    ("tc_noncausal_s10", 1, 2, 1, 390, 128, "bf16", False, 10, (0.9, 45.0)),
    ("tc_causal_s12", 1, 4, 2, 450, 128, "bf16", True, 12, (0.6, 5.0, 30.0, 200.0)),
    ("tc_noncausal_s12", 1, 2, 1, 300, 128, "bf16", False, 12, (2.5, 70.0)),
    ("tc_noncausal_s16", 1, 2, 2, 280, 128, "bf16", False, 16, (0.4, 12.0)),
    ("tc_causal_tiny_sigma", 1, 2, 1, 300, 128, "bf16", True, 16, (0.3, 0.8)),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_backward_matches_oracle(case):
    name, B, Hq, Hkv, n, d, dtype, causal, s, sig = case
    w = Workload(name, B, Hq, Hkv, n, d, dtype, causal, s, sig, qkv_seed=n + d)
    Q, K, V = make_qkv(w)
    rng = np.random.default_rng(n)
    dO = rng.standard_normal(Q.shape).astype(np.float32)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    if dtype == "bf16":
        dO = torch.from_numpy(dO).to(tdt).float().numpy()
    bins = plsh.sample_bins(n, w.sigmas(), s, seed=6)
    off, st = oracle.sample_bins(n, w.sigmas(), s, seed=6)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(tdt).cuda()
    dQ, dK, dV = plsh.alibi_attn_backward(dev(Q), dev(K), dev(V), dev(dO), bins, causal)
    plsh.stream_status()
    ref = oracle.plsh_attn_backward(Q, K, V, dO, off, st, s, causal)
    rel = 1e-4 if dtype == "f32" else 1e-2
    for got, want, what in zip((dQ, dK, dV), ref, ("dQ", "dK", "dV")):
        g = got.float().cpu().numpy().astype(np.float64)
        scale = np.abs(want).max()
        err = np.abs(g - want).max()
        assert err <= rel * scale, f"{name} {what}: max err {err:.3e} vs scale {scale:.3e}"
    bins.free()


def test_tensor_core_backward_agrees_with_cuda_cores(monkeypatch):
    """The same gradients from both kernels (bf16 outputs), a causal GQA case
    over several key tiles."""
    w = Workload("agree", 1, 4, 2, 600, 128, "bf16", True, 8, (2.0, 10.0, 60.0, 400.0),
                 qkv_seed=77)
    Q, K, V = make_qkv(w)
    dO = np.random.default_rng(5).standard_normal(Q.shape).astype(np.float32)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).cuda()
    bins = plsh.sample_bins(w.n, w.sigmas(), w.s, seed=4)
    tc = plsh.alibi_attn_backward(dev(Q), dev(K), dev(V), dev(dO), bins, True)
    plsh.stream_status()
    monkeypatch.setenv("PLSH_PATH", "simt")
    simt = plsh.alibi_attn_backward(dev(Q), dev(K), dev(V), dev(dO), bins, True)
    plsh.stream_status()
    for a, b, what in zip(tc, simt, ("dQ", "dK", "dV")):
        a = a.float().cpu().numpy()
        b = b.float().cpu().numpy()
        scale = np.abs(b).max()
        assert np.abs(a - b).max() <= 1.5e-2 * scale, what
    bins.free()


LSE_CASES = [
    # name, B, Hq, Hkv, n, causal, s, sigma, split parts
    ("causal_gqa", 1, 4, 2, 700, True, 10, (1.5, 8.0, 60.0, 400.0), 0),
    ("noncausal", 2, 2, 1, 390, False, 6, (3.0, 90.0), 0),
    ("causal_split3", 1, 2, 1, 900, True, 8, (300.0, 2000.0), 3),
]


def _lse_inputs(case):
    name, B, Hq, Hkv, n, causal, s, sig, parts = case
    w = Workload(name, B, Hq, Hkv, n, 128, "bf16", causal, s, sig, qkv_seed=n + 11)
    Q, K, V = make_qkv(w)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).cuda()
    return w, Q, K, V, dev


@pytest.mark.parametrize("case", LSE_CASES, ids=[c[0] for c in LSE_CASES])
def test_forward_lse_matches_oracle(case):
    """O from plsh_alibi_attn_lse is the O of plsh_alibi_attn, bit for bit,
    and lse_i = log2 of the oracle's unshifted row sum sum_j c_ij e^{S_ij}."""
    w, Q, K, V, dev = _lse_inputs(case)
    parts = case[-1]
    bins = plsh.sample_bins(w.n, w.sigmas(), w.s, seed=3)
    off, st = oracle.sample_bins(w.n, w.sigmas(), w.s, seed=3)
    plsh.set_split_parts(parts)
    try:
        O, lse = plsh.alibi_attn_lse(dev(Q), dev(K), dev(V), bins, w.causal)
        O2 = plsh.alibi_attn(dev(Q), dev(K), dev(V), bins, w.causal)
        plsh.stream_status()
    finally:
        plsh.set_split_parts(0)
    assert torch.equal(O, O2)
    rows = oracle.all_rows(w.B, w.Hq, w.n)
    _, den = oracle.plsh_parts_rows(Q, K, V, off, st, w.s, w.causal, rows)
    want = np.log2(den)
    got = lse.cpu().numpy().astype(np.float64)
    err = np.abs(got - want).max()
    assert err <= 2e-3, f"{case[0]}: lse max err {err:.3e}"
    bins.free()


@pytest.mark.parametrize("case", LSE_CASES[:2], ids=[c[0] for c in LSE_CASES[:2]])
def test_backward_from_saved_lse_matches_oracle(case):
    """Gradients from the forward's O and lse against the oracle's, and
    against the recomputing backward pass."""
    w, Q, K, V, dev = _lse_inputs(case)
    dO = np.random.default_rng(w.n).standard_normal(Q.shape).astype(np.float32)
    dO = torch.from_numpy(dO).to(torch.bfloat16).float().numpy()
    bins = plsh.sample_bins(w.n, w.sigmas(), w.s, seed=3)
    off, st = oracle.sample_bins(w.n, w.sigmas(), w.s, seed=3)
    q, k, v, do = dev(Q), dev(K), dev(V), dev(dO)
    O, lse = plsh.alibi_attn_lse(q, k, v, bins, w.causal)
    saved = plsh.alibi_attn_backward_lse(q, k, v, O, lse, do, bins, w.causal)
    recomputed = plsh.alibi_attn_backward(q, k, v, do, bins, w.causal)
    plsh.stream_status()
    ref = oracle.plsh_attn_backward(Q, K, V, dO, off, st, w.s, w.causal)
    for got, again, want, what in zip(saved, recomputed, ref, ("dQ", "dK", "dV")):
        g = got.float().cpu().numpy().astype(np.float64)
        scale = np.abs(want).max()
        assert np.abs(g - want).max() <= 1e-2 * scale, f"{case[0]} {what} vs oracle"
        assert np.abs(g - again.float().cpu().numpy()).max() <= 1e-2 * scale, f"{case[0]} {what}"
    bins.free()
