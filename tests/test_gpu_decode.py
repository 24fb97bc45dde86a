"""Decode step (plsh_alibi_decode) vs the fp64 oracle, through the C ABI.

A decode step is row `pos` of the approximation with the causal mask
(Methodology 3): the oracle evaluates exactly that row, per sample and per
bin, from a query tensor that holds the decode query at row `pos`.
Tolerances as for the full attention: bf16 atol 2e-3, rtol 1e-2; fp32 1e-5.
"""
import numpy as np
import pytest
import torch

import oracle
import positional_lsh_approximation_gb300 as plsh
from positional_lsh_approximation_gb300.inputs import Workload, make_qkv

pytestmark = pytest.mark.gpu

TOL = {"bf16": (2e-3, 1e-2), "f32": (1e-5, 1e-5)}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    plsh.build()
    plsh.load()


def to_dev(x, dtype):
    t = torch.from_numpy(np.ascontiguousarray(x))
    return (t.to(torch.bfloat16) if dtype == "bf16" else t).cuda()


def check(got, ref, dtype, what):
    atol, rtol = TOL[dtype]
    err = np.abs(got - ref)
    assert not np.isnan(got).any(), f"{what}: NaN"
    bad = err > atol + rtol * np.abs(ref)
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} out of tolerance, "
                           f"max err {err.max():.3e}")


def decode_vs_oracle(w: Workload, positions, seed=3):
    Q, K, V = make_qkv(w)
    sigma = w.sigmas()
    bins = plsh.sample_bins(w.n, sigma, w.s, seed=seed)
    off, st = oracle.sample_bins(w.n, sigma, w.s, seed=seed)
    k, v = to_dev(K, w.dtype), to_dev(V, w.dtype)
    for pos in positions:
        q = to_dev(Q[:, :, pos:pos + 1, :], w.dtype)
        o = plsh.alibi_decode(q, k, v, bins, pos)
        plsh.stream_status()
        got = o.float().cpu().numpy().astype(np.float64)[:, :, 0, :]
        bb, hh = np.meshgrid(np.arange(w.B), np.arange(w.Hq), indexing="ij")
        rows = (bb.ravel(), hh.ravel(), np.full(bb.size, pos))
        ref = oracle.plsh_attn_rows(Q, K, V, off, st, w.s, True, rows)
        check(got.reshape(-1, w.d), ref, w.dtype, f"{w.name} pos={pos}")
    bins.free()


CASES = [
    # name, B, Hq, Hkv, n, d, dtype, s, sigma, positions
    ("bf16_gqa", 2, 8, 2, 3000, 128, "bf16", 10, (), [2999, 1234, 0, 511, 512, 1023]),
    ("bf16_d64", 1, 4, 1, 1500, 64, "bf16", 6, (2.0, 20.0, 200.0, 2000.0), [1499, 700]),
    ("f32", 2, 2, 2, 1200, 128, "f32", 5, (3.0, 300.0), [1199, 5]),
    ("f32_d64_s64", 1, 2, 1, 800, 64, "f32", 64, (1.5, 40.0), [799, 300]),
    # one bin over the whole prefix: the envelope spans five 512-key chunks
    ("bf16_one_bin", 1, 2, 1, 2100, 128, "bf16", 3, (1e5, 1e5), [2099, 1536]),
    # three heads per KV group (two warps each, two idle), and twelve (two
    # CTAs per group: eight heads and four)
    ("bf16_g3", 2, 3, 1, 900, 128, "bf16", 4, (5.0, 60.0, 500.0), [899, 450, 63, 64]),
    ("bf16_g12", 1, 24, 2, 700, 128, "bf16", 5, (), [699, 100]),
    # grids of at least four CTAs per SM take the 8 KB stages (d = 128: 32
    # keys a block; d = 64: 64)
    ("bf16_many", 24, 8, 8, 1200, 128, "bf16", 10, (), [1199, 600]),
    ("bf16_d64_many", 32, 8, 4, 900, 64, "bf16", 6, (), [899, 64]),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_decode_matches_oracle(case):
    name, B, Hq, Hkv, n, d, dtype, s, sig, positions = case
    w = Workload(name, B, Hq, Hkv, n, d, dtype, True, s, sig, qkv_seed=n + d)
    decode_vs_oracle(w, positions)


def test_decode_singletons_return_the_value_row():
    """Bins of width one under every hash: the row's only key is pos."""
    n, d, s = 700, 128, 4
    w = Workload("single", 1, 2, 1, n, d, "bf16", True, s, (1.0,), qkv_seed=5)
    Q, K, V = make_qkv(w)
    off = np.arange(0, 2 * s * (n + 1) + 1, n + 1, dtype=np.int64)
    st = np.tile(np.arange(n + 1, dtype=np.int32), 2 * s)
    bins = plsh.bins_from_host(n, 2, s, off, st)
    k, v = to_dev(K, "bf16"), to_dev(V, "bf16")
    for pos in (0, 333, n - 1):
        o = plsh.alibi_decode(to_dev(Q[:, :, pos:pos + 1], "bf16"), k, v, bins, pos)
        plsh.stream_status()
        got = o.float().cpu().numpy()[0, :, 0, :]
        np.testing.assert_array_equal(got, np.stack([V[0, 0, pos], V[0, 0, pos]]))
    bins.free()


def test_decode_agrees_with_the_full_kernel_row():
    """The decode step and row pos of plsh_alibi_attn are the same row of T~."""
    w = Workload("rowcheck", 1, 4, 2, 2048, 128, "bf16", True, 10, (), qkv_seed=17)
    Q, K, V = make_qkv(w)
    bins = plsh.sample_bins(w.n, w.sigmas(), w.s, seed=1)
    q, k, v = to_dev(Q, "bf16"), to_dev(K, "bf16"), to_dev(V, "bf16")
    full = plsh.alibi_attn(q, k, v, bins, True).float().cpu().numpy()
    for pos in (2047, 1000, 77):
        o = plsh.alibi_decode(q[:, :, pos:pos + 1].contiguous(), k, v, bins, pos)
        plsh.stream_status()
        got = o.float().cpu().numpy()[:, :, 0, :]
        np.testing.assert_allclose(got, full[:, :, pos, :], atol=4e-3, rtol=2e-2)
    bins.free()


def test_decode_rejects_bad_arguments():
    w = Workload("bad", 1, 2, 1, 256, 128, "bf16", True, 4, (8.0,), qkv_seed=1)
    Q, K, V = make_qkv(w)
    bins = plsh.sample_bins(w.n, w.sigmas(), w.s, seed=0)
    k, v = to_dev(K, "bf16"), to_dev(V, "bf16")
    q = to_dev(Q[:, :, :1], "bf16")
    for pos in (-1, 256):
        with pytest.raises(plsh.PlshError) as err:
            plsh.alibi_decode(q, k, v, bins, pos)
        assert err.value.status == plsh.PLSH_ERR_INVALID
    with pytest.raises(plsh.PlshError):
        plsh.alibi_decode(to_dev(Q[:, :, :2], "bf16"), k, v, bins, 10)   # q has two rows
    bins.free()
