"""GPU checks of plsh_bias_error against the oracle: the exact max-norm error
and the Lanczos spectral estimate against the dense fp64 oracle on small n,
the closed forms of all-singleton bins, and the O(1/sqrt(s)) decay at
n = 16384."""
import math

import numpy as np
import pytest
import torch

import oracle
import positional_lsh_approximation_gb300 as plsh

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    plsh.build()
    plsh.load()


@pytest.mark.parametrize("n,sigma,s", [(300, 8.0, 4), (1500, 40.0, 10), (1000, 2.0, 16),
                                       (4097, 120.0, 6), (64, 1e4, 3)])
def test_bias_error_matches_dense_oracle(n, sigma, s):
    b = plsh.sample_bins(n, [sigma, 3.0], s, seed=5)
    off, st = oracle.sample_bins(n, [sigma, 3.0], s, seed=5)
    e_max, e_spec = oracle.bias_error(n, sigma, off, st, 0, s)
    g_max, g_spec = plsh.bias_error(b, sigma, 0, lanczos_iters=80, seed=1)
    assert abs(g_max - e_max) <= 1e-11 * max(1.0, e_max)
    assert abs(g_spec - e_spec) <= 1e-8 * e_spec
    b.free()


def test_bias_error_singletons_closed_form():
    n, sigma, s = 20000, 8.0, 3
    off = np.arange(0, s * (n + 1) + 1, n + 1, dtype=np.int64)
    st = np.tile(np.arange(n + 1, dtype=np.int32), s)
    b = plsh.bins_from_host(n, 1, s, off, st)
    g_max, g_spec = plsh.bias_error(b, sigma, 0, lanczos_iters=120, seed=2)
    assert abs(g_max - math.exp(-1.0 / sigma)) < 1e-12
    assert abs(g_spec / (1.0 / math.tanh(0.5 / sigma) - 1.0) - 1.0) < 1e-3
    b.free()


def test_bias_error_decays_as_inverse_sqrt_s():
    n, sigma = 16384, 32.0
    ss = [1, 4, 16, 64]
    spec = []
    for s in ss:
        b = plsh.sample_bins(n, [sigma], s, seed=11)
        spec.append(plsh.bias_error(b, sigma, 0, lanczos_iters=60, seed=3)[1])
        b.free()
    slope = np.polyfit(np.log(ss), np.log(spec), 1)[0]
    assert -0.65 < slope < -0.35, slope
