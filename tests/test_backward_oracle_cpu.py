"""Pins of the oracle's gradients of the approximation (the backward pass of
Methodology 3's estimator), independent of the formula they check: central
differences of the oracle's own forward rows, and autograd of plain softmax
attention in the case the estimator reduces to it."""
import math

import numpy as np
import pytest
import torch

import oracle


def quantised(rng, shape):
    # multiples of 2^-8 below 2: perturbing by 2^-8 or 2^-9 stays exact in fp32
    return rng.integers(-256, 256, size=shape).astype(np.float64) / 256.0


def forward_loss(Q, K, V, dO, off, st, s, causal):
    B, Hq, n, d = Q.shape
    O = oracle.plsh_attn_rows(Q, K, V, off, st, s, causal, oracle.all_rows(B, Hq, n))
    return float((O.reshape(B, Hq, n, d) * dO).sum())


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "noncausal"])
def test_gradients_match_central_differences(causal):
    rng = np.random.default_rng(7 if causal else 8)
    B, Hq, Hkv, n, d, s = 1, 2, 1, 20, 8, 3
    Q, K, V = quantised(rng, (B, Hq, n, d)), quantised(rng, (B, Hkv, n, d)), quantised(rng, (B, Hkv, n, d))
    dO = rng.standard_normal((B, Hq, n, d))
    off, st = oracle.sample_bins(n, [2.0, 9.0], s, seed=4)
    dQ, dK, dV = oracle.plsh_attn_backward(Q, K, V, dO, off, st, s, causal)
    grads = {"Q": dQ, "K": dK, "V": dV}
    for name, X in (("Q", Q), ("K", K), ("V", V)):
        for _ in range(6):
            idx = tuple(rng.integers(0, m) for m in X.shape)

            def diff(h):
                Xp, Xm = X.copy(), X.copy()
                Xp[idx] += h
                Xm[idx] -= h
                args = {"Q": Q, "K": K, "V": V}
                args[name] = Xp
                lp = forward_loss(args["Q"], args["K"], args["V"], dO, off, st, s, causal)
                args[name] = Xm
                lm = forward_loss(args["Q"], args["K"], args["V"], dO, off, st, s, causal)
                return (lp - lm) / (2 * h)
            fd = (4 * diff(2.0 ** -9) - diff(2.0 ** -8)) / 3     # Richardson: O(h^4)
            an = grads[name][idx]
            assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (name, idx, fd, an)


def test_one_bin_is_plain_softmax_attention():
    """With every hash one bin over all positions, c_ij = s for every pair, so
    the gradients are those of causal softmax attention (torch autograd, fp64)."""
    rng = np.random.default_rng(3)
    B, Hq, Hkv, n, d, s = 2, 4, 2, 30, 16, 3
    Q = rng.standard_normal((B, Hq, n, d))
    K = rng.standard_normal((B, Hkv, n, d))
    V = rng.standard_normal((B, Hkv, n, d))
    dO = rng.standard_normal((B, Hq, n, d))
    off = np.arange(0, 2 * Hq * s + 1, 2, dtype=np.int64)
    st = np.tile(np.array([0, n], dtype=np.int32), Hq * s)
    dQ, dK, dV = oracle.plsh_attn_backward(Q, K, V, dO, off, st, s, True)
    q = torch.tensor(Q, requires_grad=True)
    k = torch.tensor(K, requires_grad=True)
    v = torch.tensor(V, requires_grad=True)
    kk = k.repeat_interleave(Hq // Hkv, dim=1)
    vv = v.repeat_interleave(Hq // Hkv, dim=1)
    S = q @ kk.transpose(-1, -2) / math.sqrt(d)
    S = S.masked_fill(torch.triu(torch.ones(n, n, dtype=torch.bool), 1), float("-inf"))
    O = torch.softmax(S, dim=-1) @ vv
    (O * torch.tensor(dO)).sum().backward()
    np.testing.assert_allclose(dQ, q.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dK, k.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dV, v.grad.numpy(), rtol=1e-10, atol=1e-12)
