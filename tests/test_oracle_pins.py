"""Pins of the oracle to facts fixed by the paper and by mathematics.

"Positional LSH: Binary Block Matrix Approximation for Attention with Linear
Biases" (Wolfson & Wagner), technical summary:
  Methodology 1  L*_ij = exp(-|i-j|/sigma); contiguous non-overlapping bins;
                 L* = E_h[M(h)]
  Methodology 2  (Theorem 2.1) O(1/sqrt(s)) error in spectral and max norm;
                 b_max ~ sigma log log n; Gamma-distributed widths
  Methodology 3  (Theorem 2.2) output error = bias error against the biased
                 row sums
None of these tests reads the oracle's own formulas back: each compares it to
a closed form, a library routine, a statistical law or a second route.
"""
import math
import os

import numpy as np
import pytest
import scipy.integrate
import scipy.stats
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- helpers
def dense_mask_mean(n, offsets, starts, h, s):
    """(1/s) sum_t M(h_t) as a dense fp64 matrix, built from bin ids."""
    m = np.zeros((n, n))
    pos = np.arange(n)
    for t in range(s):
        st = starts[offsets[h * s + t]:offsets[h * s + t + 1]]
        ids = np.searchsorted(st, pos, side="right")
        m += (ids[:, None] == ids[None, :])
    return m / s


def laplace_kernel(n, sigma):
    i = np.arange(n)
    return np.exp(-np.abs(i[:, None] - i[None, :]) / sigma)


def dense_scores(Q, K, b, h, group):
    q = Q[b, h].astype(np.float64)
    k = K[b, h // group].astype(np.float64)
    return q @ k.T / math.sqrt(Q.shape[-1])


def dense_weighted(W, S, V, causal):
    """rows of (W o exp(S)) V / (W o exp(S)) 1, with a row shift for safety."""
    n = S.shape[0]
    A = np.exp(S - S.max(axis=1, keepdims=True))
    if causal:
        A = A * np.tril(np.ones((n, n)))
    WA = W * A
    return (WA @ V) / WA.sum(axis=1, keepdims=True)


def rand_qkv(B, Hq, Hkv, n, d, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    Q = (rng.standard_normal((B, Hq, n, d)) * scale).astype(np.float32)
    K = (rng.standard_normal((B, Hkv, n, d)) * scale).astype(np.float32)
    V = rng.standard_normal((B, Hkv, n, d)).astype(np.float32)
    return Q, K, V


# ------------------------------------------------------ random numbers / ln
def test_philox_known_answers():
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        lines = [l.split() for l in f if l.strip() and not l.startswith("#")]
    assert len(lines) == 3
    for parts in lines:
        words = [int(x, 16) for x in parts]
        out = oracle.philox4x32_10(words[0:4], words[4:6])
        assert [int(x) for x in out] == words[6:10]


def test_ln64_matches_libm_within_two_ulp():
    """The sampler's own ln (atanh series after reduction to [sqrt(1/2),
    sqrt(2)), 12 terms) stays within 2 ulp of the C library's log."""
    rng = np.random.default_rng(3)
    xs = np.r_[rng.random(20000), (np.arange(1, 2001) - 0.5) * 2.0 ** -32,
               1.0 - (np.arange(1, 2001) - 0.5) * 2.0 ** -32,
               np.exp2(rng.uniform(-60, 60, 4000))]
    for x in xs:
        got = oracle.ln64(float(x))
        ref = math.log(float(x))
        assert abs(got - ref) <= 2 * math.ulp(ref) + 1e-300, (x, got, ref)
    assert oracle.ln64(1.0) == 0.0


# ------------------------------------------------------------- width law
@pytest.mark.parametrize("sigma", [0.7, 4.0, 37.0])
def test_gamma2_width_law_gives_laplace_kernel(sigma):
    """P(i, j share a bin) = E_w[(1 - D/w)_+] with w ~ Gamma(2, scale sigma)
    equals exp(-D/sigma): the reading of the width law that makes
    L* = E[M(h)] (Methodology 1) hold exactly."""
    dens = lambda w: w / sigma ** 2 * math.exp(-w / sigma)
    for D in range(0, 11):
        val, _ = scipy.integrate.quad(
            lambda w: max(0.0, 1.0 - D / w) * dens(w) if w > 0 else 0.0,
            D, np.inf, limit=200)
        if D == 0:
            val = 1.0 - scipy.integrate.quad(dens, 0, 0)[0]
        assert abs(val - math.exp(-D / sigma)) < 1e-9
    # the other parametrisation (rate sigma) would not reproduce the kernel
    wrong = scipy.integrate.quad(
        lambda w: max(0.0, 1.0 - 3 / w) * (w * sigma ** 2 * math.exp(-w * sigma)),
        3, np.inf)[0]
    if sigma != 1.0:
        assert abs(wrong - math.exp(-3 / sigma)) > 1e-3


def test_draws_follow_gamma2_and_uniform_offset():
    sigma = 5.0
    N = 20000
    _, _, w, u = oracle.sample_bins(8, [sigma], N, seed=11, return_draws=True)
    x = w / sigma
    ks = scipy.stats.kstest(x, lambda z: 1.0 - (1.0 + z) * np.exp(-z))
    assert ks.pvalue > 1e-3, ks
    ks_u = scipy.stats.kstest(u / w, "uniform")
    assert ks_u.pvalue > 1e-3, ks_u
    assert np.all(u > 0) and np.all(u < w)
    # heads draw independently: same sigma, different head index
    _, _, w2, _ = oracle.sample_bins(8, [sigma, sigma], 4, seed=11,
                                     return_draws=True)
    assert not np.array_equal(w2[:4], w2[4:])
    # draws depend on the seed
    _, _, w3, _ = oracle.sample_bins(8, [sigma], 4, seed=12, return_draws=True)
    assert not np.array_equal(w3, w[:4])


# ------------------------------------------------------------ bin geometry
@pytest.mark.parametrize("n,sigma", [(1, 3.0), (7, 100.0), (300, 0.3),
                                     (1000, 2.5), (4096, 40.0), (513, 1e6)])
def test_bins_contiguous_non_overlapping(n, sigma):
    """Methodology 1: bins of the integer positions are contiguous and do not
    overlap; every position lies in exactly one bin."""
    s = 12
    offsets, starts, w, u = oracle.sample_bins(n, [sigma], s, seed=5,
                                               return_draws=True)
    for t in range(s):
        st = starts[offsets[t]:offsets[t + 1]].astype(np.int64)
        assert st[0] == 0 and st[-1] == n
        assert np.all(np.diff(st) >= 1)
        lens = np.diff(st)
        assert lens.sum() == n
        if w[t] < 1.0:
            assert np.all(lens == 1)
            continue
        first = math.ceil(u[t])
        if first < n:
            assert st[1] == first
        interior = lens[1:-1]
        if interior.size:
            assert set(np.unique(interior)) <= {math.floor(w[t]),
                                                math.ceil(w[t])}


def test_bin_membership_is_floor_of_shifted_position():
    """Position x lies in bin floor((x - u)/w) (random binning, Methodology 1);
    checked against the oracle's start lists with exact rational arithmetic
    away from ties."""
    from fractions import Fraction
    n = 400
    offsets, starts, w, u = oracle.sample_bins(n, [6.0], 20, seed=9,
                                               return_draws=True)
    for t in range(20):
        if w[t] < 1:
            continue
        st = starts[offsets[t]:offsets[t + 1]]
        ids = np.searchsorted(st, np.arange(n), side="right") - 1
        W, U = Fraction(w[t]), Fraction(u[t])
        ref = [math.floor((Fraction(x) - U) / W) + 1 for x in range(n)]
        assert list(ids) == ref


def test_expectation_of_masks_is_laplace_kernel():
    """Methodology 1: L* = E_h[M(h)], Monte Carlo over N hashes."""
    n, sigma, N = 40, 4.0, 30000
    offsets, starts = oracle.sample_bins(n, [sigma], N, seed=21)
    Mbar = dense_mask_mean(n, offsets, starts, 0, N)
    L = laplace_kernel(n, sigma)
    sd = np.sqrt(L * (1 - L) / N)
    assert np.all(np.abs(Mbar - L) <= 5 * sd + 1e-12)


def test_bmax_distribution():
    """Methodology 2: the longest block over s hashes is max_t ceil(w_t), so
    P(b_max <= x) = F(x)^s with F the Gamma(2, sigma) CDF; at s = ceil(ln n)
    this is sigma * O(log s) = sigma * O(log log n)."""
    n, sigma = 4096, 8.0
    s = math.ceil(math.log(n))          # 9
    trials = 2000
    offsets, starts = oracle.sample_bins(n, [sigma], s * trials, seed=31)
    lens = np.diff(starts.astype(np.int64))
    per_hash = np.array([lens[offsets[t]:offsets[t + 1] - 1].max()
                         for t in range(s * trials)])
    bmax = per_hash.reshape(trials, s).max(axis=1)
    F = lambda x: 1.0 - (1.0 + x / sigma) * math.exp(-x / sigma)
    for x in (16, 24, 32, 48, 64):
        p = F(x) ** s
        emp = np.mean(bmax <= x)
        assert abs(emp - p) <= 4.5 * math.sqrt(p * (1 - p) / trials) + 1e-3, x
    # median of b_max / sigma grows like log s
    for s2 in (4, 16, 64):
        offs, st = oracle.sample_bins(2048, [sigma], s2 * 300, seed=40 + s2)
        ln = np.diff(st.astype(np.int64))
        ph = np.array([ln[offs[t]:offs[t + 1] - 1].max()
                       for t in range(s2 * 300)])
        med = np.median(ph.reshape(300, s2).max(axis=1)) / sigma
        theo = scipy.optimize.brentq(lambda z: (1 - (1 + z) * math.exp(-z)) ** s2
                                     - 0.5, 0.01, 100)
        assert abs(med - theo) < 0.35, (s2, med, theo)


def test_laplace_kernel_spectral_norm_toeplitz_limit():
    """||L*||_2 tends to coth(1/(2 sigma)) (Kac-Murdock-Szego Toeplitz
    symbol), which pins the test's own L* construction used below."""
    L = laplace_kernel(2000, 16.0)
    lam = np.linalg.eigvalsh(L).max()
    assert abs(lam / (1.0 / math.tanh(1.0 / 32.0)) - 1) < 2e-3


def test_error_decays_as_inverse_sqrt_s():
    """Methodology 2 / Results: ||L* - M~|| decays like O(1/sqrt(s)) in max
    norm and spectral norm."""
    n, sigma = 192, 6.0
    L = laplace_kernel(n, sigma)
    ss = [2 ** k for k in range(0, 9)]
    spec, mx = [], []
    for s in ss:
        sp, mm = [], []
        for seed in range(8):
            offsets, starts = oracle.sample_bins(n, [sigma], s, seed=100 + seed)
            e_max, e_spec = oracle.bias_error(n, sigma, offsets, starts, 0, s)
            if seed == 0:
                # the oracle's norms are those of the test's own dense matrices
                E = dense_mask_mean(n, offsets, starts, 0, s) - L
                assert abs(e_max - np.abs(E).max()) < 1e-14
                assert abs(e_spec - np.abs(np.linalg.eigvalsh(E)).max()) < 1e-12
            sp.append(e_spec)
            mm.append(e_max)
        spec.append(np.mean(sp)); mx.append(np.mean(mm))
    slope_spec = np.polyfit(np.log(ss), np.log(spec), 1)[0]
    slope_max = np.polyfit(np.log(ss[2:]), np.log(mx[2:]), 1)[0]
    assert -0.62 < slope_spec < -0.38, slope_spec
    assert -0.62 < slope_max < -0.38, slope_max


# ---------------------------------------------------------------- attention
CASES = [  # B, Hq, Hkv, n, d, s, sigmas, causal
    (1, 1, 1, 64, 16, 1, [5.0], False),
    (1, 2, 1, 96, 16, 5, [3.0, 10.0], True),
    (2, 4, 2, 130, 8, 7, [0.8, 2.0, 9.0, 40.0], False),
    (1, 2, 2, 200, 32, 3, [60.0, 1.5], True),
]


@pytest.mark.parametrize("case", CASES)
def test_oracle_matches_dense_mask_route(case):
    """The oracle's per-sample, per-bin evaluation equals the dense matrix
    form D~^-1 (M~ o A) V (Theorem 2.2 with the averaged mask)."""
    B, Hq, Hkv, n, d, s, sig, causal = case
    Q, K, V = rand_qkv(B, Hq, Hkv, n, d, seed=n)
    offsets, starts = oracle.sample_bins(n, sig, s, seed=3)
    rows = oracle.all_rows(B, Hq, n)
    got = oracle.plsh_attn_rows(Q, K, V, offsets, starts, s, causal, rows)
    got = got.reshape(B, Hq, n, d)
    group = Hq // Hkv
    for b in range(B):
        for h in range(Hq):
            M = dense_mask_mean(n, offsets, starts, h, s)
            S = dense_scores(Q, K, b, h, group)
            ref = dense_weighted(M, S, V[b, h // group].astype(np.float64), causal)
            np.testing.assert_allclose(got[b, h], ref, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("case", CASES)
def test_exact_matches_torch_softmax(case):
    """Exact ALiBi: softmax(QK^T/sqrt(d) - |i-j|/sigma_h [+ causal mask]) V,
    computed by torch in fp64 on the CPU."""
    B, Hq, Hkv, n, d, s, sig, causal = case
    Q, K, V = rand_qkv(B, Hq, Hkv, n, d, seed=n + 1)
    rows = oracle.all_rows(B, Hq, n)
    got = oracle.alibi_exact_rows(Q, K, V, sig, causal, rows).reshape(B, Hq, n, d)
    group = Hq // Hkv
    q = torch.from_numpy(Q).double()
    k = torch.from_numpy(K).double().repeat_interleave(group, dim=1)
    v = torch.from_numpy(V).double().repeat_interleave(group, dim=1)
    idx = torch.arange(n, dtype=torch.float64)
    dist = (idx[:, None] - idx[None, :]).abs()
    logits = q @ k.transpose(-1, -2) / math.sqrt(d)
    logits = logits - dist / torch.tensor(sig, dtype=torch.float64)[None, :, None, None]
    if causal:
        logits = logits.masked_fill(idx[None, :] > idx[:, None], float("-inf"))
    ref = torch.softmax(logits, dim=-1) @ v
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_output_error_identity_and_bound(causal):
    """Methodology 3: the output error is governed by the bias error against
    the biased row sums.  Exactly:
      T~_i - T*_i = sum_j (M~ - L*)_ij A_ij (v_j - T*_i) / D~_i,
      D~_i = sum_j M~_ij A_ij, hence the row-sum bound."""
    n, d, s = 120, 16, 6
    sig = [7.0]
    Q, K, V = rand_qkv(1, 1, 1, n, d, seed=77)
    offsets, starts = oracle.sample_bins(n, sig, s, seed=8)
    rows = oracle.all_rows(1, 1, n)
    Tt = oracle.plsh_attn_rows(Q, K, V, offsets, starts, s, causal, rows)
    Ts = oracle.alibi_exact_rows(Q, K, V, sig, causal, rows)
    M = dense_mask_mean(n, offsets, starts, 0, s)
    L = laplace_kernel(n, sig[0])
    S = dense_scores(Q, K, 0, 0, 1)
    A = np.exp(S - S.max(axis=1, keepdims=True))
    if causal:
        A = A * np.tril(np.ones((n, n)))
    v = V[0, 0].astype(np.float64)
    Dt = (M * A).sum(axis=1)
    for i in range(n):
        rhs = ((M - L)[i] * A[i]) @ (v - Ts[i]) / Dt[i]
        np.testing.assert_allclose(Tt[i] - Ts[i], rhs, rtol=1e-9, atol=1e-12)
        bound = (np.abs(M - L)[i] * A[i]).sum() * np.abs(v - Ts[i]).max() / Dt[i]
        assert np.abs(Tt[i] - Ts[i]).max() <= bound + 1e-12


def test_single_full_bin_is_plain_softmax():
    """s = 1 with one bin [0, n): no positional bias, plain attention."""
    n, d = 77, 12
    Q, K, V = rand_qkv(1, 2, 1, n, d, seed=5)
    offsets = np.array([0, 2, 4], dtype=np.int64)
    starts = np.array([0, n, 0, n], dtype=np.int32)
    for causal in (False, True):
        got = oracle.plsh_attn_rows(Q, K, V, offsets, starts, 1, causal,
                                    oracle.all_rows(1, 2, n)).reshape(2, n, d)
        q = torch.from_numpy(Q[0]).double()
        k = torch.from_numpy(K[0, 0]).double()
        logits = q @ k.T / math.sqrt(d)
        if causal:
            logits = logits.masked_fill(torch.triu(torch.ones(n, n), 1).bool(),
                                        float("-inf"))
        ref = torch.softmax(logits, -1) @ torch.from_numpy(V[0, 0]).double()
        np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-13)


def test_all_singletons_return_values():
    n, d, s = 50, 8, 3
    Q, K, V = rand_qkv(1, 2, 1, n, d, seed=6, scale=5.0)
    offsets = np.arange(0, 2 * s * (n + 1) + 1, n + 1, dtype=np.int64)
    starts = np.tile(np.arange(n + 1, dtype=np.int32), 2 * s)
    for causal in (False, True):
        got = oracle.plsh_attn_rows(Q, K, V, offsets, starts, s, causal,
                                    oracle.all_rows(1, 2, n)).reshape(2, n, d)
        np.testing.assert_allclose(got[0], V[0, 0], rtol=0, atol=1e-15)
        np.testing.assert_allclose(got[1], V[0, 0], rtol=0, atol=1e-15)


def test_repeated_hash_and_sample_permutation():
    n, d = 90, 8
    Q, K, V = rand_qkv(1, 1, 1, n, d, seed=9)
    offsets, starts = oracle.sample_bins(n, [5.0], 4, seed=2)
    rows = oracle.all_rows(1, 1, n)
    one = starts[offsets[1]:offsets[2]]
    # s copies of one hash == that hash at s = 1
    rep_off = np.arange(0, 5 * one.size + 1, one.size, dtype=np.int64)
    rep = oracle.plsh_attn_rows(Q, K, V, rep_off, np.tile(one, 5), 5, True, rows)
    single = oracle.plsh_attn_rows(Q, K, V, np.array([0, one.size]), one, 1,
                                   True, rows)
    np.testing.assert_allclose(rep, single, rtol=1e-13, atol=1e-14)
    # permuting the samples changes nothing
    perm = [2, 0, 3, 1]
    pst = np.concatenate([starts[offsets[t]:offsets[t + 1]] for t in perm])
    poff = np.r_[0, np.cumsum([offsets[t + 1] - offsets[t] for t in perm])]
    a = oracle.plsh_attn_rows(Q, K, V, offsets, starts, 4, False, rows)
    b = oracle.plsh_attn_rows(Q, K, V, poff, pst, 4, False, rows)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-14)


def test_rows_lie_in_convex_hull_of_values():
    n, d, s = 256, 16, 6
    Q, K, V = rand_qkv(1, 1, 1, n, d, seed=12, scale=3.0)
    offsets, starts = oracle.sample_bins(n, [9.0], s, seed=4)
    rows = oracle.all_rows(1, 1, n)
    out = oracle.plsh_attn_rows(Q, K, V, offsets, starts, s, True, rows)
    for i in range(n):
        lo = min(starts[offsets[t]:offsets[t + 1]][
            np.searchsorted(starts[offsets[t]:offsets[t + 1]], i, "right") - 1]
            for t in range(s))
        vv = V[0, 0, lo:i + 1]
        assert np.all(out[i] >= vv.min(0) - 1e-12)
        assert np.all(out[i] <= vv.max(0) + 1e-12)


def test_numerator_and_denominator_are_unbiased():
    """E[N~/s] = (L* o A) V and E[D~/s] = (L* o A) 1 (the averaged masks are
    unbiased for L*); batch means over independent hash blocks."""
    n, d, sigma = 24, 8, 3.0
    Q, K, V = rand_qkv(1, 1, 1, n, d, seed=13, scale=0.5)
    rows = oracle.all_rows(1, 1, n)
    blocks, per = 16, 1500
    nums, dens = [], []
    for blk in range(blocks):
        offsets, starts = oracle.sample_bins(n, [sigma], per, seed=500 + blk)
        num, den = oracle.plsh_parts_rows(Q, K, V, offsets, starts, per, False,
                                          rows)
        nums.append(num / per); dens.append(den / per)
    nums, dens = np.array(nums), np.array(dens)
    S = dense_scores(Q, K, 0, 0, 1)
    LA = laplace_kernel(n, sigma) * np.exp(S)
    ref_num = LA @ V[0, 0].astype(np.float64)
    ref_den = LA.sum(axis=1)
    se_num = nums.std(axis=0, ddof=1) / math.sqrt(blocks)
    se_den = dens.std(axis=0, ddof=1) / math.sqrt(blocks)
    assert np.all(np.abs(nums.mean(0) - ref_num) <= 5 * se_num + 1e-9)
    assert np.all(np.abs(dens.mean(0) - ref_den) <= 5 * se_den + 1e-9)


def test_bias_error_closed_forms():
    """||L* - M~|| in two cases with closed forms.  All singletons: M~ = I, so
    the max-norm error is the nearest off-diagonal entry e^{-1/sigma} and the
    spectral error is max |lambda(L*) - 1| = coth(1/(2 sigma)) - 1 in the
    Toeplitz limit (Kac-Murdock-Szego).  One bin over everything: M~ = 1 1^T,
    the max-norm error is the far corner 1 - e^{-(n-1)/sigma}."""
    n, sigma, s = 1500, 8.0, 3
    offsets = np.arange(0, s * (n + 1) + 1, n + 1, dtype=np.int64)
    starts = np.tile(np.arange(n + 1, dtype=np.int32), s)
    e_max, e_spec = oracle.bias_error(n, sigma, offsets, starts, 0, s)
    assert abs(e_max - math.exp(-1.0 / sigma)) < 1e-14
    assert abs(e_spec / (1.0 / math.tanh(0.5 / sigma) - 1.0) - 1.0) < 5e-3
    offsets = np.array([0, 2, 4], dtype=np.int64)
    starts = np.array([0, 300, 0, 300], dtype=np.int32)
    e_max, _ = oracle.bias_error(300, 40.0, offsets, starts, 0, 2)
    assert abs(e_max - (1.0 - math.exp(-299.0 / 40.0))) < 1e-14


def test_bias_error_brute_force():
    """The oracle's max-norm error against an entry-by-entry loop on a tiny case."""
    n, sigma, s = 23, 3.0, 4
    offsets, starts = oracle.sample_bins(n, [sigma], s, seed=9)
    e_max, _ = oracle.bias_error(n, sigma, offsets, starts, 0, s)
    best = 0.0
    for i in range(n):
        for j in range(n):
            c = 0
            for t in range(s):
                st = list(starts[offsets[t]:offsets[t + 1]])
                bi = max(k for k in range(len(st) - 1) if st[k] <= i)
                bj = max(k for k in range(len(st) - 1) if st[k] <= j)
                c += bi == bj
            best = max(best, abs(math.exp(-abs(i - j) / sigma) - c / s))
    assert abs(e_max - best) < 1e-15
