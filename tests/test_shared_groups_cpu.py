"""Pins of the oracle's hashes shared across a GQA group: every head of a
group carries its group's start lists, and heads with equal inputs then give
equal outputs."""
import numpy as np

import oracle


def test_heads_of_a_group_carry_the_group_lists():
    n, s, G, Hq = 500, 4, 2, 8
    off, st = oracle.sample_bins(n, [5.0, 60.0], s, seed=2)
    so, ss = oracle.share_groups(off, st, G, Hq, s)
    assert len(so) == Hq * s + 1
    for h in range(Hq):
        g = h // (Hq // G)
        for t in range(s):
            a = ss[so[h * s + t]:so[h * s + t + 1]]
            b = st[off[g * s + t]:off[g * s + t + 1]]
            np.testing.assert_array_equal(a, b)


def test_equal_heads_give_equal_rows():
    rng = np.random.default_rng(4)
    n, d, s, G, Hq = 120, 16, 3, 1, 2
    off, st = oracle.sample_bins(n, [7.0], s, seed=9)
    so, ss = oracle.share_groups(off, st, G, Hq, s)
    q = rng.standard_normal((1, 1, n, d)).astype(np.float32)
    Q = np.concatenate([q, q], axis=1)
    K = rng.standard_normal((1, 1, n, d)).astype(np.float32)
    V = rng.standard_normal((1, 1, n, d)).astype(np.float32)
    O = oracle.plsh_attn_rows(Q, K, V, so, ss, s, True, oracle.all_rows(1, 2, n)).reshape(2, n, d)
    np.testing.assert_array_equal(O[0], O[1])
