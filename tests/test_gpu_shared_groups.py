"""GPU checks of plsh_bins_share_groups: exact start lists and draws against
the oracle, and attention on shared hashes against the oracle rows."""
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


def test_shared_groups_lists_draws_and_attention():
    n, s, G, Hq = 900, 6, 2, 4
    src = plsh.sample_bins(n, [12.0, 150.0], s, seed=3)
    b = plsh.bins_share_groups(src, Hq)
    off, st = oracle.sample_bins(n, [12.0, 150.0], s, seed=3)
    so, ss = oracle.share_groups(off, st, G, Hq, s)
    go, gs = b.to_host()
    np.testing.assert_array_equal(go, so)
    np.testing.assert_array_equal(gs, ss)
    w0, u0 = src.draws()
    w1, u1 = b.draws()
    for h in range(Hq):
        g = h // (Hq // G)
        np.testing.assert_array_equal(w1[h * s:(h + 1) * s], w0[g * s:(g + 1) * s])
        np.testing.assert_array_equal(u1[h * s:(h + 1) * s], u0[g * s:(g + 1) * s])
    w = Workload("shared", 1, Hq, G, n, 128, "bf16", True, s, (12.0,), qkv_seed=8)
    Q, K, V = make_qkv(w)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).cuda()
    O = plsh.alibi_attn(dev(Q), dev(K), dev(V), b, True)
    plsh.stream_status()
    rows = oracle.all_rows(1, Hq, n)
    ref = oracle.plsh_attn_rows(Q, K, V, so, ss, s, True, rows)
    got = O.float().cpu().numpy().reshape(-1, 128).astype(np.float64)
    assert (np.abs(got - ref) <= 2e-3 + 1e-2 * np.abs(ref)).all()
    b.free()
    src.free()
