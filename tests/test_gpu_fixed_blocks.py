"""plsh_bins_fixed on the GPU: the records it builds give exactly the oracle's
start lists, and attention and decode on fixed blocks match the oracle."""
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


@pytest.mark.parametrize("n,widths,s", [
    (1, [1], 1), (33, [1, 2, 40], 3), (1000, [7, 64, 128, 1000], 10),
    (4097, [5, 33, 300, 5000], 4), (8192, [2, 3, 512], 64),
])
def test_fixed_bins_match_oracle_lists(n, widths, s):
    b = plsh.bins_fixed(n, widths, s)
    off, st = b.to_host()
    ro, rs = oracle.bins_fixed(n, widths, s)
    np.testing.assert_array_equal(off, ro)
    np.testing.assert_array_equal(st, rs)
    w, u = b.draws()
    for h, wh in enumerate(widths):
        for t in range(s):
            assert w[h * s + t] == wh and u[h * s + t] == t * wh // s
    b.free()


def to_dev(x, dtype):
    t = torch.from_numpy(np.ascontiguousarray(x))
    return (t.to(torch.bfloat16) if dtype == "bf16" else t).cuda()


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "noncausal"])
def test_attention_on_fixed_blocks(causal):
    n, s, widths = 900, 4, [3, 40, 200, 1000]
    w = Workload("fixed", 1, 4, 2, n, 128, "bf16", causal, s, (1.0,), qkv_seed=23)
    Q, K, V = make_qkv(w)
    b = plsh.bins_fixed(n, widths, s)
    off, st = oracle.bins_fixed(n, widths, s)
    O = plsh.alibi_attn(to_dev(Q, "bf16"), to_dev(K, "bf16"), to_dev(V, "bf16"), b, causal)
    plsh.stream_status()
    rows = oracle.all_rows(1, 4, n)
    ref = oracle.plsh_attn_rows(Q, K, V, off, st, s, causal, rows)
    rb, rh, ri = (torch.from_numpy(np.asarray(r, dtype=np.int64)).cuda() for r in rows)
    got = O[rb, rh, ri].float().cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    assert (err <= 2e-3 + 1e-2 * np.abs(ref)).all(), err.max()
    # decode of the last position on the same blocks
    if causal:
        pos = n - 1
        o = plsh.alibi_decode(to_dev(Q[:, :, pos:pos + 1], "bf16"), to_dev(K, "bf16"),
                              to_dev(V, "bf16"), b, pos)
        plsh.stream_status()
        got = o.float().cpu().numpy().astype(np.float64)[0, :, 0, :]
        ref = oracle.plsh_attn_rows(Q, K, V, off, st, s, True,
                                    (np.zeros(4, np.int64), np.arange(4), np.full(4, pos)))
        assert (np.abs(got - ref) <= 2e-3 + 1e-2 * np.abs(ref)).all()
    b.free()


def test_fixed_bins_reject_bad_arguments():
    for widths, s in (([0], 1), ([4], 0), ([4], 65)):
        with pytest.raises(plsh.PlshError) as err:
            plsh.bins_fixed(100, widths, s)
        assert err.value.status == plsh.PLSH_ERR_INVALID
