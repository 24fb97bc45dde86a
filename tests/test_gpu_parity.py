"""CUDA path vs the fp64 oracle, through the C ABI.

Tolerances (elementwise |gpu - oracle| <= atol + rtol |oracle|):
  bf16 inputs: atol 2e-3, rtol 1e-2   (P is rounded to f16, O to bf16)
  fp32 inputs: atol 1e-5, rtol 1e-5
Bin boundaries and draws: bit-exact.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import positional_lsh_approximation_gb300 as plsh
from positional_lsh_approximation_gb300.inputs import (WORKLOADS, Workload,
                                                       alibi_sigmas, make_qkv,
                                                       sample_rows)

pytestmark = pytest.mark.gpu

TOL = {"bf16": (2e-3, 1e-2), "f32": (1e-5, 1e-5)}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    plsh.build()
    plsh.load()


def to_dev(x: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x))
    t = t.to(torch.bfloat16) if dtype == "bf16" else t
    return t.cuda()


def gather_rows(O: torch.Tensor, rows):
    rb, rh, ri = (torch.from_numpy(np.asarray(r, dtype=np.int64)).cuda() for r in rows)
    return O[rb, rh, ri].float().cpu().numpy().astype(np.float64)


def assert_close(got, ref, dtype, what=""):
    atol, rtol = TOL[dtype]
    err = np.abs(got - ref)
    bad = err > atol + rtol * np.abs(ref)
    assert not np.isnan(got).any(), f"{what}: NaN in GPU output"
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements out of "
                             f"tolerance; max err {err.max():.3e}; first {idx.tolist()}")


def run_approx(w: Workload, Q, K, V, bins, path=None, monkeypatch=None):
    if path is not None:
        monkeypatch.setenv("PLSH_PATH", path)
    O = plsh.alibi_attn(to_dev(Q, w.dtype), to_dev(K, w.dtype), to_dev(V, w.dtype),
                        bins, w.causal)
    plsh.stream_status()
    return O


# ------------------------------------------------------------------ sampler
@pytest.mark.parametrize("n,H,s,sig,seed", [
    (1, 1, 3, [2.0], 0), (31, 2, 5, [0.6, 3.0], 1), (1000, 1, 8, [16.0], 0),
    (8192, 32, 10, None, 0), (16384, 32, 40, None, 0), (131072, 40, 16, [256.0], 0),
    (4097, 3, 64, [1e6, 0.9, 50.0], 2**63 + 5)])
def test_sampler_bit_exact(n, H, s, sig, seed):
    sigma = alibi_sigmas(H) if sig is None else np.asarray(sig, dtype=np.float64)
    bins = plsh.sample_bins(n, sigma, s, seed)
    off, st = bins.to_host()
    w, u = bins.draws()
    roff, rst, rw, ru = oracle.sample_bins(n, sigma, s, seed, return_draws=True)
    assert np.array_equal(w.view(np.uint64), rw.view(np.uint64))
    assert np.array_equal(u.view(np.uint64), ru.view(np.uint64))
    assert np.array_equal(off, roff)
    assert np.array_equal(st, rst)
    # resampling in place gives a new, equally exact draw
    bins.resample(sigma * 1.5, seed + 1)
    off2, st2 = bins.to_host()
    roff2, rst2 = oracle.sample_bins(n, sigma * 1.5, s, seed + 1)
    assert np.array_equal(off2, roff2) and np.array_equal(st2, rst2)
    # same sigma, new seed (sigma stays on the device), then back to the first
    bins.resample(sigma * 1.5, seed + 2)
    off3, st3 = bins.to_host()
    roff3, rst3 = oracle.sample_bins(n, sigma * 1.5, s, seed + 2)
    assert np.array_equal(off3, roff3) and np.array_equal(st3, rst3)
    bins.resample(sigma, seed)
    off4, st4 = bins.to_host()
    assert np.array_equal(off4, roff) and np.array_equal(st4, rst)
    bins.free()


def test_bins_from_host_round_trip():
    n, H, s = 777, 3, 6
    off, st = oracle.sample_bins(n, [2.0, 9.0, 70.0], s, seed=4)
    bins = plsh.bins_from_host(n, H, s, off, st)
    off2, st2 = bins.to_host()
    assert np.array_equal(off, off2) and np.array_equal(st, st2)


# --------------------------------------------------------- small, all rows
SMALL = [
    # name, B, Hq, Hkv, n, d, dtype, causal, s, sigma
    ("f32_tiny_like", 1, 1, 1, 300, 64, "f32", False, 8, (16.0,)),
    ("f32_causal_gqa", 2, 4, 2, 260, 128, "f32", True, 5, (0.7, 3.0, 20.0, 90.0)),
    ("bf16_causal_ragged", 1, 4, 2, 1000, 128, "bf16", True, 10, (1.2, 6.0, 40.0, 300.0)),
    ("bf16_noncausal_ragged", 2, 2, 1, 777, 128, "bf16", False, 6, (3.0, 150.0)),
    ("bf16_d64", 1, 2, 1, 513, 64, "bf16", True, 4, (5.0, 60.0)),
    # d = 64 on the tensor cores (zero-padded to 128 columns): GQA, without
    # the mask, ragged tails
    ("bf16_d64_gqa_s10", 1, 4, 2, 700, 64, "bf16", True, 10, (1.2, 6.0, 40.0, 300.0)),
    ("bf16_d64_noncausal", 2, 2, 1, 390, 64, "bf16", False, 6, (3.0, 150.0)),
    ("bf16_s24", 1, 2, 1, 700, 128, "bf16", True, 24, (3.0, 50.0)),
    ("bf16_s48", 1, 2, 2, 640, 128, "bf16", True, 48, (2.0, 30.0)),
    ("bf16_s64", 1, 2, 2, 640, 128, "bf16", True, 64, (2.0, 30.0)),
    ("bf16_noncausal_s30", 1, 2, 1, 400, 128, "bf16", False, 30, (0.8, 40.0)),
    # the largest s the tensor-core kernel's shared memory holds (52 with the
    # causal mask, 29 without), and the next one up (CUDA cores)
    ("bf16_s52", 1, 2, 1, 520, 128, "bf16", True, 52, (2.0, 30.0)),
    ("bf16_s53", 1, 2, 1, 300, 128, "bf16", True, 53, (2.0, 30.0)),
    ("bf16_noncausal_s29", 1, 2, 1, 400, 128, "bf16", False, 29, (0.8, 40.0)),
    # every register-slot variant of the fused kernel (s rounded up to 4, 8,
    # 10, 12 or 16 causal; 8 or 16 without the causal mask)
    ("bf16_s7", 1, 2, 1, 900, 128, "bf16", True, 7, (2.5, 90.0)),
    ("bf16_s12", 2, 2, 1, 600, 128, "bf16", True, 12, (1.5, 20.0)),
    ("bf16_s15", 1, 4, 2, 520, 128, "bf16", True, 15, (1.1, 4.0, 30.0, 700.0)),
    ("bf16_noncausal_s13", 1, 2, 1, 450, 128, "bf16", False, 13, (2.0, 70.0)),
    ("bf16_short", 1, 3, 1, 70, 128, "bf16", True, 3, (1.0, 8.0, 1e5)),
    ("bf16_one_token", 1, 2, 1, 1, 128, "bf16", True, 2, (4.0, 4.0)),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
@pytest.mark.parametrize("path", ["auto", "simt"])
def test_small_cases_all_rows(case, path, monkeypatch):
    name, B, Hq, Hkv, n, d, dtype, causal, s, sig = case
    w = Workload(name, B, Hq, Hkv, n, d, dtype, causal, s, sig, qkv_seed=n + s)
    Q, K, V = make_qkv(w)
    sigma = w.sigmas()
    bins = plsh.sample_bins(n, sigma, s, seed=3)
    off, st = oracle.sample_bins(n, sigma, s, seed=3)
    O = run_approx(w, Q, K, V, bins, None if path == "auto" else path, monkeypatch)
    rows = oracle.all_rows(B, Hq, n)
    ref = oracle.plsh_attn_rows(Q, K, V, off, st, s, causal, rows)
    assert_close(gather_rows(O, rows), ref, dtype, f"{name}/{path}")


@pytest.mark.parametrize("case", SMALL[:5], ids=[c[0] for c in SMALL[:5]])
@pytest.mark.parametrize("path", ["auto", "simt"])
def test_exact_small_all_rows(case, path, monkeypatch):
    name, B, Hq, Hkv, n, d, dtype, causal, s, sig = case
    w = Workload(name, B, Hq, Hkv, n, d, dtype, causal, s, sig, qkv_seed=n + 1)
    Q, K, V = make_qkv(w)
    sigma = w.sigmas()
    if path == "simt":
        monkeypatch.setenv("PLSH_PATH", "simt")
    O = plsh.alibi_exact(to_dev(Q, dtype), to_dev(K, dtype), to_dev(V, dtype), sigma, causal)
    plsh.stream_status()
    rows = oracle.all_rows(B, Hq, n)
    ref = oracle.alibi_exact_rows(Q, K, V, sigma, causal, rows)
    assert_close(gather_rows(O, rows), ref, dtype, f"exact {name}/{path}")


def test_special_cases_single_bin_and_singletons():
    n, d = 300, 128
    w = Workload("sp", 1, 2, 1, n, d, "bf16", True, 1, (1.0,), qkv_seed=9)
    Q, K, V = make_qkv(w)
    # one bin [0, n) per head: plain causal softmax attention
    off = np.array([0, 2, 4], dtype=np.int64)
    st = np.array([0, n, 0, n], dtype=np.int32)
    bins = plsh.bins_from_host(n, 2, 1, off, st)
    O = run_approx(w, Q, K, V, bins)
    rows = oracle.all_rows(1, 2, n)
    ref = oracle.plsh_attn_rows(Q, K, V, off, st, 1, True, rows)
    assert_close(gather_rows(O, rows), ref, "bf16", "single bin")
    # all singletons: every output row is its own value row
    s = 3
    off = np.arange(0, 2 * s * (n + 1) + 1, n + 1, dtype=np.int64)
    st = np.tile(np.arange(n + 1, dtype=np.int32), 2 * s)
    bins = plsh.bins_from_host(n, 2, s, off, st)
    O = run_approx(w, Q, K, V, bins)
    got = O.float().cpu().numpy()
    np.testing.assert_array_equal(got[0, 0], V[0, 0])
    np.testing.assert_array_equal(got[0, 1], V[0, 0])


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "noncausal"])
def test_score_jump_in_a_later_key_tile(causal):
    """Keys 0..127 scaled by 16 (exact in bf16): every row that reaches them
    meets scores far above the running max it carried from the key tiles
    nearer its diagonal, so the kernel rescales O, l and the weights already
    written in the middle of a tile; all rows against the oracle."""
    n, s = 700, 6
    w = Workload("jump", 1, 2, 1, n, 128, "bf16", causal, s, (60.0, 400.0), qkv_seed=31)
    Q, K, V = make_qkv(w)
    K = K.copy()
    K[:, :, :128, :] *= 16.0
    sigma = w.sigmas()
    bins = plsh.sample_bins(n, sigma, s, seed=8)
    off, st = oracle.sample_bins(n, sigma, s, seed=8)
    rows = oracle.all_rows(1, 2, n)
    O = run_approx(w, Q, K, V, bins)
    ref = oracle.plsh_attn_rows(Q, K, V, off, st, s, causal, rows)
    assert_close(gather_rows(O, rows), ref, "bf16", "score jump, approx")
    E = plsh.alibi_exact(to_dev(Q, "bf16"), to_dev(K, "bf16"), to_dev(V, "bf16"), sigma, causal)
    plsh.stream_status()
    ref = oracle.alibi_exact_rows(Q, K, V, sigma, causal, rows)
    assert_close(gather_rows(E, rows), ref, "bf16", "score jump, exact")
    bins.free()


def test_peaky_rows_all_rows():
    """5 % of token rows with Q and K scaled by 8 (the Qwen-shaped inputs),
    small enough for every row against the oracle, both masks."""
    for causal in (True, False):
        w = Workload("peaky", 1, 4, 2, 900, 128, "bf16", causal, 10, (2.0, 9.0, 50.0, 250.0),
                     peaky_frac=0.05, qkv_seed=41)
        Q, K, V = make_qkv(w)
        sigma = w.sigmas()
        bins = plsh.sample_bins(w.n, sigma, w.s, seed=2)
        off, st = oracle.sample_bins(w.n, sigma, w.s, seed=2)
        rows = oracle.all_rows(1, 4, w.n)
        O = run_approx(w, Q, K, V, bins)
        ref = oracle.plsh_attn_rows(Q, K, V, off, st, w.s, causal, rows)
        assert_close(gather_rows(O, rows), ref, "bf16", f"peaky causal={causal}")
        bins.free()


def test_repeated_calls_reuse_queue_and_agree():
    w = WORKLOADS["mistral"].with_(n=2048)
    Q, K, V = make_qkv(w)
    bins = plsh.sample_bins(w.n, w.sigmas(), w.s, 0)
    q, k, v = to_dev(Q, "bf16"), to_dev(K, "bf16"), to_dev(V, "bf16")
    outs = [plsh.alibi_attn(q, k, v, bins, True) for _ in range(3)]
    plsh.stream_status()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


# ------------------------------------------------- full sizes, sampled rows
FULL = ["tiny", "mistral", "qwen_s10", "qwen_s20", "sweep_s1", "sweep_s5",
        "sweep_s10", "sweep_s20", "sweep_s40", "scout"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_rows(name):
    w = WORKLOADS[name]
    Q, K, V = make_qkv(w)
    sigma = w.sigmas()
    bins = plsh.sample_bins(w.n, sigma, w.s, w.hash_seed)
    off, st = oracle.sample_bins(w.n, sigma, w.s, w.hash_seed)
    O = run_approx(w, Q, K, V, bins)
    if name == "tiny":
        rows = oracle.all_rows(w.B, w.Hq, w.n)
    else:
        rows, (h_lo, h_hi) = sample_rows(w, per_head=24 if name == "scout" else 48)
        # every row of batch 0 for the smallest-sigma head, and for the
        # largest-sigma head where the oracle stays within seconds
        full_heads = [h_lo] + ([h_hi] if w.n * w.s <= 200_000 else [])
        rb = [rows[0]] + [np.zeros(w.n, np.int32) for _ in full_heads]
        rh = [rows[1]] + [np.full(w.n, h, np.int32) for h in full_heads]
        ri = [rows[2]] + [np.arange(w.n, dtype=np.int32) for _ in full_heads]
        rows = (np.concatenate(rb), np.concatenate(rh), np.concatenate(ri))
    ref = oracle.plsh_attn_rows(Q, K, V, off, st, w.s, w.causal, rows)
    assert_close(gather_rows(O, rows), ref, w.dtype, name)


@pytest.mark.parametrize("name", ["tiny", "mistral", "qwen_s10", "sweep_s10", "scout"])
def test_exact_full_size_sampled_rows(name):
    w = WORKLOADS[name]
    Q, K, V = make_qkv(w)
    sigma = w.sigmas()
    O = plsh.alibi_exact(to_dev(Q, w.dtype), to_dev(K, w.dtype), to_dev(V, w.dtype),
                         sigma, w.causal)
    plsh.stream_status()
    if name == "tiny":
        rows = oracle.all_rows(w.B, w.Hq, w.n)
    else:
        rows, _ = sample_rows(w, per_head=4 if name == "scout" else 12)
    ref = oracle.alibi_exact_rows(Q, K, V, sigma, w.causal, rows)
    assert_close(gather_rows(O, rows), ref, w.dtype, "exact " + name)


# ------------------------------------------------ f16 weights and values
def test_v_scaled_by_powers_of_two():
    """P V runs in f16 on the tensor cores.  V scaled by 2^12 (values up to
    about 2e4, every one an f16 value) gives O scaled by exactly 2^12, for the
    approximation and for exact ALiBi; V scaled by 2^-16 (mostly f16
    subnormals, rounded within 2^-25) stays within the scaled tolerance plus
    one subnormal step of the oracle."""
    n, s = 600, 8
    w = Workload("vscale", 1, 4, 2, n, 128, "bf16", True, s, (1.5, 7.0, 40.0, 300.0),
                 qkv_seed=17)
    Q, K, V = make_qkv(w)
    sigma = w.sigmas()
    bins = plsh.sample_bins(n, sigma, s, seed=4)
    q, k = to_dev(Q, "bf16"), to_dev(K, "bf16")
    O1 = plsh.alibi_attn(q, k, to_dev(V, "bf16"), bins, True)
    O2 = plsh.alibi_attn(q, k, to_dev(V * 4096.0, "bf16"), bins, True)
    E1 = plsh.alibi_exact(q, k, to_dev(V, "bf16"), sigma, True)
    E2 = plsh.alibi_exact(q, k, to_dev(V * 4096.0, "bf16"), sigma, True)
    plsh.stream_status()
    assert torch.equal(O2.float(), O1.float() * 4096.0)
    assert torch.equal(E2.float(), E1.float() * 4096.0)
    small = V * np.float32(2.0 ** -16)
    O3 = plsh.alibi_attn(q, k, to_dev(small, "bf16"), bins, True)
    plsh.stream_status()
    off, st = oracle.sample_bins(n, sigma, s, seed=4)
    rows = oracle.all_rows(1, 4, n)
    ref = oracle.plsh_attn_rows(Q, K, small, off, st, s, True, rows)
    got = gather_rows(O3, rows)
    bound = 2e-3 * 2.0 ** -16 + 2.0 ** -24 + 1e-2 * np.abs(ref)
    assert (np.abs(got - ref) <= bound).all(), np.abs(got - ref).max()
    bins.free()


@pytest.mark.parametrize("exact", [False, True], ids=["approx", "exact"])
def test_v_beyond_f16_range_is_reported(exact):
    """A value of V that rounds past f16's largest finite value (bf16 65536)
    is reported as PLSH_ERR_RANGE by the next plsh_stream_status, which clears
    the flag; 65280 (the largest bf16 value below it) is served."""
    n, s = 300, 4
    w = Workload("vrange", 1, 2, 1, n, 128, "bf16", True, s, (3.0, 30.0), qkv_seed=23)
    Q, K, V = make_qkv(w)
    bins = plsh.sample_bins(n, w.sigmas(), s, seed=1)
    q, k = to_dev(Q, "bf16"), to_dev(K, "bf16")

    def call(vv):
        if exact:
            return plsh.alibi_exact(q, k, to_dev(vv, "bf16"), w.sigmas(), True)
        return plsh.alibi_attn(q, k, to_dev(vv, "bf16"), bins, True)

    ok = V.copy()
    ok[0, 0, 17, 5] = 65280.0
    call(ok)
    plsh.stream_status()
    bad = V.copy()
    bad[0, 0, 211, 77] = -65536.0
    call(bad)
    with pytest.raises(plsh.PlshError) as err:
        plsh.stream_status()
    assert err.value.status == plsh.PLSH_ERR_RANGE
    plsh.stream_status()
    bins.free()


# ---------------------------------------- key-range split of long items
SPLIT_CASES = [
    # name, B, Hq, Hkv, n, d, causal, s, sigma
    ("causal_ragged", 1, 4, 2, 1000, 128, True, 10, (1.2, 6.0, 40.0, 300.0)),
    ("noncausal", 2, 2, 1, 777, 128, False, 6, (3.0, 150.0)),
    ("odd_group", 1, 3, 1, 900, 128, True, 7, (2.5, 90.0, 400.0)),
    ("sorted_lists", 1, 2, 1, 700, 128, True, 24, (3.0, 50.0)),
    ("d64", 1, 2, 1, 800, 64, True, 8, (40.0, 600.0)),
]


@pytest.mark.parametrize("parts", [2, 3])
@pytest.mark.parametrize("case", SPLIT_CASES, ids=[c[0] for c in SPLIT_CASES])
def test_forced_split_all_rows(case, parts):
    """Every work item cut into 2 or 3 key ranges (parts past an item's
    envelope do nothing), partial rows combined by the merge kernel: every
    row against the oracle, approximation and exact ALiBi."""
    name, B, Hq, Hkv, n, d, causal, s, sig = case
    w = Workload(name, B, Hq, Hkv, n, d, "bf16", causal, s, sig, qkv_seed=n + parts)
    Q, K, V = make_qkv(w)
    sigma = w.sigmas()
    bins = plsh.sample_bins(n, sigma, s, seed=9)
    off, st = oracle.sample_bins(n, sigma, s, seed=9)
    rows = oracle.all_rows(B, Hq, n)
    plsh.set_split_parts(parts)
    try:
        O = run_approx(w, Q, K, V, bins)
        E = plsh.alibi_exact(to_dev(Q, "bf16"), to_dev(K, "bf16"), to_dev(V, "bf16"), sigma,
                             causal)
        plsh.stream_status()
    finally:
        plsh.set_split_parts(0)
    ref = oracle.plsh_attn_rows(Q, K, V, off, st, s, causal, rows)
    assert_close(gather_rows(O, rows), ref, "bf16", f"split {parts} {name}")
    ref_e = oracle.alibi_exact_rows(Q, K, V, sigma, causal, rows)
    assert_close(gather_rows(E, rows), ref_e, "bf16", f"split {parts} exact {name}")
    bins.free()


def test_automatic_split_long_envelopes():
    """One pair of heads whose bins span thousands of keys: the automatic
    split cuts the long items of the last row tiles; every row of both heads
    against the oracle, and against the unsplit kernel."""
    n, s = 4096, 6
    w = Workload("long", 1, 2, 1, n, 128, "bf16", True, s, (3000.0, 4000.0), qkv_seed=21)
    Q, K, V = make_qkv(w)
    sigma = w.sigmas()
    bins = plsh.sample_bins(n, sigma, s, seed=2)
    off, st = oracle.sample_bins(n, sigma, s, seed=2)
    plsh.set_split_parts(0)
    O = run_approx(w, Q, K, V, bins)
    plsh.set_split_parts(1)
    try:
        O1 = run_approx(w, Q, K, V, bins)
    finally:
        plsh.set_split_parts(0)
    rows = oracle.all_rows(1, 2, n)
    ref = oracle.plsh_attn_rows(Q, K, V, off, st, s, True, rows)
    assert_close(gather_rows(O, rows), ref, "bf16", "automatic split")
    assert_close(gather_rows(O1, rows), ref, "bf16", "unsplit")
    bins.free()


def test_item_table_cache_eviction():
    """More shapes than the item-table cache holds: tables of shapes no call
    holds are freed in stream order behind their last use, and a shape seen
    again after its table was evicted gives the same output bit for bit."""
    d, Hq, Hkv, s = 128, 2, 1, 4
    outs = {}
    first = None
    for k in range(20):
        n = 256 + 128 * k
        w = Workload(f"ev{k}", 1, Hq, Hkv, n, d, "bf16", True, s, (3.0, 40.0), qkv_seed=500 + k)
        Q, K, V = (to_dev(x, "bf16") for x in make_qkv(w))
        bins = plsh.sample_bins(n, w.sigmas(), s, seed=11)
        O = plsh.alibi_attn(Q, K, V, bins, True)
        plsh.stream_status()
        if k == 0:
            first = (Q, K, V, bins)
            outs[k] = O.clone()
    Q, K, V, bins = first
    again = plsh.alibi_attn(Q, K, V, bins, True)
    plsh.stream_status()
    assert torch.equal(again, outs[0])


def test_item_table_built_on_another_stream():
    """A shape's first call on one stream builds its item table there; a call
    of the same shape queued at once on a second stream (no host
    synchronisation between them) waits for that upload by event and gives
    the same output bit for bit."""
    n, d, s = 1664, 128, 6
    w = Workload("xs", 1, 2, 1, n, d, "bf16", True, s, (2.0, 70.0), qkv_seed=77)
    Q, K, V = (to_dev(x, "bf16") for x in make_qkv(w))
    bins = plsh.sample_bins(n, w.sigmas(), s, seed=5)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    O1 = torch.empty_like(Q)
    O2 = torch.empty_like(Q)
    plsh.alibi_attn(Q, K, V, bins, True, out=O1, stream=s1)
    plsh.alibi_attn(Q, K, V, bins, True, out=O2, stream=s2)
    torch.cuda.synchronize()
    plsh.stream_status()
    assert torch.equal(O1, O2)
