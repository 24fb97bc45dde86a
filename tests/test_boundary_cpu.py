"""The C-ABI library builds, loads and exports every symbol of include/plsh.h;
host-side validation rejects bad arguments before touching the device."""
import ctypes
import os
import re

import numpy as np
import pytest

import positional_lsh_approximation_gb300 as plsh

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    with open(os.path.join(ROOT, "include", "plsh.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(plsh_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    plsh.build()
    return plsh.load()


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for name in ("plsh_sample_bins", "plsh_alibi_attn", "plsh_alibi_exact",
                 "plsh_bins_from_host", "plsh_bins_to_host", "plsh_bins_free",
                 "plsh_stream_status", "plsh_last_error"):
        assert name in syms


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for st in range(7):
        assert lib.plsh_status_string(st)
    assert lib.plsh_status_string(plsh.PLSH_ERR_RANGE) != lib.plsh_status_string(99)
    assert lib.plsh_last_error() is not None


@pytest.mark.parametrize("n,H,s,sigma", [(0, 1, 1, [1.0]), (10, 1, 0, [1.0]),
                                         (10, 1, 65, [1.0]), (10, 1, 2, [0.0]),
                                         (10, 1, 2, [float("nan")]),
                                         (10, 1, 2, [float("inf")]),
                                         (10, 2, 2, [1.0, -3.0])])
def test_sample_bins_rejects_bad_arguments(lib, n, H, s, sigma):
    sig = np.asarray(sigma, dtype=np.float64)
    out = ctypes.c_void_p()
    st = lib.plsh_sample_bins(n, sig.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                              H, s, 0, None, ctypes.byref(out))
    assert st == plsh.PLSH_ERR_INVALID
    assert out.value is None
    assert lib.plsh_last_error()


def test_bins_from_host_rejects_bad_lists(lib):
    def call(n, H, s, offsets, starts):
        off = np.asarray(offsets, dtype=np.int64)
        stt = np.asarray(starts, dtype=np.int32)
        out = ctypes.c_void_p()
        return lib.plsh_bins_from_host(
            n, H, s, off.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
            stt.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), None, ctypes.byref(out))
    assert call(8, 1, 1, [0, 3], [1, 4, 8]) == plsh.PLSH_ERR_INVALID   # first != 0
    assert call(8, 1, 1, [0, 3], [0, 4, 7]) == plsh.PLSH_ERR_INVALID   # last != n
    assert call(8, 1, 1, [0, 4], [0, 4, 4, 8]) == plsh.PLSH_ERR_INVALID  # not increasing
    assert call(8, 1, 1, [0, 1], [0]) == plsh.PLSH_ERR_INVALID          # too short


def test_attention_rejects_null_and_misaligned(lib):
    T = plsh._Tensor
    good = T(256, plsh.PLSH_BF16, 1, 1, 128, 128)
    bad_align = T(258, plsh.PLSH_BF16, 1, 1, 128, 128)
    bad_d = T(256, plsh.PLSH_BF16, 1, 1, 128, 96)
    sig = np.ones(1)
    sp = sig.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
    for q, o in ((bad_align, good), (bad_d, bad_d)):
        st = lib.plsh_alibi_exact(ctypes.byref(q), ctypes.byref(good), ctypes.byref(good),
                                  sp, 1, ctypes.byref(o), None)
        assert st == plsh.PLSH_ERR_INVALID
    st = lib.plsh_alibi_attn(ctypes.byref(good), ctypes.byref(good), ctypes.byref(good),
                             None, 1, ctypes.byref(good), None)
    assert st == plsh.PLSH_ERR_INVALID
    # GQA ratio must divide
    q3 = T(256, plsh.PLSH_BF16, 1, 3, 128, 128)
    k2 = T(256, plsh.PLSH_BF16, 1, 2, 128, 128)
    st = lib.plsh_alibi_exact(ctypes.byref(q3), ctypes.byref(k2), ctypes.byref(k2), sp, 1,
                              ctypes.byref(q3), None)
    assert st == plsh.PLSH_ERR_INVALID


def test_decode_rejects_bad_arguments(lib):
    T = plsh._Tensor
    q = T(256, plsh.PLSH_BF16, 2, 4, 1, 128)
    kv = T(256, plsh.PLSH_BF16, 2, 2, 512, 128)
    o = T(256, plsh.PLSH_BF16, 2, 4, 1, 128)

    def call(q_, k_, v_, o_):
        return lib.plsh_alibi_decode(ctypes.byref(q_), ctypes.byref(k_), ctypes.byref(v_),
                                     None, 7, ctypes.byref(o_), None)
    assert call(q, kv, kv, o) == plsh.PLSH_ERR_INVALID                       # bins NULL
    assert call(T(256, plsh.PLSH_BF16, 2, 4, 2, 128), kv, kv, o) == plsh.PLSH_ERR_INVALID
    assert call(T(258, plsh.PLSH_BF16, 2, 4, 1, 128), kv, kv, o) == plsh.PLSH_ERR_INVALID
    assert call(q, T(256, plsh.PLSH_F32, 2, 2, 512, 128), kv, o) == plsh.PLSH_ERR_INVALID
    assert call(q, T(256, plsh.PLSH_BF16, 2, 3, 512, 128),
                T(256, plsh.PLSH_BF16, 2, 3, 512, 128), o) == plsh.PLSH_ERR_INVALID
    assert call(q, kv, kv, T(256, plsh.PLSH_BF16, 2, 4, 1, 64)) == plsh.PLSH_ERR_INVALID
    assert call(q, kv, T(256, plsh.PLSH_BF16, 2, 2, 511, 128), o) == plsh.PLSH_ERR_INVALID


@pytest.mark.parametrize("n,widths,s", [(0, [4], 1), (10, [], 1), (10, [4], 0),
                                        (10, [4], 65), (10, [4, 0], 2), (10, [-3], 1)])
def test_bins_fixed_rejects_bad_arguments(lib, n, widths, s):
    wd = np.asarray(widths if widths else [1], dtype=np.int32)
    H = len(widths)
    out = ctypes.c_void_p()
    st = lib.plsh_bins_fixed(n, wd.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), H, s,
                             None, ctypes.byref(out))
    assert st == plsh.PLSH_ERR_INVALID
    assert out.value is None
    st = lib.plsh_bins_fixed(10, None, 1, 1, None, ctypes.byref(out))
    assert st == plsh.PLSH_ERR_INVALID


def test_bias_error_rejects_null_arguments(lib):
    mx, sp = ctypes.c_double(), ctypes.c_double()
    st = lib.plsh_bias_error(None, 8.0, 0, 60, 0, ctypes.byref(mx), ctypes.byref(sp), None)
    assert st == plsh.PLSH_ERR_INVALID


def test_backward_rejects_bad_arguments(lib):
    T = plsh._Tensor
    q = T(256, plsh.PLSH_BF16, 1, 2, 128, 128)
    k = T(256, plsh.PLSH_BF16, 1, 1, 128, 128)
    bad = T(256, plsh.PLSH_BF16, 1, 2, 64, 128)

    def call(dq, dk, dv):
        return lib.plsh_alibi_attn_backward(ctypes.byref(q), ctypes.byref(k), ctypes.byref(k),
                                            ctypes.byref(q), None, 1, ctypes.byref(dq),
                                            ctypes.byref(dk), ctypes.byref(dv), None)
    assert call(q, k, k) == plsh.PLSH_ERR_INVALID          # bins NULL
    assert call(bad, k, k) == plsh.PLSH_ERR_INVALID        # dQ shape
    assert call(q, q, k) == plsh.PLSH_ERR_INVALID          # dK shape
    assert call(q, k, T(256, plsh.PLSH_F32, 1, 1, 128, 128)) == plsh.PLSH_ERR_INVALID


def test_share_groups_rejects_null(lib):
    out = ctypes.c_void_p()
    assert lib.plsh_bins_share_groups(None, 4, None, ctypes.byref(out)) == plsh.PLSH_ERR_INVALID


def test_attn_path_query(lib):
    """plsh_attn_path names the kernel a call would take, launching nothing."""
    T = plsh._Tensor
    out = ctypes.c_int32(-1)

    def path(dtype, d, bins=None, causal=1):
        q = T(256, dtype, 1, 4, 1024, d)
        st = lib.plsh_attn_path(ctypes.byref(q), bins, causal, ctypes.byref(out))
        assert st == plsh.PLSH_OK
        return out.value

    assert path(plsh.PLSH_BF16, 128) == plsh.PLSH_PATH_TENSOR_CORES      # exact ALiBi
    assert path(plsh.PLSH_BF16, 64) == plsh.PLSH_PATH_TENSOR_CORES      # zero-padded to 128
    assert path(plsh.PLSH_F32, 128) == plsh.PLSH_PATH_CUDA_CORES
    assert lib.plsh_attn_path(None, None, 1, ctypes.byref(out)) == plsh.PLSH_ERR_INVALID


def test_split_parts_setting_is_validated(lib):
    assert lib.plsh_set_split_parts(-1) == plsh.PLSH_ERR_INVALID
    assert lib.plsh_set_split_parts(17) == plsh.PLSH_ERR_INVALID


def test_log_sum_exp_entry_points_reject_bad_arguments(lib):
    """The forward with log-sum-exp and the backward from saved statistics
    validate before any launch: a missing lse or O, an O of another shape."""
    T = plsh._Tensor
    q = T(256, plsh.PLSH_BF16, 1, 2, 128, 128)
    k = T(256, plsh.PLSH_BF16, 1, 1, 128, 128)
    o = T(256, plsh.PLSH_BF16, 1, 2, 128, 128)
    lse = ctypes.c_void_p(4096)
    st = lib.plsh_alibi_attn_lse(ctypes.byref(q), ctypes.byref(k), ctypes.byref(k), None, 1,
                                 ctypes.byref(o), None, None)
    assert st == plsh.PLSH_ERR_INVALID                     # lse NULL
    st = lib.plsh_alibi_attn_lse(ctypes.byref(q), ctypes.byref(k), ctypes.byref(k), None, 1,
                                 ctypes.byref(o), lse, None)
    assert st == plsh.PLSH_ERR_INVALID                     # bins NULL

    def bwd(o_, lse_):
        return lib.plsh_alibi_attn_backward_lse(
            ctypes.byref(q), ctypes.byref(k), ctypes.byref(k), o_, lse_, ctypes.byref(q), None, 1,
            ctypes.byref(q), ctypes.byref(k), ctypes.byref(k), None)
    assert bwd(None, lse) == plsh.PLSH_ERR_INVALID          # O NULL
    assert bwd(ctypes.byref(T(256, plsh.PLSH_BF16, 1, 2, 64, 128)), lse) == plsh.PLSH_ERR_INVALID
    assert bwd(ctypes.byref(o), None) == plsh.PLSH_ERR_INVALID   # lse NULL
