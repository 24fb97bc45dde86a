"""ctypes front of the fp64 C oracle (test infrastructure only).

Each function states the passage of "Positional LSH: Binary Block Matrix
Approximation for Attention with Linear Biases" (technical summary) that it
follows; the arithmetic itself lives in plsh_oracle.c.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "plsh_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libplsh_oracle.so")
_lock = threading.Lock()
_lib = None

_I64P = ctypes.POINTER(ctypes.c_int64)
_I32P = ctypes.POINTER(ctypes.c_int32)
_U32P = ctypes.POINTER(ctypes.c_uint32)
_F32P = ctypes.POINTER(ctypes.c_float)
_F64P = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile plsh_oracle.c with gcc (fp contraction off, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.oracle_philox4x32_10.argtypes = [_U32P, _U32P, _U32P]
        lib.oracle_ln64.argtypes = [ctypes.c_double]
        lib.oracle_ln64.restype = ctypes.c_double
        lib.oracle_draw.argtypes = [ctypes.c_double, ctypes.c_int32,
                                    ctypes.c_int32, ctypes.c_uint64, _F64P, _F64P]
        lib.oracle_bins_one.argtypes = [ctypes.c_int64, ctypes.c_double,
                                        ctypes.c_double, _I32P, ctypes.c_int64]
        lib.oracle_bins_one.restype = ctypes.c_int64
        lib.oracle_sample_bins.argtypes = [ctypes.c_int64, _F64P, ctypes.c_int32,
                                           ctypes.c_int32, ctypes.c_uint64, _I64P,
                                           _I32P, ctypes.c_int64, _F64P, _F64P]
        lib.oracle_sample_bins.restype = ctypes.c_int64
        rows_args = [_F32P, _F32P, _F32P, ctypes.c_int64, ctypes.c_int64,
                     ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]
        lib.oracle_plsh_attn_rows.argtypes = rows_args + [
            _I64P, _I32P, ctypes.c_int32, ctypes.c_int32, _I32P, _I32P, _I32P,
            ctypes.c_int64, _F64P]
        lib.oracle_plsh_parts_rows.argtypes = rows_args + [
            _I64P, _I32P, ctypes.c_int32, ctypes.c_int32, _I32P, _I32P, _I32P,
            ctypes.c_int64, _F64P, _F64P]
        lib.oracle_alibi_exact_rows.argtypes = rows_args + [
            _F64P, ctypes.c_int32, _I32P, _I32P, _I32P, ctypes.c_int64, _F64P]
        lib.oracle_set_threads.argtypes = [ctypes.c_int32]
        lib.oracle_max_threads.restype = ctypes.c_int32
        _lib = lib
        return lib


def _ptr(a: np.ndarray, typ):
    return a.ctypes.data_as(typ)


def philox4x32_10(ctr, key) -> np.ndarray:
    """Philox4x32-10 block (Salmon et al., SC'11): counter[4], key[2] -> 4 words."""
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    _load().oracle_philox4x32_10(_ptr(c, _U32P), _ptr(k, _U32P), _ptr(out, _U32P))
    return out


def ln64(x: float) -> float:
    """The sampler's own natural logarithm (atanh series, IEEE ops only)."""
    return float(_load().oracle_ln64(float(x)))


def draw(sigma: float, h: int, t: int, seed: int):
    """One random-binning draw (w, u): w ~ Gamma(2, scale sigma), u ~ U(0, w).

    Methodology item 2: the widths follow the Gamma law of random binning.
    """
    w = ctypes.c_double()
    u = ctypes.c_double()
    _load().oracle_draw(float(sigma), int(h), int(t), int(seed) & (2**64 - 1),
                        ctypes.byref(w), ctypes.byref(u))
    return w.value, u.value


def bins_one(n: int, w: float, u: float) -> np.ndarray:
    """Bin starts of one hash on 0..n-1 plus the terminal n.

    Methodology item 1: contiguous, non-overlapping bins of the integer
    positions.
    """
    cap = n + 2
    buf = np.zeros(cap, dtype=np.int32)
    got = _load().oracle_bins_one(int(n), float(w), float(u), _ptr(buf, _I32P), cap)
    if got < 0:
        raise RuntimeError("oracle_bins_one: capacity")
    return buf[:got].copy()


def sample_bins(n: int, sigma, s: int, seed: int, return_draws: bool = False):
    """All (h, t) hashes: offsets int64[H*s+1] and starts int32[total].

    Hash (h, t) owns starts[offsets[h*s+t] : offsets[h*s+t+1]], whose last
    entry is the terminal n.
    """
    sig = np.ascontiguousarray(sigma, dtype=np.float64)
    H = sig.shape[0]
    lib = _load()
    offsets = np.zeros(H * s + 1, dtype=np.int64)
    total = lib.oracle_sample_bins(int(n), _ptr(sig, _F64P), H, int(s),
                                   int(seed) & (2**64 - 1), _ptr(offsets, _I64P),
                                   None, 0, None, None)
    if total < 0:
        raise RuntimeError("oracle_sample_bins: count failed")
    starts = np.zeros(total, dtype=np.int32)
    w = np.zeros(H * s, dtype=np.float64)
    u = np.zeros(H * s, dtype=np.float64)
    got = lib.oracle_sample_bins(int(n), _ptr(sig, _F64P), H, int(s),
                                 int(seed) & (2**64 - 1), _ptr(offsets, _I64P),
                                 _ptr(starts, _I32P), total, _ptr(w, _F64P),
                                 _ptr(u, _F64P))
    if got != total:
        raise RuntimeError("oracle_sample_bins: fill failed")
    if return_draws:
        return offsets, starts, w, u
    return offsets, starts


def bins_fixed(n: int, widths, s: int):
    """Fixed blocks: hash t of head h has bin starts {0} and every position x
    in [1, n) with x >= o and (x - o) divisible by w, w = widths[h],
    o = floor(t * w / s); then the terminal n.  Same layout as sample_bins.

    The fixed-blocks baseline of the summary's fine-tuning experiment
    (Experimental validation), evaluated position by position.
    """
    offsets = [0]
    starts = []
    for w in (int(x) for x in widths):
        for t in range(s):
            o = t * w // s
            row = [x for x in range(n) if x == 0 or (x >= o and (x - o) % w == 0)]
            starts.extend(row + [n])
            offsets.append(len(starts))
    return np.asarray(offsets, dtype=np.int64), np.asarray(starts, dtype=np.int32)


def share_groups(offsets, starts, G: int, Hq: int, s: int):
    """Start lists for Hq heads where head h uses the s hashes of head
    h // (Hq // G) of the given lists (G heads): hashes shared across a GQA
    group.  Same layout as sample_bins."""
    group = Hq // G
    out_off = [0]
    out_st = []
    for h in range(Hq):
        g = h // group
        for t in range(s):
            row = list(starts[offsets[g * s + t]:offsets[g * s + t + 1]])
            out_st.extend(row)
            out_off.append(len(out_st))
    return np.asarray(out_off, dtype=np.int64), np.asarray(out_st, dtype=np.int32)


def bias_error(n: int, sigma: float, offsets, starts, h: int, s: int):
    """||L* - M~||_max and ||L* - M~||_2 for head h, as dense fp64 matrices.

    L*_ij = e^{-|i-j|/sigma} (Problem statement) and M~ = (1/s) sum_t M(h_t),
    M(h_t)_ij = 1 when i and j share a bin of hash t (Methodology 1-2); the
    summary's convergence experiment measures these two norms against s.
    Small n only (n x n matrices); the spectral norm of the symmetric
    difference is its largest eigenvalue magnitude.
    """
    pos = np.arange(n)
    m = np.zeros((n, n))
    for t in range(s):
        st = np.asarray(starts[offsets[h * s + t]:offsets[h * s + t + 1]])
        ids = np.searchsorted(st, pos, side="right")
        m += (ids[:, None] == ids[None, :])
    m /= s
    L = np.exp(-np.abs(pos[:, None] - pos[None, :]) / float(sigma))
    E = L - m
    return float(np.abs(E).max()), float(np.abs(np.linalg.eigvalsh(E)).max())


def plsh_attn_backward(Q, K, V, dO, offsets, starts, s: int, causal: bool):
    """Gradients (dQ, dK, dV) of the approximation with respect to its inputs,
    fp64, dense per (batch, head); small n only.

    Row i of the forward is O_i = sum_j P_ij v_j with P_ij = w_ij / sum_j w_ij,
    w_ij = c_ij e^{S_ij}, S_ij = q_i . k_j / sqrt(d) and c_ij the number of
    hashes that put i and j in one bin (Methodology 3: numerator and row sums
    averaged over the masks); c does not depend on Q, K, V.  The chain rule
    gives dV_j = sum_i P_ij dO_i, dP_ij = dO_i . v_j,
    dS_ij = P_ij (dP_ij - sum_l P_il dP_il), dQ_i = sum_j dS_ij k_j / sqrt(d),
    dK_j = sum_i dS_ij q_i / sqrt(d); a KV head collects the gradients of all
    the query heads that read it.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    dO = np.asarray(dO, dtype=np.float64)
    B, Hq, n, d = Q.shape
    Hkv = K.shape[1]
    group = Hq // Hkv
    pos = np.arange(n)
    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    for h in range(Hq):
        c = np.zeros((n, n))
        for t in range(s):
            st = np.asarray(starts[offsets[h * s + t]:offsets[h * s + t + 1]])
            ids = np.searchsorted(st, pos, side="right")
            c += (ids[:, None] == ids[None, :])
        if causal:
            c = np.tril(c)
        for b in range(B):
            q, k, v = Q[b, h], K[b, h // group], V[b, h // group]
            S = q @ k.T / math.sqrt(d)
            live = c > 0
            Sm = np.where(live, S, -np.inf)
            w = c * np.exp(Sm - Sm.max(axis=1, keepdims=True))
            P = w / w.sum(axis=1, keepdims=True)
            g = dO[b, h]
            dP = g @ v.T
            dS = P * (dP - (P * dP).sum(axis=1, keepdims=True))
            dV[b, h // group] += P.T @ g
            dQ[b, h] = dS @ k / math.sqrt(d)
            dK[b, h // group] += dS.T @ q / math.sqrt(d)
    return dQ, dK, dV


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def _rows(rows):
    rb = np.ascontiguousarray(rows[0], dtype=np.int32)
    rh = np.ascontiguousarray(rows[1], dtype=np.int32)
    ri = np.ascontiguousarray(rows[2], dtype=np.int32)
    assert rb.shape == rh.shape == ri.shape
    return rb, rh, ri


def all_rows(B: int, H: int, n: int):
    """Every (b, h, i) triple, b-major, as three int32 arrays."""
    b, h, i = np.meshgrid(np.arange(B), np.arange(H), np.arange(n), indexing="ij")
    return (b.ravel().astype(np.int32), h.ravel().astype(np.int32),
            i.ravel().astype(np.int32))


def plsh_attn_rows(Q, K, V, offsets, starts, s: int, causal: bool, rows):
    """Approximate ALiBi attention rows T~_i (fp64), per sample and per bin.

    Methodology item 3 (Theorem 2.2): short block attentions without
    positional bias; numerator and row sum are both taken over the s masks.
    Q [B,Hq,n,d], K/V [B,Hkv,n,d] (float32 holding the exact input values).
    """
    Q, K, V = _f32(Q), _f32(K), _f32(V)
    B, Hq, n, d = Q.shape
    Hkv = K.shape[1]
    off = np.ascontiguousarray(offsets, dtype=np.int64)
    st = np.ascontiguousarray(starts, dtype=np.int32)
    rb, rh, ri = _rows(rows)
    out = np.zeros((rb.shape[0], d), dtype=np.float64)
    _load().oracle_plsh_attn_rows(
        _ptr(Q, _F32P), _ptr(K, _F32P), _ptr(V, _F32P), B, Hq, Hkv, n, d,
        _ptr(off, _I64P), _ptr(st, _I32P), int(s), int(bool(causal)),
        _ptr(rb, _I32P), _ptr(rh, _I32P), _ptr(ri, _I32P), rb.shape[0],
        _ptr(out, _F64P))
    return out


def plsh_parts_rows(Q, K, V, offsets, starts, s: int, causal: bool, rows):
    """Unshifted numerator N~_i [R,d] and denominator D~_i [R] (fp64)."""
    Q, K, V = _f32(Q), _f32(K), _f32(V)
    B, Hq, n, d = Q.shape
    Hkv = K.shape[1]
    off = np.ascontiguousarray(offsets, dtype=np.int64)
    st = np.ascontiguousarray(starts, dtype=np.int32)
    rb, rh, ri = _rows(rows)
    num = np.zeros((rb.shape[0], d), dtype=np.float64)
    den = np.zeros(rb.shape[0], dtype=np.float64)
    _load().oracle_plsh_parts_rows(
        _ptr(Q, _F32P), _ptr(K, _F32P), _ptr(V, _F32P), B, Hq, Hkv, n, d,
        _ptr(off, _I64P), _ptr(st, _I32P), int(s), int(bool(causal)),
        _ptr(rb, _I32P), _ptr(rh, _I32P), _ptr(ri, _I32P), rb.shape[0],
        _ptr(num, _F64P), _ptr(den, _F64P))
    return num, den


def alibi_exact_rows(Q, K, V, sigma, causal: bool, rows):
    """Exact ALiBi attention rows T*_i (fp64): bias -|i-j|/sigma_h on the logits.

    Problem statement: the exact bias matrix costs O(n^2); L*_ij =
    exp(-|i-j|/sigma) (Methodology item 1).
    """
    Q, K, V = _f32(Q), _f32(K), _f32(V)
    B, Hq, n, d = Q.shape
    Hkv = K.shape[1]
    sig = np.ascontiguousarray(sigma, dtype=np.float64)
    assert sig.shape == (Hq,)
    rb, rh, ri = _rows(rows)
    out = np.zeros((rb.shape[0], d), dtype=np.float64)
    _load().oracle_alibi_exact_rows(
        _ptr(Q, _F32P), _ptr(K, _F32P), _ptr(V, _F32P), B, Hq, Hkv, n, d,
        _ptr(sig, _F64P), int(bool(causal)), _ptr(rb, _I32P), _ptr(rh, _I32P),
        _ptr(ri, _I32P), rb.shape[0], _ptr(out, _F64P))
    return out


def set_threads(nthreads: int) -> None:
    _load().oracle_set_threads(int(nthreads))


def max_threads() -> int:
    return int(_load().oracle_max_threads())
