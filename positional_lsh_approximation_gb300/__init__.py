"""Positional LSH approximate-ALiBi attention for GB300 (sm_103a).

Thin ctypes binding of the C ABI declared in include/plsh.h: argument
marshalling only.  Every step of the hot path (hash sampling, bin records,
work queue, fused block attention, exact ALiBi) runs in the library's CUDA
kernels; torch supplies device memory and streams.  There is no CPU fallback:
if the compiled library is missing, every call raises.

Method: "Positional LSH: Binary Block Matrix Approximation for Attention with
Linear Biases" (Wolfson & Wagner), technical summary, Methodology 1-3.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

from . import build as _build_mod

__all__ = ["build", "load", "sample_bins", "bins_from_host", "bins_fixed", "bins_share_groups", "Bins", "alibi_attn",
           "alibi_attn_noalloc", "alibi_attn_host",
           "alibi_exact", "alibi_decode", "alibi_attn_backward", "bias_error", "stream_status",
           "noalloc_status", "attn_path", "set_split_parts", "set_wait_limit_ns", "PlshError",
           "library_path"]

PLSH_OK, PLSH_ERR_INVALID, PLSH_ERR_CUDA, PLSH_ERR_NOMEM, PLSH_ERR_TIMEOUT, \
    PLSH_ERR_UNSUPPORTED, PLSH_ERR_RANGE = range(7)
PLSH_F32, PLSH_BF16 = 0, 1
PLSH_PATH_CUDA_CORES, PLSH_PATH_TENSOR_CORES = 0, 1

_lock = threading.Lock()
_lib = None


class PlshError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"plsh status {status}: {message}")
        self.status = status


class _Tensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32),
                ("B", ctypes.c_int64), ("H", ctypes.c_int64),
                ("n", ctypes.c_int64), ("d", ctypes.c_int64)]


def library_path() -> str:
    return _build_mod.LIB_PATH


def build(force: bool = False) -> str:
    """Compile libplsh.so for sm_103a in-tree (nvcc)."""
    return _build_mod.build(force=force)


def load():
    """Load libplsh.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libplsh.so not built ({path}); call "
                               "positional_lsh_approximation_gb300.build()")
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I32, I64, U64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64
        D = ctypes.POINTER(ctypes.c_double)
        TP = ctypes.POINTER(_Tensor)
        sig = {
            "plsh_sample_bins": [I64, D, I32, I32, U64, P, ctypes.POINTER(P)],
            "plsh_bins_resample": [P, D, U64, P],
            "plsh_bins_from_host": [I64, I32, I32, ctypes.POINTER(I64),
                                    ctypes.POINTER(I32), P, ctypes.POINTER(P)],
            "plsh_bins_info": [P, ctypes.POINTER(I64), ctypes.POINTER(I32),
                               ctypes.POINTER(I32), ctypes.POINTER(I64), P],
            "plsh_bins_to_host": [P, ctypes.POINTER(I64), ctypes.POINTER(I32), I64, P],
            "plsh_bins_draws": [P, D, D, P],
            "plsh_bins_fixed": [I64, ctypes.POINTER(I32), I32, I32, P, ctypes.POINTER(P)],
            "plsh_bins_share_groups": [P, I32, P, ctypes.POINTER(P)],
            "plsh_bias_error": [P, ctypes.c_double, I32, I32, U64, D, D, P],
            "plsh_alibi_attn_backward": [TP, TP, TP, TP, P, I32, TP, TP, TP, P],
            "plsh_alibi_attn_backward_lse": [TP, TP, TP, TP, P, TP, P, I32, TP, TP, TP, P],
            "plsh_alibi_attn_lse": [TP, TP, TP, P, I32, TP, P, P],
            "plsh_alibi_attn": [TP, TP, TP, P, I32, TP, P],
            "plsh_alibi_attn_noalloc": [TP, TP, TP, P, I32, TP, P],
            "plsh_alibi_attn_host": [TP, TP, TP, P, I32, TP, P],
            "plsh_alibi_exact": [TP, TP, TP, D, I32, TP, P],
            "plsh_alibi_decode": [TP, TP, TP, P, I64, TP, P],
            "plsh_stream_status": [P],
            "plsh_noalloc_status": [P],
            "plsh_attn_path": [TP, P, I32, ctypes.POINTER(I32)],
            "plsh_set_wait_limit_ns": [U64],
            "plsh_set_split_parts": [I32],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        lib.plsh_bins_free.argtypes = [P]
        lib.plsh_bins_free.restype = None
        lib.plsh_status_string.argtypes = [ctypes.c_int]
        lib.plsh_status_string.restype = ctypes.c_char_p
        lib.plsh_last_error.argtypes = []
        lib.plsh_last_error.restype = ctypes.c_char_p
        _lib = lib
        return lib


def _check(status: int):
    if status != PLSH_OK:
        lib = load()
        raise PlshError(status, lib.plsh_last_error().decode())


# the current stream's raw handle without building a Stream object (the
# lookup torch.cuda.current_stream() makes costs microseconds per call)
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        if _raw_stream is not None:
            return ctypes.c_void_p(_raw_stream(torch.cuda.current_device()))
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


class Bins:
    """Owner of a plsh_bins handle (s random-binning hashes per head)."""

    def __init__(self, handle: int):
        self._h = ctypes.c_void_p(handle)

    @property
    def handle(self) -> ctypes.c_void_p:
        if not self._h:
            raise RuntimeError("bins handle already freed")
        return self._h

    def info(self, stream=None):
        n, H, s, e = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int64()
        _check(load().plsh_bins_info(self.handle, ctypes.byref(n), ctypes.byref(H),
                                     ctypes.byref(s), ctypes.byref(e), _stream(stream)))
        return n.value, H.value, s.value, e.value

    def shape(self):
        n, H, s = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
        _check(load().plsh_bins_info(self.handle, ctypes.byref(n), ctypes.byref(H),
                                     ctypes.byref(s), None, None))
        return n.value, H.value, s.value

    def resample(self, sigma, seed: int, stream=None):
        sig = _f64(sigma)
        _check(load().plsh_bins_resample(
            self.handle, sig.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
            int(seed) & (2**64 - 1), _stream(stream)))

    def to_host(self, stream=None):
        """(offsets int64[H*s+1], starts int32[...]) -- synchronises."""
        n, H, s, total = self.info(stream)
        off = np.zeros(H * s + 1, dtype=np.int64)
        st = np.zeros(total, dtype=np.int32)
        _check(load().plsh_bins_to_host(
            self.handle, off.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
            st.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), total, _stream(stream)))
        return off, st

    def draws(self, stream=None):
        n, H, s = self.shape()
        w = np.zeros(H * s)
        u = np.zeros(H * s)
        _check(load().plsh_bins_draws(self.handle,
                                      w.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                                      u.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                                      _stream(stream)))
        return w, u

    def free(self):
        if self._h:
            load().plsh_bins_free(self._h)
            self._h = ctypes.c_void_p(None)

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def sample_bins(n: int, sigma, s: int, seed: int, stream=None) -> Bins:
    """plsh_sample_bins: draw s hashes per head on the current device."""
    sig = _f64(sigma)
    out = ctypes.c_void_p()
    _check(load().plsh_sample_bins(int(n), sig.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                                   int(sig.shape[0]), int(s), int(seed) & (2**64 - 1),
                                   _stream(stream), ctypes.byref(out)))
    return Bins(out.value)


def bins_from_host(n: int, H: int, s: int, offsets, starts, stream=None) -> Bins:
    """plsh_bins_from_host: explicit boundaries (same layout as Bins.to_host)."""
    off = np.ascontiguousarray(offsets, dtype=np.int64)
    st = np.ascontiguousarray(starts, dtype=np.int32)
    out = ctypes.c_void_p()
    _check(load().plsh_bins_from_host(int(n), int(H), int(s),
                                      off.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                      st.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                      _stream(stream), ctypes.byref(out)))
    return Bins(out.value)


def bins_fixed(n: int, widths, s: int, stream=None) -> Bins:
    """plsh_bins_fixed: deterministic blocks of width widths[h] per head, s
    grids shifted by floor(t * width / s) (the fixed-blocks baseline)."""
    wd = np.ascontiguousarray(widths, dtype=np.int32)
    out = ctypes.c_void_p()
    _check(load().plsh_bins_fixed(int(n), wd.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                  int(wd.shape[0]), int(s), _stream(stream), ctypes.byref(out)))
    return Bins(out.value)


def bins_share_groups(src: Bins, Hq: int, stream=None) -> Bins:
    """plsh_bins_share_groups: head h of the result uses the hashes of head
    h // (Hq // G) of `src` (G heads)."""
    out = ctypes.c_void_p()
    _check(load().plsh_bins_share_groups(src.handle, int(Hq), _stream(stream), ctypes.byref(out)))
    return Bins(out.value)


_DT = {torch.float32: PLSH_F32, torch.bfloat16: PLSH_BF16}


def _desc(t: torch.Tensor) -> _Tensor:
    if t.dim() != 4:
        raise ValueError("tensors must be [B, H, n, d]")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    if t.dtype not in _DT:
        raise ValueError("dtype must be float32 or bfloat16")
    B, H, n, d = t.shape
    return _Tensor(t.data_ptr(), _DT[t.dtype], B, H, n, d)


def _desc_host(t: torch.Tensor) -> _Tensor:
    if t.device.type != "cpu":
        raise ValueError("host-buffer call: tensors must be in host memory")
    return _desc(t)


def alibi_attn_host(Q, K, V, bins: Bins, causal: bool, out=None, stream=None):
    """plsh_alibi_attn_host: Q, K, V (and out) in host memory, preferably
    page-locked; the copies in and out overlap the kernel.  `out` is complete
    once `stream` is synchronised."""
    if out is None:
        out = torch.empty(Q.shape, dtype=Q.dtype, pin_memory=torch.cuda.is_available())
    tq, tk, tv, to = _desc_host(Q), _desc_host(K), _desc_host(V), _desc_host(out)
    _check(load().plsh_alibi_attn_host(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv),
                                       bins.handle, int(bool(causal)), ctypes.byref(to),
                                       _stream(stream)))
    return out


def _run(fn, Q, K, V, extra, causal, out, stream):
    host = Q.device.type == "cpu"
    if host:
        # host buffers: copy in, compute on the current device, copy out
        dev = torch.device("cuda", torch.cuda.current_device())
        Qd, Kd, Vd = (x.to(dev, non_blocking=True) for x in (Q, K, V))
    else:
        Qd, Kd, Vd = Q, K, V
    Od = torch.empty_like(Qd) if (out is None or host) else out
    tq, tk, tv, to = _desc(Qd), _desc(Kd), _desc(Vd), _desc(Od)
    _check(fn(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv), extra,
              int(bool(causal)), ctypes.byref(to), _stream(stream)))
    if host:
        dst = out if out is not None else torch.empty(Q.shape, dtype=Q.dtype, pin_memory=True)
        dst.copy_(Od, non_blocking=True)
        return dst
    return Od


def alibi_attn(Q, K, V, bins: Bins, causal: bool, out=None, stream=None):
    """plsh_alibi_attn: approximate ALiBi attention T~ (Methodology 3).  Host
    tensors go through plsh_alibi_attn_host (complete once `stream` is
    synchronised)."""
    if Q.device.type == "cpu":
        return alibi_attn_host(Q, K, V, bins, causal, out, stream)
    return _run(load().plsh_alibi_attn, Q, K, V, bins.handle, causal, out, stream)


def alibi_attn_lse(Q, K, V, bins: Bins, causal: bool, out=None, lse=None, stream=None):
    """plsh_alibi_attn_lse: (O, lse), lse [B*Hq*n] fp32 the rows' base-2
    log-sum-exp (device tensors, tensor-core path)."""
    O = torch.empty_like(Q) if out is None else out
    L = torch.empty(Q.shape[0] * Q.shape[1] * Q.shape[2], dtype=torch.float32,
                    device=Q.device) if lse is None else lse
    tq, tk, tv, to = _desc(Q), _desc(K), _desc(V), _desc(O)
    _check(load().plsh_alibi_attn_lse(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv),
                                      bins.handle, int(bool(causal)), ctypes.byref(to),
                                      ctypes.c_void_p(L.data_ptr()), _stream(stream)))
    return O, L


def alibi_attn_noalloc(Q, K, V, bins: Bins, causal: bool, out=None, stream=None):
    """plsh_alibi_attn_noalloc: plsh_alibi_attn without any device allocation
    inside the call (fixed scratch compiled into the library)."""
    return _run(load().plsh_alibi_attn_noalloc, Q, K, V, bins.handle, causal, out, stream)


def alibi_exact(Q, K, V, sigma, causal: bool, out=None, stream=None):
    """plsh_alibi_exact: exact ALiBi attention T* (dense comparator)."""
    sig = _f64(sigma)
    return _run(load().plsh_alibi_exact, Q, K, V,
                sig.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), causal, out, stream)


def alibi_decode(q, K, V, bins: Bins, pos: int, out=None, stream=None):
    """plsh_alibi_decode: one decode step, row `pos` of T~ (causal) for the
    query q [B, Hq, 1, d] against the cache K, V [B, Hkv, n, d] (device
    tensors)."""
    if q.device.type == "cpu":
        raise ValueError("alibi_decode: q, K, V must be device tensors")
    o = torch.empty_like(q) if out is None else out
    tq, tk, tv, to = _desc(q), _desc(K), _desc(V), _desc(o)
    _check(load().plsh_alibi_decode(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv),
                                    bins.handle, int(pos), ctypes.byref(to), _stream(stream)))
    return o


def alibi_attn_backward(Q, K, V, dO, bins: Bins, causal: bool, stream=None):
    """plsh_alibi_attn_backward: (dQ, dK, dV) of sum(T~ * dO), device tensors."""
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    t = [_desc(x) for x in (Q, K, V, dO, dQ, dK, dV)]
    _check(load().plsh_alibi_attn_backward(
        ctypes.byref(t[0]), ctypes.byref(t[1]), ctypes.byref(t[2]), ctypes.byref(t[3]),
        bins.handle, int(bool(causal)), ctypes.byref(t[4]), ctypes.byref(t[5]),
        ctypes.byref(t[6]), _stream(stream)))
    return dQ, dK, dV


def alibi_attn_backward_lse(Q, K, V, O, lse, dO, bins: Bins, causal: bool, stream=None):
    """plsh_alibi_attn_backward_lse: (dQ, dK, dV) from the forward's O and lse
    (alibi_attn_lse), device tensors."""
    if lse.dtype != torch.float32 or lse.numel() != Q.shape[0] * Q.shape[1] * Q.shape[2]:
        raise ValueError("alibi_attn_backward_lse: lse must be float32 with B*Hq*n entries")
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    t = [_desc(x) for x in (Q, K, V, O, dO, dQ, dK, dV)]
    _check(load().plsh_alibi_attn_backward_lse(
        ctypes.byref(t[0]), ctypes.byref(t[1]), ctypes.byref(t[2]), ctypes.byref(t[3]),
        ctypes.c_void_p(lse.data_ptr()), ctypes.byref(t[4]), bins.handle, int(bool(causal)),
        ctypes.byref(t[5]), ctypes.byref(t[6]), ctypes.byref(t[7]), _stream(stream)))
    return dQ, dK, dV


def bias_error(bins: Bins, sigma: float, h: int, lanczos_iters: int = 60, seed: int = 0,
               stream=None):
    """plsh_bias_error: (||L* - M~||_max, ||L* - M~||_2) for head h."""
    mx, sp = ctypes.c_double(), ctypes.c_double()
    _check(load().plsh_bias_error(bins.handle, float(sigma), int(h), int(lanczos_iters),
                                  int(seed) & (2**64 - 1), ctypes.byref(mx), ctypes.byref(sp),
                                  _stream(stream)))
    return mx.value, sp.value


def stream_status(stream=None):
    """plsh_stream_status: synchronise and raise on device-side errors."""
    _check(load().plsh_stream_status(_stream(stream)))


def noalloc_status(stream=None):
    """plsh_noalloc_status: synchronise and raise on the error word of the
    allocation-free entry point (timeouts, V out of f16 range)."""
    _check(load().plsh_noalloc_status(_stream(stream)))


def attn_path(Q, bins=None, causal: bool = True) -> str:
    """plsh_attn_path: "tensor_cores" or "cuda_cores", the kernel that
    alibi_attn (bins given) or alibi_exact (bins None) takes for Q."""
    t = _desc(Q)
    out = ctypes.c_int32()
    _check(load().plsh_attn_path(ctypes.byref(t), bins.handle if bins is not None else None,
                                 int(bool(causal)), ctypes.byref(out)))
    return "tensor_cores" if out.value == PLSH_PATH_TENSOR_CORES else "cuda_cores"


def set_split_parts(parts: int):
    """plsh_set_split_parts: 0 automatic key-range split of long work items,
    1 never, 2..16 every item in that many parts."""
    _check(load().plsh_set_split_parts(int(parts)))


def set_wait_limit_ns(ns: int):
    _check(load().plsh_set_wait_limit_ns(int(ns)))
