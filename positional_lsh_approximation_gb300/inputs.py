"""Seeded synthetic inputs and the workload table.

This module holds no arithmetic of the method: it only draws Q/K/V tensors
and lists the workload shapes.  Both the CUDA path and the oracle are fed
from here, so that they see the same values.

Workload shapes borrow the models the paper's experiments use ("Positional
LSH: Binary Block Matrix Approximation for Attention with Linear Biases",
technical summary, Experimental validation: Llama-4-Scout-17B-16E,
Mistral-7B, Qwen3-0.6B; train at 8k, evaluate at 16k).  No weights or data
are used: every tensor is i.i.d. normal noise of the model's attention shape.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


def alibi_sigmas(H: int) -> np.ndarray:
    """Per-head sigma_h = 1/m_h with the ALiBi slopes m_h = 2^(-8h/H), h = 1..H.

    The summary writes the bias as L*_ij = exp(-|i-j|/sigma) (Methodology
    item 1); sigma is the reciprocal of the ALiBi slope.
    """
    h = np.arange(1, H + 1, dtype=np.float64)
    return np.exp2(8.0 * h / H)


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    n: int
    d: int
    dtype: str          # "f32" or "bf16"
    causal: bool
    s: int
    sigma: tuple = field(default=())   # per query head; empty = ALiBi slopes
    peaky_frac: float = 0.0            # fraction of token rows scaled
    peaky_scale: float = 8.0
    qkv_seed: int = 1000
    hash_seed: int = 0

    def sigmas(self) -> np.ndarray:
        if self.sigma:
            sig = np.asarray(self.sigma, dtype=np.float64)
            if sig.shape[0] == 1:
                sig = np.full(self.Hq, sig[0])
            return sig
        return alibi_sigmas(self.Hq)

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


WORKLOADS = {
    # correctness case: fp32, non-causal, fixed sigma
    "tiny": Workload("tiny", 1, 1, 1, 1024, 64, "f32", False, 8, (16.0,),
                     qkv_seed=1000),
    # one attention layer of a Mistral-7B-shaped model (GQA 32/8)
    "mistral": Workload("mistral", 1, 32, 8, 8192, 128, "bf16", True, 10,
                        qkv_seed=1001),
    # the same layer with 64-wide heads (tensor cores, zero-padded to 128)
    "mistral_d64": Workload("mistral_d64", 1, 32, 8, 8192, 64, "bf16", True, 10,
                            qkv_seed=1005),
    # Qwen3-0.6B-shaped layer, 5% of token rows of Q and K scaled by 8
    "qwen_s10": Workload("qwen_s10", 4, 16, 8, 8192, 128, "bf16", True, 10,
                         peaky_frac=0.05, qkv_seed=1002),
    "qwen_s20": Workload("qwen_s20", 4, 16, 8, 8192, 128, "bf16", True, 20,
                         peaky_frac=0.05, qkv_seed=1002),
    # length-extrapolation sweep at 16k
    **{f"sweep_s{s}": Workload(f"sweep_s{s}", 1, 32, 8, 16384, 128, "bf16",
                               True, s, qkv_seed=1003)
       for s in (1, 5, 10, 20, 40)},
    # Llama-4-Scout-shaped long context, fixed sigma
    "scout": Workload("scout", 1, 40, 8, 131072, 128, "bf16", True, 16,
                      (256.0,), qkv_seed=1004),
}


def _round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to the storage dtype (RNE) and return float32."""
    if dtype == "f32":
        return x
    if dtype == "bf16":
        u = x.view(np.uint32).astype(np.uint64)
        # round-to-nearest-even on the upper 16 bits (inputs are finite)
        lsb = (u >> 16) & 1
        u = (u + 0x7FFF + lsb) & 0xFFFF0000
        return u.astype(np.uint32).view(np.float32)
    raise ValueError(dtype)


def make_qkv(w: Workload, seed: int | None = None):
    """Q [B,Hq,n,d], K and V [B,Hkv,n,d] as float32 arrays holding values that
    are exact in w.dtype.  N(0,1) entries; with peaky_frac > 0 a seeded
    Bernoulli(peaky_frac) set of token positions per batch element (shared by
    all heads) has its Q and K rows multiplied by peaky_scale."""
    rng = np.random.default_rng(w.qkv_seed if seed is None else seed)
    q = rng.standard_normal((w.B, w.Hq, w.n, w.d), dtype=np.float32)
    k = rng.standard_normal((w.B, w.Hkv, w.n, w.d), dtype=np.float32)
    v = rng.standard_normal((w.B, w.Hkv, w.n, w.d), dtype=np.float32)
    if w.peaky_frac > 0:
        rows = rng.random((w.B, w.n)) < w.peaky_frac
        scale = np.where(rows, np.float32(w.peaky_scale), np.float32(1.0))
        q *= scale[:, None, :, None]
        k *= scale[:, None, :, None]
    return _round_to(q, w.dtype), _round_to(k, w.dtype), _round_to(v, w.dtype)


def sample_rows(w: Workload, per_head: int = 64, seed: int = 7):
    """Row subset (b, h, i) for checks at full size: per (b, h) the first and
    last 8 positions plus random ones, and every row of the lowest- and
    highest-sigma heads of batch element 0."""
    rng = np.random.default_rng(seed)
    sig = w.sigmas()
    rb, rh, ri = [], [], []
    edge = np.r_[np.arange(min(8, w.n)), np.arange(max(0, w.n - 8), w.n)]
    for b in range(w.B):
        for h in range(w.Hq):
            extra = rng.integers(0, w.n, size=max(0, per_head - edge.size))
            idx = np.unique(np.r_[edge, extra])
            rb.append(np.full(idx.size, b)); rh.append(np.full(idx.size, h))
            ri.append(idx)
    return (np.concatenate(rb).astype(np.int32),
            np.concatenate(rh).astype(np.int32),
            np.concatenate(ri).astype(np.int32)), (int(np.argmin(sig)),
                                                   int(np.argmax(sig)))
