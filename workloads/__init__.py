"""Seeded synthetic inputs for causal GQA attention backward.

This module only draws random numbers and lays out the per-query document-start
array. It holds none of the attention arithmetic, so that both the fp64 oracle
(``oracle/``) and the CUDA path can consume the same bits without sharing code.

Workloads follow the five shapes the pages' method is exercised on:

* ``tiny``      S=64,    H=4,  Hk=2, d=32,  N(0,1),    one document
* ``causal512`` S=512,   H=4,  Hk=2, d=32,  N(0,1),    pure causal
* ``docs2k``    S=2048,  H=16, Hk=4, d=64,  N(0,1),    packed documents, lengths U[64,1024]
* ``docs4k``    S=4096,  H=32, Hk=8, d=128, N(0,1),    packed documents, lengths U[128,4096]
* ``causal16k`` S=16384, H=32, Hk=8, d=128, N(0,0.5^2), pure causal, then RoPE backward on dQ/dK

Layouts are the pages' row-major fp32 layouts (backward_attention.wgsl,
kernel ``attention_backward`` bindings): Q/dO ``[S, H*d]``, K/V ``[S, Hk*d]``,
seg ``[S]`` uint32 where ``seg[s]`` is the first position of the document that
holds position ``s``.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

__all__ = ["Workload", "WORKLOADS", "make_seg", "make_inputs", "n_pairs"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seq_len: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    sigma: float = 1.0            # standard deviation of Q, K, V, dO
    doc_lo: int | None = None     # packed documents: length range [doc_lo, doc_hi]
    doc_hi: int | None = None
    rope: bool = False            # RoPE backward on dQ and dK after the attention backward
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def describe(self) -> str:
        s = (f"S={self.seq_len} H={self.n_heads} Hk={self.n_kv_heads} d={self.head_dim} "
             f"N(0,{self.sigma}^2)")
        if self.doc_lo is not None:
            s += f" docs~U[{self.doc_lo},{self.doc_hi}]"
        else:
            s += " causal"
        if self.rope:
            s += " +rope_bwd(dQ,dK)"
        return s


WORKLOADS: dict[str, Workload] = {
    "tiny": Workload("tiny", 64, 4, 2, 32, 1.0, seed=101),
    "causal512": Workload("causal512", 512, 4, 2, 32, 1.0, seed=202),
    "docs2k": Workload("docs2k", 2048, 16, 4, 64, 1.0, 64, 1024, seed=303),
    "docs4k": Workload("docs4k", 4096, 32, 8, 128, 1.0, 128, 4096, seed=404),
    "causal16k": Workload("causal16k", 16384, 32, 8, 128, 0.5, rope=True, seed=505),
}


def make_seg(seq_len: int, doc_lo: int | None, doc_hi: int | None,
             rng: np.random.Generator) -> np.ndarray:
    """Per-query document start.

    Document lengths are drawn uniformly in ``[doc_lo, doc_hi]`` until the
    sequence is filled; the last document is cut to fit. ``doc_lo is None``
    gives one document (``seg`` all zero, pure causal).
    """
    seg = np.zeros(seq_len, dtype=np.uint32)
    if doc_lo is None or seq_len == 0:
        return seg
    pos = 0
    while pos < seq_len:
        length = int(rng.integers(doc_lo, doc_hi + 1))
        end = min(seq_len, pos + length)
        seg[pos:end] = pos
        pos = end
    return seg


def random_seg(seq_len: int, rng: np.random.Generator, monotone: bool = True,
               max_docs: int = 8) -> np.ndarray:
    """A valid but irregular document-start array for edge-case tests.

    ``monotone=False`` draws each ``seg[s]`` independently in ``[0, s]``: the
    mask reading (``seg[s] <= j <= s``) does not need documents to be
    contiguous, and the kernels must not assume it.
    """
    if seq_len == 0:
        return np.zeros(0, dtype=np.uint32)
    if not monotone:
        return np.array([rng.integers(0, s + 1) for s in range(seq_len)], dtype=np.uint32)
    n_cuts = int(rng.integers(0, max_docs))
    cuts = np.unique(rng.integers(1, max(2, seq_len), size=n_cuts)) if seq_len > 1 else []
    seg = np.zeros(seq_len, dtype=np.uint32)
    for c in cuts:
        seg[c:] = c
    return seg


def make_inputs(w: Workload, seed: int | None = None) -> dict:
    """Q, K, V, dO (fp32, row-major) and seg (uint32) for workload ``w``."""
    rng = np.random.default_rng(w.seed if seed is None else seed)
    S, H, Hk, d = w.seq_len, w.n_heads, w.n_kv_heads, w.head_dim
    seg = make_seg(S, w.doc_lo, w.doc_hi, rng)

    def draw(rows, cols):
        x = rng.standard_normal((rows, cols), dtype=np.float32)
        if w.sigma != 1.0:
            x *= np.float32(w.sigma)
        return x

    Q = draw(S, H * d)
    K = draw(S, Hk * d)
    V = draw(S, Hk * d)
    dO = draw(S, H * d)
    return {"Q": Q, "K": K, "V": V, "dO": dO, "seg": seg, "scale": w.scale,
            "seq_len": S, "n_heads": H, "n_kv_heads": Hk, "head_dim": d}


def n_pairs(seg: np.ndarray) -> int:
    """Number of unmasked (query, key) pairs: sum over s of s - seg[s] + 1."""
    s = np.arange(len(seg), dtype=np.int64)
    return int(np.sum(s - seg.astype(np.int64) + 1))
