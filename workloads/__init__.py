"""Seeded synthetic inputs for the context-parallel ring-attention step.

This module is shared by the CPU oracle and the CUDA path. It only draws
random numbers and rounds them to bf16; it holds none of the attention
arithmetic, no chunk plan and no mask.

The workloads stand in for the models the pages measure (Llama 3.1 8B
training in "Announcing Long-Context Training on TPUs with MaxText Context
Parallelism"; Llama 3 405B prefill in "Context Parallelism for Scalable
Million-Token Inference", section "Experimental Setup & Results"). Only the
attention-head geometry is taken from those models; there are no weights
and no dataset.

Recipe:
* Q, K, V and then dO are drawn, in that order, from one
  ``numpy.random.default_rng(seed)`` stream with
  ``standard_normal(dtype=float32)``, in natural token order, rows of
  ``[tokens, heads, head_dim]``. Q and K are multiplied by ``qk_scale``
  (0.5 for the 8B-shaped and the million-token workloads).
* The fp32 values are rounded to bf16 with round-to-nearest-even. The same
  bf16 bit patterns feed the GPU and the oracle (which widens them exactly
  to fp64).
* Packed-document lengths are ``floor(exp(U(ln 1024, ln 32768)))`` drawn
  from a separate ``default_rng(seed)`` until their sum reaches the total
  token count; the last one is truncated.
* Sampled rows for the largest workloads are ``default_rng(seed).choice``
  without replacement, plus the first and the last row.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

__all__ = [
    "Workload",
    "WORKLOADS",
    "f32_to_bf16_bits",
    "bf16_bits_to_f32",
    "bf16_bits_to_f64",
    "draw_bf16",
    "make_inputs",
    "doc_lengths",
    "cu_seqlens_from_lengths",
    "sample_rows",
    "make_decode_inputs",
]


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round-to-nearest-even); return uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    bias = ((u >> 16) & 1) + 0x7FFF
    out = ((u + bias) >> 16).astype(np.uint16)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32 exactly."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float64 exactly."""
    return bf16_bits_to_f32(b).astype(np.float64)


def draw_bf16(rng: np.random.Generator, shape, scale: float = 1.0,
              chunk_rows: int = 1 << 16) -> np.ndarray:
    """Draw standard normals of ``shape`` (first axis = tokens) as bf16 bits.

    Drawn in row chunks so that large tensors never hold a float32 copy;
    the stream of numbers is the same as one call of the full shape.
    """
    shape = tuple(int(s) for s in shape)
    out = np.empty(shape, dtype=np.uint16)
    rows = shape[0]
    inner = shape[1:]
    r0 = 0
    while r0 < rows:
        r1 = min(rows, r0 + chunk_rows)
        x = rng.standard_normal((r1 - r0,) + inner, dtype=np.float32)
        if scale != 1.0:
            x *= np.float32(scale)
        out[r0:r1] = f32_to_bf16_bits(x)
        r0 = r1
    return out


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, ring size, layout and mask recipe."""

    name: str
    seq_len: int                 # new (query) tokens
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    cp: int                      # virtual ring ranks R
    kv_prefix_len: int = 0       # cached tokens before the new ones
    qk_scale: float = 1.0        # multiplier applied to Q and K draws
    docs: bool = False           # packed documents (document-causal mask)
    backward: bool = False
    variants: tuple = ("pass_kv",)
    layout: str = "zigzag"
    seed: int = 0
    note: str = ""

    @property
    def kv_len(self) -> int:
        return self.kv_prefix_len + self.seq_len

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_ring", 1024, 2, 1, 64, 4,
                 note="8 half-chunks of 128, Pass-KV forward"),
        Workload("llama3_8b_layer", 32768, 32, 8, 128, 8, qk_scale=0.5,
                 backward=True,
                 note="Llama-3-8B-shaped attention layer, Pass-KV fwd+bwd"),
        Workload("packed_docs", 131072, 32, 8, 128, 16, docs=True,
                 backward=True,
                 note="log-uniform document lengths in [1024, 32768]"),
        Workload("prefill_405b_full", 131072, 128, 8, 128, 8,
                 variants=("pass_kv", "pass_q"),
                 note="405B-shaped full prefill, both ring orderings"),
        Workload("prefill_405b_partial", 4096, 128, 8, 128, 8,
                 kv_prefix_len=126976, variants=("pass_kv", "pass_q"),
                 note="4096 new tokens after a 126976-token cached prefix"),
        Workload("million_token_group", 1048576, 8, 1, 128, 64, qk_scale=0.5,
                 backward=True,
                 note="one 8-query-head GQA group over 1M tokens"),
    ]
}


def doc_lengths(total: int, lo: int = 1024, hi: int = 32768,
                seed: int = 0) -> list:
    """Log-uniform document lengths that sum to ``total`` (last one cut)."""
    rng = np.random.default_rng(seed)
    out = []
    s = 0
    while s < total:
        L = int(np.floor(np.exp(rng.uniform(np.log(lo), np.log(hi)))))
        L = min(L, total - s)
        out.append(L)
        s += L
    return out


def cu_seqlens_from_lengths(lengths) -> np.ndarray:
    """Cumulative offsets [0, l0, l0+l1, ...] as int32."""
    cu = np.zeros(len(lengths) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return cu.astype(np.int32)


def sample_rows(n: int, k: int = 4096, seed: int = 0) -> np.ndarray:
    """Sorted distinct row indices: ``k`` seeded draws plus 0 and n-1."""
    rng = np.random.default_rng(seed)
    rows = rng.choice(n, size=min(k, n), replace=False)
    rows = np.union1d(rows, np.array([0, n - 1]))
    return np.sort(rows).astype(np.int64)


@dataclass
class Inputs:
    """bf16 bit patterns in natural token order."""

    q: np.ndarray               # [seq_len, Hq, d] uint16
    k: np.ndarray               # [kv_len, Hkv, d] uint16
    v: np.ndarray               # [kv_len, Hkv, d] uint16
    dout: Optional[np.ndarray]  # [seq_len, Hq, d] uint16
    cu_seqlens: Optional[np.ndarray] = None  # int32, over kv positions
    meta: dict = field(default_factory=dict)


def make_inputs(w: Workload, with_dout: Optional[bool] = None,
                seq_len: Optional[int] = None,
                kv_prefix_len: Optional[int] = None) -> Inputs:
    """Draw the workload's tensors. ``seq_len``/``kv_prefix_len`` override
    the sizes (used for reduced-size parity cases of the same recipe)."""
    n_new = w.seq_len if seq_len is None else int(seq_len)
    prefix = w.kv_prefix_len if kv_prefix_len is None else int(kv_prefix_len)
    n_kv = prefix + n_new
    if with_dout is None:
        with_dout = w.backward
    rng = np.random.default_rng(w.seed)
    q = draw_bf16(rng, (n_new, w.n_q_heads, w.head_dim), w.qk_scale)
    k = draw_bf16(rng, (n_kv, w.n_kv_heads, w.head_dim), w.qk_scale)
    v = draw_bf16(rng, (n_kv, w.n_kv_heads, w.head_dim), 1.0)
    dout = None
    if with_dout:
        dout = draw_bf16(rng, (n_new, w.n_q_heads, w.head_dim), 1.0)
    cu = None
    if w.docs:
        cu = cu_seqlens_from_lengths(doc_lengths(n_kv, seed=w.seed))
    return Inputs(q=q, k=k, v=v, dout=dout, cu_seqlens=cu,
                  meta=dict(workload=w.name, seq_len=n_new,
                            kv_prefix_len=prefix))


def make_decode_inputs(batch: int, kv_len: int, n_q_heads: int, n_kv_heads: int,
                       head_dim: int, seed: int = 0, qk_scale: float = 1.0):
    """Decode inputs: one new query row per sequence, q [batch, Hq, d], and
    each sequence's keys and values k, v [batch, kv_len, Hkv, d] (bf16 bits,
    standard normals; Q and K multiplied by qk_scale)."""
    rng = np.random.default_rng(seed)
    q = draw_bf16(rng, (batch, n_q_heads, head_dim), qk_scale)
    k = draw_bf16(rng, (batch * kv_len, n_kv_heads, head_dim), qk_scale).reshape(
        batch, kv_len, n_kv_heads, head_dim)
    v = draw_bf16(rng, (batch * kv_len, n_kv_heads, head_dim)).reshape(
        batch, kv_len, n_kv_heads, head_dim)
    return q, k, v
