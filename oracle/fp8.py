"""E4M3 eight-bit floating point and per-tensor FP8 quantization (NumPy).

TEST INFRASTRUCTURE ONLY (see the package docstring): no product code may
import this module.

Source: [CP-Inference] "Context Parallelism for Scalable Million-Token
Inference", "Experimental Setup & Results" (Model and Quantization): the
Llama 3 405B model of the benchmarks is quantized to FP8 throughout, for
memory and throughput. The pages name neither the FP8 format nor how the
scales are chosen. Readings:

* The format is E4M3 as defined by the OCP 8-bit floating point
  specification: one sign bit, four exponent bits with bias 7, three
  mantissa bits; exponent field 0 holds subnormals m * 2^-9; there are no
  infinities; S.1111.111 is NaN, so the largest finite value is
  1.75 * 2^8 = 448.
* One scale per tensor. With amax = max |x|, an element is stored as
  RN-even(fp32(x) * fp32(448 / amax)), clamped to +-448 ("satfinite"), and
  stands for code * fp32(amax / 448). The two ratios are single fp32
  divisions and the product a single fp32 multiplication, all rounded to
  nearest even. An all-zero tensor uses scale 1.
* The attention of an FP8 model is the same attention as before, computed
  on the dequantized values: FP8 changes the inputs, not the method.
"""
from __future__ import annotations

import numpy as np

__all__ = ["E4M3_MAX", "e4m3_decode", "e4m3_encode", "quantize_per_tensor", "dequantize",
           "pv_rounding_bound", "quantize_rows"]

E4M3_MAX = 448.0
_BIAS = 7
_MANT = 3
_MIN_NORMAL_EXP = 1 - _BIAS          # exponent of the smallest normal, 2^-6
_SUB_SPACING = 2.0 ** (_MIN_NORMAL_EXP - _MANT)   # 2^-9


def e4m3_decode(codes) -> np.ndarray:
    """Value of each E4M3 code (uint8) as float64; NaN for S.1111.111."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2((e - _BIAS).astype(np.float64))
    sub = m * _SUB_SPACING
    v = sign * np.where(e == 0, sub, normal)
    return np.where((e == 0xF) & (c & 0x7 == 0x7), np.nan, v)


def e4m3_encode(x) -> np.ndarray:
    """Nearest E4M3 code of each value (ties to even mantissa), clamped to
    +-448; NaN maps to 0x7F. Works on the exact value of x."""
    x = np.asarray(x, dtype=np.float64)
    neg = np.signbit(x)
    a = np.abs(x)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, a)
    # binade of a: a = f * 2^E with f in [0.5, 1), so floor(log2 a) = E - 1
    _, E = np.frexp(a)
    e = np.maximum(E - 1, _MIN_NORMAL_EXP)          # subnormals share 2^-6's spacing
    spacing = np.exp2((e - _MANT).astype(np.float64))
    q = np.rint(a / spacing)                          # round half to even
    v = np.minimum(q * spacing, E4M3_MAX)             # a mantissa carry moves up a binade
    # fields of the rounded value
    is_sub = v < 2.0 ** _MIN_NORMAL_EXP
    _, Ev = np.frexp(np.where(v > 0, v, 1.0))
    ev = Ev - 1
    mant_norm = np.rint((v / np.exp2(ev.astype(np.float64)) - 1.0) * 8.0)
    mant_sub = np.rint(v / _SUB_SPACING)
    efield = np.where(is_sub, 0, ev + _BIAS)
    mfield = np.where(is_sub, mant_sub, mant_norm)
    code = (efield.astype(np.int64) << 3) | mfield.astype(np.int64)
    code = code | (neg.astype(np.int64) << 7)
    code = np.where(nan, 0x7F, code)
    return code.astype(np.uint8)


def quantize_per_tensor(x, amax=None):
    """(codes, scale, inv): per-tensor E4M3 quantization of the values x
    (exact in fp32, e.g. bf16 inputs). scale = fp32(amax / 448) is the
    dequantization factor, inv = fp32(448 / amax) the quantization one.
    ``amax`` gives max |x| of the whole tensor when x is only part of it."""
    x = np.asarray(x, dtype=np.float64)
    if amax is None:
        amax = np.max(np.abs(x)) if x.size else 0.0
    amax = np.float32(amax)
    if amax == 0:
        inv = np.float32(1.0)
        scale = np.float32(1.0)
    else:
        inv = np.float32(E4M3_MAX) / amax
        scale = amax / np.float32(E4M3_MAX)
    y = x.astype(np.float32) * inv                    # one fp32 multiplication
    return e4m3_encode(y.astype(np.float64)), scale, inv


def dequantize(codes, scale) -> np.ndarray:
    """The value each code stands for: code * scale, in fp64."""
    return e4m3_decode(codes) * np.float64(scale)


def pv_rounding_bound(q, k, v, qpos, kpos, cu_seqlens=None, scale=None, *, window: int = 0,
                      p_exp: int = 8, row_block: int = 256):
    """Largest change of each output element O[n, Hq, d] that E4M3 rounding
    of the probabilities can cause when the P V product takes them in E4M3.

    The FP8 step keeps the row sums in fp32 and rounds each numerator
    P_k = 2^p_exp * 2^(s_k - m) (s in log2 units, m <= the row maximum M the
    kernel holds when it meets key k) to E4M3 before P V. A normal P_k
    (>= 2^-6) moves by at most 2^-4 P_k, which after normalisation is
    2^-4 p_k (p the softmax probability); a subnormal one by at most half
    the subnormal spacing, 2^-10, which after normalisation is at most
    2^-10 / (2^p_exp L) with L = sum_k 2^(s_k - M). A key can be subnormal
    only if 2^(s_k - M) < 2^(-6 - p_exp), and for such a key 2^-4 p_k is
    below 2^(-10 - p_exp) / L as well. So, per element,
      bound = 2^-4 sum_{k normal} p_k |v_k| + 2^(-10 - p_exp) / L * sum_{k sub} |v_k|
    where "sub" are the keys with 2^(s_k - M) < 2^(-6 - p_exp). The worst
    admissible rounding reaches it when the kernel's maximum is M throughout.
    Rows without visible keys get 0.
    """
    from .ring_attention import _as_f64, _per_head, _vis, doc_index
    q = _as_f64(q)
    n, Hq, d = q.shape
    m, Hkv, _ = np.shape(k)
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    kh_ = _per_head(k)
    vh_ = [np.abs(x) for x in _per_head(v)]
    qpos = np.asarray(qpos, dtype=np.int64)
    kpos = np.asarray(kpos, dtype=np.int64)
    qdoc = doc_index(qpos, cu_seqlens)
    kdoc = doc_index(kpos, cu_seqlens)
    B = np.zeros((n, Hq, d))
    rel = 2.0 ** -4
    sub_abs = 2.0 ** (-10 - p_exp)
    sub_below = 2.0 ** (-6 - p_exp)
    for r0 in range(0, n, row_block):
        r1 = min(n, r0 + row_block)
        vis = _vis(qpos[r0:r1], qdoc[r0:r1], kpos, kdoc, window)
        has = vis.any(axis=1)
        for h in range(Hq):
            kh = h // G
            s = scale * (q[r0:r1, h, :] @ kh_[kh].T)
            s = np.where(vis, s, -np.inf)
            mx = np.where(has, s.max(axis=1), 0.0)
            e = np.exp(s - mx[:, None])                 # 2^(s - M) in log2 terms
            L = np.where(has, e.sum(axis=1), 1.0)
            p = e / L[:, None]
            sub = (e < sub_below) & vis
            b = rel * (np.where(sub, 0.0, p) @ vh_[kh]) + \
                (sub_abs / L)[:, None] * (sub.astype(np.float64) @ vh_[kh])
            B[r0:r1, h, :] = np.where(has[:, None], b, 0.0)
    return B


def quantize_rows(x):
    """(codes, scales): E4M3 quantization of each row of x (the last axis)
    with its own scale, the per-tensor rule applied row by row (the decode
    quantizes each head's query row this way)."""
    x = np.asarray(x, dtype=np.float64)
    flat = x.reshape(-1, x.shape[-1])
    codes = np.empty(flat.shape, dtype=np.uint8)
    scales = np.empty(flat.shape[0], dtype=np.float32)
    for i in range(flat.shape[0]):
        codes[i], scales[i], _ = quantize_per_tensor(flat[i])
    return codes.reshape(x.shape), scales.reshape(x.shape[:-1])
