"""ctypes binding of libcp_attn.so (include/cp_attn.h).

Argument marshalling only: every computation runs in the library's CUDA
kernels. Tensor arguments may be torch tensors (their ``data_ptr()`` is
passed), plain integers (device addresses) or None (NULL). Stream arguments
may be a ``torch.cuda.Stream``, an integer handle or None (the current torch
stream when torch is loaded with CUDA, else the legacy default stream).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

from . import build as _build

# enums (match include/cp_attn.h)
(OK, ERR_INVALID_ARG, ERR_SHAPE, ERR_UNSUPPORTED, ERR_CUDA, ERR_OOM, ERR_TIMEOUT,
 ERR_RANGE) = range(8)
LAYOUT_CONTIGUOUS, LAYOUT_ZIGZAG, LAYOUT_USP = 0, 1, 2
SPLIT_HEADS, GATHER_HEADS = 0, 1
PASS_KV, PASS_Q, VARIANT_AUTO = 0, 1, 2
WRITE_PARTIAL, ACCUMULATE = 0, 1
OP_FORWARD, OP_BACKWARD = 0, 1
TENSOR_Q, TENSOR_KV = 0, 1
TO_RANK_MAJOR, TO_NATURAL = 0, 1

LAYOUTS = {"contiguous": LAYOUT_CONTIGUOUS, "zigzag": LAYOUT_ZIGZAG, "usp": LAYOUT_USP}
VARIANTS = {"pass_kv": PASS_KV, "pass_q": PASS_Q, "auto": VARIANT_AUTO}
F32, BF16 = 0, 1
DTYPES = {"f32": F32, "bf16": BF16}
VARIANT_NAMES = {PASS_KV: "pass_kv", PASS_Q: "pass_q"}


class CpAttnError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"cp_attn status {status}: {msg}")
        self.status = status


class _PlanDesc(ctypes.Structure):
    _fields_ = [
        ("seq_len", ctypes.c_int64),
        ("kv_prefix_len", ctypes.c_int64),
        ("cp", ctypes.c_int),
        ("n_q_heads", ctypes.c_int),
        ("n_kv_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int),
        ("layout", ctypes.c_int),
        ("variant", ctypes.c_int),
        ("cu_seqlens", ctypes.POINTER(ctypes.c_int32)),
        ("n_docs", ctypes.c_int),
        ("softmax_scale", ctypes.c_float),
        ("window", ctypes.c_int64),
        ("a2a", ctypes.c_int),
        ("partial_dtype", ctypes.c_int),
        ("grad_dtype", ctypes.c_int),
        ("batch", ctypes.c_int),
    ]


class _DecodeDesc(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int),
        ("cp", ctypes.c_int),
        ("kv_len", ctypes.c_int64),
        ("n_q_heads", ctypes.c_int),
        ("n_kv_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int),
        ("softmax_scale", ctypes.c_float),
    ]


_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_SIG = {
    "cp_attn_plan": (_I, [ctypes.POINTER(_P), _I64, _I, _I, _I, _I, _I, _I,
                          ctypes.POINTER(ctypes.c_int32), _I]),
    "cp_attn_plan_ex": (_I, [ctypes.POINTER(_P), ctypes.POINTER(_PlanDesc)]),
    "cp_attn_select_variant": (_I, [_I64, _I64, _I, _I, ctypes.POINTER(_I)]),
    "cp_attn_head_a2a": (_I, [_I64, _I, _I64, _I, _I, _P, _P, _P]),
    "cp_attn_decode_workspace_size": (_I, [ctypes.POINTER(_DecodeDesc), ctypes.POINTER(ctypes.c_size_t)]),
    "cp_attn_decode": (_I, [ctypes.POINTER(_DecodeDesc), _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "cp_attn_plan_destroy": (None, [_P]),
    "cp_attn_plan_set_chaining": (_I, [_P, _I]),
    "cp_attn_decode_sync_status": (_I, [_P]),
    "cp_attn_decode_fp8": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "cp_attn_fp8_absmax": (_I, [_P, _I64, _P, _P]),
    "cp_attn_fp8_quantize": (_I, [_P, _I64, _I, _I, _P, _I, _P, _P, _P]),
    "cp_attn_step_fwd_fp8": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _I, _P, _P]),
    "cp_attn_forward_fp8": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "cp_attn_plan_info": (_I, [_P, ctypes.POINTER(_I64), _I]),
    "cp_attn_plan_positions": (_I, [_P, _I, _I, ctypes.POINTER(ctypes.c_int32)]),
    "cp_attn_plan_schedule": (_I, [_P, ctypes.POINTER(ctypes.c_int32)]),
    "cp_attn_plan_block_mask": (_I, [_P, ctypes.POINTER(ctypes.c_uint8)]),
    "cp_attn_plan_visible_pairs": (_I, [_P, _I, ctypes.POINTER(_I64)]),
    "cp_attn_workspace_size": (_I, [_P, _I, ctypes.POINTER(ctypes.c_size_t)]),
    "cp_attn_step_fwd": (_I, [_P, _I, _P, _P, _P, _P, _P, _I, _P, _P]),
    "cp_attn_half_ops_size": (_I, [_P, ctypes.POINTER(ctypes.c_size_t)]),
    "cp_attn_bwd_preprocess": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "cp_attn_step_bwd": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                              ctypes.c_size_t, _P]),
    "cp_attn_step_bwd_half": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _P]),
    "cp_attn_merge_lse": (_I, [_I, _I64, _I, _I, _P, _I64, _P, _I64, _P, _P, _P, _P]),
    "cp_attn_merge_lse_ex": (_I, [_I, _I64, _I, _I, _I, _P, _I64, _P, _I64, _P, _P, _P, _P]),
    "cp_attn_plan_work_list": (_I, [_P, _I, _I, _P, ctypes.POINTER(_I64)]),
    "cp_attn_forward": (_I, [_P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "cp_attn_forward_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P]),
    "cp_attn_forward_noalloc_capacity": (ctypes.c_size_t, []),
    "cp_attn_backward": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                              ctypes.c_size_t, _P]),
    "cp_attn_layout_apply": (_I, [_P, _I, _I, _P, _P, _I64, _P]),
    "cp_attn_sync_status": (_I, [_P, _P]),
    "cp_attn_selftest_wait_timeout": (_I, [_P, ctypes.c_uint64, _P]),
    "cp_attn_launch_count": (_I64, []),
    "cp_attn_last_error": (ctypes.c_char_p, []),
    "cp_attn_status_string": (ctypes.c_char_p, [_I]),
}

_lib = None


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libcp_attn.so (building it first if needed). Raises if the
    library cannot be built or loaded: there is no fallback path."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.build() if build_if_missing else _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"libcp_attn.so not found at {path}")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIG.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def exported_symbols():
    return list(_SIG)


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if hasattr(x, "is_contiguous") and not x.is_contiguous():
            raise ValueError("tensor arguments must be contiguous (the C ABI takes "
                             "dense row-major buffers)")
        return x.data_ptr()
    raise TypeError(f"cannot pass {type(x)} as a device pointer")


def _stream(s) -> Optional[int]:
    if s is None:
        try:
            import torch
            if torch.cuda.is_available() and torch.cuda.is_initialized():
                return torch.cuda.current_stream().cuda_stream
        except Exception:
            pass
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int):
    if status != OK:
        msg = load().cp_attn_last_error()
        raise CpAttnError(status, msg.decode() if msg else "")


def select_variant(n_new: int, n_cached: int, n_q_heads: int, n_kv_heads: int) -> str:
    """Pass KV or Pass Q for a prefill of n_new tokens after n_cached cached
    ones (cp_attn_select_variant)."""
    out = _I()
    _check(load().cp_attn_select_variant(int(n_new), int(n_cached), int(n_q_heads),
                                         int(n_kv_heads), ctypes.byref(out)))
    return VARIANT_NAMES[out.value]


def _decode_desc(batch, cp, kv_len, n_q_heads, n_kv_heads, head_dim, softmax_scale=0.0):
    d = _DecodeDesc()
    d.batch, d.cp, d.kv_len = int(batch), int(cp), int(kv_len)
    d.n_q_heads, d.n_kv_heads, d.head_dim = int(n_q_heads), int(n_kv_heads), int(head_dim)
    d.softmax_scale = float(softmax_scale)
    return d


def decode_workspace_size(batch, cp, kv_len, n_q_heads, n_kv_heads, head_dim) -> int:
    """Workspace bytes of cp_attn_decode."""
    out = ctypes.c_size_t()
    desc = _decode_desc(batch, cp, kv_len, n_q_heads, n_kv_heads, head_dim)
    _check(load().cp_attn_decode_workspace_size(ctypes.byref(desc), ctypes.byref(out)))
    return int(out.value)


def decode(q, k, v, o, lse, workspace, cp: int, softmax_scale: float = 0.0, stream=None):
    """One-row decode over the emulated ring (cp_attn_decode). q [B, Hq, d],
    k and v [B, kv_len, Hkv, d] bf16; o [B, Hq, d] bf16; lse [Hq, B] fp32."""
    B, Hq, d = q.shape
    kv_len, Hkv = k.shape[1], k.shape[2]
    desc = _decode_desc(B, cp, kv_len, Hq, Hkv, d, softmax_scale)
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().cp_attn_decode(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                 _ptr(lse), _ptr(workspace), int(nbytes), _stream(stream)))


def decode_fp8(q, k8, vt8, kv_scales, o, lse, workspace, cp: int, softmax_scale: float = 0.0,
               stream=None):
    """cp_attn_decode_fp8: q bf16 [B, Hq, 128]; k8 E4M3 [B*T, Hkv, 128]; vt8 E4M3
    [Hkv, 128, B*T]; kv_scales device [2] (K, V descale factors)."""
    B, Hq, d = q.shape
    Hkv = k8.shape[1]
    T = k8.shape[0] // B
    desc = _decode_desc(B, cp, T, Hq, Hkv, d, softmax_scale)
    _check(load().cp_attn_decode_fp8(ctypes.byref(desc), _ptr(q), _ptr(k8), _ptr(vt8),
                                     _ptr(kv_scales), _ptr(o), _ptr(lse), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(),
                                     _stream(stream)))


def decode_sync_status(stream=None):
    """Synchronise the stream and raise on a device-side error of the decode."""
    _check(load().cp_attn_decode_sync_status(_stream(stream)))


def head_a2a(x, out, a2a: int, direction: int, heads: Optional[int] = None, stream=None):
    """Sequence <-> head all-to-all (cp_attn_head_a2a). SPLIT_HEADS: x
    [rows, heads, d] -> out [a2a, rows, heads/a2a, d]; GATHER_HEADS: the
    inverse (x is then [a2a, rows, heads/a2a, d])."""
    if direction == SPLIT_HEADS:
        rows, heads, d = x.shape
    else:
        u, rows, hs, d = x.shape
        heads = u * hs
    _check(load().cp_attn_head_a2a(int(rows), int(heads), int(d * x.element_size()), int(a2a),
                                   int(direction), _ptr(x), _ptr(out), _stream(stream)))


class Plan:
    """Owner of a cp_attn_plan_t (host and device tables)."""

    def __init__(self, seq_len: int, cp: int, n_q_heads: int, n_kv_heads: int,
                 head_dim: int, layout: str = "zigzag", variant: str = "pass_kv",
                 cu_seqlens=None, kv_prefix_len: int = 0,
                 softmax_scale: float = 0.0, window: int = 0, a2a: int = 1,
                 partial_dtype: str = "f32", grad_dtype: str = "f32", batch: int = 1):
        lib = load()
        self._keep = None
        desc = _PlanDesc()
        desc.seq_len = int(seq_len)
        desc.kv_prefix_len = int(kv_prefix_len)
        desc.cp = int(cp)
        desc.n_q_heads = int(n_q_heads)
        desc.n_kv_heads = int(n_kv_heads)
        desc.head_dim = int(head_dim)
        desc.layout = LAYOUTS[layout] if isinstance(layout, str) else int(layout)
        desc.variant = VARIANTS[variant] if isinstance(variant, str) else int(variant)
        if cu_seqlens is not None:
            cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
            self._keep = cu
            desc.cu_seqlens = cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
            desc.n_docs = len(cu) - 1
        desc.softmax_scale = float(softmax_scale)
        desc.window = int(window)
        desc.a2a = int(a2a)
        desc.partial_dtype = DTYPES[partial_dtype] if isinstance(partial_dtype, str) else int(partial_dtype)
        desc.grad_dtype = DTYPES[grad_dtype] if isinstance(grad_dtype, str) else int(grad_dtype)
        desc.batch = int(batch)
        h = _P()
        _check(lib.cp_attn_plan_ex(ctypes.byref(h), ctypes.byref(desc)))
        self.handle = h
        info = (_I64 * 16)()
        _check(lib.cp_attn_plan_info(h, info, 16))
        (self.T_q, self.T_kv, self.n_q, self.n_kv, self.R, self.Hq, self.Hkv,
         self.d, self.n_qt, self.n_kt, self.n_docs, on_dev, var,
         self.window, self.a2a, self.batch) = [int(x) for x in info]
        self.on_device = bool(on_dev)
        self.layout = layout
        # the ring ordering in use ("auto" resolved by the library)
        self.variant = VARIANT_NAMES[var]
        self.kv_prefix_len = int(kv_prefix_len)
        self.partial_dtype = desc.partial_dtype
        self.grad_dtype = desc.grad_dtype

    def close(self):
        if getattr(self, "handle", None):
            load().cp_attn_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------ host queries
    def positions(self, kind: int, rank: int) -> np.ndarray:
        n = self.n_q if kind == TENSOR_Q else self.n_kv
        out = np.empty(n, dtype=np.int32)
        _check(load().cp_attn_plan_positions(
            self.handle, kind, rank, out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))))
        return out

    def schedule(self) -> np.ndarray:
        out = np.empty((self.R, self.R, 2), dtype=np.int32)
        _check(load().cp_attn_plan_schedule(
            self.handle, out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))))
        return out

    def block_mask(self) -> np.ndarray:
        out = np.empty((self.R, self.R, self.n_qt, self.n_kt), dtype=np.uint8)
        _check(load().cp_attn_plan_block_mask(
            self.handle, out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))))
        return out

    def visible_pairs(self, step: int = -1) -> int:
        out = _I64()
        _check(load().cp_attn_plan_visible_pairs(self.handle, step, ctypes.byref(out)))
        return int(out.value)

    def work_list(self, step: int, backward: bool = False) -> np.ndarray:
        """[n, 6] int32: q_owner, kv_owner, tile, lo, hi, n_full per item of
        the step's forward (or backward) work list, in launch order."""
        lib = load()
        n = _I64()
        _check(lib.cp_attn_plan_work_list(self.handle, step, 1 if backward else 0, None,
                                          ctypes.byref(n)))
        out = np.empty((int(n.value), 6), dtype=np.int32)
        _check(lib.cp_attn_plan_work_list(self.handle, step, 1 if backward else 0,
                                          out.ctypes.data, ctypes.byref(n)))
        return out

    def workspace_size(self, op: int) -> int:
        out = ctypes.c_size_t()
        _check(load().cp_attn_workspace_size(self.handle, op, ctypes.byref(out)))
        return int(out.value)

    # ------------------------------------------------------------ device calls
    def set_chaining(self, enable: bool):
        _check(load().cp_attn_plan_set_chaining(self.handle, 1 if enable else 0))

    def step_fwd(self, step, q, k, v, o_part, lse_part, mode, o_final=None, stream=None):
        _check(load().cp_attn_step_fwd(self.handle, step, _ptr(q), _ptr(k), _ptr(v),
                                       _ptr(o_part), _ptr(lse_part), mode, _ptr(o_final),
                                       _stream(stream)))

    def step_fwd_fp8(self, step, q8, k8, vt8, scales, o_part, lse_part, mode, o_final=None,
                     stream=None):
        _check(load().cp_attn_step_fwd_fp8(self.handle, step, _ptr(q8), _ptr(k8), _ptr(vt8),
                                           _ptr(scales), _ptr(o_part), _ptr(lse_part), mode,
                                           _ptr(o_final), _stream(stream)))

    def forward_fp8(self, q8, k8, vt8, scales, o, lse, workspace, workspace_bytes=None,
                    stream=None):
        if workspace_bytes is None:
            workspace_bytes = workspace.numel() * workspace.element_size()
        _check(load().cp_attn_forward_fp8(self.handle, _ptr(q8), _ptr(k8), _ptr(vt8),
                                          _ptr(scales), _ptr(o), _ptr(lse), _ptr(workspace),
                                          int(workspace_bytes), _stream(stream)))

    def half_ops_size(self) -> int:
        out = ctypes.c_size_t()
        _check(load().cp_attn_half_ops_size(self.handle, ctypes.byref(out)))
        return int(out.value)

    def bwd_preprocess(self, q, k, v, o, dout, delta, half_ops, dq=None, dk=None, dv=None,
                       o_f32=None, stream=None):
        _check(load().cp_attn_bwd_preprocess(self.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                             _ptr(o_f32), _ptr(dout), _ptr(delta),
                                             _ptr(half_ops), _ptr(dq), _ptr(dk), _ptr(dv),
                                             _stream(stream)))

    def step_bwd(self, step, q, k, v, dout, lse, delta, dq, dk, dv, workspace,
                 workspace_bytes=None, stream=None):
        if workspace_bytes is None:
            workspace_bytes = workspace.numel() * workspace.element_size()
        _check(load().cp_attn_step_bwd(self.handle, step, _ptr(q), _ptr(k), _ptr(v),
                                       _ptr(dout), _ptr(lse), _ptr(delta), _ptr(dq),
                                       _ptr(dk), _ptr(dv), _ptr(workspace),
                                       int(workspace_bytes), _stream(stream)))

    def step_bwd_half(self, step, half_ops, lse, delta, dq, dk, dv, stream=None):
        _check(load().cp_attn_step_bwd_half(self.handle, step, _ptr(half_ops), _ptr(lse),
                                            _ptr(delta), _ptr(dq), _ptr(dk), _ptr(dv),
                                            _stream(stream)))

    def forward(self, q, k, v, o, lse, workspace, workspace_bytes=None, stream=None):
        if workspace_bytes is None:
            workspace_bytes = workspace.numel() * workspace.element_size()
        _check(load().cp_attn_forward(self.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                      _ptr(lse), _ptr(workspace), int(workspace_bytes),
                                      _stream(stream)))

    def backward(self, q, k, v, o, lse, dout, dq, dk, dv, workspace,
                 workspace_bytes=None, o_f32=None, stream=None):
        if workspace_bytes is None:
            workspace_bytes = workspace.numel() * workspace.element_size()
        _check(load().cp_attn_backward(self.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                       _ptr(o_f32), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                                       _ptr(dv), _ptr(workspace), int(workspace_bytes),
                                       _stream(stream)))

    def layout_apply(self, kind, direction, x_in, x_out, row_bytes=None, stream=None):
        if row_bytes is None:
            row_bytes = x_in[0].numel() * x_in.element_size()
        _check(load().cp_attn_layout_apply(self.handle, kind, direction, _ptr(x_in),
                                           _ptr(x_out), int(row_bytes), _stream(stream)))

    def sync_status(self, stream=None):
        _check(load().cp_attn_sync_status(self.handle, _stream(stream)))


def fp8_absmax(x, n, amax, stream=None):
    """amax (device fp32) = max |x| over n bf16 values of x."""
    _check(load().cp_attn_fp8_absmax(_ptr(x), int(n), _ptr(amax), _stream(stream)))


def fp8_quantize(x, rows, heads, head_dim, amax, out, scale=None, transpose=False, stream=None):
    """E4M3 codes of x (bf16 [rows][heads][head_dim]) into out, same layout or
    [heads][head_dim][rows]; scale (device fp32) receives amax / 448."""
    _check(load().cp_attn_fp8_quantize(_ptr(x), int(rows), int(heads), int(head_dim), _ptr(amax),
                                       1 if transpose else 0, _ptr(out), _ptr(scale),
                                       _stream(stream)))


def merge_lse(n_parts, rows, heads, head_dim, o_parts, part_stride, lse_parts,
              lse_part_stride, o_out=None, o_out_f32=None, lse_out=None, stream=None,
              parts_dtype="f32"):
    """cp_attn_merge_lse (fp32 parts) or cp_attn_merge_lse_ex (parts_dtype
    "bf16"); part_stride in elements."""
    dt = DTYPES[parts_dtype] if isinstance(parts_dtype, str) else int(parts_dtype)
    if dt == F32:
        _check(load().cp_attn_merge_lse(n_parts, rows, heads, head_dim, _ptr(o_parts),
                                        int(part_stride), _ptr(lse_parts), int(lse_part_stride),
                                        _ptr(o_out), _ptr(o_out_f32), _ptr(lse_out),
                                        _stream(stream)))
    else:
        _check(load().cp_attn_merge_lse_ex(n_parts, rows, heads, head_dim, dt, _ptr(o_parts),
                                           int(part_stride), _ptr(lse_parts),
                                           int(lse_part_stride), _ptr(o_out), _ptr(o_out_f32),
                                           _ptr(lse_out), _stream(stream)))


def launch_count() -> int:
    return int(load().cp_attn_launch_count())


def status_string(status: int) -> str:
    return load().cp_attn_status_string(status).decode()
