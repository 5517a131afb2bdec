"""GB300 (sm_103a) context-parallel causal ring-attention step.

Python binding of libcp_attn.so; see ``include/cp_attn.h`` for the C ABI.
The library is built in-tree by ``build.build()`` and loaded on first use;
there is no CPU fallback.
"""
from ._abi import (  # noqa: F401
    ACCUMULATE, BF16, CpAttnError, F32, GATHER_HEADS, LAYOUT_CONTIGUOUS, LAYOUT_USP,
    LAYOUT_ZIGZAG, OP_BACKWARD, OP_FORWARD, PASS_KV, PASS_Q, SPLIT_HEADS, TENSOR_KV, TENSOR_Q,
    TO_NATURAL, TO_RANK_MAJOR, VARIANT_AUTO, WRITE_PARTIAL, Plan, decode, decode_fp8,
    decode_sync_status, decode_workspace_size, exported_symbols, fp8_absmax, fp8_quantize,
    head_a2a, launch_count, lib_path, load, merge_lse, select_variant, status_string,
)
