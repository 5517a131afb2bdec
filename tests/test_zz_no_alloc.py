"""The allocation-free forward entry point (cp_attn_forward_noalloc).

It serves callers that cannot call cudaMalloc (for example a plugin in a host
program that owns all device memory and gives it no allocator): they pass
only inputs and outputs, and the forward workspace comes from a fixed device
array inside the library. These checks call it through the C ABI, twice in a
row on each plan, and compare with cp_attn_forward given a caller-allocated
workspace, at the tolerances of the other forward tests. This file runs last
so that a failure here never hides the other tests.
"""
import ctypes

import numpy as np
import pytest

from workloads import Workload, make_inputs
from gpu_utils import DeviceRun, assert_close, assert_close_bf16, bf16_to_f64, cuda_ok, f32_to_f64

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]

if cuda_ok():
    import torch
    import context_causal_attention_ring_gb300 as cpa


def _noalloc(plan, run, o, lse):
    lib = cpa.load()
    st = lib.cp_attn_forward_noalloc(plan.handle, run.q.data_ptr(), run.k.data_ptr(),
                                     run.v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream)
    return st


@pytest.mark.parametrize("variant,shape", [
    ("pass_kv", (1024, 2, 1, 64, 4)),
    ("pass_q", (2048, 4, 2, 128, 4)),
])
def test_forward_noalloc_matches_forward(variant, shape):
    N, Hq, Hkv, d, R = shape
    w = Workload("noalloc", N, Hq, Hkv, d, R)
    plan = cpa.Plan(N, R, Hq, Hkv, d, variant=variant)
    run = DeviceRun(plan, make_inputs(w))
    assert plan.workspace_size(cpa.OP_FORWARD) <= cpa.load().cp_attn_forward_noalloc_capacity()
    o_ref, lse_ref, _ = run.forward()
    O_ref, L_ref = bf16_to_f64(o_ref), f32_to_f64(lse_ref)
    free_after = []
    for call in range(2):
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        assert _noalloc(plan, run, o, lse) == 0, cpa.load().cp_attn_last_error()
        plan.sync_status()
        assert_close_bf16(bf16_to_f64(o), O_ref, 1e-2, f"call {call} O")
        assert_close(f32_to_f64(lse), L_ref, 1e-3, f"call {call} LSE")
        free_after.append(torch.cuda.mem_get_info()[0])
    # no device memory was taken by the second call
    assert free_after[1] == free_after[0]


def test_forward_noalloc_rejects_plans_beyond_capacity():
    plan = cpa.Plan(32768, 8, 32, 8, 128)  # needs a 512 MiB fp32 workspace
    lib = cpa.load()
    assert plan.workspace_size(cpa.OP_FORWARD) > lib.cp_attn_forward_noalloc_capacity()
    n0 = cpa.launch_count()
    st = lib.cp_attn_forward_noalloc(plan.handle, 16, 16, 16, 16, 16, None)
    assert st == 2  # CP_ATTN_ERR_SHAPE, before any launch
    assert b"workspace" in lib.cp_attn_last_error()
    assert cpa.launch_count() == n0
