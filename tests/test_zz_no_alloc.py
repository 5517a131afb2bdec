"""The allocation-free forward entry point (cp_attn_forward_noalloc).

It serves callers that cannot call cudaMalloc on the compute path (for
example a plugin in a host program that owns all device memory and gives it
no allocator): they pass only inputs and outputs, and the forward workspace
comes from a fixed device array inside the library. These checks call it
through the C ABI and compare with cp_attn_forward given a caller-allocated
workspace and with the oracle, at the tolerances of the other forward tests.

Before the checked calls, another call with other inputs and the other ring
ordering runs through the same array, so a forward that read leftover
contents of the array instead of writing them first would be caught. This
file runs last so that a failure here never hides the other tests.
"""
import numpy as np
import pytest

import oracle
from workloads import Workload, bf16_bits_to_f64, make_inputs
from gpu_utils import DeviceRun, assert_close, assert_close_bf16, bf16_to_f64, cuda_ok, f32_to_f64

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]

if cuda_ok():
    import torch
    import context_causal_attention_ring_gb300 as cpa


def _noalloc(plan, run, o, lse):
    lib = cpa.load()
    return lib.cp_attn_forward_noalloc(plan.handle, run.q.data_ptr(), run.k.data_ptr(),
                                       run.v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                       torch.cuda.current_stream().cuda_stream)


def _other_call(variant, shape):
    """A forward through the array with other seeded inputs and the other
    ring ordering, leaving its contents in the array."""
    N, Hq, Hkv, d, R = shape
    other = "pass_q" if variant == "pass_kv" else "pass_kv"
    w = Workload("noalloc_other", N, Hq, Hkv, d, R, seed=7)
    plan = cpa.Plan(N, R, Hq, Hkv, d, variant=other)
    run = DeviceRun(plan, make_inputs(w))
    o = torch.empty_like(run.q)
    lse = torch.empty((Hq, plan.T_q), dtype=torch.float32, device="cuda")
    assert _noalloc(plan, run, o, lse) == 0, cpa.load().cp_attn_last_error()
    plan.sync_status()


@pytest.mark.parametrize("variant,shape", [
    ("pass_kv", (1024, 2, 1, 64, 4)),
    ("pass_q", (2048, 4, 2, 128, 4)),
])
def test_forward_noalloc_matches_forward(variant, shape):
    N, Hq, Hkv, d, R = shape
    w = Workload("noalloc", N, Hq, Hkv, d, R)
    inp = make_inputs(w)
    plan = cpa.Plan(N, R, Hq, Hkv, d, variant=variant)
    run = DeviceRun(plan, inp)
    assert plan.workspace_size(cpa.OP_FORWARD) <= cpa.load().cp_attn_forward_noalloc_capacity()
    o_ref, lse_ref, _ = run.forward()
    O_ref, L_ref = bf16_to_f64(o_ref), f32_to_f64(lse_ref)
    # the oracle on the same bf16 inputs, in the plan's rank-major row order
    pos = np.arange(N)
    O_or, L_or = oracle.attention(*(bf16_bits_to_f64(x) for x in (inp.q, inp.k, inp.v)),
                                  pos, pos)
    qidx = run.take_index(pos)
    torch.cuda.synchronize()
    free = [torch.cuda.mem_get_info()[0]]
    _other_call(variant, shape)
    for call in range(2):
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        assert _noalloc(plan, run, o, lse) == 0, cpa.load().cp_attn_last_error()
        plan.sync_status()
        got_o, got_l = bf16_to_f64(o), f32_to_f64(lse)
        assert_close_bf16(got_o, O_ref, 1e-2, f"call {call} O vs cp_attn_forward")
        assert_close(got_l, L_ref, 1e-3, f"call {call} LSE vs cp_attn_forward")
        assert_close_bf16(got_o[qidx], O_or, 1e-2, f"call {call} O vs oracle")
        assert_close(got_l[:, qidx], L_or, 1e-3, f"call {call} LSE vs oracle")
        del o, lse
        torch.cuda.synchronize()
        free.append(torch.cuda.mem_get_info()[0])
    # device memory does not grow across the checked calls (the array is part
    # of the library's device image, loaded before the first reading here)
    assert free[2] == free[1], free


def test_forward_noalloc_rejects_plans_beyond_capacity():
    plan = cpa.Plan(32768, 8, 32, 8, 128)  # needs a 512 MiB fp32 workspace
    lib = cpa.load()
    assert plan.workspace_size(cpa.OP_FORWARD) > lib.cp_attn_forward_noalloc_capacity()
    n0 = cpa.launch_count()
    st = lib.cp_attn_forward_noalloc(plan.handle, 16, 16, 16, 16, 16, None)
    assert st == 2  # CP_ATTN_ERR_SHAPE, before any launch
    assert b"workspace" in lib.cp_attn_last_error()
    assert cpa.launch_count() == n0
