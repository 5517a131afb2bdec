"""GPU parity of sliding-window masks (the window layers of models that mix
sliding-window and global layers, "Announcing Long-Context Training on TPUs
with MaxText Context Parallelism", section "What's next") against the fp64
oracle: forward (O, LSE) and backward (dQ, dK, dV) through the C ABI, for
windows shorter than a tile, exactly one tile, spanning several tiles and
crossing rank boundaries, with documents, a cached prefix, both ring
orderings and both head dimensions. Same tolerances as the unwindowed
parity tests (1e-2 on outputs and gradients, 1e-3 on LSE)."""
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

GRAD_TOL = 1e-2


def _run(w, W, variant="pass_kv", cu=None, backward=True):
    inp = make_inputs(w, with_dout=backward)
    plan = cpa.Plan(w.seq_len, w.cp, w.n_q_heads, w.n_kv_heads, w.head_dim, variant=variant,
                    cu_seqlens=cu, kv_prefix_len=w.kv_prefix_len, window=W)
    run = DeviceRun(plan, inp)
    q, k, v = (bf16_bits_to_f64(x) for x in (inp.q, inp.k, inp.v))
    P, N = w.kv_prefix_len, w.seq_len
    qp, kp = P + np.arange(N), np.arange(P + N)
    O_r, L_r = oracle.attention(q, k, v, qp, kp, cu, window=W)
    o, lse, ws = run.forward()
    plan.sync_status()
    tag = f"W={W} {variant}"
    assert_close_bf16(run.to_natural_rows(bf16_to_f64(o)), O_r, 1e-2, tag + " O")
    assert_close(run.to_natural_rows(f32_to_f64(lse), axis=1), L_r, 1e-3, tag + " LSE")
    if not backward:
        return
    do = bf16_bits_to_f64(inp.dout)
    dq_r, dk_r, dv_r = oracle.attention_backward(q, k, v, do, O_r, L_r, qp, kp, cu, window=W)
    dq = torch.empty((plan.T_q, plan.Hq, plan.d), device="cuda")
    dk = torch.empty((plan.T_kv, plan.Hkv, plan.d), device="cuda")
    dv = torch.empty_like(dk)
    wsb = torch.empty(plan.workspace_size(cpa.OP_BACKWARD), dtype=torch.uint8, device="cuda")
    plan.backward(run.q, run.k, run.v, o, lse, run.dout, dq, dk, dv, wsb, o_f32=ws)
    plan.sync_status()
    assert_close(run.to_natural_rows(f32_to_f64(dq)), dq_r, GRAD_TOL, tag + " dQ")
    assert_close(run.to_natural_rows(f32_to_f64(dk), "kv"), dk_r, GRAD_TOL, tag + " dK")
    assert_close(run.to_natural_rows(f32_to_f64(dv), "kv"), dv_r, GRAD_TOL, tag + " dV")


@pytest.mark.parametrize("W", [1, 100, 128, 300, 700])
def test_window_d64_forward_backward(W):
    w = Workload("win_d64", 1024, 2, 1, 64, 4, backward=True, seed=11)
    _run(w, W)


@pytest.mark.parametrize("W", [37, 128, 1000])
@pytest.mark.parametrize("variant", ["pass_kv", "pass_q"])
def test_window_d128_documents(W, variant):
    w = Workload("win_d128", 4096, 8, 2, 128, 2, backward=True, seed=12)
    cu = np.array([0, 700, 701, 2049, 4096], dtype=np.int32)
    _run(w, W, variant, cu, backward=(variant == "pass_kv"))


@pytest.mark.parametrize("variant", ["pass_kv", "pass_q"])
def test_window_partial_prefill(variant):
    w = Workload("win_prefix", 1024, 8, 1, 128, 2, kv_prefix_len=3072, seed=13)
    _run(w, 1500, variant, backward=False)
