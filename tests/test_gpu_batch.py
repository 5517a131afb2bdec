"""GPU parity of batched plans (cp_attn_plan_desc.batch: B independent
sequences, each sharded over the ring on its own) against the fp64 oracle,
through the C ABI. The oracle computes plain causal attention of each
sequence: the whole batch with one document per sequence. O (bf16) 1e-2 plus
half a bf16 ulp, LSE 1e-3, fp32 gradients 1e-2."""
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


def _setup(B, N, P, Hq, Hkv, d, R, variant, backward=False):
    w = Workload("batch", N, Hq, Hkv, d, R, kv_prefix_len=P, backward=backward)
    inp = make_inputs(w, seq_len=B * N, kv_prefix_len=B * P)
    plan = cpa.Plan(N, R, Hq, Hkv, d, variant=variant, kv_prefix_len=P, batch=B)
    L = N + P
    qpos = np.concatenate([b * L + P + np.arange(N) for b in range(B)])
    kpos = np.arange(B * L)
    cu = oracle.batch_cu_seqlens(N, B, P)
    return inp, plan, DeviceRun(plan, inp), qpos, kpos, cu


@pytest.mark.parametrize("B,N,P,Hq,Hkv,d,R,variant", [
    (3, 1024, 0, 4, 2, 128, 4, "pass_kv"),
    (3, 1024, 0, 4, 2, 128, 4, "pass_q"),
    (2, 512, 1536, 8, 2, 128, 2, "pass_q"),
    (2, 512, 0, 2, 1, 64, 2, "pass_kv"),
])
def test_batch_forward(B, N, P, Hq, Hkv, d, R, variant):
    inp, plan, run, qpos, kpos, cu = _setup(B, N, P, Hq, Hkv, d, R, variant)
    o, lse, _ = run.forward()
    q, k, v = (bf16_bits_to_f64(x) for x in (inp.q, inp.k, inp.v))
    O_ref, L_ref = oracle.attention(q, k, v, qpos, kpos, cu)
    what = f"batch B={B} N={N} P={P} {variant} d={d}"
    assert_close_bf16(run.to_natural_rows(bf16_to_f64(o)), O_ref, 1e-2, what + " O")
    assert_close(run.to_natural_rows(f32_to_f64(lse), axis=1), L_ref, 1e-3, what + " LSE")
    # each sequence on its own gives the same rows
    for b in range(B):
        ob, lb = oracle.attention(q[b * N:(b + 1) * N], k[b * (N + P):(b + 1) * (N + P)],
                                  v[b * (N + P):(b + 1) * (N + P)], P + np.arange(N),
                                  np.arange(N + P))
        assert np.allclose(ob, O_ref[b * N:(b + 1) * N], atol=1e-12)
        assert np.allclose(lb, L_ref[:, b * N:(b + 1) * N], atol=1e-12)


def test_batch_backward():
    B, N, Hq, Hkv, d, R = 2, 1024, 4, 2, 128, 4
    inp, plan, run, qpos, kpos, cu = _setup(B, N, 0, Hq, Hkv, d, R, "pass_kv", backward=True)
    o, lse, ws_f = run.forward()
    dq = torch.full((plan.T_q, Hq, d), float("nan"), device="cuda")
    dk = torch.full((plan.T_kv, Hkv, d), float("nan"), device="cuda")
    dv = torch.full_like(dk, float("nan"))
    ws = torch.empty(plan.workspace_size(cpa.OP_BACKWARD), dtype=torch.uint8, device="cuda")
    plan.backward(run.q, run.k, run.v, o, lse, run.dout, dq, dk, dv, ws, o_f32=ws_f)
    plan.sync_status()
    q, k, v, do = (bf16_bits_to_f64(x) for x in (inp.q, inp.k, inp.v, inp.dout))
    O, L = oracle.attention(q, k, v, qpos, kpos, cu)
    dq_r, dk_r, dv_r = oracle.attention_backward(q, k, v, do, O, L, qpos, kpos, cu)
    assert_close(run.to_natural_rows(f32_to_f64(dq)), dq_r, 1e-2, "batch dQ")
    assert_close(run.to_natural_rows(f32_to_f64(dk), "kv"), dk_r, 1e-2, "batch dK")
    assert_close(run.to_natural_rows(f32_to_f64(dv), "kv"), dv_r, 1e-2, "batch dV")
