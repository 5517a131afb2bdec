"""The whole forward and backward, captured once into a CUDA graph and
replayed: every library call is asynchronous on the caller's stream and
allocates nothing, and the chained ring steps keep their programmatic
dependencies inside the graph. Replays must reproduce the eager results:
the forward bit for bit (no atomics), the gradients within 1e-4 (the fp32 dQ
reductions add in a different order) and both within the oracle's
tolerances."""
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


@pytest.mark.parametrize("variant", ["pass_kv", "pass_q"])
def test_forward_backward_replay_matches_eager(variant):
    w = Workload("graph", 2048, 8, 2, 128, 4, backward=True)
    inp = make_inputs(w)
    plan = cpa.Plan(w.seq_len, w.cp, w.n_q_heads, w.n_kv_heads, w.head_dim, variant=variant)
    run = DeviceRun(plan, inp)
    s = torch.cuda.Stream()
    o = torch.empty_like(run.q)
    lse = torch.empty((plan.Hq, plan.T_q), dtype=torch.float32, device="cuda")
    wsf = torch.empty(plan.workspace_size(cpa.OP_FORWARD), dtype=torch.uint8, device="cuda")
    wsb = torch.empty(plan.workspace_size(cpa.OP_BACKWARD), dtype=torch.uint8, device="cuda")
    dq = torch.empty((plan.T_q, plan.Hq, plan.d), dtype=torch.float32, device="cuda")
    dk = torch.empty((plan.T_kv, plan.Hkv, plan.d), dtype=torch.float32, device="cuda")
    dv = torch.empty_like(dk)

    def pass_():
        plan.forward(run.q, run.k, run.v, o, lse, wsf, stream=s)
        plan.backward(run.q, run.k, run.v, o, lse, run.dout, dq, dk, dv, wsb, o_f32=wsf,
                      stream=s)

    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pass_()  # eager, also the warm-up before capture
    plan.sync_status(s)
    eager = [t.clone() for t in (o, lse, dq, dk, dv)]

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pass_()
    for _ in range(2):
        for t in (o, lse, dq, dk, dv):
            t.fill_(float("nan")) if t.dtype == torch.float32 else t.zero_()
        g.replay()
        torch.cuda.synchronize()
        plan.sync_status()
        assert torch.equal(o, eager[0]) and torch.equal(lse, eager[1])
        for got, want in zip((dq, dk, dv), eager[2:]):
            assert float((got - want).abs().max()) <= 1e-4

    # and the replayed results against the oracle
    q, k, v, do = (bf16_bits_to_f64(x) for x in (inp.q, inp.k, inp.v, inp.dout))
    pos = np.arange(w.seq_len)
    O_r, L_r = oracle.attention(q, k, v, pos, pos)
    assert_close_bf16(run.to_natural_rows(bf16_to_f64(o)), O_r, 1e-2, "graph O")
    assert_close(run.to_natural_rows(f32_to_f64(lse), axis=1), L_r, 1e-3, "graph LSE")
    dq_r, dk_r, dv_r = oracle.attention_backward(q, k, v, do, O_r, L_r, pos, pos)
    assert_close(run.to_natural_rows(f32_to_f64(dq)), dq_r, 1e-2, "graph dQ")
    assert_close(run.to_natural_rows(f32_to_f64(dk), kind="kv"), dk_r, 1e-2, "graph dK")
    assert_close(run.to_natural_rows(f32_to_f64(dv), kind="kv"), dv_r, 1e-2, "graph dV")
