"""GPU parity of the plan's element-type options (cp_attn_plan_desc
partial_dtype and grad_dtype) against the oracle, through the C ABI.

bf16 partials: in Pass Q each ring step's O partial is stored in bf16 (round
to nearest even) and the n-way merge reads it back. The oracle's ring does the
same with round_bf16 on its fp64 partials, so O is held to 1e-2 plus half a
bf16 ulp of the output and the LSE to 1e-3 (the LSE partials stay fp32). At
step level every bf16 WRITE_PARTIAL slot is checked against the oracle's
partial (1e-2 plus half an ulp), and cp_attn_merge_lse_ex over bf16 parts
against the oracle's merge of the very same values (fp32 arithmetic: 1e-4).

bf16 gradients: cp_attn_backward sums in fp32 and rounds once (K6). The
gradients are held to 1e-2 plus half a bf16 ulp of |exact| + 1e-2: the fp32
sums meet 1e-2, and rounding adds at most half an ulp of the rounded value.
dK and dV are summed in a fixed order, so their bf16 values must equal the
fp32 run's values rounded to nearest even, bit for bit; dQ (atomic sums in any
order) within one bf16 ulp plus 1e-5 of summation-order difference.
"""
import numpy as np
import pytest

import oracle
from workloads import Workload, bf16_bits_to_f64, make_inputs
from gpu_utils import (DeviceRun, assert_close, assert_close_bf16, bf16_half_ulp, bf16_to_f64,
                       cuda_ok, f32_to_f64)

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]

if cuda_ok():
    import torch
    import context_causal_attention_ring_gb300 as cpa

DOCS = [0, 1, 130, 1000, 1023, 1024, 1500, 2048]


def _rank_major(inp, run):
    q = bf16_bits_to_f64(inp.q)[run.q_nat]
    k = bf16_bits_to_f64(inp.k)[run.kv_nat]
    v = bf16_bits_to_f64(inp.v)[run.kv_nat]
    return q, k, v


def _positions(plan):
    return ([plan.positions(cpa.TENSOR_Q, r) for r in range(plan.R)],
            [plan.positions(cpa.TENSOR_KV, r) for r in range(plan.R)])


@pytest.mark.parametrize("N,Hq,Hkv,d,R,docs", [
    (2048, 8, 2, 128, 4, False),
    (2048, 4, 1, 128, 4, True),
    (1024, 4, 2, 64, 4, False),
])
def test_pass_q_forward_bf16_partials(N, Hq, Hkv, d, R, docs):
    w = Workload("p16", N, Hq, Hkv, d, R)
    inp = make_inputs(w, with_dout=False)
    cu = np.array(DOCS, dtype=np.int32) if docs else None
    plan = cpa.Plan(N, R, Hq, Hkv, d, variant="pass_q", cu_seqlens=cu, partial_dtype="bf16")
    run = DeviceRun(plan, inp)
    o, lse, _ = run.forward()
    q, k, v = _rank_major(inp, run)
    qpos, kvpos = _positions(plan)
    O_ref, L_ref = oracle.ring_forward(q, k, v, qpos, kvpos, cu, variant="pass_q",
                                       partial_dtype="bf16")
    what = f"bf16 partials N={N} {Hq}/{Hkv} d={d} docs={docs}"
    # the partials were rounded to bf16 before the merge (on both sides)
    assert_close_bf16(bf16_to_f64(o), O_ref, 1e-2, what + " O", flat_below=2.0)
    assert_close(f32_to_f64(lse), L_ref, 1e-3, what + " LSE")


def test_step_bf16_partials_and_merge_ex():
    w = Workload("pairs16", 1024, 4, 2, 128, 4)
    inp = make_inputs(w, with_dout=False)
    plan = cpa.Plan(w.seq_len, w.cp, w.n_q_heads, w.n_kv_heads, w.head_dim,
                    partial_dtype="bf16")
    run = DeviceRun(plan, inp)
    R, nq, nkv, Hq, d, T = plan.R, plan.n_q, plan.n_kv, plan.Hq, plan.d, plan.T_q
    o_part = torch.full((R, T, Hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse_part = torch.full((R, Hq, T), float("nan"), device="cuda")
    for t in range(R):
        plan.step_fwd(t, run.q, run.k, run.v, o_part, lse_part, cpa.WRITE_PARTIAL)
    plan.sync_status()
    q, k, v = _rank_major(inp, run)
    O = bf16_to_f64(o_part)
    L = f32_to_f64(lse_part)
    for t, pairs in enumerate(plan.schedule()):
        for qo, ko in pairs:
            qs = slice(qo * nq, (qo + 1) * nq)
            ks = slice(ko * nkv, (ko + 1) * nkv)
            Or, Lr = oracle.partial_attention(q[qs], k[ks], v[ks],
                                              plan.positions(cpa.TENSOR_Q, qo),
                                              plan.positions(cpa.TENSOR_KV, ko))
            assert_close_bf16(O[ko, qs], Or, 1e-2, f"bf16 O step {t} pair {qo},{ko}")
            assert_close(L[ko][:, qs], Lr, 1e-3, f"LSE step {t} pair {qo},{ko}")
    # the n-way merge over the bf16 parts, against the oracle's merge of the same values
    o_out = torch.empty((T, Hq, d), dtype=torch.bfloat16, device="cuda")
    o32 = torch.empty((T, Hq, d), dtype=torch.float32, device="cuda")
    lse_out = torch.empty((Hq, T), dtype=torch.float32, device="cuda")
    cpa.merge_lse(R, T, Hq, d, o_part, T * Hq * d, lse_part, Hq * T, o_out=o_out, o_out_f32=o32,
                  lse_out=lse_out, parts_dtype="bf16")
    torch.cuda.synchronize()
    M_ref, ML_ref = oracle.lse_merge([(O[i], L[i]) for i in range(R)])
    assert_close(f32_to_f64(o32), M_ref, 1e-4, "merge_ex O fp32")
    assert_close(f32_to_f64(lse_out), ML_ref, 1e-4, "merge_ex LSE")
    assert_close_bf16(bf16_to_f64(o_out), M_ref, 1e-4, "merge_ex O bf16")
    # an fp32 output on top of the bf16 parts is refused
    with pytest.raises(cpa.CpAttnError):
        cpa.merge_lse(R, T, Hq, d, o_part, T * Hq * d, lse_part, Hq * T,
                      o_out_f32=o_part.view(torch.float32), lse_out=lse_out, parts_dtype="bf16")


def _backward(plan, run, dtype):
    p = plan
    o, lse, ws_f = run.forward()
    dq = torch.full((p.T_q, p.Hq, p.d), float("nan"), dtype=dtype, device="cuda")
    dk = torch.full((p.T_kv, p.Hkv, p.d), float("nan"), dtype=dtype, device="cuda")
    dv = torch.full_like(dk, float("nan"))
    ws = torch.empty(p.workspace_size(cpa.OP_BACKWARD), dtype=torch.uint8, device="cuda")
    p.backward(run.q, run.k, run.v, o, lse, run.dout, dq, dk, dv, ws, o_f32=ws_f)
    p.sync_status()
    return dq, dk, dv


@pytest.mark.parametrize("N,Hq,Hkv,d,R,docs", [
    (2048, 8, 2, 128, 4, False),
    (2048, 4, 1, 128, 4, True),
    (1024, 2, 1, 64, 4, False),
])
def test_backward_bf16_gradients(N, Hq, Hkv, d, R, docs):
    w = Workload("g16", N, Hq, Hkv, d, R, backward=True)
    inp = make_inputs(w)
    cu = np.array(DOCS, dtype=np.int32) if docs else None
    p16 = cpa.Plan(N, R, Hq, Hkv, d, cu_seqlens=cu, grad_dtype="bf16")
    p32 = cpa.Plan(N, R, Hq, Hkv, d, cu_seqlens=cu)
    run = DeviceRun(p16, inp)
    g16 = _backward(p16, run, torch.bfloat16)
    g32 = _backward(p32, run, torch.float32)
    # K6: the bf16 gradients are the fp32 sums rounded to nearest even
    assert torch.equal(g16[1], g32[1].to(torch.bfloat16)), "dK finalize"
    assert torch.equal(g16[2], g32[2].to(torch.bfloat16)), "dV finalize"
    dq16 = bf16_to_f64(g16[0])
    dq32r = bf16_to_f64(g32[0].to(torch.bfloat16))
    # dQ: two fp32 runs differ by the order of the atomic sums (absolute, ~1e-9
    # here); their roundings then differ by at most one ulp plus that
    assert (np.abs(dq16 - dq32r) <= 2 * bf16_half_ulp(dq32r) + 1e-5).all(), "dQ finalize"
    # against the oracle
    q, k, v, do = (bf16_bits_to_f64(x) for x in (inp.q, inp.k, inp.v, inp.dout))
    pos = np.arange(N)
    O, L = oracle.attention(q, k, v, pos, pos, cu)
    refs = oracle.attention_backward(q, k, v, do, O, L, pos, pos, cu)
    for name, g, ref, kind in zip(("dQ", "dK", "dV"), g16, refs, ("q", "kv", "kv")):
        got = run.to_natural_rows(bf16_to_f64(g), kind)
        err = np.abs(got - ref)
        lim = 1e-2 + bf16_half_ulp(np.abs(ref) + 1e-2)
        assert (err <= lim).all(), f"bf16 {name}: max err {err.max():.3e}"
