"""GPU parity of the backward path (K3 preprocess, K2 backward step) against
the fp64 oracle, through the C ABI.

Gradients are produced in fp32 and compared at max-abs 1e-2 (the target's
output tolerance); delta at 2e-2. The device backward takes the forward's fp32
O for delta, as cp_attn_backward's o_f32 argument allows. The device backward consumes
the device forward's O and fp32 LSE, as a training step would; the oracle
uses its own fp64 forward.
"""
import numpy as np
import pytest

import oracle
from workloads import (WORKLOADS, Workload, bf16_bits_to_f32, bf16_bits_to_f64,
                       f32_to_bf16_bits, make_inputs, sample_rows)
from gpu_utils import DeviceRun, assert_close, cuda_ok, f32_to_f64

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]

if cuda_ok():
    import torch
    import context_causal_attention_ring_gb300 as cpa

GRAD_TOL = 1e-2


def _plan(w, variant="pass_kv", layout="zigzag", cu=None):
    return cpa.Plan(w.seq_len, w.cp, w.n_q_heads, w.n_kv_heads, w.head_dim, layout=layout,
                    variant=variant, cu_seqlens=cu, kv_prefix_len=w.kv_prefix_len)


def _grads(run):
    p = run.plan
    o, lse, run.forward_ws = run.forward()
    dq = torch.full((p.T_q, p.Hq, p.d), float("nan"), device="cuda")
    dk = torch.full((p.T_kv, p.Hkv, p.d), float("nan"), device="cuda")
    dv = torch.full_like(dk, float("nan"))
    ws = torch.empty(p.workspace_size(cpa.OP_BACKWARD), dtype=torch.uint8, device="cuda")
    # the forward leaves O in fp32 at the start of its workspace
    o_ws = run.forward_ws
    p.backward(run.q, run.k, run.v, o, lse, run.dout, dq, dk, dv, ws, o_f32=o_ws)
    p.sync_status()
    return o, lse, dq, dk, dv, ws


def _oracle_grads(inp, plan, cu):
    q, k, v, do = (bf16_bits_to_f64(x) for x in (inp.q, inp.k, inp.v, inp.dout))
    P = plan.kv_prefix_len
    N = q.shape[0]
    qp, kp = P + np.arange(N), np.arange(P + N)
    O, L = oracle.attention(q, k, v, qp, kp, cu)
    return O, L, oracle.attention_backward(q, k, v, do, O, L, qp, kp, cu)


def _check(run, cu, what):
    _, _, dq, dk, dv, ws = _grads(run)
    O, L, (dq_r, dk_r, dv_r) = _oracle_grads(run.inp, run.plan, cu)
    assert_close(run.to_natural_rows(f32_to_f64(dq)), dq_r, GRAD_TOL, what + " dQ")
    assert_close(run.to_natural_rows(f32_to_f64(dk), "kv"), dk_r, GRAD_TOL, what + " dK")
    assert_close(run.to_natural_rows(f32_to_f64(dv), "kv"), dv_r, GRAD_TOL, what + " dV")
    # delta (workspace) against the oracle's rowsum(dO * O)
    do = bf16_bits_to_f64(run.inp.dout)
    delta = f32_to_f64(ws[: run.plan.Hq * run.plan.T_q * 4].view(torch.float32)
                       .view(run.plan.Hq, run.plan.T_q))
    D_ref = np.einsum("nhd,nhd->hn", do, O)
    assert_close(run.to_natural_rows(delta, axis=1), D_ref, 2e-2, what + " delta")


def test_tiny_ring_backward():
    w = Workload("tiny_bwd", 1024, 2, 1, 64, 4, backward=True)
    run = DeviceRun(_plan(w), make_inputs(w))
    _check(run, None, "tiny")


@pytest.mark.parametrize("variant", ["pass_kv", "pass_q"])
@pytest.mark.parametrize("layout", ["zigzag", "contiguous"])
@pytest.mark.parametrize("docs", [False, True])
def test_backward_variants(variant, layout, docs):
    w = Workload("bv", 4096, 4, 2, 128, 4, backward=True)
    cu = np.array([0, 1, 130, 1000, 1023, 1024, 2500, 4096], dtype=np.int32) if docs else None
    run = DeviceRun(_plan(w, variant, layout, cu), make_inputs(w))
    _check(run, cu, f"{variant}/{layout}/docs={docs}")


@pytest.mark.parametrize("d,Hq,Hkv", [(64, 8, 1), (128, 8, 2)])
def test_backward_gqa_groups(d, Hq, Hkv):
    w = Workload("gqa", 2048, Hq, Hkv, d, 2, backward=True)
    run = DeviceRun(_plan(w), make_inputs(w))
    _check(run, None, f"gqa d={d} G={Hq // Hkv}")


def test_partial_prefill_backward():
    w = Workload("ppb", 1024, 8, 2, 128, 2, kv_prefix_len=3072, backward=True)
    run = DeviceRun(_plan(w, "pass_q"), make_inputs(w))
    _check(run, None, "partial prefill")


def test_single_step_shares():
    """One backward step adds exactly the oracle's share of that step's pairs
    (computed with the oracle's O and LSE, uploaded to the device)."""
    w = Workload("share", 2048, 4, 2, 128, 4, backward=True)
    inp = make_inputs(w)
    plan = _plan(w)
    run = DeviceRun(plan, inp)
    q, k, v, do = (bf16_bits_to_f64(x) for x in (inp.q, inp.k, inp.v, inp.dout))
    pos = np.arange(w.seq_len)
    O, L = oracle.attention(q, k, v, pos, pos)
    qn, kn = run.q_nat, run.kv_nat
    q_pos = [plan.positions(cpa.TENSOR_Q, r) for r in range(plan.R)]
    kv_pos = [plan.positions(cpa.TENSOR_KV, r) for r in range(plan.R)]
    o_dev = torch.from_numpy(O[qn].astype(np.float32)).cuda().to(torch.bfloat16)
    O_b = o_dev.float().cpu().numpy().astype(np.float64)  # the O the device sees
    lse_dev = torch.from_numpy(np.ascontiguousarray(L[:, qn], dtype=np.float32)).cuda()
    delta = torch.empty((plan.Hq, plan.T_q), dtype=torch.float32, device="cuda")
    half_ops = torch.empty(plan.half_ops_size(), dtype=torch.uint8, device="cuda")
    for t in (0, 2):
        dq = torch.empty((plan.T_q, plan.Hq, plan.d), device="cuda")
        dk = torch.empty((plan.T_kv, plan.Hkv, plan.d), device="cuda")
        dv = torch.empty_like(dk)
        plan.bwd_preprocess(run.q, run.k, run.v, o_dev, run.dout, delta, half_ops, dq, dk, dv)
        plan.step_bwd_half(t, half_ops, lse_dev, delta, dq, dk, dv)
        plan.sync_status()
        r_dq, r_dk, r_dv = oracle.ring_backward(q[qn], k[kn], v[kn], do[qn], O_b, L[:, qn],
                                                q_pos, kv_pos, steps=[t])
        msgs = []
        for name, got, ref in (("dQ", dq, r_dq), ("dK", dk, r_dk), ("dV", dv, r_dv)):
            g = f32_to_f64(got)
            err = np.abs(g - ref)
            if not err.max() <= GRAD_TOL:
                idx = np.unravel_index(np.nanargmax(err), err.shape)
                msgs.append(f"{name}: max err {err.max():.3e} at {idx} got {g[idx]:.4f} "
                            f"want {ref[idx]:.4f}; rows bad {np.unique(np.nonzero(err > GRAD_TOL)[0])[:12]}")
        assert not msgs, f"step {t}: " + " | ".join(msgs)


@pytest.mark.parametrize("d,chained,variant,docs", [(64, False, "pass_kv", False),
                                             (128, False, "pass_kv", False),
                                             (128, True, "pass_kv", False),
                                             (128, True, "pass_q", True)])
def test_step_bwd_ring_of_bf16_steps(d, chained, variant, docs):
    """cp_attn_step_bwd with bf16 q, k, v, dout and a workspace, called once
    per ring step: step 0 makes the fp16 operand copies in the workspace
    (filled with NaN patterns first), later steps reuse them; delta and the
    zeroed accumulators come from cp_attn_bwd_preprocess without copies."""
    w = Workload("stepbwd", 2048, 8, 2, d, 4, backward=True)
    cu = np.array([0, 1, 130, 1000, 1023, 1024, 1500, 2048], dtype=np.int32) if docs else None
    plan = _plan(w, variant, cu=cu)
    plan.set_chaining(chained)
    run = DeviceRun(plan, make_inputs(w))
    o, lse, fws = run.forward()
    p = plan
    delta = torch.empty((p.Hq, p.T_q), dtype=torch.float32, device="cuda")
    dq = torch.full((p.T_q, p.Hq, p.d), float("nan"), device="cuda")
    dk = torch.full((p.T_kv, p.Hkv, p.d), float("nan"), device="cuda")
    dv = torch.full_like(dk, float("nan"))
    plan.bwd_preprocess(None, None, None, o, run.dout, delta, None, dq, dk, dv, o_f32=fws)
    ws = torch.full((p.half_ops_size(),), 0xFF, dtype=torch.uint8, device="cuda")
    for t in range(p.R):
        plan.step_bwd(t, run.q, run.k, run.v, run.dout, lse, delta, dq, dk, dv, ws)
    plan.sync_status()
    _, _, (dq_r, dk_r, dv_r) = _oracle_grads(run.inp, plan, cu)
    tag = f"step_bwd ring d={d} chained={chained} {variant} docs={docs}"
    assert_close(run.to_natural_rows(f32_to_f64(dq)), dq_r, GRAD_TOL, tag + " dQ")
    assert_close(run.to_natural_rows(f32_to_f64(dk), "kv"), dk_r, GRAD_TOL, tag + " dK")
    assert_close(run.to_natural_rows(f32_to_f64(dv), "kv"), dv_r, GRAD_TOL, tag + " dV")


def test_backward_inputs_in_fp16_subnormal_range():
    """Every K element scaled by 2^-20 (exact in bf16): all of them lie below
    2^-14, where the backward's fp16 copies are subnormal and keep an
    absolute error of at most 2^-25. The gradients still meet the absolute
    1e-2 target against the oracle on the exact bf16 inputs, and dQ (which
    scales with K) matches, to 1e-2 of its size, the oracle on K rounded to
    fp16 as the documented conversion does."""
    w = Workload("small_k", 2048, 4, 2, 128, 4, backward=True)
    inp = make_inputs(w)
    k_small = bf16_bits_to_f32(inp.k) * np.float32(2.0 ** -20)
    inp.k = f32_to_bf16_bits(k_small)
    assert np.all(bf16_bits_to_f64(inp.k) == k_small.astype(np.float64))  # exact scaling
    assert np.abs(k_small).max() < 2.0 ** -14
    run = DeviceRun(_plan(w), inp)
    _, _, dq, dk, dv, _ = _grads(run)
    q, k, v, do = (bf16_bits_to_f64(x) for x in (inp.q, inp.k, inp.v, inp.dout))
    pos = np.arange(w.seq_len)
    O, L = oracle.attention(q, k, v, pos, pos)
    dq_r, dk_r, dv_r = oracle.attention_backward(q, k, v, do, O, L, pos, pos)
    DQ = run.to_natural_rows(f32_to_f64(dq))
    assert_close(DQ, dq_r, GRAD_TOL, "small K: dQ")
    assert_close(run.to_natural_rows(f32_to_f64(dk), "kv"), dk_r, GRAD_TOL, "small K: dK")
    assert_close(run.to_natural_rows(f32_to_f64(dv), "kv"), dv_r, GRAD_TOL, "small K: dV")
    # the documented conversion: K rounded to fp16 (subnormal spacing 2^-24)
    k16 = k.astype(np.float16).astype(np.float64)
    assert np.abs(k16 - k).max() <= 2.0 ** -25
    dq_16, _, _ = oracle.attention_backward(q, k16, v, do, O, L, pos, pos)
    scale_dq = np.abs(dq_16).max()
    rel16 = np.abs(DQ - dq_16).max() / scale_dq
    rel_exact = np.abs(DQ - dq_r).max() / np.abs(dq_r).max()
    assert rel16 <= 1e-2, (rel16, rel_exact)


def test_llama3_8b_layer_backward_full_head_group(oracle_pool):
    """Full-size backward in the bench's launch configuration: the whole
    forward and backward of KV head 0 and its four query heads (every row of
    dQ, every key of dK and dV), dQ of all heads at 1024 seeded rows, and dK
    and dV of all KV heads at the last 512 keys; the oracle runs on the host
    cores in parallel."""
    w = WORKLOADS["llama3_8b_layer"]
    inp = make_inputs(w)
    N, G = w.seq_len, w.group
    spec = oracle_pool.problem(inp)
    rows = sample_rows(N, 1024)
    jobs = {"head0": oracle_pool.backward_head(spec, 0),
            "dq": oracle_pool.dq_rows(spec, rows),
            "dkdv": oracle_pool.dkdv_keys(spec, N - 512, N)}
    plan = _plan(w)
    run = DeviceRun(plan, inp)
    _, _, dq, dk, dv, _ = _grads(run)
    DQ = run.to_natural_rows(f32_to_f64(dq))
    DK = run.to_natural_rows(f32_to_f64(dk), "kv")
    DV = run.to_natural_rows(f32_to_f64(dv), "kv")
    _, _, dq0, dk0, dv0 = jobs["head0"].get()
    assert_close(DQ[:, :G], dq0, GRAD_TOL, "head group 0 dQ (all rows)")
    assert_close(DK[:, 0], dk0, GRAD_TOL, "KV head 0 dK (all keys)")
    assert_close(DV[:, 0], dv0, GRAD_TOL, "KV head 0 dV (all keys)")
    assert_close(DQ[rows], jobs["dq"].get(), GRAD_TOL, "1024 sampled rows dQ")
    dk_r, dv_r = jobs["dkdv"].get()
    assert_close(DK[N - 512:], dk_r, GRAD_TOL, "last-512-key dK")
    assert_close(DV[N - 512:], dv_r, GRAD_TOL, "last-512-key dV")
    assert np.isfinite(DQ).all() and np.isfinite(DK).all() and np.isfinite(DV).all()


def test_fp16_range_violation_is_reported():
    """A finite input above the fp16 range cannot be copied exactly for the
    fp16 backward MMAs: preprocess flags CP_ATTN_ERR_RANGE."""
    w = Workload("range", 1024, 2, 1, 64, 4, backward=True)
    plan = _plan(w)
    run = DeviceRun(plan, make_inputs(w))
    k_big = run.k.clone()
    k_big[5, 0, 3] = 1.0e5
    o = torch.zeros_like(run.q)
    delta = torch.empty((plan.Hq, plan.T_q), dtype=torch.float32, device="cuda")
    half_ops = torch.empty(plan.half_ops_size(), dtype=torch.uint8, device="cuda")
    plan.bwd_preprocess(run.q, k_big, run.v, o, run.dout, delta, half_ops)
    with pytest.raises(cpa.CpAttnError) as e:
        plan.sync_status()
    assert e.value.status == 7
    plan.bwd_preprocess(run.q, run.k, run.v, o, run.dout, delta, half_ops)
    plan.sync_status()
