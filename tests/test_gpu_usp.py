"""GPU parity of the Ulysses / USP composition ("Announcing Long-Context
Training on TPUs with MaxText Context Parallelism", sections "All-to-All
(Ulysses)" and "A2A + P2P (USP)") against the fp64 oracle's monolithic
attention, through the C ABI: natural order -> pooled order (the plan's
layout permutation), head all-to-all (kernel K7), a ring of R steps per head
group over a2a-times longer chunks, all-to-all back. The all-to-all itself
is checked bit for bit against the oracle's head split. Tolerances as in
the other parity tests."""
import numpy as np
import pytest

import oracle
from workloads import Workload, bf16_bits_to_f64, make_inputs
from gpu_utils import assert_close, assert_close_bf16, bf16_to_f64, cuda_ok, f32_to_f64, to_dev

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]

if cuda_ok():
    import torch
    import context_causal_attention_ring_gb300 as cpa


def test_head_a2a_bit_exact():
    rng = np.random.default_rng(5)
    for rows, heads, d, U, dt in ((300, 8, 128, 2, torch.bfloat16), (64, 32, 64, 4, torch.bfloat16),
                                  (129, 8, 128, 8, torch.float32)):
        x = torch.from_numpy(rng.standard_normal((rows, heads, d)).astype(np.float32)).to(dt).cuda()
        y = torch.empty((U, rows, heads // U, d), dtype=dt, device="cuda")
        cpa.head_a2a(x, y, U, cpa.SPLIT_HEADS)
        want = oracle.head_split(x.float().cpu().numpy(), U)
        assert np.array_equal(y.float().cpu().numpy(), want)
        z = torch.empty_like(x)
        cpa.head_a2a(y, z, U, cpa.GATHER_HEADS)
        assert torch.equal(z, x)


def _usp_run(w, R, U, variant, cu):
    """Forward and backward of the USP pipeline; returns natural-order O, LSE,
    dQ, dK, dV (fp64 numpy) and the plan."""
    inp = make_inputs(w)
    Hq, Hkv, d = w.n_q_heads, w.n_kv_heads, w.head_dim
    hs_q, hs_kv = Hq // U, Hkv // U
    plan = cpa.Plan(w.seq_len, R, hs_q, hs_kv, d, layout="usp", a2a=U, variant=variant,
                    cu_seqlens=cu)
    T = plan.T_q

    def pooled(bits, heads, kind):
        x = to_dev(bits)
        y = torch.empty_like(x)
        plan.layout_apply(kind, cpa.TO_RANK_MAJOR, x, y, row_bytes=heads * d * 2)
        s = torch.empty((U, T, heads // U, d), dtype=x.dtype, device="cuda")
        cpa.head_a2a(y, s, U, cpa.SPLIT_HEADS)
        return s

    qs = pooled(inp.q, Hq, cpa.TENSOR_Q)
    ks = pooled(inp.k, Hkv, cpa.TENSOR_KV)
    vs = pooled(inp.v, Hkv, cpa.TENSOR_KV)
    dos = pooled(inp.dout, Hq, cpa.TENSOR_Q)
    os_ = torch.empty_like(qs)
    lse = torch.empty((Hq, T), dtype=torch.float32, device="cuda")   # [U][hs][T] == [Hq][T]
    dqs = torch.empty((U, T, hs_q, d), device="cuda")
    dks = torch.empty((U, T, hs_kv, d), device="cuda")
    dvs = torch.empty_like(dks)
    wsf = torch.empty(plan.workspace_size(cpa.OP_FORWARD), dtype=torch.uint8, device="cuda")
    wsb = torch.empty(plan.workspace_size(cpa.OP_BACKWARD), dtype=torch.uint8, device="cuda")
    for u in range(U):
        lu = lse[u * hs_q:(u + 1) * hs_q]
        plan.forward(qs[u], ks[u], vs[u], os_[u], lu, wsf)
        plan.backward(qs[u], ks[u], vs[u], os_[u], lu, dos[u], dqs[u], dks[u], dvs[u], wsb,
                      o_f32=wsf)
    plan.sync_status()

    def back(s, heads, kind, dtype):
        g = torch.empty((T, heads, d), dtype=dtype, device="cuda")
        cpa.head_a2a(s, g, U, cpa.GATHER_HEADS)
        n = torch.empty_like(g)
        plan.layout_apply(kind, cpa.TO_NATURAL, g, n, row_bytes=heads * d * g.element_size())
        return n

    o = bf16_to_f64(back(os_, Hq, cpa.TENSOR_Q, torch.bfloat16))
    perm = np.concatenate([plan.positions(cpa.TENSOR_Q, r) for r in range(R)])
    L = np.empty((Hq, T))
    L[:, perm] = f32_to_f64(lse)
    dq = f32_to_f64(back(dqs, Hq, cpa.TENSOR_Q, torch.float32))
    dk = f32_to_f64(back(dks, Hkv, cpa.TENSOR_KV, torch.float32))
    dv = f32_to_f64(back(dvs, Hkv, cpa.TENSOR_KV, torch.float32))
    return inp, o, L, dq, dk, dv


@pytest.mark.parametrize("R,U,variant", [(2, 2, "pass_kv"), (2, 4, "pass_q"), (1, 8, "pass_kv"),
                                         (4, 2, "pass_kv")])
def test_usp_pipeline_forward_backward(R, U, variant):
    w = Workload("usp", 4096, 16, 8, 128, R, backward=True, seed=21)
    cu = np.array([0, 1500, 4096], dtype=np.int32)
    inp, O, L, dq, dk, dv = _usp_run(w, R, U, variant, cu)
    q, k, v, do = (bf16_bits_to_f64(x) for x in (inp.q, inp.k, inp.v, inp.dout))
    pos = np.arange(w.seq_len)
    Or, Lr = oracle.attention(q, k, v, pos, pos, cu)
    dq_r, dk_r, dv_r = oracle.attention_backward(q, k, v, do, Or, Lr, pos, pos, cu)
    tag = f"USP R={R} a2a={U} {variant}"
    assert_close_bf16(O, Or, 1e-2, tag + " O")
    assert_close(L, Lr, 1e-3, tag + " LSE")
    assert_close(dq, dq_r, 1e-2, tag + " dQ")
    assert_close(dk, dk_r, 1e-2, tag + " dK")
    assert_close(dv, dv_r, 1e-2, tag + " dV")
