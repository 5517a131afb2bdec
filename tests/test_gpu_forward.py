"""GPU parity of the forward path (kernels K1 step forward, K4 merge, K5
layout) against the fp64 oracle, through the C ABI.

Tolerances (from the target: max-abs 1e-2 on outputs, 1e-3 on LSE):
* fp32 partial outputs and fp32 running accumulators: max-abs 1e-2;
* bf16 outputs: 1e-2 plus half a bf16 ulp of the oracle value (the rounding
  of the stored result itself, which alone exceeds 1e-2 when |O| >= 4);
* LSE (fp32, natural log): max-abs 1e-3; rows with no visible key must be
  -inf on both sides, with O exactly 0.
"""
import math

import numpy as np
import pytest

import oracle
from workloads import WORKLOADS, Workload, bf16_bits_to_f64, make_inputs, sample_rows
from gpu_utils import (DeviceRun, assert_close, assert_close_bf16, bf16_to_f64,
                       cuda_ok, f32_to_f64)

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]

if cuda_ok():
    import torch
    import context_causal_attention_ring_gb300 as cpa


def _plan(w: Workload, variant="pass_kv", layout="zigzag", cu=None, seq_len=None,
          prefix=None):
    N = w.seq_len if seq_len is None else seq_len
    P = w.kv_prefix_len if prefix is None else prefix
    return cpa.Plan(N, w.cp, w.n_q_heads, w.n_kv_heads, w.head_dim, layout=layout,
                    variant=variant, cu_seqlens=cu, kv_prefix_len=P)


def _oracle_full(inp, plan, cu):
    q = bf16_bits_to_f64(inp.q)
    k = bf16_bits_to_f64(inp.k)
    v = bf16_bits_to_f64(inp.v)
    P = plan.kv_prefix_len
    N = q.shape[0]
    return oracle.attention(q, k, v, P + np.arange(N), np.arange(P + N), cu)


def _check_forward(run, O_ref, L_ref, what):
    o, lse, _ = run.forward()
    O = run.to_natural_rows(bf16_to_f64(o))
    L = run.to_natural_rows(f32_to_f64(lse), axis=1)
    e_o = assert_close_bf16(O, O_ref, 1e-2, what + " O")
    e_l = assert_close(L, L_ref, 1e-3, what + " LSE")
    return e_o, e_l


def test_tiny_ring_forward():
    w = WORKLOADS["tiny_ring"]
    inp = make_inputs(w)
    plan = _plan(w)
    run = DeviceRun(plan, inp)
    O_ref, L_ref = _oracle_full(inp, plan, None)
    _check_forward(run, O_ref, L_ref, "tiny_ring")


@pytest.mark.parametrize("d,Hq,Hkv", [(64, 2, 1), (128, 4, 2)])
def test_step_partials_each_pair(d, Hq, Hkv):
    """WRITE_PARTIAL: every (q_owner, kv_owner) partial of every step equals
    the oracle's partial attention of that pair, including rows that see no
    key (O = 0, LSE = -inf)."""
    w = Workload("pairs", 1024, Hq, Hkv, d, 4)
    inp = make_inputs(w)
    plan = _plan(w)
    run = DeviceRun(plan, inp)
    R, nq, nkv = plan.R, plan.n_q, plan.n_kv
    q = bf16_bits_to_f64(inp.q)[run.q_nat]
    k = bf16_bits_to_f64(inp.k)[run.kv_nat]
    v = bf16_bits_to_f64(inp.v)[run.kv_nat]
    o_part = torch.full((R, plan.T_q, Hq, d), float("nan"), device="cuda")
    lse_part = torch.full((R, Hq, plan.T_q), float("nan"), device="cuda")
    sched = plan.schedule()
    for t in range(R):
        plan.step_fwd(t, run.q, run.k, run.v, o_part, lse_part, cpa.WRITE_PARTIAL)
    plan.sync_status()
    O = f32_to_f64(o_part)
    L = f32_to_f64(lse_part)
    for t in range(R):
        for qo, ko in sched[t]:
            qs = slice(qo * nq, (qo + 1) * nq)
            ks = slice(ko * nkv, (ko + 1) * nkv)
            Or, Lr = oracle.partial_attention(q[qs], k[ks], v[ks],
                                              plan.positions(cpa.TENSOR_Q, qo),
                                              plan.positions(cpa.TENSOR_KV, ko))
            assert_close(O[ko, qs], Or, 1e-2, f"O step {t} pair {qo},{ko}")
            assert_close(L[ko][:, qs], Lr, 1e-3, f"LSE step {t} pair {qo},{ko}")
            empty = np.isneginf(Lr)
            assert np.all(O[ko, qs][empty.T] == 0.0)


@pytest.mark.parametrize("chained", [False, True])
def test_running_accumulator_fp32(chained):
    """ACCUMULATE: the fp32 running merge after all steps equals monolithic
    attention at 1e-2 without any bf16 rounding of the result, with the steps
    launched normally and chained (each step overlapping the previous one's
    tail until its read-modify-write of the accumulator)."""
    w = Workload("acc", 2048, 4, 1, 128, 4)
    inp = make_inputs(w)
    plan = _plan(w)
    run = DeviceRun(plan, inp)
    plan.set_chaining(chained)
    o_acc = torch.full((plan.T_q, 4, 128), float("nan"), device="cuda")
    lse = torch.full((4, plan.T_q), float("nan"), device="cuda")
    for t in range(plan.R):
        plan.step_fwd(t, run.q, run.k, run.v, o_acc, lse, cpa.ACCUMULATE)
    plan.sync_status()
    O_ref, L_ref = _oracle_full(inp, plan, None)
    assert_close(run.to_natural_rows(f32_to_f64(o_acc)), O_ref, 1e-2, "O acc")
    assert_close(run.to_natural_rows(f32_to_f64(lse), axis=1), L_ref, 1e-3, "LSE acc")


RAGGED = [0, 1, 130, 1000, 1023, 1024, 2500, 4096]


@pytest.mark.parametrize("variant", ["pass_kv", "pass_q"])
@pytest.mark.parametrize("layout", ["zigzag", "contiguous"])
@pytest.mark.parametrize("docs", [False, True])
def test_forward_variants(variant, layout, docs):
    w = Workload("var", 4096, 4, 2, 128, 4)
    cu = np.array(RAGGED, dtype=np.int32) if docs else None
    inp = make_inputs(w)
    plan = _plan(w, variant=variant, layout=layout, cu=cu)
    run = DeviceRun(plan, inp)
    O_ref, L_ref = _oracle_full(inp, plan, cu)
    _check_forward(run, O_ref, L_ref, f"{variant}/{layout}/docs={docs}")


@pytest.mark.parametrize("variant", ["pass_kv", "pass_q"])
def test_partial_prefill_forward(variant):
    w = Workload("pp", 1024, 8, 2, 128, 2, kv_prefix_len=3072)
    inp = make_inputs(w)
    plan = _plan(w, variant=variant)
    run = DeviceRun(plan, inp)
    O_ref, L_ref = _oracle_full(inp, plan, None)
    _check_forward(run, O_ref, L_ref, f"partial prefill {variant}")


def test_pass_kv_equals_pass_q_on_device():
    w = Workload("kvq", 2048, 8, 1, 64, 4)
    inp = make_inputs(w)
    outs = []
    for variant in ("pass_kv", "pass_q"):
        plan = _plan(w, variant=variant)
        o, lse, _ = DeviceRun(plan, inp).forward()
        outs.append((bf16_to_f64(o), f32_to_f64(lse)))
    assert np.abs(outs[0][0] - outs[1][0]).max() <= 2e-2
    assert np.abs(outs[0][1] - outs[1][1]).max() <= 1e-3


@pytest.mark.parametrize("n,rows,H,d", [
    (5, 300, 3, 128),    # one warp per (row, head)
    (40, 30, 3, 128),    # many parts, few pairs: eight warps per pair
    (24, 16, 4, 64),     # the same with head_dim 64
])
def test_merge_kernel_against_oracle(n, rows, H, d):
    rng = np.random.default_rng(5)
    o = rng.standard_normal((n, rows, H, d)).astype(np.float32)
    lse = (rng.standard_normal((n, H, rows)) * 3).astype(np.float32)
    lse[1, :, ::7] = -np.inf
    lse[:, 2, 5] = -np.inf          # a row with no visible key anywhere
    o[:, 5, 2, :][np.isneginf(lse[:, 2, 5])] = 0
    parts = [(o[i].astype(np.float64), lse[i].astype(np.float64)) for i in range(n)]
    O_ref, L_ref = oracle.lse_merge(parts)
    to = torch.from_numpy(o).cuda()
    tl = torch.from_numpy(lse).cuda()
    ob = torch.empty((rows, H, d), dtype=torch.bfloat16, device="cuda")
    of = torch.empty((rows, H, d), dtype=torch.float32, device="cuda")
    lo = torch.empty((H, rows), dtype=torch.float32, device="cuda")
    cpa.merge_lse(n, rows, H, d, to, rows * H * d, tl, H * rows, ob, of, lo)
    torch.cuda.synchronize()
    assert_close(f32_to_f64(of), O_ref, 1e-4, "merge O fp32")
    assert_close_bf16(bf16_to_f64(ob), O_ref, 1e-3, "merge O bf16")
    assert_close(f32_to_f64(lo), L_ref, 1e-4, "merge LSE")
    assert np.isneginf(f32_to_f64(lo)[2, 5]) and np.all(f32_to_f64(of)[5, 2] == 0)


@pytest.mark.parametrize("n,rows,H,d", [
    (5, 300, 3, 128),    # one warp per (row, head)
    (40, 30, 3, 128),    # many parts, few pairs: a block of warps per pair
    (256, 1, 16, 128),   # a decode row's merge: 256 parts, most of them empty
])
def test_merge_never_reads_empty_parts(n, rows, H, d):
    """A part with LSE = -inf has weight 0 and its O rows are never read: they
    hold NaN here (as a slot that no kernel wrote may), and the result must
    equal the merge of the other parts alone (the LSE merge of "Ring Attention
    Algorithms": a part with no visible key contributes nothing)."""
    rng = np.random.default_rng(11)
    o = rng.standard_normal((n, rows, H, d)).astype(np.float32)
    lse = (rng.standard_normal((n, H, rows)) * 3).astype(np.float32)
    empty = rng.random(n) < 0.6
    empty[0] = False                 # every (row, head) keeps a part with keys
    lse[empty] = -np.inf
    o[empty] = np.nan
    parts = [(o[i].astype(np.float64), lse[i].astype(np.float64)) for i in range(n)
             if not empty[i]]
    O_ref, L_ref = oracle.lse_merge(parts)
    to = torch.from_numpy(o).cuda()
    tl = torch.from_numpy(lse).cuda()
    ob = torch.empty((rows, H, d), dtype=torch.bfloat16, device="cuda")
    of = torch.empty((rows, H, d), dtype=torch.float32, device="cuda")
    lo = torch.empty((H, rows), dtype=torch.float32, device="cuda")
    cpa.merge_lse(n, rows, H, d, to, rows * H * d, tl, H * rows, ob, of, lo)
    torch.cuda.synchronize()
    assert np.isfinite(f32_to_f64(of)).all() and np.isfinite(f32_to_f64(lo)).all()
    assert_close(f32_to_f64(of), O_ref, 1e-4, "merge (empty parts) O fp32")
    assert_close_bf16(bf16_to_f64(ob), O_ref, 1e-3, "merge (empty parts) O bf16")
    assert_close(f32_to_f64(lo), L_ref, 1e-4, "merge (empty parts) LSE")


@pytest.mark.parametrize("layout", ["zigzag", "contiguous"])
def test_layout_permute_bit_exact(layout):
    w = Workload("lay", 2048, 2, 1, 64, 4, kv_prefix_len=1024)
    plan = _plan(w, layout=layout)
    q_pos, kv_pos = oracle.plan_positions(2048, 4, layout, kv_prefix_len=1024)
    rows = torch.arange(plan.T_kv * 64, dtype=torch.int32, device="cuda").view(plan.T_kv, 1, 64)
    x = rows.view(torch.bfloat16).view(plan.T_kv, 2, 64)  # arbitrary bits
    y = torch.empty_like(x)
    plan.layout_apply(cpa.TENSOR_KV, cpa.TO_RANK_MAJOR, x, y)
    perm = np.concatenate(kv_pos)
    xh = x.view(torch.int16).cpu().numpy()
    assert np.array_equal(y.view(torch.int16).cpu().numpy(), xh[perm])
    z = torch.empty_like(x)
    plan.layout_apply(cpa.TENSOR_KV, cpa.TO_NATURAL, y, z)
    assert torch.equal(z.view(torch.int16), x.view(torch.int16))
    qx = torch.randn(plan.T_q, 2, 64, device="cuda").to(torch.bfloat16)
    qy = torch.empty_like(qx)
    plan.layout_apply(cpa.TENSOR_Q, cpa.TO_RANK_MAJOR, qx, qy)
    qperm = np.concatenate(q_pos) - 1024
    assert np.array_equal(qy.view(torch.int16).cpu().numpy(),
                          qx.view(torch.int16).cpu().numpy()[qperm])


def test_llama3_8b_layer_forward_sampled(oracle_pool):
    """Full-size 32768-token forward in the bench's launch configuration,
    checked on 1024 seeded sampled rows (all heads) by the oracle's
    full-prefix softmax (evaluated on the host cores in parallel), plus
    properties that hold at any size."""
    w = WORKLOADS["llama3_8b_layer"]
    inp = make_inputs(w, with_dout=False)
    rows = sample_rows(w.seq_len, 1024)
    job = oracle_pool.forward_rows(oracle_pool.problem(inp), rows)
    plan = _plan(w)
    run = DeviceRun(plan, inp)
    o, lse, _ = run.forward()
    O = run.to_natural_rows(bf16_to_f64(o))
    L = run.to_natural_rows(f32_to_f64(lse), axis=1)
    Or, Lr = job.get()
    assert_close_bf16(O[rows], Or, 1e-2, "1024 sampled rows O")
    assert_close(L[:, rows], Lr, 1e-3, "1024 sampled rows LSE")
    # row 0 sees only itself
    v0 = bf16_bits_to_f64(inp.v[0])
    assert np.abs(O[0] - v0[np.arange(w.n_q_heads) // w.group]).max() == 0.0
    assert np.isfinite(L).all()


@pytest.mark.parametrize("d", [64, 128])
def test_fp16_range_of_v_is_reported(d):
    """O += P V runs on an fp16 copy of V made by step 0 of the ring: a finite
    V value above 65504 (not representable in fp16) is reported as
    CP_ATTN_ERR_RANGE, and the next forward with valid inputs is clean."""
    w = Workload("rangef", 1024, 2, 1, d, 4)
    plan = _plan(w)
    run = DeviceRun(plan, make_inputs(w))
    v_big = run.v.clone()
    v_big[5, 0, 3] = 1.0e5
    o = torch.empty_like(run.q)
    lse = torch.empty((plan.Hq, plan.T_q), dtype=torch.float32, device="cuda")
    ws = torch.empty(plan.workspace_size(cpa.OP_FORWARD), dtype=torch.uint8, device="cuda")
    plan.forward(run.q, run.k, v_big, o, lse, ws)
    with pytest.raises(cpa.CpAttnError) as e:
        plan.sync_status()
    assert e.value.status == 7
    plan.forward(run.q, run.k, run.v, o, lse, ws)
    plan.sync_status()


def test_device_wait_timeout_is_reported():
    """A kernel wait that nothing completes gives up after its time limit and
    reports CP_ATTN_ERR_TIMEOUT through the plan's status word; the context
    stays usable."""
    w = WORKLOADS["tiny_ring"]
    plan = _plan(w)
    cpa.load().cp_attn_selftest_wait_timeout(plan.handle, 20_000_000, None)
    with pytest.raises(cpa.CpAttnError) as e:
        plan.sync_status()
    assert e.value.status == 6
    plan.sync_status()  # cleared
    x = torch.ones(16, device="cuda")
    assert float(x.sum()) == 16.0
