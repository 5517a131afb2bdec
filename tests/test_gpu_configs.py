"""GPU parity at the full sizes of the remaining workloads (packed documents,
405B-shaped full and partial prefill with both ring orderings and the
automatic choice between them, and the million-token head group), in the
launch configuration bench.py uses.

The oracle cannot afford every output at these sizes in one process, so it
runs on the host cores through tests/oracle_pool.py (its own functions on
slices of the rows, put back together) and checks:
* packed documents: the whole forward and backward of KV head 0 and its
  four query heads (every row and every key of every document, including
  the long documents that span many ranks), O and LSE at 128 seeded rows of
  every document for all heads, dQ at those rows, and dK/dV of all KV heads
  at the last 512 keys of the longest document; the three shortest
  documents are also recomputed whole, all heads;
* 405B-shaped prefill: O and LSE at 1024 seeded rows, for Pass KV, Pass Q
  and the plan that chooses between them (VARIANT_AUTO, "Ring Attention
  Algorithms"), which must pick Pass KV for the full prefill and Pass Q for
  4096 new tokens after a 126976-token cache;
* million-token head group: O and LSE at 4096 seeded rows (all heads), dQ
  at 256 seeded rows, dK and dV at the last 512 keys.
Device rows are gathered on the device so that the host never holds the
full tensors in fp64.
"""
import numpy as np
import pytest

import oracle
from workloads import WORKLOADS, bf16_bits_to_f64, make_inputs, sample_rows
from gpu_utils import DeviceRun, assert_close, assert_close_bf16, cuda_ok

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]

if cuda_ok():
    import torch
    import context_causal_attention_ring_gb300 as cpa

GRAD_TOL = 1e-2


def _plan(w, variant="pass_kv", cu=None):
    return cpa.Plan(w.seq_len, w.cp, w.n_q_heads, w.n_kv_heads, w.head_dim,
                    variant=variant, cu_seqlens=cu, kv_prefix_len=w.kv_prefix_len)


def _backward(run, o, lse, o_f32):
    p = run.plan
    dq = torch.empty((p.T_q, p.Hq, p.d), device="cuda")
    dk = torch.empty((p.T_kv, p.Hkv, p.d), device="cuda")
    dv = torch.empty_like(dk)
    ws = torch.empty(p.workspace_size(cpa.OP_BACKWARD), dtype=torch.uint8, device="cuda")
    p.backward(run.q, run.k, run.v, o, lse, run.dout, dq, dk, dv, ws, o_f32=o_f32)
    p.sync_status()
    del ws
    return dq, dk, dv


def _doc_rows(cu, per_doc, seed=0):
    """The first two and last two rows of every document plus seeded rows
    inside it, per_doc in all (fewer for short documents)."""
    rng = np.random.default_rng(seed)
    out = []
    for a, b in zip(cu[:-1], cu[1:]):
        a, b = int(a), int(b)
        ends = np.array([a, a + 1, b - 2, b - 1])
        inner = rng.choice(np.arange(a, b), size=min(per_doc - 4, b - a), replace=False)
        out.append(np.union1d(ends, inner))
    return np.unique(np.concatenate(out))


def test_packed_docs_forward_backward(oracle_pool):
    w = WORKLOADS["packed_docs"]
    inp = make_inputs(w)
    cu = inp.cu_seqlens
    lens = np.diff(cu)
    spec = oracle_pool.problem(inp)
    # the oracle works on the host cores while the device runs
    rows = _doc_rows(cu, 128)
    longest = int(np.argmax(lens))
    ka, kb = int(cu[longest + 1]) - 512, int(cu[longest + 1])
    jobs = {"head0": oracle_pool.backward_head(spec, 0),
            "fwd": oracle_pool.forward_rows(spec, rows),
            "dq": oracle_pool.dq_rows(spec, rows),
            "dkdv": oracle_pool.dkdv_keys(spec, ka, kb)}
    plan = _plan(w, cu=cu)
    run = DeviceRun(plan, inp)
    o, lse, ws = run.forward()
    dq, dk, dv = _backward(run, o, lse, ws)  # fp32 O from the forward workspace
    del ws
    N = w.seq_len
    G = w.group
    allr = np.arange(N)

    # KV head 0 and its query heads, every row and key of every document
    O0, L0, dq0, dk0, dv0 = jobs["head0"].get()
    hs = slice(0, G)
    # (heads sliced on the device before the rows are gathered)
    assert_close_bf16(run.take(o[:, hs], allr), O0, 1e-2, "head group 0 O (all rows)")
    assert_close(run.take(lse[hs], allr, axis=1), L0, 1e-3, "head group 0 LSE (all rows)")
    assert_close(run.take(dq[:, hs], allr), dq0, GRAD_TOL, "head group 0 dQ (all rows)")
    assert_close(run.take(dk[:, 0], allr, "kv"), dk0, GRAD_TOL, "KV head 0 dK (all keys)")
    assert_close(run.take(dv[:, 0], allr, "kv"), dv0, GRAD_TOL, "KV head 0 dV (all keys)")

    # all heads at rows of every document
    Or, Lr = jobs["fwd"].get()
    assert_close_bf16(run.take(o, rows), Or, 1e-2, "rows of every document O")
    assert_close(run.take(lse, rows, axis=1), Lr, 1e-3, "rows of every document LSE")
    assert_close(run.take(dq, rows), jobs["dq"].get(), GRAD_TOL, "rows of every document dQ")
    dk_r, dv_r = jobs["dkdv"].get()
    krows = np.arange(ka, kb)
    assert_close(run.take(dk, krows, "kv"), dk_r, GRAD_TOL, "longest document last-512 dK")
    assert_close(run.take(dv, krows, "kv"), dv_r, GRAD_TOL, "longest document last-512 dV")

    # the three shortest documents whole, all heads
    for doc in np.argsort(lens)[:3]:
        a, b = int(cu[doc]), int(cu[doc + 1])
        r = np.arange(a, b)
        q, k, v, do = (bf16_bits_to_f64(x[a:b]) for x in (inp.q, inp.k, inp.v, inp.dout))
        pos = np.arange(b - a)
        Od, Ld = oracle.attention(q, k, v, pos, pos)
        dq_d, dk_d, dv_d = oracle.attention_backward(q, k, v, do, Od, Ld, pos, pos)
        tag = f"document {doc} [{a},{b})"
        assert_close_bf16(run.take(o, r), Od, 1e-2, tag + " O")
        assert_close(run.take(lse, r, axis=1), Ld, 1e-3, tag + " LSE")
        assert_close(run.take(dq, r), dq_d, GRAD_TOL, tag + " dQ")
        assert_close(run.take(dk, r, "kv"), dk_d, GRAD_TOL, tag + " dK")
        assert_close(run.take(dv, r, "kv"), dv_d, GRAD_TOL, tag + " dV")
    for t in (o, lse, dq, dk, dv):
        assert bool(torch.isfinite(t.float()).all())


@pytest.mark.parametrize("name,auto_choice", [("prefill_405b_full", "pass_kv"),
                                              ("prefill_405b_partial", "pass_q")])
def test_prefill_405b_both_orderings(oracle_pool, name, auto_choice):
    w = WORKLOADS[name]
    inp = make_inputs(w, with_dout=False)
    N = w.seq_len
    rows = sample_rows(N, 1024)
    job = oracle_pool.forward_rows(oracle_pool.problem(inp, w.kv_prefix_len), rows)
    results = {}
    Or = Lr = None
    for variant in ("pass_kv", "pass_q", "auto"):
        plan = _plan(w, variant)
        if variant == "auto":
            # the selector of "Ring Attention Algorithms": full prefill keeps
            # Q still (Pass KV); a high cache-hit rate moves Q (Pass Q)
            assert plan.variant == auto_choice
        run = DeviceRun(plan, inp)
        o, lse, ws = run.forward()
        del ws
        if Or is None:
            Or, Lr = job.get()
        assert_close_bf16(run.take(o, rows), Or, 1e-2, f"{name} {variant} sampled O")
        assert_close(run.take(lse, rows, axis=1), Lr, 1e-3, f"{name} {variant} sampled LSE")
        # all plans share the same rank-major order, so outputs compare directly
        results[variant] = (o, lse)
        del run
    (o1, l1), (o2, l2) = results["pass_kv"], results["pass_q"]
    # the two orderings merge the same partial results in different orders
    assert float((o1.float() - o2.float()).abs().max()) <= 2e-2
    assert float((l1 - l2).abs().max()) <= 1e-3
    oa, la = results["auto"]
    ob, lb = results[auto_choice]
    assert torch.equal(oa, ob) and torch.equal(la, lb)  # same kernels, same order


def test_million_token_group_forward_backward(oracle_pool):
    w = WORKLOADS["million_token_group"]
    inp = make_inputs(w)
    N = w.seq_len
    spec = oracle_pool.problem(inp)
    rows = sample_rows(N, 4096)
    rows_dq = sample_rows(N, 256, seed=1)
    jobs = {"fwd": oracle_pool.forward_rows(spec, rows),
            "dq": oracle_pool.dq_rows(spec, rows_dq),
            "dkdv": oracle_pool.dkdv_keys(spec, N - 512, N)}
    plan = _plan(w)
    run = DeviceRun(plan, inp)
    o, lse, ws = run.forward()
    dq, dk, dv = _backward(run, o, lse, ws)  # fp32 O from the forward workspace
    del ws
    Or, Lr = jobs["fwd"].get()
    assert_close_bf16(run.take(o, rows), Or, 1e-2, "4096 sampled rows O")
    assert_close(run.take(lse, rows, axis=1), Lr, 1e-3, "4096 sampled rows LSE")
    assert_close(run.take(dq, rows_dq), jobs["dq"].get(), GRAD_TOL, "256 sampled rows dQ")
    # the last 512 keys are seen only by the last 512 queries
    dk_r, dv_r = jobs["dkdv"].get()
    krows = np.arange(N - 512, N)
    assert_close(run.take(dk, krows, "kv"), dk_r, GRAD_TOL, "last-512-key dK")
    assert_close(run.take(dv, krows, "kv"), dv_r, GRAD_TOL, "last-512-key dV")
    for t in (o, lse, dq, dk, dv):
        assert bool(torch.isfinite(t.float()).all())
