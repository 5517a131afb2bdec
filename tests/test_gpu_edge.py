"""GPU parity of degenerate ring shapes against the fp64 oracle, through the
C ABI: a ring of one rank (the step is plain causal flash attention), the
smallest chunk (one 128-token tile per chunk), and one-token attention, where
every query sees only itself (documents of one token, or a window of 1), so
that O must equal the query's own V row and the LSE its own scaled score.
Tolerances: O (bf16) 1e-2 plus half a bf16 ulp, LSE 1e-3, fp32 gradients
1e-2."""
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


def _forward_backward(w, variant="pass_kv", cu=None, window=0):
    inp = make_inputs(w, with_dout=True)
    plan = cpa.Plan(w.seq_len, w.cp, w.n_q_heads, w.n_kv_heads, w.head_dim, variant=variant,
                    cu_seqlens=cu, window=window)
    run = DeviceRun(plan, inp)
    o, lse, ws_f = run.forward()
    p = plan
    dq = torch.full((p.T_q, p.Hq, p.d), float("nan"), device="cuda")
    dk = torch.full((p.T_kv, p.Hkv, p.d), float("nan"), device="cuda")
    dv = torch.full_like(dk, float("nan"))
    ws = torch.empty(p.workspace_size(cpa.OP_BACKWARD), dtype=torch.uint8, device="cuda")
    p.backward(run.q, run.k, run.v, o, lse, run.dout, dq, dk, dv, ws, o_f32=ws_f)
    p.sync_status()
    q, k, v, do = (bf16_bits_to_f64(x) for x in (inp.q, inp.k, inp.v, inp.dout))
    pos = np.arange(w.seq_len)
    O_r, L_r = oracle.attention(q, k, v, pos, pos, cu, window=window)
    grads_r = oracle.attention_backward(q, k, v, do, O_r, L_r, pos, pos, cu, window=window)
    what = f"{w.name} R={w.cp} d={w.head_dim} {variant}"
    O = run.to_natural_rows(bf16_to_f64(o))
    L = run.to_natural_rows(f32_to_f64(lse), axis=1)
    assert_close_bf16(O, O_r, 1e-2, what + " O")
    assert_close(L, L_r, 1e-3, what + " LSE")
    for name, g, ref, kind in zip(("dQ", "dK", "dV"), (dq, dk, dv), grads_r, ("q", "kv", "kv")):
        assert_close(run.to_natural_rows(f32_to_f64(g), kind), ref, 1e-2, what + " " + name)
    return q, k, v, O, L


@pytest.mark.parametrize("N,Hq,Hkv,d,variant", [
    (256, 2, 1, 128, "pass_kv"),
    (256, 4, 2, 128, "pass_q"),
    (512, 2, 2, 64, "pass_kv"),
])
def test_single_rank_ring(N, Hq, Hkv, d, variant):
    _forward_backward(Workload("r1", N, Hq, Hkv, d, 1, backward=True), variant)


def test_one_tile_per_chunk():
    # R = 8, N = 2048: each of the 16 zigzag chunks is a single 128-token tile
    _forward_backward(Workload("tile_chunks", 2048, 4, 4, 128, 8, backward=True))


@pytest.mark.parametrize("how", ["docs", "window"])
def test_one_token_attention(how):
    """Every query sees only itself: O = its V row, LSE = scale * q . k."""
    w = Workload("self_only", 512, 4, 2, 64, 2, backward=True, seed=5)
    cu = np.arange(0, w.seq_len + 1, dtype=np.int32) if how == "docs" else None
    window = 1 if how == "window" else 0
    q, k, v, O, L = _forward_backward(w, cu=cu, window=window)
    G = w.n_q_heads // w.n_kv_heads
    v_rows = np.repeat(v, G, axis=1)                      # [N, Hq, d]: the query's own V
    assert_close_bf16(O, v_rows, 1e-2, how + " O = own V")
    scale = 1.0 / np.sqrt(w.head_dim)
    own = scale * np.einsum("nhd,nhd->hn", q, np.repeat(k, G, axis=1))
    assert_close(L, own, 1e-3, how + " LSE = own score")


def test_mixed_singletons_and_window():
    """Single-token documents between long ones, with a window of 3 inside
    the long ones."""
    w = Workload("mix", 1024, 4, 1, 128, 2, backward=True, seed=9)
    cu = np.array([0, 1, 2, 3, 300, 301, 700, 1024], dtype=np.int32)
    _forward_backward(w, cu=cu, window=3)
