"""Pins of the oracle's sliding-window mask and Pass KV / Pass Q choice.

Window (the window layers of models that mix sliding-window and global
layers, "Announcing Long-Context Training on TPUs with MaxText Context
Parallelism", section "What's next"): a key is visible only if it is also
fewer than W positions behind the query. Checked against pure-Python loops,
closed forms (W = 1: each query sees only itself; W >= N: no window), a
library attention with the band mask and its autograd, and the ring
decomposition.

Variant choice ("Context Parallelism for Scalable Million-Token Inference",
section "Ring Attention Algorithms"): Pass KV for full prefill and for
partial prefill with a low to medium KV-cache hit rate; Pass Q for a high hit
rate and for decode. Pinned by those statements and by the message-size
comparison at the crossover.
"""
import math

import numpy as np
import pytest

import oracle
from test_oracle_pins import _sdpa, brute_force, rand


def brute_window(q, k, v, qpos, kpos, cu, scale, W):
    """brute_force with out-of-window keys removed by giving them a position
    after every query (pure-Python distance test per pair)."""
    kpos = np.asarray(kpos)
    out_O = np.zeros(q.shape)
    out_L = np.full((q.shape[1], q.shape[0]), -np.inf)
    for i in range(q.shape[0]):
        keep = [j for j in range(len(kpos)) if qpos[i] - kpos[j] < W]
        O, L = brute_force(q[i:i + 1], k[keep], v[keep], qpos[i:i + 1], kpos[keep], cu, scale)
        out_O[i] = O[0]
        out_L[:, i] = L[:, 0]
    return out_O, out_L


def test_window_mask_brute_force():
    pos = np.arange(30)
    cu = [0, 7, 19, 30]
    for W in (1, 2, 5, 13, 29, 30, 100):
        vis = oracle.visible_mask(pos, pos, cu, window=W)
        for i in range(30):
            for j in range(30):
                doc_i = max(t for t in range(3) if cu[t] <= i)
                doc_j = max(t for t in range(3) if cu[t] <= j)
                want = (j <= i) and (doc_i == doc_j) and (i - j < W)
                assert bool(vis[i, j]) == want, (W, i, j)


@pytest.mark.parametrize("W", [1, 3, 8])
@pytest.mark.parametrize("docs", [None, [0, 5, 6, 13, 20]])
def test_window_forward_matches_brute_force(W, docs):
    N, Hq, Hkv, d = 20, 2, 1, 4
    q, k, v = rand((N, Hq, d), 61), rand((N, Hkv, d), 62), rand((N, Hkv, d), 63)
    pos = np.arange(N)
    O, L = oracle.attention(q, k, v, pos, pos, docs, 0.41, window=W)
    Ob, Lb = brute_window(q, k, v, pos, pos, docs, 0.41, W)
    np.testing.assert_allclose(O, Ob, atol=1e-13, rtol=0)
    np.testing.assert_allclose(L, Lb, atol=1e-13, rtol=0)


def test_window_one_sees_only_itself():
    N, Hq, Hkv, d = 33, 4, 2, 8
    q, k, v = rand((N, Hq, d), 64), rand((N, Hkv, d), 65), rand((N, Hkv, d), 66)
    pos = np.arange(N)
    O, L = oracle.attention(q, k, v, pos, pos, None, 0.5, window=1)
    G = Hq // Hkv
    for h in range(Hq):
        np.testing.assert_allclose(O[:, h], v[:, h // G], atol=1e-15, rtol=0)
        np.testing.assert_allclose(L[h], 0.5 * np.einsum("nd,nd->n", q[:, h], k[:, h // G]),
                                   atol=1e-14, rtol=0)


def test_window_as_long_as_sequence_is_no_window():
    N, Hq, Hkv, d = 40, 2, 1, 8
    q, k, v = rand((N, Hq, d), 67), rand((N, Hkv, d), 68), rand((N, Hkv, d), 69)
    pos = np.arange(N)
    O0, L0 = oracle.attention(q, k, v, pos, pos)
    O1, L1 = oracle.attention(q, k, v, pos, pos, window=N)
    np.testing.assert_array_equal(O0, O1)
    np.testing.assert_array_equal(L0, L1)


def test_window_equals_library_band_sdpa_and_autograd():
    torch = pytest.importorskip("torch")
    N, Hq, Hkv, d, W = 48, 4, 2, 8, 11
    q, k, v = rand((N, Hq, d), 70), rand((N, Hkv, d), 71), rand((N, Hkv, d), 72)
    do = rand((N, Hq, d), 73)
    pos = np.arange(N)
    band = (pos[None, :] <= pos[:, None]) & (pos[:, None] - pos[None, :] < W)
    O, L = oracle.attention(q, k, v, pos, pos, window=W)
    np.testing.assert_allclose(O, _sdpa(q, k, v, mask=band), atol=1e-13, rtol=0)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, O, L, pos, pos, window=W)
    G = Hq // Hkv
    tq = torch.from_numpy(q).requires_grad_()
    tk = torch.from_numpy(k).requires_grad_()
    tv = torch.from_numpy(v).requires_grad_()
    o = torch.nn.functional.scaled_dot_product_attention(
        tq.permute(1, 0, 2), tk.permute(1, 0, 2).repeat_interleave(G, 0),
        tv.permute(1, 0, 2).repeat_interleave(G, 0), attn_mask=torch.from_numpy(band))
    (o.permute(1, 0, 2) * torch.from_numpy(do)).sum().backward()
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-12)


@pytest.mark.parametrize("variant", ["pass_kv", "pass_q"])
def test_window_ring_equals_monolithic(variant):
    R, N, Hq, Hkv, d, W = 4, 64, 4, 2, 8, 13
    cu = [0, 23, 64]
    q, k, v = rand((N, Hq, d), 74), rand((N, Hkv, d), 75), rand((N, Hkv, d), 76)
    do = rand((N, Hq, d), 77)
    qp, kp = oracle.plan_positions(N, R, "zigzag")
    qperm, kperm = np.concatenate(qp), np.concatenate(kp)
    pos = np.arange(N)
    O, L = oracle.attention(q, k, v, pos, pos, cu, window=W)
    Or, Lr = oracle.ring_forward(q[qperm], k[kperm], v[kperm], qp, kp, cu, variant=variant,
                                 window=W)
    np.testing.assert_allclose(Or, O[qperm], atol=1e-13, rtol=0)
    np.testing.assert_allclose(Lr, L[:, qperm], atol=1e-13, rtol=0)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, O, L, pos, pos, cu, window=W)
    gq, gk, gv = oracle.ring_backward(q[qperm], k[kperm], v[kperm], do[qperm], O[qperm],
                                      L[:, qperm], qp, kp, cu, variant=variant, window=W)
    np.testing.assert_allclose(gq, dq[qperm], atol=1e-12, rtol=0)
    np.testing.assert_allclose(gk, dk[kperm], atol=1e-12, rtol=0)
    np.testing.assert_allclose(gv, dv[kperm], atol=1e-12, rtol=0)


def test_window_block_mask_is_tilewise_any_all():
    R, N, W = 2, 1024, 300
    qp, kp = oracle.plan_positions(N, R, "zigzag")
    bm = oracle.block_mask(qp, kp, None, window=W)
    for a in range(R):
        for b in range(R):
            vis = oracle.visible_mask(qp[a], kp[b], None, window=W)
            for i in range(bm.shape[2]):
                for j in range(bm.shape[3]):
                    t = vis[128 * i:128 * (i + 1), 128 * j:128 * (j + 1)]
                    want = 2 if t.all() else (1 if t.any() else 0)
                    assert bm[a, b, i, j] == want
    # a 300-token window leaves fully masked tiles far below the diagonal
    assert (bm == 0).sum() > 0 and (bm == 1).sum() > 0


def test_select_variant_follows_the_pages():
    # Llama 3 405B-shaped heads: 128 query heads, 8 KV heads
    Hq, Hkv = 128, 8
    # full prefill: Pass KV
    assert oracle.select_variant(131072, 0, Hq, Hkv) == "pass_kv"
    # partial prefill with a low or medium cache hit rate: Pass KV
    for hit in (0.0, 0.25, 0.5, 0.8):
        total = 100000
        new = int(round(total * (1 - hit)))
        assert oracle.select_variant(new, total - new, Hq, Hkv) == "pass_kv", hit
    # a high hit rate: Pass Q
    for hit in (0.9, 0.95, 0.99):
        total = 100000
        new = int(round(total * (1 - hit)))
        assert oracle.select_variant(new, total - new, Hq, Hkv) == "pass_q", hit
    # decode (one new token): Pass Q
    assert oracle.select_variant(1, 131071, Hq, Hkv) == "pass_q"


def test_select_variant_crossover_is_the_message_size_tie():
    # new/total = 2*Hkv/Hq exactly: equal messages, Pass KV kept
    assert oracle.select_variant(1024, 7168, 128, 8) == "pass_kv"   # 1/8
    assert oracle.select_variant(1023, 7169, 128, 8) == "pass_q"
    assert oracle.select_variant(1025, 7167, 128, 8) == "pass_kv"
    # equal head counts: the Q message is half the KV one even at full prefill
    assert oracle.select_variant(4096, 0, 32, 32) == "pass_q"
    # 8B-shaped GQA (32/8): crossover at a 50% miss rate
    assert oracle.select_variant(4096, 4096, 32, 8) == "pass_kv"
    assert oracle.select_variant(4095, 4097, 32, 8) == "pass_q"
    assert math.isclose(2 * 8 / 32, 0.5)
