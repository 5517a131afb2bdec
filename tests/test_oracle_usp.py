"""Pins of the oracle's Ulysses / USP pieces ("Announcing Long-Context
Training on TPUs with MaxText Context Parallelism", sections "All-to-All
(Ulysses)" and "A2A + P2P (USP)"): the pooled chunk plan, the head
all-to-all, and the composition (all-to-all, a ring per head group over the
pooled chunks, all-to-all back) against monolithic attention."""
import numpy as np
import pytest

import oracle
from test_oracle_pins import rand


def test_usp_figure_pairs_of_devices():
    # four devices, the all-to-all within each pair, the ring across the pairs
    assert oracle.rank_chunks(2, "usp", a2a=2) == [[0, 1, 6, 7], [2, 3, 4, 5]]
    # a2a = 1 is plain zigzag; one ring rank is pure Ulysses (the whole sequence)
    assert oracle.rank_chunks(4, "usp", a2a=1) == oracle.rank_chunks(4, "zigzag")
    assert oracle.rank_chunks(1, "usp", a2a=4) == [list(range(8))]


@pytest.mark.parametrize("R,U", [(2, 2), (4, 2), (2, 4), (3, 2)])
def test_usp_ranks_balanced_and_increasing(R, U):
    N = 2 * R * U * 8
    qp, kp = oracle.plan_positions(N, R, "usp", a2a=U)
    assert sorted(np.concatenate(qp).tolist()) == list(range(N))
    counts = [oracle.count_visible(qp[r], np.arange(N)) for r in range(R)]
    assert len(set(counts)) == 1          # every ring rank does the same work
    for r in range(R):
        assert np.all(np.diff(qp[r]) > 0)  # positions increase along the rows


def test_head_split_moves_heads_not_tokens():
    T, H, e, U = 12, 8, 3, 4
    x = np.zeros((T, H, e))
    for t in range(T):
        for h in range(H):
            x[t, h, :] = 1000 * t + 10 * h + np.arange(e)
    y = oracle.head_split(x, U)
    assert y.shape == (U, T, H // U, e)
    for u in range(U):
        for t in range(T):
            for j in range(H // U):
                assert np.array_equal(y[u, t, j], 1000 * t + 10 * (u * (H // U) + j) + np.arange(e))
    np.testing.assert_array_equal(oracle.head_gather(y), x)


@pytest.mark.parametrize("R,U", [(1, 2), (1, 4), (2, 2), (2, 4), (4, 1)])
@pytest.mark.parametrize("variant", ["pass_kv", "pass_q"])
def test_usp_composition_equals_monolithic(R, U, variant):
    N, Hq, Hkv, d = 2 * R * U * 8, 8, 4, 8
    cu = [0, N // 3, N]
    q, k, v = rand((N, Hq, d), 81), rand((N, Hkv, d), 82), rand((N, Hkv, d), 83)
    do = rand((N, Hq, d), 84)
    pos = np.arange(N)
    O, L = oracle.attention(q, k, v, pos, pos, cu)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, O, L, pos, pos, cu)
    qp, kp = oracle.plan_positions(N, R, "usp", a2a=U)
    perm = np.concatenate(qp)   # natural -> pooled (rank-major) rows
    qs, ks, vs, dos = (oracle.head_split(x[perm], U) for x in (q, k, v, do))
    outs, lses, grads = [], [], []
    for u in range(U):
        Ou, Lu = oracle.ring_forward(qs[u], ks[u], vs[u], qp, kp, cu, variant=variant)
        outs.append(Ou)
        lses.append(Lu)
        grads.append(oracle.ring_backward(qs[u], ks[u], vs[u], dos[u], Ou, Lu, qp, kp, cu,
                                          variant=variant))
    np.testing.assert_allclose(oracle.head_gather(np.stack(outs)), O[perm], atol=1e-13, rtol=0)
    np.testing.assert_allclose(np.concatenate(lses, axis=0), L[:, perm], atol=1e-13, rtol=0)
    for i, ref in enumerate((dq, dk, dv)):
        got = oracle.head_gather(np.stack([g[i] for g in grads]))
        np.testing.assert_allclose(got, ref[perm], atol=1e-12, rtol=0)
