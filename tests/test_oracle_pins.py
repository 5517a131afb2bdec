"""Pins of the CPU oracle against things other than itself.

Each test checks the oracle against a value printed on the pages (the
worked example of "Load Balancing in CP" in "Context Parallelism for
Scalable Million-Token Inference"), a closed form, a brute-force loop on
tiny inputs, an invariant of softmax attention, or a library routine that
computes a special case (torch scaled_dot_product_attention and autograd on
CPU in fp64). ``test_oracle_mutants.py`` plants mistakes in the oracle and
checks that these pins catch them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from workloads import bf16_bits_to_f64, draw_bf16

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# ---------------------------------------------------------------------------
# Chunk plan
# ---------------------------------------------------------------------------
def test_worked_example_load_balance():
    g = json.load(open(os.path.join(GOLDEN, "load_balance_worked_example.json")))
    pos = oracle.shard_positions(g["n_tokens"], g["ranks"], "zigzag")
    assert [list(map(int, p)) for p in pos] == g["rank_tokens"]
    all_pos = np.arange(g["n_tokens"])
    blocks = [oracle.count_visible(p, all_pos) for p in pos]
    assert blocks == g["compute_blocks_per_rank"]


@pytest.mark.parametrize("R,c", [(2, 1), (2, 3), (4, 128), (8, 5), (3, 7)])
def test_balanced_visible_pairs_closed_form(R, c):
    # rank r holds positions [rc, rc+c) and [(2R-1-r)c, (2R-r)c); a query at
    # position p sees p+1 keys, so every rank sees 2Rc^2 + c pairs.
    N = 2 * R * c
    q_pos, kv_pos = oracle.plan_positions(N, R, "zigzag")
    all_k = np.concatenate(kv_pos)
    counts = [oracle.count_visible(q_pos[r], all_k) for r in range(R)]
    assert counts == [2 * R * c * c + c] * R
    # no balancing with contiguous chunks: rank r sees sum_{p} (p+1)
    q_c, kv_c = oracle.plan_positions(N, R, "contiguous")
    n = N // R
    for r in range(R):
        exp = sum(p + 1 for p in range(r * n, (r + 1) * n))
        assert oracle.count_visible(q_c[r], np.concatenate(kv_c)) == exp


def test_tiny_ring_pair_count():
    # 1024 tokens, 4 ranks: 131200 visible pairs per rank and query head
    q_pos, kv_pos = oracle.plan_positions(1024, 4, "zigzag")
    allk = np.concatenate(kv_pos)
    assert [oracle.count_visible(p, allk) for p in q_pos] == [131200] * 4


@pytest.mark.parametrize("R,m", [(2, 1), (2, 2), (4, 1), (4, 3), (3, 2)])
def test_block_counts_closed_form(R, m):
    # With m tiles per half-chunk: every step t != 0 gives each rank exactly
    # 2m^2 FULL tiles and no PARTIAL; step 0 gives 2m^2 - m FULL and 2m
    # PARTIAL (the two diagonal triangles); over the ring that is
    # (2R-1)m^2 + m(m+1) non-empty tiles per rank.
    tile = 4
    c = m * tile
    N = 2 * R * c
    q_pos, kv_pos = oracle.plan_positions(N, R, "zigzag")
    bm = oracle.block_mask(q_pos, kv_pos, None, tile=tile)
    for variant in ("pass_kv", "pass_q"):
        sched = oracle.ring_schedule(R, variant)
        total = [0] * R
        for t in range(R):
            for r in range(R):
                qo, ko = sched[t][r]
                b = bm[qo, ko]
                full = int((b == 2).sum())
                part = int((b == 1).sum())
                if t == 0:
                    assert (full, part) == (2 * m * m - m, 2 * m)
                else:
                    assert (full, part) == (2 * m * m, 0)
                total[qo] += full + part
        assert total == [(2 * R - 1) * m * m + m * (m + 1)] * R


def test_block_mask_is_tilewise_any_all():
    # Tile classes of a hand-checkable 2-rank plan with two documents.
    # N=16, R=2, tile=2: rank0 positions [0..3, 12..15], rank1 [4..11].
    cu = np.array([0, 6, 16])
    q_pos, kv_pos = oracle.plan_positions(16, 2, "zigzag")
    assert list(q_pos[0]) == [0, 1, 2, 3, 12, 13, 14, 15]
    bm = oracle.block_mask(q_pos, kv_pos, cu, tile=2)
    # rank0 q tile 0 = {0,1} vs rank0 kv tile 0 = {0,1}: causal diagonal
    assert bm[0, 0, 0, 0] == 1
    # q {2,3} vs k {0,1}: all visible (same doc 0)
    assert bm[0, 0, 1, 0] == 2
    # q {12,13} (doc 1) vs k {0,1} (doc 0): empty
    assert bm[0, 0, 2, 0] == 0
    # rank1 q {6,7} (doc1) vs rank1 k {4,5} (doc0): empty
    assert bm[1, 1, 1, 0] == 0
    # rank0 q {14,15} vs rank1 k {6,7}: full (doc 1, earlier)
    assert bm[0, 1, 3, 1] == 2
    # rank1 q {4,5} vs rank1 k {4,5}: diagonal, partial
    assert bm[1, 1, 0, 0] == 1


def test_schedule_covers_every_pair_once():
    for R in (1, 2, 5, 8):
        for variant in ("pass_kv", "pass_q"):
            sched = oracle.ring_schedule(R, variant)
            pairs = [p for row in sched for p in row]
            assert sorted(pairs) == [(a, b) for a in range(R) for b in range(R)]
            for t in range(R):
                # each step is a permutation: each rank once as q and kv owner
                assert sorted(p[0] for p in sched[t]) == list(range(R))
                assert sorted(p[1] for p in sched[t]) == list(range(R))
            assert all(a == b for a, b in sched[0])


def test_partial_prefill_plan():
    # cache 8 tokens + 8 new, R=2: cache chunks of 2, new chunks of 2
    q_pos, kv_pos = oracle.plan_positions(8, 2, "zigzag", kv_prefix_len=8)
    assert list(q_pos[0]) == [8, 9, 14, 15]
    assert list(kv_pos[0]) == [0, 1, 6, 7, 8, 9, 14, 15]
    assert list(kv_pos[1]) == [2, 3, 4, 5, 10, 11, 12, 13]


# ---------------------------------------------------------------------------
# Forward
# ---------------------------------------------------------------------------
def brute_force(q, k, v, qpos, kpos, cu, scale):
    """Pure-Python loops over rows, heads and keys."""
    n, Hq, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv

    def doc(p):
        if cu is None:
            return 0
        for i in range(len(cu) - 1):
            if cu[i] <= p < cu[i + 1]:
                return i
        raise ValueError(p)

    O = np.zeros(q.shape)
    L = np.full((Hq, n), -np.inf)
    for i in range(n):
        for h in range(Hq):
            kh = h // G
            scores = []
            for j in range(k.shape[0]):
                if kpos[j] <= qpos[i] and doc(kpos[j]) == doc(qpos[i]):
                    s = sum(q[i, h, x] * k[j, kh, x] for x in range(d)) * scale
                    scores.append((s, j))
            if not scores:
                continue
            mx = max(s for s, _ in scores)
            z = sum(math.exp(s - mx) for s, _ in scores)
            for s, j in scores:
                w = math.exp(s - mx) / z
                for x in range(d):
                    O[i, h, x] += w * v[j, kh, x]
            L[h, i] = mx + math.log(z)
    return O, L


@pytest.mark.parametrize("docs", [None, [0, 5, 6, 13, 20]])
def test_forward_matches_brute_force(docs):
    N, Hq, Hkv, d = 20, 2, 1, 4
    q, k, v = rand((N, Hq, d), 1), rand((N, Hkv, d), 2), rand((N, Hkv, d), 3)
    pos = np.arange(N)
    scale = 0.37
    O, L = oracle.attention(q, k, v, pos, pos, docs, scale)
    Ob, Lb = brute_force(q, k, v, pos, pos, docs, scale)
    np.testing.assert_allclose(O, Ob, atol=1e-13, rtol=0)
    np.testing.assert_allclose(L, Lb, atol=1e-13, rtol=0)


def test_forward_brute_force_ring_shuffled_positions():
    # arbitrary position maps and a key set that leaves some rows empty
    q, k, v = rand((6, 4, 3), 4), rand((7, 2, 3), 5), rand((7, 2, 3), 6)
    qpos = np.array([9, 2, 30, 5, 0, 17])
    kpos = np.array([3, 4, 6, 10, 11, 25, 31])
    cu = [0, 8, 20, 40]
    O, L = oracle.partial_attention(q, k, v, qpos, kpos, cu, 0.5)
    Ob, Lb = brute_force(q, k, v, qpos, kpos, cu, 0.5)
    np.testing.assert_allclose(O, Ob, atol=1e-13, rtol=0)
    assert np.array_equal(np.isinf(L), np.isinf(Lb))
    fin = np.isfinite(Lb)
    np.testing.assert_allclose(L[fin], Lb[fin], atol=1e-13, rtol=0)
    # rows 1 (pos 2) and 4 (pos 0) see no key: O = 0, LSE = -inf
    assert np.all(O[[1, 4]] == 0) and np.all(np.isneginf(L[:, [1, 4]]))


def test_constant_v_returns_v():
    N, Hq, Hkv, d = 64, 4, 2, 8
    q, k = rand((N, Hq, d), 7), rand((N, Hkv, d), 8)
    vrow = rand((Hkv, d), 9)
    v = np.broadcast_to(vrow, (N, Hkv, d)).copy()
    cu = [0, 10, 40, 64]
    O, _ = oracle.attention(q, k, v, np.arange(N), np.arange(N), cu)
    for h in range(Hq):
        np.testing.assert_allclose(O[:, h, :], np.broadcast_to(vrow[h // 2], (N, d)),
                                   atol=1e-14, rtol=0)


def test_one_token_prefix_and_document_starts():
    N, Hq, Hkv, d = 48, 4, 1, 16
    q, k, v = rand((N, Hq, d), 10), rand((N, Hkv, d), 11), rand((N, Hkv, d), 12)
    cu = [0, 17, 30, 48]
    scale = 1 / math.sqrt(d)
    O, L = oracle.attention(q, k, v, np.arange(N), np.arange(N), cu, scale)
    for s in cu[:-1]:
        for h in range(Hq):
            np.testing.assert_allclose(O[s, h], v[s, 0], atol=1e-15, rtol=0)
            assert abs(L[h, s] - scale * q[s, h] @ k[s, 0]) < 1e-14


def test_documents_equal_independent_runs():
    N, Hq, Hkv, d = 50, 4, 2, 8
    q, k, v = rand((N, Hq, d), 13), rand((N, Hkv, d), 14), rand((N, Hkv, d), 15)
    cu = [0, 7, 8, 31, 50]
    O, L = oracle.attention(q, k, v, np.arange(N), np.arange(N), cu)
    for a, b in zip(cu[:-1], cu[1:]):
        pos = np.arange(b - a)
        Oi, Li = oracle.attention(q[a:b], k[a:b], v[a:b], pos, pos, None)
        np.testing.assert_allclose(O[a:b], Oi, atol=1e-14, rtol=0)
        np.testing.assert_allclose(L[:, a:b], Li, atol=1e-13, rtol=0)


def _sdpa(q, k, v, mask=None, is_causal=False, scale=None):
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    Hq, Hkv = q.shape[1], k.shape[1]
    G = Hq // Hkv
    tq = torch.from_numpy(q).permute(1, 0, 2)
    # KV head of query head h is h // G: repeat each KV head G times
    tk = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(G, dim=0)
    tv = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(G, dim=0)
    m = None if mask is None else torch.from_numpy(mask)
    o = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=m,
                                       is_causal=is_causal, scale=scale)
    return o.permute(1, 0, 2).numpy()


def test_cp1_equals_library_causal_sdpa():
    N, Hq, Hkv, d = 96, 8, 2, 16
    q, k, v = rand((N, Hq, d), 16), rand((N, Hkv, d), 17), rand((N, Hkv, d), 18)
    O, L = oracle.attention(q, k, v, np.arange(N), np.arange(N))
    Oref = _sdpa(q, k, v, is_causal=True)
    np.testing.assert_allclose(O, Oref, atol=1e-13, rtol=0)
    torch = pytest.importorskip("torch")
    s = torch.einsum("nhd,mhd->hnm", torch.from_numpy(q),
                     torch.from_numpy(np.repeat(k, 4, axis=1))) / math.sqrt(d)
    s = s.masked_fill(~torch.ones(N, N, dtype=torch.bool).tril(), -math.inf)
    np.testing.assert_allclose(L, torch.logsumexp(s, dim=-1).numpy(),
                               atol=1e-13, rtol=0)


def test_partial_prefill_equals_library_masked_sdpa():
    P, n, Hq, Hkv, d = 40, 24, 4, 1, 8
    q = rand((n, Hq, d), 19)
    k, v = rand((P + n, Hkv, d), 20), rand((P + n, Hkv, d), 21)
    O, _ = oracle.attention(q, k, v, P + np.arange(n), np.arange(P + n))
    # bottom-right aligned causal mask: query i sees keys <= P + i
    mask = np.arange(P + n)[None, :] <= (P + np.arange(n))[:, None]
    np.testing.assert_allclose(O, _sdpa(q, k, v, mask=mask), atol=1e-13, rtol=0)


@pytest.mark.parametrize("variant", ["pass_kv", "pass_q"])
@pytest.mark.parametrize("layout", ["zigzag", "contiguous"])
@pytest.mark.parametrize("docs", [False, True])
def test_ring_equals_monolithic(variant, layout, docs):
    R, N, Hq, Hkv, d = 4, 64, 4, 2, 8
    q, k, v = rand((N, Hq, d), 22), rand((N, Hkv, d), 23), rand((N, Hkv, d), 24)
    cu = [0, 9, 30, 31, 64] if docs else None
    q_pos, kv_pos = oracle.plan_positions(N, R, layout)
    perm = np.concatenate(q_pos)
    Or, Lr = oracle.ring_forward(q[perm], k[perm], v[perm], q_pos, kv_pos, cu,
                                 variant=variant)
    Om, Lm = oracle.attention(q, k, v, np.arange(N), np.arange(N), cu)
    np.testing.assert_allclose(Or, Om[perm], atol=1e-12, rtol=0)
    np.testing.assert_allclose(Lr, Lm[:, perm], atol=1e-12, rtol=0)


@pytest.mark.parametrize("variant", ["pass_kv", "pass_q"])
def test_ring_partial_prefill_equals_monolithic(variant):
    R, P, n, Hq, Hkv, d = 2, 32, 16, 4, 1, 8
    q = rand((n, Hq, d), 25)
    k, v = rand((P + n, Hkv, d), 26), rand((P + n, Hkv, d), 27)
    q_pos, kv_pos = oracle.plan_positions(n, R, "zigzag", kv_prefix_len=P)
    qperm = np.concatenate(q_pos) - P
    kperm = np.concatenate(kv_pos)
    Or, Lr = oracle.ring_forward(q[qperm], k[kperm], v[kperm], q_pos, kv_pos,
                                 variant=variant)
    Om, Lm = oracle.attention(q, k, v, P + np.arange(n), np.arange(P + n))
    np.testing.assert_allclose(Or, Om[qperm], atol=1e-12, rtol=0)
    np.testing.assert_allclose(Lr, Lm[:, qperm], atol=1e-12, rtol=0)


def test_lse_merge_special_cases():
    o1, l1 = rand((5, 2, 3), 28), rand((2, 5), 29)
    # merging with an all-empty part (-inf) is the identity
    O, L = oracle.lse_merge([(o1, l1), (np.zeros_like(o1), np.full_like(l1, -np.inf))])
    np.testing.assert_allclose(O, o1, atol=1e-15)
    np.testing.assert_allclose(L, l1, atol=1e-15)
    # two equal parts: same O, LSE + ln 2
    O, L = oracle.lse_merge([(o1, l1), (o1, l1)])
    np.testing.assert_allclose(O, o1, atol=1e-15)
    np.testing.assert_allclose(L, l1 + math.log(2), atol=1e-15)
    # all parts empty: O = 0, LSE = -inf
    O, L = oracle.lse_merge([(o1 * 0, np.full_like(l1, -np.inf))] * 3)
    assert np.all(O == 0) and np.all(np.isneginf(L))


def test_sampled_rows_equal_full():
    N, Hq, Hkv, d = 300, 4, 2, 8
    q, k, v = rand((N, Hq, d), 30), rand((N, Hkv, d), 31), rand((N, Hkv, d), 32)
    do = rand((N, Hq, d), 33)
    cu = [0, 100, 101, 300]
    pos = np.arange(N)
    rows = np.array([0, 1, 99, 100, 101, 150, 299])
    O, L = oracle.attention(q, k, v, pos, pos, cu)
    Os, Ls = oracle.sampled_forward(q, k, v, rows, pos, pos, cu)
    np.testing.assert_allclose(Os, O[rows], atol=1e-14)
    np.testing.assert_allclose(Ls, L[:, rows], atol=1e-14)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, O, L, pos, pos, cu)
    np.testing.assert_allclose(oracle.sampled_dq(q, k, v, do, rows, pos, pos, cu),
                               dq[rows], atol=1e-13)
    krows = np.arange(N - 40, N)
    dks, dvs = oracle.sampled_dkdv(q, k, v, do, krows, pos, pos, cu)
    np.testing.assert_allclose(dks, dk[krows], atol=1e-13)
    np.testing.assert_allclose(dvs, dv[krows], atol=1e-13)


def test_bf16_inputs_widen_exactly():
    rng = np.random.default_rng(0)
    b = draw_bf16(rng, (4, 3), 0.5)
    x = bf16_bits_to_f64(b)
    # every bf16 value has at most 8 significant bits
    m, e = np.frexp(x)
    assert np.all((m * 256) == np.round(m * 256))


# ---------------------------------------------------------------------------
# Backward
# ---------------------------------------------------------------------------
def _loss(q, k, v, do, pos_q, pos_k, cu, scale):
    O, _ = oracle.attention(q, k, v, pos_q, pos_k, cu, scale)
    return float((O * do).sum())


@pytest.mark.parametrize("docs", [None, [0, 4, 11, 14]])
def test_backward_finite_differences(docs):
    N, Hq, Hkv, d = 14, 4, 2, 3
    q, k, v = rand((N, Hq, d), 34), rand((N, Hkv, d), 35), rand((N, Hkv, d), 36)
    do = rand((N, Hq, d), 37)
    pos = np.arange(N)
    scale = 0.61
    O, L = oracle.attention(q, k, v, pos, pos, docs, scale)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, O, L, pos, pos, docs, scale)
    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp = x.copy(); xp[idx] += eps
            xm = x.copy(); xm[idx] -= eps
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            fp = _loss(args["q"], args["k"], args["v"], do, pos, pos, docs, scale)
            args[name] = xm
            fm = _loss(args["q"], args["k"], args["v"], do, pos, pos, docs, scale)
            num[idx] = (fp - fm) / (2 * eps)
        rel = np.abs(num - g).max() / max(np.abs(g).max(), 1e-300)
        assert rel < 1e-6, (name, rel)


def test_backward_equals_library_autograd():
    torch = pytest.importorskip("torch")
    N, Hq, Hkv, d = 40, 4, 2, 8
    q, k, v = rand((N, Hq, d), 38), rand((N, Hkv, d), 39), rand((N, Hkv, d), 40)
    do = rand((N, Hq, d), 41)
    pos = np.arange(N)
    O, L = oracle.attention(q, k, v, pos, pos)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, O, L, pos, pos)
    tq = torch.from_numpy(q).requires_grad_()
    tk = torch.from_numpy(k).requires_grad_()
    tv = torch.from_numpy(v).requires_grad_()
    G = Hq // Hkv
    o = torch.nn.functional.scaled_dot_product_attention(
        tq.permute(1, 0, 2), tk.permute(1, 0, 2).repeat_interleave(G, 0),
        tv.permute(1, 0, 2).repeat_interleave(G, 0), is_causal=True)
    (o.permute(1, 0, 2) * torch.from_numpy(do)).sum().backward()
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-12)


def test_backward_invariants():
    N, Hq, Hkv, d = 60, 4, 2, 8
    q, k, v = rand((N, Hq, d), 42), rand((N, Hkv, d), 43), rand((N, Hkv, d), 44)
    do = rand((N, Hq, d), 45)
    cu = [0, 13, 14, 60]
    pos = np.arange(N)
    O, L = oracle.attention(q, k, v, pos, pos, cu)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, O, L, pos, pos, cu)
    # a row that sees only itself has zero dQ
    for s in cu[:-1]:
        assert np.abs(dq[s]).max() < 1e-14
    # dS rows sum to zero, so sum_k dK_k = 0 per (kv head, document)
    # and sum_k dV_k = sum over the group's query heads of sum_p dO_p
    for a, b in zip(cu[:-1], cu[1:]):
        assert np.abs(dk[a:b].sum(axis=0)).max() < 1e-12
        for kh in range(Hkv):
            exp = do[a:b, 2 * kh:2 * kh + 2].sum(axis=(0, 1))
            np.testing.assert_allclose(dv[a:b, kh].sum(axis=0), exp, atol=1e-12)
    # constant V: dQ = dK = 0
    vc = np.broadcast_to(v[0], v.shape).copy()
    O, L = oracle.attention(q, k, vc, pos, pos, cu)
    dq, dk, _ = oracle.attention_backward(q, k, vc, do, O, L, pos, pos, cu)
    assert np.abs(dq).max() < 1e-13 and np.abs(dk).max() < 1e-13


@pytest.mark.parametrize("variant", ["pass_kv", "pass_q"])
@pytest.mark.parametrize("prefix", [0, 32])
def test_ring_backward_equals_monolithic(variant, prefix):
    R, n, Hq, Hkv, d = 2, 32, 4, 2, 8
    q = rand((n, Hq, d), 46)
    k, v = rand((prefix + n, Hkv, d), 47), rand((prefix + n, Hkv, d), 48)
    do = rand((n, Hq, d), 49)
    cu = [0, 20, prefix + n]
    q_pos, kv_pos = oracle.plan_positions(n, R, "zigzag", kv_prefix_len=prefix)
    qperm = np.concatenate(q_pos) - prefix
    kperm = np.concatenate(kv_pos)
    qp, kp = prefix + np.arange(n), np.arange(prefix + n)
    O, L = oracle.attention(q, k, v, qp, kp, cu)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, O, L, qp, kp, cu)
    rdq, rdk, rdv = oracle.ring_backward(q[qperm], k[kperm], v[kperm], do[qperm],
                                         O[qperm], L[:, qperm], q_pos, kv_pos, cu,
                                         variant=variant)
    np.testing.assert_allclose(rdq, dq[qperm], atol=1e-12)
    np.testing.assert_allclose(rdk, dk[kperm], atol=1e-12)
    np.testing.assert_allclose(rdv, dv[kperm], atol=1e-12)


def test_ring_backward_steps_sum_to_whole():
    R, n, Hq, Hkv, d = 4, 64, 2, 1, 4
    q, k, v = rand((n, Hq, d), 50), rand((n, Hkv, d), 51), rand((n, Hkv, d), 52)
    do = rand((n, Hq, d), 53)
    q_pos, kv_pos = oracle.plan_positions(n, R, "zigzag")
    perm = np.concatenate(q_pos)
    O, L = oracle.attention(q, k, v, np.arange(n), np.arange(n))
    args = (q[perm], k[perm], v[perm], do[perm], O[perm], L[:, perm], q_pos, kv_pos)
    whole = oracle.ring_backward(*args)
    parts = [oracle.ring_backward(*args, steps=[t]) for t in range(R)]
    for i in range(3):
        np.testing.assert_allclose(sum(p[i] for p in parts), whole[i], atol=1e-13)


# ---------------------------------------------------------------- bf16 storage rounding
def test_round_bf16_hand_values():
    """Values pinned by hand: representable values stay, ties go to the even
    significand, subnormals keep the 2^-133 spacing, the overflow point and
    above become infinite."""
    r = oracle.round_bf16
    keep = np.array([0.0, 1.0, 1.0 + 2.0 ** -7, -3.0, 2.0 ** -126, 2.0 ** -133,
                     255.0 * 2.0 ** 120, -(2.0 - 2.0 ** -7) * 2.0 ** 127])
    assert np.array_equal(r(keep), keep)
    assert r(1.0 + 2.0 ** -8) == 1.0                       # tie, down to even
    assert r(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6       # tie, up to even
    assert r(-(1.0 + 2.0 ** -8)) == -1.0
    assert r(1.0 + 2.0 ** -8 + 2.0 ** -30) == 1.0 + 2.0 ** -7  # above the tie
    assert r(1.5 * 2.0 ** -133) == 2.0 ** -132            # subnormal tie to even
    assert r(0.5 * 2.0 ** -133) == 0.0                     # half the smallest: to even (0)
    assert r((2.0 - 2.0 ** -8) * 2.0 ** 127) == np.inf     # the overflow point
    assert r((2.0 - 2.0 ** -8 - 2.0 ** -20) * 2.0 ** 127) == (2.0 - 2.0 ** -7) * 2.0 ** 127
    assert np.isnan(r(np.nan)) and r(-np.inf) == -np.inf


def test_round_bf16_matches_torch_conversion():
    """On fp32 inputs over the whole exponent range the oracle's rounding is
    the library's round-to-nearest-even fp32 -> bf16 conversion, bit for
    bit."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(200000) * np.exp2(rng.uniform(-140, 126, 200000))).astype(np.float32)
    # plus every tie of the first few binades
    ties = (np.arange(1, 4096, dtype=np.float64) * 2.0 ** -16 + 1.0).astype(np.float32)
    x = np.concatenate([x, ties, -ties])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.round_bf16(x.astype(np.float64))
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all(), x[~same][:5]


def test_ring_forward_bf16_partials_pass_q():
    """Pass Q with bf16 partial slots: each slot's O is rounded before the
    merge, so O moves by at most half a bf16 ulp of the largest partial
    (relative 2^-8 of it) and the LSE not at all; Pass KV ignores the
    option."""
    R, n, H, d = 4, 8, 2, 4
    rng = np.random.default_rng(3)
    q = rng.standard_normal((R * 2 * n, H, d))
    k = rng.standard_normal((R * 2 * n, H, d))
    v = rng.standard_normal((R * 2 * n, H, d))
    qpos, kvpos = oracle.plan_positions(R * 2 * n, R, "zigzag")
    O32, L32 = oracle.ring_forward(q, k, v, qpos, kvpos, variant="pass_q")
    O16, L16 = oracle.ring_forward(q, k, v, qpos, kvpos, variant="pass_q", partial_dtype="bf16")
    assert np.array_equal(L16, L32)
    diff = np.abs(O16 - O32)
    assert diff.max() > 0                                      # the rounding happened
    assert (diff <= 2.0 ** -8 * np.abs(v).max() + 1e-15).all()
    Ok, Lk = oracle.ring_forward(q, k, v, qpos, kvpos, variant="pass_kv", partial_dtype="bf16")
    Ok32, _ = oracle.ring_forward(q, k, v, qpos, kvpos, variant="pass_kv")
    assert np.array_equal(Ok, Ok32)


def test_batch_positions_partition_and_balance():
    """A batch's positions: the ranks together hold every position of the B
    sequences exactly once, each sequence's tokens are split evenly, and
    within each sequence every rank sees the same number of causal pairs
    (the zigzag balance of one sequence, sequence by sequence)."""
    B, N, P, R = 3, 512, 512, 2
    L = N + P
    q_pos, kv_pos = oracle.plan_positions(N, R, "zigzag", kv_prefix_len=P, batch=B)
    allkv = np.sort(np.concatenate(kv_pos))
    assert np.array_equal(allkv, np.arange(B * L))
    allq = np.sort(np.concatenate(q_pos))
    assert np.array_equal(allq, np.concatenate([b * L + P + np.arange(N) for b in range(B)]))
    cu = oracle.batch_cu_seqlens(N, B, P)
    for b in range(B):
        per_rank = []
        for r in range(R):
            mine = q_pos[r][(q_pos[r] >= b * L) & (q_pos[r] < (b + 1) * L)]
            assert len(mine) == N // R
            per_rank.append(oracle.count_visible(mine, allkv, cu))
        assert len(set(per_rank)) == 1
        # a query of sequence b sees exactly its own sequence's earlier tokens
        assert sum(per_rank) == sum(P + j + 1 for j in range(N))


def test_work_list_closed_forms():
    """The oracle's work lists on the zigzag ring against the closed forms of
    the chunk plan: over the whole ring each rank's runs cover (2R-1) m^2 +
    m (m + 1) non-empty tiles (m = tiles per half-chunk); every step after the
    first has 2 m^2 FULL tiles per rank and the first 2 m^2 - m FULL plus 2 m
    PARTIAL; run lengths never grow down a list; the backward lists cover the
    same tiles as the forward ones."""
    R, m = 4, 2
    N = 2 * R * m * oracle.TILE
    q_pos, kv_pos = oracle.plan_positions(N, R, "zigzag")
    bm = oracle.block_mask(q_pos, kv_pos)
    sched = oracle.ring_schedule(R, "pass_kv")
    per_rank = np.zeros(R, dtype=np.int64)
    for t in range(R):
        fw = oracle.work_list(bm, sched, t)
        bw = oracle.work_list(bm, sched, t, backward=True)
        for lst in (fw, bw):
            lengths = lst[:, 4] - lst[:, 3]
            assert np.all(np.diff(lengths) <= 0)
        assert (fw[:, 4] - fw[:, 3]).sum() == (bw[:, 4] - bw[:, 3]).sum()
        assert fw[:, 5].sum() == bw[:, 5].sum()
        for r in range(R):
            mine = fw[fw[:, 0] == r]
            assert len(mine) == 2 * m                       # every query tile once
            per_rank[r] += (mine[:, 4] - mine[:, 3]).sum()
            full = mine[:, 5].sum()
            if t == 0:
                # the later chunk against the earlier one (m^2 FULL) and two
                # diagonal triangles (m (m - 1) / 2 FULL and m PARTIAL each)
                assert full == 2 * m * m - m
                assert (mine[:, 4] - mine[:, 3]).sum() - full == 2 * m
            else:
                assert full == 2 * m * m
    assert np.all(per_rank == (2 * R - 1) * m * m + m * (m + 1))
