"""Host planner with sliding windows and the Pass KV / Pass Q choice, against
the oracle: bit-exact block classes and visible-pair counts for windowed
plans (with documents and a cached prefix), and the library's variant
choice over a grid of prefill shapes. No GPU needed."""
import numpy as np
import pytest

import oracle

cpa = pytest.importorskip("context_causal_attention_ring_gb300")


@pytest.mark.parametrize("W", [1, 100, 128, 129, 300, 1000, 5000])
@pytest.mark.parametrize("variant", ["pass_kv", "pass_q"])
def test_window_plan_bit_exact(W, variant):
    N, R = 4096, 4
    cu = np.array([0, 1, 130, 1000, 1023, 1024, 2500, 4096], dtype=np.int32)
    p = cpa.Plan(N, R, 2, 1, 64, variant=variant, cu_seqlens=cu, window=W)
    assert p.window == (W if W < N else 0)
    q_pos, kv_pos = oracle.plan_positions(N, R, "zigzag")
    assert np.array_equal(p.block_mask(), oracle.block_mask(q_pos, kv_pos, cu, window=W))
    sched = oracle.ring_schedule(R, variant)
    for t in range(R):
        exp = sum(oracle.count_visible(q_pos[qo], kv_pos[ko], cu, window=W) for qo, ko in sched[t])
        assert p.visible_pairs(t) == exp


@pytest.mark.parametrize("W", [64, 700, 3000])
def test_window_partial_prefill_plan_bit_exact(W):
    N, P, R = 1024, 3072, 2
    p = cpa.Plan(N, R, 2, 1, 64, kv_prefix_len=P, window=W)
    q_pos, kv_pos = oracle.plan_positions(N, R, "zigzag", kv_prefix_len=P)
    assert np.array_equal(p.block_mask(), oracle.block_mask(q_pos, kv_pos, None, window=W))
    allk = np.concatenate(kv_pos)
    assert p.visible_pairs() == sum(oracle.count_visible(x, allk, window=W) for x in q_pos)


def test_window_rejects_negative():
    with pytest.raises(cpa.CpAttnError):
        cpa.Plan(1024, 2, 2, 1, 64, window=-1)


def test_select_variant_matches_oracle_on_a_grid():
    for hq, hkv in ((128, 8), (32, 8), (32, 32), (8, 1), (64, 8)):
        for total in (1, 1000, 4096, 131072, 1 << 20):
            for new in sorted({1, total // 100 or 1, total // 16 or 1, total // 8 or 1,
                               total // 4 or 1, total // 2 or 1, total}):
                want = oracle.select_variant(new, total - new, hq, hkv)
                assert cpa.select_variant(new, total - new, hq, hkv) == want, (hq, hkv, total, new)


def test_auto_variant_plan_resolves_like_select_variant():
    # 405B-shaped heads: full prefill -> Pass KV; a 97% cache hit -> Pass Q
    full = cpa.Plan(2048, 8, 128, 8, 128, variant="auto")
    assert full.variant == "pass_kv"
    part = cpa.Plan(4096, 8, 128, 8, 128, variant="auto", kv_prefix_len=126976)
    assert part.variant == cpa.select_variant(4096, 126976, 128, 8) == "pass_q"
    sched = np.array(oracle.ring_schedule(8, "pass_q"), dtype=np.int32)
    assert np.array_equal(part.schedule(), sched)


def test_select_variant_rejects_bad_arguments():
    for args in ((0, 10, 8, 1), (10, -1, 8, 1), (10, 10, 0, 1), (10, 10, 8, 0)):
        with pytest.raises(cpa.CpAttnError):
            cpa.select_variant(*args)


@pytest.mark.parametrize("R,U,P", [(2, 2, 0), (4, 2, 0), (1, 4, 0), (2, 4, 4096), (3, 2, 0), (8, 1, 0)])
def test_usp_plan_bit_exact(R, U, P):
    N = 256 * R * U * 2
    cu = np.array([0, 300, N + P - 129, N + P], dtype=np.int32)
    p = cpa.Plan(N, R, 4, 2, 128, layout="usp", a2a=U, kv_prefix_len=P, cu_seqlens=cu)
    assert (p.R, p.a2a) == (R, U)
    q_pos, kv_pos = oracle.plan_positions(N, R, "usp", kv_prefix_len=P, a2a=U)
    for r in range(R):
        assert np.array_equal(p.positions(cpa.TENSOR_Q, r), q_pos[r])
        assert np.array_equal(p.positions(cpa.TENSOR_KV, r), kv_pos[r])
    assert np.array_equal(p.block_mask(), oracle.block_mask(q_pos, kv_pos, cu))
    allk = np.concatenate(kv_pos)
    assert p.visible_pairs() == sum(oracle.count_visible(x, allk, cu) for x in q_pos)


def test_usp_plan_rejects_bad_chunks():
    with pytest.raises(cpa.CpAttnError):
        cpa.Plan(512, 2, 4, 2, 128, layout="usp", a2a=2)   # needs 1024-token multiples
    with pytest.raises(cpa.CpAttnError):
        cpa.Plan(2048, 2, 4, 2, 128, layout="usp", a2a=0)
