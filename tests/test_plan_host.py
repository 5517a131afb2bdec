"""Host planner of the C library vs the oracle: bit-exact positions, ring
schedule, block classes and visible-pair counts; argument validation; the
exported C ABI. Runs without a GPU (plans built without a device serve the
host queries)."""
import re
import os

import numpy as np
import pytest

import oracle
from workloads import WORKLOADS, cu_seqlens_from_lengths, doc_lengths

cpa = pytest.importorskip("context_causal_attention_ring_gb300")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _plan(N, R, Hq=2, Hkv=1, d=64, layout="zigzag", variant="pass_kv", cu=None, P=0):
    return cpa.Plan(N, R, Hq, Hkv, d, layout=layout, variant=variant,
                    cu_seqlens=cu, kv_prefix_len=P)


def _check_plan(p, N, R, layout, variant, cu, P, full_mask=True, n_samples=0):
    q_pos, kv_pos = oracle.plan_positions(N, R, layout, kv_prefix_len=P)
    for r in range(R):
        assert np.array_equal(p.positions(cpa.TENSOR_Q, r), q_pos[r])
        assert np.array_equal(p.positions(cpa.TENSOR_KV, r), kv_pos[r])
    sched = np.array(oracle.ring_schedule(R, variant), dtype=np.int32)
    assert np.array_equal(p.schedule(), sched)
    bm = p.block_mask()
    if full_mask:
        assert np.array_equal(bm, oracle.block_mask(q_pos, kv_pos, cu))
    if n_samples:
        rng = np.random.default_rng(1)
        T = oracle.TILE
        for _ in range(n_samples):
            a, b = rng.integers(R, size=2)
            i = rng.integers(p.n_qt)
            j = rng.integers(p.n_kt)
            sub = oracle.block_mask([q_pos[a][i * T:(i + 1) * T]],
                                    [kv_pos[b][j * T:(j + 1) * T]], cu)[0, 0, 0, 0]
            assert bm[a, b, i, j] == sub, (a, b, i, j)
    return q_pos, kv_pos, sched


@pytest.mark.parametrize("layout", ["zigzag", "contiguous"])
@pytest.mark.parametrize("variant", ["pass_kv", "pass_q"])
def test_tiny_ring_plan_bit_exact(layout, variant):
    w = WORKLOADS["tiny_ring"]
    p = _plan(w.seq_len, w.cp, w.n_q_heads, w.n_kv_heads, w.head_dim, layout, variant)
    q_pos, kv_pos, sched = _check_plan(p, w.seq_len, w.cp, layout, variant, None, 0)
    allk = np.concatenate(kv_pos)
    assert p.visible_pairs() == sum(oracle.count_visible(x, allk) for x in q_pos)
    for t in range(w.cp):
        exp = sum(oracle.count_visible(q_pos[qo], kv_pos[ko]) for qo, ko in sched[t])
        assert p.visible_pairs(t) == exp


def test_documents_and_ragged_boundaries_bit_exact():
    N, R = 4096, 4
    cu = np.array([0, 1, 130, 1000, 1023, 1024, 2500, 4096], dtype=np.int32)
    p = _plan(N, R, cu=cu)
    q_pos, kv_pos, sched = _check_plan(p, N, R, "zigzag", "pass_kv", cu, 0)
    for t in range(R):
        exp = sum(oracle.count_visible(q_pos[qo], kv_pos[ko], cu) for qo, ko in sched[t])
        assert p.visible_pairs(t) == exp


@pytest.mark.parametrize("variant", ["pass_kv", "pass_q"])
def test_partial_prefill_plan_bit_exact(variant):
    N, P, R = 1024, 3072, 2
    p = _plan(N, R, variant=variant, P=P)
    q_pos, kv_pos, sched = _check_plan(p, N, R, "zigzag", variant, None, P)
    for t in range(R):
        exp = sum(oracle.count_visible(q_pos[qo], kv_pos[ko]) for qo, ko in sched[t])
        assert p.visible_pairs(t) == exp


def test_llama3_8b_layer_plan_bit_exact():
    w = WORKLOADS["llama3_8b_layer"]
    p = _plan(w.seq_len, w.cp, w.n_q_heads, w.n_kv_heads, w.head_dim)
    _check_plan(p, w.seq_len, w.cp, "zigzag", "pass_kv", None, 0)
    assert p.visible_pairs() == w.seq_len * (w.seq_len + 1) // 2


def test_partial_prefill_405b_plan_bit_exact():
    w = WORKLOADS["prefill_405b_partial"]
    p = _plan(w.seq_len, w.cp, w.n_q_heads, w.n_kv_heads, w.head_dim,
              variant="pass_q", P=w.kv_prefix_len)
    _check_plan(p, w.seq_len, w.cp, "zigzag", "pass_q", None, w.kv_prefix_len)
    # every new token sees the whole prefix plus its own causal triangle
    n, P = w.seq_len, w.kv_prefix_len
    assert p.visible_pairs() == n * P + n * (n + 1) // 2


def test_packed_docs_plan_sampled_tiles():
    w = WORKLOADS["packed_docs"]
    cu = cu_seqlens_from_lengths(doc_lengths(w.seq_len))
    p = _plan(w.seq_len, w.cp, w.n_q_heads, w.n_kv_heads, w.head_dim, cu=cu)
    q_pos, kv_pos, _ = _check_plan(p, w.seq_len, w.cp, "zigzag", "pass_kv", cu, 0,
                                   full_mask=False, n_samples=400)
    lens = np.diff(cu.astype(np.int64))
    assert p.visible_pairs() == int((lens * (lens + 1) // 2).sum())


def test_million_token_plan_sampled_tiles():
    w = WORKLOADS["million_token_group"]
    p = _plan(w.seq_len, w.cp, w.n_q_heads, w.n_kv_heads, w.head_dim)
    _check_plan(p, w.seq_len, w.cp, "zigzag", "pass_kv", None, 0, full_mask=False,
                n_samples=300)
    N = w.seq_len
    assert p.visible_pairs() == N * (N + 1) // 2
    # zigzag balance: every step has the same number of non-empty tiles per rank
    bm = p.block_mask()
    m = p.n_qt // 2
    counts = (bm > 0).sum(axis=(2, 3))
    for t in range(1, w.cp, 7):
        for r in range(w.cp):
            assert counts[r, (r - t) % w.cp] == 2 * m * m


@pytest.mark.parametrize("kw,status", [
    (dict(N=1000, R=4), 2),                      # not a multiple of 2*R*128
    (dict(N=1024, R=4, Hq=3, Hkv=2), 2),         # Hq % Hkv != 0
    (dict(N=1024, R=4, d=96), 3),                # head_dim unsupported
    (dict(N=1024, R=4, cu=[0, 10, 1000]), 2),    # does not end at N
    (dict(N=1024, R=4, cu=[0, 10, 10, 1024]), 2),  # not strictly increasing
    (dict(N=1024, R=0), 2),
])
def test_plan_rejects_bad_arguments(kw, status):
    with pytest.raises(cpa.CpAttnError) as e:
        _plan(**kw)
    assert e.value.status == status


def test_header_declarations_are_exported():
    hdr = open(os.path.join(ROOT, "include", "cp_attn.h")).read()
    declared = sorted(set(re.findall(r"\b(cp_attn_[a-z0-9_]+)\s*\(", hdr)))
    lib = cpa.load()
    for name in declared:
        assert hasattr(lib, name), name
    assert set(declared) == set(cpa.exported_symbols())


def test_step_chaining_flag_is_validated():
    """cp_attn_plan_set_chaining takes 0 or 1 and needs a plan (host only)."""
    plan = _plan(N=1024, R=4)
    plan.set_chaining(True)
    plan.set_chaining(False)
    lib = cpa.load()
    assert lib.cp_attn_plan_set_chaining(plan.handle, 2) == 1  # CP_ATTN_ERR_INVALID_ARG
    assert lib.cp_attn_plan_set_chaining(None, 1) == 1  # CP_ATTN_ERR_INVALID_ARG


def _round256(x):
    return (x + 255) // 256 * 256


def test_partial_and_grad_dtypes_set_the_workspace():
    """bf16 Pass-Q partials halve the R partial slots (the LSE slots stay
    fp32); bf16 gradients add the three fp32 accumulators to the backward
    workspace. Host-only plans, sizes from the element counts."""
    N, R, Hq, Hkv, d = 2048, 4, 8, 2, 128
    base = cpa.Plan(N, R, Hq, Hkv, d, variant="pass_q")
    half = cpa.Plan(N, R, Hq, Hkv, d, variant="pass_q", partial_dtype="bf16")
    o_el, l_el = N * Hq * d, N * Hq
    assert base.workspace_size(cpa.OP_FORWARD) == _round256(o_el * R * 4) + _round256(l_el * R * 4)
    assert half.workspace_size(cpa.OP_FORWARD) == _round256(o_el * R * 2) + _round256(l_el * R * 4)
    # Pass KV keeps its fp32 running output whatever the partial type
    kv = cpa.Plan(N, R, Hq, Hkv, d, variant="pass_kv", partial_dtype="bf16")
    assert kv.workspace_size(cpa.OP_FORWARD) == _round256(o_el * 4)
    g32 = cpa.Plan(N, R, Hq, Hkv, d)
    g16 = cpa.Plan(N, R, Hq, Hkv, d, grad_dtype="bf16")
    k_el = N * Hkv * d
    extra = _round256(o_el * 4) + 2 * _round256(k_el * 4)
    assert g16.workspace_size(cpa.OP_BACKWARD) == g32.workspace_size(cpa.OP_BACKWARD) + extra
    assert (half.partial_dtype, g16.grad_dtype, base.partial_dtype) == (cpa.BF16, cpa.BF16, cpa.F32)


@pytest.mark.parametrize("field", ["partial_dtype", "grad_dtype"])
def test_plan_rejects_unknown_dtype(field):
    with pytest.raises(cpa.CpAttnError) as e:
        cpa.Plan(1024, 4, 2, 1, 64, **{field: 2})
    assert e.value.status == 1  # CP_ATTN_ERR_INVALID_ARG


def test_merge_rejects_unknown_parts_dtype_and_overlap():
    """Argument checks of cp_attn_merge_lse_ex that need no device: an
    unknown dtype, and an fp32 output that overlaps bf16 parts (both fail
    before any launch; the pointers are never dereferenced)."""
    lib = cpa.load()
    base = 1 << 20
    # parts_dtype 7: ERR_INVALID_ARG
    assert lib.cp_attn_merge_lse_ex(2, 4, 1, 64, 7, base, 256, base + 4096, 4, None, None,
                                    base + 8192, None) == 1
    # bf16 parts [base, base + 2*(256 + 256)*2) and an fp32 output starting inside them
    assert lib.cp_attn_merge_lse_ex(2, 4, 1, 64, cpa.BF16, base, 256, base + 65536, 4, None,
                                    base + 512, base + 131072, None) == 1


@pytest.mark.parametrize("B,N,P,R,variant", [
    (3, 1024, 0, 4, "pass_kv"),
    (2, 512, 1536, 2, "pass_q"),
    (4, 512, 0, 2, "pass_q"),
])
def test_batch_plan_bit_exact(B, N, P, R, variant):
    """A batch of B sequences: positions (each sequence sharded on its own,
    sequence-major within a rank), the one-document-per-sequence offsets and
    the block classes bit-exact against the oracle's brute force; tiles of
    different sequences are EMPTY; visible pairs are B times one sequence's."""
    p = cpa.Plan(N, R, 2, 1, 64, variant=variant, kv_prefix_len=P, batch=B)
    assert (p.batch, p.T_q, p.T_kv, p.n_docs) == (B, B * N, B * (N + P), B)
    q_pos, kv_pos = oracle.plan_positions(N, R, "zigzag", kv_prefix_len=P, batch=B)
    cu = oracle.batch_cu_seqlens(N, B, P)
    for r in range(R):
        assert np.array_equal(p.positions(cpa.TENSOR_Q, r), q_pos[r])
        assert np.array_equal(p.positions(cpa.TENSOR_KV, r), kv_pos[r])
    bm = p.block_mask()
    assert np.array_equal(bm, oracle.block_mask(q_pos, kv_pos, cu))
    one = cpa.Plan(N, R, 2, 1, 64, variant=variant, kv_prefix_len=P)
    assert p.visible_pairs() == B * one.visible_pairs()
    sched = oracle.ring_schedule(R, variant)
    for t in range(R):
        exp = sum(oracle.count_visible(q_pos[qo], kv_pos[ko], cu) for qo, ko in sched[t])
        assert p.visible_pairs(t) == exp


def test_batch_with_documents_and_bad_offsets():
    """Documents inside a batch: cu_seqlens covers the whole batch and must
    contain every sequence start."""
    N, R, B = 1024, 2, 2
    cu = np.array([0, 300, 1024, 1500, 2048], dtype=np.int32)
    p = cpa.Plan(N, R, 2, 1, 64, cu_seqlens=cu, batch=B)
    q_pos, kv_pos = oracle.plan_positions(N, R, "zigzag", batch=B)
    assert np.array_equal(p.block_mask(), oracle.block_mask(q_pos, kv_pos, cu))
    with pytest.raises(cpa.CpAttnError) as e:   # misses the start of sequence 1 (1024)
        cpa.Plan(N, R, 2, 1, 64, cu_seqlens=[0, 300, 1500, 2048], batch=B)
    assert e.value.status == 2
    with pytest.raises(cpa.CpAttnError) as e:   # ends at one sequence's length
        cpa.Plan(N, R, 2, 1, 64, cu_seqlens=[0, 1024], batch=B)
    assert e.value.status == 2
    with pytest.raises(cpa.CpAttnError) as e:
        cpa.Plan(N, R, 2, 1, 64, batch=-1)
    assert e.value.status == 2


@pytest.mark.parametrize("kw", [
    dict(N=1024, R=4, layout="zigzag", variant="pass_kv"),
    dict(N=1024, R=4, layout="contiguous", variant="pass_q"),
    dict(N=4096, R=4, cu=[0, 1, 130, 1000, 1023, 1024, 2500, 4096]),
    dict(N=1024, R=2, P=3072, variant="pass_q"),
    dict(N=2048, R=4, window=300),
    dict(N=1024, R=2, B=3),
    dict(N=2048, R=2, layout="usp", a2a=2),
])
def test_work_lists_bit_exact(kw):
    """The work lists the step kernels consume, forward and backward, every
    step: bit-exact against the oracle's list built from its brute-force
    block classes (runs, FULL counts, longest-first order)."""
    N, R = kw["N"], kw["R"]
    layout, variant = kw.get("layout", "zigzag"), kw.get("variant", "pass_kv")
    P, B, window, a2a = kw.get("P", 0), kw.get("B", 1), kw.get("window", 0), kw.get("a2a", 1)
    cu = kw.get("cu")
    cu_arr = None if cu is None else np.array(cu, dtype=np.int32)
    p = cpa.Plan(N, R, 2, 1, 64, layout=layout, variant=variant, cu_seqlens=cu_arr,
                 kv_prefix_len=P, window=window, a2a=a2a, batch=B)
    q_pos, kv_pos = oracle.plan_positions(N, R, layout, kv_prefix_len=P, a2a=a2a, batch=B)
    docs = oracle.batch_cu_seqlens(N, B, P) if (cu is None and B > 1) else cu
    bm = oracle.block_mask(q_pos, kv_pos, docs, window=window)
    assert np.array_equal(p.block_mask(), bm)
    sched = oracle.ring_schedule(R, variant)
    for t in range(R):
        for bwd in (False, True):
            got = p.work_list(t, bwd)
            want = oracle.work_list(bm, sched, t, bwd)
            assert np.array_equal(got, want), (t, bwd)


def test_decode_fp8_argument_checks_on_the_host():
    """cp_attn_decode_fp8 refuses bad arguments before any device work: an
    unsupported head_dim, null or misaligned pointers, a short workspace and
    runs of keys that are not multiples of 128 (fake device addresses that
    are never dereferenced)."""
    import ctypes
    from context_causal_attention_ring_gb300 import _abi
    lib = cpa.load()
    base = 1 << 32

    def call(desc, ptrs=None, ws_bytes=None):
        p = ptrs or [base + i * (1 << 24) for i in range(7)]
        need = cpa.decode_workspace_size(desc.batch, desc.cp, desc.kv_len, desc.n_q_heads,
                                         desc.n_kv_heads, desc.head_dim)
        return lib.cp_attn_decode_fp8(ctypes.byref(desc), *p[:5], p[5], p[6],
                                      need if ws_bytes is None else ws_bytes, None)

    ok = _abi._decode_desc(2, 4, 4096, 8, 2, 128)
    assert call(_abi._decode_desc(2, 4, 4096, 8, 2, 64)) == 3          # head_dim 64
    ptrs = [base + i * (1 << 24) for i in range(7)]
    for i in range(7):
        bad = list(ptrs)
        bad[i] = None
        assert call(ok, bad) == 1, i                                    # a null pointer
        bad[i] = ptrs[i] + 8
        assert call(ok, bad) == 1, i                                    # misaligned
    assert call(ok, ws_bytes=16) == 2                                   # workspace too small
    assert call(_abi._decode_desc(1, 4, 256, 2, 1, 128)) == 2          # 64-key runs
