"""The parallel oracle helper of the full-size parity tests puts the oracle's
pieces back together exactly: on small inputs (with packed documents and
with a cached prefix) its results equal direct oracle calls over all rows
and keys."""
import numpy as np
import pytest

import oracle
from workloads import Workload, bf16_bits_to_f64, make_inputs
from oracle_pool import OraclePool


@pytest.fixture(scope="module")
def pool():
    p = OraclePool(3)
    yield p
    p.close()


def _direct(inp, P):
    q, k, v, do = (bf16_bits_to_f64(x) for x in (inp.q, inp.k, inp.v, inp.dout))
    N = q.shape[0]
    qp, kp = P + np.arange(N), np.arange(P + N)
    O, L = oracle.attention(q, k, v, qp, kp, inp.cu_seqlens)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, O, L, qp, kp, inp.cu_seqlens)
    return O, L, dq, dk, dv


@pytest.mark.parametrize("case", ["docs", "prefix"])
def test_pool_matches_direct_oracle(pool, case):
    if case == "docs":
        w = Workload("pool_docs", 512, 4, 2, 16, 2, docs=True, backward=True)
        inp = make_inputs(w)
        inp.cu_seqlens = np.array([0, 1, 100, 333, 512], dtype=np.int32)
        P = 0
    else:
        w = Workload("pool_prefix", 256, 4, 2, 16, 2, kv_prefix_len=192, backward=True)
        inp = make_inputs(w)
        P = 192
    O, L, dq, dk, dv = _direct(inp, P)
    spec = pool.problem(inp, P)
    N = inp.q.shape[0]
    rows = np.array([0, 1, 5, 99, 100, 101, 250, N - 1])
    fo = pool.forward_rows(spec, rows)
    fq = pool.dq_rows(spec, rows)
    a, b = P + N - 40, P + N
    fk = pool.dkdv_keys(spec, a, b)
    a2, b2 = P + 90, P + 130  # keys around a document boundary
    fk2 = pool.dkdv_keys(spec, a2, b2)
    hb = [pool.backward_head(spec, g) for g in range(2)]
    Or, Lr = fo.get()
    np.testing.assert_allclose(Or, O[rows], atol=1e-12)
    np.testing.assert_allclose(Lr, L[:, rows], atol=1e-12)
    np.testing.assert_allclose(fq.get(), dq[rows], atol=1e-12)
    for (x, y), (lo, hi) in ((fk.get(), (a, b)), (fk2.get(), (a2, b2))):
        np.testing.assert_allclose(x, dk[lo:hi], atol=1e-12)
        np.testing.assert_allclose(y, dv[lo:hi], atol=1e-12)
    for g, h in enumerate(hb):
        o, l, q_, k_, v_ = h.get()
        hs = slice(2 * g, 2 * g + 2)
        np.testing.assert_allclose(o, O[:, hs], atol=1e-12)
        np.testing.assert_allclose(l, L[hs], atol=1e-12)
        np.testing.assert_allclose(q_, dq[:, hs], atol=1e-12)
        np.testing.assert_allclose(k_, dk[:, g], atol=1e-12)
        np.testing.assert_allclose(v_, dv[:, g], atol=1e-12)
