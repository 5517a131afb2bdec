"""Pins of the oracle's decode ("Context Parallelism for Scalable
Million-Token Inference": decode is a single-row attention of the new token
over every earlier token; Pass Q for decode moves the row around the ranks
and merges the partials)."""
import numpy as np
import pytest

import oracle
from test_oracle_pins import _sdpa, rand


@pytest.mark.parametrize("R", [1, 2, 4])
def test_decode_is_the_last_row_of_causal_attention(R):
    B, T, Hq, Hkv, d = 3, 32, 8, 2, 8
    qs = rand((B, T, Hq, d), 91)
    k, v = rand((B, T, Hkv, d), 92), rand((B, T, Hkv, d), 93)
    O, L = oracle.decode(qs[:, -1], k, v, R, 0.3)
    pos = np.arange(T)
    for b in range(B):
        Of, Lf = oracle.attention(qs[b], k[b], v[b], pos, pos, None, 0.3)
        np.testing.assert_allclose(O[b], Of[-1], atol=1e-13, rtol=0)
        np.testing.assert_allclose(L[:, b], Lf[:, -1], atol=1e-13, rtol=0)


def test_decode_equals_library_sdpa_row():
    B, T, Hq, Hkv, d = 2, 40, 4, 1, 16
    q = rand((B, Hq, d), 94)
    k, v = rand((B, T, Hkv, d), 95), rand((B, T, Hkv, d), 96)
    O, _ = oracle.decode(q, k, v, 4)
    for b in range(B):
        ref = _sdpa(q[b][None], k[b], v[b])       # one row, no mask
        np.testing.assert_allclose(O[b], ref[0], atol=1e-13, rtol=0)


def test_decode_constant_values():
    B, T, Hq, Hkv, d = 2, 16, 4, 2, 8
    q, k = rand((B, Hq, d), 97), rand((B, T, Hkv, d), 98)
    v = np.broadcast_to(rand((B, 1, Hkv, d), 99), (B, T, Hkv, d)).copy()
    O, _ = oracle.decode(q, k, v, 2)
    for h in range(Hq):
        np.testing.assert_allclose(O[:, h], v[:, 0, h // 2], atol=1e-14, rtol=0)
