"""Pins of the FP8 (E4M3) oracle: the format's definition, a library cast,
and the quantization error bound. Planted mistakes in the encoder must be
caught by these pins."""
import inspect
import textwrap

import numpy as np
import pytest

import oracle.fp8 as f8


def test_known_codes():
    """Values fixed by the E4M3 definition: bias 7, three mantissa bits,
    subnormal spacing 2^-9, largest finite 448, S.1111.111 NaN."""
    v = f8.e4m3_decode(np.array([0x00, 0x01, 0x07, 0x08, 0x38, 0x39, 0x7E, 0x80, 0xFE, 0x7F, 0xFF],
                                dtype=np.uint8))
    assert v[0] == 0.0
    assert v[1] == 2.0 ** -9
    assert v[2] == 7 * 2.0 ** -9
    assert v[3] == 2.0 ** -6
    assert v[4] == 1.0
    assert v[5] == 1.125
    assert v[6] == 448.0
    assert v[7] == 0.0 and np.signbit(v[7])
    assert v[8] == -448.0
    assert np.isnan(v[9]) and np.isnan(v[10])


def test_round_trip_every_code():
    c = np.arange(256, dtype=np.uint8)
    v = f8.e4m3_decode(c)
    ok = ~np.isnan(v)
    assert ok.sum() == 254
    assert np.array_equal(f8.e4m3_encode(v[ok]), c[ok])
    # the 127 finite non-negative values are strictly increasing with the code
    assert np.all(np.diff(v[:0x7F]) > 0)


def test_ties_go_to_even_and_saturate():
    x = np.array([1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -10, 449.0, 464.0, 1e6, -1e6, -0.0,
                  240.0 + 8.0, np.nan, 2.0 ** -10 + 2.0 ** -14])
    got = f8.e4m3_encode(x)
    want = [0x38,   # halfway between 1 and 1.125 -> mantissa 0
            0x3A,   # halfway between 1.125 and 1.25 -> mantissa 2
            0x00,   # half the smallest subnormal -> 0
            0x02,   # halfway between 2^-9 and 2^-8 -> 2^-8
            0x7E, 0x7E, 0x7E, 0xFE,  # clamped to +-448
            0x80,   # -0 keeps its sign
            0x78,   # halfway between 240 and 256 -> 256 (even mantissa 0)
            0x7F,
            0x01]   # just above half the smallest subnormal -> 2^-9 (rounded once)
    assert list(got) == want


def test_encode_matches_library_cast():
    """Library special case: torch's float8_e4m3fn cast (round to nearest
    even) agrees on random values inside the range and on every midpoint
    between neighbouring values."""
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.uniform(-448, 448, 20000),
                        rng.standard_normal(20000) * np.exp2(rng.uniform(-14, 8, 20000))])
    x = np.clip(x.astype(np.float32), -448, 448).astype(np.float64)
    v = f8.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mid = (v[:-1] + v[1:]) / 2
    x = np.concatenate([x, mid, -mid])
    lib = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(f8.e4m3_encode(x), lib)


def test_quantize_error_bound_and_amax():
    """Per-tensor quantization: every dequantized value is within half a
    step of its input (2^-4 relative for normals, 2^-10 * scale for
    subnormals), and the largest magnitude maps to +-448."""
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(50000) * np.exp2(rng.uniform(-8, 3, 50000))).astype(np.float32)
    x = x.astype(np.float64)
    codes, scale, inv = f8.quantize_per_tensor(x)
    amax = np.max(np.abs(x))
    assert scale == np.float32(amax) / np.float32(448.0)
    assert inv == np.float32(448.0) / np.float32(amax)
    deq = f8.dequantize(codes, scale)
    err = np.abs(deq - x)
    bound = 2.0 ** -4 * np.abs(x) * 1.0001 + 2.0 ** -10 * float(scale) * 1.0001
    assert np.all(err <= bound)
    assert abs(f8.e4m3_decode(codes[np.argmax(np.abs(x))])) == 448.0


def test_quantize_zero_tensor():
    codes, scale, inv = f8.quantize_per_tensor(np.zeros(64))
    assert np.all(codes == 0) and scale == 1.0 and inv == 1.0


def _mutant(old, new):
    src = textwrap.dedent(inspect.getsource(f8.e4m3_encode))
    assert src.count(old) == 1, old
    ns = {}
    exec(compile(src.replace(old, new), "<mutant e4m3_encode>", "exec"), f8.__dict__, ns)
    return ns["e4m3_encode"]


MUTANTS = [
    # round half up instead of half to even
    ("q = np.rint(a / spacing)", "q = np.floor(a / spacing + 0.5)"),
    # subnormals given the spacing of their own binade
    ("e = np.maximum(E - 1, _MIN_NORMAL_EXP)", "e = E - 1"),
    # no saturation
    ("v = np.minimum(q * spacing, E4M3_MAX)", "v = q * spacing"),
    # exponent bias off by one
    ("efield = np.where(is_sub, 0, ev + _BIAS)", "efield = np.where(is_sub, 0, ev + _BIAS + 1)"),
]


@pytest.mark.parametrize("old,new", MUTANTS)
def test_planted_encoder_mistake_is_caught(old, new, monkeypatch):
    monkeypatch.setattr(f8, "e4m3_encode", _mutant(old, new))
    caught = 0
    for check in (test_round_trip_every_code, test_ties_go_to_even_and_saturate,
                  test_quantize_error_bound_and_amax, test_encode_matches_library_cast):
        try:
            check()
        except (AssertionError, ValueError, OverflowError):
            caught += 1
    assert caught > 0


def _worst_case_change(q, k, v, scale, p_exp=8):
    """Output change when every numerator 2^p_exp * 2^(s - M) of a causal
    row moves by the largest E4M3 rounding error, in the direction of its
    value's sign, column by column (one head, all keys visible up to the
    row). Written out directly: normal numerators by 2^-4 of themselves,
    subnormal ones by 2^-10."""
    n, d = q.shape
    s = scale * (q @ k.T)
    s = np.where(np.tril(np.ones((n, n), dtype=bool)), s, -np.inf)
    e = np.exp(s - s.max(axis=1, keepdims=True))
    P = 2.0 ** p_exp * e
    L = e.sum(axis=1)
    out = np.zeros((n, d))
    for j in range(d):
        sg = np.sign(v[:, j])[None, :]
        Pt = np.where(P < 2.0 ** -6, P + 2.0 ** -10 * sg, P * (1 + 2.0 ** -4 * sg))
        Pt = np.where(e > 0, Pt, 0.0)
        out[:, j] = np.abs((Pt - P) @ v[:, j]) / (2.0 ** p_exp * L)
    return out


@pytest.mark.parametrize("spread", [0.3, 9.0])
def test_pv_rounding_bound_is_reached_by_the_worst_rounding(spread):
    """The bound equals the change caused by the worst admissible rounding
    (every numerator moved by its largest error towards its value's sign):
    with close scores (all numerators normal) and with spread-out ones (many
    subnormal)."""
    rng = np.random.default_rng(11)
    n, d = 48, 8
    q = rng.standard_normal((n, 1, d)) * spread
    k = rng.standard_normal((n, 1, d))
    v = rng.standard_normal((n, 1, d))
    pos = np.arange(n)
    B = f8.pv_rounding_bound(q, k, v, pos, pos, scale=1.0 / np.sqrt(d))[:, 0, :]
    W = _worst_case_change(q[:, 0], k[:, 0], v[:, 0], 1.0 / np.sqrt(d))
    np.testing.assert_allclose(B, W, rtol=1e-9, atol=1e-15)


def test_quantize_rows_scales_each_row_on_its_own():
    """Rows of very different ranges: each row's largest magnitude maps to
    +-448 with that row's scale, and each row is within its own half-step
    bound."""
    rng = np.random.default_rng(9)
    x = rng.standard_normal((6, 128)) * np.array([1e-3, 1, 30, 0.2, 5e2, 7])[:, None]
    x = x.astype(np.float32).astype(np.float64)
    codes, scales = f8.quantize_rows(x)
    for i in range(6):
        amax = np.abs(x[i]).max()
        assert scales[i] == np.float32(amax) / np.float32(448.0)
        assert abs(f8.e4m3_decode(codes[i, np.argmax(np.abs(x[i]))])) == 448.0
        err = np.abs(f8.dequantize(codes[i], scales[i]) - x[i])
        assert np.all(err <= 2.0 ** -4 * np.abs(x[i]) * 1.0001 + 2.0 ** -10 * float(scales[i]) * 1.0001)
