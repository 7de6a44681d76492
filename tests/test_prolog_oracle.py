"""Pins of the index-prolog oracle (MXFP8 quantisation with groups of 32, cache append)
against the E4M3 / E8M0 definitions, closed forms and brute force: no GPU."""
import numpy as np
import pytest

from oracle import mx_quant as M
from oracle.dsa_oracle import decode_e4m3, decode_e8m0


def test_every_finite_code_rounds_to_itself():
    """Each finite non-negative E4M3 value, and its negation, maps back to its code."""
    codes = np.arange(0x7F, dtype=np.uint8)
    v = decode_e4m3(codes)
    assert np.array_equal(M.e4m3_round(v), codes)
    neg = M.e4m3_round(-v[1:])
    assert np.array_equal(neg, codes[1:] | 0x80)


@pytest.mark.parametrize("x, code", [
    (1.0625, 0x38),      # halfway between 1 and 1.125: the even code (1.0)
    (1.1875, 0x3A),      # halfway between 1.125 and 1.25: 1.25
    (2.0 ** -10, 0x00),  # half the smallest subnormal: 0
    (3 * 2.0 ** -10, 0x02),  # halfway between 2^-9 (code 1) and 2^-8 (code 2)
    (0.0625 + 2.0 ** -9, 0x18),  # 2^-4 + a quarter step (step 2^-7): down to 2^-4
    (449.0, 0x7E), (1e30, 0x7E),  # beyond the largest normal: saturate at 448
    (-2.0 ** -12, 0x80),  # a negative value that rounds to zero keeps its sign
])
def test_rounding_closed_forms(x, code):
    assert int(M.e4m3_round(np.array([x]))[0]) == code


def test_rounding_is_nearest_on_random_values():
    """Brute-force property: no finite E4M3 value is nearer than the chosen one."""
    rng = np.random.default_rng(5)
    v = np.ldexp(rng.uniform(-1, 1, 4000), rng.integers(-12, 10, 4000))
    c = M.e4m3_round(v)
    got = np.abs(decode_e4m3(c))
    a = np.minimum(np.abs(v), 448.0)
    table = decode_e4m3(np.arange(0x7F, dtype=np.uint8))
    nearest = np.abs(a[:, None] - table[None, :]).min(axis=1)
    assert np.allclose(np.abs(got - a), nearest, rtol=0, atol=0)
    assert np.all(np.signbit(decode_e4m3(c)) == np.signbit(v))


@pytest.mark.parametrize("amax, e", [
    (1.0, -8), (448.0, 0), (511.0, 0), (512.0, 1), (256.0, 0), (255.0, -1),
    (2.0 ** 130, 122), (2.0 ** -140, -127), (0.0, -127), (3.0 * 2.0 ** -133, -127),
])
def test_group_exponent_closed_forms(amax, e):
    assert int(M.group_exponent(np.array([amax]))[0]) == e


def test_exact_groups_round_trip():
    """A group built as E4M3 values times 2^s, with one element in [256, 448], has
    shared exponent s, so quantising it returns the codes it was built from."""
    rng = np.random.default_rng(7)
    for _ in range(50):
        s = int(rng.integers(-100, 100))
        codes = rng.integers(0, 0x7F, size=32).astype(np.uint8)
        codes |= (rng.integers(0, 2, size=32) << 7).astype(np.uint8)
        codes[rng.integers(0, 32)] = 0x78 + int(rng.integers(0, 7))  # exponent field 15: 256 .. 448
        codes[codes == 0x80] = 0x00  # -0 and +0 are the same real
        x = np.ldexp(decode_e4m3(codes), s)
        qc, qs = M.quantize_mxfp8(x[None, :])
        assert int(qs[0, 0]) == s + 127
        assert np.array_equal(qc[0], codes)
        assert np.array_equal(M.dequantize_mxfp8(qc, qs)[0], x)


def test_quantisation_error_within_half_step():
    """Every element is within half an E4M3 step (2^-3 of its binade, 2^-9 below the
    normals) of x / 2^e, the scale being the E8M0 power of two; elements whose x / 2^e
    lies in (448, 512) (only a group's largest can) saturate to 448."""
    rng = np.random.default_rng(11)
    x = rng.standard_normal((64, 128)) * np.ldexp(1.0, rng.integers(-20, 20, (64, 1)))
    c, s = M.quantize_mxfp8(x)
    back = M.dequantize_mxfp8(c, s)
    scale = np.repeat(decode_e8m0(s), 32, axis=1)
    y = np.abs(x) / scale
    assert np.all((y >= 256).reshape(64, 4, 32).any(axis=-1))  # amax / 2^e in [256, 512)
    assert np.all(y < 512)
    sat = y > 448
    assert np.all(np.abs(decode_e4m3(c[sat])) == 448.0)
    step = np.maximum(np.ldexp(1.0, np.floor(np.log2(y + 1e-300)).astype(int) - 3), 2.0 ** -9)
    ok = np.abs(back - x) <= 0.5 * step * scale
    assert np.all(ok | sat)


def test_zero_group():
    c, s = M.quantize_mxfp8(np.zeros((2, 64)))
    assert np.all(c == 0) and np.all(s == 0)


def test_append_places_rows_by_page_translation():
    rng = np.random.default_rng(3)
    pages, dim = 12, 64
    cc = rng.integers(0, 256, (pages, 64, dim)).astype(np.uint8)
    cs = rng.integers(0, 256, (pages, 64, dim // 32)).astype(np.uint8)
    bt = np.array([[5, 2, 9], [0, 11, -1]], dtype=np.int32)
    seq = np.array([0, 0, 1, 1, 1])
    pos = np.array([70, 191, 0, 100, 130])  # the last one lands on page -1: skipped
    codes = rng.integers(0, 256, (5, dim)).astype(np.uint8)
    scales = rng.integers(0, 256, (5, dim // 32)).astype(np.uint8)
    oc, os_, bad = M.append_rows(cc, cs, bt, seq, pos, codes, scales)
    assert bad == [4]
    assert np.array_equal(oc[2, 6], codes[0]) and np.array_equal(os_[2, 6], scales[0])
    assert np.array_equal(oc[9, 63], codes[1])
    assert np.array_equal(oc[0, 0], codes[2])
    assert np.array_equal(oc[11, 36], codes[3])
    touched = {(2, 6), (9, 63), (0, 0), (11, 36)}
    for p in range(pages):
        for t in range(64):
            if (p, t) not in touched:
                assert np.array_equal(oc[p, t], cc[p, t]) and np.array_equal(os_[p, t], cs[p, t])
