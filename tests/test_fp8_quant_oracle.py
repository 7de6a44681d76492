"""Pins of the FP8 block-quantisation oracle (per-token K-index rows, 128-dim latent tiles,
cache appends) against closed forms, exact rational arithmetic and properties; and
planted mistakes in it, each caught by a pin.  No GPU."""
from fractions import Fraction

import numpy as np
import pytest

from oracle import fp8_quant as F
from oracle.dsa_oracle import decode_bf16, decode_e4m3

import dsa_workloads as W


def _f32_nearest(q: Fraction) -> np.float32:
    """The binary32 value nearest to the rational q (ties to the even significand),
    found from the exact rational, independently of any floating-point division."""
    a = np.float32(float(q))                      # within one ulp of q
    cands = [np.nextafter(a, np.float32(-np.inf)), a, np.nextafter(a, np.float32(np.inf))]
    dist = [abs(Fraction(float(c)) - q) for c in cands]
    best = min(dist)
    tied = [c for c, d in zip(cands, dist) if d == best]
    if len(tied) == 1:
        return tied[0]
    return next(c for c in tied if (int(np.float32(c).view(np.uint32)) & 1) == 0)


def test_scale_is_amax_over_448_in_binary32():
    """Closed forms (powers of two, 7/448 = 2^-6) and, for random bf16 maxima, the binary32
    value nearest to the exact rational amax / 448."""
    assert F.block_scale(np.array([448.0]))[0] == 1.0
    assert F.block_scale(np.array([7.0]))[0] == 2.0 ** -6
    assert F.block_scale(np.array([448.0 * 2 ** -20]))[0] == 2.0 ** -20
    rng = np.random.default_rng(3)
    amax = decode_bf16(W.bf16_bits_from_f32(np.abs(rng.standard_normal(300)).astype(np.float32) * 10 + 1e-3))
    got = F.block_scale(amax)
    for a, s in zip(amax, got):
        assert s == _f32_nearest(Fraction(float(a)) / 448), (a, s)


def test_exact_blocks_round_trip():
    """A block of E4M3 values times a power of two s, holding +-448 s, has scale s and
    decodes back exactly."""
    rng = np.random.default_rng(4)
    vals = decode_e4m3(np.arange(0x7F, dtype=np.uint8))
    for k in (-12, -3, 0, 5):
        blk = rng.choice(vals, size=(6, 128)) * rng.choice([-1.0, 1.0], size=(6, 128))
        blk[:, 17] = 448.0
        x = np.ldexp(blk, k)
        codes, s = F.quantize_blocks(x, 128)
        assert np.all(s == 2.0 ** k)
        assert np.array_equal(F.dequantize_blocks(codes, s, 128), x)


def test_block_maximum_maps_to_448():
    rng = np.random.default_rng(5)
    x = decode_bf16(W.bf16_bits_from_f32(rng.standard_normal((200, 128)).astype(np.float32)))
    codes, s = F.quantize_blocks(x, 128)
    arg = np.abs(x).argmax(axis=1)
    top = decode_e4m3(codes[np.arange(200), arg])
    assert np.all(np.abs(top) == 448.0)
    assert np.all(np.sign(top) == np.sign(x[np.arange(200), arg]))


def test_quantisation_error_within_half_step():
    """|code * s - x| is at most half an E4M3 step at |x| / s (times s), plus the f32
    quotient's own rounding (2^-24 relative)."""
    rng = np.random.default_rng(6)
    x = decode_bf16(W.bf16_bits_from_f32((rng.standard_normal((300, 128)) * np.exp2(rng.integers(-20, 20, (300, 1))))
                                         .astype(np.float32)))
    codes, s = F.quantize_blocks(x, 128)
    y = np.abs(x) / np.repeat(s.astype(np.float64), 128, axis=1)
    # E4M3 step at magnitude y: 2^-9 below 2^-6 (subnormals), else 2^(floor(log2 y) - 3)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.maximum(y, 2.0 ** -6)))
    step = np.exp2(e - 3)
    err = np.abs(F.dequantize_blocks(codes, s, 128) - x)
    bound = np.repeat(s.astype(np.float64), 128, axis=1) * (step / 2) * (1 + 2.0 ** -20) + np.abs(x) * 2.0 ** -23
    assert np.all(err <= bound)


def test_all_zero_block_and_signed_zero():
    x = np.zeros((2, 128))
    x[1] = -0.0
    codes, s = F.quantize_blocks(x, 128)
    assert np.all(s == 1.0)
    assert np.all(codes[0] == 0) and np.all(codes[1] == 0x80)


def test_latent_tiles_are_128_wide_and_rope_is_kept():
    """Element j of the 512 latent dims uses tile j // 128; a large value in tile 2 moves
    only scale 2; the rope dims pass through bit for bit."""
    rng = np.random.default_rng(7)
    row = rng.standard_normal((3, 576)).astype(np.float32)
    row[:, 300] = 1000.0                            # tile 2 (dims 256..383)
    bits = W.bf16_bits_from_f32(row)
    codes, s, rope = F.quantize_latent_rows(bits)
    assert codes.shape == (3, 512) and s.shape == (3, 4) and rope.shape == (3, 64)
    assert np.all(s[:, 2] == F.block_scale(np.array([1000.0]))[0])
    assert np.all(s[:, [0, 1, 3]] < 0.05)
    assert np.array_equal(rope, bits[:, 512:])
    # each tile quantised on its own equals the row quantised as four blocks
    for t in range(4):
        c1, s1 = F.quantize_blocks(decode_bf16(bits[:, 128 * t:128 * (t + 1)]), 128)
        assert np.array_equal(c1, codes[:, 128 * t:128 * (t + 1)]) and np.array_equal(s1[:, 0], s[:, t])


def test_index_rows_use_one_scale_per_token():
    rng = np.random.default_rng(8)
    k = rng.integers(-8, 9, (5, 128)).astype(np.float32)
    k[:, 0] = 8.0
    codes, s = F.quantize_index_rows(W.bf16_bits_from_f32(k))
    assert s.shape == (5,) and np.all(s == 8.0 / 448.0 * np.float32(1))
    assert np.allclose(F.dequantize_blocks(codes, s[:, None], 128), k, rtol=2 ** -4, atol=0)


def test_append_places_rows_by_page_translation():
    bt = np.array([[3, 0], [1, 2]], dtype=np.int32)
    cache = np.zeros((4, 64, 2), dtype=np.int64)
    rows = np.array([[11, 12], [21, 22], [31, 32]])
    (out,), bad = F.append([cache], bt, np.array([0, 1, 1]), np.array([70, 5, 200]), [rows])
    assert bad == [2]                               # position 200 is beyond 2 pages
    assert list(out[0, 6]) == [11, 12]              # seq 0, pos 70 -> page bt[0,1] = 0, slot 6
    assert list(out[1, 5]) == [21, 22]              # seq 1, pos 5 -> page 1, slot 5
    assert out.sum() == 11 + 12 + 21 + 22


# ---------------------------------------------------------------------------------
# planted mistakes: each must fail one of the pins above
# ---------------------------------------------------------------------------------
_orig = {n: getattr(F, n) for n in ["block_scale", "quantize_blocks", "quantize_latent_rows", "append"]}


def _scale_signed_max(amax):            # "amax" from the signed maximum: the sign leaks in
    return _orig["block_scale"](amax) * np.float32(-1)


def _scale_e5m2_max(amax):
    amax = np.asarray(amax, dtype=np.float32)
    return np.where(amax > 0, amax / np.float32(57344.0), np.float32(1)).astype(np.float32)


def _scale_pow2_up(amax):              # the other common reading: amax / 448 rounded up to a power of two
    amax = np.asarray(amax, dtype=np.float64)
    with np.errstate(divide="ignore"):
        e = np.ceil(np.log2(np.where(amax > 0, amax / 448.0, 1.0)))
    return np.where(amax > 0, np.exp2(e), 1.0).astype(np.float32)


def _quant_times_scale(x, block):
    x = np.asarray(x, dtype=np.float32)
    g = x.reshape(x.shape[:-1] + (-1, block))
    s = F.block_scale(np.abs(g).max(axis=-1))
    return F.e4m3_round((g * s[..., None]).astype(np.float64)).reshape(x.shape), s


def _latent_tiles_64(row_bits):
    row_bits = np.asarray(row_bits, dtype=np.uint16)
    c, s = _orig["quantize_blocks"](decode_bf16(row_bits[..., :512]), 64)
    return c, s[..., ::2], row_bits[..., 512:].copy()


def _latent_rope_dropped(row_bits):
    c, s, r = _orig["quantize_latent_rows"](row_bits)
    return c, s, np.zeros_like(r)


def _append_slot_page_swapped(caches, bt, seq, pos, rows):
    return _orig["append"](caches, bt, seq, pos % 64 * 64 + pos // 64, rows)


MUTANTS = {
    "scale from the signed maximum": ("block_scale", _scale_signed_max),
    "scale over E5M2's 57344": ("block_scale", _scale_e5m2_max),
    "scale rounded up to a power of two": ("block_scale", _scale_pow2_up),
    "quotient x * s": ("quantize_blocks", _quant_times_scale),
    "latent tiles of 64": ("quantize_latent_rows", _latent_tiles_64),
    "rope dims dropped": ("quantize_latent_rows", _latent_rope_dropped),
    "append: slot and page swapped": ("append", _append_slot_page_swapped),
}

PINS = [test_scale_is_amax_over_448_in_binary32, test_exact_blocks_round_trip, test_block_maximum_maps_to_448,
        test_quantisation_error_within_half_step, test_all_zero_block_and_signed_zero,
        test_latent_tiles_are_128_wide_and_rope_is_kept, test_index_rows_use_one_scale_per_token,
        test_append_places_rows_by_page_translation]


@pytest.mark.parametrize("label", sorted(MUTANTS))
def test_fp8_quant_oracle_mutants(label, monkeypatch):
    name, fn = MUTANTS[label]
    monkeypatch.setattr(F, name, fn)
    caught = False
    for pin in PINS:
        try:
            pin()
        except Exception:  # an assertion or a shape error both expose the mutant
            caught = True
            break
    assert caught, f"no pin caught the mutant '{label}'"
