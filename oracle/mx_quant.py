"""Plain float64 CPU oracle of the index prolog: dynamic MXFP8 quantisation of index rows
and their append to the paged K-index cache.

TEST INFRASTRUCTURE ONLY.  Only ``tests/`` may import this module (the same rule as
``dsa_oracle``); the CUDA library never imports, links or runs it and shares no code
with it.

What it computes, with the passage each step follows:

1. MXFP8 quantisation with groups of 32: every 32 consecutive elements of a row share
   one scaling factor, chosen per group from the data ("Day0 Inference Optimization on
   Ascend CANN", section 3, "Full Quantization of LI with MXFP8"; "Adapting and
   Optimizing Inference for a New Model Architecture on Ascend", section 4.2).  The
   pages leave the rule for the factor open; this module takes the one of the OCP
   Microscaling (MX) format: the factor is the power of two 2^e with
   e = floor(log2(amax)) - 8, amax the group's largest magnitude and 8 the exponent of
   E4M3's largest normal (448 = 1.75 * 2^8), clamped to the E8M0 range [-127, 127]
   (e = -127 for an all-zero group); each element becomes the E4M3 value nearest to
   x / 2^e, ties to the even code, magnitudes beyond 448 saturating to 448.  The factor
   is stored as the E8M0 byte e + 127.
2. Append: the new key of token i (sequence b_i, position t_i) goes to physical page
   ``block_table[b_i, t_i // 64]``, slot ``t_i % 64`` (page translation as in the fused
   indexer, which "directly reads paged KV cache": "Day0 Inference Optimization on
   Ascend CANN", section 2).
"""
from __future__ import annotations

import numpy as np

from .dsa_oracle import decode_e4m3

GROUP = 32
E4M3_MAX = 448.0
# the finite non-negative E4M3 values, indexed by their code 0x00 .. 0x7E (ascending)
_E4M3_POS = decode_e4m3(np.arange(0x7F, dtype=np.uint8))


def e4m3_round(v: np.ndarray) -> np.ndarray:
    """float64 -> E4M3 codes (uint8): nearest value, ties to the even code, |v| > 448
    saturating to 448.  Brute force over the 127 non-negative finite values."""
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), E4M3_MAX).reshape(-1)
    d = np.abs(a[:, None] - _E4M3_POS[None, :])          # distance to every value
    best = d.min(axis=1, keepdims=True)
    cand = d == best                                      # one value, or two on a tie
    codes = np.arange(0x7F)
    even = cand & (codes[None, :] % 2 == 0)
    pick = np.where(even.any(axis=1), np.argmax(even, axis=1), np.argmax(cand, axis=1))
    sign = np.signbit(v.reshape(-1)).astype(np.int64) << 7
    return (pick | sign).astype(np.uint8).reshape(v.shape)


def group_exponent(amax: np.ndarray) -> np.ndarray:
    """Shared exponent e of each group from its largest magnitude (int64)."""
    amax = np.asarray(amax, dtype=np.float64)
    _, ex = np.frexp(amax)                # amax = m * 2^ex with m in [0.5, 1)
    fl = ex.astype(np.int64) - 1          # floor(log2(amax)) for amax > 0
    return np.where(amax > 0, np.clip(fl - 8, -127, 127), -127)


def quantize_mxfp8(x: np.ndarray):
    """Rows [..., dim] (dim a multiple of 32, float64 of finite values) -> (E4M3 codes
    uint8 [..., dim], E8M0 scale bytes uint8 [..., dim / 32])."""
    x = np.asarray(x, dtype=np.float64)
    dim = x.shape[-1]
    assert dim % GROUP == 0
    g = x.reshape(x.shape[:-1] + (dim // GROUP, GROUP))
    e = group_exponent(np.abs(g).max(axis=-1))
    y = np.ldexp(g, -e[..., None])        # x / 2^e, exact
    codes = e4m3_round(y).reshape(x.shape)
    return codes, (e + 127).astype(np.uint8)


def dequantize_mxfp8(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Inverse reading: E4M3 value times 2^(byte - 127) per group of 32."""
    v = decode_e4m3(codes)
    s = np.ldexp(1.0, np.asarray(scales, dtype=np.int64) - 127)
    return (v.reshape(v.shape[:-1] + (-1, GROUP)) * s[..., None]).reshape(v.shape)


def append_rows(cache_codes: np.ndarray, cache_scales: np.ndarray, block_table: np.ndarray,
                seq: np.ndarray, pos: np.ndarray, codes: np.ndarray, scales: np.ndarray):
    """Copies of the paged cache ([pages, 64, dim] codes, [pages, 64, dim / 32] scales)
    with row i written at the slot of (seq[i], pos[i]); rows whose position or page is
    outside the table are skipped and reported.  Returns (codes, scales, bad rows)."""
    out_c, out_s = cache_codes.copy(), cache_scales.copy()
    n_pages, page = cache_codes.shape[0], cache_codes.shape[1]
    bad = []
    for i in range(len(seq)):
        b, t = int(seq[i]), int(pos[i])
        if b < 0 or b >= block_table.shape[0] or t < 0 or t // page >= block_table.shape[1]:
            bad.append(i)
            continue
        pg = int(block_table[b, t // page])
        if pg < 0 or pg >= n_pages:
            bad.append(i)
            continue
        out_c[pg, t % page] = codes[i]
        out_s[pg, t % page] = scales[i]
    return out_c, out_s, bad
