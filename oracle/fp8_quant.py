"""Plain CPU oracle of FP8 block quantisation for the caches and of the cache appends.

TEST INFRASTRUCTURE ONLY.  Only ``tests/`` may import this module (the same rule as
``dsa_oracle``); the CUDA library never imports, links or runs it and shares no code
with it.

What it computes, with the passage each step follows:

1. FP8 block quantisation.  The sparse attention's KV cache is quantised to FP8 per
   token in tiles of 128 elements, which halves the bytes the attention reads ("Day0
   Inference Optimization on Ascend CANN", section 3, "FP8 Block Quantization for SFA
   KV Cache"; "Adapting and Optimizing Inference for a New Model Architecture on
   Ascend", section 4.3).  The MLA latent row has no heads, so its 512 latent dims form
   four tiles of 128; the pages do not say how the 64 rope dims are stored, and they
   stay bf16.  The K-index cache's FP8 format with one f32 scale per token (the FP8
   decode workload) is the same rule with the whole row as one block.  The pages leave
   the scale rule open; this module takes absmax scaling, the plain block-quantisation
   reading: the block's f32 scale is s = amax / 448 (amax the block's largest
   magnitude, 448 the largest finite E4M3 value), rounded to f32; each element becomes
   the E4M3 value nearest to the f32 quotient x / s, ties to the even code, magnitudes
   beyond 448 saturating to 448; an all-zero block gets s = 1 and zero codes.  Both
   divisions are IEEE binary32 divisions (correctly rounded), so a device computing them
   in f32 reaches the same codes.  Dequantisation is code * s.
2. Append: the new row of token i (sequence b_i, position t_i) goes to physical page
   ``block_table[b_i, t_i // 64]``, slot ``t_i % 64`` (page translation as everywhere on
   the path: the operators read the paged caches directly, "Day0 Inference
   Optimization on Ascend CANN", section 2).
"""
from __future__ import annotations

import numpy as np

from .dsa_oracle import decode_bf16, decode_e4m3
from .mx_quant import e4m3_round

E4M3_MAX = 448.0
TILE = 128
V_DIM = 512


def block_scale(amax: np.ndarray) -> np.ndarray:
    """f32 scale of each block from its largest magnitude: amax / 448 in binary32, or 1
    for an all-zero block."""
    amax = np.asarray(amax, dtype=np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        s = amax / np.float32(E4M3_MAX)
    return np.where(amax > 0, s, np.float32(1.0)).astype(np.float32)


def quantize_blocks(x: np.ndarray, block: int):
    """Rows [..., n] (n a multiple of `block`, finite values exactly representable in
    f32) -> (E4M3 codes uint8 [..., n], f32 scales [..., n / block])."""
    x = np.asarray(x, dtype=np.float32)
    n = x.shape[-1]
    assert n % block == 0
    g = x.reshape(x.shape[:-1] + (n // block, block))
    s = block_scale(np.abs(g).max(axis=-1))
    y = g / s[..., None]                   # binary32 quotient, correctly rounded
    codes = e4m3_round(y.astype(np.float64)).reshape(x.shape)
    return codes, s


def dequantize_blocks(codes: np.ndarray, scales: np.ndarray, block: int) -> np.ndarray:
    """code * scale per block, float64."""
    v = decode_e4m3(codes)
    s = np.asarray(scales, dtype=np.float64)
    return (v.reshape(v.shape[:-1] + (-1, block)) * s[..., None]).reshape(v.shape)


def quantize_index_rows(k_bits: np.ndarray):
    """bf16 key rows [T, d] -> (E4M3 codes [T, d], f32 per-token scales [T])."""
    codes, s = quantize_blocks(decode_bf16(k_bits), k_bits.shape[-1])
    return codes, s[..., 0]


def quantize_latent_rows(row_bits: np.ndarray):
    """bf16 latent rows [T, 576] -> (E4M3 codes of the 512 latent dims [T, 512], f32 scale
    per 128-dim tile [T, 4], the 64 rope dims as bf16 bits [T, 64], unchanged)."""
    row_bits = np.asarray(row_bits, dtype=np.uint16)
    codes, s = quantize_blocks(decode_bf16(row_bits[..., :V_DIM]), TILE)
    return codes, s, row_bits[..., V_DIM:].copy()


def append(caches, block_table: np.ndarray, seq: np.ndarray, pos: np.ndarray, rows):
    """Copies of the paged caches (each [pages, 64, ...]) with row i of every array in
    `rows` written at the slot of (seq[i], pos[i]); tokens whose position or page is
    outside the table are skipped and reported.  Returns (caches, bad tokens)."""
    out = [c.copy() for c in caches]
    n_pages, page = out[0].shape[0], out[0].shape[1]
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
        for c, r in zip(out, rows):
            c[pg, t % page] = r[i]
    return out, bad
