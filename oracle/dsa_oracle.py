"""Plain float64 CPU oracle of the DSA hot path: Lightning Indexer + Sparse Flash Attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference arm of ``bench.py`` may import this module.  The product path (the
CUDA library and its Python binding) never imports, links or runs it, and it shares no
code with that path: it reads only the seeded arrays of ``dsa_workloads``.

What it computes, step by step, with the passage each step follows:

1. Page translation -- logical token t of sequence b lives in physical page
   ``block_table[b, t // 64]`` at slot ``t % 64``: the fused indexer "directly reads
   paged KV cache" ("Day0 Inference Optimization on Ascend CANN", section 2, "Deep Fusion
   of LI and SFA"; "Inference Acceleration for Next-Gen Attention Architectures",
   section 3.2, "paged addressing and gather-read").
2. Dequantisation -- bf16 bits to the real they encode; e4m3 bytes times the per-token
   f32 scale; e4m3 bytes times 2^(E8M0 - 127) per group of 32 elements (MXFP8 with a
   group of 32: "Day0 Inference Optimization on Ascend CANN", section 3, "Full
   Quantization of LI with MXFP8"; "Adapting and Optimizing Inference for a New Model
   Architecture on Ascend", section 4.2).
3. Relevance scoring and head weighting -- per-head dot products of the indexer query
   with each key (``matmul(query, paged_k_cache, transposed)``), times the per-head
   weight, summed over heads: I[t] = sum_h w_h * (q_h . k_t) ("Adapting and Optimizing
   Inference ...", section 3.1, the fused indexer sketch; the head sum is the plain
   reading of "head weight weighting" followed by one Top-K per token).
4. Top-K -- the K largest I[t] among the visible positions t <= query position, ties to
   the lower position; returned as ascending positions padded with -1 ("Adapting and
   Optimizing Inference ...", section 3.1, ``topk_select``; "Day0 Inference Optimization
   on Ascend CANN", section 1: the indexer "selects the Top-K historical positions").
5. Sparse attention -- softmax attention of each SFA head over only the selected latent
   rows: z_j = scale * q . kv[t_j] over all 576 latent dims, p = softmax(z),
   o = sum_j p_j * kv[t_j, :512] ("Adapting and Optimizing Inference ...", section 3.1:
   the sparse attention "reads the main attention KV entries according to the selected
   indices"; DSA builds on MLA, whose latent row serves as key and, truncated to its
   first 512 dims, as value).

Every function is the definition written out in float64, with a library primitive
(matmul, sort, exp) as a step at most; nothing is blocked, fused or reordered.
"""
from __future__ import annotations

import numpy as np

PAGE_SIZE = 64


# ---------------------------------------------------------------------------------
# Storage decoders
# ---------------------------------------------------------------------------------
def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64: the top half of an IEEE binary32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def decode_e4m3(bits: np.ndarray) -> np.ndarray:
    """OCP FP8 E4M3 ("fn" variant: no infinities, S.1111.111 is NaN) -> float64.

    1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 encodes
    subnormals m/8 * 2^-6.
    """
    u = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    sign = np.where(u & 0x80, -1.0, 1.0)
    e = (u >> 3) & 0xF
    m = (u & 0x7).astype(np.float64)
    normal = np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64))
    sub = np.ldexp(m / 8.0, -6)
    v = np.where(e == 0, sub, normal) * sign
    return np.where((u & 0x7F) == 0x7F, np.nan, v)


def decode_e8m0(bits: np.ndarray) -> np.ndarray:
    """E8M0 scale byte -> float64 power of two 2^(byte - 127); 0xFF is NaN."""
    u = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    return np.where(u == 0xFF, np.nan, np.ldexp(1.0, u - 127))


# ---------------------------------------------------------------------------------
# Step 1: page translation (gathers in logical order)
# ---------------------------------------------------------------------------------
def logical_rows(cache: np.ndarray, block_table_row: np.ndarray, positions: np.ndarray) -> np.ndarray:
    """Rows of a paged cache [pages, 64, ...] for logical positions of one sequence."""
    positions = np.asarray(positions, dtype=np.int64)
    pages = block_table_row[positions // PAGE_SIZE]
    return cache[pages, positions % PAGE_SIZE]


# ---------------------------------------------------------------------------------
# Step 2: dequantisation
# ---------------------------------------------------------------------------------
def _decode(bits: np.ndarray) -> np.ndarray:
    return decode_bf16(bits) if bits.dtype == np.uint16 else decode_e4m3(bits)


def dequant_index_query(wl, token: int) -> np.ndarray:
    """Indexer query of one token, [H_I, d] float64, scales applied."""
    q = _decode(wl.idx_q[token])
    s = wl.idx_q_scale
    if s is None:
        return q
    if s.dtype == np.float32:                      # per-token f32 scale
        return q * float(s[token])
    g = s[token].shape[-1]                         # E8M0 per group of d/g elements
    return q * np.repeat(decode_e8m0(s[token]), q.shape[-1] // g, axis=-1)


def dequant_index_keys(wl, b: int, positions: np.ndarray) -> np.ndarray:
    """K-index rows of sequence b at the given logical positions, [n, d] float64."""
    k = _decode(logical_rows(wl.idx_k, wl.block_table[b], positions))
    s = wl.idx_k_scale
    if s is None:
        return k
    rows = logical_rows(s, wl.block_table[b], positions)
    if s.dtype == np.float32:
        return k * rows.astype(np.float64)[:, None]
    g = rows.shape[-1]
    return k * np.repeat(decode_e8m0(rows), k.shape[-1] // g, axis=-1)


# ---------------------------------------------------------------------------------
# Step 3: relevance scoring, head weighting, head sum
# ---------------------------------------------------------------------------------
def index_scores(q: np.ndarray, w: np.ndarray, k: np.ndarray, act: str = "identity") -> np.ndarray:
    """I[t] = sum_h w[h] * act(q[h] . k[t]);  q [H_I, d], w [H_I], k [n, d] -> [n]."""
    s = k @ q.T                                   # [n, H_I] per-head relevance
    if act == "relu":
        s = np.maximum(s, 0.0)
    elif act != "identity":
        raise ValueError(act)
    weighted = s * w[None, :]                     # head weighting
    return weighted.sum(axis=1)                   # head sum


def visible_count(wl, token: int) -> int:
    """Number of positions the query token may select: t <= q_pos and t < L_b."""
    b = int(wl.q_seq[token])
    return max(0, min(int(wl.q_pos[token]) + 1, int(wl.seq_lens[b])))


# ---------------------------------------------------------------------------------
# Step 4: Top-K
# ---------------------------------------------------------------------------------
def topk_select(scores: np.ndarray, k: int) -> np.ndarray:
    """Positions of the k largest scores, ties to the lower position.

    A full stable sort (score descending, then position ascending); the first
    min(k, n) positions are returned in ascending order, padded with -1 to length k.
    """
    n = scores.shape[0]
    s = np.where(scores == 0.0, 0.0, scores)      # -0 and +0 are the same score
    order = np.lexsort((np.arange(n), -s))        # last key is primary
    chosen = np.sort(order[:min(k, n)])
    out = np.full(k, -1, dtype=np.int32)
    out[:chosen.shape[0]] = chosen
    return out


def indexer_topk(wl, token: int, act: str = "identity"):
    """Steps 1-4 for one query token: (indices [K] int32, scores of those indices)."""
    b = int(wl.q_seq[token])
    n = visible_count(wl, token)
    pos = np.arange(n)
    scores = index_scores(dequant_index_query(wl, token), wl.head_w[token].astype(np.float64),
                          dequant_index_keys(wl, b, pos), act)
    idx = topk_select(scores, wl.spec.topk)
    sel = idx[idx >= 0]
    sc = np.full(idx.shape[0], np.nan)
    sc[:sel.shape[0]] = scores[sel]
    return idx, sc


# ---------------------------------------------------------------------------------
# Step 5: sparse attention over the selected latent rows
# ---------------------------------------------------------------------------------
def sparse_attention(q: np.ndarray, rows: np.ndarray, scale: float, v_dim: int = 512) -> np.ndarray:
    """softmax(scale * q rows^T) rows[:, :v_dim];  q [H, D], rows [n, D] -> [H, v_dim].

    With no selected row the attention has no mass and the output is 0.
    """
    if rows.shape[0] == 0:
        return np.zeros((q.shape[0], v_dim))
    z = scale * (q @ rows.T)
    z = z - z.max(axis=1, keepdims=True)
    p = np.exp(z)
    p = p / p.sum(axis=1, keepdims=True)
    return p @ rows[:, :v_dim]


def decode_latent_fp8(codes: np.ndarray, scales: np.ndarray, rope_bits: np.ndarray) -> np.ndarray:
    """FP8 latent rows -> float64 [..., 576]: each e4m3 latent element times the f32 scale
    of its 128-element tile (element j uses scale j // 128), followed by the bf16 rope
    dims.  FP8 quantisation of the SFA cache per token and head in tiles of 128 elements
    ("Day0 Inference Optimization on Ascend CANN", section 3, "FP8 Block Quantization
    for SFA KV Cache"; "Adapting and Optimizing Inference ...", section 4.3); the latent
    row has no heads, and the pages do not say how the 64 rope dims are stored: bf16
    here."""
    lat = decode_e4m3(codes) * np.repeat(np.asarray(scales, dtype=np.float64), 128, axis=-1)
    return np.concatenate([lat, decode_bf16(rope_bits)], axis=-1)


def latent_rows(wl, b: int, positions: np.ndarray) -> np.ndarray:
    """float64 latent rows [n, 576] of sequence b at the given positions (bf16 or FP8 cache)."""
    bt = wl.block_table[b]
    if wl.kv is not None:
        return decode_bf16(logical_rows(wl.kv, bt, positions))
    return decode_latent_fp8(logical_rows(wl.kv_codes, bt, positions), logical_rows(wl.kv_scale, bt, positions),
                             logical_rows(wl.kv_rope, bt, positions))


def sfa(wl, token: int, idx: np.ndarray) -> np.ndarray:
    """Sparse Flash Attention of one query token over its index list, [H, 512] float64."""
    b = int(wl.q_seq[token])
    sel = idx[idx >= 0]
    rows = latent_rows(wl, b, sel)
    return sparse_attention(decode_bf16(wl.sfa_q[token]), rows, wl.spec.softmax_scale)


def step(wl, token: int, act: str = "identity"):
    """The whole hot path for one query token: (indices, their scores, SFA output)."""
    idx, sc = indexer_topk(wl, token, act)
    return idx, sc, sfa(wl, token, idx)


# ---------------------------------------------------------------------------------
# Exactness certificate for the indexer scores in float32
# ---------------------------------------------------------------------------------
def _lsb_exponent(x: np.ndarray) -> np.ndarray:
    """Exponent of the lowest set significand bit of each finite float64 (inf for 0).

    |x| = sig * 2^e0 with sig the integer significand (implicit bit included for
    normals); the lowest set bit of sig is sig & -sig, an exact power of two.
    """
    x = np.asarray(x, dtype=np.float64)
    bits = np.abs(x).view(np.int64)
    expf = (bits >> 52) & 0x7FF
    mant = bits & ((1 << 52) - 1)
    sig = np.where(expf > 0, mant | (1 << 52), mant)
    e0 = np.where(expf > 0, expf - 1075, -1074)
    low = sig & (-sig)
    with np.errstate(divide="ignore"):
        tz = np.log2(low.astype(np.float64))
    return np.where(sig == 0, np.inf, e0 + tz)


def collapsed_query_certificate(wl, token: int) -> float:
    """max over dims d of Q_d / (2^24 A_d) for the head-collapsed query q~_d = sum_h w_h q_hd.

    With the identity activation the score is also sum_d q~_d k_td.  Q_d = sum_h
    |w_h q_hd| bounds every partial sum of q~_d and A_d is the coarsest power of two
    dividing all its terms; a value < 1 means q~ is reached exactly in float32 (any
    order), after which every product q~_d k_td and sum of them is a partial sum of the
    score's terms, exact under exactness_certificate.
    """
    q = dequant_index_query(wl, token)                   # [H, d], scales included
    w = wl.head_w[token].astype(np.float64)              # [H]
    Q = (np.abs(q) * np.abs(w)[:, None]).sum(axis=0)     # [d]
    a = (_lsb_exponent(q) + _lsb_exponent(w)[:, None]).min(axis=0)
    ratio = np.where(np.isfinite(a), Q / np.ldexp(1.0, 24) / np.exp2(np.where(np.isfinite(a), a, 0)), 0.0)
    return float(ratio.max())


def exactness_certificate(wl, token: int) -> float:
    """max over visible t of S_t / (2^24 G_t) for the score I[t].

    S_t = sum_{h,d} |w_h q_hd k_td| bounds every partial sum of the score's terms and
    G_t is the coarsest power of two dividing every term (each term is an exact product
    of its factors' significands).  Every partial sum is then a multiple of G_t no larger
    than S_t in magnitude; below 2^24 G_t such a number is an exact binary32, so a value
    < 1 means float32 arithmetic in any order and grouping reaches I[t] exactly.
    """
    b = int(wl.q_seq[token])
    n = visible_count(wl, token)
    if n == 0:
        return 0.0
    q = dequant_index_query(wl, token)
    w = wl.head_w[token].astype(np.float64)
    k = dequant_index_keys(wl, b, np.arange(n))
    S = np.abs(k) @ (np.abs(q) * np.abs(w)[:, None]).sum(axis=0)
    a = (_lsb_exponent(q) + _lsb_exponent(w)[:, None]).min(axis=0)     # [d]
    g = (_lsb_exponent(k) + a[None, :]).min(axis=1)                   # [n]
    ratio = np.where(np.isfinite(g), S / np.ldexp(1.0, 24) / np.exp2(np.where(np.isfinite(g), g, 0)), 0.0)
    return float(ratio.max())
