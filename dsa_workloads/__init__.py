"""Seeded synthetic inputs for the DSA Lightning Indexer + Sparse Flash Attention path.

This module only draws random values and lays them out in the storage formats the
operators consume (paged caches, page tables, encoded bf16 / e4m3 / E8M0 bytes).  It
holds none of the method's arithmetic: no scoring, no selection, no attention.  Both
the float64 oracle and the CUDA path read the arrays it returns.

Workload shapes follow the five DSA workloads (tiny decode, BF16 decode, FP8 decode,
causal prefill, ragged MXFP8 decode) plus small parity cases.  Value recipes:

* indexer q / K-index: small integers, uniform in [-r, r], stored as bf16 or e4m3
  (both represent every such integer exactly);
* head weights: powers of two;
* per-token scales (FP8 decode): powers of two 2^u, u in [-4, 2];
* MXFP8 (one E8M0 scale per 32 elements, as "Day0 Inference Optimization on Ascend
  CANN", section 3, fixes the group size): elements integers in [-4, 4]; key scale
  exponent = per-token base in [-4, 2] plus a per-group offset in {0, -1}, clipped to
  [-4, 2]; query scale exponent = per-head base in [-1, 1] plus a per-group offset in
  {0, -1}, clipped to [-1, 1]; head weights 2^[-3, 0];
* latent KV and SFA queries: N(0, 1) rounded to bf16 (round to nearest even).

Every slot the operators must never read (tokens past a sequence's length inside its
last page, pool pages no sequence owns) is filled with NaN encodings, so a stray read
shows up as a parity failure.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np

PAGE_SIZE = 64
KV_DIM = 576
V_DIM = 512
MX_GROUP = 32

BF16_NAN = np.uint16(0x7FC0)
E4M3_NAN = np.uint8(0x7F)
E8M0_NAN = np.uint8(0xFF)

# named random streams (index into SeedSequence.spawn)
_S_LAYOUT, _S_LENS, _S_QI, _S_QSCALE, _S_W, _S_KI, _S_KSCALE, _S_KV, _S_QS, _S_KSCALE_GRP, _S_QSCALE_GRP = range(11)


@dataclass(frozen=True)
class Spec:
    """Shape and value recipe of one synthetic workload."""
    name: str
    mode: str                      # "decode" (one query token per sequence), "multi" (several
                                   # per sequence at its last positions) or "prefill"
    batch: int
    seq_lens: tuple = ()           # explicit lengths; empty => drawn (see len_loguniform)
    len_loguniform: tuple = ()     # (lo, hi): L_b = floor(exp(U(ln lo, ln hi)))
    pool_pages: int = 0            # 0 => exactly the pages the sequences use
    idx_heads: int = 64
    idx_dim: int = 128
    idx_dtype: str = "bf16"        # "bf16" | "e4m3"
    idx_scale: str = "none"        # "none" | "per_token" | "mx"
    idx_int_range: int = 8         # q, k integers uniform in [-r, r]
    head_w_exps: tuple = (-6, 0)   # head weights 2^u, u integer in [lo, hi]
    scale_exps: tuple = (-4, 2)    # per-token f32 scales 2^u (FP8 decode)
    topk: int = 2048
    sfa_heads: int = 128
    seed: int = 0
    prefill_tokens: int = 0        # prefill: query tokens 0..T-1 of sequence 0
    tokens_per_seq: int = 1        # multi: query tokens at positions L_b - m .. L_b - 1
    kv_format: str = "bf16"        # latent cache: "bf16", or "fp8_tile128" (latent dims e4m3
                                   # with an f32 scale per 128-element tile, rope dims bf16)
    int_seed: Optional[int] = None  # seed for the integer / latent streams (defaults to seed)
    description: str = ""

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(KV_DIM)


# ---------------------------------------------------------------------------------
# The five workloads (sizes and value distributions as stated for the DSA hot path)
# ---------------------------------------------------------------------------------
TINY_DECODE = Spec(
    name="tiny_decode", mode="decode", batch=1, seq_lens=(2048,),
    idx_heads=4, idx_dim=64, idx_int_range=8, head_w_exps=(-3, 0),
    topk=128, sfa_heads=8, seed=1001,
    description="B=1, query at 2047 over 2048 tokens, 64-token pages randomly permuted; "
                "indexer 4 heads x d64 bf16; top-K 128; SFA 8 heads x 576")
BF16_DECODE = Spec(
    name="bf16_decode", mode="decode", batch=32, seq_lens=(32768,) * 32,
    idx_heads=64, idx_dim=128, idx_int_range=8, head_w_exps=(-6, 0),
    topk=2048, sfa_heads=128, seed=1002,
    description="B=32, L=32768, 64-token pages permuted; indexer 64 heads x d128 bf16; "
                "top-K 2048; SFA 128 heads x 576 bf16")
FP8_DECODE = replace(
    BF16_DECODE, name="fp8_decode", idx_dtype="e4m3", idx_scale="per_token", seed=1003,
    int_seed=1002,
    description="as bf16_decode, indexer q and K-index e4m3 with per-token f32 "
                "power-of-two scales in [2^-4, 2^2]")
CAUSAL_PREFILL = Spec(
    name="causal_prefill", mode="prefill", batch=1, seq_lens=(8192,),
    idx_heads=64, idx_dim=128, idx_int_range=4, head_w_exps=(-6, 0),
    topk=2048, sfa_heads=128, seed=1004, prefill_tokens=8192,
    description="B=1, 8192 query tokens over their own 8192-token prefix; indexer 64 "
                "heads x d128 bf16 in [-4,4], causal, top-K 2048; SFA 128 heads")
RAGGED_MXFP8_DECODE = Spec(
    name="ragged_mxfp8_decode", mode="decode", batch=8, len_loguniform=(8192, 131072),
    pool_pages=32768, idx_heads=64, idx_dim=128, idx_dtype="e4m3", idx_scale="mx",
    idx_int_range=4, head_w_exps=(-3, 0), topk=2048, sfa_heads=128, seed=1005,
    description="B=8, L log-uniform in [8192, 131072], pages scattered over a 2M-token "
                "pool; MXFP8 indexer (E8M0 per 32) 64 heads x d128; top-K 2048; SFA 128")

HEADLINE = [TINY_DECODE, BF16_DECODE, FP8_DECODE, CAUSAL_PREFILL, RAGGED_MXFP8_DECODE]

# The causal prefill with a quantised indexer (both operators run quantised in prefill
# as well as decode): the same integers, K-index and query in e4m3 with per-token f32
# scales, or MXFP8 with the ragged decode's scale recipe
CAUSAL_PREFILL_FP8 = replace(
    CAUSAL_PREFILL, name="causal_prefill_fp8", idx_dtype="e4m3", idx_scale="per_token", seed=1006,
    int_seed=1004,
    description="as causal_prefill, indexer q and K-index e4m3 with per-token f32 power-of-two scales")
CAUSAL_PREFILL_MX = replace(
    CAUSAL_PREFILL, name="causal_prefill_mxfp8", idx_dtype="e4m3", idx_scale="mx", head_w_exps=(-3, 0),
    seed=1007, int_seed=1004,
    description="as causal_prefill, MXFP8 indexer (E8M0 per 32) with the ragged decode's scale recipe")
# Multi-token decode at the BF16 decode's sizes: 4 draft tokens per sequence at its last
# four positions (the rows of a sequence share one K-index stream)
BF16_MULTI_DECODE = replace(
    BF16_DECODE, name="bf16_multi_decode", mode="multi", tokens_per_seq=4, seed=1008, int_seed=1002,
    description="as bf16_decode with 4 query tokens per sequence at its last 4 positions (128 tokens)")

# The BF16 decode with an FP8 latent cache (e4m3 latent dims, an f32 scale per 128-dim
# tile, bf16 rope dims): the attention gathers 656 instead of 1152 bytes per row
FP8KV_DECODE = replace(
    BF16_DECODE, name="bf16_decode_fp8kv", kv_format="fp8_tile128", seed=1009, int_seed=1002,
    description="as bf16_decode with an FP8 latent cache (tiles of 128, f32 scales, bf16 rope)")

EXTRA = [CAUSAL_PREFILL_FP8, CAUSAL_PREFILL_MX, BF16_MULTI_DECODE, FP8KV_DECODE]

# ---------------------------------------------------------------------------------
# Small parity cases: several tiles, ragged tails, lengths below / at / above top-K
# ---------------------------------------------------------------------------------
SMALL_DECODE_BF16 = Spec(
    name="small_decode_bf16", mode="decode", batch=6,
    seq_lens=(1, 37, 256, 257, 1000, 4133), pool_pages=120,
    idx_heads=64, idx_dim=128, topk=256, sfa_heads=128, seed=7001)
SMALL_DECODE_FP8 = replace(SMALL_DECODE_BF16, name="small_decode_fp8", idx_dtype="e4m3",
                           idx_scale="per_token", seed=7002)
SMALL_DECODE_MX = replace(SMALL_DECODE_BF16, name="small_decode_mx", idx_dtype="e4m3",
                          idx_scale="mx", idx_int_range=4, head_w_exps=(-3, 0), seed=7003)
SMALL_TIES = Spec(
    name="small_ties", mode="decode", batch=3, seq_lens=(300, 777, 2100), pool_pages=64,
    idx_heads=4, idx_dim=64, idx_int_range=1, head_w_exps=(0, 0), topk=192,
    sfa_heads=16, seed=7004)
SMALL_PREFILL = Spec(
    name="small_prefill", mode="prefill", batch=1, seq_lens=(700,), pool_pages=20,
    idx_heads=64, idx_dim=128, idx_int_range=4, topk=256, sfa_heads=128, seed=7005,
    prefill_tokens=700)
SMALL_H8 = Spec(
    name="small_h8", mode="decode", batch=2, seq_lens=(129, 2048), pool_pages=40,
    idx_heads=8, idx_dim=64, topk=128, sfa_heads=8, seed=7006)
EMPTY_AND_SHORT = Spec(
    name="empty_and_short", mode="decode", batch=4, seq_lens=(0, 1, 2, 63), pool_pages=8,
    idx_heads=64, idx_dim=128, topk=64, sfa_heads=128, seed=7007)

SMALL_MID = Spec(
    name="small_mid", mode="decode", batch=3, seq_lens=(9000, 12345, 300), pool_pages=400,
    idx_heads=64, idx_dim=128, topk=512, sfa_heads=128, seed=7008,
    description="longest row between 8K and 16K keys (the selection's four-CTA clusters)")

SMALL_SIB = Spec(
    name="small_sib", mode="decode", batch=32,
    seq_lens=(1, 2, 63, 64, 65, 100, 255, 256, 257, 300, 384, 511, 512, 513, 600, 700, 777, 900,
              1000, 1024, 1200, 1500, 1800, 2000, 2048, 2100, 2500, 2800, 3000, 3100, 3500, 4000),
    pool_pages=640, idx_heads=64, idx_dim=128, topk=512, sfa_heads=128, seed=7009,
    description="32 rows, so each token's 512 selected rows run as two splits of four 64-row "
                "tiles merged inside their cluster; rows up to 256 long leave the second split "
                "empty, rows of 257-511 leave it partly padded")

SMALL_MULTI = Spec(
    name="small_multi", mode="multi", batch=4, seq_lens=(70, 300, 1000, 2500), tokens_per_seq=4,
    pool_pages=80, idx_heads=64, idx_dim=128, topk=256, sfa_heads=128, seed=7010,
    description="multi-token decode: 4 query tokens per sequence at its last 4 positions "
                "(a speculative draft), each seeing the prefix up to itself")

# FP8 latent cache (the attention dequantises gathered rows in shared memory)
SMALL_FP8_KV = replace(SMALL_DECODE_BF16, name="small_fp8_kv", kv_format="fp8_tile128", seed=7011,
                       description="as small_decode_bf16 with an FP8 latent cache: e4m3 latent "
                                   "dims with an f32 scale per 128-dim tile, bf16 rope dims")

# e4m3 keys of 64 dims: per-token scales (the register-streamed folded-query kernel) and
# MX scales (the per-head CUDA-core kernel)
SMALL_FP8_D64 = replace(SMALL_DECODE_FP8, name="small_fp8_d64", idx_dim=64, seed=7012,
                        description="as small_decode_fp8 with 64-dim keys")
SMALL_MX_D64 = replace(SMALL_DECODE_MX, name="small_mx_d64", idx_dim=64, seed=7013,
                       description="as small_decode_mx with 64-dim keys (two MX groups per key)")

# quantised prefill (the row-blocked kernel after an exact dequantisation of the keys)
SMALL_PREFILL_FP8 = replace(SMALL_PREFILL, name="small_prefill_fp8", idx_dtype="e4m3", idx_scale="per_token",
                            seed=7015, description="as small_prefill, e4m3 indexer with per-token scales")
SMALL_PREFILL_MX = replace(SMALL_PREFILL, name="small_prefill_mx", idx_dtype="e4m3", idx_scale="mx",
                           head_w_exps=(-3, 0), seed=7016, description="as small_prefill, MXFP8 indexer")
# multi-token decode with 25 draft tokens per sequence: two row blocks per sequence (21 + 4)
SMALL_MULTI25 = Spec(
    name="small_multi25", mode="multi", batch=3, seq_lens=(40, 700, 2100), tokens_per_seq=25,
    pool_pages=60, idx_heads=64, idx_dim=128, topk=256, sfa_heads=128, seed=7017,
    description="25 query tokens per sequence at its last 25 positions")
SMALL_MULTI_FP8 = replace(SMALL_MULTI, name="small_multi_fp8", idx_dtype="e4m3", idx_scale="per_token", seed=7018,
                          description="multi-token decode with an e4m3 indexer (one key stream per token)")

# five attention heads (not a multiple of four) and eight splits per token: the split
# combine over a padded head stride
SMALL_H5 = Spec(
    name="small_h5", mode="decode", batch=3, seq_lens=(300, 777, 2100), pool_pages=60,
    idx_heads=4, idx_dim=64, head_w_exps=(-3, 0), topk=512, sfa_heads=5, seed=7019,
    description="5 SFA heads, 512 selected rows per token in eight splits")

# an MXFP8 indexer with 40 heads: the MMA's N = 48 columns, heads 32-39 in the second
# column of the query's scale factors, columns 40-47 computed and ignored
SMALL_MX_H40 = replace(SMALL_DECODE_MX, name="small_mx_h40", idx_heads=40, seed=7020,
                       description="as small_decode_mx with 40 indexer heads")

# long rows whose selection runs in clusters of eight CTAs (more than 16384 positions);
# the tests give them degenerate queries (all scores equal, or 17 distinct values) so
# that a CTA's boundary bin overflows its share of the candidate pool
LONG_ROWS = Spec(
    name="long_rows", mode="decode", batch=3, seq_lens=(40000, 34816, 9000), pool_pages=1400,
    idx_heads=64, idx_dim=128, topk=2048, sfa_heads=16, seed=7014,
    description="rows of 40000, 34816 and 9000 keys, top-K 2048")

SMALL = [SMALL_DECODE_BF16, SMALL_DECODE_FP8, SMALL_DECODE_MX, SMALL_TIES, SMALL_PREFILL,
         SMALL_H8, EMPTY_AND_SHORT, SMALL_MID, SMALL_SIB, SMALL_MULTI, SMALL_FP8_D64, SMALL_MX_D64,
         SMALL_PREFILL_FP8, SMALL_PREFILL_MX, SMALL_MULTI25, SMALL_MULTI_FP8, SMALL_FP8_KV, SMALL_H5,
         SMALL_MX_H40]

ALL = {s.name: s for s in HEADLINE + EXTRA + SMALL + [LONG_ROWS]}


# ---------------------------------------------------------------------------------
# Encoders (storage formats).  Rounding of arbitrary reals to bf16 uses torch's
# float32 -> bfloat16 conversion (round to nearest even); integers and powers of two
# are exact in every format used here.
# ---------------------------------------------------------------------------------
def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def e4m3_bits_from_f32(x: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


_ENC_CACHE: dict = {}


def _int8_encoder(fmt: str) -> np.ndarray:
    """Table mapping an int8 (viewed as its byte) to its bf16 / e4m3 encoding."""
    if fmt not in _ENC_CACHE:
        vals = np.arange(256, dtype=np.uint8).view(np.int8).astype(np.float32)
        _ENC_CACHE[fmt] = bf16_bits_from_f32(vals) if fmt == "bf16" else e4m3_bits_from_f32(vals)
    return _ENC_CACHE[fmt]


def e8m0_bits_from_exp(e: np.ndarray) -> np.ndarray:
    """E8M0 byte for the power of two 2^e (bias 127)."""
    e = np.asarray(e, dtype=np.int32)
    assert e.min(initial=0) >= -127 and e.max(initial=0) <= 127
    return (e + 127).astype(np.uint8)


# ---------------------------------------------------------------------------------
# Workload container
# ---------------------------------------------------------------------------------
@dataclass
class Workload:
    spec: Spec
    seq_lens: np.ndarray          # int32 [B]
    block_table: np.ndarray       # int32 [B, max_pages]; -1 beyond a sequence's pages
    num_pages: int
    q_seq: np.ndarray             # int32 [T]   batch row of each query token
    q_pos: np.ndarray             # int32 [T]   position of each query token
    idx_q: np.ndarray             # u16 (bf16) or u8 (e4m3) [T, H_I, d]
    idx_q_scale: Optional[np.ndarray]  # None | f32 [T] | u8 E8M0 [T, H_I, d/32]
    head_w: np.ndarray            # f32 [T, H_I]
    idx_k: np.ndarray             # u16 or u8 [num_pages, 64, d]
    idx_k_scale: Optional[np.ndarray]  # None | f32 [num_pages, 64] | u8 [num_pages, 64, d/32]
    kv: np.ndarray                # u16 (bf16) [num_pages, 64, 576]; None for an FP8 cache
    sfa_q: np.ndarray             # u16 (bf16) [T, H, 576]
    extras: dict = field(default_factory=dict)
    kv_codes: Optional[np.ndarray] = None  # FP8 cache: u8 (e4m3) [num_pages, 64, 512]
    kv_scale: Optional[np.ndarray] = None  # FP8 cache: f32 [num_pages, 64, 4], one per 128 dims
    kv_rope: Optional[np.ndarray] = None   # FP8 cache: u16 (bf16) [num_pages, 64, 64]

    @property
    def n_tokens(self) -> int:
        return int(self.q_seq.shape[0])

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])


def _streams(seed: int, n: int = 16):
    return [np.random.default_rng(s) for s in np.random.SeedSequence(seed).spawn(n)]


def draw_seq_lens(spec: Spec) -> np.ndarray:
    if spec.seq_lens:
        assert len(spec.seq_lens) == spec.batch
        return np.asarray(spec.seq_lens, dtype=np.int32)
    lo, hi = spec.len_loguniform
    rng = _streams(spec.seed)[_S_LENS]
    u = rng.uniform(math.log(lo), math.log(hi), size=spec.batch)
    return np.floor(np.exp(u)).astype(np.int32)


def _pages_needed(lens: np.ndarray) -> np.ndarray:
    return (lens.astype(np.int64) + PAGE_SIZE - 1) // PAGE_SIZE


def make(spec: Spec, n_kv_chunk_pages: int = 1024, with_latent: bool = True) -> Workload:
    """Materialise a workload (host numpy arrays) from its spec, deterministically.

    ``with_latent=False`` skips the latent KV cache and SFA queries (left as None) for
    callers that only need the indexer inputs; the indexer arrays are identical.
    """
    rs = _streams(spec.seed)
    ri = _streams(spec.int_seed if spec.int_seed is not None else spec.seed)
    B, HI, d, H = spec.batch, spec.idx_heads, spec.idx_dim, spec.sfa_heads
    lens = draw_seq_lens(spec)
    npg = _pages_needed(lens)
    used = int(npg.sum())
    pool = spec.pool_pages if spec.pool_pages else used
    assert pool >= used, f"{spec.name}: pool of {pool} pages cannot hold {used}"
    max_pages = max(1, int(npg.max(initial=0)))

    # page layout: a random permutation of the pool, handed out in per-sequence slices
    perm = ri[_S_LAYOUT].permutation(pool).astype(np.int32)
    bt = np.full((B, max_pages), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        bt[b, :npg[b]] = perm[off:off + npg[b]]
        off += int(npg[b])

    # query tokens
    if spec.mode == "decode":
        T = B
        q_seq = np.arange(B, dtype=np.int32)
        q_pos = (lens - 1).astype(np.int32)  # -1 for an empty sequence
    elif spec.mode == "multi":
        m = spec.tokens_per_seq
        assert m >= 1 and np.all(lens >= m), f"{spec.name}: every sequence needs {m} positions"
        T = B * m
        q_seq = np.repeat(np.arange(B, dtype=np.int32), m)
        q_pos = (np.repeat(lens, m) - m + np.tile(np.arange(m), B)).astype(np.int32)
    else:
        assert B == 1 and spec.prefill_tokens <= int(lens[0])
        T = spec.prefill_tokens
        q_seq = np.zeros(T, dtype=np.int32)
        q_pos = (int(lens[0]) - T + np.arange(T)).astype(np.int32)

    # physical slots in logical order: row i of the "logical" arrays below is token
    # slot (b, j, s) for b in batch order, j in page order, s in 0..63.
    phys_pages = np.concatenate([bt[b, :npg[b]] for b in range(B)]) if used else np.zeros(0, np.int32)
    live_logical = np.zeros((used, PAGE_SIZE), dtype=bool)
    off = 0
    for b in range(B):
        n = int(lens[b])
        flat = live_logical[off:off + int(npg[b])].reshape(-1)
        flat[:n] = True
        off += int(npg[b])

    unused = np.setdiff1d(np.arange(pool), phys_pages)
    # (physical page, first dead slot) of every sequence's partially filled last page
    tails = [(int(bt[b, npg[b] - 1]), int(lens[b]) - (int(npg[b]) - 1) * PAGE_SIZE)
             for b in range(B) if npg[b] > 0 and lens[b] % PAGE_SIZE]

    def scatter(logical: np.ndarray, fill) -> np.ndarray:
        out = np.empty((pool,) + logical.shape[1:], dtype=logical.dtype)
        out[unused] = fill
        if used:
            out[phys_pages] = logical
        for page, first_dead in tails:
            out[page, first_dead:] = fill
        return out

    r = spec.idx_int_range
    # indexer query and K-index integers (int8 draws, encoded through a lookup table)
    qi = ri[_S_QI].integers(-r, r + 1, size=(T, HI, d), dtype=np.int8)
    ki = ri[_S_KI].integers(-r, r + 1, size=(used, PAGE_SIZE, d), dtype=np.int8)
    wl, wh = spec.head_w_exps
    head_w = np.ldexp(np.float32(1.0), rs[_S_W].integers(wl, wh + 1, size=(T, HI))).astype(np.float32)

    idx_q_scale = idx_k_scale = None
    if spec.idx_dtype == "bf16":
        assert spec.idx_scale == "none"
        idx_q = _int8_encoder("bf16")[qi.view(np.uint8)]
        idx_k = scatter(_int8_encoder("bf16")[ki.view(np.uint8)], BF16_NAN)
    elif spec.idx_dtype == "e4m3":
        assert r <= 8, "e4m3 represents the integers in [-8, 8] exactly, not all beyond"
        idx_q = _int8_encoder("e4m3")[qi.view(np.uint8)]
        idx_k = scatter(_int8_encoder("e4m3")[ki.view(np.uint8)], E4M3_NAN)
        if spec.idx_scale == "per_token":
            lo, hi = spec.scale_exps
            idx_q_scale = np.ldexp(np.float32(1.0), rs[_S_QSCALE].integers(lo, hi + 1, size=T)).astype(np.float32)
            ks = np.ldexp(np.float32(1.0), rs[_S_KSCALE].integers(lo, hi + 1, size=(used, PAGE_SIZE))).astype(np.float32)
            idx_k_scale = scatter(ks, np.float32(np.nan))
        elif spec.idx_scale == "mx":
            assert d % MX_GROUP == 0
            ng = d // MX_GROUP
            kb = rs[_S_KSCALE].integers(-4, 3, size=(used, PAGE_SIZE, 1))
            ko = -rs[_S_KSCALE_GRP].integers(0, 2, size=(used, PAGE_SIZE, ng))
            idx_k_scale = scatter(e8m0_bits_from_exp(np.clip(kb + ko, -4, 2)), E8M0_NAN)
            qb = rs[_S_QSCALE].integers(-1, 2, size=(T, HI, 1))
            qo = -rs[_S_QSCALE_GRP].integers(0, 2, size=(T, HI, ng))
            idx_q_scale = e8m0_bits_from_exp(np.clip(qb + qo, -1, 1))
        else:
            raise ValueError(spec.idx_scale)
    else:
        raise ValueError(spec.idx_dtype)
    del qi, ki

    # latent KV cache: N(0,1) -> bf16, drawn chunk by chunk in logical page order
    if not with_latent:
        return Workload(spec=spec, seq_lens=lens, block_table=bt, num_pages=pool, q_seq=q_seq,
                        q_pos=q_pos, idx_q=idx_q, idx_q_scale=idx_q_scale, head_w=head_w,
                        idx_k=idx_k, idx_k_scale=idx_k_scale, kv=None, sfa_q=None)
    sfa_q_bits = lambda: bf16_bits_from_f32(ri[_S_QS].standard_normal((T, H, KV_DIM), dtype=np.float32))
    if spec.kv_format == "fp8_tile128":
        # latent dims: integers in [-15, 15] as e4m3 (exact) times a power-of-two scale
        # 2^u, u in [-4, -2], per 128-dim tile; rope dims N(0,1) -> bf16; dead slots NaN
        g = ri[_S_KV]
        codes = np.full((pool, PAGE_SIZE, V_DIM), E4M3_NAN, dtype=np.uint8)
        scl = np.full((pool, PAGE_SIZE, V_DIM // 128), np.nan, dtype=np.float32)
        rope = np.full((pool, PAGE_SIZE, KV_DIM - V_DIM), BF16_NAN, dtype=np.uint16)
        enc = _int8_encoder("e4m3")
        for p0 in range(0, used, n_kv_chunk_pages):
            p1 = min(used, p0 + n_kv_chunk_pages)
            n = p1 - p0
            c = enc[g.integers(-15, 16, size=(n, PAGE_SIZE, V_DIM)).astype(np.int8).view(np.uint8)]
            sc = np.ldexp(np.float32(1.0), g.integers(-4, -1, size=(n, PAGE_SIZE, V_DIM // 128))).astype(np.float32)
            rp = bf16_bits_from_f32(g.standard_normal((n, PAGE_SIZE, KV_DIM - V_DIM), dtype=np.float32))
            dead = ~live_logical[p0:p1]
            c[dead], sc[dead], rp[dead] = E4M3_NAN, np.nan, BF16_NAN
            codes[phys_pages[p0:p1]], scl[phys_pages[p0:p1]], rope[phys_pages[p0:p1]] = c, sc, rp
        return Workload(spec=spec, seq_lens=lens, block_table=bt, num_pages=pool, q_seq=q_seq,
                        q_pos=q_pos, idx_q=idx_q, idx_q_scale=idx_q_scale, head_w=head_w,
                        idx_k=idx_k, idx_k_scale=idx_k_scale, kv=None, sfa_q=sfa_q_bits(),
                        kv_codes=codes, kv_scale=scl, kv_rope=rope)
    assert spec.kv_format == "bf16", spec.kv_format
    kv = np.empty((pool, PAGE_SIZE, KV_DIM), dtype=np.uint16)
    kv[...] = BF16_NAN
    g = ri[_S_KV]
    for p0 in range(0, used, n_kv_chunk_pages):
        p1 = min(used, p0 + n_kv_chunk_pages)
        chunk = bf16_bits_from_f32(g.standard_normal((p1 - p0, PAGE_SIZE, KV_DIM), dtype=np.float32))
        chunk[~live_logical[p0:p1]] = BF16_NAN
        kv[phys_pages[p0:p1]] = chunk
    sfa_q = sfa_q_bits()

    return Workload(spec=spec, seq_lens=lens, block_table=bt, num_pages=pool, q_seq=q_seq,
                    q_pos=q_pos, idx_q=idx_q, idx_q_scale=idx_q_scale, head_w=head_w,
                    idx_k=idx_k, idx_k_scale=idx_k_scale, kv=kv, sfa_q=sfa_q)


def with_block_table(wl: Workload, new_bt_pages: np.ndarray, new_pool: int) -> Workload:
    """Re-lay the same logical caches onto another page placement.

    ``new_bt_pages[b, j]`` is the physical page that logical page j of sequence b moves
    to; the contents of every logical page are copied there unchanged.  Used to check
    that results do not depend on where pages live.
    """
    B = wl.batch
    npg = _pages_needed(wl.seq_lens)

    def move(src, fill):
        dst = np.empty((new_pool,) + src.shape[1:], dtype=src.dtype)
        dst[...] = fill
        for b in range(B):
            for j in range(int(npg[b])):
                dst[new_bt_pages[b, j]] = src[wl.block_table[b, j]]
        return dst

    bt = np.full_like(wl.block_table, -1)
    for b in range(B):
        bt[b, :npg[b]] = new_bt_pages[b, :npg[b]]
    isbf = wl.idx_k.dtype == np.uint16
    ks = None
    if wl.idx_k_scale is not None:
        ks = move(wl.idx_k_scale, np.nan if wl.idx_k_scale.dtype == np.float32 else E8M0_NAN)
    fp8 = wl.kv_codes is not None
    return replace(wl, block_table=bt, num_pages=new_pool,
                   idx_k=move(wl.idx_k, BF16_NAN if isbf else E4M3_NAN), idx_k_scale=ks,
                   kv=None if fp8 else move(wl.kv, BF16_NAN),
                   kv_codes=move(wl.kv_codes, E4M3_NAN) if fp8 else None,
                   kv_scale=move(wl.kv_scale, np.nan) if fp8 else None,
                   kv_rope=move(wl.kv_rope, BF16_NAN) if fp8 else None)
