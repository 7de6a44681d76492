"""Pins of the float64 oracle against things other than itself (CPU only).

Each test ties the oracle to a fixed point the pages or mathematics give: hand-worked
examples, library routines it must reduce to in special cases, a brute-force rank
definition of Top-K, exact integer arithmetic, and invariants (causality, page placement,
permutations).  ``test_oracle_mutants`` then plants plausible mistakes in the oracle and
checks that some pin catches each one.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import dsa_workloads as W
from oracle import dsa_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------------
# storage decoders vs torch's own conversions and textbook values
# ---------------------------------------------------------------------------------
def test_decode_bf16_all_codes():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = O.decode_bf16(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert O.decode_bf16(np.array([0x3F80], np.uint16))[0] == 1.0
    assert O.decode_bf16(np.array([0xC100], np.uint16))[0] == -8.0


def test_decode_e4m3_all_codes():
    bits = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(bits).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.decode_e4m3(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # textbook E4M3 values: 1.0, max normal 448, min normal 2^-6, min subnormal 2^-9
    v = O.decode_e4m3(np.array([0x38, 0x7E, 0x08, 0x01, 0xB8, 0x50], np.uint8))
    assert list(v) == [1.0, 448.0, 2.0 ** -6, 2.0 ** -9, -1.0, 8.0]


def test_decode_e8m0():
    v = O.decode_e8m0(np.array([127, 0, 254, 125, 129, 255], np.uint8))
    assert list(v[:5]) == [1.0, 2.0 ** -127, 2.0 ** 127, 0.25, 4.0]
    assert np.isnan(v[5])


# ---------------------------------------------------------------------------------
# hand-worked examples
# ---------------------------------------------------------------------------------
def test_golden_indexer_example():
    g = _load("indexer_worked_example.json")
    q = np.array(g["q"], float)
    w = np.array(g["w"], float)
    k = np.array(g["k"], float)
    s = O.index_scores(q, w, k)
    assert s.tolist() == g["scores"]
    for kk, want in g["topk"].items():
        assert O.topk_select(s, int(kk)).tolist() == want


def test_golden_sfa_example():
    g = _load("sfa_worked_example.json")
    out = O.sparse_attention(np.array(g["q"]), np.array(g["rows"]), g["scale"], g["v_dim"])
    assert np.allclose(out, np.array(g["out"]), rtol=0, atol=1e-15)


# ---------------------------------------------------------------------------------
# Top-K vs a brute-force rank definition (independent of any sort)
# ---------------------------------------------------------------------------------
def _rank_select(s, k):
    n = len(s)
    chosen = [t for t in range(n)
              if sum(1 for u in range(n) if s[u] > s[t] or (s[u] == s[t] and u < t)) < k]
    return chosen + [-1] * (k - len(chosen))


def test_topk_brute_force_rank():
    rng = np.random.default_rng(11)
    for trial in range(300):
        n = int(rng.integers(0, 120))
        k = int(rng.integers(1, 40))
        vals = rng.integers(-3, 4, size=n).astype(float) * (2.0 ** rng.integers(-2, 3))
        if trial % 3 == 0:
            vals = rng.standard_normal(n)
        assert O.topk_select(vals, k).tolist() == _rank_select(list(vals), k)


def test_topk_signed_zero_is_one_score():
    s = np.array([-0.0, 0.0, -1.0, -0.0])
    assert O.topk_select(s, 2).tolist() == [0, 1]
    assert O.topk_select(s, 3).tolist() == [0, 1, 3]


# ---------------------------------------------------------------------------------
# scores: exact integer arithmetic by another route (the head-collapsed form)
# ---------------------------------------------------------------------------------
def _int_scores_collapsed(q, w, k, shift):
    """sum_h w_h (q_h . k_t) == (sum_h w_h q_h) . k_t, in exact int64 (values scaled by 2^shift)."""
    qi = np.rint(q * 2.0 ** shift).astype(np.int64)
    wi = np.rint(w * 2.0 ** shift).astype(np.int64)
    ki = np.rint(k * 2.0 ** shift).astype(np.int64)
    assert np.array_equal(qi, q * 2.0 ** shift) and np.array_equal(wi, w * 2.0 ** shift)
    assert np.array_equal(ki, k * 2.0 ** shift)
    qc = (wi[:, None] * qi).sum(axis=0)           # collapsed query, int64
    return (ki @ qc).astype(np.float64) / 2.0 ** (3 * shift)


@pytest.mark.parametrize("spec", [W.SMALL_DECODE_BF16, W.SMALL_DECODE_FP8, W.SMALL_DECODE_MX,
                                  W.SMALL_TIES, W.TINY_DECODE])
def test_scores_equal_collapsed_integer_form(spec):
    wl = W.make(spec)
    for tok in range(wl.n_tokens):
        n = O.visible_count(wl, tok)
        b = int(wl.q_seq[tok])
        q = O.dequant_index_query(wl, tok)
        k = O.dequant_index_keys(wl, b, np.arange(n))
        w = wl.head_w[tok].astype(float)
        assert np.array_equal(O.index_scores(q, w, k), _int_scores_collapsed(q, w, k, 8))


def test_fp8_scores_are_scaled_integer_scores():
    wl = W.make(W.SMALL_DECODE_FP8)
    raw = W.Workload(**{**wl.__dict__, "idx_q_scale": None, "idx_k_scale": None})
    for tok in range(wl.n_tokens):
        n = O.visible_count(wl, tok)
        b = int(wl.q_seq[tok])
        pos = np.arange(n)
        w = wl.head_w[tok].astype(float)
        s = O.index_scores(O.dequant_index_query(wl, tok), w, O.dequant_index_keys(wl, b, pos))
        r = O.index_scores(O.dequant_index_query(raw, tok), w, O.dequant_index_keys(raw, b, pos))
        sk = O.logical_rows(wl.idx_k_scale, wl.block_table[b], pos).astype(float)
        assert np.array_equal(s, float(wl.idx_q_scale[tok]) * sk * r)


def test_mx_scores_group_by_group():
    """MX scores equal an explicit loop over the 32-element groups with their two scales."""
    wl = W.make(W.SMALL_DECODE_MX)
    tok = 5
    b = int(wl.q_seq[tok])
    n = O.visible_count(wl, tok)
    s = O.indexer_topk(wl, tok)  # noqa: F841  (exercise the full path once)
    pos = np.arange(n)
    q_raw = O.decode_e4m3(wl.idx_q[tok])
    k_raw = O.decode_e4m3(O.logical_rows(wl.idx_k, wl.block_table[b], pos))
    sq = O.decode_e8m0(wl.idx_q_scale[tok])                                  # [H, G]
    sk = O.decode_e8m0(O.logical_rows(wl.idx_k_scale, wl.block_table[b], pos))  # [n, G]
    w = wl.head_w[tok].astype(float)
    want = np.zeros(n)
    for g in range(sq.shape[1]):
        sl = slice(32 * g, 32 * g + 32)
        dot = k_raw[:, sl] @ q_raw[:, sl].T                                  # [n, H]
        want += (dot * (w * sq[:, g])[None, :]).sum(axis=1) * sk[:, g]
    got = O.index_scores(O.dequant_index_query(wl, tok), w, O.dequant_index_keys(wl, b, pos))
    assert np.array_equal(got, want)


# ---------------------------------------------------------------------------------
# invariants: causality, counts, duplicates, page placement
# ---------------------------------------------------------------------------------
@pytest.mark.parametrize("spec", [W.SMALL_DECODE_BF16, W.SMALL_PREFILL, W.EMPTY_AND_SHORT,
                                  W.SMALL_TIES, W.SMALL_MULTI])
def test_selection_invariants(spec):
    wl = W.make(spec)
    toks = range(wl.n_tokens) if wl.n_tokens <= 64 else list(range(0, 40)) + list(range(wl.n_tokens - 24, wl.n_tokens))
    for tok in toks:
        idx, sc = O.indexer_topk(wl, tok)
        n = O.visible_count(wl, tok)
        sel = idx[idx >= 0]
        assert sel.shape[0] == min(spec.topk, n)
        assert np.all(idx[sel.shape[0]:] == -1)
        assert np.all(np.diff(sel) > 0)                  # ascending, no duplicates
        assert sel.size == 0 or sel.max() <= wl.q_pos[tok]
        assert not np.isnan(sc[:sel.shape[0]]).any()     # never touched a NaN slot


@pytest.mark.parametrize("spec", [W.SMALL_DECODE_MX, W.SMALL_PREFILL, W.SMALL_H8, W.SMALL_FP8_KV])
def test_paged_equals_contiguous(spec):
    wl = W.make(spec)
    npg = (wl.seq_lens + 63) // 64
    ident = np.zeros_like(wl.block_table)
    off = 0
    for b in range(wl.batch):
        ident[b, :npg[b]] = np.arange(off, off + npg[b])
        off += int(npg[b])
    rng = np.random.default_rng(5)
    other = np.zeros_like(wl.block_table)
    perm = rng.permutation(off + 7)
    off = 0
    for b in range(wl.batch):
        other[b, :npg[b]] = perm[off:off + npg[b]]
        off += int(npg[b])
    a = W.with_block_table(wl, ident, int(npg.sum()))
    c = W.with_block_table(wl, other, int(npg.sum()) + 7)
    toks = range(wl.n_tokens) if wl.n_tokens <= 16 else [0, 1, 63, 64, 300, wl.n_tokens - 1]
    for tok in toks:
        i0, s0, o0 = O.step(wl, tok)
        i1, s1, o1 = O.step(a, tok)
        i2, s2, o2 = O.step(c, tok)
        assert np.array_equal(i0, i1) and np.array_equal(i0, i2)
        assert np.array_equal(s0, s1, equal_nan=True) and np.array_equal(s0, s2, equal_nan=True)
        assert np.array_equal(o0, o1) and np.array_equal(o0, o2)


# ---------------------------------------------------------------------------------
# sparse attention: special cases that reduce to textbook routines
# ---------------------------------------------------------------------------------
def test_sfa_with_k_at_least_l_is_dense_causal_attention():
    """K >= L selects every visible key, so SFA is dense attention (torch SDPA, f64)."""
    spec = W.Spec(name="dense", mode="prefill", batch=1, seq_lens=(150,), idx_heads=8,
                  idx_dim=64, topk=256, sfa_heads=8, seed=3, prefill_tokens=150)
    wl = W.make(spec)
    kv = O.decode_bf16(O.logical_rows(wl.kv, wl.block_table[0], np.arange(150)))
    q = O.decode_bf16(wl.sfa_q)                                   # [T, H, 576]
    qt = torch.from_numpy(q).permute(1, 0, 2)                     # [H, T, 576]
    kt = torch.from_numpy(kv)[None].expand(8, -1, -1)
    vt = torch.from_numpy(kv[:, :512])[None].expand(8, -1, -1)
    ref = torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, is_causal=True, scale=spec.softmax_scale).permute(1, 0, 2).numpy()
    for tok in [0, 1, 17, 64, 149]:
        idx, _, out = O.step(wl, tok)
        assert idx[:tok + 1].tolist() == list(range(tok + 1))
        assert np.allclose(out, ref[tok], rtol=0, atol=1e-12)


def test_multi_token_draft_sees_its_own_prefix():
    """Multi-token decode: the m query tokens of a sequence sit at its last m positions
    and token j sees positions 0 .. L - m + j only; where that prefix is shorter than K
    it selects all of it, so consecutive draft tokens select nested prefixes."""
    wl = W.make(W.SMALL_MULTI)
    m = W.SMALL_MULTI.tokens_per_seq
    L0 = int(wl.seq_lens[0])
    assert L0 <= W.SMALL_MULTI.topk
    for j in range(m):
        idx, _ = O.indexer_topk(wl, j)  # tokens 0 .. m - 1 belong to sequence 0
        assert int(wl.q_pos[j]) == L0 - m + j
        n = L0 - m + j + 1
        assert np.array_equal(idx[:n], np.arange(n)) and np.all(idx[n:] == -1)


def test_prefill_row0_attends_to_key0_only():
    wl = W.make(W.SMALL_PREFILL)
    idx, _, out = O.step(wl, 0)
    assert idx[0] == 0 and np.all(idx[1:] == -1)
    row0 = O.decode_bf16(O.logical_rows(wl.kv, wl.block_table[0], np.array([0])))[0, :512]
    assert np.array_equal(out, np.broadcast_to(row0, out.shape))


def test_sfa_identical_rows_return_the_row():
    rng = np.random.default_rng(2)
    row = rng.standard_normal(576)
    out = O.sparse_attention(rng.standard_normal((4, 576)), np.tile(row, (37, 1)), 0.1)
    assert np.allclose(out, np.broadcast_to(row[:512], out.shape), rtol=0, atol=1e-13)


def test_sfa_order_of_indices_does_not_matter():
    wl = W.make(W.SMALL_DECODE_BF16)
    tok = 5
    idx, _ = O.indexer_topk(wl, tok)
    o1 = O.sfa(wl, tok, idx)
    o2 = O.sfa(wl, tok, np.random.default_rng(0).permutation(idx))
    assert np.allclose(o1, o2, rtol=0, atol=1e-13)


def test_split_softmax_merge_equals_single_pass():
    """Log-sum-exp merge of per-chunk partial softmax states equals one pass (the
    identity the split-context combine relies on)."""
    rng = np.random.default_rng(4)
    q = rng.standard_normal((6, 576))
    rows = rng.standard_normal((300, 576))
    scale = 1 / math.sqrt(576)
    want = O.sparse_attention(q, rows, scale)
    cuts = np.sort(rng.choice(np.arange(1, 300), size=4, replace=False))
    parts = []
    for lo, hi in zip(np.r_[0, cuts], np.r_[cuts, 300]):
        z = scale * q @ rows[lo:hi].T
        m = z.max(axis=1)
        p = np.exp(z - m[:, None])
        parts.append((m, p.sum(axis=1), p @ rows[lo:hi, :512]))
    M = np.max([p[0] for p in parts], axis=0)
    L = sum(l * np.exp(m - M) for m, l, _ in parts)
    out = sum(o * np.exp(m - M)[:, None] for m, _, o in parts) / L[:, None]
    assert np.allclose(out, want, rtol=0, atol=1e-13)


def test_sfa_empty_selection_is_zero():
    wl = W.make(W.EMPTY_AND_SHORT)
    idx, sc, out = O.step(wl, 0)
    assert np.all(idx == -1) and np.all(out == 0)


# ---------------------------------------------------------------------------------
# exactness certificate: every generated config reaches its scores exactly in fp32
# ---------------------------------------------------------------------------------
@pytest.mark.parametrize("spec", W.SMALL + [W.TINY_DECODE])
def test_certificate_small(spec):
    wl = W.make(spec)
    for tok in range(0, wl.n_tokens, max(1, wl.n_tokens // 16)):
        assert O.exactness_certificate(wl, tok) < 1.0


@pytest.mark.parametrize("spec", W.SMALL + [W.TINY_DECODE])
def test_collapsed_query_certificate_small(spec):
    """The head-collapsed query q~ = sum_h w_h q_h (the identity-activation form the
    indexer kernel evaluates) is exact in fp32 on every sampled token."""
    wl = W.make(spec)
    for tok in range(0, wl.n_tokens, max(1, wl.n_tokens // 16)):
        assert O.collapsed_query_certificate(wl, tok) < 1.0


def test_collapsed_query_certificate_rejects_wide_weights():
    """Head weights spread over 2^-30 .. 1 with odd integer queries: q~ needs more than
    24 significant bits, and the certificate says so."""
    wl = W.make(W.SMALL_DECODE_BF16)
    wl.head_w[0] = np.exp2(-np.arange(wl.head_w.shape[1], dtype=np.float64) * 30.0 / wl.head_w.shape[1]).round(30)
    wl.head_w[0] = np.exp2(np.floor(np.log2(wl.head_w[0])))
    q = O.dequant_index_query(wl, 0)
    if not np.any(np.abs(q) % 2 == 1):
        pytest.skip("needs an odd query element")
    assert O.collapsed_query_certificate(wl, 0) >= 1.0


def test_certificate_rejects_naive_mx_reading():
    """Independent per-token key scales in [2^-4, 2^2], query scales likewise, elements in
    [-8, 8]: the fp32 score is no longer reachable exactly, and the certificate says so."""
    spec = W.replace(W.SMALL_DECODE_MX, name="naive_mx", idx_int_range=8, head_w_exps=(-6, 0))
    wl = W.make(spec)
    rng = np.random.default_rng(9)
    wl.idx_k_scale[...] = W.e8m0_bits_from_exp(rng.integers(-4, 3, size=wl.idx_k_scale.shape))
    wl.idx_q_scale[...] = W.e8m0_bits_from_exp(rng.integers(-4, 3, size=wl.idx_q_scale.shape))
    assert max(O.exactness_certificate(wl, t) for t in range(2, wl.n_tokens)) >= 1.0


def test_certificate_fp32_reproduces_scores():
    """Where the certificate holds, a float32 evaluation in a different order (per-head
    fp32 dot products, weights applied last) gives the float64 scores bit for bit."""
    wl = W.make(W.SMALL_DECODE_MX)
    tok = 5
    b = int(wl.q_seq[tok])
    n = O.visible_count(wl, tok)
    q = O.dequant_index_query(wl, tok).astype(np.float32)
    k = O.dequant_index_keys(wl, b, np.arange(n)).astype(np.float32)
    w = wl.head_w[tok].astype(np.float32)
    s32 = np.zeros(n, np.float32)
    for h in range(q.shape[0]):
        acc = np.zeros(n, np.float32)
        for d in range(q.shape[1] - 1, -1, -1):
            acc = acc + k[:, d] * q[h, d]
        s32 = s32 + acc * w[h]
    assert O.exactness_certificate(wl, tok) < 1.0
    assert np.array_equal(s32.astype(np.float64), O.indexer_topk.__globals__["index_scores"](
        O.dequant_index_query(wl, tok), wl.head_w[tok].astype(float),
        O.dequant_index_keys(wl, b, np.arange(n))))


@pytest.mark.parametrize("spec", [W.BF16_DECODE, W.FP8_DECODE, W.RAGGED_MXFP8_DECODE,
                                  W.CAUSAL_PREFILL])
def test_certificate_headline(spec):
    """Sampled query tokens of the full-size workloads: the fp32 scores are exact."""
    wl = W.make(spec, with_latent=False)
    toks = sorted(set(np.linspace(0, wl.n_tokens - 1, 6).astype(int).tolist()))
    for tok in toks:
        assert O.exactness_certificate(wl, tok) < 1.0
        assert O.collapsed_query_certificate(wl, tok) < 1.0


def test_fp8_decode_shares_integers_with_bf16_decode():
    """The FP8 workload reuses the BF16 workload's integers (only the format and the
    scales differ), so its scores are sq*sk times the BF16 scores under equal weights."""
    a = W.make(W.BF16_DECODE, with_latent=False)
    c = W.make(W.FP8_DECODE, with_latent=False)
    assert np.array_equal(O.decode_bf16(a.idx_q), O.decode_e4m3(c.idx_q))
    assert np.array_equal(O.decode_bf16(a.idx_k[:64]), O.decode_e4m3(c.idx_k[:64]))


# ---------------------------------------------------------------------------------
# FP8 latent cache (e4m3 latent dims, an f32 scale per 128-dim tile, bf16 rope dims)
# ---------------------------------------------------------------------------------
def test_fp8_latent_decode_closed_form():
    """Element j of the latent uses the scale of tile j // 128; rope dims are bf16."""
    codes = np.zeros((1, 512), dtype=np.uint8)
    codes[0, [0, 127, 128, 255, 256, 511]] = [0x38, 0x40, 0x38, 0xB8, 0x30, 0x44]  # 1, 2, 1, -1, 0.5, 3
    scales = np.array([[0.25, 0.125, 8.0, 4.0]], dtype=np.float32)
    rope = np.zeros((1, 64), dtype=np.uint16)
    rope[0, 0], rope[0, 63] = 0x3F80, 0xC000  # 1.0, -2.0
    row = O.decode_latent_fp8(codes, scales, rope)[0]
    assert row.shape == (576,)
    assert row[0] == 0.25 and row[127] == 0.5 and row[128] == 0.125 and row[255] == -0.125
    assert row[256] == 4.0 and row[511] == 12.0
    assert row[512] == 1.0 and row[575] == -2.0
    assert np.count_nonzero(row) == 8


def test_fp8_latent_sfa_equals_bf16_sfa_of_the_same_values():
    """The FP8 cache holds integers in [-15, 15] times powers of two, which bf16 also
    holds exactly: written as a bf16 cache, every token's attention is the same."""
    wl = W.make(W.SMALL_FP8_KV)
    vals = O.decode_latent_fp8(wl.kv_codes, wl.kv_scale, wl.kv_rope)  # NaN in dead slots
    bits = W.bf16_bits_from_f32(vals.astype(np.float32))
    assert np.array_equal(O.decode_bf16(bits), vals, equal_nan=True)  # exact re-encoding
    wl_bf = W.replace(wl, kv=bits, kv_codes=None, kv_scale=None, kv_rope=None)
    for tok in range(wl.n_tokens):
        idx, _ = O.indexer_topk(wl, tok)
        assert np.array_equal(O.sfa(wl, tok, idx), O.sfa(wl_bf, tok, idx))


def test_fp8_latent_workload_values():
    """The generator's FP8 latent: finite integer e4m3 codes in [-15, 15] on live slots,
    power-of-two tile scales in [2^-4, 2^-2], NaN on dead slots (a stray read shows)."""
    wl = W.make(W.SMALL_FP8_KV)
    live = ~np.isnan(wl.kv_scale[..., 0])
    v = O.decode_e4m3(wl.kv_codes[live])
    assert np.all(np.isfinite(v)) and np.all(v == np.round(v)) and np.abs(v).max() <= 15
    sc = wl.kv_scale[live]
    assert np.all(np.isin(sc, [2.0 ** -4, 2.0 ** -3, 2.0 ** -2]))
    assert np.all(np.isnan(O.decode_e4m3(wl.kv_codes[~live])))

