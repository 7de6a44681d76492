"""The C-ABI library loads, exports every symbol include/dsa.h declares, and rejects bad
arguments on the host before launching anything (no GPU needed)."""
import ctypes as C
import os
import re

import pytest
import torch

import sparse_attention_decode_dsa_gb300 as dsa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_exports_every_declared_symbol():
    hdr = open(os.path.join(ROOT, "include", "dsa.h")).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    names = set(re.findall(r"\b(dsa_[a-z_]+)\s*\(", hdr))
    assert len(names) >= 10
    raw = C.CDLL(dsa.LIB_PATH)
    missing = [n for n in sorted(names) if not hasattr(raw, n)]
    assert not missing, missing


def test_version_and_strings():
    assert dsa.lib.dsa_abi_version() == 3
    assert dsa.lib.dsa_status_string(0) == b"DSA_OK"
    assert dsa.lib.dsa_status_string(3) == b"DSA_ERR_WORKSPACE"


FAKE = 0x7F0000000000  # never dereferenced: every call below fails its host-side checks


def _structs(B=2, maxp=4, T=None, heads=64, dim=128, topk=128, dtype=dsa.DSA_BF16,
             scale=dsa.DSA_SCALE_NONE, lens=(100, 200)):
    lens_t = torch.tensor(lens, dtype=torch.int32)
    pages = dsa.PageTable(FAKE, FAKE, C.cast(C.c_void_p(lens_t.data_ptr()), C.POINTER(C.c_int32)),
                          B, maxp, 64, 16)
    toks = dsa.Tokens(T if T is not None else B, None, None, None, None)
    cache = dsa.IndexCache(FAKE, FAKE if scale else None, dtype, scale, dim)
    args = dsa.IndexerArgs(FAKE, FAKE if scale else None, dtype, scale, FAKE, heads, topk, 0)
    return pages, toks, cache, args, lens_t


def _call_indexer(pages, toks, cache, args, ws=256 * 1000, ws_bytes=1 << 30):
    return dsa.lib.dsa_indexer_topk(C.byref(args), C.byref(cache), C.byref(pages), C.byref(toks),
                                    C.c_void_p(FAKE), None, C.c_void_p(ws) if ws else None, ws_bytes,
                                    None, None)


def test_workspace_size_formula():
    pages, toks, cache, args, keep = _structs(lens=(100, 200))
    n = dsa.lib.dsa_indexer_workspace_size(C.byref(args), C.byref(cache), C.byref(pages), C.byref(toks))
    # error word (256 B) + T rows x ceil(max visible / 64) * 64 f32 scores (256-aligned)
    # + T rows x 4096 u32 key-histogram bins + the collapsed query (bf16 [T, 16, dim] and
    # f32 [T, 16] weights, each 256-aligned)
    assert n == (256 + ((2 * 256 * 4 + 255) // 256) * 256 + 2 * 4096 * 4
                 + ((2 * 16 * 128 * 2 + 255) // 256) * 256 + ((2 * 16 * 4 + 255) // 256) * 256)


@pytest.mark.parametrize("mutate,status", [
    (lambda p, t, c, a: setattr(p, "page_size", 32), dsa.DSA_ERR_UNSUPPORTED),
    (lambda p, t, c, a: setattr(a, "top_k", 0), dsa.DSA_ERR_UNSUPPORTED),
    (lambda p, t, c, a: setattr(a, "top_k", 4096), dsa.DSA_ERR_UNSUPPORTED),
    (lambda p, t, c, a: setattr(a, "n_heads", 65), dsa.DSA_ERR_UNSUPPORTED),
    (lambda p, t, c, a: setattr(c, "dim", 96), dsa.DSA_ERR_UNSUPPORTED),
    (lambda p, t, c, a: setattr(a, "q_dtype", dsa.DSA_E4M3), dsa.DSA_ERR_UNSUPPORTED),
    (lambda p, t, c, a: setattr(c, "scale_kind", dsa.DSA_SCALE_MX_E8M0_G32), dsa.DSA_ERR_UNSUPPORTED),
    (lambda p, t, c, a: setattr(t, "n_tokens", 3), dsa.DSA_ERR_INVALID_ARG),
    (lambda p, t, c, a: setattr(t, "token_seq", C.c_void_p(FAKE)), dsa.DSA_ERR_INVALID_ARG),
    (lambda p, t, c, a: setattr(p, "max_pages_per_seq", 1), dsa.DSA_ERR_INVALID_ARG),
    (lambda p, t, c, a: setattr(a, "head_w", None), dsa.DSA_ERR_INVALID_ARG),
    (lambda p, t, c, a: setattr(a, "act", 7), dsa.DSA_ERR_INVALID_ARG),
    (lambda p, t, c, a: setattr(c, "data", C.c_void_p(FAKE + 8)), dsa.DSA_ERR_INVALID_ARG),
])
def test_indexer_rejects_bad_arguments(mutate, status):
    pages, toks, cache, args, keep = _structs()
    mutate(pages, toks, cache, args)
    assert _call_indexer(pages, toks, cache, args) == status
    assert len(dsa.lib.dsa_last_error_message()) > 0


def test_e4m3_needs_scales():
    pages, toks, cache, args, keep = _structs(dtype=dsa.DSA_E4M3, scale=dsa.DSA_SCALE_PER_TOKEN_F32)
    cache.scale = None
    assert _call_indexer(pages, toks, cache, args) == dsa.DSA_ERR_INVALID_ARG


@pytest.mark.parametrize("ws,ws_bytes", [(0, 1 << 30), (FAKE + 8, 1 << 30), (FAKE, 100)])
def test_workspace_checks(ws, ws_bytes):
    pages, toks, cache, args, keep = _structs()
    assert _call_indexer(pages, toks, cache, args, ws=ws, ws_bytes=ws_bytes) == dsa.DSA_ERR_WORKSPACE


@pytest.mark.parametrize("x, rows, dim, codes, status", [
    (FAKE, 4, 48, FAKE, dsa.DSA_ERR_INVALID_ARG),       # dim not a multiple of 32
    (FAKE, 4, 0, FAKE, dsa.DSA_ERR_INVALID_ARG),
    (FAKE, -1, 128, FAKE, dsa.DSA_ERR_INVALID_ARG),
    (0, 4, 128, FAKE, dsa.DSA_ERR_INVALID_ARG),          # missing input
    (FAKE + 8, 4, 128, FAKE, dsa.DSA_ERR_INVALID_ARG),   # x not 16-byte aligned
    (FAKE, 4, 128, FAKE + 4, dsa.DSA_ERR_INVALID_ARG),   # codes not 8-byte aligned
    (FAKE, 0, 128, FAKE, dsa.DSA_OK),                     # nothing to do: nothing enqueued
])
def test_quantize_mxfp8_host_checks(x, rows, dim, codes, status):
    st = dsa.lib.dsa_quantize_mxfp8(C.c_void_p(x) if x else None, rows, dim,
                                    C.c_void_p(codes), C.c_void_p(FAKE), None)
    assert st == status


@pytest.mark.parametrize("dim, ws, ws_bytes, status", [
    (96, FAKE, 256, dsa.DSA_ERR_UNSUPPORTED),
    (128, 0, 256, dsa.DSA_ERR_WORKSPACE),
    (128, FAKE, 100, dsa.DSA_ERR_WORKSPACE),
])
def test_index_cache_append_host_checks(dim, ws, ws_bytes, status):
    pages, toks, cache, args, keep = _structs()
    st = dsa.lib.dsa_index_cache_append_mxfp8(C.c_void_p(FAKE), dim, C.byref(pages), C.byref(toks),
                                              C.c_void_p(FAKE), C.c_void_p(FAKE),
                                              C.c_void_p(ws) if ws else None, ws_bytes, None)
    assert st == status


def test_sfa_rejects_bad_shapes():
    pages, toks, cache, args, keep = _structs()
    sargs = dsa.SfaArgs(FAKE, 129, 0.04)
    lat = dsa.LatentCache(FAKE, 576, 512)
    st = dsa.lib.dsa_sparse_attn(C.byref(sargs), C.byref(lat), C.byref(pages), C.byref(toks), C.c_void_p(FAKE),
                                 128, C.c_void_p(FAKE), C.c_void_p(FAKE), 1 << 30, None, None)
    assert st == dsa.DSA_ERR_UNSUPPORTED
    sargs.n_heads = 128
    lat.dim = 512
    st = dsa.lib.dsa_sparse_attn(C.byref(sargs), C.byref(lat), C.byref(pages), C.byref(toks), C.c_void_p(FAKE),
                                 128, C.c_void_p(FAKE), C.c_void_p(FAKE), 1 << 30, None, None)
    assert st == dsa.DSA_ERR_UNSUPPORTED
    lat.dim = 576
    for q, data, out in [(FAKE + 4, FAKE, FAKE), (FAKE, FAKE + 8, FAKE), (FAKE, FAKE, FAKE + 2)]:
        sargs.q = q
        lat.data = data
        st = dsa.lib.dsa_sparse_attn(C.byref(sargs), C.byref(lat), C.byref(pages), C.byref(toks), C.c_void_p(FAKE),
                                     128, C.c_void_p(out), C.c_void_p(FAKE), 1 << 30, None, None)
        assert st == dsa.DSA_ERR_INVALID_ARG  # 16-byte alignment


def test_product_path_has_no_cpu_fallback():
    """The package imports nothing from the oracle and offers no CPU implementation."""
    pkg = os.path.join(ROOT, "sparse_attention_decode_dsa_gb300")
    for f in os.listdir(pkg):
        if f.endswith(".py"):
            src = open(os.path.join(pkg, f)).read()
            assert "oracle" not in src and "dsa_workloads" not in src, f


def test_workspace_holds_dequantised_keys_for_quantised_prefill():
    """An e4m3 indexer over many rows of one sequence (a prefill) dequantises that
    sequence's pages to bf16 once: its workspace adds bf16 [pages, 64, dim] keys, f32
    [pages * 64] scales and an int32 [batch, max_pages] page table to the per-row parts."""
    T, L, dim = 64, 4000, 128
    lens_t = torch.tensor([L], dtype=torch.int32)
    seq_t = torch.zeros(T, dtype=torch.int32)
    pos_t = torch.arange(L - T, L, dtype=torch.int32)
    hp = lambda t: C.cast(C.c_void_p(t.data_ptr()), C.POINTER(C.c_int32))
    pages = dsa.PageTable(FAKE, FAKE, hp(lens_t), 1, 63, 64, 100)
    toks = dsa.Tokens(T, FAKE, FAKE, hp(seq_t), hp(pos_t))
    cache = dsa.IndexCache(FAKE, FAKE, dsa.DSA_E4M3, dsa.DSA_SCALE_PER_TOKEN_F32, dim)
    args = dsa.IndexerArgs(FAKE, FAKE, dsa.DSA_E4M3, dsa.DSA_SCALE_PER_TOKEN_F32, FAKE, 64, 2048, 0)
    a256 = lambda n: (n + 255) // 256 * 256
    npv = (L + 63) // 64
    base = (256 + a256(T * npv * 64 * 4) + T * 4096 * 4 + a256(T * 16 * dim * 2) + a256(T * 16 * 4))
    n = dsa.lib.dsa_indexer_workspace_size(C.byref(args), C.byref(cache), C.byref(pages), C.byref(toks))
    assert n == base + a256(npv * 64 * dim * 2) + a256(npv * 64 * 4) + a256(63 * 4)
    # one row per sequence (decode): no dequantised copy
    args.act = 1  # ReLU: per-head scoring, never row-blocked
    n_relu = dsa.lib.dsa_indexer_workspace_size(C.byref(args), C.byref(cache), C.byref(pages), C.byref(toks))
    assert n_relu == base


@pytest.mark.parametrize("T,heads", [(32, 128), (8, 128), (8, 5), (2, 16), (200, 128)])
def test_attention_workspace_holds_split_partials_only_beyond_two_splits(T, heads):
    """The attention splits each token's K selected rows over s = min(SMs / (2 T), ceil(K/64),
    16) CTA pairs (at least 1), in whole 64-row tiles; one or two splits need no workspace
    beyond the 256-byte header (two merge inside their cluster), more keep f32 partials
    [T, S, 2, 256, HP] and log2-sum-exps [T, S, 2, HP] (HP = heads rounded up to 4, each
    part 256-byte aligned).  S is recomputed from the split length, so no split is empty."""
    lens = (4000,) * T
    pages, toks, cache, args, keep = _structs(B=T, maxp=64, lens=lens)
    sargs = dsa.SfaArgs(FAKE, heads, 0.04)
    K = 2048
    n = dsa.lib.dsa_sparse_attn_workspace_size(C.byref(sargs), C.byref(pages), C.byref(toks), K)
    sms = torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 148
    tiles = (K + 63) // 64
    s = max(1, min(sms // (2 * T), tiles, 16))
    split_len = -(-tiles // s) * 64
    S = -(-(tiles * 64) // split_len)
    a256 = lambda x: (x + 255) // 256 * 256
    hp = (heads + 3) // 4 * 4
    want = 256 if S <= 2 else 256 + a256(T * S * hp * 512 * 4) + a256(T * S * 2 * hp * 4)
    assert n == want
