"""Parity of the index-prolog kernels (MXFP8 quantisation with groups of 32, append of new
keys to the paged K-index cache) with the oracle, through the C ABI: E4M3 codes and E8M0
scale bytes bit for bit (the quotient x / 2^e is exact on both sides, so the rounding
decisions are taken on the same value)."""
import numpy as np
import pytest
import torch

from oracle import mx_quant as M
from oracle.dsa_oracle import decode_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    import sparse_attention_decode_dsa_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def _to_bf16_bits(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _rows(rng, n, dim):
    """bf16 rows whose 32-element groups span magnitudes 2^-30 .. 2^30, plus rows of
    zeros, signed zeros, bf16 subnormals, rounding ties, saturation and huge values."""
    x = rng.standard_normal((n, dim)).astype(np.float32)
    x *= np.repeat(np.ldexp(np.float32(1.0), rng.integers(-30, 30, (n, dim // 32))), 32, axis=1)
    x[0] = 0.0
    x[1] = 0.0
    x[1, 1::2] = -0.0
    x[1, 7] = 2.0 ** -12
    x[2] = np.ldexp(np.float32(1.0), rng.integers(-133, -127, dim)) * rng.choice([-1, 1], dim)
    x[3, :32] = [256, 1.0625, 1.1875, 2 ** -10, 3 * 2 ** -10, -1.0625, -1.1875, 2 ** -12] + [0.5] * 24
    x[4, :32] = [510, 450, -450, 448, 449] + [1.0] * 27
    x[5] = np.ldexp(np.float32(1.0), rng.integers(100, 127, dim))
    return _to_bf16_bits(x)


@pytest.mark.parametrize("shape", [(7, 128), (3, 64, 128), (5, 4, 64), (1, 32)])
def test_quantize_mxfp8_matches_oracle(dsa, shape):
    rng = np.random.default_rng(17)
    dim = shape[-1]
    n = int(np.prod(shape[:-1]))
    bits = _rows(rng, max(n, 6), dim)[:n] if n >= 6 else _rows(rng, 6, dim)[-n:]
    x = torch.from_numpy(bits.view(np.int16).reshape(shape)).cuda()
    codes, scales = dsa.quantize_mxfp8(x)
    torch.cuda.synchronize()
    want_c, want_s = M.quantize_mxfp8(decode_bf16(bits).reshape(shape))
    got_c, got_s = codes.cpu().numpy(), scales.cpu().numpy()
    assert got_s.shape == want_s.shape and np.array_equal(got_s, want_s)
    bad = np.argwhere(got_c != want_c)
    assert bad.size == 0, f"{len(bad)} codes differ, first at {bad[0].tolist()}"


def test_quantize_mxfp8_many_rows(dsa):
    """A launch of many blocks with a ragged tail (rows x dim / 8 not a multiple of 256)."""
    rng = np.random.default_rng(23)
    bits = _rows(rng, 4099, 128)
    x = torch.from_numpy(bits.view(np.int16)).cuda()
    codes, scales = dsa.quantize_mxfp8(x)
    want_c, want_s = M.quantize_mxfp8(decode_bf16(bits))
    assert np.array_equal(scales.cpu().numpy(), want_s)
    assert np.array_equal(codes.cpu().numpy(), want_c)


@pytest.mark.parametrize("dim", [64, 128])
def test_index_cache_append_matches_oracle(dsa, dim):
    rng = np.random.default_rng(29 + dim)
    pages, B, maxp = 24, 5, 6
    lens = np.array([1, 64, 65, 300, 384], dtype=np.int32)
    bt = np.full((B, maxp), -1, dtype=np.int32)
    perm = rng.permutation(pages).astype(np.int32)
    off = 0
    for b in range(B):
        npg = (lens[b] + 63) // 64
        bt[b, :npg] = perm[off:off + npg]
        off += npg
    cache_c = rng.integers(0, 256, (pages, 64, dim)).astype(np.uint8)
    cache_s = rng.integers(0, 256, (pages, 64, dim // 32)).astype(np.uint8)
    # decode append (each sequence's newest position), then a multi-token append with
    # explicit positions, one of them on an unmapped page (skipped, error bit)
    k1 = _rows(rng, 6, dim)[1:].copy()  # signed zeros, subnormals, ties, saturation, huge
    seq2 = np.array([3, 3, 3, 4, 0], dtype=np.int32)
    pos2 = np.array([200, 201, 299, 383, 70], dtype=np.int32)  # (0, 70): page 1 of row 0 is unmapped
    k2 = _rows(rng, 6, dim)[1:][::-1].copy()

    dev = lambda a: torch.from_numpy(a).cuda()
    d_c, d_s = dev(cache_c.copy()), dev(cache_s.copy())
    bt_d, lens_d, lens_h = dev(bt), dev(lens), torch.from_numpy(lens.copy())
    ws = dsa.alloc_workspace(256)
    dsa.index_cache_append_mxfp8(dev(k1.view(np.int16)), d_c, d_s, bt_d, lens_d, lens_h, ws)
    assert dsa.read_device_error(ws) == 0
    dsa.index_cache_append_mxfp8(dev(k2.view(np.int16)), d_c, d_s, bt_d, lens_d, lens_h, ws,
                                 token_seq=dev(seq2), token_pos=dev(pos2),
                                 token_seq_host=torch.from_numpy(seq2.copy()),
                                 token_pos_host=torch.from_numpy(pos2.copy()))
    assert dsa.read_device_error(ws) == dsa.DSA_DEVERR_PAGE_ID

    c1, s1 = M.quantize_mxfp8(decode_bf16(k1))
    want_c, want_s, bad = M.append_rows(cache_c, cache_s, bt, np.arange(B), lens - 1, c1, s1)
    assert bad == []
    c2, s2 = M.quantize_mxfp8(decode_bf16(k2))
    want_c, want_s, bad = M.append_rows(want_c, want_s, bt, seq2, pos2, c2, s2)
    assert bad == [4]
    assert np.array_equal(d_s.cpu().numpy(), want_s)
    assert np.array_equal(d_c.cpu().numpy(), want_c)


def test_appended_cache_feeds_the_indexer_layout(dsa):
    """Quantised rows dequantise (E4M3 value x 2^(byte - 127) per group) to within half an
    E4M3 step of the bf16 input: the layout the MX indexer reads."""
    rng = np.random.default_rng(31)
    bits = _rows(rng, 64, 128)[6:]
    x = torch.from_numpy(bits.view(np.int16)).cuda()
    codes, scales = dsa.quantize_mxfp8(x)
    back = M.dequantize_mxfp8(codes.cpu().numpy(), scales.cpu().numpy())
    ref = decode_bf16(bits)
    rel = np.abs(back - ref) / np.maximum(np.abs(ref), 1e-300)
    y = np.abs(ref) / np.repeat(np.ldexp(1.0, scales.cpu().numpy().astype(np.int64) - 127), 32, axis=1)
    normal = (y >= 2.0 ** -6) & (y <= 448)  # E4M3 normals, short of saturation
    assert normal.mean() > 0.5
    assert np.all(rel[normal] <= 2.0 ** -4)
    assert np.all(np.abs(back[y > 448]) == 448 * np.ldexp(1.0, scales.cpu().numpy().astype(np.int64) - 127).repeat(32, axis=1)[y > 448])


# ---------------------------------------------------------------------------------
# appends of new rows to bf16 / FP8 K-index caches and latent caches
# ---------------------------------------------------------------------------------
def _paged_layout(rng, pages=24):
    B, maxp = 5, 6
    lens = np.array([1, 64, 65, 300, 384], dtype=np.int32)
    bt = np.full((B, maxp), -1, dtype=np.int32)
    perm = rng.permutation(pages).astype(np.int32)
    off = 0
    for b in range(B):
        npg = (lens[b] + 63) // 64
        bt[b, :npg] = perm[off:off + npg]
        off += npg
    # a multi-token append with explicit positions, one on an unmapped page (skipped)
    seq2 = np.array([3, 3, 3, 4, 0], dtype=np.int32)
    pos2 = np.array([200, 201, 299, 383, 70], dtype=np.int32)
    return pages, B, lens, bt, seq2, pos2


def _run_two_appends(dsa, fn, k1, k2, bt, lens, seq2, pos2):
    """fn(x, bt, lens, lens_host, ws, **tokens): a decode append (each sequence's newest
    position) then the explicit multi-token one; returns the two error words."""
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    bt_d, lens_d, lens_h = dev(bt), dev(lens), torch.from_numpy(lens.copy())
    ws = dsa.alloc_workspace(256)
    fn(dev(k1.view(np.int16)), bt_d, lens_d, lens_h, ws)
    e1 = dsa.read_device_error(ws)
    dsa.clear_device_error(ws)
    fn(dev(k2.view(np.int16)), bt_d, lens_d, lens_h, ws, token_seq=dev(seq2), token_pos=dev(pos2),
       token_seq_host=torch.from_numpy(seq2.copy()), token_pos_host=torch.from_numpy(pos2.copy()))
    return e1, dsa.read_device_error(ws)


@pytest.mark.parametrize("fmt", ["bf16", "fp8"])
@pytest.mark.parametrize("dim", [64, 128])
def test_index_cache_append_formats_match_oracle(dsa, fmt, dim):
    """bf16 rows copied; e4m3 rows with one f32 scale per token (absmax / 448) bit for bit
    (codes and scale bits), including zero rows, signed zeros, subnormals and huge values."""
    from oracle import fp8_quant as F
    rng = np.random.default_rng(41 + dim)
    pages, B, lens, bt, seq2, pos2 = _paged_layout(rng)
    k1 = _rows(rng, 6, dim)[1:].copy()
    k2 = _rows(rng, 6, dim)[::-1][:5].copy()
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    if fmt == "bf16":
        cache0 = [rng.integers(0, 2 ** 16, (pages, 64, dim)).astype(np.uint16)]
        d_c = dev(cache0[0].view(np.int16))
        d_s = None
        rows = lambda k: [k]
    else:
        cache0 = [rng.integers(0, 256, (pages, 64, dim)).astype(np.uint8),
                  rng.standard_normal((pages, 64)).astype(np.float32)]
        d_c, d_s = dev(cache0[0]), dev(cache0[1])
        rows = lambda k: list(F.quantize_index_rows(k))
    fn = lambda x, bt_d, lens_d, lens_h, ws, **kw: dsa.index_cache_append(x, d_c, d_s, bt_d, lens_d, lens_h, ws, **kw)
    e1, e2 = _run_two_appends(dsa, fn, k1, k2, bt, lens, seq2, pos2)
    assert e1 == 0 and e2 == dsa.DSA_DEVERR_PAGE_ID
    want, bad = F.append(cache0, bt, np.arange(B), lens - 1, rows(k1))
    assert bad == []
    want, bad = F.append(want, bt, seq2, pos2, rows(k2))
    assert bad == [4]
    got = [d_c.cpu().numpy()] + ([d_s.cpu().numpy()] if d_s is not None else [])
    for g, w in zip(got, want):
        assert np.array_equal(g.view(np.uint8), np.ascontiguousarray(w).view(np.uint8))


@pytest.mark.parametrize("fmt", ["bf16", "fp8"])
def test_latent_cache_append_matches_oracle(dsa, fmt):
    """bf16 latent rows copied; FP8 rows: each 128-dim latent tile quantised (absmax / 448)
    to e4m3 codes and an f32 scale, the 64 rope dims copied, all bit for bit."""
    from oracle import fp8_quant as F
    rng = np.random.default_rng(53)
    pages, B, lens, bt, seq2, pos2 = _paged_layout(rng)
    k1 = _rows(rng, 6, 576)[1:].copy()
    k2 = _rows(rng, 6, 576)[::-1][:5].copy()
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    if fmt == "bf16":
        cache0 = [rng.integers(0, 2 ** 16, (pages, 64, 576)).astype(np.uint16)]
        dc = [dev(cache0[0].view(np.int16))]
        fn = lambda x, bt_d, lens_d, lens_h, ws, **kw: dsa.latent_cache_append(x, dc[0], bt_d, lens_d, lens_h, ws, **kw)
        rows = lambda k: [k]
    else:
        cache0 = [rng.integers(0, 256, (pages, 64, 512)).astype(np.uint8),
                  rng.standard_normal((pages, 64, 4)).astype(np.float32),
                  rng.integers(0, 2 ** 16, (pages, 64, 64)).astype(np.uint16)]
        dc = [dev(cache0[0]), dev(cache0[1]), dev(cache0[2].view(np.int16))]
        fn = lambda x, bt_d, lens_d, lens_h, ws, **kw: dsa.latent_cache_append(
            x, dc[0], bt_d, lens_d, lens_h, ws, cache_scale=dc[1], cache_rope=dc[2], **kw)
        rows = lambda k: list(F.quantize_latent_rows(k))
    e1, e2 = _run_two_appends(dsa, fn, k1, k2, bt, lens, seq2, pos2)
    assert e1 == 0 and e2 == dsa.DSA_DEVERR_PAGE_ID
    want, bad = F.append(cache0, bt, np.arange(B), lens - 1, rows(k1))
    want, bad = F.append(want, bt, seq2, pos2, rows(k2))
    assert bad == [4]
    for g, w in zip(dc, want):
        assert np.array_equal(g.cpu().numpy().view(np.uint8), np.ascontiguousarray(w).view(np.uint8))
