"""Parity of the CUDA path (through the C ABI) with the float64 oracle.

Workspaces are poisoned (every byte after the error word set to 0xFF, NaN as f32), so a
kernel that reads scratch nobody wrote fails these checks instead of reading zeros.

Indices and their scores must match bit for bit (the exactness certificate guarantees the
fp32 scores are exact).  Attention outputs must satisfy, against the float64 oracle,
max |err| <= 2e-2 and relative RMS (||o - r|| / ||r|| over the compared tensor) <= 1e-2:
the BF16 tolerance of the DSA hot path.  Every sparse-attention output here is bf16 from
bf16 inputs, so that tolerance applies to all configs, including those whose indexer
runs in FP8.
"""
import numpy as np
import pytest
import torch

import dsa_workloads as W
from oracle import dsa_oracle as O

pytestmark = pytest.mark.gpu

ATOL = 2e-2
RRMS = 1e-2
# FP8 paths (an FP8 latent cache feeds the attention): the looser bar for FP8
ATOL_FP8 = 6e-2
RRMS_FP8 = 3e-2


@pytest.fixture(scope="module")
def dsa():
    import sparse_attention_decode_dsa_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def _device(wl):
    from dsa_workloads.device import to_device
    return to_device(wl)


def _run_fused(dsa, plan, T, K, H):
    out_idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
    ws = dsa.alloc_workspace(plan.ws_fused(), poison=True)
    dsa.fused_decode(plan, out_idx, out, ws)
    torch.cuda.synchronize()
    assert dsa.read_device_error(ws) == 0
    return out_idx.cpu().numpy(), out.float().cpu().numpy().astype(np.float64)


def _run_indexer(dsa, plan, T, K):
    out_idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
    out_sc = torch.empty((T, K), dtype=torch.float32, device="cuda")
    ws = dsa.alloc_workspace(plan.ws_indexer(), poison=True)
    dsa.indexer_topk(plan, out_idx, ws, out_score=out_sc)
    torch.cuda.synchronize()
    assert dsa.read_device_error(ws) == 0
    return out_idx.cpu().numpy(), out_sc.cpu().numpy().astype(np.float64)


def _run_sfa(dsa, plan, idx_np, H):
    T, K = idx_np.shape
    idx = torch.from_numpy(np.ascontiguousarray(idx_np, dtype=np.int32)).cuda()
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
    ws = dsa.alloc_workspace(plan.ws_sfa(), poison=True)
    dsa.sparse_attn(plan, idx, out, ws)
    torch.cuda.synchronize()
    assert dsa.read_device_error(ws) == 0
    return out.float().cpu().numpy().astype(np.float64)


def _check_attn(got, want, label, fp8=False):
    err = np.abs(got - want)
    denom = np.linalg.norm(want)
    rrms = np.linalg.norm(got - want) / denom if denom > 0 else np.linalg.norm(got)
    atol, rr = (ATOL_FP8, RRMS_FP8) if fp8 else (ATOL, RRMS)
    assert err.max() <= atol, f"{label}: max |err| {err.max():.3e}"
    assert rrms <= rr, f"{label}: relative RMS {rrms:.3e}"
    return err.max(), rrms


def _check_config(dsa, spec, tokens=None):
    wl = W.make(spec)
    d = _device(wl)
    plan = dsa.Plan(d)
    T, K, H = wl.n_tokens, spec.topk, spec.sfa_heads
    toks = list(range(T)) if tokens is None else tokens
    ref = {t: O.step(wl, t) for t in toks}

    idx_g, sc_g = _run_indexer(dsa, plan, T, K)
    for t in toks:
        ri, rs, _ = ref[t]
        assert np.array_equal(idx_g[t], ri), f"{spec.name} token {t}: indices differ"
        assert np.array_equal(sc_g[t], rs, equal_nan=True), f"{spec.name} token {t}: scores differ"

    fidx, fout = _run_fused(dsa, plan, T, K, H)
    assert np.array_equal(fidx[toks], idx_g[toks])
    want = np.stack([ref[t][2] for t in toks])
    fp8kv = spec.kv_format != "bf16"
    _check_attn(fout[toks], want, f"{spec.name} fused", fp8kv)

    # the attention fed the oracle's own indices (indexer and attention checked apart)
    oidx = idx_g.copy()
    for t in toks:
        oidx[t] = ref[t][0]
    sout = _run_sfa(dsa, plan, oidx, H)
    _check_attn(sout[toks], want, f"{spec.name} sfa", fp8kv)
    return wl


@pytest.mark.parametrize("spec", W.SMALL, ids=lambda s: s.name)
def test_small_configs(dsa, spec):
    _check_config(dsa, spec)


def test_tiny_decode(dsa):
    _check_config(dsa, W.TINY_DECODE)


def test_bf16_decode_sampled(dsa):
    _check_config(dsa, W.BF16_DECODE, tokens=[0, 13, 31])


def test_fp8_decode_sampled(dsa):
    _check_config(dsa, W.FP8_DECODE, tokens=[1, 30])


def test_ragged_mxfp8_decode_sampled(dsa):
    _check_config(dsa, W.RAGGED_MXFP8_DECODE, tokens=[0, 3, 6, 7])


def test_causal_prefill_sampled(dsa):
    _check_config(dsa, W.CAUSAL_PREFILL, tokens=[0, 1, 63, 64, 2046, 2047, 2048, 5000, 8191])


@pytest.mark.parametrize("spec", [W.CAUSAL_PREFILL_FP8, W.CAUSAL_PREFILL_MX], ids=lambda s: s.name)
def test_causal_prefill_quantised_sampled(dsa, spec):
    """The 8192-token causal prefill with an e4m3 (per-token scales) or MXFP8 indexer: the
    keys are dequantised exactly to bf16 once, then the row-blocked tensor-core kernel
    scores 21 rows per key tile; indices and scores bit-exact on sampled rows."""
    _check_config(dsa, spec, tokens=[0, 1, 63, 64, 2047, 2048, 5000, 8191])


def test_fp8_latent_decode_sampled(dsa):
    """The BF16 decode's sizes with an FP8 latent cache (e4m3 latent dims with an f32 scale
    per 128-dim tile, bf16 rope dims): two splits per token merged in their cluster."""
    _check_config(dsa, W.FP8KV_DECODE, tokens=[0, 17, 31])


def test_multi_token_decode_sampled(dsa):
    """Four draft tokens per sequence at the BF16 decode's sizes (128 tokens, 32768-token
    contexts): the four rows of a sequence share each K-index tile."""
    _check_config(dsa, W.BF16_MULTI_DECODE, tokens=[0, 1, 2, 3, 62, 125, 127])


@pytest.mark.parametrize("spec", [W.SMALL_DECODE_BF16, W.SMALL_DECODE_FP8, W.SMALL_DECODE_MX, W.SMALL_FP8_D64,
                                  W.SMALL_MX_D64, W.SMALL_MX_H40, W.SMALL_H8, W.SMALL_PREFILL, W.SMALL_MULTI],
                         ids=lambda s: s.name)
def test_relu_activation(dsa, spec):
    """The per-head ReLU variant against the oracle's 'relu' reading, in every key format
    and width (per-head tensor-core kernel for 128-dim keys, the CUDA-core kernel for
    64-dim e4m3 keys)."""
    wl = W.make(spec, with_latent=False)
    d = _device(wl)
    d.act = dsa.DSA_ACT_RELU
    plan = dsa.Plan(d)
    idx_g, sc_g = _run_indexer(dsa, plan, wl.n_tokens, spec.topk)
    for t in range(wl.n_tokens):
        ri, rs = O.indexer_topk(wl, t, act="relu")
        assert np.array_equal(idx_g[t], ri)
        assert np.array_equal(sc_g[t], rs, equal_nan=True)


def test_bad_page_id_sets_error_bit_and_gpu_stays_usable(dsa):
    spec = W.SMALL_DECODE_BF16
    wl = W.make(spec)
    d = _device(wl)
    d.block_table[5, 3] = wl.num_pages + 100     # outside the cache
    plan = dsa.Plan(d)
    ws = dsa.alloc_workspace(plan.ws_fused())
    out_idx = torch.empty((wl.n_tokens, spec.topk), dtype=torch.int32, device="cuda")
    out = torch.empty((wl.n_tokens, spec.sfa_heads, 512), dtype=torch.bfloat16, device="cuda")
    dsa.fused_decode(plan, out_idx, out, ws)
    err = dsa.read_device_error(ws)
    assert err & dsa.DSA_DEVERR_PAGE_ID
    dsa.clear_device_error(ws)
    assert dsa.read_device_error(ws) == 0
    _check_config(dsa, W.SMALL_H8)               # the context is still healthy


def test_out_of_range_index_sets_error_bit(dsa):
    spec = W.SMALL_DECODE_BF16
    wl = W.make(spec)
    plan = dsa.Plan(_device(wl))
    idx = np.full((wl.n_tokens, spec.topk), -1, np.int32)
    idx[:, 0] = 0
    idx[1, 1] = 5000                             # beyond sequence 1's 37 tokens
    ws = dsa.alloc_workspace(plan.ws_sfa())
    out = torch.empty((wl.n_tokens, spec.sfa_heads, 512), dtype=torch.bfloat16, device="cuda")
    dsa.sparse_attn(plan, torch.from_numpy(idx).cuda(), out, ws)
    assert dsa.read_device_error(ws) & dsa.DSA_DEVERR_INDEX


def test_repeated_calls_are_deterministic(dsa):
    spec = W.SMALL_DECODE_MX
    wl = W.make(spec)
    plan = dsa.Plan(_device(wl))
    a = _run_fused(dsa, plan, wl.n_tokens, spec.topk, spec.sfa_heads)
    b = _run_fused(dsa, plan, wl.n_tokens, spec.topk, spec.sfa_heads)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("spec", [W.SMALL_DECODE_BF16, W.SMALL_PREFILL, W.SMALL_DECODE_FP8],
                         ids=lambda s: s.name)
def test_cuda_graph_replay_matches_eager(dsa, spec):
    """The fused call captured into a CUDA graph and replayed gives the eager call's
    indices and outputs bit for bit (the library launches only kernels and holds no
    host-side state a replay could miss); the workspace is reused across replays."""
    wl = W.make(spec)
    plan = dsa.Plan(_device(wl))
    T, K, H = wl.n_tokens, spec.topk, spec.sfa_heads
    want = _run_fused(dsa, plan, T, K, H)
    out_idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
    ws = dsa.alloc_workspace(plan.ws_fused())
    dsa.fused_decode(plan, out_idx, out, ws)  # first call on the device outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=cap):
        dsa.fused_decode(plan, out_idx, out, ws, stream=cap)
    for _ in range(3):
        out_idx.fill_(-7)
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert dsa.read_device_error(ws) == 0
        assert np.array_equal(out_idx.cpu().numpy(), want[0])
        assert np.array_equal(out.float().cpu().numpy().astype(np.float64), want[1])


def _indexer_vs_oracle(dsa, wl, label):
    d = _device(wl)
    plan = dsa.Plan(d)
    idx_g, sc_g = _run_indexer(dsa, plan, wl.n_tokens, wl.spec.topk)
    for t in range(wl.n_tokens):
        ri, rs = O.indexer_topk(wl, t)
        assert np.array_equal(idx_g[t], ri), f"{label} token {t}: indices differ"
        assert np.array_equal(sc_g[t], rs, equal_nan=True), f"{label} token {t}: scores differ"
    return idx_g


def test_topk_all_scores_equal_on_long_rows(dsa):
    """An all-zero indexer query gives every key the same score, the method's degenerate
    case: the answer is positions 0..K-1 (ties to the lower position).  Every CTA's
    boundary bin then holds all its keys, far more than its share of the candidate pool,
    so the selection takes the rescanning radix select on rows of 40000, 34816 and 9000
    keys (clusters of eight CTAs)."""
    wl = W.make(W.LONG_ROWS, with_latent=False)
    wl.idx_q[...] = 0                              # bf16 +0
    idx_g = _indexer_vs_oracle(dsa, wl, "all-equal")
    assert np.array_equal(idx_g, np.tile(np.arange(W.LONG_ROWS.topk, dtype=np.int32), (wl.n_tokens, 1)))


def test_topk_boundary_bin_near_pool_capacity(dsa):
    """One nonzero query element: each score is w * q * k_t0 with k_t0 an integer in
    [-8, 8], so the scores take 17 values and the K-th largest sits in a bin holding
    about 1/17 of each CTA's keys -- close to a CTA's share of the candidate pool (256 of
    2048 in a cluster of eight), below it in some CTAs and above it in others, on the
    34816-key row in particular.  Both the pooled select and its fallback must give the
    oracle's answer."""
    wl = W.make(W.LONG_ROWS, with_latent=False)
    wl.idx_q[...] = 0
    wl.idx_q[:, 0, 0] = 0x3F80                     # bf16 1.0 in head 0, dim 0
    _indexer_vs_oracle(dsa, wl, "17 values")


def test_indexer_wait_timeout_unwinds_and_the_context_stays_usable(dsa):
    """Every pipeline wait of the indexer's tensor-core kernels is bounded.  With the
    limit lowered to 300 cycles the ordinary waits (a TMA load landing, an MMA completing,
    an accumulator freed) run out: each call must return with DSA_DEVERR_TIMEOUT in the
    error word, and -- the kernels having let their in-flight copies and MMAs finish and
    freed their tensor memory -- full parity checks on the same context afterwards must be
    green.  The per-head, row-blocked and MX paths wait for the query's TMA load right
    after issuing it, so a wait always runs out there; the folded FP8 path's loads may
    land before its first probe, so it need only return with no other error bit."""
    specs = [W.SMALL_DECODE_BF16, W.SMALL_PREFILL, W.SMALL_DECODE_MX, W.SMALL_DECODE_FP8]
    assert dsa.lib.dsa_set_indexer_wait_limit(-1) == dsa.DSA_ERR_INVALID_ARG
    assert dsa.lib.dsa_set_indexer_wait_limit(300) == dsa.DSA_OK
    try:
        for spec in specs:
            wl = W.make(spec, with_latent=False)
            plan = dsa.Plan(_device(wl))
            out_idx = torch.empty((wl.n_tokens, spec.topk), dtype=torch.int32, device="cuda")
            ws = dsa.alloc_workspace(plan.ws_indexer(), poison=True)
            dsa.indexer_topk(plan, out_idx, ws)
            torch.cuda.synchronize()
            err = dsa.read_device_error(ws)
            assert err & ~dsa.DSA_DEVERR_TIMEOUT == 0, f"{spec.name}: error word {err:#x}"
            if spec is not W.SMALL_DECODE_FP8:
                assert err & dsa.DSA_DEVERR_TIMEOUT, f"{spec.name}: no wait ran out"
    finally:
        assert dsa.lib.dsa_set_indexer_wait_limit(0) == dsa.DSA_OK
    for spec in specs:
        _check_config(dsa, spec)


@pytest.mark.parametrize("spec", [W.BF16_DECODE, W.FP8_DECODE, W.RAGGED_MXFP8_DECODE, W.FP8KV_DECODE],
                         ids=lambda s: s.name)
def test_back_to_back_steps_agree(dsa, spec):
    """Thirty fused steps issued back to back, each kernel's set-up overlapping the previous
    one's tail, give bit-identical indices and outputs equal to an isolated step's, and
    leave the error word clear.  A pipeline race (a barrier phase taken for another, a
    stage refilled while still read) shows up here as a differing step or a timeout."""
    wl = W.make(spec)
    plan = dsa.Plan(_device(wl))
    T, K, H = wl.n_tokens, spec.topk, spec.sfa_heads
    ref_idx, ref_out = _run_fused(dsa, plan, T, K, H)
    n = 30
    ws = dsa.alloc_workspace(plan.ws_fused(), poison=True)
    idx = [torch.empty((T, K), dtype=torch.int32, device="cuda") for _ in range(n)]
    out = [torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    for i in range(n):
        dsa.fused_decode(plan, idx[i], out[i], ws)
    torch.cuda.synchronize()
    assert dsa.read_device_error(ws) == 0
    want_idx = torch.from_numpy(ref_idx).cuda()
    want_out = torch.from_numpy(ref_out).cuda()
    for i in range(n):
        assert torch.equal(idx[i], want_idx), f"step {i}: indices differ from the isolated step"
        assert torch.equal(out[i].double(), want_out), f"step {i}: outputs differ from the isolated step"
