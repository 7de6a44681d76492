"""dsa_indexer_topk_noalloc: the indexer entry point for callers that cannot allocate.

Some callers of this library cannot call cudaMalloc: plugin hosts or serving runtimes
that give it no allocator and fix their memory budget up front, and request paths that
must not touch the driver's allocator (it can synchronise the device).  For them the
library offers an indexer entry point whose scratch is a fixed 8 MiB array built into
the library.  This test calls it through the C ABI twice in a row and checks both
results against dsa_indexer_topk run with a caller workspace: indices and their
scores must match bit for bit (the indexer's parity bar).  It also checks the claim the
entry point exists for: once the first call has loaded the library's module on the
device (the fixed array is part of that module), a further call changes neither the
device's free memory nor what torch's allocator holds.  An oversized request must be
refused before any launch.

The file is named so that pytest collects it last: it adds an entry point beside the
hot path rather than testing the path itself, so when it fails, a run that stops at the
first failure (``-x``) has already run every other test.  It depends on nothing those
tests leave behind and passes when run alone in a fresh process.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import dsa_workloads as W

pytestmark = pytest.mark.gpu


def _lib_and_plan(dsa, spec):
    from dsa_workloads.device import to_device
    wl = W.make(spec, with_latent=False)
    plan = dsa.Plan(to_device(wl))
    fn = dsa.lib.dsa_indexer_topk_noalloc
    P = C.POINTER
    fn.argtypes = [P(dsa.IndexerArgs), P(dsa.IndexCache), P(dsa.PageTable), P(dsa.Tokens), C.c_void_p,
                   C.c_void_p, C.c_void_p]
    fn.restype = C.c_int
    return wl, plan, fn


def _noalloc(dsa, fn, plan, out_idx, out_sc):
    return fn(C.byref(plan.iargs), C.byref(plan.icache), C.byref(plan.pages), C.byref(plan.tokens),
              C.c_void_p(out_idx.data_ptr()), C.c_void_p(out_sc.data_ptr()),
              C.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("spec", [W.SMALL_DECODE_MX, W.TINY_DECODE, W.BF16_DECODE], ids=lambda s: s.name)
def test_noalloc_matches_workspace_entry_point(spec):
    import sparse_attention_decode_dsa_gb300 as dsa
    wl, plan, fn = _lib_and_plan(dsa, spec)
    T, K = wl.n_tokens, spec.topk
    ref_idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
    ref_sc = torch.empty((T, K), dtype=torch.float32, device="cuda")
    ws = dsa.alloc_workspace(plan.ws_indexer())
    dsa.indexer_topk(plan, ref_idx, ws, out_score=ref_sc)
    outs = [(torch.full((T, K), -7, dtype=torch.int32, device="cuda"),
             torch.full((T, K), -7.0, dtype=torch.float32, device="cuda")) for _ in range(2)]
    torch.cuda.synchronize()
    for call, (idx, sc) in enumerate(outs):
        if call == 1:  # the module holding the fixed array is loaded by now
            free0, held0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
        assert _noalloc(dsa, fn, plan, idx, sc) == dsa.DSA_OK, dsa.lib.dsa_last_error_message()
        torch.cuda.synchronize()
        if call == 1:
            assert torch.cuda.mem_get_info()[0] == free0, "the call changed the device's free memory"
            assert torch.cuda.memory_allocated() == held0
        assert torch.equal(idx, ref_idx), f"call {call}: indices differ"
        assert np.array_equal(sc.cpu().numpy(), ref_sc.cpu().numpy(), equal_nan=True), f"call {call}: scores differ"


def test_noalloc_refuses_requests_beyond_its_scratch():
    import sparse_attention_decode_dsa_gb300 as dsa
    spec = W.replace(W.SMALL_PREFILL, name="noalloc_big", seq_lens=(4160,), prefill_tokens=4160, pool_pages=70)
    wl, plan, fn = _lib_and_plan(dsa, spec)          # 4160 rows x 4160 scores x 4 B > 8 MiB
    idx = torch.empty((wl.n_tokens, spec.topk), dtype=torch.int32, device="cuda")
    sc = torch.empty((wl.n_tokens, spec.topk), dtype=torch.float32, device="cuda")
    assert _noalloc(dsa, fn, plan, idx, sc) == dsa.DSA_ERR_WORKSPACE
    assert b"fixed scratch" in dsa.lib.dsa_last_error_message()
