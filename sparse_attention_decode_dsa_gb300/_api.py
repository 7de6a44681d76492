"""Marshalling from torch tensors to the C structs of include/dsa.h and back."""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass
from typing import Optional

import torch

from . import (lib, _check, PageTable, Tokens, IndexCache, IndexerArgs, LatentCache, SfaArgs, Trace,
               DSA_BF16, DSA_E4M3, DSA_SCALE_NONE, DSA_SCALE_PER_TOKEN_F32, DSA_SCALE_MX_E8M0_G32,
               DSA_ACT_IDENTITY)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return C.c_void_p(t.data_ptr())


def _i32_host_ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    assert t.device.type == "cpu" and t.dtype == torch.int32 and t.is_contiguous()
    return C.cast(C.c_void_p(t.data_ptr()), C.POINTER(C.c_int32))


def _stream_ptr(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


@dataclass
class DeviceInputs:
    """Device-resident inputs of one DSA step (caller-owned torch tensors).

    Storage dtypes: bf16 tensors may be torch.bfloat16 or raw uint16/int16 bits; e4m3
    tensors are torch.float8_e4m3fn or uint8 bytes; E8M0 scales are uint8.
    """
    block_table: torch.Tensor            # int32 [B, max_pages] (device)
    seq_lens: torch.Tensor               # int32 [B] (device)
    seq_lens_host: torch.Tensor          # int32 [B] (host)
    num_pages: int
    idx_q: torch.Tensor                  # [T, H_I, d]
    head_w: torch.Tensor                 # f32 [T, H_I]
    idx_k: torch.Tensor                  # [num_pages, 64, d]
    top_k: int
    idx_q_scale: Optional[torch.Tensor] = None
    idx_k_scale: Optional[torch.Tensor] = None
    kv: Optional[torch.Tensor] = None    # bf16 [num_pages, 64, 576]
    kv_codes: Optional[torch.Tensor] = None  # FP8 latent cache: e4m3 codes [num_pages, 64, 512]
    kv_scale: Optional[torch.Tensor] = None  #   f32 [num_pages, 64, 4], one per 128-dim tile
    kv_rope: Optional[torch.Tensor] = None   #   bf16 [num_pages, 64, 64]
    sfa_q: Optional[torch.Tensor] = None  # bf16 [T, H, 576]
    softmax_scale: float = 576 ** -0.5
    token_seq: Optional[torch.Tensor] = None
    token_pos: Optional[torch.Tensor] = None
    token_seq_host: Optional[torch.Tensor] = None
    token_pos_host: Optional[torch.Tensor] = None
    act: int = DSA_ACT_IDENTITY

    @property
    def n_tokens(self) -> int:
        return int(self.idx_q.shape[0]) if self.idx_q is not None else int(self.sfa_q.shape[0])


class Plan:
    """C structs for one set of device inputs, kept alive together with the tensors."""

    def __init__(self, d: DeviceInputs):
        self.d = d
        B, maxp = d.block_table.shape
        self.pages = PageTable(_ptr(d.block_table), _ptr(d.seq_lens), _i32_host_ptr(d.seq_lens_host),
                               B, maxp, 64, d.num_pages)
        self.tokens = Tokens(d.n_tokens, _ptr(d.token_seq), _ptr(d.token_pos),
                             _i32_host_ptr(d.token_seq_host), _i32_host_ptr(d.token_pos_host))
        dt = DSA_BF16 if d.idx_k.element_size() == 2 else DSA_E4M3
        if d.idx_k_scale is None:
            sk = DSA_SCALE_NONE
        elif d.idx_k_scale.dtype == torch.float32:
            sk = DSA_SCALE_PER_TOKEN_F32
        else:
            sk = DSA_SCALE_MX_E8M0_G32
        self.icache = IndexCache(_ptr(d.idx_k), _ptr(d.idx_k_scale), dt, sk, int(d.idx_k.shape[-1]))
        self.iargs = IndexerArgs(_ptr(d.idx_q), _ptr(d.idx_q_scale), dt, sk, _ptr(d.head_w),
                                 int(d.idx_q.shape[1]), int(d.top_k), int(d.act))
        if d.kv_codes is not None:
            self.lcache = LatentCache(_ptr(d.kv_codes), 576, 512, DSA_E4M3, _ptr(d.kv_scale), _ptr(d.kv_rope))
        else:
            self.lcache = LatentCache(_ptr(d.kv), 576, 512, DSA_BF16, None, None) if d.kv is not None else None
        self.sargs = (SfaArgs(_ptr(d.sfa_q), int(d.sfa_q.shape[1]), float(d.softmax_scale))
                      if d.sfa_q is not None else None)

    def ws_indexer(self) -> int:
        return lib.dsa_indexer_workspace_size(C.byref(self.iargs), C.byref(self.icache),
                                              C.byref(self.pages), C.byref(self.tokens))

    def ws_sfa(self) -> int:
        return lib.dsa_sparse_attn_workspace_size(C.byref(self.sargs), C.byref(self.pages),
                                                  C.byref(self.tokens), int(self.d.top_k))

    def ws_fused(self) -> int:
        return lib.dsa_fused_workspace_size(C.byref(self.iargs), C.byref(self.icache), C.byref(self.sargs),
                                            C.byref(self.pages), C.byref(self.tokens))


def workspace_size(plan: Plan, which: str = "fused") -> int:
    return {"fused": plan.ws_fused, "indexer": plan.ws_indexer, "sfa": plan.ws_sfa}[which]()


def alloc_workspace(nbytes: int, device="cuda", poison: bool = False) -> torch.Tensor:
    """A 256-byte aligned workspace (torch allocations are 512-byte aligned), zeroed.

    ``poison=True`` fills everything after the 256-byte header (whose error word must
    start at zero) with 0xFF bytes -- NaN as f32, 0xFFFFFFFF as a counter -- so that a
    kernel reading scratch it has not written shows up as a wrong result."""
    ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
    if poison:
        ws[256:].fill_(0xFF)
    return ws


def indexer_topk(plan: Plan, out_idx: torch.Tensor, ws: torch.Tensor, out_score: Optional[torch.Tensor] = None,
                 stream=None, trace: Optional[Trace] = None):
    _check(lib.dsa_indexer_topk(C.byref(plan.iargs), C.byref(plan.icache), C.byref(plan.pages),
                                C.byref(plan.tokens), _ptr(out_idx), _ptr(out_score), _ptr(ws),
                                ws.numel() * ws.element_size(), _stream_ptr(stream),
                                C.byref(trace) if trace is not None else None), "dsa_indexer_topk")


def sparse_attn(plan: Plan, idx: torch.Tensor, out: torch.Tensor, ws: torch.Tensor, stream=None,
                trace: Optional[Trace] = None):
    _check(lib.dsa_sparse_attn(C.byref(plan.sargs), C.byref(plan.lcache), C.byref(plan.pages),
                               C.byref(plan.tokens), _ptr(idx), int(idx.shape[-1]), _ptr(out), _ptr(ws),
                               ws.numel() * ws.element_size(), _stream_ptr(stream),
                               C.byref(trace) if trace is not None else None), "dsa_sparse_attn")


def fused_decode(plan: Plan, out_idx: torch.Tensor, out: torch.Tensor, ws: torch.Tensor, stream=None,
                 trace: Optional[Trace] = None):
    _check(lib.dsa_fused_decode(C.byref(plan.iargs), C.byref(plan.icache), C.byref(plan.sargs),
                                C.byref(plan.lcache), C.byref(plan.pages), C.byref(plan.tokens),
                                _ptr(out_idx), _ptr(out), _ptr(ws), ws.numel() * ws.element_size(),
                                _stream_ptr(stream), C.byref(trace) if trace is not None else None),
           "dsa_fused_decode")


def read_device_error(ws: torch.Tensor, stream=None) -> int:
    v = C.c_uint32(0)
    _check(lib.dsa_read_device_error(_ptr(ws), C.byref(v), _stream_ptr(stream)), "dsa_read_device_error")
    return int(v.value)


def clear_device_error(ws: torch.Tensor, stream=None):
    _check(lib.dsa_clear_device_error(_ptr(ws), _stream_ptr(stream)), "dsa_clear_device_error")


def quantize_mxfp8(x: torch.Tensor, codes: Optional[torch.Tensor] = None, scales: Optional[torch.Tensor] = None,
                   stream=None):
    """MXFP8 (groups of 32) of bf16 rows x [..., dim] -> (e4m3 codes uint8 [..., dim], E8M0
    scales uint8 [..., dim / 32]), computed by the library's kernel."""
    assert x.is_cuda and x.element_size() == 2 and x.is_contiguous()
    dim = int(x.shape[-1])
    rows = x.numel() // dim if dim else 0
    if codes is None:
        codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(x.shape[:-1] + (dim // 32,), dtype=torch.uint8, device=x.device)
    _check(lib.dsa_quantize_mxfp8(_ptr(x), rows, dim, _ptr(codes), _ptr(scales), _stream_ptr(stream)),
           "dsa_quantize_mxfp8")
    return codes, scales


def index_cache_append_mxfp8(k_new: torch.Tensor, cache_codes: torch.Tensor, cache_scales: torch.Tensor,
                             block_table: torch.Tensor, seq_lens: torch.Tensor, seq_lens_host: torch.Tensor,
                             ws: torch.Tensor, token_seq: Optional[torch.Tensor] = None,
                             token_pos: Optional[torch.Tensor] = None, token_seq_host: Optional[torch.Tensor] = None,
                             token_pos_host: Optional[torch.Tensor] = None, stream=None):
    """Quantises the new key of every token (bf16 k_new [T, dim]) and writes it to that
    token's (page, slot) of the paged MXFP8 cache (codes [pages, 64, dim], scales
    [pages, 64, dim / 32]).  Token i is batch row token_seq[i] (or i) at position
    token_pos[i] (or seq_len - 1)."""
    assert k_new.is_cuda and k_new.element_size() == 2 and k_new.is_contiguous()
    B, maxp = block_table.shape
    pages = PageTable(_ptr(block_table), _ptr(seq_lens), _i32_host_ptr(seq_lens_host), B, maxp, 64,
                      int(cache_codes.shape[0]))
    tokens = Tokens(int(k_new.shape[0]), _ptr(token_seq), _ptr(token_pos), _i32_host_ptr(token_seq_host),
                    _i32_host_ptr(token_pos_host))
    _check(lib.dsa_index_cache_append_mxfp8(_ptr(k_new), int(k_new.shape[-1]), C.byref(pages), C.byref(tokens),
                                            _ptr(cache_codes), _ptr(cache_scales), _ptr(ws),
                                            ws.numel() * ws.element_size(), _stream_ptr(stream)),
           "dsa_index_cache_append_mxfp8")


def _pages_tokens(block_table, seq_lens, seq_lens_host, num_pages, n_tokens, token_seq, token_pos, token_seq_host,
                  token_pos_host):
    B, maxp = block_table.shape
    pages = PageTable(_ptr(block_table), _ptr(seq_lens), _i32_host_ptr(seq_lens_host), B, maxp, 64, int(num_pages))
    tokens = Tokens(int(n_tokens), _ptr(token_seq), _ptr(token_pos), _i32_host_ptr(token_seq_host),
                    _i32_host_ptr(token_pos_host))
    return pages, tokens


def index_cache_append(k_new: torch.Tensor, cache: torch.Tensor, cache_scale: Optional[torch.Tensor],
                       block_table: torch.Tensor, seq_lens: torch.Tensor, seq_lens_host: torch.Tensor,
                       ws: torch.Tensor, token_seq=None, token_pos=None, token_seq_host=None, token_pos_host=None,
                       stream=None):
    """Writes the new key of every token (bf16 k_new [T, dim]) to its (page, slot) of the
    paged K-index cache: bf16 cache [pages, 64, dim] (copied), or e4m3 (uint8) with
    per-token f32 scales [pages, 64] or MX E8M0 scales [pages, 64, dim / 32]."""
    assert k_new.is_cuda and k_new.element_size() == 2 and k_new.is_contiguous()
    if cache.element_size() == 2:
        dt, sk = DSA_BF16, DSA_SCALE_NONE
    else:
        dt = DSA_E4M3
        sk = DSA_SCALE_PER_TOKEN_F32 if cache_scale.dtype == torch.float32 else DSA_SCALE_MX_E8M0_G32
    icache = IndexCache(_ptr(cache), _ptr(cache_scale), dt, sk, int(cache.shape[-1]))
    pages, tokens = _pages_tokens(block_table, seq_lens, seq_lens_host, cache.shape[0], k_new.shape[0], token_seq,
                                  token_pos, token_seq_host, token_pos_host)
    _check(lib.dsa_index_cache_append(_ptr(k_new), C.byref(icache), C.byref(pages), C.byref(tokens), _ptr(ws),
                                      ws.numel() * ws.element_size(), _stream_ptr(stream)), "dsa_index_cache_append")


def latent_cache_append(rows_new: torch.Tensor, cache: torch.Tensor, block_table: torch.Tensor,
                        seq_lens: torch.Tensor, seq_lens_host: torch.Tensor, ws: torch.Tensor,
                        cache_scale: Optional[torch.Tensor] = None, cache_rope: Optional[torch.Tensor] = None,
                        token_seq=None, token_pos=None, token_seq_host=None, token_pos_host=None, stream=None):
    """Writes the new latent row of every token (bf16 rows_new [T, 576]) to its (page,
    slot) of the paged latent cache: bf16 cache [pages, 64, 576] (copied), or FP8 (codes
    uint8 [pages, 64, 512], f32 scales [pages, 64, 4] per 128-dim tile, bf16 rope
    [pages, 64, 64])."""
    assert rows_new.is_cuda and rows_new.element_size() == 2 and rows_new.is_contiguous()
    fp8 = cache.element_size() == 1
    lcache = LatentCache(_ptr(cache), 576, 512, DSA_E4M3 if fp8 else DSA_BF16, _ptr(cache_scale), _ptr(cache_rope))
    pages, tokens = _pages_tokens(block_table, seq_lens, seq_lens_host, cache.shape[0], rows_new.shape[0], token_seq,
                                  token_pos, token_seq_host, token_pos_host)
    _check(lib.dsa_latent_cache_append(_ptr(rows_new), C.byref(lcache), C.byref(pages), C.byref(tokens), _ptr(ws),
                                       ws.numel() * ws.element_size(), _stream_ptr(stream)), "dsa_latent_cache_append")
