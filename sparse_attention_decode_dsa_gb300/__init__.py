"""Python binding of the GB300 DSA library (include/dsa.h): argument marshalling only.

Every step of the indexer and of the sparse attention runs in the CUDA kernels of
``libdsa.so``; this module builds the C structs from torch tensors (device pointers,
the current stream) and calls the C entry points of the same names.  There is no
fallback: importing fails loudly when the library is missing and cannot be built.
"""
from __future__ import annotations

import ctypes as C
import os

from . import _build

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsa.so")

DSA_OK, DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED, DSA_ERR_WORKSPACE, DSA_ERR_CUDA = range(5)
DSA_BF16, DSA_E4M3 = 0, 1
DSA_SCALE_NONE, DSA_SCALE_PER_TOKEN_F32, DSA_SCALE_MX_E8M0_G32 = 0, 1, 2
DSA_ACT_IDENTITY, DSA_ACT_RELU = 0, 1
DSA_DEVERR_PAGE_ID, DSA_DEVERR_SEQ_LEN, DSA_DEVERR_INDEX, DSA_DEVERR_TOKEN, DSA_DEVERR_TIMEOUT = 1, 2, 4, 8, 16
DSA_TRACE_MAX = 8

_vp = C.c_void_p
_i32p = C.POINTER(C.c_int32)


class PageTable(C.Structure):
    _fields_ = [("block_table", _vp), ("seq_lens", _vp), ("seq_lens_host", _i32p),
                ("batch", C.c_int32), ("max_pages_per_seq", C.c_int32),
                ("page_size", C.c_int32), ("num_pages", C.c_int32)]


class Tokens(C.Structure):
    _fields_ = [("n_tokens", C.c_int32), ("token_seq", _vp), ("token_pos", _vp),
                ("token_seq_host", _i32p), ("token_pos_host", _i32p)]


class IndexCache(C.Structure):
    _fields_ = [("data", _vp), ("scale", _vp), ("dtype", C.c_int), ("scale_kind", C.c_int),
                ("dim", C.c_int32)]


class IndexerArgs(C.Structure):
    _fields_ = [("q", _vp), ("q_scale", _vp), ("q_dtype", C.c_int), ("q_scale_kind", C.c_int),
                ("head_w", _vp), ("n_heads", C.c_int32), ("top_k", C.c_int32), ("act", C.c_int)]


class LatentCache(C.Structure):
    _fields_ = [("data", _vp), ("dim", C.c_int32), ("v_dim", C.c_int32), ("dtype", C.c_int),
                ("scale", _vp), ("rope", _vp)]


class SfaArgs(C.Structure):
    _fields_ = [("q", _vp), ("n_heads", C.c_int32), ("softmax_scale", C.c_float)]


class Trace(C.Structure):
    _fields_ = [("begin", _vp * DSA_TRACE_MAX), ("end", _vp * DSA_TRACE_MAX),
                ("n_recorded", C.c_int32), ("name", C.c_char_p * DSA_TRACE_MAX)]


def _load() -> C.CDLL:
    if not os.path.exists(LIB_PATH) or not _build.up_to_date():
        _build.build()
    lib = C.CDLL(LIB_PATH)
    P = C.POINTER
    sz = C.c_size_t
    lib.dsa_indexer_workspace_size.argtypes = [P(IndexerArgs), P(IndexCache), P(PageTable), P(Tokens)]
    lib.dsa_indexer_workspace_size.restype = sz
    lib.dsa_indexer_topk.argtypes = [P(IndexerArgs), P(IndexCache), P(PageTable), P(Tokens), _vp, _vp,
                                     _vp, sz, _vp, P(Trace)]
    lib.dsa_indexer_topk.restype = C.c_int
    lib.dsa_sparse_attn_workspace_size.argtypes = [P(SfaArgs), P(PageTable), P(Tokens), C.c_int32]
    lib.dsa_sparse_attn_workspace_size.restype = sz
    lib.dsa_sparse_attn.argtypes = [P(SfaArgs), P(LatentCache), P(PageTable), P(Tokens), _vp, C.c_int32,
                                    _vp, _vp, sz, _vp, P(Trace)]
    lib.dsa_sparse_attn.restype = C.c_int
    lib.dsa_fused_workspace_size.argtypes = [P(IndexerArgs), P(IndexCache), P(SfaArgs), P(PageTable),
                                             P(Tokens)]
    lib.dsa_fused_workspace_size.restype = sz
    lib.dsa_fused_decode.argtypes = [P(IndexerArgs), P(IndexCache), P(SfaArgs), P(LatentCache),
                                     P(PageTable), P(Tokens), _vp, _vp, _vp, sz, _vp, P(Trace)]
    lib.dsa_fused_decode.restype = C.c_int
    lib.dsa_quantize_mxfp8.argtypes = [_vp, C.c_int64, C.c_int32, _vp, _vp, _vp]
    lib.dsa_quantize_mxfp8.restype = C.c_int
    lib.dsa_index_cache_append_mxfp8.argtypes = [_vp, C.c_int32, P(PageTable), P(Tokens), _vp, _vp, _vp,
                                                 C.c_size_t, _vp]
    lib.dsa_index_cache_append_mxfp8.restype = C.c_int
    lib.dsa_index_cache_append.argtypes = [_vp, P(IndexCache), P(PageTable), P(Tokens), _vp, C.c_size_t, _vp]
    lib.dsa_index_cache_append.restype = C.c_int
    lib.dsa_latent_cache_append.argtypes = [_vp, P(LatentCache), P(PageTable), P(Tokens), _vp, C.c_size_t, _vp]
    lib.dsa_latent_cache_append.restype = C.c_int
    lib.dsa_set_indexer_wait_limit.argtypes = [C.c_int64]
    lib.dsa_set_indexer_wait_limit.restype = C.c_int
    lib.dsa_read_device_error.argtypes = [_vp, P(C.c_uint32), _vp]
    lib.dsa_read_device_error.restype = C.c_int
    lib.dsa_clear_device_error.argtypes = [_vp, _vp]
    lib.dsa_clear_device_error.restype = C.c_int
    lib.dsa_status_string.argtypes = [C.c_int]
    lib.dsa_status_string.restype = C.c_char_p
    lib.dsa_last_error_message.argtypes = []
    lib.dsa_last_error_message.restype = C.c_char_p
    lib.dsa_abi_version.argtypes = []
    lib.dsa_abi_version.restype = C.c_int32
    return lib


lib = _load()


class DsaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = lib.dsa_last_error_message().decode()
        super().__init__(f"{where}: {lib.dsa_status_string(status).decode()}: {msg}")


def _check(status: int, where: str):
    if status != DSA_OK:
        raise DsaError(status, where)


from ._api import (  # noqa: E402  (needs `lib` above)
    DeviceInputs, Plan, indexer_topk, sparse_attn, fused_decode, read_device_error,
    clear_device_error, workspace_size, alloc_workspace, quantize_mxfp8, index_cache_append_mxfp8,
    index_cache_append, latent_cache_append)

__all__ = ["lib", "DsaError", "DeviceInputs", "Plan", "indexer_topk", "sparse_attn", "fused_decode",
           "read_device_error", "clear_device_error", "workspace_size", "alloc_workspace", "Trace",
           "quantize_mxfp8", "index_cache_append_mxfp8", "index_cache_append", "latent_cache_append"]
