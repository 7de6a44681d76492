"""Copies a seeded workload's host arrays to the GPU as the library's DeviceInputs.

Only moves bytes: no arithmetic of the method happens here.
"""
from __future__ import annotations

import numpy as np
import torch


def _dev(a, device, dtype=None):
    if a is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to(device, non_blocking=False)


def to_device(wl, device="cuda", with_latent=True):
    from sparse_attention_decode_dsa_gb300 import DeviceInputs
    decode = wl.spec.mode == "decode"
    fp8kv = with_latent and wl.kv_codes is not None
    bf = torch.bfloat16
    kbits = torch.bfloat16 if wl.idx_k.dtype == np.uint16 else torch.uint8
    qs = wl.idx_q_scale
    ks = wl.idx_k_scale
    return DeviceInputs(
        block_table=_dev(wl.block_table, device),
        seq_lens=_dev(wl.seq_lens, device),
        seq_lens_host=torch.from_numpy(np.ascontiguousarray(wl.seq_lens, dtype=np.int32)),
        num_pages=int(wl.num_pages),
        idx_q=_dev(wl.idx_q.view(np.int16) if wl.idx_q.dtype == np.uint16 else wl.idx_q, device,
                   kbits if kbits is torch.bfloat16 else None),
        head_w=_dev(wl.head_w, device),
        idx_k=_dev(wl.idx_k.view(np.int16) if wl.idx_k.dtype == np.uint16 else wl.idx_k, device,
                   kbits if kbits is torch.bfloat16 else None),
        top_k=int(wl.spec.topk),
        idx_q_scale=_dev(qs, device),
        idx_k_scale=_dev(ks, device),
        kv=_dev(wl.kv.view(np.int16), device, bf) if (with_latent and wl.kv is not None) else None,
        kv_codes=_dev(wl.kv_codes, device) if fp8kv else None,
        kv_scale=_dev(wl.kv_scale, device) if fp8kv else None,
        kv_rope=_dev(wl.kv_rope.view(np.int16), device, bf) if fp8kv else None,
        sfa_q=_dev(wl.sfa_q.view(np.int16), device, bf) if (with_latent and wl.sfa_q is not None) else None,
        softmax_scale=float(wl.spec.softmax_scale),
        token_seq=None if decode else _dev(wl.q_seq, device),
        token_pos=None if decode else _dev(wl.q_pos, device),
        token_seq_host=None if decode else torch.from_numpy(np.ascontiguousarray(wl.q_seq, dtype=np.int32)),
        token_pos_host=None if decode else torch.from_numpy(np.ascontiguousarray(wl.q_pos, dtype=np.int32)),
    )
