"""Plant plausible mistakes in the oracle (on the CPU) and check that a pin catches each.

A pin set that no mutant can slip past is what makes the oracle trustworthy without
another implementation to compare with.  Each mutant replaces one oracle function by a
subtly wrong copy; the pins from ``test_oracle_pins`` run against it and at least one
must fail.
"""
import numpy as np
import pytest

import dsa_workloads as W
from oracle import dsa_oracle as O
from tests import test_oracle_pins as P

_orig = {name: getattr(O, name) for name in
         ["index_scores", "topk_select", "sparse_attention", "visible_count",
          "dequant_index_keys", "dequant_index_query", "logical_rows", "decode_e4m3",
          "decode_e8m0", "decode_bf16", "decode_latent_fp8"]}


def _scores_no_weights(q, w, k, act="identity"):
    return _orig["index_scores"](q, np.ones_like(w), k, act)


def _scores_reversed_weights(q, w, k, act="identity"):
    return _orig["index_scores"](q, w[::-1].copy(), k, act)


def _scores_max_over_heads(q, w, k, act="identity"):
    return ((k @ q.T) * w[None, :]).max(axis=1)


def _topk_high_index_wins(scores, k):
    n = scores.shape[0]
    order = np.lexsort((-np.arange(n), -scores))
    out = np.full(k, -1, np.int32)
    ch = np.sort(order[:min(k, n)])
    out[:ch.shape[0]] = ch
    return out


def _topk_score_order(scores, k):
    n = scores.shape[0]
    order = np.lexsort((np.arange(n), -scores))[:min(k, n)]
    out = np.full(k, -1, np.int32)
    out[:order.shape[0]] = order
    return out


def _topk_smallest(scores, k):
    return _orig["topk_select"](-scores, k)


def _attn_tail_values(q, rows, scale, v_dim=512):
    if rows.shape[0] == 0:
        return np.zeros((q.shape[0], v_dim))
    z = scale * (q @ rows.T)
    p = np.exp(z - z.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    return p @ rows[:, rows.shape[1] - v_dim:]


def _attn_no_scale(q, rows, scale, v_dim=512):
    return _orig["sparse_attention"](q, rows, 1.0, v_dim)


def _attn_rope_dropped(q, rows, scale, v_dim=512):
    return _orig["sparse_attention"](q[:, :v_dim], rows[:, :v_dim], scale, v_dim)


def _visible_excludes_self(wl, token):
    return max(0, _orig["visible_count"](wl, token) - 1)


def _keys_no_scale(wl, b, positions):
    k = _orig["logical_rows"](wl.idx_k, wl.block_table[b], positions)
    return O.decode_bf16(k) if k.dtype == np.uint16 else O.decode_e4m3(k)


def _query_no_scale(wl, token):
    q = wl.idx_q[token]
    return O.decode_bf16(q) if q.dtype == np.uint16 else O.decode_e4m3(q)


def _logical_rows_swapped(cache, bt_row, positions):
    positions = np.asarray(positions, dtype=np.int64)
    return cache[bt_row[positions % 64 % bt_row.shape[0]], positions // 64 % 64]


def _logical_rows_unpaged(cache, bt_row, positions):
    positions = np.asarray(positions, dtype=np.int64)
    return cache[positions // 64, positions % 64]


def _e4m3_bias8(bits):
    return _orig["decode_e4m3"](bits) / 2.0


def _e8m0_bias126(bits):
    return _orig["decode_e8m0"](bits) * 2.0


def _latent_fp8_tile64(codes, scales, rope_bits):
    sc = np.asarray(scales, dtype=np.float64)
    lat = O.decode_e4m3(codes) * np.repeat(np.concatenate([sc, sc], axis=-1), 64, axis=-1)
    return np.concatenate([lat, O.decode_bf16(rope_bits)], axis=-1)


def _latent_fp8_no_scale(codes, scales, rope_bits):
    return _orig["decode_latent_fp8"](codes, np.ones_like(scales), rope_bits)


MUTANTS = {
    "scores: head weights dropped": ("index_scores", _scores_no_weights),
    "scores: head weights misaligned": ("index_scores", _scores_reversed_weights),
    "scores: max instead of head sum": ("index_scores", _scores_max_over_heads),
    "topk: ties to the higher position": ("topk_select", _topk_high_index_wins),
    "topk: output in score order": ("topk_select", _topk_score_order),
    "topk: smallest instead of largest": ("topk_select", _topk_smallest),
    "sfa: value = last 512 dims": ("sparse_attention", _attn_tail_values),
    "sfa: softmax scale dropped": ("sparse_attention", _attn_no_scale),
    "sfa: rope dims dropped from the logits": ("sparse_attention", _attn_rope_dropped),
    "causality: query position excluded": ("visible_count", _visible_excludes_self),
    "dequant: key scale dropped": ("dequant_index_keys", _keys_no_scale),
    "dequant: query scale dropped": ("dequant_index_query", _query_no_scale),
    "paging: page and slot swapped": ("logical_rows", _logical_rows_swapped),
    "paging: page table ignored": ("logical_rows", _logical_rows_unpaged),
    "e4m3: exponent bias 8": ("decode_e4m3", _e4m3_bias8),
    "e8m0: exponent bias 126": ("decode_e8m0", _e8m0_bias126),
    "fp8 latent: tiles of 64 elements": ("decode_latent_fp8", _latent_fp8_tile64),
    "fp8 latent: tile scale dropped": ("decode_latent_fp8", _latent_fp8_no_scale),
}

PINS = [
    P.test_decode_e4m3_all_codes,
    P.test_decode_e8m0,
    P.test_golden_indexer_example,
    P.test_golden_sfa_example,
    P.test_topk_brute_force_rank,
    lambda: P.test_scores_equal_collapsed_integer_form(W.SMALL_DECODE_MX),
    P.test_fp8_scores_are_scaled_integer_scores,
    P.test_mx_scores_group_by_group,
    lambda: P.test_selection_invariants(W.SMALL_PREFILL),
    lambda: P.test_paged_equals_contiguous(W.SMALL_H8),
    P.test_sfa_with_k_at_least_l_is_dense_causal_attention,
    P.test_prefill_row0_attends_to_key0_only,
    P.test_fp8_latent_decode_closed_form,
]


@pytest.mark.parametrize("label", sorted(MUTANTS))
def test_oracle_mutants(label, monkeypatch):
    name, fn = MUTANTS[label]
    monkeypatch.setattr(O, name, fn)
    caught = []
    for pin in PINS:
        try:
            pin()
        except Exception as e:  # an assertion or a shape error both expose the mutant
            caught.append(type(e).__name__)
            break
    assert caught, f"no pin caught the mutant '{label}'"
