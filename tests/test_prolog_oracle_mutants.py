"""Plant plausible mistakes in the index-prolog oracle (MXFP8 quantisation, cache append)
on the CPU and check that one of its pins catches each."""
import numpy as np
import pytest

from oracle import mx_quant as M
from tests import test_prolog_oracle as P

_orig = {name: getattr(M, name) for name in ["e4m3_round", "group_exponent", "quantize_mxfp8", "append_rows"]}


def _exp_emax7(amax):
    return np.where(np.asarray(amax) > 0, np.clip(_orig["group_exponent"](amax) + 1, -127, 127), -127)


def _exp_ceil(amax):
    amax = np.asarray(amax, dtype=np.float64)
    with np.errstate(divide="ignore"):
        c = np.ceil(np.log2(np.where(amax > 0, amax, 1.0))).astype(np.int64)
    return np.where(amax > 0, np.clip(c - 8, -127, 127), -127)


def _round_ties_away(v):
    v = np.asarray(v, dtype=np.float64)
    c = _orig["e4m3_round"](v)
    # move every exact tie to the code away from zero
    a = np.minimum(np.abs(v), 448.0)
    lo = M.decode_e4m3((c & 0x7F).astype(np.uint8))
    step_up = M.decode_e4m3(np.minimum((c & 0x7F) + 1, 0x7E).astype(np.uint8))
    tie = np.isclose(a - lo, step_up - a, rtol=0, atol=0) & (a > lo)
    return np.where(tie, (c & 0x80) | np.minimum((c & 0x7F) + 1, 0x7E), c).astype(np.uint8)


def _round_no_saturation(v):
    v = np.asarray(v, dtype=np.float64)
    c = _orig["e4m3_round"](v)
    return np.where(np.abs(v) > 464, (c & 0x80) | 0x7F, c).astype(np.uint8)  # overflow to NaN


def _round_sign_dropped(v):
    return (_orig["e4m3_round"](v) & 0x7F).astype(np.uint8)


def _quant_bias126(x):
    c, s = _orig["quantize_mxfp8"](x)
    return c, (s.astype(np.int64) - 1).clip(0, 255).astype(np.uint8)


def _append_slot_page_swapped(cc, cs, bt, seq, pos, codes, scales):
    return _orig["append_rows"](cc, cs, bt, seq, pos % 64 * 64 + pos // 64, codes, scales)


MUTANTS = {
    "mx: element exponent 7 (largest normal 240)": ("group_exponent", _exp_emax7),
    "mx: ceil instead of floor of log2(amax)": ("group_exponent", _exp_ceil),
    "e4m3: ties away from zero": ("e4m3_round", _round_ties_away),
    "e4m3: no saturation (overflow to NaN)": ("e4m3_round", _round_no_saturation),
    "e4m3: sign dropped": ("e4m3_round", _round_sign_dropped),
    "e8m0: scale byte bias 126": ("quantize_mxfp8", _quant_bias126),
    "append: slot and page swapped": ("append_rows", _append_slot_page_swapped),
}

PINS = [
    P.test_every_finite_code_rounds_to_itself,
    lambda: P.test_rounding_closed_forms(1.0625, 0x38),
    lambda: P.test_rounding_closed_forms(3 * 2.0 ** -10, 0x02),
    lambda: P.test_rounding_closed_forms(449.0, 0x7E),
    lambda: P.test_group_exponent_closed_forms(1.0, -8),
    lambda: P.test_group_exponent_closed_forms(511.0, 0),
    P.test_exact_groups_round_trip,
    P.test_quantisation_error_within_half_step,
    P.test_append_places_rows_by_page_translation,
]


@pytest.mark.parametrize("label", sorted(MUTANTS))
def test_prolog_oracle_mutants(label, monkeypatch):
    name, fn = MUTANTS[label]
    monkeypatch.setattr(M, name, fn)
    caught = []
    for pin in PINS:
        try:
            pin()
        except Exception as e:  # an assertion or a shape error both expose the mutant
            caught.append(type(e).__name__)
            break
    assert caught, f"no pin caught the mutant '{label}'"


def test_pins_pass_on_the_unmutated_oracle():
    for pin in PINS:
        pin()
