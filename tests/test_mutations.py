"""Mutation tests: each planted mistake in the oracle must fail at least one pin.

The mistakes are compiled into throw-away copies of the oracle (CPU only); the
pins of tests/test_oracle.py then run against each copy.  Mutant 1 is the
clamped group index min(h / heads_per_group, 1) that vllm.cpp #1362 uses as its
own mutation; mutant 3 is the dropped chunk carry; the others are a reversed
conv tap order, y read from the pre-update state, a dropped dt bias and a
flipped decay sign in the chunk form; mutants 7-9 are in the gated group
RMSNorm: one norm over the whole row, eps outside the square root, and the
gate applied before the norm.  Mutants 10-12 are in the chunk form's clamp
(TensorRT-Model-Connect #2207 "Implementation": gamma_S is the last element
of the cumulative sum, not a separate reduction, and every exponent is
clamped at 0): no clamp at all, gamma_L from a separate fp32 reduction with
its state exponent unclamped, and gamma_t, gamma_s clamped one by one.
Mutant 13 chains two segments' states without the second segment's decay.
"""
import pytest

import oracle
from tests import test_oracle as pins

PINS = [
    pins.test_single_step_hand_values,
    pins.test_softplus_and_bias_hand_values,
    pins.test_three_step_unrolled_sum,
    pins.test_dt_zero_leaves_state_unchanged,
    pins.test_zero_input_is_geometric_decay,
    pins.test_A_zero_is_prefix_sum,
    lambda: pins.test_chunked_equals_sequential([7, 4], True),
    lambda: pins.test_chunked_equals_sequential([3, 1, 5, 2], False),
    pins.test_group_mapping_equals_expanded_groups,
    pins.test_conv_matches_numpy_correlate,
    pins.test_conv_impulse_returns_reversed_taps,
    pins.test_linearity_in_x_and_h0,
    pins.test_decode_steps_equal_sequential_rows,
    pins.test_rmsnorm_constant_group_hand_value,
    pins.test_rmsnorm_groups_are_independent,
    pins.test_rmsnorm_gate_acts_after_the_norm,
    pins.test_chunk_form_clamp_hand_values,
    pins.test_chunk_form_clamp_carries_across_chunks,
    lambda: pins.test_huge_decay_limit("chunked"),
    pins.test_state_combine_hand_values,
    lambda: pins.test_segments_chained_by_combine_equal_one_call([3, 8]),
]


@pytest.mark.parametrize("mutant", [1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13])
def test_pins_catch_mutant(mutant, tmp_path, monkeypatch):
    lib = oracle.open_library(oracle.build(out_path=str(tmp_path / f"m{mutant}.so"),
                                           mutant=mutant))
    monkeypatch.setattr(oracle, "_lib", lib)
    failed = 0
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed >= 1, f"mutant {mutant} passed every pin"


def test_unmutated_copy_passes_every_pin(tmp_path, monkeypatch):
    lib = oracle.open_library(oracle.build(out_path=str(tmp_path / "m0.so"), force=True))
    monkeypatch.setattr(oracle, "_lib", lib)
    for pin in PINS:
        pin()
