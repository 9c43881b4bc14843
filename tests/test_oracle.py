"""The CPU oracle against its pins: the pages' printed figures, closed forms,
library routines, brute force on tiny inputs and invariants."""
import pytest

from oracle import nvfp4_moe as O
from tests import oracle_pins as P

PINS = [
    P.check_e2m1_decode, P.check_e2m1_ties, P.check_e2m1_brute_force,
    P.check_e4m3_decode_library, P.check_e4m3_brute_force, P.check_e4m3_library_cast,
    P.check_e4m3_saturation, P.check_bf16_rounding,
    P.check_sf_layout_points, P.check_sf_layout_structure, P.check_fused_swizzle,
    P.check_quantize_block_hand, P.check_pack_order, P.check_quantize_error_bound,
    P.check_grouping_brute, P.check_gather, P.check_gemm_brute_force, P.check_gemm_invariants,
    P.check_swiglu_closed_form, P.check_scatter_hand, P.check_layer_batch_invariance,
    P.check_unused_slots, P.check_gemv_w4a16_lossless, P.check_gemv_w4a16_brute_force, P.check_layer_w4a16,
]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(O)


def test_e4m3_fold_figures(pages):
    P.check_e4m3_fold_figures(O, pages)


def test_quantize_bytes(pages):
    P.check_quantize_bytes(O, pages)


def test_sizes(pages):
    P.check_sizes(pages)
