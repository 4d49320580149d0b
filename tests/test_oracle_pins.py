"""The CPU oracle against what the pages and the mathematics fix (no GPU)."""
import pytest

import oracle
import workloads as wl
from tests import pins

ALL_FMTS = [wl.MLX_AFFINE4_G64, wl.MXFP4, wl.NVFP4, wl.Q6K, wl.Q5_0, wl.Q5_1, wl.Q5_K]


def test_e2m1_table_is_the_page_set():
    pins.check_e2m1(oracle)


def test_e8m0_matches_library_decoder():
    pins.check_e8m0(oracle)


def test_e4m3_matches_library_decoder():
    pins.check_e4m3(oracle)


def test_bf16_rounding_once():
    pins.check_bf16_rounding(oracle)


def test_bits_per_weight_and_q6k_output_layer_bytes():
    pins.check_bpw(oracle)


def test_q6k_half_operand_identity():
    pins.check_q6k_operand(oracle)


def test_q5_half_operand_identity():
    pins.check_q5_operand(oracle)


def test_q6k_old_seed_identity():
    pins.check_q6k_old_seed()


@pytest.mark.parametrize("fmt", ALL_FMTS)
def test_dequant_is_one_rounding_of_exact_value(fmt):
    pins.check_dequant_exact(oracle, fmt)


@pytest.mark.parametrize("fmt", ALL_FMTS)
@pytest.mark.parametrize("m", [1, 4])
def test_gemv_brute_force_exact_rational(fmt, m):
    pins.check_gemv_brute_force(oracle, fmt, m, residual=(m == 4))


@pytest.mark.parametrize("fmt", ALL_FMTS)
def test_unit_scales_reduce_to_dense_matmul(fmt):
    pins.check_dense_special_case(oracle, fmt)


def test_route_brute_force_and_invariance():
    pins.check_route_brute_force(oracle)


def test_route_statistics_match_page():
    pins.check_route_statistics(oracle)


def test_silu():
    pins.check_silu(oracle)


def test_sigmoid():
    pins.check_sigmoid(oracle)


def test_moe_shared_gate():
    pins.check_moe_shared_gate(oracle)


def test_moe_chain_composition():
    pins.check_moe_composition(oracle)


@pytest.mark.parametrize("fmt", ALL_FMTS)
def test_bf16_operand(fmt):
    pins.check_operand_bf16(oracle, fmt)


def test_tolerance_output_ulp():
    pins.check_tolerance_output_ulp(oracle)


def test_e2m1_encode_closed_form():
    pins.check_e2m1_encode(oracle)


def test_e4m3_encode_matches_library():
    pins.check_e4m3_encode(oracle)


def test_act_quant_round_trip():
    pins.check_act_quant_round_trip(oracle)


def test_act_quant_nearest_grid_points():
    pins.check_act_quant_nearest(oracle)


def test_w4a4_reduces_to_w4a16():
    pins.check_w4a4_reduces_to_w4a16(oracle)


def test_w4a4_brute_force_exact_rational():
    pins.check_w4a4_brute_force(oracle)


def test_tolerance_base_term_and_row_norms():
    pins.check_tolerance_base(oracle)
