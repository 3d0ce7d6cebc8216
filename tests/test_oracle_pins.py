"""Pins of the fp64 oracle against what the pages and the mathematics fix.

The bodies live in tests/_pins.py so the same checks can also be run against
deliberately broken copies of the oracle (tests/test_oracle_mutants.py).

* closed forms at points where tanh and sigmoid are rational (tests/golden/closed_forms.txt);
* limits, symmetries and the small-argument expansion of the definition;
* the SwiGLU limit (beta, lbeta -> infinity), a textbook special case;
* central finite differences of  Λ(x, p) = Σ_r p_r Σ_j g_rj a_rj(x)  for every dx and dp;
* a brute-force tiny expert  y = Σ_e p_e W_e a_e(x_e)  for the router-gradient rewrite;
* the definition run under PyTorch autograd in float64 (an independent derivative).

Definition: "Frontier-scale RL with Kimi K3", section "Streaming activations".
Router rewrite: "Kimi K3 模型结构（9）：显存", section "MoE 反向：推一下为什么可以不存 expert 输出".
"""
import pytest

import _pins
import oracle


@pytest.mark.parametrize("row", _pins.closed_form_rows(), ids=lambda r: r[0])
def test_closed_forms(row):
    _pins._pin_closed_form_row(oracle, row)


def test_bf16_bits_exact():
    _pins.pin_bf16_bits_exact(oracle)


def test_zero_rows():
    _pins.pin_zero_rows(oracle)


def test_saturation_limits():
    _pins.pin_saturation_limits(oracle)


def test_small_argument_expansion():
    _pins.pin_small_argument_expansion(oracle)


def test_symmetries():
    _pins.pin_symmetries(oracle)


def test_swiglu_limit():
    _pins.pin_swiglu_limit(oracle)


@pytest.mark.parametrize("beta,lbeta", [(4.0, 25.0), (2.0, 5.0)])
def test_finite_differences_every_output(beta, lbeta):
    _pins.pin_finite_differences(oracle, beta, lbeta)


def test_tiny_expert_router_rewrite():
    _pins.pin_tiny_expert_router_rewrite(oracle)


@pytest.mark.parametrize("beta,lbeta", [(4.0, 25.0), (3.0, 11.0)])
def test_autograd_of_definition(beta, lbeta):
    _pins.pin_autograd_of_definition(oracle, beta, lbeta)


def test_bf16_entry_matches_f64_entry():
    _pins.pin_bf16_entry_matches_f64_entry(oracle)


def test_thread_count_independent():
    _pins.pin_thread_count_independent(oracle)


def test_extreme_finite_inputs_give_finite_outputs():
    _pins.pin_extreme_finite_inputs(oracle)


def test_empty_rows_ok():
    _pins.pin_empty_rows(oracle)


def test_e4m3_codec():
    _pins.pin_e4m3_codec(oracle)


def test_fp8_block_quantization():
    _pins.pin_fp8_block_quantization(oracle)


def test_fp8_backward_is_backward_of_dequantized():
    _pins.pin_fp8_backward_is_backward_of_dequantized(oracle)


def test_grouped_dgrad():
    _pins.pin_grouped_dgrad(oracle)


def test_round_bf16():
    _pins.pin_round_bf16(oracle)


def test_grouped_gateup():
    _pins.pin_grouped_gateup(oracle)


def test_adam_matches_torch():
    _pins.pin_adam_matches_torch(oracle)


def test_adam_first_step_closed_form():
    _pins.pin_adam_first_step_closed_form(oracle)


def test_adam_stored_is_a_rounding_of_f64():
    _pins.pin_adam_stored_is_a_rounding_of_f64(oracle)
