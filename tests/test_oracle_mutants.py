"""The oracle's pins are sensitive: each plausible mistake, planted in a copy of the oracle
source and compiled on the CPU, must make at least one pin fail.

Mutations only change arithmetic or in-bounds indexing (no out-of-range access).
An unmodified copy compiled the same way must pass every pin (control).
"""
import numpy as np
import pytest

import _pins
import oracle

PINS = [
    ("closed_forms", _pins.pin_closed_forms),
    ("bf16_bits", _pins.pin_bf16_bits_exact),
    ("zero_rows", _pins.pin_zero_rows),
    ("saturation", _pins.pin_saturation_limits),
    ("small_argument", _pins.pin_small_argument_expansion),
    ("symmetries", _pins.pin_symmetries),
    ("swiglu_limit", _pins.pin_swiglu_limit),
    ("fd_4_25", lambda o: _pins.pin_finite_differences(o, 4.0, 25.0)),
    ("fd_2_5", lambda o: _pins.pin_finite_differences(o, 2.0, 5.0)),
    ("tiny_expert", _pins.pin_tiny_expert_router_rewrite),
    ("autograd", lambda o: _pins.pin_autograd_of_definition(o, 4.0, 25.0)),
    ("bf16_vs_f64", _pins.pin_bf16_entry_matches_f64_entry),
    ("extreme", _pins.pin_extreme_finite_inputs),
    ("e4m3_codec", _pins.pin_e4m3_codec),
    ("fp8_blocks", _pins.pin_fp8_block_quantization),
    ("fp8_bwd", _pins.pin_fp8_backward_is_backward_of_dequantized),
    ("round_bf16", _pins.pin_round_bf16),
    ("gateup", _pins.pin_grouped_gateup),
    ("adam_torch", _pins.pin_adam_matches_torch),
    ("adam_first_step", _pins.pin_adam_first_step_closed_form),
    ("adam_stored", _pins.pin_adam_stored_is_a_rounding_of_f64),
]

MUTANTS = {
    "drop_second_term_of_Gprime": ("double Gp = (1.0 - T * T) * S + beta * T * S * (1.0 - S);",
                                   "double Gp = (1.0 - T * T) * S;"),
    "wrong_sign_in_Gprime": ("(1.0 - T * T) * S + beta * T * S * (1.0 - S)",
                             "(1.0 - T * T) * S - beta * T * S * (1.0 - S)"),
    "sigmoid_negative_branch": ("return e / (1.0 + e);", "return 1.0 / (1.0 + e);"),
    "sigmoid_positive_sign": ("return 1.0 / (1.0 + exp(-u));", "return 1.0 / (1.0 + exp(u));"),
    "gate_linear_swapped": ("oracle_situ_point(xr[j], xr[H + j],", "oracle_situ_point(xr[H + j], xr[j],"),
    "p_folded_into_dp": ("acc += gr[j] * a;", "acc += p * gr[j] * a;"),
    "dx_without_p": ("dxr[j] = p * gr[j] * L * Gp;", "dxr[j] = gr[j] * L * Gp;"),
    "dgate_dlinear_swapped": ("dxr[j] = p * gr[j] * L * Gp;\n        dxr[H + j] = p * gr[j] * G * Lp;",
                              "dxr[j] = p * gr[j] * G * Lp;\n        dxr[H + j] = p * gr[j] * L * Gp;"),
    "Lprime_not_squared": ("double Lp = 1.0 - W * W;", "double Lp = 1.0 - W;"),
    "gate_missing_beta": ("double G = beta * T * S;", "double G = T * S;"),
    "tanh_argument_inverted": ("double T = tanh(u / beta);", "double T = tanh(u * beta);"),
    "linear_missing_lbeta": ("double L = lbeta * W;", "double L = W;"),
    "linear_uses_beta": ("double W = tanh(v / lbeta);", "double W = tanh(v / beta);"),
    "dp_abs_not_absolute": ("acc_abs += fabs(gr[j] * a);", "acc_abs += gr[j] * a;"),
    "bf16_shift_wrong": ("((uint32_t)bits) << 16;", "((uint32_t)bits) << 15;"),
    "bf16_row_stride_wrong": ("(const uint16_t*)jb->x + r * 2 * H;", "(const uint16_t*)jb->x + r * H;"),
    "bf16_p_index_wrong": ("p = (double)((const float*)jb->p)[r];", "p = (double)((const float*)jb->p)[0];"),
    "g_row_off_by_one": ("gr = (const double*)jb->g + r * H;",
                         "gr = (const double*)jb->g + (r > 0 ? r - 1 : 0) * H;"),
    # block-wise FP8 saved x
    "e4m3_ties_not_to_even": ("if (d_hi < d_lo || (d_hi == d_lo && (c & 1))) c = c + 1;",
                              "if (d_hi <= d_lo) c = c + 1;"),
    "e4m3_overflow_to_nan": ("if (a >= 448.0f) return sign | 0x7E;", "if (a >= 448.0f) return sign | 0x7F;"),
    "e4m3_subnormal_scale": ("if (e == 0) return ldexpf((float)m, -9);", "if (e == 0) return ldexpf((float)m, -10);"),
    "e4m3_bias": ("return ldexpf((float)(8 + m), e - 10);", "return ldexpf((float)(8 + m), e - 9);"),
    "fp8_scale_divisor": ("s[bi] = amax / 448.0f;", "s[bi] = amax / 256.0f;"),
    "fp8_no_amax_floor": ("if (amax < floor_amax) amax = floor_amax;", "(void)floor_amax;"),
    "fp8_linear_scales_overwrite_gate": ("s + r * 2 * nb + nb, block);", "s + r * 2 * nb, block);"),
    "fp8_dequant_ignores_half": ("float sc = s[r * 2 * nb + half * nb + j / block];",
                                 "float sc = s[r * 2 * nb + j / block];"),
    # bf16 rounding of the gate/up projection
    "bf16_ties_away": ("if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0)) n = fl + 1.0;",
                       "if (rem >= 0.5) n = fl + 1.0;"),
    "bf16_truncates": ("if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0)) n = fl + 1.0;", "(void)rem;"),
    "bf16_seven_bits": ("    double ulp = ldexp(1.0, ex - 7);\n    double q = a / ulp;",
                        "    double ulp = ldexp(1.0, ex - 6);\n    double q = a / ulp;"),
    "bf16_no_subnormal_clamp": ("    if (ex < -126) ex = -126;\n    double ulp = ldexp(1.0, ex - 7);\n    double q = a / ulp;",
                                "    double ulp = ldexp(1.0, ex - 7);\n    double q = a / ulp;"),
    "bf16_overflow_at_max": ("uint16_t b = r > ldexp(255.0, 120) ? 0x7F80", "uint16_t b = r >= ldexp(255.0, 120) ? 0x7F80"),
    "bf16_sign_dropped": ("return (uint16_t)((signbit(v) ? 0x8000 : 0) | b);", "return b;"),
    # Adam on host-resident state
    "adam_f64_no_bc2": ("const double denom = sqrt(v[i]) / sqrt(bc2) + hp->eps;",
                        "const double denom = sqrt(v[i]) + hp->eps;"),
    "adam_f64_ascent": ("w[i] = w[i] - (hp->lr / bc1) * m[i] / denom;", "w[i] = w[i] + (hp->lr / bc1) * m[i] / denom;"),
    "adam_f64_coupled_decay": ("if (hp->weight_decay > 0.0) w[i] = w[i] * (1.0 - hp->lr * hp->weight_decay);",
                               "if (hp->weight_decay > 0.0) w[i] = w[i] * (1.0 - hp->weight_decay);"),
    "adam_no_bc1": ("const float s = (float)(hp->lr / bc1);", "const float s = (float)(hp->lr);"),
    "adam_no_sqrt": ("t = sqrtf(v1); float sq = t;", "t = v1; float sq = t;"),
    "adam_eps_inside_sqrt": ("        t = sqrtf(v1); float sq = t;\n        t = sq * r; float qa = t;\n        t = qa + eps; float q = t;",
                             "        t = sqrtf(v1 + eps); float sq = t;\n        t = sq * r; float qa = t;\n        t = qa; float q = t;"),
    "adam_betas_swapped": ("t = b1 * bf16_bits_to_float(m[i]); float ma = t;", "t = b2 * bf16_bits_to_float(m[i]); float ma = t;"),
    "adam_g_not_squared": ("t = gb * gb; float gg = t;", "t = gb; float gg = t;"),
    "adam_decay_ignored": ("if (decay) { t = w1 * d; w1 = t; }", "(void)d;"),
    "adam_working_weight_stale": ("w_out[i] = oracle_round_bf16((double)w2);", "w_out[i] = oracle_round_bf16((double)w1);"),
    "adam_m_without_gradient": ("m[i] = oracle_round_bf16((double)m1);", "m[i] = oracle_round_bf16((double)ma);"),
}


def failing_pins(o):
    failed = []
    with np.errstate(all="ignore"):
        for name, pin in PINS:
            try:
                pin(o)
            except AssertionError:
                failed.append(name)
    return failed


def test_unmodified_copy_passes_every_pin(tmp_path):
    o = oracle.compile_variant(oracle.source_text(), str(tmp_path / "control.so"))
    assert failing_pins(o) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    find, repl = MUTANTS[name]
    text = oracle.source_text()
    assert find in text, f"mutation anchor not found: {name}"
    o = oracle.compile_variant(text.replace(find, repl), str(tmp_path / f"{name}.so"))
    failed = failing_pins(o)
    assert failed, f"no pin catches the planted mistake {name}"


# ---------------------------------------------------------------- the oracle's numpy parts
# The expert-grouped projections are numpy code (an fp64 matmul per expert): planted mistakes
# there replace one oracle function with a wrong one and must trip the GEMM pins.

class Shim:
    """The oracle module with some of its functions replaced."""

    def __init__(self, **over):
        self.__dict__.update(over)

    def __getattr__(self, name):
        return getattr(oracle, name)


def _bits_f64(b):
    return (np.asarray(b).view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _gateup_fwd_from(grouped, rounding="rne", out_from="rounded"):
    def gateup_fwd(h, w, off, beta=4.0, lbeta=25.0, nthreads=0):
        x, mag = grouped(h, w, off)
        if rounding == "rne":
            xb = oracle.round_bf16_array(x)
        else:                                   # truncation toward zero
            xb = (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        src = xb if out_from == "rounded" else None
        out = oracle.fwd_bf16(src, beta, lbeta) if src is not None else oracle.fwd_f64(x, beta, lbeta)
        return x, xb, out, mag
    return gateup_fwd


def _swap_halves(grouped):
    def f(h, w, off):
        x, mag = grouped(h, w, off)
        H = x.shape[1] // 2
        idx = np.r_[H:2 * H, 0:H]
        return x[:, idx], mag[:, idx]
    return f


def _next_expert_weights_gateup(h, w, off):
    return oracle.grouped_gateup(h, np.roll(np.asarray(w), -1, axis=0), off)


def _dp_times_p(x, dy, wt, off, p, *a, **k):
    dx, dp, dpa = oracle.dgrad_bwd_router(x, dy, wt, off, p, *a, **k)
    return dx, dp * np.asarray(p, dtype=np.float64), dpa


def _dgrad_without_p_in_dx(x, dy, wt, off, p, *a, **k):
    return oracle.dgrad_bwd_router(x, dy, wt, off, np.ones_like(np.asarray(p)), *a, **k)


NUMPY_MUTANTS = {
    "dgrad_next_expert_weights": ("dgrad", lambda: Shim(
        grouped_dgrad=lambda dy, wt, off: oracle.grouped_dgrad(dy, np.roll(np.asarray(wt), -1, axis=0), off))),
    "dgrad_rows_shifted": ("dgrad", lambda: Shim(
        grouped_dgrad=lambda dy, wt, off: np.roll(oracle.grouped_dgrad(dy, wt, off), 1, axis=0))),
    "dgrad_weights_not_transposed": ("dgrad", lambda: Shim(
        grouped_dgrad=lambda dy, wt, off: oracle.grouped_dgrad(
            dy, np.ascontiguousarray(np.asarray(wt).reshape(wt.shape[0], -1)[:, :wt.shape[1] * wt.shape[2]]
                                     .reshape(wt.shape[0], wt.shape[2], wt.shape[1]).transpose(0, 2, 1)), off))),
    "dgrad_dp_times_p": ("dgrad", lambda: Shim(dgrad_bwd_router=_dp_times_p)),
    "dgrad_router_weight_ignored": ("dgrad", lambda: Shim(dgrad_bwd_router=_dgrad_without_p_in_dx)),
    "gateup_halves_swapped": ("gateup", lambda: Shim(
        grouped_gateup=_swap_halves(oracle.grouped_gateup),
        gateup_fwd=_gateup_fwd_from(_swap_halves(oracle.grouped_gateup)))),
    "gateup_next_expert_weights": ("gateup", lambda: Shim(
        grouped_gateup=_next_expert_weights_gateup, gateup_fwd=_gateup_fwd_from(_next_expert_weights_gateup))),
    "gateup_truncating_rounding": ("gateup", lambda: Shim(
        gateup_fwd=_gateup_fwd_from(oracle.grouped_gateup, rounding="trunc"))),
    "gateup_out_from_unrounded_x": ("gateup", lambda: Shim(
        gateup_fwd=_gateup_fwd_from(oracle.grouped_gateup, out_from="exact"))),
}

GEMM_PINS = {"dgrad": _pins.pin_grouped_dgrad, "gateup": _pins.pin_grouped_gateup}


def test_numpy_control_passes():
    for pin in GEMM_PINS.values():
        pin(Shim())
    _pins.pin_grouped_gateup(Shim(gateup_fwd=_gateup_fwd_from(oracle.grouped_gateup)))


@pytest.mark.parametrize("name", sorted(NUMPY_MUTANTS))
def test_planted_mistake_in_numpy_part_is_caught(name):
    which, make = NUMPY_MUTANTS[name]
    with np.errstate(all="ignore"), pytest.raises((AssertionError, ValueError)):
        GEMM_PINS[which](make())
