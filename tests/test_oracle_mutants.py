"""The oracle's pins have teeth: each planted mistake fails at least one pin.

Every mutant below is a copy of gdn_oracle.c with one plausible slip (a
dropped term, a wrong sign, a swapped index or operand), compiled into a
temporary library on the CPU.  The battery of pin tests from
test_oracle_pins.py and test_oracle_layer.py runs against it, and at least
one of them must fail.  All mutants keep every memory access in bounds.
"""
import os
import subprocess

import pytest

import oracle
import test_oracle_layer as L
import test_oracle_pins as P
import test_oracle_proj as J

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.c")

MUTANTS = {
    "conv taps reversed": ("acc += w[(long)c * W + j] *", "acc += w[(long)c * W + (W - 1 - j)] *"),
    "conv state rows reversed": ("return state[(long)(W - 1 + tau) * n_ch + c];",
                                 "return state[(long)(-1 - tau) * n_ch + c];"),
    "softplus sign": ("log1p(exp(-fabs(x)))", "log1p(exp(-x))"),
    "decay sign": ("*g = -exp(A_log) * or_softplus(a + dt_bias);",
                   "*g = exp(A_log) * or_softplus(a + dt_bias);"),
    "dt_bias dropped": ("or_softplus(a + dt_bias)", "or_softplus(a)"),
    "A_log not exponentiated": ("*g = -exp(A_log) *", "*g = -A_log *"),
    "sigmoid sign": ("return 1.0 / (1.0 + exp(-x));", "return 1.0 / (1.0 + exp(x));"),
    "silu is identity": ("double or_silu(double x) { return x / (1.0 + exp(-x)); }",
                         "double or_silu(double x) { return x; }"),
    "l2 eps outside sqrt": ("double r = 1.0 / sqrt(ss + eps);", "double r = 1.0 / (sqrt(ss) + eps);"),
    "q scale on k": ("or_l2norm(dk, yk + t * dk, dm->l2_eps, 1.0, kn + t * dk);",
                     "or_l2norm(dk, yk + t * dk, dm->l2_eps, 1.0 / sqrt((double)dk), kn + t * dk);"),
    "decay dropped": ("for (long e = 0; e < (long)d_v * d_k; ++e) S[e] *= decay;",
                      "for (long e = 0; e < (long)d_v * d_k; ++e) S[e] *= 1.0;"),
    "beta dropped": ("double u = beta * (v[i] - sk);", "double u = (v[i] - sk);"),
    "delta sign": ("double u = beta * (v[i] - sk);", "double u = beta * (v[i] + sk);"),
    "output reads k": ("acc += S[(long)i * d_k + j] * q[j];", "acc += S[(long)i * d_k + j] * k[j];"),
    "state transposed in prediction": ("sk += S[(long)i * d_k + j] * k[j];",
                                       "sk += S[(long)(j % d_v) * d_k + (i % d_k)] * k[j];"),
    "rms uses sum not mean": ("ms /= d;", "ms /= 1;"),
    "gate before silu": ("out[i] = o[i] * r * w[i] * or_silu(z[i]);",
                         "out[i] = o[i] * r * w[i] * z[i];"),
    "norm weight dropped": ("out[i] = o[i] * r * w[i] * or_silu(z[i]);",
                            "out[i] = o[i] * r * or_silu(z[i]);"),
    "gqa h mod Hk": ("kh = h / G;", "kh = h % Hk;"),
    "q and k blocks swapped": ("const int chq = kh * dk, chk = Hk * dk + kh * dk,",
                               "const int chk = kh * dk, chq = Hk * dk + kh * dk,"),
    "z of wrong head": ("z + ((t0 + t) * Hv + h) * dv", "z + ((t0 + t) * Hv + (Hv - 1 - h)) * dv"),
    "chunk decay flipped": ("val = beta[c0 + i] * exp(gam[i] - gam[j]) * kk;",
                            "val = beta[c0 + i] * exp(gam[j] - gam[i]) * kk;"),
    "chunk diag excluded": ("for (int s = 0; s <= i; ++s) {", "for (int s = 0; s < i; ++s) {"),
    "chunk state decay dropped": ("double acc = exp(gl) * S0[e * d_k + j];",
                                  "double acc = S0[e * d_k + j];"),
    "products beta dropped": ("acc += beta[s] * v[s * d_v + i] * k[s * d_k + x] * P[x * d_k + c];",
                              "acc += v[s * d_v + i] * k[s * d_k + x] * P[x * d_k + c];"),
    "conv handoff from wrong rows": (
        "conv_input(qkv + t0 * Cc, Cc, st, Cc, W, T - (W - 1) + r, c);",
        "conv_input(qkv + t0 * Cc, Cc, st, Cc, W, (T - (W - 1) + r) < 0 ? (T - (W - 1) + r) : 0, c);"),
    "projection reads w reversed": ("acc += x[m * K + k] * w[n * K + k];",
                                    "acc += x[m * K + k] * w[n * K + (K - 1 - k)];"),
    "projection drops the last term": ("for (long k = 0; k < K; ++k) acc +=",
                                       "for (long k = 0; k + 1 < K; ++k) acc +="),
    "projection reads x row of n": ("acc += x[m * K + k] * w[n * K + k];",
                                    "acc += x[(n % M) * K + k] * w[n * K + k];"),
    "bf16 rounding truncates": ("y[i] = ldexp(nearbyint(ldexp(m, 8)), e - 8);",
                                "y[i] = ldexp(trunc(ldexp(m, 8)), e - 8);"),
    "bf16 ties away from zero": ("y[i] = ldexp(nearbyint(ldexp(m, 8)), e - 8);",
                                 "y[i] = ldexp(round(ldexp(m, 8)), e - 8);"),
    "bf16 keeps 9 bits": ("y[i] = ldexp(nearbyint(ldexp(m, 8)), e - 8);",
                          "y[i] = ldexp(nearbyint(ldexp(m, 9)), e - 9);"),
}

BATTERY = [
    P.test_softplus_closed_forms, P.test_sigmoid_and_silu_closed_forms,
    P.test_gates_closed_forms, P.test_conv_identity_tap_gives_silu,
    P.test_conv_oldest_tap_reads_state_rows_in_order, P.test_conv_box_filter_is_moving_sum,
    P.test_conv_state_carry_identity, lambda: P.test_conv_short_sequence_mixes_state(1),
    P.test_l2norm_closed_form, P.test_gated_rmsnorm_closed_forms,
    P.test_hand_expanded_first_step_from_zero, P.test_hand_expanded_two_steps,
    P.test_beta0_g0_leaves_state_bitwise, P.test_beta1_overwrites_key_direction,
    P.test_full_decay_resets_state, lambda: P.test_products_form_equals_sequential(5, True),
    lambda: P.test_chunked_equals_sequential(16, True), P.test_chunked_survives_decay_underflow,
    L.test_value_head_reads_key_head_floor_h_over_G, L.test_zero_key_block_leaves_pure_decay,
    L.test_first_token_from_zero_state_closed_form, L.test_zero_gate_input_zeroes_only_that_head,
    L.test_write_gate_one_overwrites_key_direction,
    L.test_prefill_then_decode_equals_longer_prefill,
    lambda: L.test_tiny_fp32_sequential_equals_chunked16(True),
    J.test_linear_identity_weight_returns_input, J.test_linear_one_hot_rows_pick_input_columns,
    J.test_linear_hand_computed_2x3, J.test_round_bf16_nearest_even_on_constructed_ties,
    J.test_in_proj_splits_columns_in_the_documented_order, J.test_out_proj_reads_heads_in_row_major_order,
]


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutant '{name}': anchor not found exactly once"
    c = tmp_path / "mutant.c"
    c.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-fPIC", "-shared", "-fopenmp", "-std=c11", "-o", str(so),
                    str(c), "-lm"], check=True)
    return str(so)


def test_unmutated_battery_passes():
    for fn in BATTERY:
        fn()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    so = _build_mutant(tmp_path, name, old, new)
    caught = []
    with oracle.using_library(so):
        for fn in BATTERY:
            try:
                fn()
            except (AssertionError, ValueError, FloatingPointError):
                caught.append(getattr(fn, "__name__", "lambda"))
    assert caught, f"no pin caught the mutant '{name}'"
