"""Planted mistakes in the oracle must each trip at least one pin.

Every case copies ``oracle/ssm_oracle.c``, applies one plausible slip (a
dropped term, a wrong sign or index, a swapped operand, a wrong activation),
compiles the copy with gcc into a temporary directory and runs the pins on it.
A mutant that passes every pin would mean the pins cannot see that mistake.
The real oracle source is never modified.
"""
import os

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "oracle", "ssm_oracle.c")

# the input stage's forward loop body
CONV_FWD = ("double pre = bias ? bias[d] : 0.0;\n"
            "                for (int64_t k = 0; k < K; ++k) {\n"
            "                    const int64_t s = t - (K - 1) + k;\n"
            "                    if (s >= 0) pre += w[d * K + k] * x[(b * L + s) * dim + d];\n"
            "                }\n"
            "                u[(b * L + t) * dim + d] = oracle_silu(pre);")

# (name, text in the oracle source, replacement)
MUTANTS = [
    ("drop_D_skip", "if (j->D) y += j->D[d] * xv;", ""),
    ("wrong_sign_in_exp", "exp(dt * j->A[d * N + n])", "exp(-dt * j->A[d * N + n])"),
    ("transposed_A", "exp(dt * j->A[d * N + n])", "exp(dt * j->A[n * j->dim + d])"),
    ("Bbar_without_delta", "const double dBx = dt * j->B[", "const double dBx = j->B["),
    ("B_time_index_off_by_one", "j->B[(b * L + t) * N + n]",
     "j->B[(b * L + (t > 0 ? t - 1 : 0)) * N + n]"),
    ("C_reads_B", "acc += j->C[(b * L + t) * N + n] * h[n];",
     "acc += j->B[(b * L + t) * N + n] * h[n];"),
    ("y_reads_state_before_update",
     "h[n] = dA * h[n] + dBx;\n            acc += j->C[(b * L + t) * N + n] * h[n];",
     "acc += j->C[(b * L + t) * N + n] * h[n];\n            h[n] = dA * h[n] + dBx;"),
    ("drop_delta_bias", "if (j->delta_bias) dt += j->delta_bias[d];", ""),
    ("bias_after_softplus",
     "if (j->delta_bias) dt += j->delta_bias[d];\n        if (j->delta_softplus) dt = oracle_softplus(dt);",
     "if (j->delta_softplus) dt = oracle_softplus(dt);\n        if (j->delta_bias) dt += j->delta_bias[d];"),
    ("softplus_wrong_sign", "log1p(exp(-fabs(v)))", "log1p(exp(fabs(v)))"),
    ("gate_sigmoid_not_silu", "return z / (1.0 + exp(-z));", "return 1.0 / (1.0 + exp(-z));"),
    ("gate_before_D", "if (j->D) y += j->D[d] * xv;\n        if (j->z) y *= oracle_silu(j->z[e]);",
     "if (j->z) y *= oracle_silu(j->z[e]);\n        if (j->D) y += j->D[d] * xv;"),
    ("h0_ignored", "h[n] = j->h0 ? j->h0[(b * dim + d) * N + n] : 0.0;", "h[n] = 0.0;"),
    ("final_state_index_transposed", "j->final_state[(b * dim + d) * N + n] = h[n];",
     "j->final_state[(b * dim + d) + n * (j->batch * dim)] = h[n];"),
    ("decode_drops_delta_in_exp", "*h = exp(dt * A[d * N + n]) * (*h)",
     "*h = exp(A[d * N + n]) * (*h)"),
    ("decode_wrong_B_row", "dt * B[b * N + n] * xv", "dt * B[n] * xv"),
    ("core_recurrence_drops_state", "h[n] = Abar[t * N + n] * h[n] + Bbar[t * N + n] * x[t];",
     "h[n] = Abar[t * N + n] + Bbar[t * N + n] * x[t];"),
    ("core_readout_drops_C", "acc += C[t * N + n] * h[n];", "acc += h[n];"),
    # the forward's window (the backward recomputes the same pre-activation)
    ("conv_kernel_flipped", CONV_FWD, CONV_FWD.replace("w[d * K + k]", "w[d * K + (K - 1 - k)]")),
    ("conv_shift_off_by_one", CONV_FWD, CONV_FWD.replace("t - (K - 1) + k", "t - K + k")),
    ("conv_drops_bias", CONV_FWD, CONV_FWD.replace("bias ? bias[d] : 0.0", "0.0")),
    ("conv_without_silu", "u[(b * L + t) * dim + d] = oracle_silu(pre);",
     "u[(b * L + t) * dim + d] = pre;"),
    ("zoh_phi_drops_division", "return z == 0.0 ? 1.0 : expm1(z) / z;",
     "return z == 0.0 ? 1.0 : expm1(z);"),
    ("zoh_ignored_in_scan", "* (j->zoh ? oracle_phi(dt * j->A[d * N + n]) : 1.0);", "* 1.0;"),
    ("zoh_phi_wrong_sign", "oracle_phi(dt * j->A[d * N + n])", "oracle_phi(-dt * j->A[d * N + n])"),
    ("zoh_ignored_in_decode", "* (zoh ? oracle_phi(dt * A[d * N + n]) : 1.0);", "* 1.0;"),
    ("bwd_dC_reads_state_before_update", "j->dC[(b * L + t) * N + n] += dy * ht;",
     "j->dC[(b * L + t) * N + n] += dy * hprev;"),
    ("bwd_carry_drops_decay", "G[n] = a * g;", "G[n] = g;"),
    ("bwd_ddt_drops_input_term", "ddt += g * ((j->zoh ? a : 1.0) * xv * Bt[n] + Ad[n] * a * hprev);",
     "ddt += g * (Ad[n] * a * hprev);"),
    ("bwd_softplus_derivative_missing",
     "const double dd = j->delta_softplus ? ddt * oracle_sigmoid(j->delta[e] + bias) : ddt;",
     "const double dd = ddt;"),
    ("bwd_silu_derivative_wrong", "s * (1.0 + j->z[e] * (1.0 - s))", "s"),
    ("bwd_dA_missing_dt", "j->dA[d * N + n] += g * (dt * a * hprev",
     "j->dA[d * N + n] += g * (a * hprev"),
    ("bwd_dx_drops_D", "double dx = j->D ? dy * j->D[d] : 0.0;", "double dx = 0.0;"),
    ("bwd_dB_drops_x", "j->dB[(b * L + t) * N + n] += g * dt * p * xv;",
     "j->dB[(b * L + t) * N + n] += g * dt * p;"),
    ("bwd_dh0_one_step_late", "j->dh0[(b * dim + d) * N + n] = G[n];",
     "j->dh0[(b * dim + d) * N + n] = G[n] / exp(dtv[0] * Ad[n]);"),
    ("phi_prime_series_wrong_denominator", "sum += term / (k + 2);", "sum += term / (k + 1);"),
    ("phi_prime_closed_form_wrong_sign", "(exp(z) * (z - 1.0) + 1.0)", "(exp(z) * (z + 1.0) - 1.0)"),
    ("bwd_zoh_recompute_first_order",
     "const double p = j->zoh ? oracle_phi(dt * Ad[n]) : 1.0;\n            h[n] =",
     "const double p = 1.0;\n            h[n] ="),
    ("bwd_zoh_dB_drops_phi", "j->dB[(b * L + t) * N + n] += g * dt * p * xv;",
     "j->dB[(b * L + t) * N + n] += g * dt * xv;"),
    ("bwd_zoh_dx_drops_phi", "dx += g * dt * p * Bt[n];", "dx += g * dt * Bt[n];"),
    ("bwd_zoh_ddt_first_order_input_term", "(j->zoh ? a : 1.0) * xv * Bt[n]", "xv * Bt[n]"),
    ("bwd_zoh_dA_drops_hold_term", "(j->zoh ? dt * dt * oracle_phi_prime(dt * Ad[n])",
     "(0 ? dt * dt * oracle_phi_prime(dt * Ad[n])"),
    ("bwd_zoh_dA_hold_term_one_dt", "dt * dt * oracle_phi_prime(dt * Ad[n])",
     "dt * oracle_phi_prime(dt * Ad[n])"),
    ("conv_bwd_sigmoid_not_silu_derivative", "du[(b * L + t) * dim + d] * sg * (1.0 + pre * (1.0 - sg))",
     "du[(b * L + t) * dim + d] * sg"),
    ("conv_bwd_dx_flipped_taps", "dx[(b * L + s) * dim + d] += dpre * w[d * K + k];",
     "dx[(b * L + s) * dim + d] += dpre * w[d * K + (K - 1 - k)];"),
    ("conv_bwd_dw_reads_current_token", "if (dw) dw[d * K + k] += dpre * x[(b * L + s) * dim + d];",
     "if (dw) dw[d * K + k] += dpre * x[(b * L + t) * dim + d];"),
    ("conv_bwd_drops_bias_in_pre", "double pre = bias ? bias[d] : 0.0;\n                for (int64_t k = 0; k < K; ++k) {\n                    const int64_t s = t - (K - 1) + k;\n                    if (s >= 0) pre += w[d * K + k] * x[(b * L + s) * dim + d];\n                }\n                const double sg",
     "double pre = 0.0;\n                for (int64_t k = 0; k < K; ++k) {\n                    const int64_t s = t - (K - 1) + k;\n                    if (s >= 0) pre += w[d * K + k] * x[(b * L + s) * dim + d];\n                }\n                const double sg"),
    ("conv_bwd_dbias_drops_derivative", "if (dbias) dbias[d] += dpre;",
     "if (dbias) dbias[d] += du[(b * L + t) * dim + d];"),
    ("ssd_group_interleaved", "g = hd / (H / G);", "g = hd % G;"),
    ("ssd_drops_dt_bias", "if (j->dt_bias) dt += j->dt_bias[hd];", ""),
    ("ssd_decay_without_dt", "const double a = exp(dt * j->A[hd]);", "const double a = exp(j->A[hd]);"),
    ("ssd_drops_decay", "h[p * N + n] = a * h[p * N + n] + dt * j->x[e] * Bt[n];",
     "h[p * N + n] = h[p * N + n] + dt * j->x[e] * Bt[n];"),
    ("ssd_reads_B_for_C", "acc += Ct[n] * h[p * N + n];", "acc += Bt[n] * h[p * N + n];"),
    ("ssd_drops_D", "j->y[e] = acc + (j->D ? j->D[hd] * j->x[e] : 0.0);", "j->y[e] = acc;"),
    ("ssd_dt_per_channel_slot", "double dt = j->dt[(b * L + t) * H + hd];",
     "double dt = j->dt[(b * L + t) * H + (hd + 1) % H];"),
    ("ssd_h0_ignored", "h[i] = j->h0 ? j->h0[pair * P * N + i] : 0.0;", "h[i] = 0.0;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation anchor not found exactly once: %s" % name
    path = tmp_path / ("mut_%s.c" % name)
    path.write_text(src.replace(old, new))
    lib = oracle.compile_source(str(path), str(tmp_path / ("libmut_%s.so" % name)))
    orc = oracle.Oracle(lib)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, RuntimeError, ValueError, FloatingPointError):
            failed.append(pin.__name__)
    assert failed, "mutant %s passed every pin" % name
