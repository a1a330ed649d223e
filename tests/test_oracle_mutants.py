"""Every plausible mistake planted in a copy of the oracle must fail at least one pin.

Each mutant is the oracle's C source with one textual edit (a dropped term, a
wrong sign, a transposed index or operand, ...), compiled on the CPU into a
temporary library and run through the pins of ``oracle_pins``.  A mutant
that passes every pin would mean the pins cannot tell that mistake from the
correct oracle.
"""
import os

import pytest

import oracle
from oracle_pins import ALL_PINS

# (name, text in the oracle source, replacement); the text must occur exactly once
MUTANTS = [
    ("sign_of_A", "exp(dt * a);", "exp(-dt * a);"),
    ("drop_delta_in_Bbar", "? expm1(dt * a) / a : dt;", "? expm1(dt * a) / a : 1.0;"),
    ("zoh_exp_not_expm1", "? expm1(dt * a) / a : dt;", "? exp(dt * a) / a : dt;"),
    ("zoh_times_A", "? expm1(dt * a) / a : dt;", "? expm1(dt * a) * a : dt;"),
    ("zoh_ignored", "(j->zoh && a != 0.0)", "(0 && a != 0.0)"),
    ("zoh_missing_delta_limit", "(j->zoh && a != 0.0)", "(j->zoh)"),
    ("conv_not_causal", "const int64_t tt = t - (width - 1) + k;", "const int64_t tt = t + k;"),
    ("conv_taps_reversed", "acc += (double)w[d * width + k] * load_in", "acc += (double)w[d * width + width - 1 - k] * load_in"),
    ("conv_bias_ignored", "double acc = cb ? (double)cb[d] : 0.0;", "double acc = 0.0;"),
    ("conv_no_silu", "u_out[(b * dim + d) * seqlen + t] = silu(acc);", "u_out[(b * dim + d) * seqlen + t] = acc;"),
    ("u_override_ignored", "const double u = j->u_f64 ? j->u_f64[e]", "const double u = 0 ? j->u_f64[e]"),
    ("reverse_ignored", "j->reverse ? (L - 1 - s) : s;", "s;"),
    ("reverse_off_by_one", "j->reverse ? (L - 1 - s) : s;", "j->reverse ? (L - 1 - s + (s > 0)) : s;"),
    ("drop_D_term", "    y += Dd * u;\n", "\n"),
    ("read_state_before_update",
     "      h[n] = abar * h[n] + bbar * Bv * u;  /* h_t = Ā·h_{t-1} + B̄·u */\n"
     "      y += Cv * h[n];                      /* C·h_t reads the updated state */\n",
     "      y += Cv * h[n];\n      h[n] = abar * h[n] + bbar * Bv * u;\n"),
    ("no_gate", "if (j->z) y *= silu(", "if (0) y *= silu("),
    ("gate_before_D", "    y += Dd * u;\n    if (j->z) y *= silu(load_in(j->z, e, j->in_dtype));\n",
     "    if (j->z) y *= silu(load_in(j->z, e, j->in_dtype));\n    y += Dd * u;\n"),
    ("BC_layout_transposed", "(b * N + n) * L + t; /* index into [B, N, L] */", "(b * L + t) * N + n;"),
    ("B_C_swapped", "const double Bv = load_in(j->B, bc, j->in_dtype);\n      const double Cv = load_in(j->C, bc",
     "const double Bv = load_in(j->C, bc, j->in_dtype);\n      const double Cv = load_in(j->B, bc"),
    ("softplus_identity", "return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));", "return x;"),
    ("softplus_wrong_sign", "log1p(exp(-fabs(x)))", "log1p(exp(fabs(x)))"),
    ("softplus_drops_linear_part", "return (x > 0.0 ? x : 0.0) + log1p", "return 0.0 + log1p"),
    ("bias_ignored", "load_in(j->delta, e, j->in_dtype) + bias;", "load_in(j->delta, e, j->in_dtype);"),
    ("h0_ignored", "h[n] = j->h0_f64 ? j->h0_f64[s0] : (j->h0 ? (double)j->h0[s0] : 0.0);", "h[n] = 0.0;"),
    ("silu_wrong_sign", "return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    ("sigmoid_instead_of_silu", "return z / (1.0 + exp(-z));", "return 1.0 / (1.0 + exp(-z));"),
    ("bf16_shift", "[i]) << 16;", "[i]) << 15;"),
    ("A_index_transposed", "(double)j->A[d * N + n];", "(double)j->A[n * Dm + d];"),
    ("D_index_wrong", "(double)j->D[d] : 0.0;", "(double)j->D[0] : 0.0;"),
    ("bias_index_wrong", "(double)j->delta_bias[d] : 0.0;\n  const double Dd",
     "(double)j->delta_bias[0] : 0.0;\n  const double Dd"),
    ("u_index_off_by_one", "j->u_f64 ? j->u_f64[e] : load_in(j->u, e, j->in_dtype);",
     "j->u_f64 ? j->u_f64[e] : load_in(j->u, t > 0 ? e - 1 : e, j->in_dtype);"),
    ("h_last_not_final", "for (int64_t n = 0; n < N; n++) hl_row[n] = h[n];",
     "for (int64_t n = 0; n < N; n++) hl_row[n] = 0.5 * h[n];"),
    ("step_sign_of_A", "*h = exp(dt * (double)A[d * dstate + n]) * (*h)", "*h = exp(-dt * (double)A[d * dstate + n]) * (*h)"),
    ("step_drop_delta_in_Bbar", "* (*h) + dt * Bv * uu;", "* (*h) + Bv * uu;"),
    ("step_drop_D", "y += (D ? (double)D[d] : 0.0) * uu;", "y += 0.0 * uu;"),
    ("step_no_gate", "if (z) y *= silu(load_in(z, e, in_dtype));", "if (0) y *= silu(load_in(z, e, in_dtype));"),
    ("step_bias_ignored", "x = load_in(delta, e, in_dtype) + (delta_bias ? (double)delta_bias[d] : 0.0);",
     "x = load_in(delta, e, in_dtype);"),
    # the backward
    ("bwd_sign_of_A_in_sweep", "exp(a * dt); /* Ā_t[n] */", "exp(-a * dt); /* Ā_t[n] */"),
    ("bwd_recompute_sign_of_A", "const double abar = exp(dt * (double)j->A[d * N + n]);",
     "const double abar = exp(-dt * (double)j->A[d * N + n]);"),
    ("bwd_no_decay_of_g", "      g[n] = G * abar;\n", "      g[n] = G;\n"),
    ("bwd_dC_with_h_prev", "w->dC[bc] += dy * hs[(t + 1) * N + n];", "w->dC[bc] += dy * hs[t * N + n];"),
    ("bwd_dA_with_h_t", "w->dA[d * N + n] += G * abar * hprev * dt;", "w->dA[d * N + n] += G * abar * hs[(t + 1) * N + n] * dt;"),
    ("bwd_dA_sign", "w->dA[d * N + n] += G * abar * hprev * dt;", "w->dA[d * N + n] -= G * abar * hprev * dt;"),
    ("bwd_ddt_drops_decay_term", "ddt += G * (Bv * u + a * abar * hprev);", "ddt += G * Bv * u;"),
    ("bwd_ddt_drops_input_term", "ddt += G * (Bv * u + a * abar * hprev);", "ddt += G * a * abar * hprev;"),
    ("bwd_du_drops_D", "double du = dy * Dd, ddt = 0.0;", "double du = 0.0, ddt = 0.0;"),
    ("bwd_du_drops_delta", "du += G * dt * Bv;", "du += G * Bv;"),
    ("bwd_dB_uses_dy", "w->dB[bc] += G * dt * u;", "w->dB[bc] += dy * dt * u;"),
    ("bwd_G_without_readout", "const double G = g[n] + dy * Cv;", "const double G = g[n];"),
    ("bwd_softplus_derivative_missing", "ddt * sigmoid(x) : ddt;", "ddt : ddt;"),
    ("bwd_dz_missing_silu_slope", "sg * (1.0 + zz * (1.0 - sg));", "sg;"),
    ("bwd_dy_ungated", "dy = j->dout[e] * zz * sg;", "dy = j->dout[e];"),
    ("bwd_dD_uses_dout", "if (w->dD) w->dD[d] += dy * u;", "if (w->dD) w->dD[d] += j->dout[e] * u;"),
    ("bwd_dh_last_ignored", "g[n] = j->dh_last ? j->dh_last[(b * Dm + d) * N + n] : 0.0;", "g[n] = 0.0;"),
    ("bwd_recompute_without_h0", "hs[n] = j->h0 ? (double)j->h0[(b * Dm + d) * N + n] : 0.0;", "hs[n] = 0.0;"),
    ("bwd_dbias_uses_ddt", "if (w->dbias) w->dbias[d] += dx;", "if (w->dbias) w->dbias[d] += ddt;"),
    ("bwd_reduction_drops_worker", "for (size_t i = 0; dB && i < nbc; i++) dB[i] += ws[k].dB[i];",
     "for (size_t i = 0; dB && i < nbc && k == 0; i++) dB[i] += ws[k].dB[i];"),
]


@pytest.fixture(scope="module")
def source():
    with open(oracle.SRC) as f:
        return f.read()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, source, name, old, new):
    assert source.count(old) == 1, f"mutation site for {name} not found exactly once"
    src = tmp_path / f"mutant_{name}.c"
    src.write_text(source.replace(old, new))
    lib = oracle.load(oracle.compile_oracle(str(src), str(tmp_path / f"libmutant_{name}.so")))
    caught = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"


def test_unmutated_copy_passes(tmp_path, source):
    src = tmp_path / "copy.c"
    src.write_text(source)
    lib = oracle.load(oracle.compile_oracle(str(src), str(tmp_path / "libcopy.so")))
    for pin in ALL_PINS:
        pin(lib)
