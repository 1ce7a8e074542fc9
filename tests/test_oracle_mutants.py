"""Planted mistakes in the oracle (on the CPU): every plausible slip in the
recurrence must make at least one pin fail. Each mutant is a textual edit of a
temporary copy of oracle/ss_oracle.c, compiled separately; the committed
oracle is never modified."""

import os
import shutil
import tempfile

import pytest

import pins
from oracle import build as obuild

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "ss_oracle.c")

MUTANTS = {
    "exp_sign": ("exp(delta * (double)j->A[d * N + n])", "exp(-delta * (double)j->A[d * N + n])"),
    "drop_skip": ("y += dsk * x;", "y += 0.0 * dsk * x;"),
    "readout_uses_B": ("y += widen(j->C, j->in_dtype, r + n) * h[n];", "y += widen(j->B, j->in_dtype, r + n) * h[n];"),
    "gate_without_sigmoid": ("if (j->z) y *= silu(", "if (j->z) y *= (1.0 + 0.0 * "),
    "drop_bias": ("softplus(widen(j->delta_raw, j->in_dtype, i) + bias)", "softplus(widen(j->delta_raw, j->in_dtype, i))"),
    "A_transposed": ("(double)j->A[d * N + n]", "(double)j->A[(n * Dm + d) % (Dm * N)]"),
    "softplus_is_exp": ("return log1p(exp(x));", "return exp(x);"),
    "h0_ignored": ("h[n] = j->h0 ? (double)j->h0[(b * Dm + d) * N + n] : 0.0;", "h[n] = 0.0;"),
    "bbar_without_delta": ("const double bbar_x = delta * widen(j->B", "const double bbar_x = 1.0 * widen(j->B"),
    "B_time_lag": ("const int64_t r = (b * L + t) * N;", "const int64_t r = (b * L + (t > 0 ? t - 1 : 0)) * N;"),
    "readout_before_update": ("h[n] = abar * h[n] + bbar_x;\n      y += widen(j->C, j->in_dtype, r + n) * h[n];",
                              "y += widen(j->C, j->in_dtype, r + n) * h[n];\n      h[n] = abar * h[n] + bbar_x;"),
    "skip_outside_gate": ("    y += dsk * x;\n    if (j->z) y *= silu(widen(j->z, j->in_dtype, i));",
                          "    if (j->z) y *= silu(widen(j->z, j->in_dtype, i));\n    y += dsk * x;"),
    "batch_stride_B": ("const int64_t r = (b * L + t) * N;", "const int64_t r = (t) * N;"),
    "decode_exp_sign": ("hs[n] = exp(delta * (double)A[d * dstate + n]) * hs[n] +",
                        "hs[n] = exp(-delta * (double)A[d * dstate + n]) * hs[n] +"),
    # backward pass
    "bwd_no_decay_of_adjoint": ("lam[n] *= a; /* becomes", "lam[n] *= 1.0; /* becomes"),
    "bwd_dA_uses_h_t": ("dA[d * N + n] += lam[n] * hist[t * N + n] * a * delta[t];",
                        "dA[d * N + n] += lam[n] * hist[(t + 1) * N + n] * a * delta[t];"),
    "bwd_dC_uses_lambda": ("dC[r + n] += dyv * hist[(t + 1) * N + n];", "dC[r + n] += lam[n] * hist[(t + 1) * N + n];"),
    "bwd_dB_without_delta": ("dB[r + n] += lam[n] * delta[t] * x;", "dB[r + n] += lam[n] * x;"),
    "bwd_no_softplus_derivative": ("ddelta_raw[i] = ddel * sg;", "ddelta_raw[i] = ddel;"),
    "bwd_dh_last_ignored": ("lam[n] = dh_last ? (double)dh_last[(b * Dm + d) * N + n] : 0.0;", "lam[n] = 0.0;"),
    "bwd_gate_derivative_is_sigmoid": ("return s * (1.0 + z * (1.0 - s));", "return s;"),
    # generalised scan
    "gen_zoh_without_division_by_A": ("expm1(delta * a) / a : delta", "expm1(delta * a) : delta"),
    "gen_zoh_exp_instead_of_expm1": ("expm1(delta * a) / a : delta", "exp(delta * a) / a : delta"),
    "gen_zoh_ignored": ("(j->disc == 1 && a != 0.0)", "(j->disc == 7 && a != 0.0)"),
    "gen_group_by_modulo": ("const int64_t g = d / (Dm / G);", "const int64_t g = d % G;"),
    "gen_row_without_groups": ("const int64_t r = ((b * L + t) * G + g) * N;", "const int64_t r = ((b * L + t) + g) * N;"),
    "gen_A_row_of_16": ("const double a = (double)j->A[d * N + n];", "const double a = (double)j->A[d * 16 + n % 16];"),
    # convolution front-end
    "conv_taps_reversed": ("pre += (double)w[d * width + k] * e[t + k];",
                           "pre += (double)w[d * width + (width - 1 - k)] * e[t + k];"),
    "conv_drop_bias": ("double pre = bias ? (double)bias[d] : 0.0;\n        for (int64_t k = 0; k < width; k++)",
                       "double pre = 0.0;\n        for (int64_t k = 0; k < width; k++)"),
    "conv_not_causal": ("for (int64_t k = 0; k < width; k++) pre += (double)w[d * width + k] * e[t + k];",
                        "for (int64_t k = 0; k < width; k++) pre += (double)w[d * width + k] * e[t + k + (t + k + 1 < seqlen + H ? 1 : 0)];"),
    "conv_state_ignored": ("e[q] = state_in ? widen(state_in, in_dtype, (b * dim + d) * H + q) : 0.0;", "e[q] = 0.0;"),
    "conv_state_out_shift": ("state_out[(b * dim + d) * H + k] = e[seqlen + k];",
                             "state_out[(b * dim + d) * H + k] = e[seqlen + k - (seqlen + k > 0 ? 1 : 0)];"),
    "conv_decode_no_shift": ("for (int64_t k = 0; k + 1 < H; k++) s[k] = s[k + 1];", ""),
    "conv_decode_x_tap": ("pre += (double)w[d * width + H] * xv;", "pre += (double)w[d * width + 0] * xv;"),
}


@pytest.fixture(scope="module")
def tmpdir_mod():
    d = tempfile.mkdtemp(prefix="ss_oracle_mut_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmpdir_mod):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new, 1)
    csrc = os.path.join(tmpdir_mod, f"{name}.c")
    with open(csrc, "w") as f:
        f.write(mutated)
    lib = obuild.build(csrc, os.path.join(tmpdir_mod, f"lib_{name}.so"), extra=("-Wno-unused",))
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"


# Planted mistakes in the state-space-dual wrapper (oracle.ssd expands heads
# into channels of the generalised scan): each must fail the semiseparable pin.
SSD_MUTANTS = {
    "ssd_dt_tiled_not_repeated": ("dt.repeat_interleave(P, dim=2)", "dt.repeat(1, 1, P)"),
    "ssd_A_tiled_not_repeated": ('_f32(x["A"]).repeat_interleave(P)', '_f32(x["A"]).repeat(P)'),
    "ssd_zero_order_hold": ('ngroups, "euler"', 'ngroups, "zoh"'),
    "ssd_bias_dropped": ('if x.get("dt_bias") is not None else None', 'if False else None'),
}


@pytest.mark.parametrize("name", sorted(SSD_MUTANTS))
def test_ssd_wrapper_mutant_is_caught(name, monkeypatch):
    import inspect
    import textwrap

    import oracle

    old, new = SSD_MUTANTS[name]
    src = textwrap.dedent(inspect.getsource(oracle.ssd))
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), f"<{name}>", "exec"), ns)
    monkeypatch.setattr(oracle, "ssd", ns["ssd"])
    with pytest.raises(AssertionError):
        pins.pin_ssd_semiseparable()
