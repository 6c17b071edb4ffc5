"""Planted mistakes in the oracle, on the CPU.

Each mutant is the oracle's C source with one plausible error written in: a
dropped term, a wrong sign, index or rounding rule, a transposed operand, a
skipped step.  It is compiled into a library of its own, swapped in for the
oracle, and at least one pin of test_oracle_pins.py or test_oracle_flips.py
has to fail on it: the pins hold the oracle to the pages and to mathematics,
not only on its own happy path.  The unmodified source passes every pin (the
control case).
"""
import inspect
import itertools
import os
import subprocess

import pytest

import oracle
import oracle.build as ob
import test_oracle_flips as flip_pins
import test_oracle_pins as pins

SRC = os.path.join(ob.HERE, "moe_oracle.c")

# (name, text of the oracle, text of the mutant); each text occurs once
MUTANTS = [
    ("bf16_truncates", "return (uint16_t)((b + 0x7FFFu + lsb) >> 16);", "return (uint16_t)(b >> 16);"),
    ("q2k_drops_min_term", "w[e] = d * sc * q - dmin * mn;", "w[e] = d * sc * q;"),
    ("q2k_swaps_scale_and_min", "int sc = scales[b] & 15, mn = scales[b] >> 4;",
     "int sc = scales[b] >> 4, mn = scales[b] & 15;"),
    ("q2k_wrong_plane_shift", "int q = (qs[32 * h + l] >> (2 * j)) & 3;\n    int sc",
     "int q = (qs[32 * h + l] >> j) & 3;\n    int sc"),
    ("q3k_high_bit_sign", "int q = lo - (hb ? 0 : 4);", "int q = lo - (hb ? 4 : 0);"),
    ("q3k_scale_without_offset", "w[e] = d * (orc_q3k_scale_code(scales, b) - 32) * q;",
     "w[e] = d * orc_q3k_scale_code(scales, b) * q;"),
    ("q3k_high_scale_bits", "int hi2 = (scales12[8 + b % 4] >> (2 * (b / 4))) & 3;",
     "int hi2 = (scales12[8 + b / 4] >> (2 * (b % 4))) & 3;"),
    ("q8_1_half_to_even", "static float round_half_away(float v) { return roundf(v); }",
     "static float round_half_away(float v) { return rintf(v); }"),
    ("q8_1_divides_by_128", "float d = amax / 127.0f;", "float d = amax / 128.0f;"),
    ("q8_1_sum_without_d", "uint16_t s16 = orc_f16_from_f32(d * (float)sum);",
     "uint16_t s16 = orc_f16_from_f32((float)sum);"),
    ("router_transposed_weight", "orc_bf16_value(W[(size_t)e * D + d]);",
     "orc_bf16_value(W[(size_t)d * N + e]);"),
    ("score_without_sqrt", "return (float)sqrt(log1p(exp((double)t)));", "return (float)log1p(exp((double)t));"),
    ("score_ignores_temperature", "float orc_score(float z, float gate_temp) {\n  float t = z / gate_temp;",
     "float orc_score(float z, float gate_temp) {\n  float t = z;"),
    ("sigmoid_sign", "s[e] = (float)(1.0 / (1.0 + exp(-(double)t)));", "s[e] = (float)(1.0 / (1.0 + exp((double)t)));"),
    ("nan_key_ranks_first", "if (na != nb) return nb;", "if (na != nb) return na;"),
    ("ties_to_higher_id", "  return a < b;\n}", "  return a > b;\n}"),
    ("weights_from_biased_keys", "w_out[i] = s[order[i]];", "w_out[i] = key[order[i]];"),
    ("no_renormalisation", "if (c->norm_topk_prob && k > 1) {", "if (0) {"),
    ("route_scale_dropped", "for (int i = 0; i < k; ++i) w_out[i] *= c->route_scale;", ""),
    ("image_tokens_ignore_bias_vl",
     "const float* bias = (L->image_mask && L->bias_vl && L->image_mask[t]) ? L->bias_vl : L->bias;",
     "const float* bias = L->bias;"),
    ("swiglu_sigma_of_up", "double sig = 1.0 / (1.0 + exp(-g));", "double sig = 1.0 / (1.0 + exp(-u));"),
    ("swiglu_clamps_gate_below", "if (u > limit) { u = limit;", "if (g < -limit) g = -limit;\n    if (u > limit) { u = limit;"),
    ("h_not_requantised", "orc_dequant_q8_1(hq8, I, hh);", "for (int j = 0; j < I; ++j) hh[j] = h[j];"),
    ("shared_h_not_bf16", "hb[r] = orc_bf16_value(orc_bf16_from_f32(h));", "hb[r] = h;"),
    ("shared_down_transposed", "acc += orc_bf16_value(w2[(size_t)d * I + j]) * hb[j];",
     "acc += orc_bf16_value(w2[(size_t)j * D + d]) * hb[j];"),
    ("routed_outputs_unweighted", "double g = (double)w[slot];", "double g = 1.0;"),
    ("shared_expert_dropped", "for (int d = 0; d < D; ++d) out[d] = y[d] + E[d];",
     "for (int d = 0; d < D; ++d) out[d] = y[d];"),
    ("q2k_d_and_dmin_swapped", "double d = orc_f16_value((uint16_t)(blk[80] | (blk[81] << 8)));",
     "double d = orc_f16_value((uint16_t)(blk[82] | (blk[83] << 8)));"),
    ("q3k_hmask_bit_transposed", "int hb = (hmask[l] >> (4 * h + j)) & 1;", "int hb = (hmask[l] >> (h + 4 * j)) & 1;"),
    ("q3k_upper_scales_low_nibble", "(scales12[b - 8] >> 4)", "(scales12[b - 8] & 15)"),
    ("q8_1_signed_max", "float a = fabsf(xb[i]);", "float a = xb[i];"),
    ("keys_ascending", "if (!na && ka != kb) return ka > kb;", "if (!na && ka != kb) return ka < kb;"),
    ("no_epsilon", "sum += 1e-20f;", ""),
    ("normalises_over_all_experts", "for (int i = 0; i < k; ++i) sum += w_out[i];",
     "for (int i = 0; i < N; ++i) sum += s[i];"),
    ("normalises_single_pick", "if (c->norm_topk_prob && k > 1) {", "if (c->norm_topk_prob) {"),
    ("softmax_without_shift", "double mx = -INFINITY, sum = 0.0;\n    int any_nan = 0;\n    for (int e = 0; e < N; ++e) {\n"
     "      float t = z[e] / c->gate_temp;\n      if (isnan(t)) any_nan = 1;\n      else if (t > mx) mx = t;\n",
     "double mx = 0.0, sum = 0.0;\n    int any_nan = 0;\n    for (int e = 0; e < N; ++e) {\n"
     "      float t = z[e] / c->gate_temp;\n      if (isnan(t)) any_nan = 1;\n"),
    ("up_clamped_only_above", "if (u < -limit) { u = -limit; if (clipped) ++*clipped; }", ""),
    ("clamps_at_zero_limit", "if (limit > 0) {", "if (limit >= 0) {"),
    ("gate_and_up_swapped", "const uint8_t* w1 = L->experts[3 * e + 0];\n    const uint8_t* w3 = L->experts[3 * e + 1];",
     "const uint8_t* w1 = L->experts[3 * e + 1];\n    const uint8_t* w3 = L->experts[3 * e + 0];"),
    # the requantisation flip candidates
    ("flip_code_change_sign", "f->coef[0] = G * (double)(qq - q[i]) * dv;", "f->coef[0] = G * (double)(q[i] - qq) * dv;"),
    ("flip_code_unscaled", "f->coef[0] = G * (double)(qq - q[i]) * dv;", "f->coef[0] = (double)(qq - q[i]) * dv;"),
    ("flip_scale_keeps_codes", "int q2 = q8_code(hb[i], d2, ends[e]);", "int q2 = q[i];"),
    ("flip_scale_one_column", "for (int i = 0; i < f->n; ++i) s += f->coef[i] * row[f->j0 + i];",
     "for (int i = 0; i < f->n; ++i) s += f->coef[i] * row[f->j0];"),
    ("flip_window_on_gate_only", "swiglu_range(g, u, kappa * sg, kappa * su, c->swiglu_limit, &lo[r], &hi[r]);",
     "swiglu_range(g, u, kappa * sg, 0.0, c->swiglu_limit, &lo[r], &hi[r]);"),
    ("flip_bf16_ends_only", "if (key == kh || (k1 - k0 > BF16_SPAN && key != k0 && key != k1)) continue;",
     "if (key == kh || (key != k0 && key != k1)) continue;"),
    ("flip_bf16_change_from_zero", "f->coef[0] = orc_bf16_value(alt) - orc_bf16_value(hb);",
     "f->coef[0] = orc_bf16_value(alt);"),
]


def _pin_cases():
    """Every pin of the two pin modules with each of its parameter sets."""
    for mod in (pins, flip_pins):
        for name, fn in inspect.getmembers(mod, inspect.isfunction):
            if not name.startswith("test_") or fn.__module__ != mod.__name__:
                continue
            sets = []
            for mk in getattr(fn, "pytestmark", []):
                if mk.name != "parametrize":
                    continue
                argnames, values = mk.args[:2]
                names = [a.strip() for a in argnames.split(",")] if isinstance(argnames, str) else list(argnames)
                sets.append([dict(zip(names, v if len(names) > 1 else (v,))) for v in values])
            for combo in itertools.product(*sets):
                kw = {}
                for d in combo:
                    kw.update(d)
                yield name, fn, kw


def _first_failing_pin():
    for name, fn, kw in _pin_cases():
        try:
            fn(**kw)
        except Exception:  # an assertion, or an error the pin's own checks raise
            return name
    return None


def _use_library(monkeypatch, so):
    monkeypatch.setattr(oracle, "SO", so)
    monkeypatch.setattr(oracle, "_lib", None)


def test_every_pin_passes_on_the_oracle(tmp_path, monkeypatch):
    so = str(tmp_path / "liboracle_control.so")
    subprocess.run(ob.command(SRC, so), check=True, capture_output=True)
    _use_library(monkeypatch, so)
    assert _first_failing_pin() is None


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_a_pin_catches_the_planted_mistake(name, old, new, tmp_path, monkeypatch):
    text = open(SRC).read()
    assert text.count(old) == 1, f"{name}: the text to change must occur exactly once"
    src = tmp_path / "moe_oracle_mutant.c"
    src.write_text(text.replace(old, new))
    so = str(tmp_path / "liboracle_mutant.so")
    p = subprocess.run(ob.command(str(src), so), capture_output=True, text=True)
    assert p.returncode == 0, p.stdout + p.stderr
    _use_library(monkeypatch, so)
    assert _first_failing_pin() is not None, f"no pin fails with the planted mistake {name}"
