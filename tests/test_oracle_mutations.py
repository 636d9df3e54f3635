"""Plant plausible mistakes in a copy of the oracle and check that the pins
catch each one. The copy is built from the oracle's source text with one
substitution and loaded as a separate module; the real oracle is untouched.
"""
import importlib.util
import inspect
import types

import pytest

from oracle import pa_oracle
import tests.test_oracle_pins as pins

MUTANTS = {
    "rope_first_half_sign": ("seg[:half] = a * c - b * s", "seg[:half] = a * c + b * s"),
    "rope_second_half_sign": ("seg[half:] = b * c + a * s", "seg[half:] = b * c - a * s"),
    "rope_interleaved_sign": ("seg[0::2] = a * c - b * s", "seg[0::2] = a * c + b * s"),
    "rope_wrong_position": ("c = cos_tab[pos, :half]", "c = cos_tab[max(pos - 1, 0), :half]"),
    "window_off_by_one": ("max(0, pos - window)", "max(0, pos - window + 1)"),
    "causal_excludes_self": ("return range(lo, pos + 1)", "return range(lo, max(pos, lo + 1))"),
    "softcap_dropped": ('s = p["softcap"] * np.tanh(s / p["softcap"])', "pass"),
    "softcap_before_scale": ('s = (q @ K.T) * p["scale"]', 's = (q @ K.T)'),
    "value_wrong_channels": ("(w @ K[:, :vhs])", "(w @ K[:, hs - vhs:])"),
    "block_offset_wrong": ("return phys * block_size + j % block_size",
                           "return phys * block_size + (j + 1) % block_size"),
    "position_ignores_past": ("return b, int(past[b]) + (t - int(cumseq[b]))",
                              "return b, (t - int(cumseq[b]))"),
    "rounding_truncates": ("r = np.rint(x / spacing) * spacing",
                           "r = np.trunc(x / spacing) * spacing"),
    "slot_minus_one_written": ("if slot < 0:\n            continue",
                               "if slot < -1:\n            continue"),
    "softmax_not_normalised": ("out = (w @ K[:, :vhs]) / den", "out = (w @ K[:, :vhs])"),
    "scales_prob_not_squared": ("n_p = np.sqrt(np.maximum((prob * prob) @ V2, 0.0))",
                                "n_p = np.sqrt(np.maximum(prob @ V2, 0.0))"),
    "scales_score_centre_dropped": ("var_a = (a @ V2) - 2.0 * out * (a @ V)",
                                    "var_a = (a @ V2) - 0.0 * out * (a @ V)"),
    "scales_diag_wrong_channel": ("np.abs(q[:, :vhs])", "np.abs(q[:, -vhs:])"),
    "e4m3_bias_8": ("np.ldexp(1.0, e - 7)", "np.ldexp(1.0, e - 8)"),
    "e4m3_subnormal_scale": ("np.where(e == 0, m * 2.0 ** -9,", "np.where(e == 0, m * 2.0 ** -10,"),
    "e4m3_truncates": ("r = np.minimum(np.rint(ax / spacing) * spacing, E4M3_MAX)",
                       "r = np.minimum(np.floor(ax / spacing) * spacing, E4M3_MAX)"),
    "e4m3_saturates_too_high": ("E4M3_MAX = 448.0", "E4M3_MAX = 480.0"),
    "fp8_read_unscaled": ("return e4m3_to_f64(self.codes[idx]) * self.k_scale",
                          "return e4m3_to_f64(self.codes[idx])"),
    "fp8_multiplies": ("q32 = v32 / np.float32(k_scale)", "q32 = v32 * np.float32(k_scale)"),
    "sep_kv_head_wrong": ("        g = h // grp\n", "        g = h % kvh\n"),
    "sep_sink_not_in_denominator": ("        den = w.sum() + extra", "        den = w.sum()"),
    "sep_rms_sum": ("np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)",
                    "np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)"),
    "sep_value_rotated": ("            vcache.put(slot * kvh + g, v[g])",
                          "            vcache.put(slot * kvh + g, rope_row(v[g], pos, p[\"rotary_offset\"], p[\"rotary_dim\"], cos_tab, sin_tab, False))"),
}

PINS = [
    lambda: pins.test_round_bf16_matches_torch_cast(),
    lambda: pins.test_round_f16_matches_numpy_cast(),
    lambda: pins.test_rope_is_complex_rotation(0),
    lambda: pins.test_rope_is_complex_rotation(1),
    lambda: pins.test_rope_relative_position(0),
    lambda: pins.test_attention_matches_naive_contiguous(0.0, -1),
    lambda: pins.test_attention_matches_naive_contiguous(1.5, -1),
    lambda: pins.test_attention_matches_naive_contiguous(0.0, 3),
    lambda: pins.test_absorbed_equals_decomposed_mla(128, 32, 32, 64, 3),
    lambda: pins.test_slot_minus_one_leaves_cache_untouched(),
    lambda: pins.test_two_key_softcap_closed_form(),
    lambda: pins.test_error_scales_single_key(),
    lambda: pins.test_error_scales_equal_probabilities(),
    lambda: pins.test_error_scales_probability_term_monte_carlo(),
    lambda: pins.test_error_scales_score_term_monte_carlo(),
    lambda: pins.test_error_scales_diagonal_term_is_a_derivative(),
    lambda: pins.test_e4m3_decode_matches_torch(),
    lambda: pins.test_e4m3_rounding_matches_torch_cast_in_range(),
    lambda: pins.test_e4m3_saturates_to_448(),
    lambda: pins.test_fp8_write_is_exact_for_representable_rows(),
    lambda: pins.test_fp8_read_equals_plain_read_of_dequantized_cache(),
    lambda: pins.test_fp8_quantization_divides_by_k_scale_in_float32(),
    lambda: pins.test_separate_matches_naive_dense(dict(num_heads=4, kv_num_heads=2, head_size=32,
                                                        rotary_dim=16)),
    lambda: pins.test_separate_matches_naive_dense(dict(num_heads=8, kv_num_heads=2, head_size=64,
                                                        rotary_dim=64, head_sink=True,
                                                        qk_norm=True, softcap=2.0,
                                                        local_window_size=5)),
    lambda: pins.test_rms_norm_matches_torch(),
    lambda: pins.test_head_sink_closed_forms(),
]


def _mutant(old, new):
    src = inspect.getsource(pa_oracle)
    assert src.count(old) == 1, old
    mod = types.ModuleType("pa_oracle_mutant")
    exec(compile(src.replace(old, new), "pa_oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, monkeypatch):
    mod = _mutant(*MUTANTS[name])
    monkeypatch.setattr(pins, "O", mod)
    caught = []
    for pin in PINS:
        try:
            pin()
        except Exception as e:  # AssertionError, or the mutant breaking outright
            caught.append(type(e).__name__)
    assert caught, f"no pin caught mutant {name}"
