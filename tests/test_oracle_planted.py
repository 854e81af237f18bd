"""Planted mistakes: each plausible error, put into a copy of the oracle on
the CPU, must make at least one pin (test_oracle.py, test_oracle_out_proj.py,
test_oracle_ln_qkv.py, test_oracle_mlp.py) fail.

The copy is made by a textual edit of the oracle's C source, compiled into a
temporary library and swapped in for the duration of the check; the oracle
itself is never modified.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
from oracle import build as obuild
import test_oracle as T
import test_oracle_out_proj as P
import test_oracle_ln_qkv as N
import test_oracle_mlp as M

# (name, original source fragment, planted fragment)
PLANTS = [
    ("rope_sign", "y[m] = a * c - b * s;", "y[m] = a * c + b * s;"),
    ("rope_interleaved_pairs", "double a = x[m], b = x[m + half];",
     "double a = x[2 * m], b = x[2 * m + 1];"),
    ("no_scale", "sc[j - j0] = acc * scale;", "sc[j - j0] = acc;"),
    ("window_exclusive", "return d <= (int64_t)half_window;", "return d < (int64_t)half_window;"),
    ("band_one_short", "hi = i + half_window + 1;", "hi = i + half_window;"),
    ("positions_not_restarting", "const int64_t i = row - row0;  ", "const int64_t i = row;  "),
    ("values_from_key_block", "+ 2 * c->heads * c->head_dim + c->h * c->head_dim;",
     "+ c->heads * c->head_dim + c->h * c->head_dim;"),
    ("softmax_without_max", "den += exp(scores[j] - m);", "den += exp(scores[j]);"),
    ("freq_exponent", "inv_freq[m] = pow(theta, -2.0 * (double)m / (double)head_dim);",
     "inv_freq[m] = pow(theta, -1.0 * (double)m / (double)head_dim);"),
    ("out_proj_transposed", "acc += ar[c] * w[(int64_t)o * d + c];",
     "acc += ar[c] * w[(int64_t)c * d + o];"),
    ("out_proj_without_residual", "y[k * d + o] = bf16_to_f64(x[t * d + o]) + acc;\n        }\n        free(ar);",
     "y[k * d + o] = acc;\n        }\n        free(ar);"),
    ("ln_unbiased_variance", "const double sd = sqrt(sq / d + eps);",
     "const double sd = sqrt(sq / (d - 1) + eps);"),
    ("ln_eps_outside_sqrt", "const double sd = sqrt(sq / d + eps);",
     "const double sd = sqrt(sq / d) + eps;"),
    ("ln_mean_not_subtracted", "h[c] = (bf16_to_f64(x[c]) - mean) / sd * bf16_to_f64(w[c]);",
     "h[c] = bf16_to_f64(x[c]) / sd * bf16_to_f64(w[c]);"),
    ("ln_weight_ignored", "h[c] = (bf16_to_f64(x[c]) - mean) / sd * bf16_to_f64(w[c]);",
     "h[c] = (bf16_to_f64(x[c]) - mean) / sd;"),
    ("qkv_weight_transposed", "acc += h[c] * wm[(int64_t)j * d + c];",
     "acc += h[c] * wm[(int64_t)c * n_out + j];"),
    ("gelu_tanh_form", "return 0.5 * z * (1.0 + erf(z / sqrt(2.0)));",
     "return 0.5 * z * (1.0 + tanh(sqrt(2.0 / 3.14159265358979323846) * (z + 0.044715 * z * z * z)));"),
    ("mlp_halves_swapped", "m[j] = gelu_erf(g) * u;", "m[j] = gelu_erf(u) * g;"),
    ("round_bf16_seven_bits", "return ldexp(nearbyint(ldexp(m, 8)), e - 8);",
     "return ldexp(nearbyint(ldexp(m, 7)), e - 7);"),
    ("round_bf16_truncates", "return ldexp(nearbyint(ldexp(m, 8)), e - 8);",
     "return ldexp(trunc(ldexp(m, 8)), e - 8);"),
    ("rounded_keys_not_rounded", "        if (c->round_operands)\n            for (int e = 0; e < c->head_dim; e++)\n                k[e] = oracle_round_bf16(k[e]);\n",
     ""),
    ("mlp_without_residual", "y[k * d + o] = bf16_to_f64(x[t * d + o]) + acc;\n        }\n        free(h);",
     "y[k * d + o] = acc;\n        }\n        free(h);"),
]

# every exported function whose ctypes signature the copies must share
_FUNCS = ("oracle_inv_freq", "oracle_rope_row", "oracle_key_counts", "oracle_sdpa_dense",
          "oracle_attention", "oracle_out_proj", "oracle_layernorm", "oracle_ln_qkv",
          "oracle_gelu", "oracle_mlp", "oracle_max_threads", "oracle_attention_rounded",
          "oracle_round_bf16", "oracle_round_bf16_n", "oracle_rope_rows")


def _pins():
    """The pins, as zero-argument callables."""
    table = T._read_table("key_counts.txt")
    out = [
        T.test_worked_example_weights_match_page,
        T.test_dense_rows_sum_to_one_and_mask_zeroes,
        T.test_inv_freq_matches_printed_values,
        T.test_rope_matches_complex_multiplication,
        T.test_rope_relative_position_and_norm,
        T.test_key_counts_closed_form,
        T.test_global_equals_band_covering_sequence,
        T.test_offset_in_pack_does_not_matter,
        T.test_length_one_sequence_returns_its_value,
        T.test_unit_values_give_unit_outputs,
    ]
    out += [P.test_hand_worked_example, P.test_permutation_weight_permutes_columns,
            P.test_zero_weight_returns_the_residual, P.test_power_of_two_diagonal]
    out += [N.test_page_worked_example, N.test_mean_zero_and_spread_closed_form,
            N.test_constant_row_gives_zero, N.test_scale_invariance_without_eps,
            N.test_shift_invariance_on_integers, N.test_weight_scales_positions,
            N.test_matches_torch_layer_norm, N.test_ln_qkv_equals_library_matmul,
            N.test_identity_norm_of_layer_zero, N.test_three_way_split_with_selection_weights]
    out += [M.test_gelu_printed_values, M.test_gelu_matches_torch_exact_form,
            M.test_zero_down_projection_returns_the_residual,
            M.test_selection_weights_give_gelu_times_gate, M.test_matches_library_composition]
    out += [T.test_round_bf16_matches_torch_and_bit_rounding,
            T.test_rounded_operands_at_position_zero_are_exact]
    out += [(lambda lengths=lengths, kind=kind: T.test_rounded_operands_match_bruteforce(lengths, kind))
            for lengths in ([5, 64, 65],) for kind in ("global", "local")]
    out += [(lambda r=r: T.test_key_counts_match_pages(r)) for r in table]
    for lengths in ([5, 64, 65], [130, 7, 200]):
        for kind in ("global", "local"):
            out.append(lambda lengths=lengths, kind=kind: T.test_attention_matches_bruteforce(lengths, kind))
    return out


def _compile_variant(tmp_path, original, planted):
    src = open(obuild.SRC).read()
    assert src.count(original) == 1, f"fragment not unique in the oracle: {original!r}"
    path = tmp_path / "planted.c"
    path.write_text(src.replace(original, planted))
    lib = tmp_path / "libplanted.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-shared",
                    "-fPIC", "-o", str(lib), str(path), "-lm"], check=True)
    return str(lib)


@pytest.mark.parametrize("name,original,planted", PLANTS, ids=[p[0] for p in PLANTS])
def test_planted_mistake_fails_a_pin(tmp_path, name, original, planted):
    good = oracle.lib()
    libpath = _compile_variant(tmp_path, original, planted)
    bad = ctypes.CDLL(libpath)
    for fn in _FUNCS:
        getattr(bad, fn).argtypes = getattr(good, fn).argtypes
        getattr(bad, fn).restype = getattr(good, fn).restype
    failed = []
    oracle._lib = bad
    try:
        for pin in _pins():
            try:
                pin()
            except (AssertionError, ValueError):
                failed.append(pin)
    finally:
        oracle._lib = good
    assert failed, f"planted mistake {name!r} passed every pin"


def test_unplanted_copy_passes_every_pin(tmp_path):
    """Control: the same machinery with no edit passes all pins."""
    good = oracle.lib()
    src = open(obuild.SRC).read()
    path = tmp_path / "copy.c"
    path.write_text(src)
    lib = tmp_path / "libcopy.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-shared",
                    "-fPIC", "-o", str(lib), str(path), "-lm"], check=True)
    copy = ctypes.CDLL(str(lib))
    for fn in _FUNCS:
        getattr(copy, fn).argtypes = getattr(good, fn).argtypes
        getattr(copy, fn).restype = getattr(good, fn).restype
    oracle._lib = copy
    try:
        for pin in _pins():
            pin()
    finally:
        oracle._lib = good
