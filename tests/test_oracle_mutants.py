"""Planted mistakes in the oracle, on the CPU: every mutant below of oracle/pg_oracle.c or of
oracle/dense.py must fail at least one of the independent pins (test_oracle_pins.py,
test_nf4_export_pins.py, test_fp8_pins.py), which check the oracle against what the pages and
the mathematics fix. The stored hash-version-1 values are left out: they were written by the
oracle itself and any change at all would fail them.

Each C mutant is compiled from a copy of the source into a temporary directory and loaded in
place of the oracle's library for that test only."""
import numpy as np
import pytest

from oracle import dense
from oracle import oracle as orc
from tests import test_fp8_pins as F8
from tests import test_nf4_export_pins as NX
from tests import test_oracle_pins as P

# (what the mistake is, text of pg_oracle.c, the text that replaces it); each text occurs once
C_MUTANTS = [
    ("page row with K and S swapped",
     "((uint64_t)p * d->K + k) * d->S + slot", "((uint64_t)p * d->S + k) * d->K + slot"),
    ("page index modulo one page too many", "% d->pages[o];", "% (d->pages[o] + 1u);"),
    ("slot modulo one slot too few",
     "% (uint32_t)d->S;", "% (uint32_t)(d->S > 1 ? d->S - 1 : 1);"),
    ("suffix window shifted one token back",
     "int64_t src = b * L + (t - j);", "int64_t src = b * L + (t - j > 0 ? t - j - 1 : 0);"),
    ("positions before the sequence read as token 0",
     "if (t - j < 0) { c[j] = ORC_PAD; continue; }", "if (t - j < 0) { c[j] = 0; continue; }"),
    ("canonical map not applied",
     "c[j] = canon_map ? canon_map[x] : (uint32_t)x;", "c[j] = (uint32_t)x;"),
    ("n-gram hashed without its oldest token",
     "for (int j = 0; j < n; ++j) h ^=", "for (int j = 0; j + 1 < n; ++j) h ^="),
    ("all heads of an order share one slot hash",
     "uint32_t slot = orc_fold32(orc_hash64(d->seed, 1, o, k, nord, c))",
     "uint32_t slot = orc_fold32(orc_hash64(d->seed, 1, o, 0, nord, c))"),
    ("sign taken from the next element's bit",
     "return (int)((words[i / 64] >> (i % 64)) & 1ull);",
     "return (int)((words[i / 64] >> ((i + 1) % 64)) & 1ull);"),
    ("signs never applied", "return (int)((words[i / 64] >> (i % 64)) & 1ull);", "return 0 * i + 0 * (int)words[0];"),
    ("flat sum subtracts the later orders", "acc = (o == 0) ? v : acc + v;", "acc = (o == 0) ? v : acc - v;"),
    ("heads concatenated head-major", "(int64_t)(o * H + k) * r + i", "(int64_t)(k * O + o) * r + i"),
    ("Engram subtables taken head-major",
     "    for (int i = 0; i < d->num_orders; ++i)\n      for (int j = 0; j < d->K; ++j) {\n"
     "        if (i == o && j == k) return base;",
     "    for (int j = 0; j < d->K; ++j)\n      for (int i = 0; i < d->num_orders; ++i) {\n"
     "        if (i == o && j == k) return base;"),
    ("NF4 nibbles swapped",
     "int code = (i % 2 == 0) ? (byte & 0x0F) : (byte >> 4);",
     "int code = (i % 2 == 0) ? (byte >> 4) : (byte & 0x0F);"),
    ("NF4 scale read big-endian",
     "(uint16_t)(row[32] | ((uint16_t)row[33] << 8))", "(uint16_t)(row[33] | ((uint16_t)row[32] << 8))"),
    ("one NF4 level one ulp off", "0xbf3239b1u", "0xbf3239b2u"),
    ("bf16 conversion truncates", "u += 0x7FFFu + lsb;", "u += 0u * lsb;"),
    ("fp16 exponent bias off by one", "((e + 112u) << 23)", "((e + 111u) << 23)"),
    ("splitmix64 first shift off by one",
     "z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;", "z = (z ^ (z >> 29)) * 0xBF58476D1CE4E5B9ull;"),
    ("multipliers not forced odd",
     "return orc_mix64(seed + ORC_GOLDEN * (1ull + fid)) | 1ull;",
     "return orc_mix64(seed + ORC_GOLDEN * (1ull + fid)) & ~1ull;"),
    ("teaching bucket with its operands swapped", "(3ull * a + b) % m", "(3ull * b + a) % m"),
    ("NF4 export: ties go to the higher code", "if (dk < dbest) {", "if (dk <= dbest) {"),
    ("fp16 scale rounded toward zero",
     "if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1u;", "(void)rem;"),
    ("E4M3 encoding with exponent bias 8",
     "uint32_t h = (a >> 20) - ((127u - 7u) << 3);", "uint32_t h = (a >> 20) - ((127u - 8u) << 3);"),
    ("E4M3 decoding with exponent bias 6",
     "else v = bits_to_f32(((e + 120u) << 23) | (m << 20));",
     "else v = bits_to_f32(((e + 121u) << 23) | (m << 20));"),
    ("FP8 row scale from 240 instead of 448", "const float s = a / 448.0f;", "const float s = a / 240.0f;"),
    ("the largest out-of-range position reported",
     "if (bad < 0 || src < bad) bad = src;", "if (bad < 0 || src > bad) bad = src;"),
    ("Engram head reduced modulo the previous head's subtable size",
     "% d->rows[o][k];", "% d->rows[o][k > 0 ? k - 1 : 0];"),
    ("fp16 subnormals scaled by 2^-23", "(float)m * bits_to_f32(0x33800000u)", "(float)m * bits_to_f32(0x34000000u)"),
    ("NF4 export of a zero row with code 8", "code[i] = 7;", "code[i] = 8;"),
    ("E4M3 saturating only past 480 (464 .. 480 round to the NaN pattern)",
     "if (a > 0x43E80000u)", "if (a > 0x43F00000u)"),
]


def _silu_negated(c):
    c = np.asarray(c, np.float64)
    return c * (1.0 / (1.0 + np.exp(c)))


def _rmsnorm_eps_outside(z, gamma, eps):
    z = np.asarray(z, np.float64)
    return z / (np.sqrt(np.mean(z * z, axis=-1, keepdims=True)) + eps) * np.asarray(gamma, np.float64)


def _rmsnorm_sum(z, gamma, eps):
    z = np.asarray(z, np.float64)
    return z / np.sqrt(np.sum(z * z, axis=-1, keepdims=True) + eps) * np.asarray(gamma, np.float64)


def _fetch_rows_shifted(table_bytes, rows):
    flat = rows.reshape(-1)
    out = np.zeros((flat.size, table_bytes.shape[1]), np.uint8)
    ok = flat != orc.NO_ROW
    out[ok] = table_bytes[np.minimum(flat[ok].astype(np.int64) + 1, table_bytes.shape[0] - 1)]
    return out.reshape(rows.shape + (table_bytes.shape[1],))


def _collisions_keyed_on_head_k(rows):
    r = np.asarray(rows).astype(np.uint64)
    shared = np.zeros(r.shape[1], np.int64)
    for k in range(r.shape[1]):
        _, c = np.unique(r[:, k], return_counts=True)
        shared[k] = int((c.astype(np.int64) * (c.astype(np.int64) - 1) // 2).sum())
    return int(shared[0]), shared


def _python_mutants():
    """(what the mistake is, module, attribute, replacement)"""
    rms, proj, conv = dense.rmsnorm, dense.project, dense.conv_residual
    deq, fp8deq = orc.nf4_dequantize, orc.fp8_dequantize
    return [
        ("rows fetched one row further on", orc, "fetch_rows", _fetch_rows_shifted),
        ("NF4 rows decoded with their nibbles swapped", orc, "nf4_dequantize",
         lambda rows: deq(np.concatenate([((np.asarray(rows)[:, :32] & 15) << 4) | (np.asarray(rows)[:, :32] >> 4),
                                          np.asarray(rows)[:, 32:]], axis=1).astype(np.uint8))),
        ("FP8 rows decoded with the scale applied twice", orc, "fp8_dequantize",
         lambda q, sc: fp8deq(q, sc) * np.asarray(sc, np.float64)[:, None]),
        ("head collisions counted on head k alone", orc, "collision_counts", _collisions_keyed_on_head_k),
    ] + [(what, dense, name, fn) for what, name, fn in _dense_mutants(rms, proj, conv)]


def _dense_mutants(rms, proj, conv):
    return [
        ("SiLU as c * sigmoid(-c)", "silu", _silu_negated),
        ("RMSNorm without its gain", "rmsnorm", lambda z, g, eps: rms(z, np.ones_like(np.asarray(g)), eps)),
        ("RMSNorm with eps outside the root", "rmsnorm", _rmsnorm_eps_outside),
        ("RMSNorm over the sum instead of the mean", "rmsnorm", _rmsnorm_sum),
        ("projection with W's rows reversed", "project", lambda e, W: proj(e, np.asarray(W)[::-1])),
        ("gate without the 1/sqrt(d) scale", "context_gate",
         lambda h, k, gh, gk, eps: dense.sigmoid(np.sum(rms(h, gh, eps) * rms(k, gk, eps), axis=-1))),
        ("conv taps in reverse order", "conv_residual",
         lambda v, a, g, w, dil, eps, H: conv(v, a, g, np.ascontiguousarray(np.asarray(w)[:, ::-1]), dil, eps, H)),
        ("conv without the residual alpha v", "conv_residual",
         lambda v, a, g, w, dil, eps, H: conv(v, a, g, w, dil, eps, H)
         - np.asarray(a, np.float64)[..., None] * np.asarray(v, np.float64)[None]),
    ]


# every pin that checks the oracle against something other than itself, fast ones first;
# parametrised pins at one of their parameter sets
PINS = [
    (P.test_toy_bucket_worked_values, {}),
    (P.test_mix64_matches_splitmix64_reference_outputs, {}),
    (P.test_multipliers_odd_and_distinct, {}),
    (P.test_number_conversions_against_libraries, {}),
    (P.test_nf4_format_arithmetic_and_levels, {}),
    (P.test_nf4_levels_are_qlora_published_table, {}),
    (P.test_nf4_decode_special_rows, {}),
    (P.test_bf16_sign_flip_is_exact, {}),
    (P.test_concat_order_and_sign_flip, {}),
    (P.test_flat_sum_of_two_signed_rows, {}),
    (P.test_pagegram_heads_share_one_page_and_stay_in_range, {"S": 4}),
    (P.test_pagegram_heads_share_one_page_and_stay_in_range, {"S": 15}),
    (P.test_engram_and_flat_rows_inside_their_subtables, {}),
    (P.test_rows_depend_exactly_on_the_suffix_window, {}),
    (P.test_sequences_do_not_leak_into_each_other, {}),
    (P.test_positions_before_the_start_are_padding_not_a_token, {}),
    (P.test_canonical_map_folds_ids_and_is_surjective, {}),
    (P.test_out_of_range_ids_are_reported, {}),
    (P.test_toy_mode_through_the_ngram_window, {}),
    (P.test_slot_count_extremes, {}),
    (P.test_sign_bits_are_balanced, {}),
    (P.test_projection_and_gate_against_torch, {}),
    (P.test_conv_residual_against_torch_conv1d, {"ks": 4, "dil": 3}),
    (P.test_zero_table_leaves_the_residual_stream_unchanged, {}),
    (P.test_zero_conv_weights_give_the_identity_path, {}),
    (P.test_causality_of_the_whole_path, {}),
    (P.test_parameter_budgets_match_the_report, {}),
    (P.test_bucket_loads_are_poisson_like, {}),
    (P.test_collision_counts_equal_brute_force, {"n": 60, "K": 8, "hi": 4, "seed": 3}),
    (P.test_collision_counts_closed_forms, {}),
    (P.test_collision_counts_on_pagegram_rows, {"S": 4}),
    (P.test_pagegram_extra_shared_heads, {"S": 4, "expect": 7 / 4}),
    (P.test_engram_second_head_recollision_is_about_one_over_M, {}),
    (NX.test_fp16_scale_rounding_matches_ieee_conversion, {}),
    (NX.test_zero_row_is_exact, {}),
    (NX.test_rows_of_exact_levels_return_their_codes, {}),
    (NX.test_exact_ties_between_two_levels_take_the_lower_code, {}),
    (NX.test_nibble_order_and_scale_bytes, {}),
    (NX.test_export_is_idempotent_through_the_stored_format, {}),
    (NX.test_error_within_the_quantisation_bound, {"dist": "normal"}),
    (F8.test_e4m3_encoding_matches_torch_below_the_saturation_point, {}),
    (F8.test_e4m3_saturates_where_torch_overflows, {}),
    (F8.test_e4m3_decoding_matches_torch_for_every_byte, {}),
    (F8.test_fp8_rows_zero_row_and_extremes, {}),
    (F8.test_fp8_rows_error_within_the_rounding_bound, {"dist": "normal"}),
]


def _first_failing_pin():
    for fn, kw in PINS:
        try:
            fn(**kw)
        except Exception:       # an assertion, or an error such as a row outside the table
            return fn.__name__
    return None


def test_every_pin_passes_on_the_oracle_as_it_stands():
    assert _first_failing_pin() is None


@pytest.mark.parametrize("what,orig,mut", C_MUTANTS, ids=[m[0] for m in C_MUTANTS])
def test_c_oracle_mistake_fails_a_pin(tmp_path, monkeypatch, what, orig, mut):
    with open(orc._SRC) as f:
        src = f.read()
    assert src.count(orig) == 1, what
    path = tmp_path / "pg_oracle_mutant.c"
    path.write_text(src.replace(orig, mut))
    monkeypatch.setattr(orc, "_SRC", str(path))
    monkeypatch.setattr(orc, "_LIB", str(tmp_path / "liboracle_mutant.so"))
    monkeypatch.setattr(orc, "_lib", None)
    assert _first_failing_pin() is not None, f"no pin fails when the oracle has this mistake: {what}"


@pytest.mark.parametrize("k", range(12))
def test_python_oracle_mistake_fails_a_pin(monkeypatch, k):
    what, module, name, fn = _python_mutants()[k]
    monkeypatch.setattr(module, name, fn)
    assert _first_failing_pin() is not None, f"no pin fails when the oracle has this mistake: {what}"
