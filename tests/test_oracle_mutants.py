"""Planted mistakes: each mutant copy of the oracle must fail at least one pin.

A copy of ``oracle/attn_ref.c`` is edited in a temporary directory (one
plausible slip per mutant), compiled with gcc, swapped in through
``oracle.use_library`` and run through the pins of ``test_oracle.py``.  The
real oracle source is never modified.  CPU only.
"""
import os
import subprocess

import pytest

import oracle
import test_oracle as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_ref.c")

MUTANTS = {
    "scale_dropped": ("double s = scale * dot;", "double s = dot;"),
    "score_sign": ("double s = scale * dot;", "double s = -scale * dot;"),
    "values_as_keys": ("const double *k_row = kmat + j * d;",
                       "const double *k_row = vmat + j * d;"),
    "causal_reversed": ("if (causal && i + 1 < hi) hi = i + 1;",
                        "if (causal && i > lo) lo = i;"),
    "causal_no_diagonal": ("if (causal && i + 1 < hi) hi = i + 1;",
                           "if (causal && i + 1 < hi) hi = (i > 0 ? i : 1);"),
    "window_left_off_by_one": ("if (wl >= 0 && i - wl > lo) lo = i - wl;",
                               "if (wl >= 0 && i - wl + 1 > lo) lo = i - wl + 1;"),
    "window_right_ignored": ("if (wr >= 0 && i + wr + 1 < hi) hi = i + wr + 1;",
                             "if (0) hi = i + wr + 1;"),
    "gqa_head_mapping": ("long bh = b * H + h, bkv = b * H_kv + h / group;",
                         "long bh = b * H + h, bkv = b * H_kv + h % H_kv;"),
    "lse_base2": ("double lse = m + log(sum);", "double lse = m + log2(sum);"),
    "lse_without_max": ("double lse = m + log(sum);", "double lse = log(sum);"),
    "no_max_subtraction": ("sum += exp(scores[j] - m);", "sum += exp(scores[j]);"),
    "unnormalised_output": ("double p = exp(scores[j] - lse);",
                            "double p = exp(scores[j] - m);"),
    "varlen_kv_head": ("gather_rows(k + (k0 * H_kv + hk) * d",
                       "gather_rows(k + (k0 * H_kv + h % H_kv) * d"),
    "varlen_row_stride": ("gather_rows(q + (q0 * H + h) * d, H * d,",
                          "gather_rows(q + (q0 * H + h) * d, d,"),
    "varlen_lse_layout": ("lse + h * total_q + q0 + i", "lse + (q0 + i) * H + h"),
    "varlen_global_positions": ("key_range(nk, i + nk - nq, causal, wl, wr, &j0, &j1);",
                                "key_range(nk, i + q0 + nk - nq < nk ? i + q0 + nk - nq : nk - 1,"
                                " causal, wl, wr, &j0, &j1);"),
    "varlen_top_left_alignment": ("key_range(nk, i + nk - nq, causal, wl, wr, &j0, &j1);",
                                  "key_range(nk, i, causal, wl, wr, &j0, &j1);"),
    "varlen_used_k_ignored": ("seq_rows(cu_k, used_k,", "seq_rows(cu_k, NULL,"),
    "varlen_key_rows_from_query_offsets": ("        seq_rows(cu_k, used_k, b, total_k, &k0, &nk);\n"
                                           "        if (nq == 0) continue;",
                                           "        seq_rows(cu_k, used_k, b, total_k, &k0, &nk);\n"
                                           "        k0 = q0;\n        if (nq == 0) continue;"),
    "bwd_dk_unscaled": ("dkj[c] += scale * ds * qi[c];", "dkj[c] += ds * qi[c];"),
    "bwd_rowsum_without_p": ("dsi += exp(s[j] - l) * dp;", "dsi += dp;"),
    "bwd_dv_from_ds": ("dvj[c] += p * doi[c];", "dvj[c] += ds * doi[c];"),
    "bwd_key_mask_ignored": ("if (j < j0 || j >= j1) continue;", "if (j < 0) continue;"),
    "bwd_dq_transposed": ("dqi[c] += scale * ds * kd[j * d + c];",
                          "dqi[c] += scale * ds * vd[j * d + c];"),
    "bwd_qk_top_left_alignment": ("const long shift = Nk - Nq;", "const long shift = 0;"),
    "bwd_qk_shift_sign": ("const long shift = Nk - Nq;", "const long shift = Nq - Nk;"),
    "bwd_qk_key_pass_unshifted": ("key_range(Nk, i + shift, causal, wl, wr, &j0, &j1);\n"
                                  "                    if (j < j0 || j >= j1) continue;",
                                  "key_range(Nk, i, causal, wl, wr, &j0, &j1);\n"
                                  "                    if (j < j0 || j >= j1) continue;"),
    "e4m3_bias": ("else mag = ldexp(8.0 + mant, expo - 10);",
                  "else mag = ldexp(8.0 + mant, expo - 11);"),
    "e4m3_subnormal": ("if (expo == 0) mag = ldexp((double)mant, -9);",
                       "if (expo == 0) mag = ldexp((double)mant, -10);"),
    "fp8_descale_v_dropped": ("vd[t] = dv * e4m3_to_double(v[bkv * slice + t]);",
                              "vd[t] = e4m3_to_double(v[bkv * slice + t]);"),
    "bf16_decoder_shift": ("uint32_t bits = (uint32_t)b << 16;",
                           "uint32_t bits = (uint32_t)b << 15;"),
    "half_decoder_bias": ("expo - 25", "expo - 24"),
}

PIN_CALLS = [
    (pins.test_golden_hand_worked, dict(path="f64", causal=False)),
    (pins.test_golden_hand_worked, dict(path="f64", causal=True)),
    (pins.test_golden_hand_worked, dict(path="bf16", causal=True)),
    (pins.test_golden_hand_worked, dict(path="fp16", causal=False)),
    (pins.test_decoder_exhaustive, dict(dtype=pins.torch.float16)),
    (pins.test_decoder_exhaustive, dict(dtype=pins.torch.bfloat16)),
    (pins.test_matches_torch_sdpa_f64, dict(shape=(2, 3, 33, 16), causal=False)),
    (pins.test_matches_torch_sdpa_f64, dict(shape=(2, 3, 33, 16), causal=True)),
    (pins.test_large_scores_no_overflow, {}),
    (pins.test_probabilities_sum_to_one, dict(causal=True)),
    (pins.test_causal_row_zero, {}),
    (pins.test_zero_queries_closed_form, dict(causal=True)),
    (pins.test_single_key_closed_form, {}),
    (pins.test_window_matches_sdpa_mask, dict(causal=False)),
    (pins.test_window_closed_forms, {}),
    (pins.test_grouped_heads_equal_repeated_heads, {}),
    (pins.test_varlen_equal_lengths_is_the_batched_definition,
     dict(causal=True, window=(5, 3))),
    (pins.test_varlen_matches_torch_per_sequence, dict(causal=True, window=(4, 2))),
    (pins.test_varlen_zero_queries_closed_form, {}),
    (pins.test_varlen_qk_matches_torch_per_sequence, dict(causal=True, window=(4, 2), case=0)),
    (pins.test_varlen_qk_used_lengths_are_a_prefix, dict(causal=True)),
    (pins.test_varlen_qk_decode_and_zero_query_closed_forms, {}),
    (pins.test_bwd_matches_torch_autograd, dict(causal=True, window=(6, 3), H=4, H_kv=2)),
    (pins.test_bwd_directional_finite_difference, dict(causal=True)),
    (pins.test_bwd_sum_identities, dict(causal=False, window=(5, 2))),
    (pins.test_bwd_qk_matches_torch_autograd, dict(Nq=23, Nk=9, causal=True, window=(4, 2))),
    (pins.test_bwd_qk_matches_torch_autograd, dict(Nq=9, Nk=23, causal=True, window=(-1, -1))),
    (pins.test_bwd_qk_keyless_rows_drop_out, {}),
    (pins.test_e4m3_decoder_exhaustive, {}),
    (pins.test_fp8_matches_torch_on_decoded_inputs, dict(causal=True)),
    (pins.test_fp8_descale_folds_into_scale, {}),
]


def _build_mutant(tmp_path, old, new):
    with open(SRC) as f:
        text = f.read()
    assert text.count(old) >= 1, f"mutation anchor not found: {old!r}"
    src = tmp_path / "attn_ref_mutant.c"
    src.write_text(text.replace(old, new))
    lib = tmp_path / "libattn_ref_mutant.so"
    subprocess.run(["gcc", "-O1", "-std=c99", "-shared", "-fPIC", str(src), "-o",
                    str(lib), "-lm"], check=True, capture_output=True)
    return str(lib)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    path = _build_mutant(tmp_path, old, new)
    caught = []
    oracle.use_library(path)
    try:
        for fn, kwargs in PIN_CALLS:
            try:
                fn(**kwargs)
            except AssertionError:
                caught.append(fn.__name__)
    finally:
        oracle.use_library(None)
    assert caught, f"mutant {name!r} passed every pin"


def test_unmutated_copy_passes_every_pin(tmp_path):
    path = _build_mutant(tmp_path, "double s = scale * dot;", "double s = scale * dot;")
    oracle.use_library(path)
    try:
        for fn, kwargs in PIN_CALLS:
            fn(**kwargs)
    finally:
        oracle.use_library(None)
