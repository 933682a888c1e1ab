"""Mutation test of the oracle's pins: plausible mistakes planted in a copy of
the oracle's C source (a swapped index, a dropped term, a wrong operand or
sign) must each make at least one pin of tests/test_oracle.py fail.

Each mutant is compiled with gcc into a temporary library and its pins run
in a subprocess (so a mutant that crashes also counts as caught).  Nothing
here touches the GPU; the real oracle is never modified.
"""
import os
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

# (name, text in pgd_oracle.c, replacement, replace every occurrence?)
MUTANTS = [
    ("page index takes t % BS", "MB + t / BS];", "MB + t % BS];", False),
    ("row within the page takes t / BS", "(t % BS) * x.token", "(t / BS) * x.token", False),
    ("head and token strides swapped", "g * x.head + (t % BS) * x.token",
     "g * x.token + (t % BS) * x.head", False),
    ("weights: KV head h % Hkv", "s, h / (Hq / Hkv), L, D, BS, MB);", "s, h % Hkv, L, D, BS, MB);",
     False),
    ("decode: KV head h % Hkv",
     "int g = h / G;\n        long L = seq_lens[s];\n        double *o = out + sh * D;",
     "int g = h % Hkv;\n        long L = seq_lens[s];\n        double *o = out + sh * D;", False),
    ("scale dropped", "z[t] = scale * dot;", "z[t] = dot;", False),
    ("q . q instead of q . k",
     "dot += g_h2d[qh[d]] * g_h2d[kt[d]];\n        z[t]",
     "dot += g_h2d[qh[d]] * g_h2d[qh[d]];\n        z[t]", False),
    ("softmax exponent sign flipped", "exp(z[t] - zmax)", "exp(zmax - z[t])", True),
    ("max taken as min", "if (z[t] > zmax)", "if (z[t] < zmax)", False),
    ("V read from the K cache",
     "kv_row(v_cache, x, block_tables, s, t, g, BS, MB);\n            for (int d = 0; d < D; ++d)\n                o[d] += w * g_h2d[vt[d]];",
     "kv_row(k_cache, x, block_tables, s, t, g, BS, MB);\n            for (int d = 0; d < D; ++d)\n                o[d] += w * g_h2d[vt[d]];", False),
    ("partials: log2(e) dropped", "exp2(z[t] * log2e - m)", "exp2(z[t] - m)", True),
    ("partials: output not normalised",
     "                o[d] /= l;\n            m_out", "\n            m_out", False),
    ("reduce: exp-sum weight dropped", "double w = l * exp2(", "double w = exp2(", False),
    ("reduce: partial outputs unweighted", "o[d] += w * o_in[", "o[d] += o_in[", False),
    ("online: running sum not rescaled", "l = alpha * l + p;", "l = l + p;", False),
    ("fp16 exponent bias off by one", "expo - 25", "expo - 24", False),
    ("page reads one past the end", "j < npages ? block_tables", "j <= npages ? block_tables",
     False),
    ("append row off by one", "((L - 1) % BS) * x.token", "(L % BS) * x.token", False),
    ("varlen: position one early", "- n + (r - cu_q[s]);", "- n + (r - cu_q[s]) - 1;", False),
    ("varlen: causal bound dropped", "long count = pos + 1;", "long count = seq_lens[s];",
     False),
    ("varlen: query row of the sequence, not of the token", "logits(z, q + rh * D,",
     "logits(z, q + ((long)s * Hq + h) * D,", False),
    ("varlen: owner of a row off by one", "while (cu_q[s + 1] <= r)", "while (cu_q[s + 1] < r)",
     False),
    ("q8: scale and bias swapped", "meta[2 * gidx]) * codes[i] +\n               oracle_bf16_to_double(meta[2 * gidx + 1]);",
     "meta[2 * gidx + 1]) * codes[i] +\n               oracle_bf16_to_double(meta[2 * gidx]);", False),
    ("q8: V dequantised with the K metadata",
     "                                  v_meta + pp * mx.page", "                                  k_meta + pp * mx.page",
     False),
    ("q8: pairs' head and token strides swapped", "k_meta + pp * mx.page + g * mx.head + (t % BS) * mx.token",
     "k_meta + pp * mx.page + g * mx.token + (t % BS) * mx.head", False),
    ("q8: bf16 bits shifted by 15", "(uint32_t)h << 16", "(uint32_t)h << 15", False),
    ("quantiser: codes truncated", "float t = rintf(diff / S);", "float t = truncf(diff / S);",
     False),
    ("quantiser: ties rounded up", "float t = rintf(diff / S);", "float t = floorf(diff / S + 0.5f);",
     False),
    ("quantiser: 256 steps", "range / 255.0f", "range / 256.0f", False),
    ("quantiser: bias from the maximum", "bb = f32_to_bf16_rne(mn)", "bb = f32_to_bf16_rne(mx)",
     False),
    ("quantiser: bf16 truncated", "    u += 0x7FFFu + ((u >> 16) & 1u);\n", "", False),
    ("quantiser: codes from the unrounded bias", "float diff = (float)g_h2d[x[i]] - B;",
     "float diff = (float)g_h2d[x[i]] - mn;", False),
    ("quantiser: row within the page off by one", "h * cx.head + row * cx.token;",
     "h * cx.head + ((row + 1) % BS) * cx.token;", False),
    ("append q8: newest row one late", "(int32_t)(page * (long)BS + (L - 1) % BS)",
     "(int32_t)(page * (long)BS + L % BS)", False),
]


def _pins():
    import test_oracle as T
    import test_oracle_varlen as V
    import test_oracle_q8 as Q
    import test_oracle_quantise as Z
    return [
        ("half decoding", T.test_half_decoding_matches_numpy),
        ("hand case 0", lambda: T.test_hand_cases(0)),
        ("hand case 1", lambda: T.test_hand_cases(1)),
        ("sdpa 8/2 BS4", lambda: T.test_dense_sdpa_special_case(8, 2, 4)),
        ("sdpa 6/1 BS8", lambda: T.test_dense_sdpa_special_case(6, 1, 8)),
        ("length one", T.test_length_one_returns_v),
        ("constant v", T.test_constant_v),
        ("weights sum", T.test_weights_sum_to_one),
        ("weights dense", T.test_weights_match_dense_softmax),
        ("scale zero", T.test_scale_zero_gives_mean),
        ("gqa mapping", T.test_gqa_head_mapping),
        ("zero length", T.test_zero_length),
        ("page permutation", T.test_page_permutation_invariance),
        ("poison", T.test_poison_never_read),
        ("online", T.test_online_log2_equals_definition),
        ("split P=7", lambda: T.test_split_invariance(7)),
        ("split P=100", lambda: T.test_split_invariance(100)),
        ("merge empty", T.test_merge_skips_empty_partitions),
        ("append rows", T.test_append_writes_only_the_newest_rows),
        ("append closed forms", T.test_append_then_decode_closed_forms),
        ("strided layouts", T.test_strided_layouts_equal_head_major),
        ("strided append", T.test_strided_append_equals_head_major_append),
        ("varlen hand case", V.test_hand_case),
        ("varlen sdpa", lambda: V.test_dense_causal_sdpa(8, 2, 4)),
        ("varlen prefix decode", V.test_each_row_is_a_decode_of_its_prefix),
        ("varlen n = 1", V.test_single_token_rows_equal_decode),
        ("varlen prompt row 0", V.test_prompt_first_row_is_v0),
        ("varlen permutation", V.test_page_permutation_invariance),
        ("q8 worked example", Q.test_worked_example),
        ("q8 bf16", Q.test_bf16_decoding_matches_torch),
        ("q8 exact fp16", Q.test_equals_fp16_decode_on_exact_values),
        ("q8 sdpa", lambda: Q.test_dense_sdpa_on_dequantised_values(8, 2, 8)),
        ("q8 strided", lambda: Q.test_strided_q8_equals_head_major(128, 8)),
        ("q8 strided append", Q.test_strided_q8_append_equals_head_major),
        ("quantise example", Z.test_worked_example_inverted),
        ("quantise grid", Z.test_exact_grid),
        ("quantise ties", Z.test_ties_go_to_even),
        ("quantise constant", Z.test_constant_group),
        ("quantise bound", Z.test_round_trip_bound),
        ("quantise pair", Z.test_pair_is_bf16_of_min_and_step),
        ("quantise rows", Z.test_rows_land_at_their_slots),
        ("quantise append", Z.test_append_is_the_newest_row),
        ("quantise stored bias", Z.test_codes_count_from_the_stored_bias),
    ]


def _run_pins(lib_path):
    """Subprocess body: run every pin against the library; print the failures."""
    sys.path.insert(0, HERE)
    sys.path.insert(0, ROOT)
    import oracle
    failed = []
    with oracle.using(lib_path):
        for name, pin in _pins():
            try:
                pin()
            except Exception as e:  # an assertion or the oracle rejecting its own input
                failed.append(f"{name}: {type(e).__name__}")
    print("FAILED:" + "|".join(failed))


def test_unmutated_copy_passes_every_pin(tmp_path):
    import oracle
    so = oracle.compile_source(oracle.source_text(), str(tmp_path / "same.so"))
    r = subprocess.run([sys.executable, __file__, so], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    assert "FAILED:\n" in r.stdout or r.stdout.strip() == "FAILED:", r.stdout


@pytest.mark.parametrize("name,find,repl,all_", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, find, repl, all_, tmp_path):
    import oracle
    src = oracle.source_text()
    assert find in src, f"mutation target of '{name}' not found"
    if not all_:
        assert src.count(find) >= 1
    mutated = src.replace(find, repl) if all_ else src.replace(find, repl, 1)
    assert mutated != src
    so = oracle.compile_source(mutated, str(tmp_path / "mutant.so"))
    r = subprocess.run([sys.executable, __file__, so], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    if r.returncode != 0:
        return  # the mutant crashed the pins: caught
    line = [l for l in r.stdout.splitlines() if l.startswith("FAILED:")][-1]
    caught = [x for x in line[len("FAILED:"):].split("|") if x]
    assert caught, f"mutant '{name}' passed every pin"


if __name__ == "__main__":
    _run_pins(sys.argv[1])
