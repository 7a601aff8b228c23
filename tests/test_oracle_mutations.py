"""Plants one plausible mistake at a time in a copy of the oracle's C source and
checks that the pin battery rejects every such build."""
import os
import subprocess
import sys

import pytest

import oracle as O

SRC = os.path.join(os.path.dirname(O.__file__), "csa_oracle.c")

MUTATIONS = [
    ("relu_dropped", "const double relu = dot[h] > 0.0 ? dot[h] : 0.0;", "const double relu = dot[h];"),
    ("weight_dropped", "logit += relu * (double)P->w[(int64_t)b * H + h];", "logit += relu;"),
    ("weight_of_row0", "logit += relu * (double)P->w[(int64_t)b * H + h];", "logit += relu * (double)P->w[h];"),
    ("e4m3_bias_8", "v = ldexp(1.0 + (double)m / 8.0, E - 7);", "v = ldexp(1.0 + (double)m / 8.0, E - 8);"),
    ("e4m3_subnormal_exp", "v = ldexp((double)m / 8.0, -6);", "v = ldexp((double)m / 8.0, -7);"),
    ("e4m3_nan_all_E15", "if (E == 15 && m == 7) return NAN;", "if (E == 15) return NAN;"),
    ("e4m3_sign_dropped", "return sign ? -v : v;", "return v;"),
    ("scale_ignored", "const double kd = oracle_e4m3(rec[d]) * s;", "const double kd = oracle_e4m3(rec[d]);"),
    ("scale_big_endian",
     "uint32_t u = (uint32_t)rec[OR_D] | ((uint32_t)rec[OR_D + 1] << 8) |\n               ((uint32_t)rec[OR_D + 2] << 16) | ((uint32_t)rec[OR_D + 3] << 24);",
     "uint32_t u = (uint32_t)rec[OR_D + 3] | ((uint32_t)rec[OR_D + 2] << 8) |\n               ((uint32_t)rec[OR_D + 1] << 16) | ((uint32_t)rec[OR_D] << 24);"),
    ("q_transposed", "qT[d * H + h] = oracle_bf16(qb[h * OR_D + d]);", "qT[d * H + h] = oracle_bf16(qb[d * H + h]);"),
    ("bf16_low_half", "uint32_t u = (uint32_t)h << 16;", "uint32_t u = (uint32_t)h << 15;"),
    ("tie_break_reversed", "return (x->pos > y->pos) - (x->pos < y->pos);", "return (x->pos < y->pos) - (x->pos > y->pos);"),
    ("length_off_by_one",
     "for (int64_t r = 0; r < OR_PAGE && p * OR_PAGE + r < L; ++r) {\n          if (pos) pos[n] = p * OR_PAGE + r;\n          if (col) col[n] = p * OR_PAGE + r;",
     "for (int64_t r = 0; r < OR_PAGE && p * OR_PAGE + r <= L; ++r) {\n          if (pos) pos[n] = p * OR_PAGE + r;\n          if (col) col[n] = p * OR_PAGE + r;"),
    ("resident_column_is_position", "if (col) col[n] = j * OR_PAGE + r;", "if (col) col[n] = p * OR_PAGE + r;"),
    ("page_table_ignored", "int32_t phys = P->page_table[(int64_t)req * P->pt_stride + p];\n  const uint8_t* rec",
     "int32_t phys = (int32_t)p;\n  const uint8_t* rec"),
    ("sigmoid_sign", "return 1.0 / (1.0 + exp(-x));", "return 1.0 / (1.0 + exp(x));"),
    ("padding_score_half", "if (score) score[o] = 0.0;\n        if (logit) logit[o] = -INFINITY;",
     "if (score) score[o] = 0.5;\n        if (logit) logit[o] = -INFINITY;"),
    ("resident_bound_off", "if (p < 0 || p >= npages) {", "if (p < 0 || p > npages) {"),
    ("bad_request_kept", "if (req < 0 || req >= P->num_req) {", "if (req < 0) {"),
    # compressed-K writer
    ("encode_ties_to_odd", "(d == best_d && (c & 1) == 0 && (best & 1) == 1)",
     "(d == best_d && (c & 1) == 1 && (best & 1) == 0)"),
    ("encode_truncates", "if (d < best_d || (d == best_d", "if ((oracle_e4m3((uint8_t)c) <= a && d < best_d) || (d == best_d"),
    ("encode_sign_dropped", "return (uint8_t)(sign | best);", "return (uint8_t)best;"),
    ("writer_scale_240", "const float scale = amax / 448.0f;", "const float scale = amax / 240.0f;"),
    ("writer_scale_big_endian", "rec[OR_D + j] = (uint8_t)(bits >> (8 * j));",
     "rec[OR_D + j] = (uint8_t)(bits >> (8 * (3 - j)));"),
    ("writer_record_off_by_one", "memcpy(kv + phys * page_stride + (p % OR_PAGE) * OR_REC_BYTES, rec, OR_REC_BYTES);",
     "memcpy(kv + phys * page_stride + (p % OR_PAGE + 1) * OR_REC_BYTES, rec, OR_REC_BYTES);"),
    ("writer_page_table_ignored", "const int64_t phys = page_table[r * pt_stride + p / OR_PAGE];",
     "const int64_t phys = p / OR_PAGE;"),
    ("writer_amax_signed", "const float a = fabsf(x[d]);", "const float a = x[d];"),
    ("writer_scale_underflow_kept", "    if (scale == 0.0f) {", "    if (amax == 0.0f) {"),
    # Level-1 recall
    ("recall_max_is_min", "*a = ensemble_mean ? *a + sc : (sc > *a ? sc : *a);",
     "*a = ensemble_mean ? *a + sc : (sc < *a ? sc : *a);"),
    ("recall_mean_not_divided", "const double e = ensemble_mean ? acc[o] / n_layers : acc[o];",
     "const double e = acc[o];"),
    ("recall_threshold_strict", "const int k = e >= threshold || n < sink || n >= L - recent;",
     "const int k = e > threshold || n < sink || n >= L - recent;"),
    ("recall_sink_off_by_one", "const int k = e >= threshold || n < sink || n >= L - recent;",
     "const int k = e >= threshold || n <= sink || n >= L - recent;"),
    ("recall_tail_off_by_one", "const int k = e >= threshold || n < sink || n >= L - recent;",
     "const int k = e >= threshold || n < sink || n > L - recent;"),
    ("recall_sigmoid_skipped", "const double sc = valid[o] ? oracle_sigmoid(logit[o]) : 0.0;",
     "const double sc = valid[o] ? logit[o] : 0.0;"),
    ("recall_unreadable_scores_half", "const double sc = valid[o] ? oracle_sigmoid(logit[o]) : 0.0;",
     "const double sc = valid[o] ? oracle_sigmoid(logit[o]) : 0.5;"),
    ("recall_rows_of_each_layer", "    P.q_len = layers[0].q_len;\n    P.q_req = layers[0].q_req;\n", ""),
    # FP4 (MXFP4) variant
    ("fp4_emax_1", "    e = (E2 - 1) - 2;", "    e = (E2 - 1) - 1;"),
    ("fp4_scale_ceil", "    e = (E2 - 1) - 2;", "    e = E2 - 2;"),
    ("fp4_ties_odd",
     "const double d = fabs(oracle_e2m1(c) - a);\n    if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) {",
     "const double d = fabs(oracle_e2m1(c) - a);\n    if (d < best_d || (d == best_d && (c & 1) == 1 && (best & 1) == 0)) {"),
    ("fp4_subnormal_quarter", "const double v = E == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, E - 1);",
     "const double v = E == 0 ? 0.25 * m : ldexp(1.0 + 0.5 * m, E - 1);"),
    ("fp4_nibbles_swapped", "rec[j] = (uint8_t)((codes[2 * j] & 15) | ((codes[2 * j + 1] & 15) << 4));",
     "rec[j] = (uint8_t)((codes[2 * j + 1] & 15) | ((codes[2 * j] & 15) << 4));"),
    ("fp4_decode_block0_scale", "k[d] = oracle_e2m1(code) * oracle_ue8m0(rec[OR_D / 2 + d / OR_FP4_BLOCK]);",
     "k[d] = oracle_e2m1(code) * oracle_ue8m0(rec[OR_D / 2]);"),
    ("fp4_query_unrounded", "for (int d = 0; d < OR_D; ++d) dot += k[d] * qr[d];",
     "for (int d = 0; d < OR_D; ++d) dot += k[d] * qf[d];"),
    ("fp4_relu_dropped", "const double relu = dot > 0.0 ? dot : 0.0;", "const double relu = dot;"),
    ("fp4_paged_record_stride", "r * (P->format == 1 ? OR_FP4_REC_BYTES : OR_REC_BYTES)", "r * OR_REC_BYTES"),
    ("fp4_paged_query_unrounded", "  if (P->format == 1) {\n    for (int h = 0; h < H; ++h) {",
     "  if (P->format == 2) {\n    for (int h = 0; h < H; ++h) {"),
    ("fp4_writer_row_stride", "kv + phys * page_stride + (p % OR_PAGE) * OR_FP4_REC_BYTES);",
     "kv + phys * page_stride + (p % OR_PAGE) * OR_REC_BYTES);"),
    ("fp4_writer_nonfinite_kept", "    if (!finite) {\n      flags |= OR_FLAG_RANGE;\n      continue;\n    }\n    oracle_fp4_record(",
     "    if (!finite) {\n      flags |= OR_FLAG_RANGE;\n    }\n    oracle_fp4_record("),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {name}"
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"lib{name}.so"
    c.write_text(src.replace(old, new, 1))
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-shared", "-fPIC",
                    "-o", str(so), str(c), "-lm"], check=True)
    # The battery runs in a child process: a mutant may also crash outright (an
    # out-of-range write), which counts as caught as well.
    r = subprocess.run([sys.executable, "-c", _RUNNER, str(so)], capture_output=True, text=True,
                       cwd=os.path.dirname(os.path.dirname(os.path.abspath(__file__))), timeout=600)
    assert r.returncode != 0, f"no pin rejects the planted mistake '{name}':\n{r.stdout}{r.stderr}"
    assert r.returncode == 3 or r.returncode < 0, r.stderr


_RUNNER = """
import sys
sys.path[:0] = ['.', 'tests']
import _pins, oracle as O
o = O.load_build(sys.argv[1])
for pin in _pins.ALL_PINS:
    try:
        pin(o)
    except AssertionError:
        print('caught by', pin.__name__)
        sys.exit(3)
sys.exit(0)
"""
