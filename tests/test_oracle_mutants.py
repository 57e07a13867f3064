"""Mutation check for the oracle pins (CPU only).

Each case copies oracle/dsa_oracle.c, plants one plausible mistake (a dropped
term, a wrong sign or index, a transposed operand, a reversed tie-break),
compiles the copy and runs tests/test_oracle_pins.py against it in a
subprocess.  The pins must fail for every mutant; the unmodified source must
pass.  Mistakes are planted only in the oracle copy, never in product code.
"""
import os
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(ROOT, "oracle", "dsa_oracle.c")

MUTANTS = {
    "indexer_drop_relu": ("s += w[h] * (dot > 0.0 ? dot : 0.0);", "s += w[h] * dot;"),
    "indexer_drop_weight": ("s += w[h] * (dot > 0.0 ? dot : 0.0);", "s += (dot > 0.0 ? dot : 0.0);"),
    "indexer_ignore_doc_start": ("ki + (int64_t)(start_rows[r] + j) * d", "ki + (int64_t)(j) * d"),
    "indexer_drop_diagonal": ("if (j >= len_rows[r]) {", "if (j + 1 >= len_rows[r]) {"),
    "indexer_transposed_q": ("dot += qi[h * d + c] * k[c];", "dot += qi[c * Hi + h] * k[c];"),
    "topk_tiebreak_reversed": ("return (x->j < y->j) ? -1 : (x->j > y->j);",
                               "return (x->j > y->j) ? -1 : (x->j < y->j);"),
    "topk_ascending_scores": ("if (x->score > y->score) return -1;\n  if (x->score < y->score) return 1;",
                              "if (x->score < y->score) return -1;\n  if (x->score > y->score) return 1;"),
    "topk_unsorted_ids": ("qsort(out, (size_t)n, sizeof(int32_t), cmp_i32_asc);", ""),
    "attn_drop_sink": ("double z = zkv + exp(sk - ref);", "double z = zkv;"),
    "attn_sign_in_exp": ("double p = exp(s[j] - ref);", "double p = exp(ref - s[j]);"),
    "attn_drop_scale": ("s[j] = scale * dot;", "s[j] = dot;"),
    "attn_lse_kv_with_sink": ("if (lse_kv) lse_kv[rh] = ref + log(zkv);", "if (lse_kv) lse_kv[rh] = ref + log(z);"),
    "lse_indexer_prefix_off_by_one": ("while (np < n && slot[np] < indexer_topk) ++np;",
                                      "while (np < n && slot[np] <= indexer_topk) ++np;"),
    "lse_indexer_counts_valid_ids": ("while (np < n && slot[np] < indexer_topk) ++np;",
                                     "while (np < n && np < indexer_topk) ++np;"),
    "lse_indexer_with_sink": ("lse_indexer[rh] = zp > 0.0 ? mp + log(zp) : INFINITY;",
                              "lse_indexer[rh] = zp > 0.0 ? mp + log(zp + exp(sk - mp)) : INFINITY;"),
    "topk_softmax_ignores_start": ("l = scores[(int64_t)r * ld + (idx[(int64_t)r * K + j] - base)];",
                                   "l = scores[(int64_t)r * ld + idx[(int64_t)r * K + j]];"),
    "topk_softmax_lse_over_all_slots": ("for (int j = 0; j < n; ++j) z += exp(logits[(int64_t)r * K + j] - m);",
                                        "for (int j = 0; j < K; ++j) z += exp(logits[(int64_t)r * K + j] - m) + 1e-3;"),
    "topk_softmax_divides_by_max": ("softmax[(int64_t)r * K + j] = j < n ? exp(logits[(int64_t)r * K + j] - lz) : 0.0;",
                                    "softmax[(int64_t)r * K + j] = j < n ? exp(logits[(int64_t)r * K + j] - m) : 0.0;"),
    "compact_keeps_key_count": ("(int64_t)id < key_count", "(int64_t)id <= key_count"),
    "pack_wrong_batch_stride": ("v = b * S + id;", "v = b * W + id;"),
    "metadata_len_off_by_one": ("len[t] = t - cu[b] + 1;", "len[t] = t - cu[b];"),
    "e4m3_bias_eight": ("ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    "e4m3_subnormal_as_normal": ("e == 0 ? ldexp((double)m / 8.0, 1 - 7)", "e == 0 ? ldexp(1.0 + (double)m / 8.0, -7)"),
    "e4m3_no_nan": ("if (e == 15 && m == 7) return NAN;", ""),
    "fp8_descale_wrong_row": ("out[r * len + i] = oracle_e4m3_value(codes[r * len + i]) * (double)scales[r];",
                              "out[r * len + i] = oracle_e4m3_value(codes[r * len + i]) * (double)scales[0];"),
    "e8m0_bias_126": ("return ldexp(1.0, (int)e - 127);", "return ldexp(1.0, (int)e - 126);"),
    "e8m0_no_nan": ("  if (e == 255) return NAN;\n  return ldexp", "  return ldexp"),
    "mxfp8_block_of_16": ("oracle_e8m0_value(scales[r * nb + i / 32])", "oracle_e8m0_value(scales[r * nb + i / 16])"),
    "mxfp8_scale_row_ignored": ("oracle_e8m0_value(scales[r * nb + i / 32])", "oracle_e8m0_value(scales[i / 32])"),
    "bwd_drop_delta": ("const double ds = p * (dp - delta);", "const double ds = p * dp;"),
    "bwd_dq_without_scale": ("for (int c = 0; c < Dqk; ++c) dq[c] += scale * ds * k[c];",
                             "for (int c = 0; c < Dqk; ++c) dq[c] += ds * k[c];"),
    "bwd_drop_value_grad": ("for (int c = 0; c < Dv; ++c) g[c] += p * dout[c];", ""),
    "bwd_sink_sign": ("dsink[h] += -exp(sk - L) * delta;", "dsink[h] += exp(sk - L) * delta;"),
    "bwd_normaliser_without_sink": ("const double p = exp(scale * dot - L);", "const double p = exp(scale * dot - lkv);"),
    "ratio_drop_plus_one": ("const int64_t num = off + (t - cu_q[b]) + 1;",
                            "const int64_t num = off + (t - cu_q[b]);"),
    "ratio_ceil_not_floor": ("int64_t bound = num >= 0 ? num / ratio : -((-num + ratio - 1) / ratio);",
                             "int64_t bound = num >= 0 ? (num + ratio - 1) / ratio : -((-num) / ratio);"),
    "ratio_no_clamp_to_prefix": ("if (bound > seqlen_k) bound = seqlen_k;", ""),
    "ratio_ignores_offset": ("const int64_t off = q_off ? q_off[b] : 0;", "const int64_t off = 0;"),
    "ratio_start_from_queries": ("start[t] = cu_k[b];", "start[t] = cu_q[b];"),
}


def _build(tmp_path, text, name):
    c = tmp_path / f"{name}.c"
    c.write_text(text)
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", "-o", str(so), str(c), "-lm"],
                   check=True, capture_output=True)
    return str(so)


def _run_pins(lib):
    env = dict(os.environ, DSA_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(HERE, "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode


def test_unmodified_oracle_passes_pins(tmp_path):
    assert _run_pins(_build(tmp_path, open(SRC).read(), "orig")) == 0


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    src = open(SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    assert _run_pins(_build(tmp_path, src.replace(old, new), name)) != 0, f"pins missed mutant {name}"
