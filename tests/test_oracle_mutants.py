"""The pins must catch plausible mistakes in the oracle.

Each case copies ``oracle.c`` to a temporary directory, plants one mistake by
text substitution (on the CPU, never in the real file), compiles it and runs
every pin against it: at least one pin must fail.  A mutant that passes every
pin would mean that part of the oracle is not pinned.
"""
import os

import pytest

import oracle
from pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, text in oracle.c, replacement)
MUTANTS = [
    ("drop_inv_sqrt_d", "lg[j] = dot_row(s, q_spec, q_off, K, k_off) * inv_sqrt_d;",
     "lg[j] = dot_row(s, q_spec, q_off, K, k_off);"),
    ("lse_sign", "lse[g] = m + log(sum);", "lse[g] = m - log(sum);"),
    ("lse_no_shift", "lse[g] = m + log(sum);", "lse[g] = log(sum);"),
    ("gqa_head_map", "const int h = hk * G + g;\n    const int64_t q_off = ((int64_t)b * s->n_q_heads + h) * d;\n    double* lg",
     "const int h = g * s->n_kv_heads + hk;\n    const int64_t q_off = ((int64_t)b * s->n_q_heads + h) * d;\n    double* lg"),
    ("swap_b_hk_in_k", "const int64_t k_off = (((int64_t)b * s->n_kv_heads + hk) * n + j) * d;",
     "const int64_t k_off = (((int64_t)hk * s->batch + b) * n + j) * d;"),
    ("group_score_logits", "acc += exp(logits[(int64_t)g * n + j] - lse[g]);",
     "acc += logits[(int64_t)g * n + j];"),
    ("group_score_first_head_only", "acc += exp(logits[(int64_t)g * n + j] - lse[g]);",
     "acc += exp(logits[j] - lse[0]);"),
    ("tiebreak_high_index", "return (p->j < q->j) ? -1 : (p->j > q->j);\n}\n\nstatic int by_index_asc",
     "return (p->j > q->j) ? -1 : (p->j < q->j);\n}\n\nstatic int by_index_asc"),
    ("window_off_by_one", "const int span = s->ctx_len - s->window, k = s->top_k;",
     "const int span = s->ctx_len - s->window + 1, k = s->top_k;"),
    ("select_ascending", "if (p->a > q->a) return -1;\n  if (p->a < q->a) return 1;",
     "if (p->a < q->a) return -1;\n  if (p->a > q->a) return 1;"),
    ("gap_wrong_denominator", "(c[k - 1].a - c[k].a) / c[k - 1].a", "(c[k - 1].a - c[k].a) / c[k].a"),
    ("bf16_shift", "(uint32_t)((const uint16_t*)p)[i] << 16", "(uint32_t)((const uint16_t*)p)[i] << 15"),
    ("attn_window_offset", "const int64_t j = (r < n_idx) ? idx[r] : (n - n_win + (r - n_idx));\n      e[r]",
     "const int64_t j = (r < n_idx) ? idx[r] : (n - n_win + (r - n_idx) - 1);\n      e[r]"),
    ("attn_no_normalise", "const double p = exp(e[r] - m) / z;", "const double p = exp(e[r] - m);"),
    ("attn_v_unit", "o[t] += p * widen(V, s->dtype, (unit_row0 + j) * d + t);",
     "o[t] += p * widen(V, s->dtype, j * d + t);"),
    ("attn_no_scale", "e[r] = dot_row(s, q, q_off, K, (unit_row0 + j) * d) * inv_sqrt_d;",
     "e[r] = dot_row(s, q, q_off, K, (unit_row0 + j) * d);"),
    ("attn_drop_window", "const int64_t n_win = include_window ? s->window : 0;",
     "const int64_t n_win = 0;"),
    ("landmark_mean_denominator", "L[(int64_t)m * d + t] = acc / chunk;",
     "L[(int64_t)m * d + t] = acc / (chunk + 1);"),
    ("landmark_row_stride", "acc += widen(K, s->dtype, (row0 + (int64_t)m * chunk + r) * d + t);",
     "acc += widen(K, s->dtype, (row0 + (int64_t)m + r) * d + t);"),
    ("landmark_rows_shifted", "rows[i * chunk + r] = c[i].j * chunk + r;",
     "rows[i * chunk + r] = c[i].j * chunk + r + 1;"),
    ("landmark_first_head_only", "for (int m = 0; m < M; ++m) a[m] += exp(lg[m] - l);",
     "if (g == 0) for (int m = 0; m < M; ++m) a[m] += exp(lg[m] - l);"),
    ("landmark_no_scale", "lg[m] = acc * inv_sqrt_d;", "lg[m] = acc;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation site for {name} not unique"
    src = tmp_path / "oracle_mutant.c"
    src.write_text(text.replace(old, new))
    lib = oracle.build(str(src), str(tmp_path / "liboracle_mutant.so"))
    orc = oracle.Oracle(lib)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError, IndexError, OverflowError) as e:  # noqa: PERF203
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
