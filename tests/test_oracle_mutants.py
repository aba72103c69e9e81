"""Plant plausible mistakes in copies of the oracle; each must trip a pin.

The mistakes are planted in temporary copies of ``oracle/oracle.c`` on the CPU;
the oracle itself is never modified.
"""
import os
import subprocess

import pytest

import oracle
import oracle_pins as P

MUTANTS = {
    # gather: logical block and in-block offset swapped
    "gather_swap": ("const int32_t logical = t / block_size;",
                    "const int32_t logical = t % block_size;"),
    # gather: rows of a block read in reverse order (stays inside the pool)
    "gather_rows_reversed": ("const int32_t off = t % block_size;",
                             "const int32_t off = (block_size - 1) - t % block_size;"),
    # causal limit one token short
    "causal_off_by_one": ("const int32_t lim = T - n_query_per_seq + j; /* last visible position */",
                          "const int32_t lim = T - n_query_per_seq + j - 1;"),
    # GQA: query heads interleaved across kv heads instead of grouped
    "gqa_interleaved": ("const int32_t qh = h * group + g;",
                        "const int32_t qh = g * num_kv_heads + h;"),
    # scale dropped from the scores
    "no_scale": ("w[t] = scale * dot;", "w[t] = dot;"),
    # softmax normaliser dropped
    "no_normaliser": ("w[t] /= z;", "w[t] /= 1.0;"),
    # append writes one slot too far
    "append_offset": ("const int64_t off = slot % block_size;",
                      "const int64_t off = (slot + 1) % block_size;"),
    # merge: rescale factor with the wrong sign
    "merge_sign": ("const double f = exp(m[i] - M);", "const double f = exp(M - m[i]);"),
    # weighted sum over K instead of V
    "sum_over_k": ("o[d] += w[t] * V[(int64_t)t * head_dim + d];",
                   "o[d] += w[t] * K[(int64_t)t * head_dim + d];"),
    # query/sequence order of the q rows transposed
    "q_row_order": ("const int64_t row = ((int64_t)s * n_query_per_seq + j) * num_q_heads + qh;\n"
                    "                double *o",
                    "const int64_t row = ((int64_t)j * num_seqs + s) * num_q_heads + qh;\n"
                    "                double *o"),
    # partial state: running sum not rescaled by the range maximum
    "partial_no_shift": ("const double e = exp(x[t] - m);", "const double e = exp(x[t]);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    src = open(oracle.SOURCE).read()
    before, after = MUTANTS[name]
    assert src.count(before) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(before, after, 1)
    path = tmp_path / "mut.c"
    path.write_text(mutated)
    lib = tmp_path / "mut.so"
    oracle.build(str(path), str(lib), force=True)
    m = oracle.Oracle(oracle.load(str(lib)))
    failures = []
    for pin in P.ALL_PINS:
        try:
            pin(m)
        except (AssertionError, ValueError) as e:  # a pin caught the mistake
            failures.append(pin.__name__)
    assert failures, f"no pin caught mutant {name}"
