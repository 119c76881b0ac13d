"""Plant one mistake at a time in a copy of the oracle; the pins must catch it.

Every mutant keeps its reads in bounds, so a mutant can only give wrong
numbers, never crash the test process.
"""
import os

import pytest

import oracle_pins

MUTANTS = {
    "no_scale": ("s[t - t0] = J->scale * dot;", "s[t - t0] = dot;"),
    "causal_off_by_one": ("n = J->seqlens[b] - J->s_q + 1 + i;", "n = J->seqlens[b] - J->s_q + i;"),
    "lse_log2": ("const double lse = m + log(sum);", "const double lse = m + log2(sum);"),
    "value_offset": ("o[d] += w * bf16_to_double(vrow[d]);",
                     "o[d] += w * bf16_to_double(vrow[d + 64]);"),
    "weight_sign": ("const double w = exp(s[t - t0] - lse);",
                    "const double w = exp(lse - s[t - t0]);"),
    "no_max_in_sum": ("sum += exp(s[t - t0] - m);", "sum += exp(s[t - t0]);"),
    "q_transposed": ("(((size_t)b * J->s_q + i) * J->h_q + h) * D_QK",
                     "(((size_t)b * J->h_q + h) * J->s_q + i) * D_QK"),
    "slot_shift": ("return J->kv + ((size_t)page * PAGE + (t % PAGE)) * D_QK;",
                   "return J->kv + ((size_t)page * PAGE + ((t + 1) % PAGE)) * D_QK;"),
    "sparse_ignores_list": ("t = J->indices[(size_t)b * J->topk + j];", "t = j;"),
    "sparse_first_entry_list": ("t = J->indices[(size_t)b * J->topk + j];",
                                "t = J->indices[j];"),
    "sparse_count_short": ("n = J->counts[b];", "n = J->counts[b] > 0 ? J->counts[b] - 1 : 0;"),
    "combine_weight": ("const double w = exp(lse_parts[j] - *lse);",
                       "const double w = exp(lse_parts[j] - m);"),
    "dot_short": ("for (int d = 0; d < D_QK; ++d)\n            dot +=",
                  "for (int d = 0; d < D_V; ++d)\n            dot +="),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path, oracle_mod):
    old, new = MUTANTS[name]
    src = open(oracle_mod.SOURCE).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path = tmp_path / f"mutant_{name}.c"
    path.write_text(src.replace(old, new))
    lib = oracle_mod.compile_source(str(path), str(tmp_path / f"libmutant_{name}.so"))
    orc = oracle_mod.Oracle(lib)
    caught = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(orc)
        except AssertionError:
            caught.append(check.__name__)
    assert caught, f"no pin rejects mutant {name}"
