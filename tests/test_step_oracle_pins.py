"""The cache-append / query-absorption, GEMM and dense-attention oracles
against their pins, and planted mistakes in copies of each that the pins
must catch.  Every mutant keeps its reads in bounds."""
import pytest

import attention_pins
import gemm_pins
import prologue_pins


@pytest.mark.parametrize("check", prologue_pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_prologue_pin(check, oracle_mod):
    check(oracle_mod.prologue())


@pytest.mark.parametrize("check", gemm_pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_gemm_pin(check, oracle_mod):
    check(oracle_mod.gemm_oracle())


@pytest.mark.parametrize("check", attention_pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_attention_pin(check, oracle_mod):
    check(oracle_mod.attention_oracle())


ATTENTION_MUTANTS = {
    "causal_off_by_one": ("const int n = J->causal ? i + 1 : J->S;",
                          "const int n = J->causal ? (i > 0 ? i : 1) : J->S;"),
    "no_scale": ("s[t] = J->scale * dot;", "s[t] = dot;"),
    "lse_log2": ("const double lse = m + log(sum);", "const double lse = m + log2(sum);"),
    "value_from_key_row": ("const uint16_t* v = J->v + (((size_t)b * J->S + t) * J->H + h) * J->dv;",
                           "const uint16_t* v = J->v + (((size_t)b * J->S + 0) * J->H + h) * J->dv;"),
    "head_seq_swapped": ("const uint16_t* q = J->q + (((size_t)b * J->S + i) * J->H + h) * J->dqk;",
                         "const uint16_t* q = J->q + (((size_t)b * J->S + (i % J->S)) * J->H + (h + i) % J->H) * J->dqk;"),
    "short_dot": ("for (int d = 0; d < J->dqk; ++d)", "for (int d = 0; d < J->dqk - 1; ++d)"),
    "weights_not_normalised": ("const double w = exp(s[t] - lse);", "const double w = exp(s[t] - m);"),
}


PROLOGUE_MUTANTS = {
    "append_slot_shift": ("uint16_t* dst = kv_cache + ((size_t)page * PAGE + t % PAGE) * ROW;",
                          "uint16_t* dst = kv_cache + ((size_t)page * PAGE + (t + 1) % PAGE) * ROW;"),
    "append_position_first_token": ("const int t = seqlens[b] - s_q + i;",
                                    "const int t = seqlens[b] - s_q + i - i;"),
    "append_page_of_entry_0": ("block_table[(size_t)b * max_pages + t / PAGE]",
                               "block_table[t / PAGE]"),
    "absorb_w_transposed": ("bf16_value(w[(size_t)d * d_c + c])",
                            "bf16_value(w[((size_t)c * d_nope + d) % ((size_t)d_nope * d_c)])"),
    "absorb_head_0_weights": ("const uint16_t* w = w_uk + (size_t)h * d_nope * d_c;",
                              "const uint16_t* w = w_uk;"),
    "absorb_short_sum": ("for (int d = 0; d < d_nope; ++d)\n                    acc +=",
                         "for (int d = 1; d < d_nope; ++d)\n                    acc +="),
}

GEMM_MUTANTS = {
    "b_transposed": ("b = B[(size_t)k * N + n]", "b = B[(size_t)n * K + k]"),
    "f16_bias_14": ("v = ldexp(1.0 + (double)f / 1024.0, e - 15);",
                    "v = ldexp(1.0 + (double)f / 1024.0, e - 14);"),
    "f16_no_subnormals": ("v = ldexp((double)f, -24);", "v = 0.0;"),
    "f16_sign_dropped": ("return sign ? -v : v;", "return v;"),
    "short_k_loop": ("for (int k = 0; k < K; ++k) {", "for (int k = 0; k < K - 1; ++k) {"),
    "entry_n_for_m": ("J->out[w] = gemm_entry(J->A, J->B, J->N, J->K, J->fmt, m, n);",
                      "J->out[w] = gemm_entry(J->A, J->B, J->N, J->K, J->fmt, m % J->N, n % J->M);"),
}


def _caught(oracle_mod, source, old, new, tmp_path, name, cls, checks):
    src = open(source).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path = tmp_path / f"mutant_{name}.c"
    path.write_text(src.replace(old, new))
    lib = oracle_mod.compile_source(str(path), str(tmp_path / f"libmutant_{name}.so"))
    orc = cls(lib)
    caught = []
    for check in checks:
        try:
            check(orc)
        except AssertionError:
            caught.append(check.__name__)
    return caught


@pytest.mark.parametrize("name", sorted(PROLOGUE_MUTANTS))
def test_prologue_mutant_is_caught(name, tmp_path, oracle_mod):
    old, new = PROLOGUE_MUTANTS[name]
    assert _caught(oracle_mod, oracle_mod.PROLOGUE_SOURCE, old, new, tmp_path, name,
                   oracle_mod.Prologue, prologue_pins.ALL_CHECKS), f"no pin rejects {name}"


@pytest.mark.parametrize("name", sorted(GEMM_MUTANTS))
def test_gemm_mutant_is_caught(name, tmp_path, oracle_mod):
    old, new = GEMM_MUTANTS[name]
    assert _caught(oracle_mod, oracle_mod.GEMM_SOURCE, old, new, tmp_path, name,
                   oracle_mod.Gemm, gemm_pins.ALL_CHECKS), f"no pin rejects {name}"


@pytest.mark.parametrize("name", sorted(ATTENTION_MUTANTS))
def test_attention_mutant_is_caught(name, tmp_path, oracle_mod):
    old, new = ATTENTION_MUTANTS[name]
    assert _caught(oracle_mod, oracle_mod.ATTENTION_SOURCE, old, new, tmp_path, name,
                   oracle_mod.Attention, attention_pins.ALL_CHECKS), f"no pin rejects {name}"
