"""Plant plausible mistakes in copies of the oracle source and check a pin fails.

Each mutant is oracle.c with one textual substitution (a dropped term, a wrong
sign, an off-by-one mask, a swapped operand or index), compiled into a temporary
directory.  The real oracle is never modified.
"""
import os

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "causal_off_by_one": ("if (p->causal && j > p->q_offset + i) return 0;",
                          "if (p->causal && j >= p->q_offset + i) return 0;"),
    "causal_ignores_offset": ("if (p->causal && j > p->q_offset + i) return 0;",
                              "if (p->causal && j > i) return 0;"),
    "key_len_off_by_one": ("j >= p->key_len[b]) return 0;", "j > p->key_len[b]) return 0;"),
    "lse_drops_log_l": ("*lse_i = m + log(l);", "*lse_i = m;"),
    "unnormalised_weights": ("const double w = exp(srow[j] - m) / l;",
                             "const double w = exp(srow[j] - m);"),
    "out_uses_k_for_v": ("const double* vj = v + k_at(p, b, j, h);",
                         "const double* vj = k + k_at(p, b, j, h);"),
    "scale_dropped_in_scores": ("srow[j] = p->scale * dot(", "srow[j] = dot("),
    "dq_sign_of_D": ("const double dS = P * (dP - J->D[i - J->i0]);\n            const double* kj",
                     "const double dS = P * (dP + J->D[i - J->i0]);\n            const double* kj"),
    "dkv_sign_of_D": ("const double dS = P * (dP - J->D[i - J->i0]);\n            for",
                      "const double dS = P * (dP + J->D[i - J->i0]);\n            for"),
    "dk_drops_scale": ("dkj[c] += p->scale * dS * qi[c];", "dkj[c] += dS * qi[c];"),
    "dv_uses_dS": ("dvj[c] += P * doi[c];", "dvj[c] += dS * doi[c];"),
    "dq_uses_v": ("const double* kj = J->k + k_at(p, J->b, j, J->h);",
                  "const double* kj = J->v + k_at(p, J->b, j, J->h);"),
    "D_uses_q": ("J->D[i - J->i0] = dot(doi, o, p->d);",
                 "J->D[i - J->i0] = dot(doi, J->q + q_at(p, J->b, i, J->h), p->d);"),
    "head_groups_strided": ("const int r = t / sl, u = t % sl, head = g * hl + j;",
                            "const int r = t / sl, u = t % sl, head = j * N + g;"),
    "shards_interleaved": ("const int r = t / sl, u = t % sl, head = g * hl + j;",
                           "const int r = t % N, u = t / N, head = g * hl + j;"),
    "merge_weight_unnormalised": ("const double w = exp(lses[k * lse_part + li] - total);",
                                  "const double w = exp(lses[k * lse_part + li] - m);"),
    "merge_lse_drops_max": ("const double total = m + log(s);", "const double total = log(s);"),
    "key_mask_ignored": ("if (p->key_mask != NULL && p->key_mask[(size_t)b * p->sk + j] == 0) return 0;",
                         "if (0) return 0;"),
    "key_mask_inverted": ("if (p->key_mask != NULL && p->key_mask[(size_t)b * p->sk + j] == 0) return 0;",
                          "if (p->key_mask != NULL && p->key_mask[(size_t)b * p->sk + j] != 0) return 0;"),
    "key_mask_batch_stride": ("p->key_mask[(size_t)b * p->sk + j] == 0",
                              "p->key_mask[(size_t)j] == 0"),
    "head2seq_groups_strided": ("const int g = head / hl, j = head % hl, t = r * sl + u;",
                                "const int g = head % N, j = head / N, t = r * sl + u;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) >= 1, f"mutation site for {name} not found"
    mutated = tmp_path / "oracle_mutant.c"
    mutated.write_text(text.replace(old, new, 1))
    lib = oracle.open_library(oracle.compile_source(str(mutated), str(tmp_path / "m.so")))
    orc = oracle.Oracle(lib)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_fails_a_generated_property(name, tmp_path):
    """The same mutants against the generated properties of test_oracle_properties.py:
    hypothesis searches (without shrinking) for a case on which the broken oracle
    disagrees with torch's fp64 attention, the split-key merge identity or torch's
    regrouping."""
    from hypothesis import Phase, find, settings
    from hypothesis.errors import NoSuchExample
    from test_oracle_properties import PROPERTIES
    old, new = MUTANTS[name]
    mutated = tmp_path / "oracle_mutant.c"
    mutated.write_text(open(SRC).read().replace(old, new, 1))
    orc = oracle.Oracle(oracle.open_library(
        oracle.compile_source(str(mutated), str(tmp_path / "m.so"))))
    search = settings(max_examples=60, phases=[Phase.generate], derandomize=True,
                      database=None, deadline=None)

    def fails(check, case):
        try:
            check(orc, case)
        except (AssertionError, ValueError):
            return True
        return False

    for strategy, check in PROPERTIES:
        try:
            find(strategy, lambda case, check=check: fails(check, case), settings=search)
            return
        except NoSuchExample:
            continue
    pytest.fail(f"mutant {name} passed every generated property")
