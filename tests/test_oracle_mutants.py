"""The pins must catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of the oracle's C source (on the CPU),
builds it, swaps it in, and runs the pin battery of test_oracle_pins.py; at
least one pin must fail.  No GPU.
"""
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "ulysses_oracle.c")

# (name, text in the source, replacement): one plausible slip each.
MUTANTS = [
    ("causal mask off by one", "long n_keys = sh->causal ? i + 1 : S;\n    attend_row(D, n_keys, qi",
     "long n_keys = sh->causal ? i : S;\n    attend_row(D, n_keys, qi"),
    ("strided head ownership", "(((long)b * Sl + t) * heads + ((long)dst * hp + j)) * D",
     "(((long)b * Sl + t) * heads + ((long)j * P + dst)) * D"),
    ("pieces in reverse source order", "double *to = y + (((long)b * S + ((long)src * Sl + t)) * hp + j) * D;",
     "double *to = y + (((long)b * S + ((long)(P - 1 - src) * Sl + t)) * hp + j) * D;"),
    ("inverse transpose takes the wrong heads", "double *to = x + (((long)b * Sl + t) * heads + ((long)src * hp + j)) * D;",
     "double *to = x + (((long)b * Sl + t) * heads + ((long)j * P + src)) * D;"),
    ("self piece counted as traffic", "      if (src != dst) {\n        long long piece",
     "      {\n        long long piece"),
    ("rope sign flipped", "v[i] = x1 * c[i] - x2 * s[i];", "v[i] = x1 * c[i] + x2 * s[i];"),
    ("rope uses local position", "const double p = (double)r * Sl + t;", "const double p = (double)t;"),
    ("rope frequency schedule", "pow(base, -2.0 * i / D)", "pow(base, -1.0 * i / D)"),
    ("softmax scale dropped", "w[k] = scale * dot;", "w[k] = dot;"),
    ("grouped kv heads interleaved", "return g / (sh->n_head / sh->n_kv_head);", "return g % sh->n_kv_head;"),
    ("lse misses the max", "*lse = m + log(l);", "*lse = log(l);"),
    ("softmax not normalised", "for (int e = 0; e < D; ++e) o[e] /= l;", ""),
    ("backward drops delta", "double ds = p * (dp - dd);", "double ds = p * dp;"),
    ("dk misses the scale", "dkr[e] += sh->scale * ds * qi[e];", "dkr[e] += ds * qi[e];"),
    ("dv uses dS", "dvr[e] += p * doi[e];", "dvr[e] += ds * doi[e];"),
    ("dk/dv causal range off by one", "for (long i = sh->causal ? kk : 0; i < S; ++i)",
     "for (long i = sh->causal ? kk + 1 : 0; i < S; ++i)"),
    ("dq transposed operand", "dqi[e] += sh->scale * ds * kr[e];", "dqi[e] += sh->scale * ds * vr[e];"),
    ("replicated kv-heads dealt round-robin", "const int kv = dst / R;", "const int kv = dst % heads;"),
    ("gradient reduce drops a replica", "for (int j = 0; j < R; ++j) {", "for (int j = 1; j < R; ++j) {"),
    ("replica rank holds the wrong kv-head", "r / (sh->P / sh->n_kv_head);", "r % sh->n_kv_head;"),
]


def battery():
    """Run the pins; return the names of those that failed."""
    cases = [
        ("ownership", lambda: pins.test_ownership_example_matches_page()),
        ("identity", lambda: pins.test_pack_then_unpack_is_identity(4, 1, 7, 8, 3)),
        ("volume", lambda: pins.test_bytes_moved_match_page_formula(4, 2, 3, 8, 4, 2)),
        ("rope-global", lambda: pins.test_rope_position_zero_is_identity_and_positions_are_global()),
        ("rope-norm", lambda: pins.test_rope_preserves_pair_norms_and_inverts()),
        ("rope-relative", lambda: pins.test_rope_scores_depend_on_relative_position_only()),
        ("brute-gqa", lambda: pins.test_oracle_matches_brute_force(2, 2, 6, 4, 2, 6, False, True)),
        ("brute-causal", lambda: pins.test_oracle_matches_brute_force(4, 1, 16, 4, 4, 4, True, True)),
        ("brute-gqa-causal", lambda: pins.test_oracle_matches_brute_force(4, 1, 8, 8, 4, 2, True, False)),
        ("torch", lambda: pins.test_single_rank_matches_torch_sdpa_and_autograd(True)),
        ("closed-forms", lambda: pins.test_closed_forms()),
        ("unsharded", lambda: pins.test_ulysses_equals_unsharded_attention_bit_exact(4, 2, 64, 8, 4, 8, True, True)),
        ("unsharded-replicated", lambda: pins.test_ulysses_equals_unsharded_attention_bit_exact(8, 2, 64, 8, 1, 4, True, True)),
        ("brute-replicated", lambda: pins.test_oracle_matches_brute_force(4, 1, 8, 4, 2, 4, True, True)),
        ("replicated-adjoint", lambda: pins.test_replicated_reduce_is_the_adjoint_of_the_replicating_all_to_all(4, 1, 3, 2, 4)),
    ]
    failed = []
    for name, fn in cases:
        try:
            fn()
        except Exception:  # an assertion, or a mutant that makes a call fail
            failed.append(name)
    return failed


def test_unmutated_oracle_passes_battery():
    assert battery() == []


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {name}"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new, 1))  # first occurrence only
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                           "-o", str(so), str(path), "-lm"])
    saved = oracle._lib
    oracle._lib = oracle.load_library(str(so))
    try:
        failed = battery()
    finally:
        oracle._lib = saved
    assert failed, f"no pin caught the planted mistake: {name}"
