"""The pins must catch plausible slips: each test here compiles a copy of the
oracle with one deliberate mistake (on the CPU, in a temporary directory) and
checks that at least one pin in test_oracle_pins fails against it."""
import os
import subprocess

import numpy as np

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.cpp")

FWD_PINS = [pins.test_hand_worked_cases, pins.test_gqa_head_map_contiguous_groups,
            pins.test_beta_zero_is_pure_decay, pins.test_orthonormal_keys_store_values_exactly,
            pins.test_reset_at_boundaries_equals_separate_runs, pins.test_empty_documents_pass_the_state_through,
            lambda: pins.test_brute_force_quadratic_form(17, 8, 5)]
BWD_PINS = [pins.test_backward_matches_finite_differences]
# the block recompute of the backward only runs past its first block on documents over 64 tokens
CKPT_PINS = [pins.test_backward_finite_differences_across_checkpoints]

# (name, original text, mutated text, which pins)
MUTANTS = [
    ("decay dropped", "for (int c = 0; c < w; ++c) S[r * w + c] *= a;", "for (int c = 0; c < w; ++c) S[r * w + c] *= 1.0;", FWD_PINS),
    ("correction sign", "d[c] = b * (vt[c] - p[c]);", "d[c] = b * (vt[c] + p[c]);", FWD_PINS),
    ("beta dropped", "d[c] = b * (vt[c] - p[c]);", "d[c] = (vt[c] - p[c]);", FWD_PINS),
    ("output reads k", "double qr = qt[r];", "double qr = kt[r];", FWD_PINS),
    ("interleaved head map", "const int hk = h / G;\n    std::vector<std::vector<double>> fin(N);",
     "const int hk = h % Hk;\n    std::vector<std::vector<double>> fin(N);", FWD_PINS),
    ("no reset", "std::fill(S, S + (size_t)s.Dk * w, 0.0);", "(void)S;", FWD_PINS),
    ("dg sign", "dgt += dS[e] * Sp[e];", "dgt -= dS[e] * Sp[e];", BWD_PINS),
    ("dk drops prediction term", "acc += Sp[(size_t)r * w + c] * dp[c];", "acc += 0.0;", BWD_PINS),
    ("dbeta uses v", "dbt += ddel[c] * vp[c];", "dbt += ddel[c] * vt[c];", BWD_PINS),
    ("decay not carried into dS", "for (size_t e = 0; e < SZ; ++e) dS[e] *= a;", "(void)a;", BWD_PINS),
    ("block restarts from the previous checkpoint", "std::copy(ckpt[bi].begin(), ckpt[bi].end(), states.begin());",
     "std::copy(ckpt[bi ? bi - 1 : 0].begin(), ckpt[bi ? bi - 1 : 0].end(), states.begin());", CKPT_PINS),
    ("block edge off by one", "const int64_t tb = t0 + bi * CK, te = std::min(t1, tb + CK);",
     "const int64_t tb = t0 + bi * CK - (bi > 0 ? 1 : 0), te = std::min(t1, tb + CK);", CKPT_PINS),
    ("checkpoint repeats the previous one", "ckpt[bi] = S;\n        for (int64_t t = t0 + bi * CK;",
     "ckpt[bi] = bi ? ckpt[bi - 1] : S;\n        for (int64_t t = t0 + bi * CK;", CKPT_PINS),
]


@pytest.mark.parametrize("name,orig,mut,which", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(name, orig, mut, which, tmp_path, monkeypatch):
    src = open(SRC).read()
    assert src.count(orig) >= 1, f"mutation site for '{name}' not found"
    bad = src.replace(orig, mut, 1)
    cpp = tmp_path / "mut.cpp"
    cpp.write_text(bad)
    so = tmp_path / "libmut.so"
    subprocess.check_call(["g++", "-O1", "-std=c++17", "-shared", "-fPIC", "-pthread", str(cpp), "-o", str(so)])
    monkeypatch.setattr(oracle, "_lib", oracle.load_library(str(so)))
    failed = []
    for pin in which:
        try:
            pin()
        except AssertionError:
            failed.append(getattr(pin, "__name__", "pin"))
    assert failed, f"no pin caught the '{name}' mutant"
    if which is CKPT_PINS:
        # only the pin that crosses a checkpoint sees these: the short-document pin passes
        pins.test_backward_matches_finite_differences()


# The normalisation of q and k is plain numpy in oracle/__init__.py: its mutants are substituted
# functions, and the finite-difference pin must reject each of them.
L2_MUTANTS = [
    ("projection term dropped", lambda x, dy, eps=1e-6: dy / np.sqrt(np.sum(x * x, -1, keepdims=True) + eps)),
    ("r to the first power in the projection",
     lambda x, dy, eps=1e-6: (lambda r: r * dy - r * np.sum(x * dy, -1, keepdims=True) * x)(
         1.0 / np.sqrt(np.sum(x * x, -1, keepdims=True) + eps))),
    ("projection sign", lambda x, dy, eps=1e-6: (lambda r, y: r * (dy + np.sum(y * dy, -1, keepdims=True) * y))(
        1.0 / np.sqrt(np.sum(x * x, -1, keepdims=True) + eps),
        x / np.sqrt(np.sum(x * x, -1, keepdims=True) + eps))),
]


@pytest.mark.parametrize("name,fn", L2_MUTANTS, ids=[m[0] for m in L2_MUTANTS])
def test_l2norm_pin_catches_mutant(name, fn, monkeypatch):
    monkeypatch.setattr(oracle, "l2norm_rows_bwd", fn)
    with pytest.raises(AssertionError):
        pins.test_l2norm_rows_bwd_matches_finite_differences()
