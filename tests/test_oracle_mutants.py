"""Planted-mistake check for the oracle's pins.

Each case copies attention_oracle.c to a temporary directory, plants one
plausible mistake (dropped scale, off-by-one mask, transposed index, wrong sign,
wrong operand), compiles the copy with gcc and runs the pin battery of
test_oracle_pins.py against it.  Every mutant must fail at least one pin; the
unmodified source must pass them all.  Nothing here touches the committed oracle.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attention_oracle.c")

MUTANTS = {
    "drop_scale_in_scores": ("s[j] = h->scale * dot_rows(", "s[j] = dot_rows("),
    "causal_off_by_one": ("if (h->causal && j > i) return 0;", "if (h->causal && j >= i) return 0;"),
    "kv_len_off_by_one": ("if (j >= h->kv_len) return 0;", "if (j > h->kv_len) return 0;"),
    "block_mask_transposed": ("[(long)(i / h->tile) * h->n_tiles + (j / h->tile)]",
                              "[(long)(j / h->tile) * h->n_tiles + (i / h->tile)]"),
    "dS_sign_rows": ("const double ds = p * (dp[j] - D);", "const double ds = p * (dp[j] + D);"),
    "dS_sign_cols": ("const double ds = p * (dpij - ctx->Dsum[i]);", "const double ds = p * (dpij + ctx->Dsum[i]);"),
    "dq_drops_scale": ("dq[c] += h->scale * ds * kj[c];", "dq[c] += ds * kj[c];"),
    "dk_wrong_operand": ("dk[c] += h->scale * ds * qi[c];", "dk[c] += h->scale * ds * kj[c];"),
    "dv_wrong_operand": ("dv[c] += p * doi[c];", "dv[c] += p * vj[c];"),
    "dP_uses_keys": ("dp[j] = dot_rows(doi, h->v + (long)j * d, d);", "dp[j] = dot_rows(doi, h->k + (long)j * d, d);"),
    "lse_drops_max": ("ctx->lse[item] = m + log(l);", "ctx->lse[item] = log(l);"),
    "output_not_normalised": ("const double p = exp(s[j] - m) / l;\n    const double *vj",
                              "const double p = exp(s[j] - m);\n    const double *vj"),
    "scores_transposed": ("s[j] = h->scale * dot_rows(qi, h->k + (long)j * d, d);",
                          "s[j] = h->scale * dot_rows(h->q + (long)j * d, h->k + (long)i * d, d);"),
}


def _battery():
    """Run the pins; return the names of those that failed."""
    failed = []
    cases = [
        (pins.test_golden_hand_derived, [("non_causal",), ("causal",)]),
        (pins.test_identical_keys_give_mean_of_values, [(False, None), (True, 11)]),
        (pins.test_softmax_rows_sum_to_one, [(True, 23, True)]),
        (pins.test_backward_sum_identities, [(True, 9)]),
        (pins.test_gradients_match_central_differences, [(True, 6, True)]),
        (pins.test_against_torch_sdpa_fp64, [(True, True, True), (False, False, False)]),
    ]
    for fn, params in cases:
        for p in params:
            try:
                fn(*p)
            except (AssertionError, ValueError, FloatingPointError):
                failed.append(f"{fn.__name__}{p}")
    return failed


def _compile(tmp_path, name, text):
    src = tmp_path / f"{name}.c"
    src.write_text(text)
    lib = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-pthread", "-o", str(lib), str(src), "-lm"],
                   check=True)
    return oracle.bind(ctypes.CDLL(str(lib)))


def test_unmodified_oracle_passes_battery(tmp_path, monkeypatch):
    monkeypatch.setattr(oracle, "_lib", _compile(tmp_path, "clean", open(SRC).read()))
    assert _battery() == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path, monkeypatch):
    text = open(SRC).read()
    find, repl = MUTANTS[name]
    assert text.count(find) == 1, f"mutation site for {name} not unique"
    monkeypatch.setattr(oracle, "_lib", _compile(tmp_path, name, text.replace(find, repl)))
    assert _battery(), f"no pin caught the planted mistake {name}"
