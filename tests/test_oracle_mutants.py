"""Planted mistakes: each mutant of the oracle's C source must fail a pin.

A mutant is the oracle's own source with one plausible slip written into it
(a dropped scale, a flipped exponent, a wrong GQA head, an off-by-one causal
mask (top-left or bottom-right), a bias subtracted or read from the wrong query, a missing normalisation, V swapped for K, a log2 for a log, a missing
Delta or scale in the backward).  Each is compiled with gcc into a temporary
library, swapped in for the real one, and run through a battery of the pins
in test_oracle.py; the test passes only if the battery rejects it.  All on the
CPU; nothing here touches the CUDA path.
"""
import os
import subprocess

import pytest

import oracle
import tests.test_oracle as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

MUTANTS = {
    "dropped_scale": ("s[j] = scale * dot;", "s[j] = dot;"),
    "flipped_exponent": ("s[j] = exp(s[j] - m);", "s[j] = exp(m - s[j]);"),
    "causal_off_by_one": ("return (i + 1 < Nk) ? (i + 1) : Nk;",
                          "return (i + 2 < Nk) ? (i + 2) : Nk;"),
    "gqa_strided_heads": ("const int64_t g = h / G;", "const int64_t g = h % jb->Hkv;"),
    "no_normalisation": ("const double w = s[j] / l;", "const double w = s[j];"),
    "values_are_keys": ("const double *v_row = v_head + j * D;",
                        "const double *v_row = k_head + j * D;"),
    "lse_log2": ("*lse_out = m + log(l);", "*lse_out = m + log2(l);"),
    "bwd_no_delta": ("const double ds = p[j] * (dp[j] - delta);",
                     "const double ds = p[j] * dp[j];"),
    "bwd_dk_unscaled": ("dk_head[j * D + d] += jb->scale * ds * q_row[d];",
                        "dk_head[j * D + d] += ds * q_row[d];"),
    "bwd_dv_transposed": ("dv_head[j * D + d] += p[j] * do_row[d];",
                          "dv_head[j * D + d] += p[j] * q_row[d];"),
    "bottom_right_off_by_one": ("? i + (jb->Nk - jb->Nq) : i;", "? i + (jb->Nk - jb->Nq) - 1 : i;"),
    "bottom_right_as_top_left": ("? i + (jb->Nk - jb->Nq) : i;", "? i : i;"),
    "mask_subtracted": ("if (bias_row) s[j] += bias_row[j];", "if (bias_row) s[j] -= bias_row[j];"),
    "mask_query_stride_ignored": ("+ i * jb->bsq : NULL;\n        fwd_one_row", "+ 0 * jb->bsq : NULL;\n        fwd_one_row"),
    "bwd_mask_ignored": ("if (bias_row) p[j] += bias_row[j];", "if (bias_row) p[j] += 0.0;"),
}


def battery():
    """The pins most likely to see a slip; returns the names that failed."""
    checks = [
        ("hand_fwd", pins.test_hand_worked_example_forward, ()),
        ("hand_bwd", pins.test_hand_worked_example_backward, ()),
        ("sdpa_gqa_causal", pins.test_matches_torch_sdpa_f64, (1, 4, 2, 33, 33, 16, True)),
        ("sdpa_gqa7", pins.test_matches_torch_sdpa_f64, (1, 7, 1, 45, 45, 32, False)),
        ("autograd_gqa", pins.test_backward_matches_torch_autograd, (4, 2, True)),
        ("prefix_means", pins.test_zero_query_causal_gives_prefix_means, ()),
        ("single_key", pins.test_single_key_returns_its_value_row, ()),
        ("bottom_right", pins.test_bottom_right_matches_torch_causal_lower_right,
         (2, 4, 2, 1, 23, 16)),
        ("bottom_right_prefix", pins.test_zero_query_bottom_right_gives_prefix_means, ()),
        ("mask_closed_forms", pins.test_mask_closed_forms, ()),
        ("mask_sdpa", pins.test_mask_matches_torch_sdpa_f64, ((2, 4, 13, 23), "additive", True)),
        ("mask_autograd", pins.test_masked_backward_matches_torch_autograd, ("bool",)),
    ]
    failed = []
    for name, fn, args in checks:
        try:
            fn(*args)
        except AssertionError:
            failed.append(name)
    return failed


@pytest.fixture
def swap_lib(tmp_path, monkeypatch):
    def _swap(mutation):
        src = open(SRC).read()
        old, new = mutation
        assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
        path = tmp_path / "mut.c"
        path.write_text(src.replace(old, new))
        so = tmp_path / "libmut.so"
        subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-o", str(so), str(path), "-lm"])
        import ctypes
        lib = ctypes.CDLL(str(so))
        real = oracle._load()
        for fname in ("oracle_attn_fwd_rows", "oracle_attn_fwd_rows_bias", "oracle_attn_bwd",
                      "oracle_attn_bwd_bias"):
            getattr(lib, fname).argtypes = getattr(real, fname).argtypes
            getattr(lib, fname).restype = getattr(real, fname).restype
        monkeypatch.setattr(oracle, "_lib", lib)
    return _swap


def test_unmutated_oracle_passes_battery():
    assert battery() == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, swap_lib):
    swap_lib(MUTANTS[name])
    assert battery(), f"mutant {name} passed every pin"
