"""Shared helpers for the parity tests: run the oracle on exactly the rows a
test checks, and compare with the stated tolerances.

Tolerances (absolute, per element, against the fp64 oracle on the same
rounded inputs): O <= 2e-3 for fp16 and <= 1e-2 for bf16; LSE <= 1e-3;
backward <= 2e-2 (bf16) and <= 1e-2 (fp16).  O and the gradients are stored
in the 16-bit input dtype, so even the exactly rounded value is off by up to
half a unit in the last place (ulp) of that dtype.  Where that half ulp fits
under the tolerance the tolerance applies unchanged; only where it does not
(bf16 |x| >= 4 for 1e-2, fp16 |x| >= 8 for 2e-3; bf16 |x| >= 8 for 2e-2,
fp16 |x| >= 16 for 1e-2) is the bound the tolerance plus that half ulp.

Every comparison is recorded (largest error, its bound, and how many elements
needed the widened bound); conftest.py prints the records at the end of the
session.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle

TOL_O = {torch.float16: 2e-3, torch.bfloat16: 1e-2}
TOL_LSE = 1e-3
TOL_BWD = {torch.float16: 1e-2, torch.bfloat16: 2e-2}


def oracle_rows(q, k, v, rows, causal, scale=None):
    """Oracle O/LSE for flattened rows (b*Hq + h)*Nq + i, one head at a time
    so that only that head's K/V are widened to fp64."""
    B, Hq, Nq, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    rows = np.asarray(rows, dtype=np.int64)
    o = np.empty((rows.size, D))
    lse = np.empty(rows.size)
    bh = rows // Nq
    for key in np.unique(bh):
        sel = np.nonzero(bh == key)[0]
        b, h = divmod(int(key), Hq)
        g = h // G
        o_h, lse_h = oracle.attention_fwd(q[b:b + 1, h:h + 1], k[b:b + 1, g:g + 1],
                                          v[b:b + 1, g:g + 1], causal=causal, scale=scale,
                                          rows=rows[sel] % Nq)
        o[sel] = o_h
        lse[sel] = lse_h
    return o, lse


def gpu_rows(out, lse, rows):
    D = out.shape[-1]
    idx = torch.as_tensor(np.asarray(rows, dtype=np.int64), device=out.device)
    o = out.reshape(-1, D).index_select(0, idx).double().cpu().numpy()
    l_ = lse.reshape(-1).index_select(0, idx).double().cpu().numpy()
    return o, l_


def max_err(a, b) -> float:
    return float(np.max(np.abs(np.asarray(a) - np.asarray(b)))) if np.size(a) else 0.0


_MANT_BITS = {torch.float16: 10, torch.bfloat16: 7}


def ulp(ref, dtype):
    """One unit in the last place of `dtype` at |ref| (normal range)."""
    a = np.maximum(np.abs(np.asarray(ref, dtype=np.float64)), 2.0 ** -14)
    return np.exp2(np.floor(np.log2(a)) - _MANT_BITS[dtype])


# (what, name, elements, max error, tolerance, elements under the widened
# bound, largest error among elements under the flat tolerance, max |ref|)
RECORDS: list = []


def bound_for(ref, tol, dtype):
    """Per-element bound: tol where half an ulp of the stored dtype at |ref|
    is at most tol, else tol + that half ulp."""
    half = 0.5 * ulp(ref, dtype)
    return np.where(half > tol, tol + half, tol)


def assert_close_elementwise(got, ref, tol, dtype, what, name):
    got, ref = np.asarray(got), np.asarray(ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite {name}"
    bound = bound_for(ref, tol, dtype)
    err = np.abs(got - ref)
    widened = bound > tol
    flat_err = float(err[~widened].max()) if np.any(~widened) else 0.0
    RECORDS.append((what, name, int(err.size), float(err.max()) if err.size else 0.0, tol,
                    int(widened.sum()), flat_err,
                    float(np.abs(ref).max()) if err.size else 0.0))
    worst = np.unravel_index(np.argmax(err - bound), err.shape) if err.size else None
    if err.size:
        n_bad = int(np.sum(err > bound))
        assert n_bad == 0, (
            f"{what}: |{name}-oracle| = {err[worst]:.3e} > bound {bound[worst]:.3e} "
            f"at |ref| = {abs(ref[worst]):.3f} (max err {err.max():.3e}; {n_bad} of "
            f"{err.size} elements over their bound)")
    return float(err.max()) if err.size else 0.0


def assert_fwd_close(o_gpu, lse_gpu, o_ref, lse_ref, dtype, what=""):
    eo = assert_close_elementwise(o_gpu, o_ref, TOL_O[dtype], dtype, what, "O")
    el = max_err(lse_gpu, lse_ref)
    assert np.all(np.isfinite(lse_gpu)), f"{what}: non-finite LSE"
    RECORDS.append((what, "LSE", int(np.size(lse_gpu)), el, TOL_LSE, 0, el, 0.0))
    assert el <= TOL_LSE, f"{what}: max|LSE-oracle| = {el:.3e} > {TOL_LSE}"
    return eo, el


def default_scale(D):
    return 1.0 / math.sqrt(D)
