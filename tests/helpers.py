"""Shared helpers for the parity tests: run the oracle on exactly the rows a
test checks, and compare with the stated tolerances.

Tolerances (max-abs, against the fp64 oracle on the same rounded inputs):
O <= 2e-3 for fp16 and <= 1e-2 for bf16; LSE <= 1e-3; backward (bf16)
<= 2e-2, fp16 backward <= 1e-2.
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


def assert_fwd_close(o_gpu, lse_gpu, o_ref, lse_ref, dtype, what=""):
    eo = max_err(o_gpu, o_ref)
    el = max_err(lse_gpu, lse_ref)
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite O"
    assert np.all(np.isfinite(lse_gpu)), f"{what}: non-finite LSE"
    assert eo <= TOL_O[dtype], f"{what}: max|O-oracle| = {eo:.3e} > {TOL_O[dtype]}"
    assert el <= TOL_LSE, f"{what}: max|LSE-oracle| = {el:.3e} > {TOL_LSE}"
    return eo, el


def default_scale(D):
    return 1.0 / math.sqrt(D)
