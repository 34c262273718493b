"""Pins for the fp64 CPU oracle (no GPU).

The pages print no numeric example, so the oracle is pinned to what the
mathematics fixes: a hand-worked example (tests/golden/hand_worked.json),
closed forms, invariants, an independent library routine (torch's fp64 CPU
scaled_dot_product_attention and its autograd) and finite differences.  Each
pin is chosen so that a plausible slip in the oracle -- a dropped scale, a
flipped exponent sign, a transposed operand, a wrong GQA head mapping, an
off-by-one causal mask, a missing normalisation -- fails at least one test.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from tiled_memory_efficient_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(shape, seed, std=1.0):
    g = np.random.default_rng(seed)
    return g.standard_normal(shape) * std


def sdpa_f64(q, k, v, causal, scale):
    """torch's own CPU fp64 SDPA; GQA by repeat_interleave of K/V heads."""
    q, k, v = (torch.as_tensor(np.asarray(x), dtype=torch.float64) for x in (q, k, v))
    G = q.shape[1] // k.shape[1]
    k = k.repeat_interleave(G, dim=1)
    v = v.repeat_interleave(G, dim=1)
    return F.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=scale).numpy()


def lse_f64(q, k, causal, scale):
    """torch.logsumexp over the scaled scores (library reduction)."""
    q, k = (torch.as_tensor(np.asarray(x), dtype=torch.float64) for x in (q, k))
    G = q.shape[1] // k.shape[1]
    k = k.repeat_interleave(G, dim=1)
    s = scale * q @ k.transpose(-1, -2)
    if causal:
        nq, nk = s.shape[-2:]
        mask = torch.ones(nq, nk, dtype=torch.bool).tril()
        s = s.masked_fill(~mask, -math.inf)
    return torch.logsumexp(s, dim=-1).numpy()


# --------------------------------------------------------------------------- golden

def test_hand_worked_example_forward():
    gd = json.load(open(os.path.join(GOLDEN, "hand_worked.json")))
    q = np.array(gd["q"])[None, None]
    k = np.array(gd["k"])[None, None]
    v = np.array(gd["v"])[None, None]
    for causal, key in ((False, "noncausal"), (True, "causal")):
        o, lse = oracle.attention_fwd(q, k, v, causal=causal, scale=gd["scale"])
        np.testing.assert_allclose(o[0, 0], np.array(gd[key]["o"]), rtol=0, atol=1e-14)
        np.testing.assert_allclose(lse[0, 0], np.array(gd[key]["lse"]), rtol=0, atol=1e-14)


def test_hand_worked_example_backward():
    gd = json.load(open(os.path.join(GOLDEN, "hand_worked.json")))
    q = np.array(gd["q"])[None, None]
    k = np.array(gd["k"])[None, None]
    v = np.array(gd["v"])[None, None]
    bw = gd["backward_noncausal"]
    do = np.array(bw["dout"])[None, None]
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal=False, scale=gd["scale"])
    np.testing.assert_allclose(dq[0, 0], np.array(bw["dq"]), atol=1e-14)
    np.testing.assert_allclose(dk[0, 0], np.array(bw["dk"]), atol=1e-14)
    np.testing.assert_allclose(dv[0, 0], np.array(bw["dv"]), atol=1e-14)


# --------------------------------------------------------------------------- library routine

@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,D,causal", [
    (1, 2, 2, 37, 37, 16, False),
    (2, 3, 3, 40, 29, 8, False),
    (1, 4, 2, 33, 33, 16, True),
    (1, 6, 2, 20, 31, 8, True),     # Nq != Nk, top-left causal
    (1, 7, 1, 45, 45, 32, False),   # G = 7 as in the GQA prefill shape
])
def test_matches_torch_sdpa_f64(B, Hq, Hkv, Nq, Nk, D, causal):
    q = rnd((B, Hq, Nq, D), 1)
    k = rnd((B, Hkv, Nk, D), 2)
    v = rnd((B, Hkv, Nk, D), 3)
    scale = 1.0 / math.sqrt(D)
    o, lse = oracle.attention_fwd(q, k, v, causal=causal)
    np.testing.assert_allclose(o, sdpa_f64(q, k, v, causal, scale), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_f64(q, k, causal, scale), rtol=0, atol=1e-12)


def test_explicit_scale_is_used():
    q, k, v = rnd((1, 1, 9, 4), 4), rnd((1, 1, 9, 4), 5), rnd((1, 1, 9, 4), 6)
    o, lse = oracle.attention_fwd(q, k, v, scale=0.37)
    np.testing.assert_allclose(o, sdpa_f64(q, k, v, False, 0.37), atol=1e-12)
    np.testing.assert_allclose(lse, lse_f64(q, k, False, 0.37), atol=1e-12)


@pytest.mark.parametrize("Hq,Hkv,causal", [(2, 2, False), (4, 2, True), (3, 1, False)])
def test_backward_matches_torch_autograd(Hq, Hkv, causal):
    B, N, D = 2, 19, 8
    q, k, v, do = rnd((B, Hq, N, D), 7), rnd((B, Hkv, N, D), 8), rnd((B, Hkv, N, D), 9), \
        rnd((B, Hq, N, D), 10)
    qt, kt, vt = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    G = Hq // Hkv
    out = F.scaled_dot_product_attention(qt, kt.repeat_interleave(G, 1),
                                         vt.repeat_interleave(G, 1), is_causal=causal)
    out.backward(torch.tensor(do))
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal=causal)
    np.testing.assert_allclose(dq, qt.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dk, kt.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dv, vt.grad.numpy(), atol=1e-11)


# --------------------------------------------------------------------------- brute force

def test_rows_subset_equals_full():
    B, Hq, Hkv, N, D = 2, 4, 2, 23, 8
    q, k, v = rnd((B, Hq, N, D), 11), rnd((B, Hkv, N, D), 12), rnd((B, Hkv, N, D), 13)
    o, lse = oracle.attention_fwd(q, k, v, causal=True)
    rows = np.array([0, 5, 22, 23, 60, B * Hq * N - 1])
    o_r, lse_r = oracle.attention_fwd(q, k, v, causal=True, rows=rows)
    np.testing.assert_array_equal(o_r, o.reshape(-1, D)[rows])
    np.testing.assert_array_equal(lse_r, lse.reshape(-1)[rows])


def test_finite_differences_backward():
    B, Hq, Hkv, N, D = 1, 2, 1, 6, 4
    q, k, v, do = rnd((B, Hq, N, D), 14), rnd((B, Hkv, N, D), 15), rnd((B, Hkv, N, D), 16), \
        rnd((B, Hq, N, D), 17)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal=True)

    def loss(q_, k_, v_):
        o, _ = oracle.attention_fwd(q_, k_, v_, causal=True)
        return float((o * do).sum())

    eps = 1e-6
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            fp = loss(args["q"], args["k"], args["v"])
            args[name] = xm
            fm = loss(args["q"], args["k"], args["v"])
            num[idx] = (fp - fm) / (2 * eps)
        np.testing.assert_allclose(grad, num, rtol=1e-6, atol=1e-8, err_msg=name)


# --------------------------------------------------------------------------- closed forms

def test_single_key_returns_its_value_row():
    q, k, v = rnd((1, 3, 5, 8), 20), rnd((1, 3, 1, 8), 21), rnd((1, 3, 1, 8), 22)
    o, lse = oracle.attention_fwd(q, k, v)
    np.testing.assert_allclose(o, np.broadcast_to(v, o.shape), atol=1e-15)
    expect = (q @ k.transpose(0, 1, 3, 2))[..., 0] / math.sqrt(8)
    np.testing.assert_allclose(lse, expect, atol=1e-13)


def test_identical_keys_give_mean_of_values():
    N, D = 17, 8
    q = rnd((1, 2, N, D), 23)
    k = np.broadcast_to(rnd((1, 2, 1, D), 24), (1, 2, N, D)).copy()
    v = rnd((1, 2, N, D), 25)
    o, lse = oracle.attention_fwd(q, k, v)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape),
                               atol=1e-13)
    expect = (q @ k[:, :, :1].transpose(0, 1, 3, 2))[..., 0] / math.sqrt(D) + math.log(N)
    np.testing.assert_allclose(lse, expect, atol=1e-13)


def test_zero_query_causal_gives_prefix_means():
    N, D = 21, 4
    q = np.zeros((1, 1, N, D))
    k, v = rnd((1, 1, N, D), 26), rnd((1, 1, N, D), 27)
    o, lse = oracle.attention_fwd(q, k, v, causal=True)
    prefix = np.cumsum(v[0, 0], axis=0) / np.arange(1, N + 1)[:, None]
    np.testing.assert_allclose(o[0, 0], prefix, atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], np.log(np.arange(1, N + 1)), atol=1e-14)
    o_nc, lse_nc = oracle.attention_fwd(q, k, v, causal=False)
    np.testing.assert_allclose(o_nc[0, 0], np.broadcast_to(v[0, 0].mean(0), (N, D)), atol=1e-14)
    np.testing.assert_allclose(lse_nc, math.log(N), atol=1e-14)


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,D", [
    (1, 2, 2, 5, 19, 8),      # Nq < Nk
    (2, 4, 2, 1, 23, 16),     # one query (decode) with GQA
    (1, 7, 1, 12, 40, 8),     # G = 7
    (1, 2, 1, 17, 17, 8),     # Nq = Nk
])
def test_bottom_right_matches_torch_causal_lower_right(B, Hq, Hkv, Nq, Nk, D):
    """Bottom-right causal against torch's own lower-right causal bias (an
    independent library routine) and torch.logsumexp over a tril mask."""
    from torch.nn.attention.bias import causal_lower_right
    q, k, v = rnd((B, Hq, Nq, D), 81), rnd((B, Hkv, Nk, D), 82), rnd((B, Hkv, Nk, D), 83)
    scale = 1.0 / math.sqrt(D)
    o, lse = oracle.attention_fwd(q, k, v, causal="bottom_right")
    G = Hq // Hkv
    qt, kt, vt = (torch.as_tensor(x) for x in (q, k, v))
    kt, vt = kt.repeat_interleave(G, dim=1), vt.repeat_interleave(G, dim=1)
    ref = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=causal_lower_right(Nq, Nk))
    np.testing.assert_allclose(o, ref.numpy(), rtol=0, atol=1e-12)
    s = scale * qt @ kt.transpose(-1, -2)
    mask = torch.ones(Nq, Nk, dtype=torch.bool).tril(diagonal=Nk - Nq)
    ref_lse = torch.logsumexp(s.masked_fill(~mask, -math.inf), dim=-1)
    np.testing.assert_allclose(lse, ref_lse.numpy(), rtol=0, atol=1e-12)


def test_zero_query_bottom_right_gives_prefix_means():
    """Q = 0, bottom-right: query i averages V[0 .. i + Nk - Nq] and its LSE
    is ln(i + Nk - Nq + 1) (closed form)."""
    Nq, Nk, D = 6, 15, 4
    q = np.zeros((1, 1, Nq, D))
    k, v = rnd((1, 1, Nk, D), 84), rnd((1, 1, Nk, D), 85)
    o, lse = oracle.attention_fwd(q, k, v, causal="bottom_right")
    n = np.arange(Nq) + (Nk - Nq) + 1
    prefix = np.cumsum(v[0, 0], axis=0)[n - 1] / n[:, None]
    np.testing.assert_allclose(o[0, 0], prefix, atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], np.log(n), atol=1e-14)
    assert [oracle.attended_keys(i, Nk, "bottom_right", Nq) for i in range(Nq)] == list(n)


def test_bottom_right_special_cases():
    """Square: bottom-right is top-left.  The last query sees every key."""
    q, k, v = rnd((1, 2, 11, 8), 86), rnd((1, 2, 11, 8), 87), rnd((1, 2, 11, 8), 88)
    a = oracle.attention_fwd(q, k, v, causal="bottom_right")
    b = oracle.attention_fwd(q, k, v, causal=True)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    k2, v2 = rnd((1, 2, 30, 8), 89), rnd((1, 2, 30, 8), 90)
    o, lse = oracle.attention_fwd(q, k2, v2, causal="bottom_right")
    o_nc, lse_nc = oracle.attention_fwd(q[:, :, -1:], k2, v2)
    np.testing.assert_allclose(o[:, :, -1:], o_nc, atol=1e-15)
    np.testing.assert_allclose(lse[:, :, -1:], lse_nc, atol=1e-15)


def test_bottom_right_argument_checks():
    q, k = rnd((1, 1, 9, 4), 91), rnd((1, 1, 5, 4), 92)
    with pytest.raises(RuntimeError):
        oracle.attention_fwd(q, k, k, causal="bottom_right")   # Nq > Nk
    with pytest.raises(RuntimeError):
        oracle.attention_bwd(q[:, :, :5], k, k, q[:, :, :5], causal="bottom_right")


@pytest.mark.parametrize("shape,kind,causal", [
    ((2, 1, 1, 23), "bool", False),       # key padding, broadcast over heads and queries
    ((2, 1, 13, 23), "bool", True),       # per-query mask with the causal mask on top
    ((1, 4, 13, 23), "additive", False),  # per-head bias (ALiBi-like)
    ((2, 4, 13, 23), "additive", True),
    ((13, 23), "additive", False),        # 2-D mask, broadcast over batch and heads
])
def test_mask_matches_torch_sdpa_f64(shape, kind, causal):
    """attn_mask against torch's fp64 SDPA (an independent library routine)
    and torch.logsumexp of the biased scores."""
    B, Hq, Hkv, Nq, Nk, D = 2, 4, 2, 13, 23, 8
    q, k, v = rnd((B, Hq, Nq, D), 101), rnd((B, Hkv, Nk, D), 102), rnd((B, Hkv, Nk, D), 103)
    g = torch.Generator().manual_seed(104)
    if kind == "bool":
        mask = torch.rand(shape, generator=g) > 0.4
        mask[..., 0] = True   # every row keeps key 0 (so no row is empty)
    else:
        mask = torch.randn(shape, generator=g, dtype=torch.float64) * 2.0
    o, lse = oracle.attention_fwd(q, k, v, causal=causal, mask=mask)
    qt, kt, vt = (torch.as_tensor(x) for x in (q, k, v))
    kt, vt = kt.repeat_interleave(Hq // Hkv, dim=1), vt.repeat_interleave(Hq // Hkv, dim=1)
    bias = mask if kind == "additive" else torch.zeros(shape, dtype=torch.float64).masked_fill(
        ~mask, -math.inf)
    if causal:
        bias = bias + torch.zeros(Nq, Nk, dtype=torch.float64).masked_fill(
            ~torch.ones(Nq, Nk, dtype=torch.bool).tril(), -math.inf)
    ref = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=bias)
    np.testing.assert_allclose(o, ref.numpy(), rtol=0, atol=1e-12)
    s = qt @ kt.transpose(-1, -2) / math.sqrt(D) + bias
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), rtol=0, atol=1e-12)


def test_mask_closed_forms():
    """A constant bias c leaves O alone and adds c to the LSE; with Q = 0 a
    bias ln w_j gives the w-weighted mean of V and LSE = ln sum w; a mask that
    keeps one key returns that key's value row; a row with every key masked
    is O = 0, LSE = -inf."""
    Nq, Nk, D = 5, 11, 4
    q, k, v = rnd((1, 1, Nq, D), 105), rnd((1, 1, Nk, D), 106), rnd((1, 1, Nk, D), 107)
    o0, l0 = oracle.attention_fwd(q, k, v)
    o1, l1 = oracle.attention_fwd(q, k, v, mask=np.full((Nq, Nk), 0.75))
    np.testing.assert_allclose(o1, o0, atol=1e-14)
    np.testing.assert_allclose(l1, l0 + 0.75, atol=1e-14)
    w = np.exp(rnd((Nk,), 108))
    oz, lz = oracle.attention_fwd(np.zeros_like(q), k, v, mask=np.log(w)[None, :])
    np.testing.assert_allclose(oz[0, 0], np.broadcast_to(w @ v[0, 0] / w.sum(), (Nq, D)),
                               atol=1e-14)
    np.testing.assert_allclose(lz, math.log(w.sum()), atol=1e-14)
    keep = np.zeros((Nq, Nk), dtype=bool)
    keep[np.arange(Nq), np.arange(Nq) * 2] = True
    keep[4] = False                     # row 4: every key masked
    om, lm = oracle.attention_fwd(q, k, v, mask=torch.as_tensor(keep))
    for i in range(4):
        np.testing.assert_allclose(om[0, 0, i], v[0, 0, 2 * i], atol=1e-15)
        np.testing.assert_allclose(lm[0, 0, i], q[0, 0, i] @ k[0, 0, 2 * i] / math.sqrt(D),
                                   atol=1e-14)
    np.testing.assert_array_equal(om[0, 0, 4], 0.0)
    assert lm[0, 0, 4] == -math.inf


@pytest.mark.parametrize("kind", ["bool", "additive"])
def test_masked_backward_matches_torch_autograd(kind):
    """Gradients with an attn_mask against torch.autograd through fp64 SDPA
    (GQA by repeat_interleave, so dk/dv are summed over the group); a query
    row with every key masked contributes nothing."""
    B, Hq, Hkv, Nq, Nk, D = 2, 4, 2, 11, 17, 8
    q, k, v = rnd((B, Hq, Nq, D), 111), rnd((B, Hkv, Nk, D), 112), rnd((B, Hkv, Nk, D), 113)
    do = rnd((B, Hq, Nq, D), 114)
    g = torch.Generator().manual_seed(115)
    if kind == "bool":
        mask = torch.rand(B, 1, Nq, Nk, generator=g) > 0.4
        mask[..., 0] = True
        mask[1, 0, 5] = False             # an empty row
        bias = torch.zeros(B, 1, Nq, Nk, dtype=torch.float64).masked_fill(~mask, -math.inf)
    else:
        mask = torch.randn(1, Hq, Nq, Nk, generator=g, dtype=torch.float64)
        bias = mask
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, mask=mask)
    qt, kt, vt = (torch.as_tensor(x).requires_grad_(True) for x in (q, k, v))
    G = Hq // Hkv
    keep = torch.isfinite(bias).any(-1, keepdim=True)         # torch gives NaN on empty rows
    safe = torch.where(keep, bias, torch.zeros_like(bias))
    out = F.scaled_dot_product_attention(qt, kt.repeat_interleave(G, 1), vt.repeat_interleave(G, 1),
                                         attn_mask=safe) * keep
    out.backward(torch.as_tensor(do))
    for name, got, ref in (("dq", dq, qt.grad), ("dk", dk, kt.grad), ("dv", dv, vt.grad)):
        np.testing.assert_allclose(got, ref.numpy(), rtol=0, atol=1e-11, err_msg=name)
    if kind == "bool":
        np.testing.assert_array_equal(dq[1, 0, 5], 0.0)


def test_causal_row_zero_is_first_value():
    q, k, v = rnd((2, 2, 9, 8), 28), rnd((2, 2, 9, 8), 29), rnd((2, 2, 9, 8), 30)
    o, _ = oracle.attention_fwd(q, k, v, causal=True)
    np.testing.assert_allclose(o[:, :, 0], v[:, :, 0], atol=1e-15)


def test_rows_sum_to_one_via_constant_values():
    q, k = rnd((1, 2, 11, 8), 31, std=3.0), rnd((1, 2, 13, 8), 32, std=3.0)
    v = np.ones((1, 2, 13, 8))
    for causal in (False, True):
        o, _ = oracle.attention_fwd(q, k, v, causal=causal)
        np.testing.assert_allclose(o, 1.0, atol=1e-14)


def test_key_shift_leaves_output_and_moves_lse():
    D = 8
    q, k, v = rnd((1, 1, 10, D), 33), rnd((1, 1, 12, D), 34), rnd((1, 1, 12, D), 35)
    u = rnd((D,), 36)
    o, lse = oracle.attention_fwd(q, k, v)
    o2, lse2 = oracle.attention_fwd(q, k + u, v)
    np.testing.assert_allclose(o2, o, atol=1e-13)
    np.testing.assert_allclose(lse2, lse + (q @ u) / math.sqrt(D), atol=1e-12)


# --------------------------------------------------------------------------- invariants

def test_permuting_keys_and_values_together():
    q, k, v = rnd((1, 2, 14, 8), 37), rnd((1, 2, 19, 8), 38), rnd((1, 2, 19, 8), 39)
    perm = np.random.default_rng(40).permutation(19)
    o, lse = oracle.attention_fwd(q, k, v)
    o2, lse2 = oracle.attention_fwd(q, k[:, :, perm], v[:, :, perm])
    np.testing.assert_allclose(o2, o, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, atol=1e-13)


def test_gqa_equals_mha_on_repeated_heads():
    q, k, v = rnd((1, 6, 15, 8), 41), rnd((1, 2, 15, 8), 42), rnd((1, 2, 15, 8), 43)
    for causal in (False, True):
        o, lse = oracle.attention_fwd(q, k, v, causal=causal)
        o2, lse2 = oracle.attention_fwd(q, np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1),
                                        causal=causal)
        np.testing.assert_array_equal(o, o2)
        np.testing.assert_array_equal(lse, lse2)
    # contiguous groups: query heads 0..2 use KV head 0, so changing KV head 1
    # must leave them alone and change heads 3..5
    k2 = k.copy()
    k2[:, 1] = rnd((1, 15, 8), 99)
    o, _ = oracle.attention_fwd(q, k, v)
    o3, _ = oracle.attention_fwd(q, k2, v)
    np.testing.assert_array_equal(o3[:, :3], o[:, :3])
    assert np.abs(o3[:, 3:] - o[:, 3:]).max() > 1e-3


def test_output_is_linear_in_values():
    q, k = rnd((1, 1, 8, 4), 44), rnd((1, 1, 8, 4), 45)
    v1, v2 = rnd((1, 1, 8, 4), 46), rnd((1, 1, 8, 4), 47)
    o1, _ = oracle.attention_fwd(q, k, v1)
    o2, _ = oracle.attention_fwd(q, k, v2)
    o3, _ = oracle.attention_fwd(q, k, 2.0 * v1 - 3.0 * v2)
    np.testing.assert_allclose(o3, 2.0 * o1 - 3.0 * o2, atol=1e-13)


def test_backward_invariants():
    B, Hq, Hkv, N, D = 1, 4, 2, 13, 8
    q, k = rnd((B, Hq, N, D), 48), rnd((B, Hkv, N, D), 49)
    do = rnd((B, Hq, N, D), 50)
    # identical value rows: output is constant in q and k, so dq = dk = 0
    v_same = np.broadcast_to(rnd((B, Hkv, 1, D), 51), (B, Hkv, N, D)).copy()
    dq, dk, dv = oracle.attention_bwd(q, k, v_same, do, causal=True)
    np.testing.assert_allclose(dq, 0.0, atol=1e-13)
    np.testing.assert_allclose(dk, 0.0, atol=1e-13)
    # softmax rows sum to one: sum_j dv_j = sum over the group's rows of dout;
    # shifting every key by u leaves O alone: sum_j dk_j = 0
    v = rnd((B, Hkv, N, D), 52)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal=False)
    group_do = do.reshape(B, Hkv, Hq // Hkv, N, D).sum(axis=(2, 3))
    np.testing.assert_allclose(dv.sum(axis=2), group_do, atol=1e-12)
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12)


# --------------------------------------------------------------------------- inputs and host logic

def test_inputs_are_seeded_and_rounded():
    w = inputs.WORKLOADS["tiny"]
    a = inputs.make_inputs(w, 256)
    b = inputs.make_inputs(w, 256)
    for key in ("q", "k", "v"):
        assert a[key].dtype == torch.float16
        assert torch.equal(a[key], b[key])
    assert a["q"].shape == (1, 2, 256, 64)


def test_outlier_keys_recipe():
    w = inputs.Workload("t", 9, 1, 2, 2, 16, torch.bfloat16, False, (300,), outlier_keys=True)
    x = inputs.make_inputs(w, 300)
    norms = x["k"].float().norm(dim=-1)
    big = (norms > 3 * norms.median()).sum(dim=-1)
    assert big.tolist() == [[3, 3]]   # floor(0.01 * 300) rows per KV head


def test_sample_rows_cover_edges():
    rows = inputs.sample_rows(1, 2, 1000, per_head=4, seed=3)
    r = set(rows.tolist())
    for base in (0, 1000):
        assert {base, base + 999, base + 127, base + 128, base + 255, base + 256} <= r


def test_flops_formula():
    w = inputs.WORKLOADS["gqa_prefill"]
    assert w.flops_fwd(1024) == 4 * 14 * 1024 * 1024 * 64 / 2
