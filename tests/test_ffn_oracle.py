"""Pins for the fp64 FFN oracle (no GPU): torch's own fp64 linear layers and
activations (independent library routines), closed forms, and the property
chunking rests on (every output row depends on its own input row only)."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import ffn


def rnd(shape, seed, std=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * std


def torch_ffn(x, w1, b1, w2, b2, act):
    x, w1, b1, w2, b2 = (torch.as_tensor(t) for t in (x, w1, b1, w2, b2))
    a = F.linear(x, w1, b1)
    if act == "swiglu":
        g, u = a.chunk(2, dim=-1)
        h = F.silu(g) * u
    elif act == "gelu_tanh":
        h = F.gelu(a, approximate="tanh")
    elif act == "silu":
        h = F.silu(a)
    elif act == "relu":
        h = F.relu(a)
    else:
        h = a
    return F.linear(h, w2, b2).numpy()


@pytest.mark.parametrize("act", ["none", "relu", "gelu_tanh", "silu", "swiglu"])
def test_matches_torch_f64(act):
    T, d, f = 37, 24, 40
    n1 = 2 * f if act == "swiglu" else f
    x, w1, b1 = rnd((T, d), 1), rnd((n1, d), 2, 0.3), rnd((n1,), 3)
    w2, b2 = rnd((d, f), 4, 0.2), rnd((d,), 5)
    y, _ = ffn.ffn_fwd(x, w1, b1, w2, b2, act)
    np.testing.assert_allclose(y, torch_ffn(x, w1, b1, w2, b2, act), rtol=0, atol=1e-12)


def test_closed_forms():
    T, d = 9, 8
    x = rnd((T, d), 6)
    eye, b1, b2 = np.eye(d), rnd((d,), 7), rnd((d,), 8)
    y, _ = ffn.ffn_fwd(x, eye, b1, eye, b2, "none")
    np.testing.assert_allclose(y, x + b1 + b2, atol=1e-14)
    # relu of a negative pre-activation is 0: only b2 is left
    y, _ = ffn.ffn_fwd(np.abs(x), -eye, None, rnd((d, d), 9), b2, "relu")
    np.testing.assert_allclose(y, np.broadcast_to(b2, (T, d)), atol=1e-14)
    # swiglu with a zero up projection is 0 whatever the gate
    w1 = np.concatenate([rnd((d, d), 10), np.zeros((d, d))])
    y, h = ffn.ffn_fwd(x, w1, None, rnd((d, d), 11), None, "swiglu")
    np.testing.assert_array_equal(h, 0.0)
    np.testing.assert_array_equal(y, 0.0)
    # the activations at a few points fixed by their definitions
    a = np.array([0.0, 30.0, -30.0])
    np.testing.assert_allclose(ffn.activation(a, "gelu_tanh"), [0.0, 30.0, 0.0], atol=1e-12)
    np.testing.assert_allclose(ffn.activation(a, "silu"), [0.0, 30.0, -30.0 * math.exp(-30)],
                               atol=1e-12)


def test_rows_are_independent():
    """The property chunking rests on: a chunk of rows gives the same rows."""
    T, d, f = 50, 16, 32
    x, w1, w2 = rnd((T, d), 12), rnd((2 * f, d), 13), rnd((d, f), 14)
    y, _ = ffn.ffn_fwd(x, w1, None, w2, None, "swiglu")
    for lo, hi in ((0, 7), (7, 31), (31, 50)):
        yc, _ = ffn.ffn_fwd(x[lo:hi], w1, None, w2, None, "swiglu")
        np.testing.assert_allclose(yc, y[lo:hi], rtol=0, atol=1e-12)


def test_intermediate_rounded_to_dtype():
    T, d, f = 5, 8, 16
    x, w1, w2 = rnd((T, d), 15), rnd((f, d), 16), rnd((d, f), 17)
    _, h = ffn.ffn_fwd(x, w1, None, w2, None, "gelu_tanh", h_dtype=torch.bfloat16)
    np.testing.assert_array_equal(h, torch.as_tensor(h).to(torch.bfloat16).double().numpy())
    _, h64 = ffn.ffn_fwd(x, w1, None, w2, None, "gelu_tanh")
    assert np.max(np.abs(h - h64) / np.maximum(np.abs(h64), 1e-30)) <= 2.0 ** -8
