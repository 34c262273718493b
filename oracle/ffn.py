"""fp64 CPU oracle for the token-chunked feed-forward network -- TEST
INFRASTRUCTURE (only the test suite, the package's smoke check and the
benchmark's CPU legs may import it; it shares no code with the CUDA library).

The noflash-attention forum post (ai-navigate-news, section "The DIY
approach", list "What worked") names FFN chunking, with a runtime safety
check, as a further memory saving next to the tiled attention: the
feed-forward block of a transformer acts on every token independently, so it
can run a slice of tokens at a time and never hold the [tokens x d_ff]
intermediate for the whole sequence.  What it computes is the plain
definition, per token row x:

    h = act(x W1^T + b1)               (d_ff values)
    y = h W2^T + b2                    (d_model values)

with act one of relu, gelu (tanh form), silu, or swiglu, where W1 stacks a
gate and an up projection ([Wg; Wu], 2*d_ff rows) and h = silu(x Wg^T + bg) *
(x Wu^T + bu).  Reading of the pages (they give no formula): h is stored in
the input dtype between the two products, as a PyTorch fp16/bf16 FFN stores
its activation, so the oracle rounds h to that dtype when one is given; all
other arithmetic is fp64.  Chunking changes nothing in this definition: each
output row depends on its own input row only.
"""
from __future__ import annotations

import math

import numpy as np

ACTS = ("none", "relu", "gelu_tanh", "silu", "swiglu")


def _f64(x):
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def activation(a: np.ndarray, act: str) -> np.ndarray:
    """The element-wise activations, written from their definitions:
    relu max(0, a); gelu (tanh form, Hendrycks & Gimpel)
    0.5 a (1 + tanh(sqrt(2/pi) (a + 0.044715 a^3))); silu a / (1 + e^-a)."""
    if act == "none":
        return a
    if act == "relu":
        return np.maximum(a, 0.0)
    if act == "gelu_tanh":
        return 0.5 * a * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (a + 0.044715 * a ** 3)))
    if act == "silu":
        return a / (1.0 + np.exp(-a))
    raise ValueError(f"unknown activation {act!r}")


def round_to(x: np.ndarray, dtype) -> np.ndarray:
    """Round fp64 values to a torch 16-bit dtype (round to nearest even) and
    back to fp64."""
    import torch
    return torch.as_tensor(x).to(dtype).double().numpy()


def ffn_fwd(x, w1, b1, w2, b2, act: str, h_dtype=None):
    """y = act(x W1^T + b1) W2^T + b2 for x [T, d_model]; W1 [d_ff or 2*d_ff
    (swiglu), d_model], b1 matching or None; W2 [d_model, d_ff], b2 [d_model]
    or None.  h is rounded to ``h_dtype`` (a torch dtype) when given.
    Returns (y, h) in fp64."""
    x, w1, w2 = _f64(x), _f64(w1), _f64(w2)
    a = x @ w1.T
    if b1 is not None:
        a = a + _f64(b1)
    if act == "swiglu":
        f = w1.shape[0] // 2
        h = activation(a[:, :f], "silu") * a[:, f:]
    else:
        h = activation(a, act)
    if h_dtype is not None:
        h = round_to(h, h_dtype)
    y = h @ w2.T
    if b2 is not None:
        y = y + _f64(b2)
    return y, h
