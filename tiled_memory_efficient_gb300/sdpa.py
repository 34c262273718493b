"""Drop-in scaled-dot-product attention on the tiled CUDA kernels.

The forum post "I've been using a couple 32GB MI50s..." (ai-navigate-news,
section "Other areas where this could be useful") describes the library as a
patch of every ``F.scaled_dot_product_attention`` call, with an autograd tier
for training.  This module provides that surface on GB300:

* ``attention(q, k, v, is_causal=False, scale=None)`` -- a differentiable
  function (``torch.autograd.Function``) whose forward and backward both run in
  the library's kernels;
* ``scaled_dot_product_attention(...)`` -- the SDPA signature, accepting the
  arguments the kernels implement and raising for the rest;
* ``patch()`` / ``unpatch()`` -- opt-in replacement of
  ``torch.nn.functional.scaled_dot_product_attention``.

There is no backend probing and no fallback to another implementation: an
argument the kernels do not support (dropout, another head dim or dtype, a CPU
tensor) raises ``NotImplementedError`` or ``ValueError``.
"""
from __future__ import annotations

import math

import torch

from . import _lib

__all__ = ["attention", "scaled_dot_product_attention", "patch", "unpatch", "is_patched"]

_SUPPORTED_D = (64, 128)
_original_sdpa = None


class _TiledAttentionMasked(torch.autograd.Function):
    """Attention with an attn_mask (the mask itself gets no gradient)."""
    @staticmethod
    def forward(ctx, q, k, v, mask, is_causal, scale):
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        out, lse = _lib.attn_fwd(q, k, v, causal=is_causal, scale=scale, mask=mask)
        ctx.save_for_backward(q, k, v, out, lse, mask)
        ctx.is_causal = is_causal
        ctx.scale = scale
        return out

    @staticmethod
    def backward(ctx, dout):
        q, k, v, out, lse, mask = ctx.saved_tensors
        dq, dk, dv = _lib.attn_bwd(q, k, v, out, dout.contiguous(), lse, causal=ctx.is_causal,
                                   scale=ctx.scale, mask=mask)
        return dq, dk, dv, None, None, None


class _TiledAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, is_causal, scale):
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        B, Hq, Nq, D = q.shape
        Hkv, Nk = k.shape[1], k.shape[2]
        # Short query blocks against long keys (decode) leave most SMs idle
        # in one CTA per query-tile pair: cut the keys into ranges then.
        splits = _lib.num_splits(B, Hq, Hkv, Nq, Nk, D)
        if splits > 1:
            out, lse = _lib.attn_fwd_splitkv(q, k, v, causal=is_causal, scale=scale,
                                             splits=splits)
        else:
            # bf16: the value tiles are converted to fp16 once, in a workspace
            # torch allocates (fp16: the plain forward)
            out, lse = _lib.attn_fwd_ws(q, k, v, causal=is_causal, scale=scale)
        ctx.save_for_backward(q, k, v, out, lse)
        ctx.is_causal = is_causal
        ctx.scale = scale
        return out

    @staticmethod
    def backward(ctx, dout):
        q, k, v, out, lse = ctx.saved_tensors
        dq, dk, dv = _lib.attn_bwd(q, k, v, out, dout.contiguous(), lse,
                                   causal=ctx.is_causal, scale=ctx.scale)
        return dq, dk, dv, None, None


def _validate(q, k, v):
    for name, t in (("query", q), ("key", k), ("value", v)):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a tensor")
        if t.dim() != 4:
            raise NotImplementedError(f"{name} must be 4-D [batch, heads, seq_len, dim]")
        if t.device.type != "cuda":
            raise NotImplementedError(f"{name} must be on a CUDA device")
        if t.dtype not in (torch.float16, torch.bfloat16):
            raise NotImplementedError(f"{name} dtype {t.dtype} is not float16/bfloat16")
    if q.shape[-1] not in _SUPPORTED_D:
        raise NotImplementedError(f"head dim {q.shape[-1]} is not one of {_SUPPORTED_D}")
    if k.shape[1] == 0 or q.shape[1] % k.shape[1] != 0:
        raise ValueError("query heads must be a multiple of key/value heads")


def attention(q, k, v, is_causal: bool = False, scale: float | None = None, attn_mask=None):
    """Differentiable tiled attention.  q [B,Hq,Nq,D]; k, v [B,Hkv,Nk,D] with
    Hq a multiple of Hkv (query head h uses KV head h // (Hq//Hkv)); causal is
    top-left aligned; scale defaults to 1/sqrt(D).  attn_mask: bool (True
    keeps a key) or additive, broadcastable to [B,Hq,Nq,Nk]."""
    _validate(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    if attn_mask is not None:
        return _TiledAttentionMasked.apply(q, k, v, attn_mask, bool(is_causal), float(scale))
    return _TiledAttention.apply(q, k, v, bool(is_causal), float(scale))


def scaled_dot_product_attention(query, key, value, attn_mask=None, dropout_p=0.0,
                                 is_causal=False, scale=None, enable_gqa=False):
    """The SDPA call, served by the tiled kernels.

    Supported: dropout_p == 0, fp16/bf16 CUDA tensors [B, H, N, D] with D in
    (64, 128), an optional attn_mask (bool or floating, broadcastable to
    [B, Hq, Nq, Nk]; it gets no gradient).  With
    Hq != Hkv, enable_gqa must be set (as for torch's own SDPA).  Anything
    else raises.
    """
    if dropout_p != 0.0:
        raise NotImplementedError("dropout is not supported by the tiled kernels")
    if query.dim() == 4 and key.dim() == 4 and query.shape[1] != key.shape[1] and not enable_gqa:
        raise ValueError("query and key head counts differ: pass enable_gqa=True")
    return attention(query, key, value, is_causal=is_causal, scale=scale, attn_mask=attn_mask)


def patch():
    """Route torch.nn.functional.scaled_dot_product_attention to the tiled
    kernels (opt-in; unsupported arguments then raise instead of running)."""
    global _original_sdpa
    import torch.nn.functional as F
    if _original_sdpa is None:
        _original_sdpa = F.scaled_dot_product_attention
        F.scaled_dot_product_attention = scaled_dot_product_attention


def unpatch():
    """Restore the original torch.nn.functional.scaled_dot_product_attention."""
    global _original_sdpa
    import torch.nn.functional as F
    if _original_sdpa is not None:
        F.scaled_dot_product_attention = _original_sdpa
        _original_sdpa = None


def is_patched() -> bool:
    return _original_sdpa is not None
