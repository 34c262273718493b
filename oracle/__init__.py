"""fp64 CPU oracle for scaled-dot-product attention -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's
``cpu_baseline`` / reference leg may import this package.  The CUDA library
never does, and this package never imports the CUDA library: the two share
no code.  The arithmetic lives in ``attn_oracle.c`` (plain C, fp64, one query
row at a time); this module only builds it with gcc and marshals arrays.

What it computes is the plain definition of attention that the tiled method
reaches by a faster route (noflash-attention forum post, ai-navigate-news,
section "The DIY approach": tiling gives the same math with O(N) memory):
``O = softmax(scale * Q K^T) V`` per row, ``LSE = log sum_j exp(scale q.k_j)``,
GQA by ``h_kv = h_q // (Hq // Hkv)``, an optional causal mask (top-left, or
for the forward also bottom-right: the queries are the last Nq positions of
the key sequence, as in KV-cache decoding), and the gradients of that map
(no mask or top-left).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into oracle/_build/liboracle.so with gcc."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64 = ctypes.c_int64
            lib.oracle_attn_fwd_rows.argtypes = [_dp, _dp, _dp, i64, i64, i64, i64, i64, i64,
                                                 ctypes.c_double, ctypes.c_int, _i64p, i64,
                                                 _dp, _dp, ctypes.c_int]
            lib.oracle_attn_fwd_rows.restype = ctypes.c_int
            lib.oracle_attn_fwd_rows_bias.argtypes = [_dp, _dp, _dp, i64, i64, i64, i64, i64, i64,
                                                      ctypes.c_double, ctypes.c_int,
                                                      _dp, i64, i64, i64, _i64p, i64,
                                                      _dp, _dp, ctypes.c_int]
            lib.oracle_attn_fwd_rows_bias.restype = ctypes.c_int
            lib.oracle_attn_bwd.argtypes = [_dp, _dp, _dp, _dp, i64, i64, i64, i64, i64, i64,
                                            ctypes.c_double, ctypes.c_int, _dp, _dp, _dp,
                                            ctypes.c_int]
            lib.oracle_attn_bwd.restype = ctypes.c_int
            lib.oracle_attn_bwd_bias.argtypes = [_dp, _dp, _dp, _dp, i64, i64, i64, i64, i64, i64,
                                                 ctypes.c_double, ctypes.c_int, _dp, i64, i64, i64,
                                                 _dp, _dp, _dp, ctypes.c_int]
            lib.oracle_attn_bwd_bias.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    """Widen a torch tensor or array (fp16/bf16/fp32/fp64) to contiguous fp64."""
    if hasattr(x, "detach"):  # torch tensor: go through fp32 (exact for fp16/bf16)
        x = x.detach().to("cpu")
        if x.dtype != _torch_f64():
            x = x.float()
        x = x.numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _torch_f64():
    import torch
    return torch.float64


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_dp)


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _shapes(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [B, H, N, D]")
    B, Hq, Nq, D = q.shape
    Bk, Hkv, Nk, Dk = k.shape
    if v.shape != k.shape or Bk != B or Dk != D or Hq % Hkv != 0:
        raise ValueError(f"incompatible shapes q{q.shape} k{k.shape} v{v.shape}")
    return B, Hq, Hkv, Nq, Nk, D


def _bias_f64(mask, B, Hq, Nq, Nk):
    """An SDPA-style attn_mask as an fp64 additive bias and its element
    strides over (batch, query head, query): bool -> 0 where True, -inf where
    False; any other dtype is taken as an additive bias.  The mask must
    broadcast to [B, Hq, Nq, Nk]; size-1 dimensions get stride 0."""
    if hasattr(mask, "detach"):          # a torch tensor
        t = mask.detach().cpu()
        m = t.numpy() if str(t.dtype) == "torch.bool" else t.double().numpy()
    else:
        m = np.asarray(mask)
    if m.dtype == np.bool_:
        m = np.where(m, 0.0, -np.inf)
    m = np.asarray(m, dtype=np.float64)
    while m.ndim < 4:
        m = m[None]
    if m.ndim != 4 or m.shape[-1] != Nk:
        raise ValueError(f"mask must broadcast to {(B, Hq, Nq, Nk)}, got {m.shape}")
    for dim, full in zip(m.shape[:3], (B, Hq, Nq)):
        if dim not in (1, full):
            raise ValueError(f"mask shape {m.shape} does not broadcast to {(B, Hq, Nq, Nk)}")
    m = np.ascontiguousarray(m)
    strides = tuple(0 if m.shape[i] == 1 else m.strides[i] // 8 for i in range(3))
    return m, strides


def attention_fwd(q, k, v, causal=False, scale: float | None = None,
                  rows=None, threads: int | None = None, mask=None):
    """Forward definition in fp64.

    q: [B,Hq,Nq,D]; k, v: [B,Hkv,Nk,D].  Returns (o, lse) as fp64 arrays.  With
    ``rows`` (flattened ids ``(b*Hq + h)*Nq + i``) only those rows are
    computed and o is [len(rows), D], lse [len(rows)]; otherwise o is
    [B,Hq,Nq,D] and lse [B,Hq,Nq].  ``mask``: optional attn_mask broadcastable
    to [B,Hq,Nq,Nk], boolean (True keeps a key) or additive.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Hkv, Nq, Nk, D = _shapes(q, k, v)
    bias, bstr = (None, (0, 0, 0)) if mask is None else _bias_f64(mask, B, Hq, Nq, Nk)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if rows is None:
        o = np.empty((B, Hq, Nq, D), np.float64)
        lse = np.empty((B, Hq, Nq), np.float64)
        rows_p, n = None, 0
    else:
        rows_a = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
        n = rows_a.size
        o = np.empty((n, D), np.float64)
        lse = np.empty((n,), np.float64)
        rows_p = rows_a.ctypes.data_as(_i64p)
        if n == 0:
            return o, lse
    rc = _load().oracle_attn_fwd_rows_bias(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Nq, Nk, D,
                                           float(scale), causal_code(causal),
                                           None if bias is None else _ptr(bias), *bstr,
                                           rows_p, n, _ptr(o), _ptr(lse),
                                           int(threads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_fwd_rows_bias failed with {rc}")
    return o, lse


def attention_bwd(q, k, v, dout, causal: bool = False, scale: float | None = None,
                  threads: int | None = None, mask=None):
    """Gradients of the forward definition, in fp64: returns (dq, dk, dv).
    ``mask`` as for attention_fwd (rows with every key masked get zero)."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, Hq, Hkv, Nq, Nk, D = _shapes(q, k, v)
    bias, bstr = (None, (0, 0, 0)) if mask is None else _bias_f64(mask, B, Hq, Nq, Nk)
    if dout.shape != q.shape:
        raise ValueError("dout must have q's shape")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    rc = _load().oracle_attn_bwd_bias(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), B, Hq, Hkv, Nq, Nk,
                                      D, float(scale), causal_code(causal),
                                      None if bias is None else _ptr(bias), *bstr,
                                      _ptr(dq), _ptr(dk), _ptr(dv),
                                      int(threads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_bwd_bias failed with {rc}")
    return dq, dk, dv


def causal_code(causal) -> int:
    """0 none, 1 top-left (True), 2 bottom-right ("bottom_right")."""
    if causal is None or causal is False:
        return 0
    if causal is True:
        return 1
    if isinstance(causal, str):
        return {"none": 0, "top_left": 1, "bottom_right": 2}[causal]
    return int(causal)


def attended_keys(i: int, nk: int, causal, nq: int | None = None) -> int:
    """How many keys query i attends to: all, j <= i (top-left), or
    j <= i + nk - nq (bottom-right; needs nq)."""
    c = causal_code(causal)
    if c == 0:
        return nk
    pos = i + (nk - nq) if c == 2 else i
    return max(0, min(pos + 1, nk))
