"""ctypes binding of the C ABI in include/attn.h (argument marshalling only).

Every step of the computation runs in libattn.so's CUDA kernels; torch is used
only to own device memory and to name the current stream.  There is no CPU
fallback: if the library is missing or the device is not an sm_103 GPU, the
calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os
import re
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_build", "libattn.so")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")
HEADERS = [os.path.join(INCLUDE, "attn.h"), os.path.join(INCLUDE, "ffn.h")]

ATTN_OK = 0
ATTN_ERR_INVALID = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_ALIGN = 3
ATTN_ERR_CUDA = 4
ATTN_ERR_TIMEOUT = 5
ATTN_ERR_WORKSPACE = 6
ATTN_ERR_MISMATCH = 7
FFN_ACTS = {"none": 0, "relu": 1, "gelu_tanh": 2, "silu": 3, "swiglu": 4}
ATTN_F16 = 0
ATTN_BF16 = 1
ATTN_CAUSAL_NONE = 0
ATTN_CAUSAL_TOP_LEFT = 1
ATTN_CAUSAL_BOTTOM_RIGHT = 2
ATTN_MASK_BOOL = 1
ATTN_MASK_ADDITIVE = 2
_CAUSAL_NAMES = {"none": ATTN_CAUSAL_NONE, "top_left": ATTN_CAUSAL_TOP_LEFT,
                 "bottom_right": ATTN_CAUSAL_BOTTOM_RIGHT}

_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_i = ctypes.c_int
_SIGNATURES = {
    "attn_fwd": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, ctypes.c_float, _i, _i, _vp],
                 _i),
    "attn_fwd_masked": ([_vp, _vp, _vp, _vp, _vp, _vp, _i, ctypes.c_longlong, ctypes.c_longlong,
                         ctypes.c_longlong, _i, _i, _i, _i, _i, _i, ctypes.c_float, _i, _i, _vp],
                        _i),
    "attn_fwd_splitkv": ([_vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _i, _i, _i, _i, _i, _i,
                          ctypes.c_float, _i, _i, _i, _vp], _i),
    "attn_fwd_splitkv_workspace_size": ([_i, _i, _i, _i, _i, _i, _i], ctypes.c_size_t),
    "attn_fwd_ws": ([_vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _i, _i, _i, _i, _i, _i,
                     ctypes.c_float, _i, _i, _vp], _i),
    "attn_fwd_workspace_size": ([_i, _i, _i, _i, _i, _i, _i], ctypes.c_size_t),
    "attn_fwd_ws_splits": ([_i, _i, _i, _i, _i, _i, _i, _i], _i),
    "attn_fwd_half_positions": ([_i, _i, _i, _i, _i, _i, _i, _i, _i], _i),
    "attn_bwd_splits": ([_i, _i, _i, _i, _i, _i, _i, _i], _i),
    "attn_fwd_num_splits": ([_i, _i, _i, _i, _i, _i, _i], _i),
    "attn_bwd_workspace_size": ([_i, _i, _i, _i, _i, _i, _i], ctypes.c_size_t),
    "attn_bwd": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t,
                  _i, _i, _i, _i, _i, _i, ctypes.c_float, _i, _i, _vp], _i),
    "attn_bwd_masked": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp,
                         _i, ctypes.c_longlong, ctypes.c_longlong, ctypes.c_longlong,
                         _i, _i, _i, _i, _i, _i, ctypes.c_float, _i, _i, _vp], _i),
    "attn_bwd_noalloc": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                          _i, _i, _i, _i, _i, _i, ctypes.c_float, _i, _i, _vp], _i),
    "attn_sync_status": ([_vp], _i),
    "ffn_workspace_size": ([_i, _i, _i], ctypes.c_size_t),
    "ffn_forward": ([_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, ctypes.c_size_t, _i,
                     _vp], _i),
    "ffn_check_chunking": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp,
                            ctypes.c_size_t, _i, _vp], _i),
    "attn_selftest_timeout": ([ctypes.c_ulonglong, _vp], _i),
    "attn_strerror": ([_i], ctypes.c_char_p),
    "attn_version": ([], _i),
}


class AttnError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {code} ({strerror(code)})")


def declared_functions() -> list:
    """Names of the functions include/attn.h and include/ffn.h declare."""
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names.update(re.findall(r"\b((?:attn|ffn)_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def load(path: str | None = None):
    """dlopen libattn.so (built by __graft_entry__.build()) and set signatures."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(f"{p} is missing: run __graft_entry__.build() first")
            lib = ctypes.CDLL(p)
            for name, (args, res) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


def strerror(code: int) -> str:
    return load().attn_strerror(code).decode()


def _stream_handle(device) -> int:
    import torch
    return torch.cuda.current_stream(device).cuda_stream


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return ATTN_F16
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    raise TypeError(f"unsupported dtype {t.dtype}: use float16 or bfloat16")


def causal_code(causal) -> int:
    """Mask code of the C ABI: False/None -> none, True -> top-left (the SDPA
    is_causal convention), or one of "none", "top_left", "bottom_right", or
    the integer code itself."""
    if causal is None or causal is False:
        return ATTN_CAUSAL_NONE
    if causal is True:
        return ATTN_CAUSAL_TOP_LEFT
    if isinstance(causal, str):
        if causal not in _CAUSAL_NAMES:
            raise ValueError(f"causal must be one of {sorted(_CAUSAL_NAMES)}, got {causal!r}")
        return _CAUSAL_NAMES[causal]
    return int(causal)


def _check(q, k, v):
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous [B, H, N, D]")
        if t.dim() != 4:
            raise ValueError(f"{name} must be 4-D [B, H, N, D]")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype")
    if k.shape != v.shape or k.shape[0] != q.shape[0] or k.shape[3] != q.shape[3]:
        raise ValueError(f"shapes q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")


def prepare_mask(mask, q, Nk: int):
    """An SDPA attn_mask as the C ABI's (tensor, kind, strides): bool stays a
    byte mask (True keeps the key); a floating mask becomes an additive bias
    in q's dtype.  It must broadcast to [B, Hq, Nq, Nk].  If its rows are not
    16-byte aligned it is copied into a padded buffer (same values),
    allocated on the current stream, the one the kernel runs on."""
    import torch
    B, Hq, Nq, _ = q.shape
    if not isinstance(mask, torch.Tensor) or mask.device != q.device:
        raise ValueError("attn_mask must be a tensor on q's device")
    if mask.dtype == torch.bool:
        kind, m = ATTN_MASK_BOOL, mask
    elif mask.is_floating_point():
        kind, m = ATTN_MASK_ADDITIVE, mask.to(q.dtype)
    else:
        raise TypeError(f"attn_mask dtype {mask.dtype} is neither bool nor floating point")
    while m.dim() < 4:
        m = m.unsqueeze(0)
    if m.dim() != 4 or m.shape[-1] != Nk or any(
            d not in (1, full) for d, full in zip(m.shape[:3], (B, Hq, Nq))):
        raise ValueError(f"attn_mask shape {tuple(mask.shape)} does not broadcast to "
                         f"{(B, Hq, Nq, Nk)}")
    if m.stride(-1) != 1:
        m = m.contiguous()
    esz = m.element_size()

    def strides(t):
        return [0 if t.shape[i] == 1 else t.stride(i) for i in range(3)]
    st = strides(m)
    if m.data_ptr() % 16 or any((x * esz) % 16 for x in st):
        per = 16 // esz
        buf = torch.zeros((*m.shape[:3], (Nk + per - 1) // per * per), dtype=m.dtype,
                          device=m.device)
        buf[..., :Nk] = m
        m = buf
        st = strides(m)
    return m, kind, st


def attn_fwd(q, k, v, causal=False, scale: float | None = None, out=None, lse=None, mask=None):
    """O, LSE = attention(q, k, v).  q [B,Hq,Nq,D]; k, v [B,Hkv,Nk,D] (CUDA).

    Returns (out [B,Hq,Nq,D] in q's dtype, lse [B,Hq,Nq] fp32 natural log).
    causal: see causal_code.  mask: optional SDPA-style attn_mask (see
    prepare_mask).  Enqueued on torch's current stream; no synchronisation.
    """
    import torch
    _check(q, k, v)
    B, Hq, Nq, D = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Nq), device=q.device, dtype=torch.float32)
    if mask is not None:
        m, kind, (sb, sh, sq) = prepare_mask(mask, q, Nk)
        rc = load().attn_fwd_masked(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                    lse.data_ptr(), m.data_ptr(), kind, sb, sh, sq, B, Hq, Hkv, Nq,
                                    Nk, D, float(scale), causal_code(causal), _dtype_code(q),
                                    _stream_handle(q.device))
        if rc != ATTN_OK:
            raise AttnError("attn_fwd_masked", rc)
        # (a converted / padded copy was allocated on this stream, after which
        # the kernel is queued: the allocator reuses it only for later work
        # on the same stream, so it may be released now)
        return out, lse
    rc = load().attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                         lse.data_ptr(), B, Hq, Hkv, Nq, Nk, D, float(scale), causal_code(causal),
                         _dtype_code(q), _stream_handle(q.device))
    if rc != ATTN_OK:
        raise AttnError("attn_fwd", rc)
    return out, lse


def fwd_workspace_size(B, Hq, Hkv, Nq, Nk, D, dtype) -> int:
    """Bytes of workspace attn_fwd_ws needs on the current device (0: none)."""
    code = dtype if isinstance(dtype, int) else (ATTN_BF16 if str(dtype).endswith("bfloat16")
                                                 else ATTN_F16)
    return load().attn_fwd_workspace_size(B, Hq, Hkv, Nq, Nk, D, code)


def fwd_ws_splits(B, Hq, Hkv, Nq, Nk, D, causal=False, num_sms: int = 0) -> int:
    """Key ranges attn_fwd_ws cuts its cut units into on a device of num_sms
    SMs (0: the current device; 1: the grid is not cut, no merge kernel)."""
    return load().attn_fwd_ws_splits(B, Hq, Hkv, Nq, Nk, D, causal_code(causal), num_sms)


def fwd_half_positions(B, Hq, Hkv, Nq, Nk, D, causal=True, dtype="float16",
                       num_sms: int = 0) -> int:
    """Heaviest pair positions per head that the causal forward runs as two
    one-tile CTAs per pair (0: none; see attn_fwd_half_positions)."""
    code = dtype if isinstance(dtype, int) else (ATTN_BF16 if str(dtype).endswith("bfloat16")
                                                 else ATTN_F16)
    return load().attn_fwd_half_positions(B, Hq, Hkv, Nq, Nk, D, causal_code(causal), code,
                                          num_sms)


def bwd_splits(B, Hq, Hkv, Nq, Nk, D, causal=False, num_sms: int = 0) -> int:
    """Query ranges attn_bwd cuts the dK/dV work into with its recommended
    workspace on a device of num_sms SMs (0: the current device; 1: no
    partial-sum kernel)."""
    return load().attn_bwd_splits(B, Hq, Hkv, Nq, Nk, D, causal_code(causal), num_sms)


def attn_fwd_ws(q, k, v, causal=False, scale: float | None = None, out=None, lse=None,
                workspace=None):
    """attn_fwd through attn_fwd_ws, with a workspace (allocated here on q's
    device when not given): for bf16 inputs the value tiles are converted to
    fp16 once into it, instead of inside every CTA, and grids that fill the
    GPU unevenly cut some units' keys into ranges whose partials it holds."""
    import torch
    _check(q, k, v)
    B, Hq, Nq, D = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Nq), device=q.device, dtype=torch.float32)
    lib = load()
    ws_bytes = lib.attn_fwd_workspace_size(B, Hq, Hkv, Nq, Nk, D, _dtype_code(q))
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes, device=q.device, dtype=torch.uint8)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib.attn_fwd_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                         ws_ptr, ws_len, B, Hq, Hkv, Nq, Nk, D, float(scale), causal_code(causal),
                         _dtype_code(q), _stream_handle(q.device))
    if rc != ATTN_OK:
        raise AttnError("attn_fwd_ws", rc)
    return out, lse


def num_splits(B, Hq, Hkv, Nq, Nk, D, num_sms: int = 0) -> int:
    """The library's key-range count for attn_fwd_splitkv (num_sms 0: ask the
    current device)."""
    return load().attn_fwd_num_splits(B, Hq, Hkv, Nq, Nk, D, int(num_sms))


def splitkv_workspace_size(B, Hq, Hkv, Nq, Nk, D, splits: int) -> int:
    return load().attn_fwd_splitkv_workspace_size(B, Hq, Hkv, Nq, Nk, D, int(splits))


def attn_fwd_splitkv(q, k, v, causal=False, scale: float | None = None, splits: int | None = None,
                     out=None, lse=None, workspace=None):
    """attn_fwd with the keys cut into ``splits`` ranges (None: the library's
    choice for this device) and the partial results merged; for short query
    blocks against long keys, e.g. decoding against a KV cache (use
    causal="bottom_right" when the queries are the newest positions)."""
    import torch
    _check(q, k, v)
    B, Hq, Nq, D = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    lib = load()
    if splits is None:
        splits = lib.attn_fwd_num_splits(B, Hq, Hkv, Nq, Nk, D, 0)
    ws_bytes = lib.attn_fwd_splitkv_workspace_size(B, Hq, Hkv, Nq, Nk, D, int(splits))
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes, device=q.device, dtype=torch.uint8)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Nq), device=q.device, dtype=torch.float32)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib.attn_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                              lse.data_ptr(), ws_ptr, ws_len, B, Hq, Hkv, Nq, Nk, D, float(scale),
                              causal_code(causal), _dtype_code(q), int(splits),
                              _stream_handle(q.device))
    if rc != ATTN_OK:
        raise AttnError("attn_fwd_splitkv", rc)
    return out, lse


def attn_bwd(q, k, v, out, dout, lse, causal: bool = False, scale: float | None = None,
             dq=None, dk=None, dv=None, workspace=None, mask=None):
    """dq, dk, dv of attn_fwd (dk, dv summed over each GQA group); with the
    forward's mask, of attn_fwd(mask=...)."""
    import torch
    _check(q, k, v)
    B, Hq, Nq, D = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dt = _dtype_code(q)
    lib = load()
    ws_bytes = lib.attn_bwd_workspace_size(B, Hq, Hkv, Nq, Nk, D, dt)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), device=q.device, dtype=torch.uint8)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if mask is not None:
        m, kind, (sb, sh, sq) = prepare_mask(mask, q, Nk)
        rc = lib.attn_bwd_masked(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                 dout.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                 dv.data_ptr(), workspace.data_ptr(),
                                 workspace.numel() * workspace.element_size(), m.data_ptr(), kind,
                                 sb, sh, sq, B, Hq, Hkv, Nq, Nk, D, float(scale),
                                 causal_code(causal), dt, _stream_handle(q.device))
        if rc != ATTN_OK:
            raise AttnError("attn_bwd_masked", rc)
        return dq, dk, dv
    rc = lib.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), dout.data_ptr(),
                      lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                      workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                      B, Hq, Hkv, Nq, Nk, D, float(scale), causal_code(causal), dt,
                      _stream_handle(q.device))
    if rc != ATTN_OK:
        raise AttnError("attn_bwd", rc)
    return dq, dk, dv


def sync_status(device=None) -> int:
    """Synchronise the current stream and return (and clear) the device status."""
    import torch
    dev = device if device is not None else torch.cuda.current_device()
    return load().attn_sync_status(_stream_handle(dev))


def _ptr(t):
    return None if t is None else t.data_ptr()


def ffn_forward(x, w1, b1, w2, b2, act: str = "gelu_tanh", chunk: int = 4096, out=None,
                workspace=None):
    """y = act(x W1^T + b1) W2^T + b2 over x [T, d_model], `chunk` tokens at a
    time (include/ffn.h).  swiglu: W1 = [Wg; Wu] of 2*d_ff rows."""
    import torch
    T, d_model = x.shape
    d_ff = w2.shape[1]
    for name, t in (("x", x), ("w1", w1), ("w2", w2)):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != x.dtype:
            raise ValueError(f"{name} must be a contiguous CUDA tensor of x's dtype")
    lib = load()
    if workspace is None:
        workspace = torch.empty(max(16, lib.ffn_workspace_size(T, d_ff, chunk)),
                                dtype=torch.uint8, device=x.device)
    y = torch.empty((T, d_model), dtype=x.dtype, device=x.device) if out is None else out
    rc = lib.ffn_forward(x.data_ptr(), w1.data_ptr(), _ptr(b1), w2.data_ptr(), _ptr(b2),
                         y.data_ptr(), T, d_model, d_ff, FFN_ACTS[act], int(chunk),
                         workspace.data_ptr(), workspace.numel(), _dtype_code(x),
                         _stream_handle(x.device))
    if rc != ATTN_OK:
        raise AttnError("ffn_forward", rc)
    return y


def ffn_check_chunking(x, w1, b1, w2, b2, act: str = "gelu_tanh", chunk: int = 4096):
    """Runs the FFN chunked and unchunked and compares bit for bit on the
    device; returns (y, ok)."""
    import torch
    T, d_model = x.shape
    d_ff = w2.shape[1]
    lib = load()
    ws = torch.empty(max(16, lib.ffn_workspace_size(T, d_ff, T)), dtype=torch.uint8,
                     device=x.device)
    y = torch.empty((T, d_model), dtype=x.dtype, device=x.device)
    y_ref = torch.empty_like(y)
    rc = lib.ffn_check_chunking(x.data_ptr(), w1.data_ptr(), _ptr(b1), w2.data_ptr(), _ptr(b2),
                                y.data_ptr(), y_ref.data_ptr(), T, d_model, d_ff, FFN_ACTS[act],
                                int(chunk), ws.data_ptr(), ws.numel(), _dtype_code(x),
                                _stream_handle(x.device))
    if rc not in (ATTN_OK, ATTN_ERR_MISMATCH):
        raise AttnError("ffn_check_chunking", rc)
    return y, rc == ATTN_OK
