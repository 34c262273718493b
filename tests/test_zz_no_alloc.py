"""attn_bwd_noalloc: the backward for callers that cannot allocate device
memory (it takes its scratch from a fixed array in the library instead of a
caller-provided workspace).  Checked through the C ABI against attn_bwd with a
caller workspace, on two calls in a row (the array is shared and keeps the
previous call's contents).  This file is collected last on purpose.
"""
import pytest
import torch

from tests import helpers
from tiled_memory_efficient_gb300 import _lib, inputs

pytestmark = pytest.mark.gpu


def _ptr(t):
    return t.data_ptr()


def test_noalloc_matches_workspace_entry_point_on_two_calls(cuda_lib):
    lib = cuda_lib
    B, Hq, Hkv, N, D = 1, 4, 2, 300, 128
    dtype = torch.bfloat16
    x = inputs.make_custom(B, Hq, Hkv, N, N, D, dtype, seed=31, with_grad=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    out, lse = _lib.attn_fwd(q, k, v, causal=True)
    ref = _lib.attn_bwd(q, k, v, out, do, lse, causal=True)
    stream = torch.cuda.current_stream().cuda_stream
    scale = 1.0 / D ** 0.5
    for call in range(2):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        rc = lib.attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(do), _ptr(lse),
                                  _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, N, N, D, scale, 1,
                                  _lib.ATTN_BF16, stream)
        assert rc == _lib.ATTN_OK, _lib.strerror(rc)
        assert lib.attn_sync_status(stream) == _lib.ATTN_OK
        for name, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            helpers.assert_close_elementwise(got.double().cpu().numpy(),
                                             want.double().cpu().numpy(),
                                             helpers.TOL_BWD[dtype], dtype, f"call {call}", name)


def test_noalloc_rejects_problems_beyond_its_scratch(cuda_lib):
    lib = cuda_lib
    # 2 arrays x 64 groups x 16384 rows x 4 bytes = 8 MiB > 4 MiB: rejected before launch
    need = lib.attn_bwd_workspace_size(1, 64, 64, 16384, 16384, 64, 0)
    assert need > 4 * 1024 * 1024
    rc = lib.attn_bwd_noalloc(256, 256, 256, 256, 256, 256, 256, 256, 256,
                              1, 64, 64, 16384, 16384, 64, 0.125, 0, 0, None)
    assert rc == _lib.ATTN_ERR_WORKSPACE
