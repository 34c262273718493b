"""attn_bwd_noalloc: the backward for callers that cannot allocate device
memory (it takes its scratch from a fixed array in the library instead of a
caller-provided workspace).  Checked through the C ABI against attn_bwd with a
caller workspace of the same size, bit for bit, and with the recommended
workspace within the backward tolerance, on calls in a row (the array is
shared and keeps the previous call's contents).  This file is collected last
on purpose.
"""
import pytest
import torch

from tests import helpers
from tiled_memory_efficient_gb300 import _lib, inputs

pytestmark = pytest.mark.gpu


def _ptr(t):
    return t.data_ptr()


SCRATCH = 4 << 20   # the library's fixed scratch array


def _noalloc(lib, x, causal, dtype_code):
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    B, Hq, Nq, D = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    out, lse = _lib.attn_fwd(q, k, v, causal=causal)
    # attn_bwd with a caller workspace of the same size as the scratch array
    # (the workspace size decides how the dK/dV work is cut, hence the bits),
    # and with the size attn_bwd_workspace_size recommends
    same = _lib.attn_bwd(q, k, v, out, do, lse, causal=causal,
                         workspace=torch.empty(SCRATCH, device="cuda", dtype=torch.uint8))
    rec = _lib.attn_bwd(q, k, v, out, do, lse, causal=causal)
    stream = torch.cuda.current_stream().cuda_stream
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    rc = lib.attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(do), _ptr(lse),
                              _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, Nq, Nk, D,
                              1.0 / D ** 0.5, 1 if causal else 0, dtype_code, stream)
    assert rc == _lib.ATTN_OK, _lib.strerror(rc)
    assert lib.attn_sync_status(stream) == _lib.ATTN_OK
    return (dq, dk, dv), same, rec


def test_noalloc_matches_workspace_entry_point_on_two_calls(cuda_lib):
    """The backward is deterministic for a given workspace size, so the
    allocation-free call must give the same bits as attn_bwd with a 4 MiB
    workspace, and agree with attn_bwd at its recommended workspace within the
    backward tolerance.  The first call is a larger problem of another shape
    (it leaves its own data in more of the shared scratch); the next two are a
    smaller problem that reads a scratch region the first call wrote."""
    lib = cuda_lib
    dtype = torch.bfloat16
    big = inputs.make_custom(2, 8, 2, 1000, 1000, 128, dtype, seed=30, with_grad=True)
    small = inputs.make_custom(1, 4, 2, 300, 300, 128, dtype, seed=31, with_grad=True)
    for call, (x, causal) in enumerate(((big, False), (small, True), (small, True))):
        got, same, rec = _noalloc(lib, x, causal, _lib.ATTN_BF16)
        for name, g, r, r2 in zip(("dq", "dk", "dv"), got, same, rec):
            assert torch.equal(g, r), f"call {call}: {name} differs from attn_bwd (4 MiB)"
            helpers.assert_close_elementwise(g.double().cpu().numpy(), r2.double().cpu().numpy(),
                                             helpers.TOL_BWD[dtype], dtype, f"noalloc call {call}",
                                             name)


def test_noalloc_rejects_problems_beyond_its_scratch(cuda_lib):
    lib = cuda_lib
    # 2 arrays x 64 groups x 16384 rows x 4 bytes = 8 MiB > 4 MiB: rejected before launch
    need = lib.attn_bwd_workspace_size(1, 64, 64, 16384, 16384, 64, 0)
    assert need > 4 * 1024 * 1024
    rc = lib.attn_bwd_noalloc(256, 256, 256, 256, 256, 256, 256, 256, 256,
                              1, 64, 64, 16384, 16384, 64, 0.125, 0, 0, None)
    assert rc == _lib.ATTN_ERR_WORKSPACE
