"""Split-key forward (attn_fwd_splitkv) and the bottom-right causal mask on the
GPU, through the C ABI, against the fp64 oracle on the same seeded, rounded
inputs.  Every row of every case is checked.

The shapes are those of decoding against a KV cache (one or a few new query
positions per head, long key sequences, GQA as in the Qwen 2.5 model of the
forum post's LLM-inference table), plus prefill shapes cut into key ranges so
that some ranges hold no visible key for some query tiles.
"""
import numpy as np
import pytest
import torch

from tests import helpers
from tiled_memory_efficient_gb300 import _lib, inputs

pytestmark = pytest.mark.gpu

F16, BF16 = torch.float16, torch.bfloat16


def make(B, Hq, Hkv, Nq, Nk, D, dtype, seed):
    return inputs.make_custom(B, Hq, Hkv, Nq, Nk, D, dtype, seed=seed)


def check_all_rows(x, out, lse, causal, what):
    q = x["q"]
    rows = np.arange(q.shape[0] * q.shape[1] * q.shape[2])
    o_ref, lse_ref = helpers.oracle_rows(q, x["k"], x["v"], rows, causal)
    o_gpu, lse_gpu = helpers.gpu_rows(out, lse, rows)
    return helpers.assert_fwd_close(o_gpu, lse_gpu, o_ref, lse_ref, q.dtype, what)


CASES = [
    # B, Hq, Hkv, Nq, Nk, D, dtype, causal, splits (None: the library's choice)
    (2, 14, 2, 1, 4133, 64, F16, "bottom_right", None),   # decode, GQA 7, ragged keys
    (2, 14, 2, 1, 4133, 64, F16, False, 7),
    (1, 4, 4, 3, 9000, 128, BF16, "bottom_right", 64),    # 71 tiles in 64 requested ranges
    (1, 8, 2, 200, 5000, 128, BF16, "bottom_right", 5),   # two query tiles, ragged
    (1, 2, 2, 1000, 1000, 64, F16, True, 4),              # empty ranges above the diagonal
    (1, 14, 2, 130, 2100, 64, F16, True, 6),              # top-left, Nq < Nk, tiles cross heads
    (1, 2, 2, 700, 700, 128, BF16, "bottom_right", 3),    # square: bottom-right = top-left
    (1, 3, 3, 17, 300, 64, F16, False, 256),              # more ranges asked than key tiles
    (1, 2, 2, 64, 128, 64, F16, False, 2),                # one key tile: a single range
]


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,D,dtype,causal,splits", CASES)
def test_splitkv_matches_oracle(cuda_lib, B, Hq, Hkv, Nq, Nk, D, dtype, causal, splits):
    x = make(B, Hq, Hkv, Nq, Nk, D, dtype, seed=Nq * 7919 + Nk)
    q, k, v = (x[n].cuda() for n in "qkv")
    out, lse = _lib.attn_fwd_splitkv(q, k, v, causal=causal, splits=splits)
    assert _lib.sync_status() == _lib.ATTN_OK
    eo, el = check_all_rows(x, out, lse, causal, f"splitkv {B,Hq,Hkv,Nq,Nk,D} {causal} {splits}")
    print(f"splits={splits}: max|dO|={eo:.2e} max|dLSE|={el:.2e}")


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,D,dtype", [
    (1, 14, 2, 100, 3000, 64, F16),
    (2, 4, 4, 1, 777, 128, BF16),
    (1, 2, 2, 300, 301, 128, F16),
])
def test_bottom_right_unsplit_matches_oracle(cuda_lib, B, Hq, Hkv, Nq, Nk, D, dtype):
    x = make(B, Hq, Hkv, Nq, Nk, D, dtype, seed=Nk)
    q, k, v = (x[n].cuda() for n in "qkv")
    out, lse = _lib.attn_fwd(q, k, v, causal="bottom_right")
    assert _lib.sync_status() == _lib.ATTN_OK
    check_all_rows(x, out, lse, "bottom_right", f"bottom-right {B,Hq,Hkv,Nq,Nk,D}")


def test_single_range_is_attn_fwd_bitwise(cuda_lib):
    x = make(1, 14, 2, 33, 2000, 64, F16, seed=5)
    q, k, v = (x[n].cuda() for n in "qkv")
    a = _lib.attn_fwd(q, k, v, causal="bottom_right")
    b = _lib.attn_fwd_splitkv(q, k, v, causal="bottom_right", splits=1)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_square_bottom_right_is_top_left_bitwise(cuda_lib):
    x = make(1, 4, 2, 520, 520, 128, BF16, seed=6)
    q, k, v = (x[n].cuda() for n in "qkv")
    a = _lib.attn_fwd(q, k, v, causal=True)
    b = _lib.attn_fwd(q, k, v, causal="bottom_right")
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_splitkv_is_deterministic(cuda_lib):
    x = make(2, 14, 2, 1, 20000, 64, F16, seed=7)
    q, k, v = (x[n].cuda() for n in "qkv")
    a = _lib.attn_fwd_splitkv(q, k, v, causal="bottom_right", splits=40)
    b = _lib.attn_fwd_splitkv(q, k, v, causal="bottom_right", splits=40)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_long_kv_cache_decode(cuda_lib):
    """A long cache: 4 sequences, 14 query heads on 2 KV heads, one new token
    each, 65,613 cached keys (ragged tail), the library's range count."""
    x = make(4, 14, 2, 1, 65613, 64, F16, seed=8)
    q, k, v = (x[n].cuda() for n in "qkv")
    splits = _lib.num_splits(4, 14, 2, 1, 65613, 64)
    assert splits > 1
    out, lse = _lib.attn_fwd_splitkv(q, k, v, causal="bottom_right")
    assert _lib.sync_status() == _lib.ATTN_OK
    eo, el = check_all_rows(x, out, lse, "bottom_right", "decode 65613")
    print(f"decode 65613 keys, {splits} ranges: max|dO|={eo:.2e} max|dLSE|={el:.2e}")


def test_splitkv_rejects_short_workspace(cuda_lib):
    x = make(1, 2, 2, 1, 4096, 64, F16, seed=9)
    q, k, v = (x[n].cuda() for n in "qkv")
    need = _lib.splitkv_workspace_size(1, 2, 2, 1, 4096, 64, 8)
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(_lib.AttnError) as e:
        _lib.attn_fwd_splitkv(q, k, v, splits=8, workspace=ws)
    assert e.value.code == _lib.ATTN_ERR_WORKSPACE


@pytest.mark.parametrize("nk", inputs.WORKLOADS["gqa_decode"].seq_lens)
def test_gqa_decode_workload_every_row(cuda_lib, nk):
    """The decode workload exactly as the benchmark times it (8 sequences,
    14 query heads on 2 KV heads, one new token, bottom-right causal, the
    library's range count): every output row against the oracle."""
    w = inputs.WORKLOADS["gqa_decode"]
    x = inputs.make_inputs(w, nk)
    q, k, v = (x[n].cuda() for n in "qkv")
    out, lse = _lib.attn_fwd_splitkv(q, k, v, causal=w.causal)
    assert _lib.sync_status() == _lib.ATTN_OK
    check_all_rows(x, out, lse, w.causal, f"gqa_decode Nk={nk}")
