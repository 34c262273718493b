"""Backward parity on the GPU: dQ, dK, dV from the CUDA path (forward then
backward, through the C ABI) against the fp64 oracle's gradients on the same
seeded, rounded inputs.  Small shapes and the training workload (B=2, H=16,
N=8192, D=128, bf16, causal; every head, each an independent MHA problem, at
the full sequence length) are checked in full.
"""
import numpy as np
import pytest
import torch

import oracle
from tests import helpers
from tiled_memory_efficient_gb300 import _lib, inputs

pytestmark = pytest.mark.gpu

F16, BF16 = torch.float16, torch.bfloat16


def gpu_grads(x, causal, scale=None):
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    out, lse = _lib.attn_fwd(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = _lib.attn_bwd(q, k, v, out, do, lse, causal=causal, scale=scale)
    assert _lib.sync_status() == _lib.ATTN_OK
    return dq, dk, dv


def check(got, ref, dtype, what):
    tol = helpers.TOL_BWD[dtype]
    errs = []
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        errs.append(helpers.assert_close_elementwise(
            g.double().cpu().numpy(), r, tol, dtype, what, name))
    return errs


SMALL = [
    # B, Hq, Hkv, Nq, Nk, D, dtype, causal
    (1, 2, 2, 128, 128, 64, F16, False),
    (1, 2, 2, 256, 256, 128, BF16, True),
    (1, 2, 2, 300, 300, 64, F16, True),      # ragged tail
    (2, 4, 2, 200, 333, 64, BF16, False),    # GQA G=2, Nq != Nk, ragged
    (1, 14, 2, 250, 250, 64, F16, True),     # GQA G=7, tiles cross head boundaries
    (1, 7, 1, 37, 37, 128, BF16, True),      # tiny heads flattened into one tile
    (1, 2, 2, 129, 700, 128, F16, True),     # Nq < Nk (late key tiles see no query)
    (1, 3, 3, 1, 1, 64, F16, False),         # single query and key
    (1, 2, 2, 1024, 1024, 128, BF16, True),  # several tiles each way
]


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,D,dtype,causal", SMALL)
def test_backward_small_shapes(cuda_lib, B, Hq, Hkv, Nq, Nk, D, dtype, causal):
    x = inputs.make_custom(B, Hq, Hkv, Nq, Nk, D, dtype, seed=3 * Nq + Nk + D, with_grad=True)
    got = gpu_grads(x, causal)
    ref = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], causal=causal)
    errs = check(got, ref, dtype, f"{(B, Hq, Hkv, Nq, Nk, D, dtype, causal)}")
    print(f"{(B, Hq, Hkv, Nq, Nk, D, str(dtype), causal)}: max err dq/dk/dv = {errs}")


def test_backward_explicit_scale(cuda_lib):
    x = inputs.make_custom(1, 2, 2, 256, 256, 64, F16, seed=77, with_grad=True)
    got = gpu_grads(x, False, scale=0.2)
    ref = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], causal=False, scale=0.2)
    check(got, ref, F16, "scale=0.2")


def test_training_workload_every_head(cuda_lib):
    """The training workload (B=2, H=16, N=8192, D=128, bf16, causal) as the
    benchmark runs it: dQ, dK and dV of every head against the oracle."""
    w = inputs.WORKLOADS["training"]
    n = w.seq_lens[0]
    x = inputs.make_inputs(w, n)
    dq, dk, dv = gpu_grads(x, w.causal)
    for b in range(w.B):
        for h in range(w.Hq):
            sl = {m: x[m][b:b + 1, h:h + 1] for m in ("q", "k", "v", "do")}
            ref = oracle.attention_bwd(sl["q"], sl["k"], sl["v"], sl["do"], causal=w.causal)
            got = (dq[b:b + 1, h:h + 1], dk[b:b + 1, h:h + 1], dv[b:b + 1, h:h + 1])
            errs = check(got, ref, w.dtype, f"training head b={b} h={h}")
            print(f"training N={n} head ({b},{h}): max err dq/dk/dv = {errs}")


def test_backward_deterministic(cuda_lib):
    x = inputs.make_custom(1, 4, 2, 500, 500, 128, BF16, seed=21, with_grad=True)
    g1 = gpu_grads(x, True)
    g2 = gpu_grads(x, True)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


def test_backward_chain_on_a_side_stream(cuda_lib):
    """The backward's kernels are chained as programmatic dependent launches
    (statistics, dQ, dK/dV, the reduction of the dK/dV ranges).  On a side
    stream, two calls back to back and plain kernels reading the gradients
    right after them (no host synchronisation in between) see exactly the
    default-stream results."""
    x = inputs.make_custom(1, 14, 2, 1024, 1024, 64, F16, seed=63, with_grad=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    out, lse = _lib.attn_fwd(q, k, v, causal=True)
    ref = _lib.attn_bwd(q, k, v, out, do, lse, causal=True)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        a = _lib.attn_bwd(q, k, v, out, do, lse, causal=True)
        b = _lib.attn_bwd(q, k, v, out, do, lse, causal=True)
        doubled = [t * 2 for t in (*a, *b)]   # ordinary kernels right behind the chain
    side.synchronize()
    assert _lib.sync_status() == _lib.ATTN_OK
    for r, ga, gb in zip(ref, a, b):
        assert torch.equal(r, ga) and torch.equal(r, gb)
    for d, r in zip(doubled, (*ref, *ref)):
        assert torch.equal(d, r * 2)


def test_backward_workspace_contents_do_not_matter(cuda_lib):
    x = inputs.make_custom(1, 2, 2, 300, 300, 64, F16, seed=22, with_grad=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    out, lse = _lib.attn_fwd(q, k, v, causal=True)
    lib = _lib.load()
    ws_bytes = lib.attn_bwd_workspace_size(1, 2, 2, 300, 300, 64, 0)
    res = []
    for fill in (0, 255):
        ws = torch.full((ws_bytes,), fill, device="cuda", dtype=torch.uint8)
        res.append(_lib.attn_bwd(q, k, v, out, do, lse, causal=True, workspace=ws))
    assert _lib.sync_status() == _lib.ATTN_OK
    for a, b in zip(*res):
        assert torch.equal(a, b)


def test_backward_range_plan(cuda_lib):
    """dK/dV query ranges on a 152-SM GB300: without the causal mask as many as
    fill one wave; with it enough that key tile 0's CTAs (which meet every
    query tile) do no more than the average work per SM."""
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the plan below is for 152 SMs")
    # GQA 14:2, D = 64: 2 KV groups x Nk / 128 key tiles
    assert _lib.bwd_splits(1, 14, 2, 2048, 2048, 64, True) == 9
    assert _lib.bwd_splits(1, 14, 2, 4096, 4096, 64, True) == 5
    assert _lib.bwd_splits(1, 14, 2, 8192, 8192, 64, True) == 3
    assert _lib.bwd_splits(1, 14, 2, 4096, 4096, 64, False) == 3
    assert _lib.bwd_splits(2, 16, 16, 8192, 8192, 128, True) == 1   # 2048 key-tile CTAs


def test_gqa_backward_split_every_head(cuda_lib):
    """GQA 14:2 at N = 2048 (causal, fp16): 2 KV heads x 16 key tiles are far
    fewer dK/dV CTAs than SMs, so the query tiles of each key tile are cut
    into ranges whose fp32 partial sums a last kernel adds.  Every head of
    every gradient against the oracle."""
    x = inputs.make_custom(1, 14, 2, 2048, 2048, 64, F16, seed=61, with_grad=True)
    got = gpu_grads(x, True)
    ref = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], causal=True)
    errs = check(got, ref, F16, "gqa 14:2 N=2048 split backward")
    print(f"gqa 14:2 N=2048 backward: max err dq/dk/dv = {errs}")


def test_backward_split_matches_unsplit(cuda_lib):
    """The same backward with the statistics-only workspace (no split of the
    dK/dV work) and with the recommended one agree within the tolerance, and
    each is deterministic."""
    x = inputs.make_custom(1, 8, 2, 1024, 1024, 128, BF16, seed=62, with_grad=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    out, lse = _lib.attn_fwd(q, k, v, causal=False)
    lib = _lib.load()
    rec = lib.attn_bwd_workspace_size(1, 8, 2, 1024, 1024, 128, 1)
    stats = 2 * 2 * (4 * 1024) * 4        # 2 arrays x 2 KV heads x G*Nq rows x 4 bytes
    assert rec > stats                    # 16 dK/dV CTAs: the work is split
    res = []
    for nbytes in (stats, rec, stats, rec):
        ws = torch.empty(nbytes, device="cuda", dtype=torch.uint8)
        res.append(_lib.attn_bwd(q, k, v, out, do, lse, causal=False, workspace=ws))
    assert _lib.sync_status() == _lib.ATTN_OK
    for a, b in zip(res[0], res[2]):
        assert torch.equal(a, b)
    for a, b in zip(res[1], res[3]):
        assert torch.equal(a, b)
    for name, a, b in zip(("dq", "dk", "dv"), res[0], res[1]):
        helpers.assert_close_elementwise(a.double().cpu().numpy(), b.double().cpu().numpy(),
                                         helpers.TOL_BWD[BF16], BF16, "split vs unsplit", name)
