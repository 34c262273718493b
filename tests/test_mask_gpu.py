"""Forward with an attention mask (attn_fwd_masked, the SDPA attn_mask) on the
GPU, through the C ABI, against the fp64 oracle on the same seeded inputs and
the same (dtype-rounded) mask.  Every row is checked; rows whose every key is
masked must come back as O = 0 and LSE = -inf, the oracle's reading."""
import math

import numpy as np
import pytest
import torch

import oracle
from tests import helpers
from tiled_memory_efficient_gb300 import _lib, inputs, sdpa

pytestmark = pytest.mark.gpu

F16, BF16 = torch.float16, torch.bfloat16


def make_mask(shape, kind, dtype, seed, Nk, empty_rows=False):
    g = torch.Generator().manual_seed(seed)
    if kind == "padding":                 # [B,1,1,Nk]: per-sequence key lengths
        B = shape[0]
        lens = torch.randint(Nk // 3, Nk + 1, (B,), generator=g)
        lens[0] = Nk
        return (torch.arange(Nk)[None, :] < lens[:, None]).reshape(B, 1, 1, Nk)
    if kind == "bool":
        m = torch.rand(shape, generator=g) > 0.35
        if empty_rows:
            m[..., 3, :] = False          # query row 3: no key at all
        return m
    m = torch.randn(shape, generator=g) * 2.0
    m = m.masked_fill(torch.rand(shape, generator=g) < 0.1, -math.inf)
    return m.to(dtype)                    # the kernel reads the bias in the input dtype


def check(x, out, lse, causal, mask, what):
    o_ref, lse_ref = oracle.attention_fwd(x["q"], x["k"], x["v"], causal=causal, mask=mask)
    o_gpu = out.double().cpu().numpy()
    lse_gpu = lse.double().cpu().numpy()
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse_gpu), empty), f"{what}: empty rows differ"
    assert np.all(o_gpu[empty] == 0.0), f"{what}: an empty row is not zero"
    keep = ~empty
    eo, el = helpers.assert_fwd_close(o_gpu[keep], lse_gpu[keep], o_ref[keep], lse_ref[keep],
                                      x["q"].dtype, what)
    return eo, el, int(empty.sum())


CASES = [
    # B, Hq, Hkv, Nq, Nk, D, dtype, causal, mask shape (None: padding), kind
    (2, 4, 4, 300, 300, 64, F16, False, None, "padding"),
    (1, 14, 2, 250, 517, 64, F16, True, (1, 1, 250, 517), "bool"),
    (1, 4, 2, 200, 333, 128, BF16, False, (1, 4, 200, 333), "additive"),
    (2, 3, 3, 128, 256, 128, BF16, True, (2, 3, 128, 256), "additive"),
    (1, 2, 2, 64, 1000, 64, F16, False, (1000,), "bool"),           # 1-D: over keys only
    (1, 6, 2, 77, 77, 128, F16, False, (77, 77), "additive"),       # rows not 16-byte aligned
    (2, 2, 1, 130, 140, 64, BF16, "bottom_right", (2, 1, 130, 140), "bool"),
    # key-only boolean masks at D=64 run in the split layout:
    (2, 14, 2, 200, 700, 64, BF16, True, None, "padding"),          # GQA, causal, Nq < Nk
    (2, 4, 4, 150, 260, 64, F16, "bottom_right", (2, 4, 1, 260), "bool"),  # per head, G = 1
    (1, 3, 3, 300, 4100, 64, BF16, False, (1, 1, 1, 4100), "bool"), # many key tiles, ragged
    # a per-head key mask with G > 1 takes the general masked layout:
    (1, 6, 2, 100, 300, 64, F16, False, (1, 6, 1, 300), "bool"),
    # D=64 general masks (bias staged in shared memory a key tile ahead):
    # GQA with partly real warps and a ragged last key tile; many whole key
    # tiles; heads of 90 rows, so Q tiles and warps span heads
    (1, 4, 2, 300, 600, 64, F16, False, (1, 4, 300, 600), "additive"),
    (1, 2, 2, 256, 2048, 64, F16, False, (1, 1, 256, 2048), "additive"),
    (1, 6, 2, 90, 390, 64, BF16, True, (1, 6, 90, 390), "additive"),
    (2, 2, 2, 200, 1024, 64, F16, "bottom_right", (2, 2, 200, 1024), "bool"),
]


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,D,dtype,causal,shape,kind", CASES)
def test_masked_forward_matches_oracle(cuda_lib, B, Hq, Hkv, Nq, Nk, D, dtype, causal, shape, kind):
    x = inputs.make_custom(B, Hq, Hkv, Nq, Nk, D, dtype, seed=Nq + 3 * Nk)
    mask = make_mask(shape or (B, 1, 1, Nk), kind, dtype, seed=Nk, Nk=Nk)
    q, k, v = (x[n].cuda() for n in "qkv")
    out, lse = _lib.attn_fwd(q, k, v, causal=causal, mask=mask.cuda())
    assert _lib.sync_status() == _lib.ATTN_OK
    eo, el, n_empty = check(x, out, lse, causal, mask, f"mask {kind} {shape} {causal}")
    print(f"{kind} {shape}: max|dO|={eo:.2e} max|dLSE|={el:.2e} empty rows={n_empty}")


@pytest.mark.parametrize("causal", [False, True])
def test_padding_mask_with_an_empty_sequence(cuda_lib, causal):
    """A key-padding mask whose second sequence keeps no key: every row of
    that sequence is O = 0, LSE = -inf; the first keeps 200 of 333 keys."""
    x = inputs.make_custom(2, 4, 2, 160, 333, 64, F16, seed=13)
    mask = (torch.arange(333)[None, :] < torch.tensor([200, 0])[:, None]).reshape(2, 1, 1, 333)
    q, k, v = (x[n].cuda() for n in "qkv")
    out, lse = _lib.attn_fwd(q, k, v, causal=causal, mask=mask.cuda())
    assert _lib.sync_status() == _lib.ATTN_OK
    _, _, n_empty = check(x, out, lse, causal, mask, f"padding with an empty sequence {causal}")
    assert n_empty >= 4 * 160


def test_rows_with_every_key_masked(cuda_lib):
    x = inputs.make_custom(1, 2, 2, 40, 300, 64, F16, seed=11)
    mask = make_mask((1, 2, 40, 300), "bool", F16, seed=12, Nk=300, empty_rows=True)
    q, k, v = (x[n].cuda() for n in "qkv")
    out, lse = _lib.attn_fwd(q, k, v, mask=mask.cuda())
    assert _lib.sync_status() == _lib.ATTN_OK
    _, _, n_empty = check(x, out, lse, False, mask, "empty rows")
    assert n_empty == 2


def test_all_true_mask_is_the_unmasked_forward(cuda_lib):
    """A mask that keeps every key gives the unmasked result (to rounding:
    the masked kernel scales the scores before the max)."""
    x = inputs.make_custom(1, 4, 4, 256, 384, 128, BF16, seed=13)
    q, k, v = (x[n].cuda() for n in "qkv")
    a = _lib.attn_fwd(q, k, v)
    b = _lib.attn_fwd(q, k, v, mask=torch.ones(384, dtype=torch.bool, device="cuda"))
    torch.cuda.synchronize()
    assert (a[0].float() - b[0].float()).abs().max().item() <= 1e-2
    assert (a[1] - b[1]).abs().max().item() <= 1e-4


@pytest.mark.parametrize("causal", [False, True])
def test_all_true_padding_mask_is_the_unmasked_forward_bitwise(cuda_lib, causal):
    """At D=64 a key-only keep-mask runs in the unmasked kernel's layout and
    only drops keys: keeping every key must give the unmasked result bit for
    bit."""
    x = inputs.make_custom(2, 14, 2, 300, 700, 64, F16, seed=16)
    q, k, v = (x[n].cuda() for n in "qkv")
    a = _lib.attn_fwd(q, k, v, causal=causal)
    b = _lib.attn_fwd(q, k, v, causal=causal,
                      mask=torch.ones((2, 1, 1, 700), dtype=torch.bool, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("causal", [False, True])
def test_all_true_general_mask_d64_is_the_unmasked_forward_bitwise(cuda_lib, causal):
    """At D=64 (fp16) a general boolean mask runs in the unmasked kernel's
    split layout, its bias staged in shared memory, and only drops keys:
    keeping every key must give the unmasked result bit for bit."""
    x = inputs.make_custom(1, 6, 2, 300, 700, 64, F16, seed=17)
    q, k, v = (x[n].cuda() for n in "qkv")
    a = _lib.attn_fwd(q, k, v, causal=causal)
    b = _lib.attn_fwd(q, k, v, causal=causal,
                      mask=torch.ones((1, 6, 300, 700), dtype=torch.bool, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_sdpa_with_attn_mask(cuda_lib):
    x = inputs.make_custom(2, 4, 2, 200, 200, 64, F16, seed=14)
    mask = make_mask((2, 1, 1, 200), "padding", F16, seed=15, Nk=200)
    q, k, v = (x[n].cuda() for n in "qkv")
    out = sdpa.scaled_dot_product_attention(q, k, v, attn_mask=mask.cuda(), enable_gqa=True)
    o_ref, _ = oracle.attention_fwd(x["q"], x["k"], x["v"], mask=mask)
    helpers.assert_close_elementwise(out.double().cpu().numpy(), o_ref, helpers.TOL_O[F16], F16,
                                     "sdpa mask", "O")


BWD_CASES = [
    # B, Hq, Hkv, N, D, dtype, causal, mask shape (None: padding), kind
    (2, 4, 2, 300, 64, F16, False, None, "padding"),
    (1, 4, 4, 257, 128, BF16, True, (1, 4, 257, 257), "additive"),
    (2, 6, 2, 200, 128, BF16, False, (2, 1, 200, 200), "bool"),
    (1, 14, 2, 90, 64, F16, True, (90, 90), "bool"),     # heads of 90 rows: tiles span heads
    # D=64 dQ stages 32 keys of bias per warp (16 warps): an additive bias with
    # a ragged last key tile and partly real warps; bf16 heads of 90 rows;
    # a GQA padding mask under the causal mask (keep bytes 32 keys at a time)
    (1, 4, 2, 300, 64, F16, False, (1, 4, 300, 300), "additive"),
    (1, 6, 2, 90, 64, BF16, True, (1, 6, 90, 90), "additive"),
    (2, 14, 2, 500, 64, F16, True, None, "padding"),
]


@pytest.mark.parametrize("B,Hq,Hkv,N,D,dtype,causal,shape,kind", BWD_CASES)
def test_masked_backward_matches_oracle(cuda_lib, B, Hq, Hkv, N, D, dtype, causal, shape, kind):
    x = inputs.make_custom(B, Hq, Hkv, N, N, D, dtype, seed=7 * N + D, with_grad=True)
    mask = make_mask(shape or (B, 1, 1, N), kind, dtype, seed=N + 1, Nk=N)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    mc = mask.cuda()
    out, lse = _lib.attn_fwd(q, k, v, causal=causal, mask=mc)
    dq, dk, dv = _lib.attn_bwd(q, k, v, out, do, lse, causal=causal, mask=mc)
    assert _lib.sync_status() == _lib.ATTN_OK
    ref = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], causal=causal, mask=mask)
    for name, t, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        e = helpers.assert_close_elementwise(t.double().cpu().numpy(), r, helpers.TOL_BWD[dtype],
                                             dtype, f"masked bwd {kind} {shape}", name)
        print(f"{kind} {shape} {name}: max err {e:.2e}")


def test_sdpa_masked_autograd(cuda_lib):
    x = inputs.make_custom(1, 4, 4, 256, 256, 128, BF16, seed=16, with_grad=True)
    mask = make_mask((1, 1, 256, 256), "bool", BF16, seed=17, Nk=256, empty_rows=True)
    q, k, v = (x[n].cuda().requires_grad_(True) for n in "qkv")
    out = sdpa.scaled_dot_product_attention(q, k, v, attn_mask=mask.cuda())
    out.backward(x["do"].cuda())
    ref = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], mask=mask)
    for name, t, r in zip(("dq", "dk", "dv"), (q, k, v), ref):
        helpers.assert_close_elementwise(t.grad.double().cpu().numpy(), r, helpers.TOL_BWD[BF16],
                                         BF16, "sdpa masked bwd", name)


@pytest.mark.parametrize("B,Hq,Hkv,N,D,dtype,causal,lens", [
    (2, 14, 2, 1000, 64, F16, False, (1000, 300)),    # sequence 1: key tiles 3-7 all masked
    (2, 4, 4, 700, 128, BF16, True, (130, 700)),      # sequence 0: key tiles 2-5 all masked
])
def test_padding_mask_whole_key_tiles_masked(cuda_lib, B, Hq, Hkv, N, D, dtype, causal, lens):
    """A key-padding mask ([B,1,1,N]) whose sequences end in whole masked key
    tiles: the forward stops at each sequence's last kept key, the dQ kernel
    does the same, and dK/dV CTAs of masked key tiles visit no query.  Forward
    and backward against the oracle."""
    x = inputs.make_custom(B, Hq, Hkv, N, N, D, dtype, seed=N + D, with_grad=True)
    mask = (torch.arange(N)[None, :] < torch.tensor(lens)[:, None]).reshape(B, 1, 1, N)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    mc = mask.cuda()
    out, lse = _lib.attn_fwd(q, k, v, causal=causal, mask=mc)
    assert _lib.sync_status() == _lib.ATTN_OK
    check(x, out, lse, causal, mask, f"padding {lens}")
    dq, dk, dv = _lib.attn_bwd(q, k, v, out, do, lse, causal=causal, mask=mc)
    assert _lib.sync_status() == _lib.ATTN_OK
    ref = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], causal=causal, mask=mask)
    for name, t, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        helpers.assert_close_elementwise(t.double().cpu().numpy(), r, helpers.TOL_BWD[dtype],
                                         dtype, f"padding {lens} bwd", name)
