"""The drop-in SDPA surface: argument handling on the CPU, and on the GPU the
autograd function's forward and gradients against the fp64 oracle, plus the
opt-in patch of torch.nn.functional.scaled_dot_product_attention."""
import pytest
import torch
import torch.nn.functional as F

import oracle
from tests import helpers
from tiled_memory_efficient_gb300 import inputs, sdpa


def test_unsupported_arguments_raise_without_a_gpu():
    q = torch.zeros(1, 2, 8, 64, dtype=torch.float16)
    with pytest.raises(NotImplementedError):
        sdpa.scaled_dot_product_attention(q, q, q, attn_mask=torch.zeros(8, 8))
    with pytest.raises(NotImplementedError):
        sdpa.scaled_dot_product_attention(q, q, q, dropout_p=0.1)
    with pytest.raises(NotImplementedError):   # CPU tensors: no CPU fallback
        sdpa.scaled_dot_product_attention(q, q, q)
    k = torch.zeros(1, 1, 8, 64, dtype=torch.float16)
    with pytest.raises(ValueError):            # GQA must be asked for, as in torch
        sdpa.scaled_dot_product_attention(q, k, k)


def test_patch_is_opt_in_and_reversible():
    original = F.scaled_dot_product_attention
    assert not sdpa.is_patched()
    sdpa.patch()
    try:
        assert F.scaled_dot_product_attention is sdpa.scaled_dot_product_attention
        sdpa.patch()   # idempotent
        assert sdpa.is_patched()
    finally:
        sdpa.unpatch()
    assert F.scaled_dot_product_attention is original
    assert not sdpa.is_patched()


@pytest.mark.gpu
@pytest.mark.parametrize("Hq,Hkv,causal,dtype", [(4, 4, True, torch.bfloat16),
                                                 (6, 2, False, torch.float16)])
def test_autograd_function_matches_oracle(cuda_lib, Hq, Hkv, causal, dtype):
    x = inputs.make_custom(1, Hq, Hkv, 333, 333, 64, dtype, seed=41, with_grad=True)
    q, k, v = (x[n].cuda().requires_grad_(True) for n in ("q", "k", "v"))
    out = sdpa.attention(q, k, v, is_causal=causal)
    out.backward(x["do"].cuda())
    o_ref, _ = oracle.attention_fwd(x["q"], x["k"], x["v"], causal=causal)
    helpers.assert_close_elementwise(out.detach().double().cpu().numpy(), o_ref,
                                     helpers.TOL_O[dtype], dtype, "sdpa fwd", "O")
    ref = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], causal=causal)
    for name, t, r in zip(("dq", "dk", "dv"), (q, k, v), ref):
        helpers.assert_close_elementwise(t.grad.double().cpu().numpy(), r,
                                         helpers.TOL_BWD[dtype], dtype, "sdpa bwd", name)


@pytest.mark.gpu
def test_patched_torch_sdpa_runs_on_the_tiled_kernels(cuda_lib):
    x = inputs.make_custom(2, 4, 2, 256, 256, 128, torch.bfloat16, seed=42)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    sdpa.patch()
    try:
        out = F.scaled_dot_product_attention(q, k, v, is_causal=True, enable_gqa=True)
    finally:
        sdpa.unpatch()
    o_ref, _ = oracle.attention_fwd(x["q"], x["k"], x["v"], causal=True)
    helpers.assert_close_elementwise(out.double().cpu().numpy(), o_ref, 1e-2, torch.bfloat16,
                                     "patched sdpa", "O")


@pytest.mark.gpu
def test_decode_shape_takes_the_split_path_and_trains(cuda_lib):
    """One query per head against 5000 keys: the forward runs split (the
    library picks several key ranges for this grid) and the backward uses its
    LSE; both against the oracle."""
    from tiled_memory_efficient_gb300 import _lib
    assert _lib.num_splits(2, 14, 2, 1, 5000, 64) > 1
    x = inputs.make_custom(2, 14, 2, 1, 5000, 64, torch.float16, seed=43, with_grad=True)
    q, k, v = (x[n].cuda().requires_grad_(True) for n in ("q", "k", "v"))
    out = sdpa.scaled_dot_product_attention(q, k, v, enable_gqa=True)
    out.backward(x["do"].cuda())
    o_ref, _ = oracle.attention_fwd(x["q"], x["k"], x["v"])
    helpers.assert_close_elementwise(out.detach().double().cpu().numpy(), o_ref,
                                     helpers.TOL_O[torch.float16], torch.float16, "decode", "O")
    ref = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"])
    for name, t, r in zip(("dq", "dk", "dv"), (q, k, v), ref):
        helpers.assert_close_elementwise(t.grad.double().cpu().numpy(), r,
                                         helpers.TOL_BWD[torch.float16], torch.float16,
                                         "decode bwd", name)
