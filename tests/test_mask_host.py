"""Host-side handling of attention masks, no GPU: the binding's conversion of
an SDPA attn_mask into the C ABI's (pointer, kind, strides), and the C ABI's
rejection of masks it cannot read, before any device work."""
import pytest
import torch

from tiled_memory_efficient_gb300 import _lib


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build_library()
    return _lib.load()


def q_of(B, Hq, Nq, D=64, dtype=torch.float16):
    return torch.zeros(B, Hq, Nq, D, dtype=dtype)


def test_bool_padding_mask_is_used_in_place():
    q = q_of(2, 4, 10)
    mask = torch.ones(2, 1, 1, 64, dtype=torch.bool)
    m, kind, st = _lib.prepare_mask(mask, q, 64)
    assert kind == _lib.ATTN_MASK_BOOL
    assert m.data_ptr() == mask.data_ptr()
    assert st == [64, 0, 0]          # batch stride; broadcast head and query


def test_unaligned_rows_are_copied_into_padded_rows():
    q = q_of(2, 3, 5)
    mask = torch.rand(2, 3, 5, 300) > 0.5
    m, kind, st = _lib.prepare_mask(mask, q, 300)
    assert m.shape[-1] == 304 and m.data_ptr() != mask.data_ptr()
    assert torch.equal(m[..., :300], mask)
    assert st == [3 * 5 * 304, 5 * 304, 304]
    assert all((s * m.element_size()) % 16 == 0 for s in st)


def test_float_mask_becomes_an_additive_bias_in_q_dtype():
    q = q_of(1, 2, 8, dtype=torch.bfloat16)
    mask = torch.randn(8, 32)
    m, kind, st = _lib.prepare_mask(mask, q, 32)
    assert kind == _lib.ATTN_MASK_ADDITIVE
    assert m.dtype == torch.bfloat16 and m.shape == (1, 1, 8, 32)
    assert st == [0, 0, 32]
    assert torch.equal(m[0, 0], mask.to(torch.bfloat16))


def test_key_only_mask_has_zero_strides():
    q = q_of(1, 2, 8)
    m, kind, st = _lib.prepare_mask(torch.ones(48, dtype=torch.bool), q, 48)
    assert st == [0, 0, 0] and m.shape == (1, 1, 1, 48)


@pytest.mark.parametrize("mask,exc", [
    (torch.ones(2, 1, 1, 63, dtype=torch.bool), ValueError),    # wrong key count
    (torch.ones(3, 1, 1, 64, dtype=torch.bool), ValueError),    # batch does not broadcast
    (torch.ones(1, 1, 1, 64, dtype=torch.int32), TypeError),    # neither bool nor float
    ([[True] * 64], ValueError),                                # not a tensor
])
def test_bad_masks_are_rejected(mask, exc):
    with pytest.raises(exc):
        _lib.prepare_mask(mask, q_of(2, 4, 10), 64)


P = 256  # a fake, 16-byte-aligned "device" address: validation fails before any use


@pytest.mark.parametrize("mask,kind,sb,sh,sq,code", [
    (0, 1, 0, 0, 0, _lib.ATTN_ERR_INVALID),           # no mask
    (P, 0, 0, 0, 0, _lib.ATTN_ERR_INVALID),           # unknown kind
    (P, 3, 0, 0, 0, _lib.ATTN_ERR_INVALID),
    (P, 1, -16, 0, 0, _lib.ATTN_ERR_INVALID),         # negative stride
    (P + 8, 1, 0, 0, 0, _lib.ATTN_ERR_ALIGN),         # mask not 16-byte aligned
    (P, 1, 0, 0, 300, _lib.ATTN_ERR_ALIGN),           # bool rows of 300 bytes
    (P, 2, 0, 12, 0, _lib.ATTN_ERR_ALIGN),            # additive: 12 elements = 24 bytes
])
def test_masked_forward_rejects_unreadable_masks(lib, mask, kind, sb, sh, sq, code):
    rc = lib.attn_fwd_masked(P, P, P, P, P, mask, kind, sb, sh, sq, 1, 2, 2, 128, 128, 64,
                             0.125, 0, 0, None)
    assert rc == code


def test_readable_mask_still_gets_the_shape_checks(lib):
    # 8 16-bit elements per head are 16 bytes: the mask passes, the batch size does not
    rc = lib.attn_fwd_masked(P, P, P, P, P, P, 2, 0, 8, 0, 0, 2, 2, 128, 128, 64, 0.125, 0, 0,
                             None)
    assert rc == _lib.ATTN_ERR_INVALID
