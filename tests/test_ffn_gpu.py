"""The token-chunked FFN on the GPU (include/ffn.h), through the C ABI,
against the fp64 FFN oracle on the same seeded, rounded inputs.

Tolerance, derived from the arithmetic: the kernel accumulates in fp32 and
rounds h to the 16-bit dtype like the oracle, but its gelu / silu use the
hardware tanh / exp2 approximations (relative error about 2^-10 at most), so
an element of h may land one or two units in the last place away from the
oracle's rounded h.  Per output element the bound is therefore
    sum_f |W2[n,f]| (2 ulp(h_f) + 2^-10 |h_f|) + ulp(y_n) + 2^-20 sum_f |W2[n,f] h_f|.
Chunking must change no bit at all (every output row is one fixed-order
reduction of its own input row)."""
import numpy as np
import pytest
import torch

from oracle import ffn as ffn_oracle
from tests import helpers
from tiled_memory_efficient_gb300 import _lib

pytestmark = pytest.mark.gpu

F16, BF16 = torch.float16, torch.bfloat16


def make(T, d, f, act, dtype, seed, bias=True):
    g = torch.Generator().manual_seed(seed)
    n1 = 2 * f if act == "swiglu" else f
    x = torch.randn(T, d, generator=g).to(dtype)
    w1 = (torch.randn(n1, d, generator=g) / d ** 0.5).to(dtype)
    w2 = (torch.randn(d, f, generator=g) / f ** 0.5).to(dtype)
    b1 = (torch.randn(n1, generator=g) * 0.1).to(dtype) if bias else None
    b2 = (torch.randn(d, generator=g) * 0.1).to(dtype) if bias else None
    return x, w1, b1, w2, b2


def check(y_gpu, x, w1, b1, w2, b2, act, dtype, rows=None, what=""):
    xs = x if rows is None else x[rows]
    y_ref, h = ffn_oracle.ffn_fwd(xs, w1, b1, w2, b2, act, h_dtype=dtype)
    w2a = np.abs(w2.double().numpy())
    bound = (w2a @ (2 * helpers.ulp(h, dtype) + 2.0 ** -10 * np.abs(h)).T).T
    bound += helpers.ulp(y_ref, dtype) + 2.0 ** -20 * (np.abs(h) @ w2a.T)
    got = y_gpu.double().cpu().numpy() if rows is None else y_gpu[rows].double().cpu().numpy()
    err = np.abs(got - y_ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), (f"{what}: |y - oracle| = {err[worst]:.3e} > bound "
                                  f"{bound[worst]:.3e} at {worst}")
    return float(err.max())


CASES = [
    # T, d_model, d_ff, act, dtype, chunk
    (300, 64, 200, "gelu_tanh", BF16, 128),    # ragged rows and columns, several chunks
    (257, 128, 264, "swiglu", BF16, 100),      # chunk not a multiple of 128
    (130, 96, 136, "silu", F16, 1000),         # one chunk
    (64, 64, 128, "relu", F16, 64),
    (200, 136, 72, "none", BF16, 50),
    (1, 8, 8, "gelu_tanh", BF16, 1),           # one token, the narrowest rows (16 bytes)
    (3, 16, 24, "swiglu", F16, 2),             # tiles far larger than the problem
    (129, 64, 8, "silu", BF16, 128),           # a one-row second chunk
    (150, 256, 512, "relu", F16, 64),          # 256-column tiles in both products
    (100, 480, 160, "gelu_tanh", F16, 64),     # 160-column tiles: three across d_model
]


@pytest.mark.parametrize("T,d,f,act,dtype,chunk", CASES)
def test_ffn_matches_oracle(cuda_lib, T, d, f, act, dtype, chunk):
    x, w1, b1, w2, b2 = make(T, d, f, act, dtype, seed=T + f)
    dev = [t.cuda() if t is not None else None for t in (x, w1, b1, w2, b2)]
    y = _lib.ffn_forward(*dev, act=act, chunk=chunk)
    assert _lib.sync_status() == _lib.ATTN_OK
    e = check(y, x, w1, b1, w2, b2, act, dtype, what=f"ffn {act} {T}x{d}x{f}")
    print(f"{act} {dtype}: max err {e:.2e}")


@pytest.mark.parametrize("act", ["swiglu", "gelu_tanh"])
def test_chunking_is_bit_exact(cuda_lib, act):
    x, w1, b1, w2, b2 = make(1000, 128, 384, act, BF16, seed=3)
    dev = [t.cuda() for t in (x, w1, b1, w2, b2)]
    y, ok = _lib.ffn_check_chunking(*dev, act=act, chunk=192)
    assert ok
    y_full = _lib.ffn_forward(*dev, act=act, chunk=1000)
    y_small = _lib.ffn_forward(*dev, act=act, chunk=77)
    torch.cuda.synchronize()
    assert torch.equal(y, y_full) and torch.equal(y_small, y_full)


def test_qwen_sized_swiglu_sampled(cuda_lib):
    """The MLP shape of the Qwen 2.5 0.5B model of the forum post's LLM table
    (d_model 896, d_ff 4864, SwiGLU, no biases), 4096 tokens in chunks of
    1024; 64 rows checked against the oracle."""
    x, w1, b1, w2, b2 = make(4096, 896, 4864, "swiglu", BF16, seed=4, bias=False)
    dev = [t.cuda() if t is not None else None for t in (x, w1, b1, w2, b2)]
    y = _lib.ffn_forward(*dev, act="swiglu", chunk=1024)
    assert _lib.sync_status() == _lib.ATTN_OK
    rows = np.sort(np.random.default_rng(5).choice(4096, 64, replace=False))
    rows[0], rows[-1] = 0, 4095
    e = check(y, x, w1, b1, w2, b2, "swiglu", BF16, rows=rows, what="qwen mlp")
    print(f"qwen-sized swiglu: max err {e:.2e}")


def test_ffn_benchmark_config_sampled(cuda_lib):
    """The FFN exactly as the benchmark times it (16384 tokens in chunks of
    4096, d_model 896, d_ff 4864, swiglu, bf16, no biases, the benchmark's
    seed and scaling): 64 sampled rows, including both ends of every chunk."""
    g = torch.Generator().manual_seed(9000)
    T, d, f = 16384, 896, 4864
    x = torch.randn(T, d, generator=g).to(BF16)
    w1 = (torch.randn(2 * f, d, generator=g) / d ** 0.5).to(BF16)
    w2 = (torch.randn(d, f, generator=g) / f ** 0.5).to(BF16)
    y = _lib.ffn_forward(x.cuda(), w1.cuda(), None, w2.cuda(), None, act="swiglu", chunk=4096)
    assert _lib.sync_status() == _lib.ATTN_OK
    edges = [c + e for c in range(0, T, 4096) for e in (0, 4095)]
    rows = np.unique(np.concatenate([edges, np.random.default_rng(6).choice(T, 56, replace=False)]))
    e = check(y, x, w1, None, w2, None, "swiglu", BF16, rows=rows, what="ffn bench config")
    print(f"ffn benchmark config: max err {e:.2e}")
