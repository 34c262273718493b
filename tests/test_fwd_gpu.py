"""Forward parity on the GPU: the CUDA path (through the C ABI) against the
fp64 oracle on the same seeded, rounded inputs.

Small shapes are checked on every row; the full-size workloads on a seeded
sample of rows (always rows 0, N-1 and the 128-row tile edges of each head),
since a full fp64 check would cost tens of TFLOP on the CPU.
"""
import numpy as np
import pytest
import torch

from tests import helpers
from tiled_memory_efficient_gb300 import _lib, inputs

pytestmark = pytest.mark.gpu

F16, BF16 = torch.float16, torch.bfloat16


def run_fwd(x, causal, scale=None):
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    out, lse = _lib.attn_fwd(q, k, v, causal=causal, scale=scale)
    assert _lib.sync_status() == _lib.ATTN_OK
    return out, lse


def check_full(x, causal, scale=None, what=""):
    out, lse = run_fwd(x, causal, scale)
    o_ref, lse_ref = helpers.oracle_rows(x["q"], x["k"], x["v"],
                                         np.arange(x["q"].shape[0] * x["q"].shape[1] *
                                                   x["q"].shape[2]), causal, scale)
    o_gpu, lse_gpu = out.reshape(-1, out.shape[-1]).double().cpu().numpy(), \
        lse.reshape(-1).double().cpu().numpy()
    return helpers.assert_fwd_close(o_gpu, lse_gpu, o_ref, lse_ref, x["q"].dtype, what)


def test_tiny_workload_every_row(cuda_lib):
    w = inputs.WORKLOADS["tiny"]
    x = inputs.make_inputs(w, 256)
    eo, el = check_full(x, w.causal, what="tiny")
    print(f"tiny: max|dO|={eo:.2e} max|dLSE|={el:.2e}")


SMALL = [
    # B, Hq, Hkv, Nq, Nk, D, dtype, causal
    (1, 2, 2, 128, 128, 64, F16, False),
    (1, 2, 2, 300, 300, 64, F16, True),       # ragged tail, causal
    (2, 3, 3, 1, 1, 64, F16, False),          # single query and key
    (1, 3, 3, 1, 517, 128, BF16, False),      # one query row, many keys
    (1, 4, 4, 200, 333, 128, BF16, False),    # Nq != Nk, both ragged
    (1, 14, 2, 250, 250, 64, F16, True),      # GQA G=7, tiles cross head boundaries
    (1, 7, 1, 37, 37, 128, BF16, True),       # tiny heads flattened into one tile
    (2, 4, 2, 1024, 1024, 128, BF16, True),   # several key tiles, causal skipping
    (1, 2, 2, 129, 1000, 64, F16, True),      # Nq < Nk, top-left causal
    (1, 2, 2, 1000, 129, 64, F16, True),      # Nq > Nk: late rows see every key
    (1, 4, 1, 512, 2048, 128, F16, False),    # GQA G=4, D=128 fp16
    (1, 2, 2, 640, 640, 64, BF16, False),
]


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,D,dtype,causal", SMALL)
def test_small_shapes_every_row(cuda_lib, B, Hq, Hkv, Nq, Nk, D, dtype, causal):
    x = inputs.make_custom(B, Hq, Hkv, Nq, Nk, D, dtype, seed=Nq * 7 + Nk + D)
    check_full(x, causal, what=f"{(B, Hq, Hkv, Nq, Nk, D, dtype, causal)}")


@pytest.mark.parametrize("v_std", [0.5, 1.0])
@pytest.mark.parametrize("dtype", [F16, BF16])
def test_large_scores_stress_ftz_and_rescale(cuda_lib, dtype, v_std):
    # q, k with std 4: scaled scores of std ~16, so rows are nearly one-hot,
    # the running max moves often and many terms fall under the flush
    # threshold.  With v of std 1 many outputs are a single value row of
    # magnitude 2 to 4, where half an ulp of the stored output takes most of
    # the bound (bf16: 0.0078 of 0.01); v of std 0.5 keeps |O| below 2.
    x = inputs.make_custom(1, 2, 2, 384, 700, 64, dtype, seed=5, std=4.0, v_std=v_std)
    check_full(x, False, what=f"std4 v_std={v_std}")
    check_full(x, True, what=f"std4 v_std={v_std} causal")


@pytest.mark.parametrize("dtype", [F16, BF16])
def test_large_scores_stress_d128(cuda_lib, dtype):
    # the same regime at D = 128 (one thread per 128-key row), with a ragged tail
    x = inputs.make_custom(1, 3, 3, 300, 520, 128, dtype, seed=6, std=4.0, v_std=1.0)
    check_full(x, False, what="std4 D=128")
    check_full(x, True, what="std4 D=128 causal")


def test_explicit_scale(cuda_lib):
    x = inputs.make_custom(1, 2, 2, 256, 256, 128, F16, seed=9)
    check_full(x, False, scale=0.3, what="scale=0.3")


SAMPLED = [("sweep", n) for n in inputs.WORKLOADS["sweep"].seq_lens] + \
          [("gqa_prefill", n) for n in inputs.WORKLOADS["gqa_prefill"].seq_lens] + \
          [("video_dit", n) for n in inputs.WORKLOADS["video_dit"].seq_lens] + \
          [("training", 8192)]


FULL = [("sweep", n) for n in inputs.WORKLOADS["sweep"].seq_lens] + \
       [("gqa_prefill", n) for n in inputs.WORKLOADS["gqa_prefill"].seq_lens] + \
       [("video_dit", 17600), ("training", 8192)]


@pytest.mark.parametrize("name,n", FULL)
def test_workloads_every_row(cuda_lib, name, n):
    """The benchmark workloads exactly as the benchmark runs them (all but
    video-DiT at N = 75600, which is row-sampled below): every output row of
    every head against the oracle."""
    w = inputs.WORKLOADS[name]
    x = inputs.make_inputs(w, n)
    eo, el = check_full(x, w.causal, what=f"{name} N={n} every row")
    print(f"{name} N={n} every row: max|dO|={eo:.2e} max|dLSE|={el:.2e}")


@pytest.mark.parametrize("name,n", SAMPLED)
def test_workloads_sampled_rows(cuda_lib, name, n):
    w = inputs.WORKLOADS[name]
    x = inputs.make_inputs(w, n)
    out, lse = run_fwd(x, w.causal)
    rows = inputs.sample_rows(w.B, w.Hq, n, per_head=6, seed=n)
    o_gpu, lse_gpu = helpers.gpu_rows(out, lse, rows)
    o_ref, lse_ref = helpers.oracle_rows(x["q"], x["k"], x["v"], rows, w.causal)
    eo, el = helpers.assert_fwd_close(o_gpu, lse_gpu, o_ref, lse_ref, w.dtype, f"{name} N={n}")
    print(f"{name} N={n}: rows={len(rows)} max|dO|={eo:.2e} max|dLSE|={el:.2e}")


# The causal forward at short sequences runs the heaviest pair positions as
# two one-tile CTAs per pair (attn_fwd_half_positions): the split changes which
# CTA computes a row, not its arithmetic.  A key-only all-true mask (which
# takes the same split-softmax layout without the split) must agree bit for
# bit, and every row matches the oracle.

HALF_SHAPES = [
    # B, Hq, Hkv, Nq, Nk, causal
    (1, 14, 2, 2048, 2048, True),            # the GQA prefill at N = 2048: 3 positions split
    (1, 2, 2, 512, 512, True),               # one position split
    (1, 2, 2, 512, 1000, "bottom_right"),    # Nk > Nq: every row sees 488 more keys
    (2, 4, 2, 768, 768, True),               # B = 2, GQA 2:1, three pairs per head
]


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,causal", HALF_SHAPES)
def test_half_pairs_every_row_and_bitwise(cuda_lib, B, Hq, Hkv, Nq, Nk, causal):
    h = _lib.fwd_half_positions(B, Hq, Hkv, Nq, Nk, 64, causal, F16)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms == 152:
        assert h > 0
    x = inputs.make_custom(B, Hq, Hkv, Nq, Nk, 64, F16, seed=Nq + Nk + Hq)
    check_full(x, causal, what=f"half pairs {(B, Hq, Hkv, Nq, Nk, causal)}")
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    a = _lib.attn_fwd(q, k, v, causal=causal)
    b = _lib.attn_fwd(q, k, v, causal=causal,
                      mask=torch.ones((B, 1, 1, Nk), dtype=torch.bool, device="cuda"))
    c = _lib.attn_fwd_ws(q, k, v, causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert torch.equal(a[0], c[0]) and torch.equal(a[1], c[1])


def test_output_canaries_untouched(cuda_lib):
    B, Hq, Hkv, N, D = 1, 3, 3, 200, 64
    x = inputs.make_custom(B, Hq, Hkv, N, N, D, F16, seed=11)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    pad = 4096
    o_buf = torch.full((B * Hq * N * D + 2 * pad,), 7.0, device="cuda", dtype=F16)
    l_buf = torch.full((B * Hq * N + 2 * pad,), 7.0, device="cuda", dtype=torch.float32)
    out = o_buf[pad:pad + B * Hq * N * D].view(B, Hq, N, D)
    lse = l_buf[pad:pad + B * Hq * N].view(B, Hq, N)
    _lib.attn_fwd(q, k, v, causal=True, out=out, lse=lse)
    assert _lib.sync_status() == _lib.ATTN_OK
    assert torch.all(o_buf[:pad] == 7.0) and torch.all(o_buf[-pad:] == 7.0)
    assert torch.all(l_buf[:pad] == 7.0) and torch.all(l_buf[-pad:] == 7.0)
    assert torch.all(torch.isfinite(out))


def test_runs_on_side_stream(cuda_lib):
    x = inputs.make_custom(1, 2, 2, 256, 256, 64, F16, seed=12)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    ref_out, ref_lse = _lib.attn_fwd(q, k, v)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out, lse = _lib.attn_fwd(q, k, v)
    s.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


def test_calls_from_a_fresh_host_thread(cuda_lib):
    # A new host thread has no current CUDA context until something makes one
    # current; the library must still encode its tensor maps and launch.
    import threading
    x = inputs.make_custom(1, 2, 2, 200, 200, 64, F16, seed=15, with_grad=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    ref_out, ref_lse = _lib.attn_fwd(q, k, v, causal=True)
    ref_g = _lib.attn_bwd(q, k, v, ref_out, do, ref_lse, causal=True)
    torch.cuda.synchronize()
    res = {}

    def worker():
        try:
            out, lse = _lib.attn_fwd(q, k, v, causal=True)
            g = _lib.attn_bwd(q, k, v, out, do, lse, causal=True)
            torch.cuda.synchronize()
            res["v"] = (out, lse) + tuple(g)
        except Exception as e:  # reported below
            res["e"] = e

    t = threading.Thread(target=worker)
    t.start()
    t.join()
    assert "e" not in res, res.get("e")
    for a, b in zip(res["v"], (ref_out, ref_lse) + tuple(ref_g)):
        assert torch.equal(a, b)


def test_deterministic(cuda_lib):
    x = inputs.make_custom(1, 4, 2, 700, 700, 128, BF16, seed=13)
    o1, l1 = run_fwd(x, True)
    o2, l2 = run_fwd(x, True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_bounded_wait_reports_timeout(cuda_lib):
    lib = cuda_lib
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.attn_sync_status(stream) == _lib.ATTN_OK
    assert lib.attn_selftest_timeout(1_000_000, stream) == _lib.ATTN_OK   # 1 ms
    assert lib.attn_sync_status(stream) == _lib.ATTN_ERR_TIMEOUT
    assert lib.attn_sync_status(stream) == _lib.ATTN_OK                  # cleared
    # the context is still usable afterwards
    x = inputs.make_custom(1, 2, 2, 128, 128, 64, F16, seed=14)
    check_full(x, False, what="after timeout")


# ---------------------------------------------------------------- attn_fwd_ws
# bf16 inputs: the value tiles are converted to fp16 once into a workspace
# instead of inside every CTA; fp16 inputs take attn_fwd itself.

WS_SHAPES = [
    # B, Hq, Hkv, Nq, Nk, D, causal
    (1, 2, 2, 300, 300, 128, False),
    (1, 2, 2, 300, 300, 128, True),
    (1, 4, 4, 200, 333, 128, False),     # Nq != Nk, both ragged
    (1, 14, 2, 250, 250, 64, True),      # GQA G=7, D=64
    (2, 4, 2, 1024, 1024, 128, True),    # several key tiles, causal skipping
    (1, 3, 3, 1, 517, 64, False),        # one query row
]


def run_fwd_ws(x, causal, scale=None):
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    out, lse = _lib.attn_fwd_ws(q, k, v, causal=causal, scale=scale)
    assert _lib.sync_status() == _lib.ATTN_OK
    return out, lse


def check_ws(x, causal, what):
    out, lse = run_fwd_ws(x, causal)
    o_ref, lse_ref = helpers.oracle_rows(x["q"], x["k"], x["v"],
                                         np.arange(x["q"].shape[0] * x["q"].shape[1] *
                                                   x["q"].shape[2]), causal)
    return helpers.assert_fwd_close(out.reshape(-1, out.shape[-1]).double().cpu().numpy(),
                                    lse.reshape(-1).double().cpu().numpy(), o_ref, lse_ref,
                                    x["q"].dtype, what)


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,D,causal", WS_SHAPES)
def test_ws_small_shapes_every_row(cuda_lib, B, Hq, Hkv, Nq, Nk, D, causal):
    x = inputs.make_custom(B, Hq, Hkv, Nq, Nk, D, BF16, seed=Nq * 5 + Nk + D)
    check_ws(x, causal, f"ws {(B, Hq, Hkv, Nq, Nk, D, causal)}")


def test_ws_stress_one_hot_rows(cuda_lib):
    x = inputs.make_custom(1, 3, 3, 300, 520, 128, BF16, seed=6, std=4.0, v_std=1.0)
    check_ws(x, False, "ws std4 D=128")
    check_ws(x, True, "ws std4 D=128 causal")


@pytest.mark.parametrize("name,n", [("video_dit", 17600), ("training", 8192)])
def test_ws_matches_attn_fwd_bitwise(cuda_lib, name, n):
    """Every value tile of these workloads converts, so both paths run the
    same fp16 PV products: the outputs agree bit for bit (attn_fwd itself is
    checked against the oracle on every row of both workloads)."""
    w = inputs.WORKLOADS[name]
    x = inputs.make_inputs(w, n)
    a = run_fwd(x, w.causal)
    b = run_fwd_ws(x, w.causal)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("path", ["attn_fwd", "attn_fwd_ws"])
def test_value_tile_below_fp16_precision_stays_bf16(cuda_lib, path):
    """A value tile whose largest magnitude is below 2^-8 stays bf16 (its
    small values would lose bits as fp16 subnormals); the other tiles still
    convert.  Both paths against the oracle at the usual bound."""
    x = inputs.make_custom(1, 2, 2, 384, 700, 128, BF16, seed=41)
    v = x["v"].clone()
    v[0, 1, 256:384] *= 1.0e-4           # key tile 2 of head 1
    x["v"] = v.to(BF16)
    if path == "attn_fwd":
        check_full(x, False, what="tiny value tile attn_fwd")
    else:
        check_ws(x, False, "tiny value tile attn_fwd_ws")


@pytest.mark.parametrize("path", ["attn_fwd", "attn_fwd_ws"])
def test_value_tile_beyond_fp16_range_stays_bf16(cuda_lib, path):
    """A value of magnitude 2^16 or more (here 1e5) does not fit fp16: its
    tile (attn_fwd) or the CTAs that read it (attn_fwd_ws) keep bf16 values
    and pack P as bf16.  bf16 P is rounded to 2^-8 relative, which moves O by
    up to 2^-8 of the weighted mean of |v| -- about half an ulp of the large
    outputs this value makes -- so the bound here adds 2^-7 * sum_j p_j |v_j|
    (exact softmax weights p) to the usual one."""
    x = inputs.make_custom(1, 2, 2, 384, 700, 128, BF16, seed=41)
    v = x["v"].clone()
    v[0, 0, 200, 5] = 1.0e5              # key tile 1 of head 0
    x["v"] = v.to(BF16)
    out, lse = run_fwd(x, False) if path == "attn_fwd" else run_fwd_ws(x, False)
    q, k, vv = (x[n][0].double().numpy() for n in ("q", "k", "v"))
    o_ref, lse_ref = helpers.oracle_rows(x["q"], x["k"], x["v"], np.arange(2 * 384), False)
    slack = np.concatenate([
        (lambda s: (np.exp(s - s.max(1, keepdims=True)) /
                    np.exp(s - s.max(1, keepdims=True)).sum(1, keepdims=True)) @ np.abs(vv[h]))(
            q[h] @ k[h].T / np.sqrt(128))
        for h in range(2)])
    got = out.reshape(-1, 128).double().cpu().numpy()
    err = np.abs(got - o_ref)
    bound = helpers.bound_for(o_ref, helpers.TOL_O[BF16], BF16) + 2.0 ** -7 * slack
    assert np.all(np.isfinite(got)) and np.all(err <= bound), float((err - bound).max())
    assert helpers.max_err(lse.reshape(-1).double().cpu().numpy(), lse_ref) <= helpers.TOL_LSE


def test_ws_fp16_is_attn_fwd(cuda_lib):
    """fp16 with a grid that is not cut: attn_fwd itself, no workspace."""
    x = inputs.make_custom(1, 2, 2, 300, 300, 64, F16, seed=43)
    assert _lib.fwd_workspace_size(1, 2, 2, 300, 300, 64, F16) == 0
    a = run_fwd(x, True)
    b = run_fwd_ws(x, True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


# attn_fwd_ws also evens out the grid (one CTA per SM per unit of a KV group
# and 256 query rows): the last wave's units are cut into 2 to 4 key ranges
# when a model of the last wave's time says it pays (no causal mask, >= 8 key
# tiles), and a grid under
# one wave has every unit's keys cut into ranges of >= 16 key tiles; the cut
# units' partials are merged by a second kernel.  The shapes below are cut on
# a 152-SM GB300.

CUT_SHAPES = [
    # B, Hq, Hkv, Nq, Nk, D, dtype, causal
    (1, 4, 4, 10240, 1000, 64, F16, False),    # 160 units: 152 whole, 8 in halves; ragged keys
    (1, 8, 2, 5120, 1100, 64, F16, False),     # GQA 4:1, 9 key tiles: halves of 5 and 4
    (1, 4, 4, 10240, 2048, 64, F16, False),    # 16 key tiles: the 8 tail units in quarters
    (1, 4, 4, 10100, 1000, 64, F16, False),    # heads of 10100 rows: the cut rows end mid-pair
    (1, 4, 4, 10240, 1000, 128, BF16, False),  # bf16 with the fp16 copy of V
    (1, 2, 2, 1000, 8000, 64, F16, False),     # 8 units: 3 ranges of 21 key tiles (the last 21)
    (1, 2, 2, 1000, 8000, 64, F16, "bottom_right"),  # causal: a range may hold no visible key
    (2, 6, 2, 300, 4200, 128, BF16, "bottom_right"),  # GQA 3:1, 2 ranges of 17 and 16
]


def cut_plan(B, Hq, Hkv, Nq, Nk, D, causal, sms):
    """(first output row of the cut units, ranges) as the library plans it:
    a tail of several waves cut into S = 2..4 ranges when the model of the
    last wave's time (rounds of 1/S of a unit, ~15 us per extra round, ~4 us
    for the merge, ~1.1 / 2.2 us per key tile at D = 64 / 128) says it pays."""
    rows = Hq // Hkv * Nq
    n_pairs = -(-rows // 256)
    units = B * Hkv * n_pairs
    tiles = -(-Nk // 128)
    if units >= sms:
        waves = -(-units // sms)
        tail = units - (waves - 1) * sms
        if causal or tiles < 8 or waves < 2:
            return None, 1
        unit_us = tiles * (2.2 if D == 128 else 1.1)
        best, best_s = 1.0, 1
        for S in (2, 3, 4):
            if tiles < 4 * S:
                break
            rounds = -(-tail * S // sms)
            cost = rounds / S + (rounds - 1) * 15.0 / unit_us + 4.0 / unit_us
            if cost < best - 0.02:
                best, best_s = cost, S
        if best_s < 2:
            return None, 1
        whole = units - tail
        tps = -(-tiles // best_s)
        return (whole // n_pairs) * rows + (whole % n_pairs) * 256, -(-tiles // tps)
    want = min(sms // units, tiles // 16, 256)
    if want < 2:
        return None, 1
    tps = -(-tiles // want)
    return 0, -(-tiles // tps)


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,D,dtype,causal", CUT_SHAPES)
def test_ws_cut_grid_every_row(cuda_lib, B, Hq, Hkv, Nq, Nk, D, dtype, causal):
    """Every row against the oracle; the rows of whole units are attn_fwd's
    bit for bit (fp16: the same kernel arithmetic), the merged rows agree
    with the oracle at the usual bound."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    row0, splits = cut_plan(B, Hq, Hkv, Nq, Nk, D, bool(causal), sms)
    assert _lib.fwd_ws_splits(B, Hq, Hkv, Nq, Nk, D, causal) == splits
    if sms == 152:
        assert splits > 1
    ws = _lib.fwd_workspace_size(B, Hq, Hkv, Nq, Nk, D, dtype)
    assert (ws > 0) == (splits > 1 or dtype == BF16)
    x = inputs.make_custom(B, Hq, Hkv, Nq, Nk, D, dtype, seed=Nq + 3 * Nk + D)
    check_ws(x, causal, f"cut grid {(B, Hq, Hkv, Nq, Nk, D, causal)}")
    if dtype == F16 and row0 is not None:
        a_o, a_l = run_fwd(x, causal)
        b_o, b_l = run_fwd_ws(x, causal)
        a_o, b_o = a_o.reshape(-1, D), b_o.reshape(-1, D)
        a_l, b_l = a_l.reshape(-1), b_l.reshape(-1)
        assert torch.equal(a_o[:row0], b_o[:row0]) and torch.equal(a_l[:row0], b_l[:row0])


def test_ws_cut_workspace_is_checked(cuda_lib):
    """A cut fp16 grid needs its workspace: a smaller one is refused before
    anything runs."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms != 152:
        pytest.skip("the cut shape is planned for 152 SMs")
    ws = _lib.fwd_workspace_size(1, 4, 4, 10240, 1000, 64, F16)
    assert ws > 0
    x = inputs.make_custom(1, 4, 4, 10240, 1000, 64, F16, seed=5)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    small = torch.empty(ws - 256, device="cuda", dtype=torch.uint8)
    with pytest.raises(_lib.AttnError):
        _lib.attn_fwd_ws(q, k, v, workspace=small)


@pytest.mark.parametrize("D,dtype", [(64, F16), (128, BF16)])
def test_out_only_16_byte_aligned(cuda_lib, D, dtype):
    """The epilogue writes 32-byte sectors when out is 32-byte aligned and
    16-byte chunks when it is only 16-byte aligned: both give the same bits."""
    x = inputs.make_custom(1, 2, 2, 300, 300, D, dtype, seed=44)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    ref, ref_lse = _lib.attn_fwd(q, k, v, causal=True)
    n = q.numel()
    buf = torch.zeros(n + 64, device="cuda", dtype=dtype)
    assert buf.data_ptr() % 32 == 0
    out = buf[8:8 + n].view_as(q)          # 16 bytes past a 32-byte boundary
    assert out.data_ptr() % 32 == 16
    _, lse = _lib.attn_fwd(q, k, v, causal=True, out=out)
    assert _lib.sync_status() == _lib.ATTN_OK
    assert torch.equal(out, ref) and torch.equal(lse, ref_lse)
    assert torch.all(buf[:8] == 0) and torch.all(buf[8 + n:] == 0)
