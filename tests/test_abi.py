"""C-ABI checks that need no GPU: the library builds, loads, exports every
symbol include/attn.h declares, and rejects bad arguments before touching the
device."""
import ctypes
import os

import pytest

from tiled_memory_efficient_gb300 import _lib


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build_library()
    return _lib.load()


def test_header_declares_the_boundary():
    names = _lib.declared_functions()
    for required in ("attn_fwd", "attn_bwd", "attn_bwd_workspace_size", "attn_sync_status",
                     "attn_strerror", "attn_selftest_timeout", "attn_version", "attn_fwd_splitkv",
                     "attn_fwd_splitkv_workspace_size", "attn_fwd_num_splits", "attn_fwd_masked",
                     "attn_bwd_masked", "ffn_forward", "ffn_check_chunking",
                     "ffn_workspace_size", "attn_fwd_ws", "attn_fwd_workspace_size",
                     "attn_fwd_ws_splits", "attn_bwd_splits", "attn_fwd_half_positions"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in _lib.declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib._SIGNATURES, f"binding lacks a signature for {name}"


def test_strerror_and_version(lib):
    assert lib.attn_strerror(0) == b"ok"
    assert b"aligned" in lib.attn_strerror(3)
    assert lib.attn_strerror(99) == b"unknown status"
    assert lib.attn_version() >= 100


P = 256  # a fake, 16-byte-aligned "device" address: validation fails before any use


@pytest.mark.parametrize("args,code", [
    # null pointer
    ((0, P, P, P, P, 1, 2, 2, 128, 128, 64, 0.125, 0, 0), 1),
    # non-positive sizes
    ((P, P, P, P, P, 0, 2, 2, 128, 128, 64, 0.125, 0, 0), 1),
    ((P, P, P, P, P, 1, 2, 2, 128, 0, 64, 0.125, 0, 0), 1),
    # Hq not a multiple of Hkv
    ((P, P, P, P, P, 1, 3, 2, 128, 128, 64, 0.125, 0, 0), 1),
    # bad scale, bad dtype
    ((P, P, P, P, P, 1, 2, 2, 128, 128, 64, 0.0, 0, 0), 1),
    ((P, P, P, P, P, 1, 2, 2, 128, 128, 64, float("nan"), 0, 0), 1),
    ((P, P, P, P, P, 1, 2, 2, 128, 128, 64, 0.125, 0, 7), 1),
    # unsupported head dim
    ((P, P, P, P, P, 1, 2, 2, 128, 128, 96, 0.125, 0, 0), 2),
    # misaligned pointer
    ((P + 2, P, P, P, P, 1, 2, 2, 128, 128, 64, 0.125, 0, 0), 3),
    ((P, P, P, P, P + 4, 1, 2, 2, 128, 128, 64, 0.125, 0, 1), 3),
    # unknown causal mode; bottom-right with more queries than keys
    ((P, P, P, P, P, 1, 2, 2, 128, 128, 64, 0.125, 3, 0), 1),
    ((P, P, P, P, P, 1, 2, 2, 129, 128, 64, 0.125, 2, 0), 1),
])
def test_fwd_rejects_without_launch(lib, args, code):
    assert lib.attn_fwd(*args, None) == code


def test_bwd_validation_and_workspace(lib):
    ws = lib.attn_bwd_workspace_size(2, 16, 16, 8192, 8192, 128, 1)
    assert ws >= 2 * 16 * 8192 * 2 * 4 and ws % 256 == 0
    # per-group rows padded to a multiple of 128: G*Nq = 7*37 = 259 -> 384
    assert lib.attn_bwd_workspace_size(1, 7, 1, 37, 37, 64, 0) == 2 * 384 * 4
    assert lib.attn_bwd_workspace_size(1, 3, 2, 10, 10, 64, 0) == 0
    base = [P] * 9
    # workspace too small
    assert lib.attn_bwd(*base, P, 16, 2, 16, 16, 8192, 8192, 128, 0.08, 1, 1, None) == 6
    # null workspace
    assert lib.attn_bwd(*base, 0, ws, 2, 16, 16, 8192, 8192, 128, 0.08, 1, 1, None) == 1
    # misaligned dout
    bad = [P] * 9
    bad[4] = P + 8
    assert lib.attn_bwd(*bad, P, ws, 2, 16, 16, 8192, 8192, 128, 0.08, 1, 1, None) == 3


def test_fwd_ws_workspace_size_and_validation(lib):
    """bf16: the fp16 copy of v and one flag byte per (KV head, 128-key tile),
    each padded to 256 bytes; fp16 needs none.  Workspace errors come before
    any device call."""
    # 2*16 KV heads x 8192 keys x 128 dims x 2 bytes, then 32 x 64 flag bytes
    assert lib.attn_fwd_workspace_size(2, 16, 16, 8192, 8192, 128, 1) == \
        2 * 16 * 8192 * 128 * 2 + 2048
    # ragged: 1 x 2 heads x 300 keys x 64 x 2 = 76800 -> 76800; 2 x 3 flags -> 256
    assert lib.attn_fwd_workspace_size(1, 14, 2, 300, 300, 64, 1) == 76800 + 256
    assert lib.attn_fwd_workspace_size(1, 2, 2, 300, 300, 64, 0) == 0
    assert lib.attn_fwd_workspace_size(1, 3, 2, 300, 300, 64, 1) == 0   # invalid sizes
    ws = lib.attn_fwd_workspace_size(1, 2, 2, 128, 128, 64, 1)
    args = (1, 2, 2, 128, 128, 64, 0.125, 0, 1, None)
    assert lib.attn_fwd_ws(*([P] * 5), 0, ws, *args) == 1          # null workspace
    assert lib.attn_fwd_ws(*([P] * 5), P + 8, ws, *args) == 3      # misaligned workspace
    assert lib.attn_fwd_ws(*([P] * 5), P, ws - 1, *args) == 6      # too small
    assert lib.attn_fwd_ws(*([P] * 5), P, ws, 1, 2, 2, 128, 128, 96, 0.125, 0, 1, None) == 2
    # plan queries: small grids whose ranges would be under 4 key tiles (or no
    # device) are not cut; invalid sizes give 0
    assert lib.attn_fwd_ws_splits(1, 2, 2, 300, 300, 64, 0, 0) == 1
    assert lib.attn_fwd_ws_splits(1, 3, 2, 300, 300, 64, 0, 152) == 0
    assert lib.attn_bwd_splits(1, 2, 2, 300, 300, 64, 1, 0) == 1
    assert lib.attn_bwd_splits(1, 3, 2, 300, 300, 64, 0, 152) == 0


def test_launch_plans_for_152_sms(lib):
    """The grid plans for a 152-SM GB300, computed on the host.
    attn_fwd_ws: the last wave's units cut into 2..4 key ranges when a model
    of that wave says it pays; a grid under one wave cut into ranges of >= 16
    key tiles.  attn_bwd: dK/dV query ranges filling one wave, or (causal)
    sized so key tile 0's CTAs do no more than the average work per SM."""
    fwd = lambda B, Hq, Hkv, N, D, causal=0, Nk=None: lib.attn_fwd_ws_splits(
        B, Hq, Hkv, N, Nk or N, D, causal, 152)
    # the sweep (B=1, H=16, D=64): only N = 8192 (a last wave of 56 units) is cut
    assert [fwd(1, 16, 16, n, 64) for n in (256, 1024, 2048, 4096, 8192, 16384)] == [1, 1, 1, 1, 2, 1]
    assert fwd(1, 24, 24, 17600, 128) == 1 and fwd(1, 24, 24, 75600, 128) == 4   # video-DiT
    assert fwd(2, 16, 16, 8192, 128, causal=1) == 1          # causal grids are not cut
    assert fwd(1, 4, 4, 10240, 64, Nk=1000) == 2             # the parity cases of the cut
    assert fwd(1, 4, 4, 10240, 64, Nk=2048) == 4
    assert fwd(8, 14, 2, 1, 64, Nk=65536) == 9               # decode shape: 16 units, 512 key tiles
    bwd = lambda B, Hq, Hkv, N, D, causal: lib.attn_bwd_splits(B, Hq, Hkv, N, N, D, causal, 152)
    assert [bwd(1, 14, 2, n, 64, 1) for n in (2048, 4096, 8192, 16384)] == [9, 5, 3, 1]
    assert bwd(1, 14, 2, 4096, 64, 0) == 3
    assert bwd(2, 16, 16, 8192, 128, 1) == 1


def test_half_positions_for_152_sms(lib):
    """The causal forward's one-tile CTAs (D=64 fp16, Nq % 256 == 0): the
    heaviest pair positions run as two CTAs when a simulation of the grid on
    152 SMs says it saves >= 2%.  The GQA prefill (B=1, 14:2) splits at N =
    1024, 2048 and 4096 only."""
    half = lambda B, Hq, Hkv, N, D=64, causal=1, dtype=0, Nk=None, sms=152: \
        lib.attn_fwd_half_positions(B, Hq, Hkv, N, Nk or N, D, causal, dtype, sms)
    assert [half(1, 14, 2, n) for n in (1024, 2048, 4096, 8192, 16384)] == [2, 3, 1, 0, 0]
    assert half(1, 2, 2, 512) == 1 and half(1, 2, 2, 512, causal=2, Nk=1000) == 2
    # shapes the split does not serve
    assert half(1, 14, 2, 1024, causal=0) == 0            # no causal mask
    assert half(1, 14, 2, 1024, dtype=1) == 0             # bf16: one thread per row
    assert half(1, 14, 2, 1024, D=128) == 0
    assert half(1, 14, 2, 1000) == 0                      # Nq not a multiple of 256
    assert half(2, 16, 16, 8192, D=128, dtype=1) == 0     # the training forward
    assert half(1, 14, 2, 1024, sms=0) in (0, 2)          # current device (0 without one)
    assert half(1, 14, 3, 1024) == -1                     # invalid sizes
    assert half(1, 14, 2, 1024, causal=3) == -1


def _model_cut(B, Hq, Hkv, Nq, Nk, D, causal, sms):
    """Key ranges of attn_fwd_ws's grid, restated: several waves (no causal
    mask, >= 8 key tiles) cut the last wave into S = 2..4 ranges when rounds / S
    + (rounds - 1) * 15 us + 4 us of merge (in units of ~1.1 / 2.2 us per key
    tile at D = 64 / 128) beats a whole unit by 2%; under one wave every unit
    is cut into as many ranges of >= 16 key tiles as fill the SMs."""
    rows = Hq // Hkv * Nq
    units = B * Hkv * -(-rows // 256)
    tiles = -(-Nk // 128)
    if units >= sms:
        if causal or tiles < 8:
            return 1
        waves = -(-units // sms)
        tail = units - (waves - 1) * sms
        if waves < 2:
            return 1
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
            return 1
        tps = -(-tiles // best_s)
        return -(-tiles // tps)
    want = min(sms // units, tiles // 16, 256)
    if want < 2:
        return 1
    tps = -(-tiles // want)
    splits = -(-tiles // tps)
    return splits if splits >= 2 else 1


def _model_half(B, Hq, Nq, Nk, causal, sms, half=0.70, cta=2.5):
    """Heaviest pair positions run as one-tile CTAs, restated: simulate the
    grid's in-order assignment to the first free SM for each count h of split
    positions (a one-tile CTA costs `half` of its pair's key tiles, every CTA
    `cta` key tiles more) and keep the first h that beats the best so far by
    2%; grids of more than 8 waves of pairs are not split."""
    import heapq
    if Nq % 256:
        return 0
    m, heads = Nq // 256, B * Hq
    if heads * m > 8 * sms:
        return 0
    off = Nk - Nq if causal == 2 else 0
    t = []
    for i in range(m):
        keys = min((m - 1 - i) * 256 + 256 + off, Nk)
        t.append(0 if keys <= 0 else -(-keys // 128))
    best, best_h = None, 0
    for h in range(m + 1):
        free = [0.0] * sms
        end = 0.0
        for i in range(m):
            costs = [half * t[i] + cta] * 2 if i < h else [t[i] + cta]
            for _ in range(heads):
                for c in costs:
                    t0 = heapq.heappop(free)
                    heapq.heappush(free, t0 + c)
                    end = max(end, t0 + c)
        if best is None or end < 0.98 * best:
            best, best_h = end, h
    return best_h


def test_fwd_plans_match_a_model(lib):
    """Host-only: attn_fwd_ws's key ranges and the causal forward's one-tile
    positions on a 152-SM device agree with an independent restatement of the
    two plans over a grid of shapes."""
    import itertools
    n_cut = n_half = 0
    for (B, Hq, Hkv), N, extra, D in itertools.product(
            [(1, 16, 16), (1, 14, 2), (2, 4, 2), (1, 2, 2), (4, 24, 24)],
            [256, 512, 1024, 2048, 4096, 8192, 10240, 16384], [0, 300], [64, 128]):
        Nk = N + extra
        for causal in (0, 1):
            got = lib.attn_fwd_ws_splits(B, Hq, Hkv, N, Nk, D, causal, 152)
            want = _model_cut(B, Hq, Hkv, N, Nk, D, causal, 152)
            assert got == want, (B, Hq, Hkv, N, Nk, D, causal, got, want)
            n_cut += got > 1
        if D == 64 and N <= 4096:
            for causal in (1, 2):
                got = lib.attn_fwd_half_positions(B, Hq, Hkv, N, Nk, 64, causal, 0, 152)
                want = _model_half(B, Hq, N, Nk, causal, 152)
                assert got == want, (B, Hq, Hkv, N, Nk, causal, got, want)
                n_half += got > 0
    assert n_cut > 5 and n_half > 5   # the grid exercises both plans


def _model_bwd(B, Hq, Hkv, Nq, Nk, causal, sms):
    """dK/dV query ranges, restated: none when the (group, key tile) CTAs fill
    the SMs; otherwise enough ranges to fill one wave, or (causal) enough that
    key tile 0's CTAs, which meet every query tile, do no more than the average
    work per SM; at least 4 query tiles per range, at most 32 ranges."""
    groups, ktiles = B * Hkv, -(-Nk // 128)
    n_qtiles = -(-(Hq // Hkv) * Nq // 128)
    units = groups * ktiles
    if units >= sms:
        return 1
    want = -(-sms // units)
    if causal:
        tq = -(-Nq // 128)
        total = sum(tq - kt for kt in range(min(ktiles, tq)))
        if total > 0:
            want = -(-tq * sms // (groups * total))
    want = min(want, n_qtiles // 4, 32)
    if want <= 1:
        return 1
    per = -(-n_qtiles // want)
    return -(-n_qtiles // per)


def test_bwd_plan_matches_a_model(lib):
    """Host-only: attn_bwd's dK/dV query ranges on a 152-SM device agree with
    an independent restatement of the plan over a grid of shapes."""
    import itertools
    cut = 0
    for (B, Hq, Hkv), N, extra, causal in itertools.product(
            [(1, 14, 2), (2, 16, 16), (1, 4, 4), (8, 8, 1), (1, 2, 2)],
            [128, 512, 1024, 2048, 4096, 8192, 16384], [0, 700], (0, 1)):
        got = lib.attn_bwd_splits(B, Hq, Hkv, N, N + extra, 64, causal, 152)
        want = _model_bwd(B, Hq, Hkv, N, N + extra, causal, 152)
        assert got == want, (B, Hq, Hkv, N, N + extra, causal, got, want)
        cut += got > 1
    assert cut > 10


def test_bwd_rejects_bottom_right(lib):
    ws = lib.attn_bwd_workspace_size(1, 2, 2, 128, 256, 64, 0)
    assert lib.attn_bwd(*([P] * 9), P, ws, 1, 2, 2, 128, 256, 64, 0.125, 2, 0, None) == 2
    assert lib.attn_bwd(*([P] * 9), P, ws, 1, 2, 2, 128, 256, 64, 0.125, 5, 0, None) == 1


def test_num_splits_heuristic(lib):
    """Host-only: one wave of CTAs on num_sms SMs, >= 2 key tiles per range,
    and no empty range."""
    # decode, 8 sequences, Qwen-like GQA (14:2): 16 units -> 9 wanted on 152
    # SMs; 32 key tiles in ranges of 4 -> 8 ranges
    assert lib.attn_fwd_num_splits(8, 14, 2, 1, 4096, 64, 152) == 8
    # a grid that already fills the GPU is not split
    assert lib.attn_fwd_num_splits(1, 16, 16, 16384, 16384, 64, 152) == 1
    # two key tiles: at most one range
    assert lib.attn_fwd_num_splits(1, 2, 2, 1, 200, 64, 152) == 1
    # one unit, long keys: 152 ranges of 7 tiles cover 1024 tiles in 147
    assert lib.attn_fwd_num_splits(1, 1, 1, 1, 131072, 128, 152) == 147
    assert lib.attn_fwd_num_splits(1, 3, 2, 1, 4096, 64, 152) == 1   # invalid sizes
    # the decode benchmark's cache lengths: the counts a GB300 sweep of 1-32 ranges found
    # fastest (1K: 4 or 8 tied; 4K: 8 or 9 tied; 16K and 64K: 9)
    for nk, best in ((1024, (4, 8)), (4096, (8, 9)), (16384, (9,)), (65536, (9,))):
        assert lib.attn_fwd_num_splits(8, 14, 2, 1, nk, 64, 152) in best, nk


def test_splitkv_workspace_and_validation(lib):
    ws = lib.attn_fwd_splitkv_workspace_size(8, 14, 2, 1, 4096, 64, 8)
    rows = 8 * 14 * 1
    assert ws == 8 * rows * 64 * 4 + ((8 * rows * 4 + 255) // 256) * 256
    # 9 requested on 32 tiles is ranges of 4 tiles: 8 ranges
    assert lib.attn_fwd_splitkv_workspace_size(8, 14, 2, 1, 4096, 64, 9) == ws
    assert lib.attn_fwd_splitkv_workspace_size(8, 14, 2, 1, 4096, 64, 1) == 0
    assert lib.attn_fwd_splitkv_workspace_size(8, 14, 2, 1, 4096, 64, 257) == 0
    assert lib.attn_fwd_splitkv_workspace_size(8, 14, 3, 1, 4096, 64, 8) == 0
    args = (8, 14, 2, 1, 4096, 64, 0.125, 0, 0)
    # bad range count, null / misaligned / short workspace: all before any device call
    assert lib.attn_fwd_splitkv(P, P, P, P, P, P, ws, *args, 0, None) == 1
    assert lib.attn_fwd_splitkv(P, P, P, P, P, 0, ws, *args, 8, None) == 1
    assert lib.attn_fwd_splitkv(P, P, P, P, P, P + 8, ws, *args, 8, None) == 3
    assert lib.attn_fwd_splitkv(P, P, P, P, P, P, ws - 16, *args, 8, None) == 6


def test_ffn_host_checks(lib):
    assert lib.ffn_workspace_size(1000, 4864, 256) == 256 * 4864 * 2
    assert lib.ffn_workspace_size(100, 4864, 256) == (100 * 4864 * 2 + 255) // 256 * 256
    assert lib.ffn_workspace_size(0, 4864, 256) == 0
    ws = lib.ffn_workspace_size(1000, 4864, 256)
    args = (1000, 896, 4864, 4, 256, P, ws, 1, None)
    # null x, unknown activation, d_model not a multiple of 8, misaligned, short workspace
    assert lib.ffn_forward(0, P, 0, P, 0, P, *args) == 1
    assert lib.ffn_forward(P, P, 0, P, 0, P, 1000, 896, 4864, 9, 256, P, ws, 1, None) == 1
    assert lib.ffn_forward(P, P, 0, P, 0, P, 1000, 900, 4864, 4, 256, P, ws, 1, None) == 2
    assert lib.ffn_forward(P + 8, P, 0, P, 0, P, *args) == 3
    assert lib.ffn_forward(P, P, 0, P, 0, P, 1000, 896, 4864, 4, 256, P, ws - 256, 1, None) == 6
    assert lib.attn_strerror(7) == b"results that must agree differ"
