"""Decode-update variants of the CUDA path against the oracle's general form (GPU).

cconv_update_ex through the C ABI: state length L = W (one token more than the window),
padding rows (index -1 touches nothing when the mode is on, and is an invalid negative
index when it is off), activation None, on the vector and the scalar paths; the plain
settings must reproduce cconv_update bit for bit.  Pools are compared bit for bit, y within
the forward tolerance; rows the call must not write are checked against a sentinel.
"""
import numpy as np
import pytest
import torch

import depthwise_causal_short_gb300 as cc
import oracle
from depthwise_causal_short_gb300 import _build, inputs
from tests.helpers import FWD_TOL, bits, f64, rel_err

pytestmark = pytest.mark.gpu

SENTINEL = 0x7F7F  # a bf16 bit pattern no computed y row is expected to hold everywhere


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    return cc.load()


def _pool(S, D, L, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(S, D, L, generator=g).to(torch.bfloat16)


def _steps(W, L, D, ldpad, pad, act, idx_rows, steps, seed, wdtype=torch.float32):
    """Runs `steps` decode steps on the GPU and the oracle side by side."""
    S = max(29, max(idx_rows) + 1)
    N = len(idx_rows)
    _, xr, _, w, b = inputs.decode_inputs(S, N, D, W, True, n_x=steps, seed=seed, wdtype=wdtype)
    state = _pool(S, D, L, seed + 1)
    rows = torch.zeros(steps, N, D + ldpad, dtype=torch.bfloat16)
    rows[:, :, :D] = xr
    rows_g = rows.cuda()
    state_g, wg, bg = state.cuda(), w.cuda(), b.cuda()
    idx = torch.tensor(idx_rows, dtype=torch.int32)
    idx_g = idx.cuda()
    st_ref = bits(state)
    live = idx >= 0
    for k in range(steps):
        y = torch.full((N, D), 0, dtype=torch.int16)
        y[:] = SENTINEL
        y = y.view(torch.bfloat16).cuda()
        _, status = cc.cconv_update_ex(rows_g[k, :, :D], state_g, wg, bg, idx_g, pad_rows=pad,
                                       activation=act, y=y)
        torch.cuda.synchronize()
        assert status.tolist() == [0, 0], f"step {k}: status {status.tolist()}"
        rc, y_ref, st_ref = oracle.update_ex(bits(xr[k]), st_ref, idx.numpy(), f64(w), f64(b),
                                             pad=pad, activation=act)
        assert rc == 0
        yc = y.cpu()
        e = rel_err(f64(yc[live]), y_ref[live.numpy()])
        assert e <= FWD_TOL, f"W={W} L={L} step {k}: y err {e:.2e}"
        assert np.all(bits(yc[~live]) == SENTINEL), "a padding row's y was written"
    assert np.array_equal(bits(state_g), st_ref), f"W={W} L={L}: pool differs"


@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("D,ldpad", [(4096, 0), (1000, 8), (1001, 0)])
@pytest.mark.parametrize("act", ["silu", None], ids=["silu", "none"])
def test_state_length_w(W, D, ldpad, act):
    _steps(W, W, D, ldpad, False, act, [4, 17, 0, 28, 9, 3, 11], steps=4, seed=W + D)


@pytest.mark.parametrize("W", [2, 4])
@pytest.mark.parametrize("L_off", [0, 1])
@pytest.mark.parametrize("D,ldpad", [(2048, 0), (1001, 0)])
def test_padding_rows(W, L_off, D, ldpad):
    _steps(W, W - 1 + L_off, D, ldpad, True, "silu", [5, -1, 12, -1, -1, 0, 27, 6, -1],
           steps=3, seed=40 + W)


def test_many_rows_state_length_w():
    """256 rows (the decode workload's batch) with L = W over 6 steps: the row-blocked
    kernel; then the pool holds the last 4 tokens of every row, bit for bit."""
    g = torch.Generator().manual_seed(77)
    idx = torch.randperm(512, generator=g)[:256].tolist()
    _steps(4, 4, 4096, 0, False, "silu", idx, steps=6, seed=77)


def test_plain_settings_equal_cconv_update():
    S, N, D, W = 64, 40, 2048, 4
    state, xr, idx, w, b = inputs.decode_inputs(S, N, D, W, True, n_x=2, seed=50)
    a, c = state.cuda(), state.cuda()
    ya, sa = cc.cconv_update(xr[0].cuda(), a, w.cuda(), b.cuda(), idx.cuda())
    yc, sc = cc.cconv_update_ex(xr[0].cuda(), c, w.cuda(), b.cuda(), idx.cuda())
    torch.cuda.synchronize()
    assert sa.tolist() == sc.tolist() == [0, 0]
    assert torch.equal(ya.view(torch.int16), yc.view(torch.int16))
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))


@pytest.mark.parametrize("pad,idx,mask", [
    (True, [3, -2, 5], 1),          # -2 is no padding marker
    (True, [3, -1, 3], 4),          # repeats among real rows still fail
    (True, [3, -1, 99], 2),
    (False, [3, -1, 5], 1),         # without the mode -1 is a negative index
])
def test_invalid_with_padding_mode(pad, idx, mask):
    S, D, W = 8, 512, 4
    state = _pool(S, D, W, 60).cuda()
    before = state.clone()
    g = torch.Generator().manual_seed(61)
    x = torch.randn(len(idx), D, generator=g).to(torch.bfloat16).cuda()
    w = torch.rand(D, W, generator=g).cuda()
    y = torch.zeros(len(idx), D, dtype=torch.bfloat16).cuda()
    _, status = cc.cconv_update_ex(x, state, w, None, torch.tensor(idx, dtype=torch.int32).cuda(),
                                   pad_rows=pad, y=y)
    torch.cuda.synchronize()
    assert status.tolist() == [-8, mask]
    assert torch.equal(state.view(torch.int16), before.view(torch.int16))
    assert not y.float().any(), "y written on a rejected call"


def _ring_steps(W, L, D, ldpad, pad, act, idx_rows, steps, seed, start):
    """Circular-buffer decode: `steps` steps with cache_seqlens = start + step, against the
    oracle's circular form; pools bit for bit, y within tolerance, padding y untouched."""
    S = max(29, max(idx_rows) + 1)
    N = len(idx_rows)
    _, xr, _, w, b = inputs.decode_inputs(S, N, D, W, True, n_x=steps, seed=seed)
    state = _pool(S, D, L, seed + 1)
    rows = torch.zeros(steps, N, D + ldpad, dtype=torch.bfloat16)
    rows[:, :, :D] = xr
    rows_g = rows.cuda()
    state_g, wg, bg = state.cuda(), w.cuda(), b.cuda()
    idx = torch.tensor(idx_rows, dtype=torch.int32)
    idx_g = idx.cuda()
    st_ref = bits(state)
    live = idx >= 0
    for k in range(steps):
        pos = torch.tensor([start[i] + k for i in range(N)], dtype=torch.int32)
        y = torch.full((N, D), 0, dtype=torch.int16)
        y[:] = SENTINEL
        y = y.view(torch.bfloat16).cuda()
        _, status = cc.cconv_update_ex(rows_g[k, :, :D], state_g, wg, bg, idx_g, pad_rows=pad,
                                       cache_seqlens=pos.cuda(), activation=act, y=y)
        torch.cuda.synchronize()
        assert status.tolist() == [0, 0], f"step {k}: status {status.tolist()}"
        rc, y_ref, st_ref = oracle.update_ring(bits(xr[k]), st_ref, idx.numpy(), pos.numpy(),
                                               f64(w), f64(b), pad=pad, activation=act)
        assert rc == 0
        yc = y.cpu()
        e = rel_err(f64(yc[live]), y_ref[live.numpy()])
        assert e <= FWD_TOL, f"ring W={W} L={L} step {k}: y err {e:.2e}"
        assert np.all(bits(yc[~live]) == SENTINEL), "a padding row's y was written"
    assert np.array_equal(bits(state_g), st_ref), f"ring W={W} L={L}: pool differs"


@pytest.mark.parametrize("D,N,W,L_off,pad", [(808, 157, 4, 1, True), (4096, 200, 3, 0, False),
                                              (2048, 300, 4, 1, False)])
def test_row_lane_layouts_general(D, N, W, L_off, pad):
    """The general kernels on the 256-thread CTAs: a partial channel block, row groups split
    unevenly, padding rows mixed in."""
    g = torch.Generator().manual_seed(D + N)
    idx = torch.randperm(N + 40, generator=g)[:N]
    if pad:
        idx[::7] = -1
    _steps(W, W - 1 + L_off, D, 0, pad, "silu", idx.tolist(), steps=2, seed=D + N)


@pytest.mark.parametrize("W,L", [(4, 3), (4, 4), (3, 2), (3, 3), (2, 1), (2, 2), (1, 1)])
@pytest.mark.parametrize("D,ldpad", [(4096, 0), (1000, 8), (1001, 0)])
def test_circular_buffer(W, L, D, ldpad):
    start = [0, 1, 5, 2, 7, 100, 3]        # different positions per row, wrapping
    _ring_steps(W, L, D, ldpad, False, "silu", [4, 17, 0, 28, 9, 3, 11], steps=5, seed=W + L,
                start=start)


def test_circular_buffer_padding_and_no_activation():
    start = [3, 0, 9, 0, 1, 4, 0, 2, 6]
    _ring_steps(4, 4, 2048, 0, True, None, [5, -1, 12, -1, -1, 0, 27, 6, -1], steps=4, seed=90,
                start=start)


def test_circular_buffer_many_rows():
    g = torch.Generator().manual_seed(91)
    idx = torch.randperm(512, generator=g)[:256].tolist()
    start = torch.randint(0, 50, (256,), generator=g).tolist()
    _ring_steps(4, 3, 4096, 0, False, "silu", idx, steps=4, seed=91, start=start)


def test_circular_buffer_negative_position():
    """cache_seqlens is taken modulo L, non-negative: -1 is entry L - 1."""
    _ring_steps(4, 3, 512, 0, False, "silu", [0, 1, 2], steps=3, seed=92, start=[-1, -5, -3])
