"""Decode-update parity of the CUDA path against the oracle (GPU).

The decode workload (pool [512, 4096, 3] bf16, 256 active rows, W=4, bias) runs its 1000
steps through the C ABI; every step's y is compared with the oracle and the pool is
compared bit for bit.  Invalid index vectors (negative, out of range, duplicate) must be
rejected with the oracle's offence bits and leave the pool and y untouched, without a
trap.  Narrow widths, the scalar path (D not a multiple of 8, padded rows), NULL indices
and the largest pool the in-kernel check accepts are covered too.
"""
import numpy as np
import pytest
import torch

import depthwise_causal_short_gb300 as cc
import oracle
from depthwise_causal_short_gb300 import _build, inputs
from tests.helpers import FWD_TOL, bits, f64, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    return cc.load()


def _step_and_check(xg, state_g, wg, bg, idx_g, st_ref, x_cpu, idx_cpu, w, b, what):
    y, status = cc.cconv_update(xg, state_g, wg, bg, idx_g)
    torch.cuda.synchronize()
    assert status.tolist() == [0, 0], f"{what}: status {status.tolist()}"
    rc, y_ref, st_ref = oracle.update(bits(x_cpu), st_ref, None if idx_cpu is None else
                                      idx_cpu.numpy(), f64(w), f64(b))
    assert rc == 0
    e = rel_err(y.double().cpu().numpy(), y_ref)
    assert e <= FWD_TOL, f"{what}: y err {e:.2e}"
    return st_ref


def test_decode_workload_1000_steps():
    sh = inputs.DECODE_SHAPE
    state, xr, idx, w, b = inputs.decode_inputs(sh.S, sh.N, sh.D, sh.W, sh.bias, n_x=16)
    state_g, xr_g, idx_g, wg, bg = state.cuda(), xr.cuda(), idx.cuda(), w.cuda(), b.cuda()
    st_ref = bits(state)
    for step in range(sh.steps):
        k = step % xr.shape[0]
        st_ref = _step_and_check(xr_g[k], state_g, wg, bg, idx_g, st_ref, xr[k], idx, w, b,
                                 f"step {step}")
        if step % 100 == 99 or step == sh.steps - 1:
            assert np.array_equal(bits(state_g), st_ref), f"pool differs after step {step}"


@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("D,pad", [(4096, 0), (1000, 8), (1001, 0), (24, 5)])
def test_widths_and_layouts(W, D, pad):
    S, N = 37, 11
    state, xr, idx, w, b = inputs.decode_inputs(S, N, D, W, True, n_x=3, seed=W * 10 + D)
    rows = torch.zeros(xr.shape[0], N, D + pad, dtype=torch.bfloat16)
    rows[:, :, :D] = xr
    rows_g = rows.cuda()
    state_g, idx_g, wg, bg = state.cuda(), idx.cuda(), w.cuda(), b.cuda()
    st_ref = bits(state)
    for k in range(3):
        st_ref = _step_and_check(rows_g[k, :, :D], state_g, wg, bg, idx_g, st_ref, xr[k], idx,
                                 w, b, f"W{W} D{D} pad{pad} step {k}")
    assert np.array_equal(bits(state_g), st_ref)


# Batches large enough for the 256-thread CTAs (32 channel vectors x 8 row lanes with staged
# taps): a partial last channel block (D=808: 101 vectors), row groups split unevenly over a
# grid sized to the SM count, 1-, 2- and 4-row kernels, bf16 and fp32 taps, no bias, and a
# grid of more than one wave (D=8192 N=512).
ROW_LANE_CASES = [
    (808, 157, 4, torch.float32, True),
    (808, 157, 3, torch.bfloat16, False),
    (1024, 192, 1, torch.float32, True),
    (2048, 300, 2, torch.bfloat16, True),
    (4096, 128, 4, torch.float32, True),
    (4096, 200, 4, torch.float32, False),
    (8192, 512, 4, torch.float32, True),
]


@pytest.mark.parametrize("D,N,W,wdtype,bias", ROW_LANE_CASES,
                         ids=[f"D{c[0]}-N{c[1]}-W{c[2]}-{str(c[3])[6:]}-b{int(c[4])}"
                              for c in ROW_LANE_CASES])
def test_row_lane_layouts(D, N, W, wdtype, bias):
    S = N + 37
    state, xr, idx, w, b = inputs.decode_inputs(S, N, D, W, bias, n_x=2, seed=D + N + W,
                                                wdtype=wdtype)
    state_g, xr_g, idx_g, wg = state.cuda(), xr.cuda(), idx.cuda(), w.cuda()
    bg = None if b is None else b.cuda()
    st_ref = bits(state)
    for k in range(2):
        st_ref = _step_and_check(xr_g[k], state_g, wg, bg, idx_g, st_ref, xr[k], idx, w, b,
                                 f"D{D} N{N} W{W} step {k}")
    assert np.array_equal(bits(state_g), st_ref)
    # rows outside the index vector keep their state
    untouched = np.setdiff1d(np.arange(S), idx.numpy())
    assert np.array_equal(bits(state_g)[untouched], bits(state)[untouched])


def test_null_indices_and_bf16_weights():
    S, N, D, W = 20, 16, 512, 4
    state, xr, _, w, b = inputs.decode_inputs(S, N, D, W, True, n_x=2, seed=21,
                                              wdtype=torch.bfloat16)
    state_g, xr_g, wg, bg = state.cuda(), xr.cuda(), w.cuda(), b.cuda()
    st_ref = bits(state)
    for k in range(2):
        st_ref = _step_and_check(xr_g[k], state_g, wg, bg, None, st_ref, xr[k], None, w, b,
                                 f"null idx step {k}")
    assert np.array_equal(bits(state_g), st_ref)


INVALID = {
    "negative": ([3, -1, 7, 2], 1),
    "out_of_range": ([3, 16, 7, 2], 2),
    "duplicate": ([3, 9, 7, 9], 4),
    "negative_and_duplicate": ([5, 5, -7, 1], 5),
    "all_three": ([16, -2, 4, 4], 7),
}


@pytest.mark.parametrize("case", sorted(INVALID))
def test_invalid_indices_fail_closed(case):
    S, N, D, W = 16, 4, 256, 4
    idx_list, mask = INVALID[case]
    state, xr, _, w, b = inputs.decode_inputs(S, N, D, W, True, n_x=1, seed=31)
    idx = torch.tensor(idx_list, dtype=torch.int32)
    assert oracle.validate(idx.numpy(), S) == mask
    state_g = state.cuda()
    before = bits(state_g)
    y = torch.full((N, D), 7.0, dtype=torch.bfloat16, device="cuda")
    status = torch.full((2,), 99, dtype=torch.int32, device="cuda")
    cc.cconv_update(xr[0].cuda(), state_g, w.cuda(), b.cuda(), idx.cuda(), y=y, status=status)
    torch.cuda.synchronize()
    assert status.tolist() == [-8, mask]
    assert np.array_equal(bits(state_g), before), "pool changed on a rejected call"
    assert torch.all(y == 7.0), "y written on a rejected call"
    # the context is still usable and a valid call afterwards succeeds
    y2, st2 = cc.cconv_update(xr[0].cuda(), state_g, w.cuda(), b.cuda(),
                              torch.tensor([0, 1, 2, 3], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert st2.tolist() == [0, 0]


def test_largest_pool():
    S, N, D, W = 393216, 8, 8, 4
    state = torch.zeros(S, D, W - 1, dtype=torch.bfloat16, device="cuda")
    x = torch.ones(N, D, dtype=torch.bfloat16, device="cuda")
    w = torch.full((D, W), 0.25, device="cuda")
    idx = torch.tensor([0, 1, 2, 3, S - 4, S - 3, S - 2, S - 1], dtype=torch.int32, device="cuda")
    y, status = cc.cconv_update(x, state, w, None, idx)
    torch.cuda.synchronize()
    assert status.tolist() == [0, 0]
    assert torch.all(state[S - 1, :, W - 2] == 1.0) and torch.all(state[4:S - 4] == 0)
    with pytest.raises(cc.CConvError) as e:
        cc.cconv_update(x, torch.zeros(S + 1, D, W - 1, dtype=torch.bfloat16, device="cuda"),
                        w, None, idx)
    assert e.value.status == -2


def test_sequential_updates_match_gpu_forward():
    """T decode steps from a zero state give the forward's rows (both on the GPU)."""
    B, T, D, W = 3, 12, 256, 4
    x, _, w, b = inputs.fwd_bwd_inputs(B, T, D, W, True, seed=41)
    xg, wg, bg = x.cuda(), w.cuda(), b.cuda()
    y_full = cc.cconv_fwd(xg, wg, bg)
    state = torch.zeros(B, D, W - 1, dtype=torch.bfloat16, device="cuda")
    for t in range(T):
        y, st = cc.cconv_update(xg[:, t, :], state, wg, bg, None)
        torch.cuda.synchronize()
        assert st.tolist() == [0, 0]
        assert rel_err(y.double().cpu().numpy(), y_full[:, t, :].double().cpu().numpy()) <= 1e-2
    assert np.array_equal(bits(state), bits(xg[:, T - 3:, :].permute(0, 2, 1)))
