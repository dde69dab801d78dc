"""Largest shapes (GPU): very wide rows and a very long sequence, against the oracle.

Very wide: D = 2^20 + 8 channels (1025 forward channel groups, several waves of CTAs) over
a few rows, compared in full.  Very long: one sequence of 2^24 rows at D = 8 (row indices
past 2^24, 268 MB per activation tensor); the packed-sequence forward over the same rows
must equal the batched one bit for bit.  The oracle runs in chunks: a chunk of the sequence
with the 3 rows before it as its initial state has exactly the forward and the dw / dbias
contributions of those rows, so dw / dbias are checked in full and y / dx on sampled
windows (dx away from each window's end, where g past it would be needed).
"""
import numpy as np
import pytest
import torch

import depthwise_causal_short_gb300 as cc
import oracle
from depthwise_causal_short_gb300 import _build, inputs
from tests.helpers import BWD_TOL, FWD_TOL, f64, oracle_bwd, oracle_fwd, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    return cc.load()


def test_very_wide_rows():
    B, T, D, W = 1, 7, (1 << 20) + 8, 4
    x, dy, w, b = inputs.fwd_bwd_inputs(B, T, D, W, True, seed=80)
    dev = torch.device("cuda", 0)
    y = cc.cconv_fwd(x.to(dev), w.to(dev), b.to(dev))
    dx, dw, db = cc.cconv_bwd(x.to(dev), dy.to(dev), w.to(dev), b.to(dev))
    torch.cuda.synchronize()
    assert rel_err(f64(y), oracle_fwd(x, w, b)) <= FWD_TOL
    rdx, rdw, rdb = oracle_bwd(x, dy, w, b)
    for name, g, r in (("dx", dx, rdx), ("dw", dw, rdw), ("dbias", db, rdb)):
        assert rel_err(f64(g), r) <= BWD_TOL, name


def test_very_long_sequence():
    T, D, W = 1 << 24, 8, 4
    g = torch.Generator().manual_seed(81)
    x = torch.randn(1, T, D, generator=g).to(torch.bfloat16)
    dy = torch.randn(1, T, D, generator=g).to(torch.bfloat16)
    w = torch.rand(D, W, generator=g) - 0.5
    b = (torch.rand(D, generator=g) - 0.5) * 0.2
    dev = torch.device("cuda", 0)
    xg, dyg = x.to(dev), dy.to(dev)
    y = cc.cconv_fwd(xg, w.to(dev), b.to(dev))
    dx, dw, db = cc.cconv_bwd(xg, dyg, w.to(dev), b.to(dev))
    # the packed-sequence path over the same rows, as one sequence
    cu = torch.tensor([0, T], dtype=torch.int32, device=dev)
    yv, _, _ = cc.cconv_fwd_varlen(xg.view(T, D), cu, w.to(dev), b.to(dev))
    torch.cuda.synchronize()
    assert torch.equal(y.view(T, D).view(torch.int16), yv.view(torch.int16))
    # host copies in fp32 (exact for bf16); fp64 only chunk by chunk
    y, dx = y[0].float().cpu().numpy(), dx[0].float().cpu().numpy()
    xs, dys = x[0].float().numpy(), dy[0].float().numpy()
    wd, bd = f64(w), f64(b)

    def init_before(r):
        out = np.zeros((1, D, W - 1))
        k = min(r, W - 1)
        if k:
            out[0, :, W - 1 - k:] = xs[r - k:r].T
        return out

    chunk = 1 << 21
    dw_ref = np.zeros((D, W))
    db_ref = np.zeros(D)
    rng = np.random.default_rng(82)
    for c0 in range(0, T, chunk):
        xc = xs[c0:c0 + chunk].astype(np.float64)
        dyc = dys[c0:c0 + chunk].astype(np.float64)
        cu_c = np.array([0, xc.shape[0]], np.int64)
        _, cdw, cdb, _ = oracle.bwd_seq(xc, dyc, cu_c, wd, bd, init_before(c0))
        dw_ref += cdw
        db_ref += cdb
        # sampled windows of y and dx (dx away from the window's end, where g past it
        # would be needed)
        for s_ in rng.integers(0, chunk - 512, size=2):
            lo = c0 + int(s_)
            xw = xs[lo:lo + 256].astype(np.float64)
            dyw = dys[lo:lo + 256].astype(np.float64)
            cu_w = np.array([0, 256], np.int64)
            yw = oracle.fwd_seq(xw, cu_w, wd, bd, init_before(lo))
            assert rel_err(y[lo:lo + 256], yw) <= FWD_TOL, f"y window at {lo}"
            dxw = oracle.bwd_seq(xw, dyw, cu_w, wd, bd, init_before(lo))[0]
            assert rel_err(dx[lo:lo + 250], dxw[:250]) <= BWD_TOL, f"dx window at {lo}"
    assert rel_err(f64(dw), dw_ref) <= BWD_TOL
    assert rel_err(f64(db), db_ref) <= BWD_TOL
