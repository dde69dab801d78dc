"""Forward / backward parity of the CUDA path against the fp64 oracle (GPU).

All five training-shaped workloads run at their full sizes through the C ABI, in the same
launch configuration the benchmark times, and are compared element by element with the
oracle.  Smaller grids cover the ragged cases (T and D tails, T < 4, B = 1, W < 4, no bias,
bf16 weights, strided inputs); guard bands check that nothing is written outside y / dx;
the backward is checked to be bit-for-bit repeatable; a CUDA-graph replay must equal the
eager calls bit for bit.
"""
import numpy as np
import pytest
import torch

import depthwise_causal_short_gb300 as cc
from depthwise_causal_short_gb300 import _build, inputs
from tests.helpers import BWD_TOL, FWD_TOL, bits, oracle_bwd, oracle_fwd, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    return cc.load()


def _run(x, dy, w, b, want_dbias=None):
    xg, dyg, wg = x.cuda(), dy.cuda(), w.cuda()
    bg = None if b is None else b.cuda()
    y = cc.cconv_fwd(xg, wg, bg)
    dx, dw, db = cc.cconv_bwd(xg, dyg, wg, bg, want_dbias=want_dbias)
    torch.cuda.synchronize()
    return y, dx, dw, db


def _check(x, dy, w, b, y, dx, dw, db, what):
    y_ref = oracle_fwd(x, w, b)
    e = rel_err(y.double().cpu().numpy(), y_ref)
    assert e <= FWD_TOL, f"{what}: fwd err {e:.2e}"
    dx_ref, dw_ref, db_ref = oracle_bwd(x, dy, w, b, want_dbias=db is not None)
    for name, g, r in (("dx", dx, dx_ref), ("dw", dw, dw_ref), ("dbias", db, db_ref)):
        if g is None:
            continue
        e = rel_err(g.double().cpu().numpy(), r)
        assert e <= BWD_TOL, f"{what}: {name} err {e:.2e}"


@pytest.mark.parametrize("wdtype", [torch.float32, torch.bfloat16], ids=["w_f32", "w_bf16"])
@pytest.mark.parametrize("shape", inputs.FWD_BWD_SHAPES, ids=lambda s: s.name)
def test_workloads_full_size(shape, wdtype):
    x, dy, w, b = inputs.fwd_bwd_inputs(shape.B, shape.T, shape.D, shape.W, shape.bias,
                                        wdtype=wdtype)
    y, dx, dw, db = _run(x, dy, w, b, want_dbias=True)
    _check(x, dy, w, b, y, dx, dw, db, shape.name)


EDGE = [
    (1, 1, 8, 4), (1, 2, 8, 4), (1, 3, 16, 4), (2, 4, 8, 3), (3, 5, 24, 2), (2, 17, 264, 4),
    (1, 33, 1000, 1), (2, 100, 136, 4), (1, 777, 512, 3), (5, 31, 2056, 4), (1, 4097, 256, 4),
]


@pytest.mark.parametrize("with_bias", [True, False])
@pytest.mark.parametrize("B,T,D,W", EDGE)
def test_edge_shapes(B, T, D, W, with_bias):
    x, dy, w, b = inputs.fwd_bwd_inputs(B, T, D, W, with_bias, seed=B * 1000 + T + D + W)
    y, dx, dw, db = _run(x, dy, w, b, want_dbias=True)
    _check(x, dy, w, b, y, dx, dw, db, f"B{B} T{T} D{D} W{W}")


def test_strided_inputs():
    B, T, D, W = 3, 300, 512, 4
    x, dy, w, b = inputs.fwd_bwd_inputs(B, T, D, W, True, seed=5)
    # x: a channel slice of a wider activation; dy: a [T,B,D] buffer viewed as [B,T,D]
    wide = torch.zeros(B, T, D + 256, dtype=torch.bfloat16, device="cuda")
    wide[:, :, 128:128 + D] = x.cuda()
    xv = wide[:, :, 128:128 + D]
    tbd = dy.transpose(0, 1).contiguous().cuda()
    dyv = tbd.transpose(0, 1)
    assert xv.stride() == (T * (D + 256), D + 256, 1) and dyv.stride() == (D, B * D, 1)
    wg, bg = w.cuda(), b.cuda()
    y = cc.cconv_fwd(xv, wg, bg)
    dx, dw, db = cc.cconv_bwd(xv, dyv, wg, bg)
    torch.cuda.synchronize()
    _check(x, dy, w, b, y, dx, dw, db, "strided")


def test_outputs_stay_in_bounds():
    B, T, D, W = 2, 123, 1000, 4
    x, dy, w, b = inputs.fwd_bwd_inputs(B, T, D, W, True, seed=9)
    n = B * T * D
    guard = 4096
    canary = torch.full((n + 2 * guard,), 12345, dtype=torch.int16, device="cuda")
    y = canary.view(torch.bfloat16)[guard:guard + n].view(B, T, D)
    canary2 = canary.clone()
    dx = canary2.view(torch.bfloat16)[guard:guard + n].view(B, T, D)
    xg, dyg, wg, bg = x.cuda(), dy.cuda(), w.cuda(), b.cuda()
    cc.cconv_fwd(xg, wg, bg, y=y)
    cc.cconv_bwd(xg, dyg, wg, bg, dx=dx)
    torch.cuda.synchronize()
    for c in (canary, canary2):
        assert torch.all(c[:guard] == 12345) and torch.all(c[guard + n:] == 12345)
    _check(x, dy, w, b, y, dx, None, None, "guarded")


def test_backward_is_deterministic():
    s = inputs.PROD
    x, dy, w, b = inputs.fwd_bwd_inputs(s.B, s.T, s.D, s.W, True, seed=3)
    xg, dyg, wg, bg = x.cuda(), dy.cuda(), w.cuda(), b.cuda()
    ws = torch.empty(cc.cconv_bwd_workspace_bytes(s.B, s.T, s.D, s.W), dtype=torch.uint8,
                     device="cuda")
    r1 = cc.cconv_bwd(xg, dyg, wg, bg, workspace=ws)
    r1 = [t.clone() for t in r1]
    ws.fill_(0xFF)  # stale workspace contents must not matter
    r2 = cc.cconv_bwd(xg, dyg, wg, bg, workspace=ws)
    torch.cuda.synchronize()
    assert np.array_equal(bits(r1[0]), bits(r2[0]))
    assert torch.equal(r1[1], r2[1]) and torch.equal(r1[2], r2[2])


def test_cuda_graph_replay_matches_eager():
    B, T, D, W = 2, 1024, 2048, 4
    x, dy, w, b = inputs.fwd_bwd_inputs(B, T, D, W, True, seed=4)
    xg, dyg, wg, bg = x.cuda(), dy.cuda(), w.cuda(), b.cuda()
    y0 = cc.cconv_fwd(xg, wg, bg)
    dx0, dw0, db0 = cc.cconv_bwd(xg, dyg, wg, bg)
    y = torch.empty_like(y0)
    dx, dw, db = torch.empty_like(dx0), torch.empty_like(dw0), torch.empty_like(db0)
    ws = torch.empty(cc.cconv_bwd_workspace_bytes(B, T, D, W), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            cc.cconv_fwd(xg, wg, bg, y=y)
            cc.cconv_bwd(xg, dyg, wg, bg, dx=dx, dw=dw, dbias=db, workspace=ws)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(bits(y), bits(y0))
    assert np.array_equal(bits(dx), bits(dx0))
    assert torch.equal(dw, dw0) and torch.equal(db, db0)


def test_gpu_side_argument_errors():
    B, T, D, W = 1, 64, 256, 4
    x = torch.zeros(B, T, D + 8, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(D, W, device="cuda")
    with pytest.raises(cc.CConvError) as e:
        cc.cconv_fwd(x[:, :, 1:D + 1], w)  # base not 16-byte aligned
    assert e.value.status == -4
    dy = torch.zeros(B, T, D, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cc.CConvError) as e:
        cc.cconv_bwd(dy, dy, w, workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == -7


def test_no_device_fault_recorded():
    assert cc.cconv_device_fault() == 0


@pytest.mark.parametrize("scale", [1e-4, 30.0, 1e3], ids=["tiny", "saturating", "huge"])
def test_extreme_magnitudes(scale):
    """x scaled far from N(0,1): tiny values, values where tanh saturates (|z| >> 1, the
    SiLU's linear and zero sides), and huge ones; all within the forward / backward
    tolerances of the oracle."""
    B, T, D, W = 2, 300, 520, 4
    x, dy, w, b = inputs.fwd_bwd_inputs(B, T, D, W, True, seed=95)
    x = (x.float() * scale).to(torch.bfloat16)
    y, dx, dw, db = _run(x, dy, w, b, want_dbias=True)
    assert torch.isfinite(y.float()).all() and torch.isfinite(dx.float()).all()
    _check(x, dy, w, b, y, dx, dw, db, f"scale {scale}")
