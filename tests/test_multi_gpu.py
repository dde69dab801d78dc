"""Several convolutions in one launch (the q, k, v short convolutions of a layer) (GPU).

cconv_fwd_multi / cconv_bwd_multi through the C ABI against the fp64 oracle, problem by
problem, and against separate single-problem calls: y and dx must be bit-identical to them
(each row's arithmetic does not depend on how rows are split among CTAs), dw and dbias
within the backward tolerance.  Covers the KDA layout (D, D, 2D), ragged widths per
problem, strided inputs, bf16 weights, problems with and without bias, n = 1 and n = 4.
"""
import pytest
import torch

import depthwise_causal_short_gb300 as cc
from depthwise_causal_short_gb300 import _build, inputs
from tests.helpers import BWD_TOL, FWD_TOL, f64, oracle_bwd, oracle_fwd, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    return cc.load()


def _problems(B, T, Ds, W, biases, wdtype, seed):
    out = []
    for k, (D, hb) in enumerate(zip(Ds, biases)):
        out.append(inputs.fwd_bwd_inputs(B, T, D, W, hb, wdtype=wdtype, seed=seed + k))
    return out


def _run_and_check(B, T, Ds, W, biases, wdtype=torch.float32, seed=0, strided=False):
    probs = _problems(B, T, Ds, W, biases, wdtype, seed)
    xs, dys = [], []
    for x, dy, _, _ in probs:
        if strided:  # rows of a wider buffer, as slices of a fused projection output
            big = torch.zeros(B, T, x.shape[2] + 64, dtype=torch.bfloat16)
            big[:, :, 32:32 + x.shape[2]] = x
            xs.append(big.cuda()[:, :, 32:32 + x.shape[2]])
        else:
            xs.append(x.cuda())
        dys.append(dy.cuda())
    wg = [w.cuda() for _, _, w, _ in probs]
    bg = [None if b is None else b.cuda() for _, _, _, b in probs]
    ys = cc.cconv_fwd_multi(xs, wg, bg)
    dxs, dws, dbs = cc.cconv_bwd_multi(xs, dys, wg, bg, want_dbias=True)
    torch.cuda.synchronize()
    for k, (x, dy, w, b) in enumerate(probs):
        y1 = cc.cconv_fwd(xs[k], wg[k], bg[k])
        dx1, _, _ = cc.cconv_bwd(xs[k], dys[k], wg[k], bg[k])
        torch.cuda.synchronize()
        assert torch.equal(ys[k].view(torch.int16), y1.view(torch.int16)), f"problem {k}: y"
        assert torch.equal(dxs[k].view(torch.int16), dx1.view(torch.int16)), f"problem {k}: dx"
        e = rel_err(f64(ys[k]), oracle_fwd(x, w, b))
        assert e <= FWD_TOL, f"problem {k}: y err {e:.2e}"
        rdx, rdw, rdb = oracle_bwd(x, dy, w, b, want_dbias=True)
        for name, g, r in (("dx", dxs[k], rdx), ("dw", dws[k], rdw), ("dbias", dbs[k], rdb)):
            e = rel_err(f64(g), r)
            assert e <= BWD_TOL, f"problem {k}: {name} err {e:.2e}"


def test_kda_qkv_layout():
    """q, k at D = 8 heads x 128, v at twice that."""
    _run_and_check(2, 2048, [1024, 1024, 2048], 4, [False, False, False])


@pytest.mark.parametrize("wdtype", [torch.float32, torch.bfloat16], ids=["w_f32", "w_bf16"])
def test_ragged_widths(wdtype):
    _run_and_check(3, 777, [1000, 264, 2056], 3, [True, False, True], wdtype=wdtype, seed=10)


def test_strided_inputs():
    _run_and_check(2, 300, [512, 512, 1024], 4, [True, True, True], seed=20, strided=True)


@pytest.mark.parametrize("Ds", [[4096], [128, 256, 384, 1024]], ids=["n1", "n4"])
def test_problem_counts(Ds):
    _run_and_check(1, 1500, Ds, 4, [True] * len(Ds), seed=30)


def test_short_rows():
    _run_and_check(2, 3, [64, 8, 72], 2, [True, True, False], seed=40)


def test_backward_deterministic():
    B, T, W = 2, 1000, 4
    Ds = [512, 512, 1024]
    probs = [inputs.fwd_bwd_inputs(B, T, D, W, True, seed=60 + k) for k, D in enumerate(Ds)]
    xs = [p[0].cuda() for p in probs]
    dys = [p[1].cuda() for p in probs]
    ws = [p[2].cuda() for p in probs]
    bs = [p[3].cuda() for p in probs]
    a = cc.cconv_bwd_multi(xs, dys, ws, bs, want_dbias=True)
    c = cc.cconv_bwd_multi(xs, dys, ws, bs, want_dbias=True)
    torch.cuda.synchronize()
    for u_list, v_list in zip(a, c):
        for u, v in zip(u_list, v_list):
            if u.dtype == torch.bfloat16:
                assert torch.equal(u.view(torch.int16), v.view(torch.int16))
            else:
                assert torch.equal(u, v)
