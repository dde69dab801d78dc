"""causal_conv1d (the differentiable entry point) against the direct calls (GPU).

Its forward and the gradients autograd produces must equal, bit for bit, what the library
calls it dispatches to return: the batched pair for the plain case, the packed-sequence
pair with initial / final states, no activation, or cu_seqlens.
"""
import pytest
import torch

import depthwise_causal_short_gb300 as cc
from depthwise_causal_short_gb300 import _build, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    return cc.load()


def _same(a, b):
    if a.dtype == torch.bfloat16:
        return torch.equal(a.view(torch.int16), b.view(torch.int16))
    return torch.equal(a, b)


@pytest.mark.parametrize("wdtype", [torch.float32, torch.bfloat16], ids=["w_f32", "w_bf16"])
def test_batched(wdtype):
    x, dy, w, b = inputs.fwd_bwd_inputs(2, 700, 1000 - 1000 % 8, 4, True, wdtype=wdtype, seed=100)
    xg = x.cuda().requires_grad_(True)
    wg = w.cuda().requires_grad_(True)
    bg = b.cuda().requires_grad_(True)
    y, fin = cc.causal_conv1d(xg, wg, bg)
    assert fin is None
    y.backward(dy.cuda())
    y0 = cc.cconv_fwd(x.cuda(), w.cuda(), b.cuda())
    dx0, dw0, db0 = cc.cconv_bwd(x.cuda(), dy.cuda(), w.cuda(), b.cuda(), want_dbias=True)
    torch.cuda.synchronize()
    assert _same(y.detach(), y0)
    assert _same(xg.grad, dx0) and _same(wg.grad, dw0) and _same(bg.grad, db0)


@pytest.mark.parametrize("act", ["silu", None], ids=["silu", "none"])
def test_packed_with_states(act):
    lens = [300, 0, 2, 457, 31]
    x, dy, cu, w, b, init = inputs.varlen_inputs(lens, 512, 4, bias=True, seed=101)
    D = x.shape[1]
    xg = x.cuda().view(1, -1, D).requires_grad_(True)
    wg = w.cuda().requires_grad_(True)
    bg = b.cuda().requires_grad_(True)
    ig = init.cuda().requires_grad_(True)
    y, fin = cc.causal_conv1d(xg, wg, bg, initial_state=ig, output_final_state=True,
                              activation=act, cu_seqlens=cu.cuda())
    assert not fin.requires_grad
    y.backward(dy.cuda().view(1, -1, D))
    y0, fin0, _ = cc.cconv_fwd_varlen(x.cuda(), cu.cuda(), w.cuda(), b.cuda(), activation=act,
                                      initial_state=init.cuda(), final_state=True)
    dx0, dw0, db0, di0 = cc.cconv_bwd_varlen(x.cuda(), dy.cuda(), cu.cuda(), w.cuda(), b.cuda(),
                                             activation=act, initial_state=init.cuda(),
                                             want_dbias=True)
    torch.cuda.synchronize()
    assert _same(y.detach().view(-1, D), y0) and _same(fin, fin0)
    assert _same(xg.grad.view(-1, D), dx0) and _same(wg.grad, dw0) and _same(bg.grad, db0)
    assert _same(ig.grad, di0)


def test_batch_rows_with_initial_states_and_only_x_grad():
    """No cu_seqlens but initial states: each batch row is one sequence; only x needs a
    gradient."""
    B, T, D, W = 3, 200, 256, 4
    x, dy, w, b = inputs.fwd_bwd_inputs(B, T, D, W, False, seed=102)
    g = torch.Generator().manual_seed(103)
    init = torch.randn(B, D, W - 1, generator=g).to(torch.bfloat16).cuda()
    xg = x.cuda().requires_grad_(True)
    y, _ = cc.causal_conv1d(xg, w.cuda(), None, initial_state=init)
    y.backward(dy.cuda())
    cu = torch.arange(0, (B + 1) * T, T, dtype=torch.int32, device="cuda")
    y0, _, _ = cc.cconv_fwd_varlen(x.cuda().view(-1, D), cu, w.cuda(), None, initial_state=init)
    dx0, _, _, _ = cc.cconv_bwd_varlen(x.cuda().view(-1, D), dy.cuda().view(-1, D), cu, w.cuda(),
                                       None, initial_state=init)
    torch.cuda.synchronize()
    assert _same(y.detach().view(-1, D), y0) and _same(xg.grad.view(-1, D), dx0)


def test_first_call_on_a_fresh_thread():
    """A thread whose first CUDA work is a library call (as autograd's device thread can
    be) has no context current yet; the calls must bind one, not fail."""
    import threading

    x, dy, w, b = inputs.fwd_bwd_inputs(2, 300, 512, 4, True, seed=104)
    xg, dyg, wg, bg = x.cuda(), dy.cuda(), w.cuda(), b.cuda()
    y0 = cc.cconv_fwd(xg, wg, bg)
    ref = cc.cconv_bwd(xg, dyg, wg, bg, want_dbias=True)
    outs = {}
    for name in ("fwd", "bwd"):
        y1 = torch.empty_like(y0)
        dx1, dw1, db1 = torch.empty_like(ref[0]), torch.empty_like(ref[1]), torch.empty_like(ref[2])
        ws = torch.empty(cc.cconv_bwd_workspace_bytes(2, 300, 512, 4), dtype=torch.uint8,
                         device="cuda")
        torch.cuda.synchronize()
        err = []

        def run():
            try:
                if name == "fwd":
                    cc.cconv_fwd(xg, wg, bg, y=y1)
                else:
                    cc.cconv_bwd(xg, dyg, wg, bg, dx=dx1, dw=dw1, dbias=db1, workspace=ws)
                torch.cuda.synchronize()
            except Exception as e:  # reported to the main thread
                err.append(e)

        t = threading.Thread(target=run)
        t.start()
        t.join()
        assert not err, err
        outs[name] = (y1,) if name == "fwd" else (dx1, dw1, db1)
    assert _same(outs["fwd"][0], y0)
    for u, v in zip(outs["bwd"], ref):
        assert _same(u, v)
