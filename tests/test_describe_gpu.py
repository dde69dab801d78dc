"""Launch descriptions (cconv_describe_begin / cconv_describe_end) on the GPU.

While recording, a call runs its host checks and planning and reports the kernels it would
launch, with their resources, and nothing runs: outputs keep their contents.  The backward
at the production shape is a one-wave lockstep stream kernel (one CTA per SM) plus its
reduction; below 512 channels an independent-pipeline stream kernel plus the reduction.
"""
import pytest
import torch

import depthwise_causal_short_gb300 as cc
from depthwise_causal_short_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda", 0)


def test_backward_description(dev):
    B, T, D, W = 2, 8192, 4096, 4
    x, dy, w, _ = inputs.fwd_bwd_inputs(B, T, D, W, False)
    x, dy, w = x.to(dev), dy.to(dev), w.to(dev)
    dx = torch.full_like(x, 7.0)
    dw = torch.full_like(w, 7.0)
    ks = cc.describe(lambda: cc.cconv_bwd(x, dy, w, dx=dx, dw=dw))
    torch.cuda.synchronize()
    assert [k["name"].split("(")[0].split("<")[0].split("::")[-1] for k in ks] == [
        "cconv_bwd_ls_kernel", "cconv_bwd_reduce1_kernel"]
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    stream = ks[0]
    assert stream["ctas"] <= sms and stream["ctas"] >= sms - 8
    assert stream["ctas_per_sm"] >= 1 and stream["threads"] == 288
    assert stream["registers"] > 0 and stream["local_bytes"] == 0
    assert stream["dynamic_shared_bytes"] > 100_000
    assert (dx == 7.0).all() and (dw == 7.0).all(), "a recorded call must not run"


def test_every_call_describes(dev):
    B, T, D, W = 2, 300, 512, 4
    x, dy, w, b = (t.to(dev) for t in inputs.fwd_bwd_inputs(B, T, D, W, True))
    assert len(cc.describe(lambda: cc.cconv_fwd(x, w, b))) == 1
    st, xr, idx, wd, bd = (t.to(dev) for t in inputs.decode_inputs(16, 8, D, W, True, n_x=1))
    ks = cc.describe(lambda: cc.cconv_update(xr[0], st, wd, bd, idx))
    assert len(ks) == 1 and "cconv_update_kernel" in ks[0]["name"]
    lens = [100, 0, 250, 250]
    vx, vdy, cu, vw, vb, init = (t.to(dev) for t in inputs.varlen_inputs(lens, D, W, seed=2))
    assert len(cc.describe(lambda: cc.cconv_fwd_varlen(vx, cu, vw, vb, initial_state=init,
                                                       final_state=True))) == 1
    assert len(cc.describe(lambda: cc.cconv_bwd_varlen(vx, vdy, cu, vw, vb,
                                                       initial_state=init))) == 2
    narrow = [t[..., :256] for t in (x, dy)]
    ks = cc.describe(lambda: cc.cconv_bwd(*narrow, w[:256].contiguous()))
    assert [k["name"].split("(")[0].split("<")[0].split("::")[-1] for k in ks] == [
        "cconv_bwd_kernel", "cconv_bwd_reduce1_kernel"]
    xs = [x, x[..., :256]]
    ws = [w, w[:256].contiguous()]
    assert len(cc.describe(lambda: cc.cconv_fwd_multi(xs, ws))) == 1
    assert len(cc.describe(lambda: cc.cconv_bwd_multi(xs, [dy, dy[..., :256]], ws))) == 2
    # recording stops at the end: the next call runs
    y = cc.cconv_fwd(x, w, b)
    torch.cuda.synchronize()
    assert torch.isfinite(y.float()).all() and y.abs().sum() > 0
