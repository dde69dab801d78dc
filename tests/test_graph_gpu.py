"""CUDA-graph capture of the newer entry points (GPU).

Every call enqueues on the caller's stream with no host synchronisation and allocates
nothing, so it can be captured.  One graph holds: a packed-sequence forward writing final
states from the stream kernel, another into a decode pool in place through state indices
(second kernel), the packed-sequence backward, a decode update with the variants, and the
q/k/v forward and backward in one launch each.  Its replay must equal eager execution bit
for bit.
"""
import numpy as np
import pytest
import torch

import depthwise_causal_short_gb300 as cc
from depthwise_causal_short_gb300 import _build, inputs
from tests.helpers import bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    return cc.load()


def _work(dev):
    D, W = 512, 4
    lens = [300, 0, 2, 457, 31]
    x, dy, cu, w, b, init = inputs.varlen_inputs(lens, D, W, bias=True, seed=70)
    g = torch.Generator().manual_seed(71)
    pool = torch.randn(40, D, W - 1, generator=g).to(torch.bfloat16)
    idx = torch.randperm(40, generator=g)[:len(lens)].to(torch.int32)
    dpool = torch.randn(64, D, W, generator=g).to(torch.bfloat16)
    xd = torch.randn(20, D, generator=g).to(torch.bfloat16)
    didx = torch.randperm(64, generator=g)[:20].to(torch.int32)
    didx[3] = -1
    qkv = [inputs.fwd_bwd_inputs(2, 300, d, W, True, seed=72 + k)
           for k, d in enumerate((256, 256, 512))]
    t = dict(x=x, dy=dy, cu=cu, w=w, b=b, init=init, pool=pool, idx=idx, dpool=dpool, xd=xd,
             didx=didx)
    out = {k: v.to(dev) for k, v in t.items()}
    out["qkv"] = [tuple(u.to(dev) for u in p) for p in qkv]
    return out


def _outputs(t):
    D, W = t["w"].shape
    n = t["cu"].numel() - 1
    o = dict(
        y=torch.empty_like(t["x"]), fin=torch.empty(n, D, W - 1, dtype=torch.bfloat16,
                                                    device=t["x"].device),
        y2=torch.empty_like(t["x"]), status=torch.empty(2, dtype=torch.int32, device=t["x"].device),
        dx=torch.empty_like(t["x"]), dw=torch.empty_like(t["w"]), db=torch.empty_like(t["b"]),
        di=torch.empty_like(t["init"]),
        ws=torch.empty(cc.cconv_bwd_varlen_workspace_bytes(t["x"].shape[0], D, W),
                       dtype=torch.uint8, device=t["x"].device),
        yd=torch.zeros(t["xd"].shape, dtype=torch.bfloat16, device=t["x"].device),
        dstatus=torch.empty(2, dtype=torch.int32, device=t["x"].device),
        qy=[torch.empty_like(p[0]) for p in t["qkv"]],
        qdx=[torch.empty_like(p[0]) for p in t["qkv"]],
        qdw=[torch.empty_like(p[2]) for p in t["qkv"]],
        qdb=[torch.empty_like(p[3]) for p in t["qkv"]],
        qws=torch.empty(cc.cconv_bwd_multi_workspace_bytes([p[0].shape[2] for p in t["qkv"]], 2,
                                                           300, W),
                        dtype=torch.uint8, device=t["x"].device),
    )
    return o


def _calls(t, o, stream):
    cc.cconv_fwd_varlen(t["x"], t["cu"], t["w"], t["b"], initial_state=t["init"],
                        final_state=o["fin"], y=o["y"], stream=stream)
    cc.cconv_fwd_varlen(t["x"], t["cu"], t["w"], t["b"], initial_state=t["pool"],
                        final_state=t["pool"], state_indices=t["idx"], status=o["status"],
                        y=o["y2"], stream=stream)
    cc.cconv_bwd_varlen(t["x"], t["dy"], t["cu"], t["w"], t["b"], initial_state=t["init"],
                        want_dbias=True, dx=o["dx"], dw=o["dw"], dbias=o["db"],
                        d_initial_state=o["di"], workspace=o["ws"], stream=stream)
    cc.cconv_update_ex(t["xd"], t["dpool"], t["w"], t["b"], t["didx"], pad_rows=True,
                       activation=None, y=o["yd"], status=o["dstatus"], stream=stream)
    xs = [p[0] for p in t["qkv"]]
    cc.cconv_fwd_multi(xs, [p[2] for p in t["qkv"]], [p[3] for p in t["qkv"]], ys=o["qy"],
                       stream=stream)
    cc.cconv_bwd_multi(xs, [p[1] for p in t["qkv"]], [p[2] for p in t["qkv"]],
                       [p[3] for p in t["qkv"]], want_dbias=True, dxs=o["qdx"], dws=o["qdw"],
                       dbiases=o["qdb"], workspace=o["qws"], stream=stream)


def _snapshot(t, o):
    out = {}
    for k, v in o.items():
        if k in ("ws", "qws"):
            continue
        vs = v if isinstance(v, list) else [v]
        out[k] = [u.detach().cpu().clone() for u in vs]
    out["pool"] = [t["pool"].cpu().clone()]
    out["dpool"] = [t["dpool"].cpu().clone()]
    return out


def test_graph_replay_equals_eager():
    dev = torch.device("cuda", 0)
    eager_t = _work(dev)
    eager_o = _outputs(eager_t)
    _calls(eager_t, eager_o, torch.cuda.current_stream())
    torch.cuda.synchronize()
    want = _snapshot(eager_t, eager_o)
    assert want["status"][0].tolist() == [0, 0] and want["dstatus"][0].tolist() == [0, 0]

    t = _work(dev)
    o = _outputs(t)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            _calls(t, o, s)
    torch.cuda.synchronize()
    # capture ran nothing: restore the mutable pools, then replay once
    fresh = _work(dev)
    t["pool"].copy_(fresh["pool"])
    t["dpool"].copy_(fresh["dpool"])
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    got = _snapshot(t, o)
    for k, vs in want.items():
        for a, c in zip(vs, got[k]):
            if a.dtype == torch.bfloat16:
                assert np.array_equal(bits(a), bits(c)), k
            else:
                assert torch.equal(a, c), k
