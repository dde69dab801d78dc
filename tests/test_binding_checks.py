"""The Python binding refuses every tensor whose shape, dtype, layout or device disagrees
with the call, before anything is enqueued.

The C ABI sees pointers and sizes only and the kernels size every access from x's
[B, T, D], the pool's S and the number of sequences, so a mismatched tensor that reached a
kernel would be read or written past its end.  Each case below builds a small, otherwise
valid call with one tensor wrong.

- On the CPU (no GPU needed) the shape / dtype / layout checks run before the device
  check, so every case raises the same way with CPU tensors, and the valid calls get as
  far as the device check ("must be a CUDA tensor").
- On the GPU every case raises, and every output tensor passed in keeps its contents bit
  for bit (nothing ran).
"""
import pytest
import torch

import depthwise_causal_short_gb300 as cc

B, T, D, W = 2, 16, 64, 4
N, S = 4, 8
LENS = [5, 0, 11]
NSEQ = len(LENS)
TOTAL = sum(LENS)


def _t(dev, *shape, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(sum(shape) + 7)
    return torch.randn(*shape, generator=g).to(dtype).to(dev)


def _base(dev):
    """Tensors of a valid call of every kind."""
    z = {}
    z["x"], z["dy"] = _t(dev, B, T, D), _t(dev, B, T, D)
    z["w"], z["b"] = _t(dev, D, W, dtype=torch.float32), _t(dev, D, dtype=torch.float32)
    z["y"], z["dx"] = _t(dev, B, T, D), _t(dev, B, T, D)
    z["dw"], z["db"] = _t(dev, D, W, dtype=torch.float32), _t(dev, D, dtype=torch.float32)
    z["xd"], z["yd"] = _t(dev, N, D), _t(dev, N, D)
    z["state"] = _t(dev, S, D, W - 1)
    z["idx"] = torch.tensor([3, 0, 5, 1], dtype=torch.int32, device=dev)
    z["status"] = torch.zeros(2, dtype=torch.int32, device=dev)
    z["pos"] = torch.tensor([0, 1, 2, 7], dtype=torch.int32, device=dev)
    z["xv"], z["dyv"] = _t(dev, TOTAL, D), _t(dev, TOTAL, D)
    z["yv"], z["dxv"] = _t(dev, TOTAL, D), _t(dev, TOTAL, D)
    cu = [0]
    for n in LENS:
        cu.append(cu[-1] + n)
    z["cu"] = torch.tensor(cu, dtype=torch.int32, device=dev)
    z["init"], z["fin"] = _t(dev, NSEQ, D, W - 1), _t(dev, NSEQ, D, W - 1)
    z["dinit"] = _t(dev, NSEQ, D, W - 1)
    z["ws"] = torch.empty(1 << 20, dtype=torch.uint8, device=dev)
    z["qx"] = [_t(dev, B, T, d) for d in (64, 64, 128)]
    z["qdy"] = [_t(dev, B, T, d) for d in (64, 64, 128)]
    z["qw"] = [_t(dev, d, W, dtype=torch.float32) for d in (64, 64, 128)]
    z["qy"] = [_t(dev, B, T, d) for d in (64, 64, 128)]
    z["qdx"] = [_t(dev, B, T, d) for d in (64, 64, 128)]
    z["qdw"] = [_t(dev, d, W, dtype=torch.float32) for d in (64, 64, 128)]
    return z


def _fwd(z, **o):
    a = dict(x=z["x"], w=z["w"], bias=z["b"], y=z["y"]) | o
    return cc.cconv_fwd(a.pop("x"), a.pop("w"), a.pop("bias"), **a), ("y",)


def _bwd(z, **o):
    a = dict(x=z["x"], dy=z["dy"], w=z["w"], bias=z["b"], dx=z["dx"], dw=z["dw"], dbias=z["db"],
             workspace=z["ws"]) | o
    return cc.cconv_bwd(a.pop("x"), a.pop("dy"), a.pop("w"), a.pop("bias"), **a)


def _noalloc(z, **o):
    a = dict(x=z["x"], dy=z["dy"], w=z["w"], bias=z["b"], dx=z["dx"], dw=z["dw"],
             dbias=z["db"]) | o
    return cc.cconv_bwd_noalloc(a.pop("x"), a.pop("dy"), a.pop("w"), a.pop("bias"), **a)


def _upd(z, **o):
    a = dict(x=z["xd"], state=z["state"], w=z["w"], bias=z["b"], state_indices=z["idx"],
             y=z["yd"], status=z["status"]) | o
    return cc.cconv_update(a.pop("x"), a.pop("state"), a.pop("w"), a.pop("bias"),
                           a.pop("state_indices"), **a)


def _updx(z, **o):
    a = dict(x=z["xd"], state=z["state"], w=z["w"], bias=z["b"], state_indices=z["idx"],
             cache_seqlens=None, y=z["yd"], status=z["status"]) | o
    return cc.cconv_update_ex(a.pop("x"), a.pop("state"), a.pop("w"), a.pop("bias"),
                              a.pop("state_indices"), **a)


def _fwdv(z, **o):
    a = dict(x=z["xv"], cu=z["cu"], w=z["w"], bias=z["b"], initial_state=z["init"],
             final_state=z["fin"], y=z["yv"]) | o
    return cc.cconv_fwd_varlen(a.pop("x"), a.pop("cu"), a.pop("w"), a.pop("bias"), **a)


def _bwdv(z, **o):
    a = dict(x=z["xv"], dy=z["dyv"], cu=z["cu"], w=z["w"], bias=z["b"], initial_state=z["init"],
             dx=z["dxv"], dw=z["dw"], dbias=z["db"], d_initial_state=z["dinit"],
             workspace=z["ws"]) | o
    return cc.cconv_bwd_varlen(a.pop("x"), a.pop("dy"), a.pop("cu"), a.pop("w"), a.pop("bias"),
                               **a)


def _fwdm(z, **o):
    a = dict(xs=z["qx"], ws=z["qw"], ys=z["qy"]) | o
    return cc.cconv_fwd_multi(a.pop("xs"), a.pop("ws"), **a)


def _bwdm(z, **o):
    a = dict(xs=z["qx"], dys=z["qdy"], ws=z["qw"], dxs=z["qdx"], dws=z["qdw"],
             workspace=z["ws"]) | o
    return cc.cconv_bwd_multi(a.pop("xs"), a.pop("dys"), a.pop("ws"), **a)


def _auto(z, **o):
    a = dict(x=z["x"], weight=z["w"]) | o
    return cc.causal_conv1d(a.pop("x"), a.pop("weight"), **a)


def _noncontig(t):
    """Same shape and values, not contiguous."""
    big = torch.empty(*t.shape[:-1], 2 * t.shape[-1], dtype=t.dtype, device=t.device)
    big[..., ::2] = t
    return big[..., ::2]


def _strided_rows(t):
    """Same shape and values, contiguous channels, rows padded (allowed for inputs)."""
    big = torch.zeros(*t.shape[:-1], t.shape[-1] + 8, dtype=t.dtype, device=t.device)
    big[..., : t.shape[-1]] = t
    return big[..., : t.shape[-1]]


V, Ty = ValueError, TypeError
# (name, call, overrides(z) -> dict, exception)
CASES = [
    ("fwd x fp32", _fwd, lambda z: dict(x=z["x"].float()), Ty),
    ("fwd x 2-D", _fwd, lambda z: dict(x=z["x"][0]), V),
    ("fwd x channel stride 2", _fwd, lambda z: dict(x=_noncontig(z["x"])), V),
    ("fwd w wrong D", _fwd, lambda z: dict(w=z["w"][: D - 8]), V),
    ("fwd w W=5", _fwd, lambda z: dict(w=torch.cat([z["w"], z["w"][:, :1]], 1)), V),
    ("fwd w not contiguous", _fwd, lambda z: dict(w=z["w"].t().contiguous().t()), V),
    ("fwd w fp16", _fwd, lambda z: dict(w=z["w"].half(), bias=None), Ty),
    ("fwd bias wrong D", _fwd, lambda z: dict(bias=z["b"][:-8]), V),
    ("fwd bias dtype", _fwd, lambda z: dict(bias=z["b"].bfloat16()), Ty),
    ("fwd y shape", _fwd, lambda z: dict(y=z["y"][:, :-1]), V),
    ("fwd y not contiguous", _fwd, lambda z: dict(y=_strided_rows(z["y"])), V),
    ("fwd y fp32", _fwd, lambda z: dict(y=z["y"].float()), Ty),
    ("fwd y is x", _fwd, lambda z: dict(y=z["x"]), V),
    ("bwd dy shorter", _bwd, lambda z: dict(dy=z["dy"][:, :-1]), V),
    ("bwd dy narrower", _bwd, lambda z: dict(dy=z["dy"][..., :-8]), V),
    ("bwd dy fp32", _bwd, lambda z: dict(dy=z["dy"].float()), Ty),
    ("bwd dx shape", _bwd, lambda z: dict(dx=z["dx"][:1]), V),
    ("bwd dx not contiguous", _bwd, lambda z: dict(dx=_strided_rows(z["dx"])), V),
    ("bwd dx overlaps dy", _bwd, lambda z: dict(dx=z["dy"]), V),
    ("bwd dw shape", _bwd, lambda z: dict(dw=z["dw"][:, :3]), V),
    ("bwd dw dtype", _bwd, lambda z: dict(dw=z["dw"].bfloat16()), Ty),
    ("bwd dbias shape", _bwd, lambda z: dict(dbias=z["db"][:-1]), V),
    ("bwd w wrong D", _bwd, lambda z: dict(w=z["w"][:32], dw=z["dw"][:32]), V),
    ("bwd workspace not contiguous", _bwd, lambda z: dict(workspace=z["ws"][::2]), V),
    ("noalloc dx shape", _noalloc, lambda z: dict(dx=z["dx"][:, :8]), V),
    ("noalloc dy shorter", _noalloc, lambda z: dict(dy=z["dy"][:, :8]), V),
    ("noalloc dw shape", _noalloc, lambda z: dict(dw=z["dw"][:8]), V),
    ("update state W-2 entries", _upd, lambda z: dict(state=z["state"][..., :2].contiguous()), V),
    ("update state wrong D", _upd, lambda z: dict(state=z["state"][:, :32].contiguous()), V),
    ("update state not contiguous", _upd, lambda z: dict(state=z["state"][::2]), V),
    ("update state fp32", _upd, lambda z: dict(state=z["state"].float()), Ty),
    ("update indices too long", _upd,
     lambda z: dict(state_indices=torch.cat([z["idx"], z["idx"][:1]])), V),
    ("update indices int64", _upd, lambda z: dict(state_indices=z["idx"].long()), Ty),
    ("update y shape", _upd, lambda z: dict(y=z["yd"][:2]), V),
    ("update status int64", _upd, lambda z: dict(status=z["status"].long()), V),
    ("update status one word", _upd, lambda z: dict(status=z["status"][:1]), V),
    ("update S < N without indices", _upd,
     lambda z: dict(state=z["state"][:2].contiguous(), state_indices=None), V),
    ("update w wrong D", _upd, lambda z: dict(w=z["w"][:32]), V),
    ("update_ex state L = W+1", _updx,
     lambda z: dict(state=torch.cat([z["state"], z["state"][..., :2]], 2)), V),
    ("update_ex positions too short", _updx, lambda z: dict(cache_seqlens=z["pos"][:3]), V),
    ("update_ex positions int64", _updx, lambda z: dict(cache_seqlens=z["pos"].long()), Ty),
    ("fwd_varlen cu int64", _fwdv, lambda z: dict(cu=z["cu"].long()), Ty),
    ("fwd_varlen cu one entry", _fwdv, lambda z: dict(cu=z["cu"][:1]), V),
    ("fwd_varlen initial W-2 entries", _fwdv,
     lambda z: dict(initial_state=z["init"][..., :2].contiguous()), V),
    ("fwd_varlen final wrong D", _fwdv, lambda z: dict(final_state=z["fin"][:, :32].contiguous()), V),
    ("fwd_varlen states too few", _fwdv,
     lambda z: dict(initial_state=z["init"][:2].contiguous(), final_state=None), V),
    ("fwd_varlen indices too short", _fwdv,
     lambda z: dict(state_indices=z["idx"][:2], status=z["status"]), V),
    ("fwd_varlen y shape", _fwdv, lambda z: dict(y=z["yv"][:-1]), V),
    ("fwd_varlen x 3-D", _fwdv, lambda z: dict(x=z["xv"][None]), V),
    ("bwd_varlen dy shorter", _bwdv, lambda z: dict(dy=z["dyv"][:-1]), V),
    ("bwd_varlen initial one too many", _bwdv,
     lambda z: dict(initial_state=torch.cat([z["init"], z["init"][:1]])), V),
    ("bwd_varlen d_initial wrong entries", _bwdv,
     lambda z: dict(d_initial_state=z["dinit"][..., :2].contiguous()), V),
    ("bwd_varlen dx shape", _bwdv, lambda z: dict(dx=z["dxv"][:, :32]), V),
    ("multi fwd weight count", _fwdm, lambda z: dict(ws=z["qw"][:2]), V),
    ("multi fwd weight wrong D", _fwdm, lambda z: dict(ws=[z["qw"][0], z["qw"][2], z["qw"][2]]), V),
    ("multi fwd W differs", _fwdm,
     lambda z: dict(ws=[z["qw"][0], z["qw"][1][:, :3].contiguous(), z["qw"][2]]), V),
    ("multi fwd y shape", _fwdm, lambda z: dict(ys=[z["qy"][0][:1], z["qy"][1], z["qy"][2]]), V),
    ("multi fwd T differs", _fwdm, lambda z: dict(xs=[z["qx"][0], z["qx"][1][:, :8], z["qx"][2]]), V),
    ("multi bwd dy shape", _bwdm,
     lambda z: dict(dys=[z["qdy"][0], z["qdy"][1][..., :32], z["qdy"][2]]), V),
    ("multi bwd dw shape", _bwdm, lambda z: dict(dws=[z["qdw"][0][:8], z["qdw"][1], z["qdw"][2]]), V),
    ("autograd x 2-D", _auto, lambda z: dict(x=z["x"][0]), V),
    ("autograd initial state count", _auto,
     lambda z: dict(initial_state=z["init"][:1].contiguous()), V),
]
IDS = [c[0] for c in CASES]


def _outputs(z):
    return [t for k, t in z.items() if k in ("y", "dx", "dw", "db", "yd", "state", "status",
                                            "yv", "dxv", "fin", "dinit")] + z["qy"] + z["qdx"] + \
        z["qdw"]


@pytest.mark.parametrize("name,call,over,exc", CASES, ids=IDS)
def test_mismatch_raises_on_cpu(name, call, over, exc):
    z = _base("cpu")
    with pytest.raises(exc):
        call(z, **over(z))


@pytest.mark.parametrize("call", [_fwd, _bwd, _noalloc, _upd, _updx, _fwdv, _bwdv, _fwdm, _bwdm],
                         ids=lambda f: f.__name__)
def test_valid_calls_reach_the_device_check(call):
    z = _base("cpu")
    with pytest.raises(ValueError, match="CUDA tensor"):
        call(z)


@pytest.mark.gpu
@pytest.mark.parametrize("name,call,over,exc", CASES, ids=IDS)
def test_mismatch_raises_before_launch(name, call, over, exc):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    z = _base("cuda")
    o = over(z)
    outs = _outputs(z) + [t for t in o.values() if isinstance(t, torch.Tensor)]
    before = [t.detach().clone() for t in outs]
    torch.cuda.synchronize()
    with pytest.raises(exc):
        call(z, **o)
    torch.cuda.synchronize()
    for a, b in zip(outs, before):
        assert torch.equal(a.view(torch.uint8) if a.dtype == torch.bool else a, b)


@pytest.mark.gpu
def test_valid_calls_run():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    z = _base("cuda")
    for call in (_fwd, _bwd, _noalloc, _upd, _updx, _fwdv, _bwdv, _fwdm, _bwdm):
        call(z)
    torch.cuda.synchronize()
    assert z["status"].tolist() == [0, 0]
    assert cc.cconv_device_fault() == 0


@pytest.mark.gpu
def test_tensors_on_another_device_are_refused():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    z = _base("cuda")
    with pytest.raises(ValueError, match="CUDA tensor"):
        cc.cconv_fwd(z["x"], z["w"].cpu(), z["b"], y=z["y"])
    with pytest.raises(ValueError, match="CUDA tensor"):
        cc.cconv_update(z["xd"], z["state"], z["w"], z["b"], z["idx"].cpu(), y=z["yd"],
                        status=z["status"])
