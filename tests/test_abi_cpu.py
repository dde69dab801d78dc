"""The C ABI without a GPU: the library builds, loads, exports exactly the functions
include/cconv.h declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes

import pytest
import torch

import depthwise_causal_short_gb300 as cc
from depthwise_causal_short_gb300 import _build

BF16, F32 = 0, 1
OK, ENULL, ESHAPE, EWIDTH, EALIGN, ESTRIDE, EDTYPE = 0, -1, -2, -3, -4, -5, -6

P = 0x100000  # a fake, 16-byte aligned device address; never dereferenced by these tests


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return cc.load()


def test_exports_match_header(lib):
    declared = cc.header_functions()
    assert set(declared) == {"cconv_fwd", "cconv_bwd_workspace_bytes", "cconv_bwd",
                             "cconv_bwd_noalloc", "cconv_update", "cconv_status_str",
                             "cconv_device_fault", "cconv_fwd_varlen",
                             "cconv_bwd_varlen_workspace_bytes", "cconv_bwd_varlen",
                             "cconv_update_ex", "cconv_fwd_multi",
                             "cconv_bwd_multi_workspace_bytes", "cconv_bwd_multi",
                             "cconv_describe_begin", "cconv_describe_end"}
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in cconv.h but not exported"


def test_only_header_symbols_exported():
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", str(cc.lib_path())],
                         capture_output=True, text=True, check=True).stdout
    names = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert names == set(cc.header_functions())


def test_status_strings(lib):
    for code in range(-10, 1):
        s = cc.cconv_status_str(code)
        assert s.startswith(cc.binding.STATUS[code])
    assert "unknown" in cc.cconv_status_str(-99)


def _fwd(lib, x=P, B=2, T=16, D=64, sxb=16 * 64, sxt=64, w=P, bias=None, wdt=F32, W=4, y=P):
    return lib.cconv_fwd(x, B, T, D, sxb, sxt, w, bias, wdt, W, y, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(x=None), ENULL), (dict(w=None), ENULL), (dict(y=None), ENULL),
    (dict(W=0), EWIDTH), (dict(W=5), EWIDTH), (dict(wdt=7), EDTYPE),
    (dict(B=0), ESHAPE), (dict(T=0), ESHAPE), (dict(D=0), ESHAPE), (dict(T=1 << 31), ESHAPE),
    (dict(D=60, sxt=64), EALIGN), (dict(x=P + 2), EALIGN), (dict(y=P + 8), EALIGN),
    (dict(sxt=68), EALIGN), (dict(sxb=16 * 64 + 4), EALIGN),
    (dict(sxt=0), ESTRIDE), (dict(sxt=-64), ESTRIDE), (dict(sxb=0), ESTRIDE),
    (dict(w=P + 2, wdt=F32), EALIGN), (dict(bias=P + 1, wdt=BF16), EALIGN),
])
def test_fwd_rejects(lib, kw, expect):
    assert _fwd(lib, **kw) == expect


def _bwd(lib, x=P, dy=P, B=2, T=16, D=64, w=P, bias=None, wdt=F32, W=4, dx=P, dw=P,
         dbias=None, ws=P, wsb=1 << 30, sxb=16 * 64, sxt=64, sdb=16 * 64, sdt=64):
    return lib.cconv_bwd(x, sxb, sxt, dy, sdb, sdt, B, T, D, w, bias, wdt, W, dx, dw, dbias, ws,
                         wsb, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(x=None), ENULL), (dict(dy=None), ENULL), (dict(dx=None), ENULL), (dict(dw=None), ENULL),
    (dict(W=9), EWIDTH), (dict(wdt=2), EDTYPE), (dict(T=0), ESHAPE), (dict(D=12), EALIGN),
    (dict(dy=P + 4), EALIGN), (dict(dx=P + 2), EALIGN), (dict(sdt=-8), ESTRIDE),
    (dict(sdb=12), EALIGN), (dict(dbias=P + 2, wdt=F32), EALIGN),
])
def test_bwd_rejects(lib, kw, expect):
    assert _bwd(lib, **kw) == expect


def test_workspace_query_rejects(lib):
    n = ctypes.c_size_t(0)
    assert lib.cconv_bwd_workspace_bytes(1, 1, 8, 4, None) == ENULL
    assert lib.cconv_bwd_workspace_bytes(1, 0, 8, 4, ctypes.byref(n)) == ESHAPE
    assert lib.cconv_bwd_workspace_bytes(1, 1, 8, 0, ctypes.byref(n)) == EWIDTH


def _upd(lib, x=P, N=4, D=64, ldx=64, state=P, S=8, idx=P, w=P, bias=None, wdt=F32, W=4, y=P,
         status=P):
    return lib.cconv_update(x, N, D, ldx, state, S, idx, w, bias, wdt, W, y, status, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(x=None), ENULL), (dict(w=None), ENULL), (dict(y=None), ENULL),
    (dict(status=None), ENULL), (dict(state=None), ENULL), (dict(W=5), EWIDTH),
    (dict(wdt=3), EDTYPE), (dict(N=0), ESHAPE), (dict(D=0), ESHAPE), (dict(S=-1), ESHAPE),
    (dict(ldx=63), ESTRIDE), (dict(idx=None, S=3), ESHAPE),
    (dict(S=393217), ESHAPE), (dict(idx=P + 2), EALIGN), (dict(status=P + 2), EALIGN),
    (dict(x=P + 1), EALIGN), (dict(w=P + 2), EALIGN),
])
def test_update_rejects(lib, kw, expect):
    assert _upd(lib, **kw) == expect


def _fwdv(lib, x=P, total=64, D=64, sxt=64, cu=P, nseq=2, w=P, bias=None, wdt=F32, W=4, act=0,
          init=None, fin=None, idx=None, S=2, status=None, y=P):
    return lib.cconv_fwd_varlen(x, total, D, sxt, cu, nseq, w, bias, wdt, W, act, init, fin, idx,
                                S, status, y, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(cu=None), ENULL), (dict(w=None), ENULL), (dict(x=None), ENULL), (dict(y=None), ENULL),
    (dict(W=0), EWIDTH), (dict(wdt=5), EDTYPE), (dict(act=2), ESHAPE), (dict(nseq=0), ESHAPE),
    (dict(total=-1), ESHAPE), (dict(total=1 << 31), ESHAPE), (dict(D=0), ESHAPE),
    (dict(D=60, sxt=64), EALIGN), (dict(cu=P + 2), EALIGN), (dict(x=P + 2), EALIGN),
    (dict(y=P + 4), EALIGN), (dict(sxt=0), ESTRIDE), (dict(sxt=12), EALIGN),
    (dict(fin=P, S=1), ESHAPE), (dict(init=P + 8), EALIGN), (dict(fin=P + 2), EALIGN),
    (dict(idx=P), ENULL), (dict(idx=P, status=P, S=0), ESHAPE),
    (dict(idx=P, status=P, S=393217), ESHAPE), (dict(idx=P + 1, status=P), EALIGN),
])
def test_fwd_varlen_rejects(lib, kw, expect):
    assert _fwdv(lib, **kw) == expect


def _bwdv(lib, x=P, sxt=64, dy=P, sdt=64, total=64, D=64, cu=P, nseq=2, w=P, bias=None,
          wdt=F32, W=4, act=0, init=None, idx=None, S=2, status=None, dx=P, dw=P, dbias=None,
          dinit=None, ws=P, wsb=1 << 30):
    return lib.cconv_bwd_varlen(x, sxt, dy, sdt, total, D, cu, nseq, w, bias, wdt, W, act, init,
                                idx, S, status, dx, dw, dbias, dinit, ws, wsb, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(cu=None), ENULL), (dict(dw=None), ENULL), (dict(dy=None), ENULL),
    (dict(dx=None), ENULL), (dict(W=5), EWIDTH), (dict(wdt=9), EDTYPE), (dict(act=-1), ESHAPE),
    (dict(nseq=0), ESHAPE), (dict(D=20), EALIGN), (dict(sdt=-64), ESTRIDE),
    (dict(dx=P + 8), EALIGN), (dict(dinit=P + 1), EALIGN), (dict(cu=P + 1), EALIGN),
    (dict(init=P, idx=P), ENULL), (dict(init=P, idx=P, status=P, S=0), ESHAPE),
    (dict(init=P, idx=P, status=P, S=393217), ESHAPE), (dict(idx=P + 2, status=P), EALIGN),
    (dict(idx=P, status=P + 2), EALIGN),
])
def test_bwd_varlen_rejects(lib, kw, expect):
    assert _bwdv(lib, **kw) == expect


def _updx(lib, x=P, N=4, D=64, ldx=64, state=P, S=8, L=3, idx=P, pad=0, pos=None, w=P,
          bias=None, wdt=F32, W=4, act=0, y=P, status=P):
    return lib.cconv_update_ex(x, N, D, ldx, state, S, L, idx, pad, pos, w, bias, wdt, W, act, y,
                               status, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(L=2), ESHAPE), (dict(L=5), ESHAPE), (dict(W=2, L=3), ESHAPE), (dict(act=3), ESHAPE),
    (dict(status=None), ENULL), (dict(state=None), ENULL), (dict(W=1, L=1, state=None), ENULL),
    (dict(W=7, L=6), EWIDTH), (dict(ldx=60), ESTRIDE), (dict(x=None), ENULL),
    (dict(W=1, L=0, pos=P), ESHAPE), (dict(pos=P + 2), EALIGN),
])
def test_update_ex_rejects(lib, kw, expect):
    assert _updx(lib, **kw) == expect


def _arr(ctype, vals):
    return (ctype * len(vals))(*vals)


def _fwdm(lib, n=3, x=(P, P, P), D=(64, 64, 128), sxb=(16 * 64, 16 * 64, 16 * 128),
          sxt=(64, 64, 128), w=(P, P, P), bias=None, y=(P, P, P), B=2, T=16, wdt=F32, W=4):
    V, I = ctypes.c_void_p, ctypes.c_int64
    return lib.cconv_fwd_multi(n, _arr(V, x), _arr(I, D), _arr(I, sxb), _arr(I, sxt), _arr(V, w),
                               None if bias is None else _arr(V, bias), _arr(V, y), B, T, wdt, W,
                               None)


@pytest.mark.parametrize("kw,expect", [
    (dict(n=0), ESHAPE), (dict(n=5, x=(P,) * 5, D=(64,) * 5, sxb=(1024,) * 5, sxt=(64,) * 5,
                                 w=(P,) * 5, y=(P,) * 5), ESHAPE),
    (dict(x=(P, None, P)), ENULL), (dict(y=(P, P, None)), ENULL), (dict(W=5), EWIDTH),
    (dict(wdt=4), EDTYPE), (dict(T=0), ESHAPE), (dict(D=(64, 60, 128)), EALIGN),
    (dict(D=(64, 0, 128)), ESHAPE), (dict(y=(P, P + 8, P)), EALIGN), (dict(sxt=(64, 64, 0)), ESTRIDE),
    (dict(bias=(None, P + 1, None)), EALIGN),
])
def test_fwd_multi_rejects(lib, kw, expect):
    assert _fwdm(lib, **kw) == expect


def test_bwd_multi_workspace_query_rejects(lib):
    n = ctypes.c_size_t(0)
    D = _arr(ctypes.c_int64, [64, 64])
    assert lib.cconv_bwd_multi_workspace_bytes(2, D, 2, 16, 4, None) == ENULL
    assert lib.cconv_bwd_multi_workspace_bytes(0, D, 2, 16, 4, ctypes.byref(n)) == ESHAPE
    assert lib.cconv_bwd_multi_workspace_bytes(2, D, 2, 16, 6, ctypes.byref(n)) == EWIDTH
    assert lib.cconv_bwd_multi_workspace_bytes(2, _arr(ctypes.c_int64, [64, 12]), 2, 16, 4,
                                               ctypes.byref(n)) == EALIGN


def test_causal_conv1d_rejects_unknown_activation():
    x = torch.zeros(1, 4, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        cc.causal_conv1d(x, torch.zeros(8, 4), activation="gelu")


def test_describe_records_nothing_without_calls(lib):
    n = ctypes.c_int(-1)
    assert lib.cconv_describe_begin() == OK
    assert lib.cconv_describe_end(None, 0, ctypes.byref(n)) == OK
    assert n.value == 0
    assert lib.cconv_describe_end(None, 0, None) == ENULL
    assert lib.cconv_describe_end(None, 1, ctypes.byref(n)) == ENULL


def test_describe_keeps_host_checks(lib):
    # A call recorded between begin and end still runs its host checks and launches nothing.
    n = ctypes.c_int(-1)
    assert lib.cconv_describe_begin() == OK
    assert _fwd(lib, W=5) == EWIDTH
    assert lib.cconv_describe_end(None, 0, ctypes.byref(n)) == OK
    assert n.value == 0
