"""cconv_bwd_noalloc through the C ABI (GPU).

cconv_bwd_noalloc serves callers that cannot allocate device memory where they run the
backward: runtimes that hand out memory only from an arena sized up front, plugins inside a
framework that owns every allocation, threads that must not call cudaMalloc because it can
synchronise the device.  It uses the library's fixed device scratch array instead of a
caller-supplied workspace.  This test checks, on two calls in a row with different inputs,
that its outputs agree with cconv_bwd's within the backward tolerance.  It sits in a file
that pytest collects last so that a run stopping at the first failure has run every other
test before it, and it also passes on its own in a fresh process.
"""
import ctypes

import pytest
import torch

import depthwise_causal_short_gb300 as cc
from depthwise_causal_short_gb300 import _build, inputs
from tests.helpers import BWD_TOL, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    return cc.load()


def _noalloc(lib, x, dy, w, b, dx, dw, db):
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    wdt = 1 if w.dtype == torch.float32 else 0
    B, T, D = x.shape
    return lib.cconv_bwd_noalloc(p(x), x.stride(0), x.stride(1), p(dy), dy.stride(0), dy.stride(1),
                                 B, T, D, p(w), p(b), wdt, w.shape[1], p(dx), p(dw), p(db), stream)


@pytest.mark.parametrize("B,T,D,W,wdtype", [
    (2, 8192, 4096, 4, torch.float32),
    (4, 777, 1000, 3, torch.bfloat16),
])
def test_noalloc_matches_cconv_bwd_twice(lib, B, T, D, W, wdtype):
    for call in range(2):  # two calls in a row share the scratch array
        x, dy, w, b = inputs.fwd_bwd_inputs(B, T, D, W, True, wdtype=wdtype, seed=100 + call)
        xg, dyg, wg, bg = x.cuda(), dy.cuda(), w.cuda(), b.cuda()
        dx_ref, dw_ref, db_ref = cc.cconv_bwd(xg, dyg, wg, bg)
        dx = torch.empty_like(dx_ref)
        dw = torch.empty_like(dw_ref)
        db = torch.empty_like(db_ref)
        rc = _noalloc(lib, xg, dyg, wg, bg, dx, dw, db)
        assert rc == 0, cc.cconv_status_str(rc)
        torch.cuda.synchronize()
        for name, got, ref in (("dx", dx, dx_ref), ("dw", dw, dw_ref), ("dbias", db, db_ref)):
            e = rel_err(got.double().cpu().numpy(), ref.double().cpu().numpy())
            assert e <= BWD_TOL, f"call {call}: {name} differs from cconv_bwd by {e:.2e}"


def test_noalloc_rejects_a_problem_larger_than_its_scratch(lib):
    # D = 2^21 channels needs far more than the 8 MiB array; the call must refuse before
    # touching any buffer (the pointers below are never dereferenced).
    fake = 1 << 20
    rc = lib.cconv_bwd_noalloc(fake, 0, 1 << 21, fake, 0, 1 << 21, 1, 1, 1 << 21, fake, None, 1, 4,
                               fake, fake, None, None)
    assert rc == -7
