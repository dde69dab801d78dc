"""cconv_bwd_noalloc through the C ABI (GPU).

cconv_bwd_noalloc serves callers that cannot allocate device memory where they run the
backward: runtimes that hand out memory only from an arena sized up front, plugins inside a
framework that owns every allocation, threads that must not call cudaMalloc because it can
synchronise the device.  It runs the same kernels with the same work split as cconv_bwd,
with the partial sums in the library's fixed device scratch array instead of a
caller-supplied workspace, so its outputs must equal cconv_bwd's bit for bit.

The test queues two calls with different inputs back to back on one stream, into separate
outputs and with no launch or synchronisation between them (the second call's stream
kernel may start while the first call's reduction still reads the shared array), then
checks both against cconv_bwd bit for bit and against the fp64 oracle within the backward
tolerance.  After a warm-up call, further calls must leave the device's free memory
unchanged.  The file sits where pytest collects it last, so that a run stopping at the
first failure has run every other test before it; it also passes on its own in a fresh
process.
"""
import ctypes

import pytest
import torch

import depthwise_causal_short_gb300 as cc
from depthwise_causal_short_gb300 import _build, inputs
from tests.helpers import BWD_TOL, oracle_bwd, rel_err

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


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


@pytest.mark.parametrize("B,T,D,W,wdtype", [
    (2, 8192, 4096, 4, torch.float32),
    (4, 777, 1000, 3, torch.bfloat16),
])
def test_noalloc_equals_cconv_bwd_on_two_queued_calls(lib, B, T, D, W, wdtype):
    calls = []
    for k in range(2):
        x, dy, w, b = inputs.fwd_bwd_inputs(B, T, D, W, True, wdtype=wdtype, seed=100 + k)
        g = [t.cuda() for t in (x, dy, w, b)]
        ref = cc.cconv_bwd(*g)  # dx, dw, dbias through the workspace call
        out = (torch.empty_like(ref[0]), torch.empty_like(ref[1]), torch.empty_like(ref[2]))
        calls.append(((x, dy, w, b), g, ref, out))
    torch.cuda.synchronize()
    for _, g, _, out in calls:  # both calls queued, nothing in between
        rc = _noalloc(lib, *g, *out)
        assert rc == 0, cc.cconv_status_str(rc)
    torch.cuda.synchronize()
    for k, (host, _, ref, out) in enumerate(calls):
        want = oracle_bwd(*host, want_dbias=True)
        for name, got, r, o in zip(("dx", "dw", "dbias"), out, ref, want):
            assert torch.equal(_bits(got), _bits(r)), f"call {k}: {name} differs from cconv_bwd"
            e = rel_err(got.double().cpu().numpy(), o)
            assert e <= BWD_TOL, f"call {k}: {name} differs from the oracle by {e:.2e}"


def test_noalloc_leaves_free_memory_unchanged(lib):
    B, T, D, W = 2, 4096, 2048, 4
    x, dy, w, b = (t.cuda() for t in inputs.fwd_bwd_inputs(B, T, D, W, True, seed=7))
    dx, dw, db = torch.empty_like(x), torch.empty_like(w), torch.empty_like(b)
    assert _noalloc(lib, x, dy, w, b, dx, dw, db) == 0  # warm-up: may load the device code
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert _noalloc(lib, x, dy, w, b, dx, dw, db) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"
    ref = cc.cconv_bwd(x, dy, w, b)
    torch.cuda.synchronize()
    for got, r in zip((dx, dw, db), ref):
        assert torch.equal(_bits(got), _bits(r))


def test_noalloc_rejects_a_problem_larger_than_its_scratch(lib):
    # D = 2^21 channels needs far more than the 8 MiB array; the call must refuse before
    # touching any buffer (the pointers below are never dereferenced).
    fake = 1 << 20
    rc = lib.cconv_bwd_noalloc(fake, 0, 1 << 21, fake, 0, 1 << 21, 1, 1, 1 << 21, fake, None, 1, 4,
                               fake, fake, None, None)
    assert rc == -7
