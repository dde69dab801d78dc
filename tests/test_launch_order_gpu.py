"""The packed-sequence kernels read cu_seqlens only after their programmatic dependency wait.

Every kernel of the library is launched as a programmatic dependent of the kernel before it
on the stream, so it may start while that kernel still runs; whatever that kernel writes
must not be read before griddepcontrol.wait.  Here the kernel before the packed-sequence
calls (tests/gpu_support/late_writer.cu, built with nvcc for this test) lets its dependents
start at once and writes the real cu_seqlens over a zeroed one only 200 us later.  Row
ranges split from the zeroed vector would all be empty, so a call that read cu_seqlens too
early would leave most of its outputs unwritten.  Each result is checked against the
oracle on the real vector, for the forward and for both backward CTA forms (lockstep from
512 channels, independent warp pipelines below).
"""
import ctypes
import subprocess
from pathlib import Path

import pytest
import torch

import depthwise_causal_short_gb300 as cc
import oracle
from depthwise_causal_short_gb300 import _build, inputs
from tests.helpers import BWD_TOL, FWD_TOL, bits, f64, rel_err

pytestmark = pytest.mark.gpu

SUPPORT = Path(__file__).resolve().parent / "gpu_support"
DELAY_NS = 200_000


@pytest.fixture(scope="module")
def writer():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    src = SUPPORT / "late_writer.cu"
    out = SUPPORT / "_build" / "liblate_writer.so"
    if not out.exists() or out.stat().st_mtime < src.stat().st_mtime:
        out.parent.mkdir(parents=True, exist_ok=True)
        subprocess.run([_build.nvcc(), *_build.ARCH, "-O2", "-shared", "-Xcompiler", "-fPIC",
                        "-cudart", "static", "-o", str(out), str(src)], check=True,
                       capture_output=True)
    lib = ctypes.CDLL(str(out))
    lib.late_copy.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                              ctypes.c_ulonglong, ctypes.c_void_p]
    lib.late_copy.restype = ctypes.c_int
    return lib


def _late_cu(writer, cu: torch.Tensor) -> torch.Tensor:
    """A zeroed device cu_seqlens that the late writer overwrites with `cu` on the stream."""
    dst = torch.zeros_like(cu).cuda()
    src = cu.cuda()
    torch.cuda.synchronize()
    rc = writer.late_copy(dst.data_ptr(), src.data_ptr(), cu.numel(), DELAY_NS,
                          torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    dst._keep = src  # the copy's source lives as long as the destination
    return dst


@pytest.mark.parametrize("D", [256, 2048])
def test_cu_seqlens_from_the_previous_kernel(writer, D):
    W = 4
    lens = [3000, 1, 0, 700, 2, 5000, 129, 64, 3]
    x, dy, cu, w, b, init = inputs.varlen_inputs(lens, D, W, bias=True, seed=21)
    xg, dyg, wg, bg, ig = (t.cuda() for t in (x, dy, w, b, init))
    assert cc.cconv_device_fault() == 0

    y, fin, _ = cc.cconv_fwd_varlen(xg, _late_cu(writer, cu), wg, bg, initial_state=ig,
                                    final_state=True)
    dx, dw, db, di = cc.cconv_bwd_varlen(xg, dyg, _late_cu(writer, cu), wg, bg,
                                         initial_state=ig, want_dbias=True)
    torch.cuda.synchronize()
    assert cc.cconv_device_fault() == 0

    ry, rfin = oracle.fwd_seq(f64(x), cu.numpy(), f64(w), f64(b), f64(init), "silu",
                              want_final=True)
    assert rel_err(f64(y), ry) <= FWD_TOL
    assert (bits(fin).astype("int64") == bits(torch.from_numpy(rfin).to(torch.bfloat16))
            .astype("int64")).all()
    rdx, rdw, rdb, rdi = oracle.bwd_seq(f64(x), f64(dy), cu.numpy(), f64(w), f64(b), f64(init),
                                        want_dinit=True)
    for name, got, ref in (("dx", dx, rdx), ("dw", dw, rdw), ("dbias", db, rdb),
                           ("d_initial_state", di, rdi)):
        assert rel_err(f64(got), ref) <= BWD_TOL, name
