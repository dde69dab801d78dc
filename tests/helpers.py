"""Shared helpers for the GPU parity tests: tolerances, error metric, oracle calls."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# max |gpu - ref| / max |ref| per output tensor, ref in fp64 (the pages' budgets on bf16
# outputs: kernel-fun 0.2.0.dev1 wheel, cconv/_kernels/strip.py, `_sigmoid` comment).
FWD_TOL = 5e-3
BWD_TOL = 8e-3


def f64(t: torch.Tensor | None):
    return None if t is None else t.detach().to("cpu", torch.float64).numpy()


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def rel_err(gpu, ref) -> float:
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    err = float(np.max(np.abs(gpu - ref)))
    scale = float(np.max(np.abs(ref)))
    return err / scale if scale > 0 else err


def oracle_fwd(x, w, b):
    return oracle.fwd(f64(x), f64(w), f64(b))


def oracle_bwd(x, dy, w, b, want_dbias=True):
    return oracle.bwd(f64(x), f64(dy), f64(w), f64(b), want_dbias=want_dbias)
