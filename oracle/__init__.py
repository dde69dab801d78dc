"""fp64 CPU oracle for the depthwise causal short convolution with fused SiLU.

TEST INFRASTRUCTURE ONLY.  The oracle defines the correct results that the CUDA library
is compared against.  Only the tests, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline / reference arm may import it; the product path never does, and the two
share no code.  The arithmetic lives in ``cconv_oracle.c`` (plain C, fp64, libm); this
module only marshals numpy arrays into it.

Sources followed (page title, file / section):
  * kernel-fun 0.2.0.dev1 wheel, kernel_fun/cconv/_kernels/strip.py: ``_tap``,
    ``_ld_ring``, ``_silu``, ``_dsilu``, ``_bwd4`` and the partial store of
    ``cconv_bwd_strip`` (forward / backward definitions);
  * "Add experimental causal conv1d decode update - #797" (NVIDIA/cudnn-frontend),
    PR summary (decode update, fail-closed index validation, full-sequence-to-decode
    state handoff);
  * kernel-fun 0.2.0.dev1 wheel, kernel_fun/_common/compat.py: the keywords of fla's
    causal_conv1d (initial_state, output_final_state, activation, cu_seqlens), which the
    packed-sequence forms ``fwd_seq`` / ``bwd_seq`` follow.

Conventions: the forward and backward take float64 values (the exact bf16 / fp32 values
the GPU receives, widened); the decode update takes the bf16 token and state as their
uint16 bit patterns, because it moves state bits.  Outputs are float64 and unrounded.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

import numpy as np

from . import build as _build

IDX_NEGATIVE = 1
IDX_OUT_OF_RANGE = 2
IDX_DUPLICATE = 4

_P = ctypes.c_void_p
_I64 = ctypes.c_int64


class Oracle:
    """Handle on one compiled copy of the oracle (the default one, or a test's variant)."""

    def __init__(self, lib_path: str | Path | None = None):
        if lib_path is None:
            lib_path = _build.build()
        self.path = Path(lib_path)
        lib = ctypes.CDLL(str(self.path))
        lib.oracle_fwd.argtypes = [_I64, _I64, _I64, ctypes.c_int, _P, _P, _P, _P, _P]
        lib.oracle_fwd.restype = ctypes.c_int
        lib.oracle_bwd.argtypes = [_I64, _I64, _I64, ctypes.c_int, _P, _P, _P, _P, _P, _P, _P]
        lib.oracle_bwd.restype = ctypes.c_int
        lib.oracle_validate.argtypes = [_I64, _I64, _P]
        lib.oracle_validate.restype = ctypes.c_int
        lib.oracle_update.argtypes = [_I64, _I64, ctypes.c_int, _P, _P, _I64, _P, _P, _P, _P]
        lib.oracle_update.restype = ctypes.c_int
        lib.oracle_validate_pad.argtypes = [_I64, _I64, _P, ctypes.c_int]
        lib.oracle_validate_pad.restype = ctypes.c_int
        lib.oracle_update_ex.argtypes = [_I64, _I64, ctypes.c_int, ctypes.c_int, _P, _P, _I64, _P,
                                         ctypes.c_int, _P, _P, ctypes.c_int, _P]
        lib.oracle_update_ex.restype = ctypes.c_int
        lib.oracle_update_ring.argtypes = [_I64, _I64, ctypes.c_int, ctypes.c_int, _P, _P, _I64,
                                           _P, ctypes.c_int, _P, _P, _P, ctypes.c_int, _P]
        lib.oracle_update_ring.restype = ctypes.c_int
        lib.oracle_fwd_seq.argtypes = [_I64, _P, _I64, ctypes.c_int, _P, _P, _P, _P, ctypes.c_int,
                                       _P, _P]
        lib.oracle_fwd_seq.restype = ctypes.c_int
        lib.oracle_bwd_seq.argtypes = [_I64, _P, _I64, ctypes.c_int, _P, _P, _P, _P, _P,
                                       ctypes.c_int, _P, _P, _P, _P]
        lib.oracle_bwd_seq.restype = ctypes.c_int
        self.lib = lib

    # -- marshalling helpers -------------------------------------------------------------
    @staticmethod
    def _bits(a) -> np.ndarray:
        a = np.ascontiguousarray(a)
        if a.dtype == np.int16:
            a = a.view(np.uint16)
        if a.dtype != np.uint16:
            raise TypeError(f"bf16 tensors are passed as uint16 bit patterns, got {a.dtype}")
        return a

    @staticmethod
    def _f64(a) -> np.ndarray | None:
        if a is None:
            return None
        return np.ascontiguousarray(a, dtype=np.float64)

    @staticmethod
    def _ptr(a) -> int | None:
        return None if a is None else a.ctypes.data

    # -- the four definitions --------------------------------------------------------------
    def fwd(self, x, w, bias=None, return_z: bool = False):
        """y = silu(bias + sum_k w[:, W-1-k] x[t-k]) for x [B,T,D], w [D,W]."""
        x = self._f64(x)
        B, T, D = x.shape
        w = self._f64(w)
        W = w.shape[1]
        assert w.shape == (D, W)
        b = self._f64(bias)
        y = np.empty((B, T, D), np.float64)
        z = np.empty((B, T, D), np.float64) if return_z else None
        rc = self.lib.oracle_fwd(B, T, D, W, self._ptr(x), self._ptr(w), self._ptr(b),
                                 self._ptr(y), self._ptr(z))
        if rc != 0:
            raise RuntimeError(f"oracle_fwd failed ({rc})")
        return (y, z) if return_z else y

    def bwd(self, x, dy, w, bias=None, want_dbias: bool = True):
        """(dx [B,T,D], dw [D,W], dbias [D] or None) for the forward above and upstream dy."""
        x = self._f64(x)
        dy = self._f64(dy)
        B, T, D = x.shape
        assert dy.shape == x.shape
        w = self._f64(w)
        W = w.shape[1]
        b = self._f64(bias)
        dx = np.empty((B, T, D), np.float64)
        dw = np.empty((D, W), np.float64)
        db = np.empty((D,), np.float64) if want_dbias else None
        rc = self.lib.oracle_bwd(B, T, D, W, self._ptr(x), self._ptr(dy), self._ptr(w),
                                 self._ptr(b), self._ptr(dx), self._ptr(dw), self._ptr(db))
        if rc != 0:
            raise RuntimeError(f"oracle_bwd failed ({rc})")
        return dx, dw, db

    def validate(self, idx, S: int) -> int:
        """Offence mask of a state_indices vector against a pool of S slots (0 = valid)."""
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        return int(self.lib.oracle_validate(idx.shape[0], S, self._ptr(idx)))

    def update(self, x_bits, state_bits, idx, w, bias=None):
        """One decode step.  Returns (status, y, new_state); the input state is not modified.

        status is 0, or the offence mask (> 0), in which case new_state equals the input
        and y is None."""
        x = self._bits(x_bits)
        N, D = x.shape
        st = np.array(self._bits(state_bits), copy=True)
        S = st.shape[0]
        w = self._f64(w)
        W = w.shape[1]
        assert st.shape == (S, D, W - 1)
        b = self._f64(bias)
        ix = None if idx is None else np.ascontiguousarray(idx, dtype=np.int32)
        y = np.empty((N, D), np.float64)
        rc = self.lib.oracle_update(N, D, W, self._ptr(x), self._ptr(st), S, self._ptr(ix),
                                    self._ptr(w), self._ptr(b), self._ptr(y))
        if rc < 0:
            raise RuntimeError(f"oracle_update failed ({rc})")
        return rc, (y if rc == 0 else None), st

    def validate_pad(self, idx, S: int, pad: bool) -> int:
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        return int(self.lib.oracle_validate_pad(idx.size, S, self._ptr(idx), int(pad)))

    def update_ex(self, x_bits, state_bits, idx, w, bias=None, *, pad: bool = False,
                  activation="silu"):
        """General decode update: state [S, D, Ls] with Ls >= W-1 (its newest W-1 entries
        feed the window); pad: index -1 marks a padding row (no state access, y row NaN);
        activation 'silu' or None.  Returns (status, y, new_state) like update()."""
        x = self._bits(x_bits)
        N, D = x.shape
        st = np.array(self._bits(state_bits), copy=True)
        S, _, Ls = st.shape
        w = self._f64(w)
        W = w.shape[1]
        b = self._f64(bias)
        ix = None if idx is None else np.ascontiguousarray(idx, dtype=np.int32)
        act = {"silu": 0, None: 1, "none": 1}[activation]
        y = np.empty((N, D), np.float64)
        rc = self.lib.oracle_update_ex(N, D, W, Ls, self._ptr(x), self._ptr(st), S,
                                       self._ptr(ix), int(pad), self._ptr(w), self._ptr(b), act,
                                       self._ptr(y))
        if rc < 0:
            raise RuntimeError(f"oracle_update_ex failed ({rc})")
        return rc, (y if rc == 0 else None), st

    def update_ring(self, x_bits, state_bits, idx, pos, w, bias=None, *, pad: bool = False,
                    activation="silu"):
        """Circular-buffer decode update: state [S, D, Ls] is a ring per channel, pos [N]
        the tokens each row's slot has seen; the token goes to ring entry pos mod Ls and the
        window is the W-1 entries before it.  Returns (status, y, new_state)."""
        x = self._bits(x_bits)
        N, D = x.shape
        st = np.array(self._bits(state_bits), copy=True)
        S, _, Ls = st.shape
        w = self._f64(w)
        W = w.shape[1]
        b = self._f64(bias)
        ix = None if idx is None else np.ascontiguousarray(idx, dtype=np.int32)
        ps = np.ascontiguousarray(pos, dtype=np.int32)
        act = {"silu": 0, None: 1, "none": 1}[activation]
        y = np.empty((N, D), np.float64)
        rc = self.lib.oracle_update_ring(N, D, W, Ls, self._ptr(x), self._ptr(st), S,
                                         self._ptr(ix), int(pad), self._ptr(ps), self._ptr(w),
                                         self._ptr(b), act, self._ptr(y))
        if rc < 0:
            raise RuntimeError(f"oracle_update_ring failed ({rc})")
        return rc, (y if rc == 0 else None), st

    # -- packed sequences, initial / final state, activation ---------------------------------
    @staticmethod
    def _cu(cu_seqlens):
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
        assert cu.ndim == 1 and cu.size >= 1 and cu[0] == 0
        return cu

    def fwd_seq(self, x, cu_seqlens, w, bias=None, initial_state=None, activation="silu",
                want_final: bool = False):
        """Packed-sequence forward.  x [total, D]; cu_seqlens [nseq+1]; initial_state
        [nseq, D, W-1] or None.  Returns y [total, D] (and final_state [nseq, D, W-1])."""
        x = self._f64(x)
        total, D = x.shape
        cu = self._cu(cu_seqlens)
        assert cu[-1] == total
        nseq = cu.size - 1
        w = self._f64(w)
        W = w.shape[1]
        b = self._f64(bias)
        init = self._f64(initial_state)
        act = {"silu": 0, None: 1, "none": 1}[activation]
        y = np.empty((total, D), np.float64)
        fin = np.empty((nseq, D, W - 1), np.float64) if want_final else None
        rc = self.lib.oracle_fwd_seq(nseq, self._ptr(cu), D, W, self._ptr(x), self._ptr(w),
                                     self._ptr(b), self._ptr(init), act, self._ptr(y),
                                     self._ptr(fin))
        if rc != 0:
            raise RuntimeError(f"oracle_fwd_seq failed ({rc})")
        return (y, fin) if want_final else y

    def bwd_seq(self, x, dy, cu_seqlens, w, bias=None, initial_state=None, activation="silu",
                want_dbias: bool = True, want_dinit: bool = False):
        """Packed-sequence backward: (dx [total, D], dw [D, W], dbias [D] or None,
        d_initial_state [nseq, D, W-1] or None)."""
        x = self._f64(x)
        dy = self._f64(dy)
        total, D = x.shape
        cu = self._cu(cu_seqlens)
        nseq = cu.size - 1
        w = self._f64(w)
        W = w.shape[1]
        b = self._f64(bias)
        init = self._f64(initial_state)
        act = {"silu": 0, None: 1, "none": 1}[activation]
        dx = np.empty((total, D), np.float64)
        dw = np.empty((D, W), np.float64)
        db = np.empty((D,), np.float64) if want_dbias else None
        di = np.empty((nseq, D, W - 1), np.float64) if want_dinit else None
        rc = self.lib.oracle_bwd_seq(nseq, self._ptr(cu), D, W, self._ptr(x), self._ptr(dy),
                                     self._ptr(w), self._ptr(b), self._ptr(init), act,
                                     self._ptr(dx), self._ptr(dw), self._ptr(db), self._ptr(di))
        if rc != 0:
            raise RuntimeError(f"oracle_bwd_seq failed ({rc})")
        return dx, dw, db, di


_default: Oracle | None = None


def get() -> Oracle:
    """The oracle built from ``cconv_oracle.c`` (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def fwd(*a, **k):
    return get().fwd(*a, **k)


def bwd(*a, **k):
    return get().bwd(*a, **k)


def validate(*a, **k):
    return get().validate(*a, **k)


def update(*a, **k):
    return get().update(*a, **k)


def update_ex(*a, **k):
    return get().update_ex(*a, **k)


def validate_pad(*a, **k):
    return get().validate_pad(*a, **k)


def update_ring(*a, **k):
    return get().update_ring(*a, **k)


def fwd_seq(*a, **k):
    return get().fwd_seq(*a, **k)


def bwd_seq(*a, **k):
    return get().bwd_seq(*a, **k)
