"""ctypes binding of libcconv.so, with the C ABI's names (argument marshalling only).

Every step of the computation runs in the library's CUDA kernels; this module only turns
torch tensors into pointers, sizes and strides, allocates outputs with torch when the
caller does not pass them, and raises on a nonzero status.  There is no fallback: if the
library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import re
from pathlib import Path

import torch

from . import _build

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_INT = ctypes.c_int

CCONV_BF16 = 0
CCONV_F32 = 1
CCONV_ACT_SILU = 0
CCONV_ACT_NONE = 1
STATUS = {
    0: "CCONV_OK", -1: "CCONV_ERR_NULL", -2: "CCONV_ERR_SHAPE", -3: "CCONV_ERR_WIDTH",
    -4: "CCONV_ERR_ALIGN", -5: "CCONV_ERR_STRIDE", -6: "CCONV_ERR_DTYPE",
    -7: "CCONV_ERR_WORKSPACE", -8: "CCONV_ERR_INDEX", -9: "CCONV_ERR_CUDA",
    -10: "CCONV_ERR_DEVICE",
}
IDX_NEGATIVE = 1
IDX_OUT_OF_RANGE = 2
IDX_DUPLICATE = 4


class CConvError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        super().__init__(f"{call}: {STATUS.get(status, status)} ({status})")


class KernelDesc(ctypes.Structure):
    """cconv_kernel_desc of include/cconv.h."""
    _fields_ = [("name", ctypes.c_char * 160), ("registers", ctypes.c_int),
                ("local_bytes", ctypes.c_int), ("static_shared_bytes", ctypes.c_int),
                ("dynamic_shared_bytes", ctypes.c_int), ("threads", ctypes.c_int),
                ("ctas_per_sm", ctypes.c_int), ("ctas", ctypes.c_int64)]


_lib = None


def lib_path() -> Path:
    return _build.LIB


def load(path: str | Path | None = None):
    """Load libcconv.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = Path(path) if path else _build.LIB
    if not p.exists():
        raise RuntimeError(
            f"{p} is missing: build the CUDA library first "
            "(python -m depthwise_causal_short_gb300._build, or __graft_entry__.build())")
    lib = ctypes.CDLL(str(p))
    lib.cconv_fwd.argtypes = [_P, _I64, _I64, _I64, _I64, _I64, _P, _P, _INT, _INT, _P, _P]
    lib.cconv_fwd.restype = _INT
    lib.cconv_bwd_workspace_bytes.argtypes = [_I64, _I64, _I64, _INT, ctypes.POINTER(ctypes.c_size_t)]
    lib.cconv_bwd_workspace_bytes.restype = _INT
    lib.cconv_bwd.argtypes = [_P, _I64, _I64, _P, _I64, _I64, _I64, _I64, _I64, _P, _P, _INT,
                              _INT, _P, _P, _P, _P, ctypes.c_size_t, _P]
    lib.cconv_bwd.restype = _INT
    lib.cconv_bwd_noalloc.argtypes = [_P, _I64, _I64, _P, _I64, _I64, _I64, _I64, _I64, _P, _P,
                                      _INT, _INT, _P, _P, _P, _P]
    lib.cconv_bwd_noalloc.restype = _INT
    lib.cconv_update.argtypes = [_P, _I64, _I64, _I64, _P, _I64, _P, _P, _P, _INT, _INT, _P, _P, _P]
    lib.cconv_update.restype = _INT
    lib.cconv_fwd_varlen.argtypes = [_P, _I64, _I64, _I64, _P, _I64, _P, _P, _INT, _INT, _INT,
                                     _P, _P, _P, _I64, _P, _P, _P]
    lib.cconv_fwd_varlen.restype = _INT
    lib.cconv_bwd_varlen_workspace_bytes.argtypes = [_I64, _I64, _INT,
                                                     ctypes.POINTER(ctypes.c_size_t)]
    lib.cconv_bwd_varlen_workspace_bytes.restype = _INT
    lib.cconv_bwd_varlen.argtypes = [_P, _I64, _P, _I64, _I64, _I64, _P, _I64, _P, _P, _INT, _INT,
                                     _INT, _P, _P, _I64, _P, _P, _P, _P, _P, _P, ctypes.c_size_t,
                                     _P]
    lib.cconv_bwd_varlen.restype = _INT
    lib.cconv_update_ex.argtypes = [_P, _I64, _I64, _I64, _P, _I64, _INT, _P, _INT, _P, _P, _P,
                                    _INT, _INT, _INT, _P, _P, _P]
    lib.cconv_update_ex.restype = _INT
    _PA = ctypes.POINTER(ctypes.c_void_p)
    _IA = ctypes.POINTER(ctypes.c_int64)
    lib.cconv_fwd_multi.argtypes = [_INT, _PA, _IA, _IA, _IA, _PA, _PA, _PA, _I64, _I64, _INT, _INT,
                                    _P]
    lib.cconv_fwd_multi.restype = _INT
    lib.cconv_bwd_multi_workspace_bytes.argtypes = [_INT, _IA, _I64, _I64, _INT,
                                                    ctypes.POINTER(ctypes.c_size_t)]
    lib.cconv_bwd_multi_workspace_bytes.restype = _INT
    lib.cconv_bwd_multi.argtypes = [_INT, _PA, _IA, _IA, _PA, _IA, _IA, _IA, _PA, _PA, _PA, _PA,
                                    _PA, _I64, _I64, _INT, _INT, _P, ctypes.c_size_t, _P]
    lib.cconv_bwd_multi.restype = _INT
    lib.cconv_status_str.argtypes = [_INT]
    lib.cconv_status_str.restype = ctypes.c_char_p
    lib.cconv_device_fault.argtypes = [ctypes.POINTER(ctypes.c_int32)]
    lib.cconv_device_fault.restype = _INT
    lib.cconv_describe_begin.argtypes = []
    lib.cconv_describe_begin.restype = _INT
    lib.cconv_describe_end.argtypes = [ctypes.POINTER(KernelDesc), _INT, ctypes.POINTER(_INT)]
    lib.cconv_describe_end.restype = _INT
    if path is None:
        _lib = lib
    return lib


def header_functions() -> list[str]:
    """Names of the functions include/cconv.h declares (CCONV_API ... name(...))."""
    text = (_build.INCLUDE / "cconv.h").read_text()
    return re.findall(r"CCONV_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


# ---------------------------------------------------------------------------------------
# argument checks and marshalling
#
# The C ABI sees pointers and sizes only, and the kernels size every access from those
# sizes (x's [B, T, D], the pool's S, the number of sequences).  A tensor smaller than the
# sizes imply (a dy shorter than x, a [S, D, 2] state with W = 4, a non-contiguous output)
# would be read or written past its end.  So every wrapper checks, before anything is
# enqueued, the shape, dtype, layout and device of every tensor the call touches: shape,
# dtype and layout first (TypeError / ValueError), then that all of them live on one CUDA
# device (ValueError).  The call then runs with that device current, on its current stream
# unless a stream is given.
# ---------------------------------------------------------------------------------------

_WDTYPES = (torch.float32, torch.bfloat16)


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _wdt(w: torch.Tensor) -> int:
    return CCONV_F32 if w.dtype == torch.float32 else CCONV_BF16


def _check(rc: int, call: str):
    if rc != 0:
        raise CConvError(rc, call)


def _tensor(t, name: str):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor, got {type(t).__name__}")


def _rows(t, name: str, dim: int):
    """bf16 activations with `dim` dimensions and channel stride 1 (other strides free)."""
    _tensor(t, name)
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    if t.dim() != dim:
        raise ValueError(f"{name} must have {dim} dimensions, got shape {tuple(t.shape)}")
    if t.shape[-1] > 1 and t.stride(-1) != 1:
        raise ValueError(f"{name} must have channel stride 1, got strides {t.stride()}")


def _weights(w, D: int, name: str = "w") -> int:
    """w [D, W] contiguous, fp32 or bf16, 1 <= W <= 4; returns W."""
    _tensor(w, name)
    if w.dtype not in _WDTYPES:
        raise TypeError(f"{name} dtype must be float32 or bfloat16, got {w.dtype}")
    if w.dim() != 2 or w.shape[0] != D:
        raise ValueError(f"{name} must be [D={D}, W], got shape {tuple(w.shape)}")
    if not 1 <= w.shape[1] <= 4:
        raise ValueError(f"{name}: W must be in [1, 4], got {w.shape[1]}")
    if not w.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return int(w.shape[1])


def _exact(t, shape, dtype, name: str):
    """A tensor the kernels address densely: exactly `shape` and `dtype`, contiguous."""
    _tensor(t, name)
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _int32_vec(t, n: int, name: str):
    """int32 [n] contiguous (indices, positions)."""
    _exact(t, (n,), torch.int32, name)


def _status(t):
    _tensor(t, "status")
    if t.dtype != torch.int32 or t.numel() < 2 or not t.is_contiguous():
        raise ValueError("status must be a contiguous int32 tensor of at least 2 elements")


def _workspace(t):
    _tensor(t, "workspace")
    if not t.is_contiguous():
        raise ValueError("workspace must be contiguous")


def _bias(b, D: int, w: torch.Tensor, name: str = "bias"):
    if b is not None:
        _exact(b, (D,), w.dtype, name)


def _extent(t: torch.Tensor):
    """[first, last) byte range a tensor's elements span."""
    n = t.numel()
    if n == 0:
        return (0, 0)
    a = t.data_ptr()
    if t.is_contiguous():
        return (a, a + n * t.element_size())
    span = 1
    for size, stride in zip(t.shape, t.stride()):
        span += (size - 1) * stride
    return (a, a + span * t.element_size())


def _disjoint(outs, ins):
    """No output may overlap what the call reads.  outs, ins: sequences of (name, tensor or
    None)."""
    spans = [(n, _extent(t)) for n, t in ins if t is not None]
    for on, o in outs:
        if o is None:
            continue
        a0, a1 = _extent(o)
        for n, (b0, b1) in spans:
            if a0 < b1 and b0 < a1:
                raise ValueError(f"{on} overlaps {n}")


def _device(names, tensors) -> torch.device:
    """Every given tensor (None entries skipped) is a CUDA tensor on the first one's device;
    returns that device.  names: the tensors' names, a sequence or a function of the
    position (only used for the error message)."""
    idx = -2
    for i, t in enumerate(tensors):
        if t is None:
            continue
        d = t.get_device()
        if d >= 0 and (idx == -2 or d == idx):
            idx = d
            continue
        name = names(i) if callable(names) else names[i]
        if d < 0:
            raise ValueError(f"{name} must be a CUDA tensor, got device {t.device}")
        raise ValueError(f"{name} is on cuda:{d}, but the call's tensors are on cuda:{idx}")
    return torch.device("cuda", idx)


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, dev: torch.device) -> ctypes.c_void_p:
    if stream is None:
        if _raw_stream is not None:
            return ctypes.c_void_p(_raw_stream(dev.index))
        return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    if hasattr(stream, "cuda_stream"):
        sdev = getattr(stream, "device", None)
        if sdev is not None and torch.device(sdev) != dev:
            raise ValueError(f"stream belongs to {sdev}, but the call's tensors are on {dev}")
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _run(dev: torch.device, fn, *args):
    """fn(*args) with `dev` current (the library launches on the current device)."""
    if dev.index == torch.cuda.current_device():
        return fn(*args)
    with torch.cuda.device(dev):
        return fn(*args)


# ---------------------------------------------------------------------------------------
# the three calls
# ---------------------------------------------------------------------------------------

def cconv_fwd(x: torch.Tensor, w: torch.Tensor, bias: torch.Tensor | None = None, *,
              y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y = silu(bias + causal depthwise conv(x, w)); x [B,T,D] bf16, w [D,W]."""
    _rows(x, "x", 3)
    B, T, D = x.shape
    W = _weights(w, D)
    _bias(bias, D, w)
    if y is not None:
        _exact(y, (B, T, D), torch.bfloat16, "y")
        _disjoint((("y", y),), (("x", x),))
    dev = _device(("x", "w", "bias", "y"), (x, w, bias, y))
    if y is None:
        y = torch.empty((B, T, D), dtype=torch.bfloat16, device=dev)
    rc = _run(dev, load().cconv_fwd, _ptr(x), B, T, D, x.stride(0), x.stride(1), _ptr(w),
              _ptr(bias), _wdt(w), W, _ptr(y), _stream(stream, dev))
    _check(rc, "cconv_fwd")
    return y


def cconv_bwd_workspace_bytes(B: int, T: int, D: int, W: int, device=None) -> int:
    """Workspace cconv_bwd needs on `device` (default: the current CUDA device)."""
    n = ctypes.c_size_t(0)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    _check(_run(dev, load().cconv_bwd_workspace_bytes, B, T, D, W, ctypes.byref(n)),
           "cconv_bwd_workspace_bytes")
    return int(n.value)


def _bwd_args(x, dy, w, bias, dx, dw, dbias, want_dbias):
    """Checks shared by cconv_bwd and cconv_bwd_noalloc; returns (B, T, D, W, dev)."""
    _rows(x, "x", 3)
    _rows(dy, "dy", 3)
    B, T, D = x.shape
    if dy.shape != x.shape:
        raise ValueError(f"dy must have x's shape {tuple(x.shape)}, got {tuple(dy.shape)}")
    W = _weights(w, D)
    _bias(bias, D, w)
    if dx is not None:
        _exact(dx, (B, T, D), torch.bfloat16, "dx")
        _disjoint((("dx", dx),), (("x", x), ("dy", dy)))
    if dw is not None:
        _exact(dw, (D, W), w.dtype, "dw")
    if want_dbias and dbias is not None:
        _bias(dbias, D, w, "dbias")
    return B, T, D, W


def cconv_bwd(x: torch.Tensor, dy: torch.Tensor, w: torch.Tensor,
              bias: torch.Tensor | None = None, *, want_dbias: bool | None = None,
              dx: torch.Tensor | None = None, dw: torch.Tensor | None = None,
              dbias: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
              stream=None):
    """(dx, dw, dbias) for upstream gradient dy; dbias is None unless wanted (default:
    when a bias is given)."""
    if want_dbias is None:
        want_dbias = bias is not None or dbias is not None
    B, T, D, W = _bwd_args(x, dy, w, bias, dx, dw, dbias, want_dbias)
    if workspace is not None:
        _workspace(workspace)
    dev = _device(("x", "dy", "w", "bias", "dx", "dw", "dbias", "workspace"),
                  (x, dy, w, bias, dx, dw, dbias if want_dbias else None, workspace))
    if dx is None:
        dx = torch.empty((B, T, D), dtype=torch.bfloat16, device=dev)
    if dw is None:
        dw = torch.empty((D, W), dtype=w.dtype, device=dev)
    if want_dbias and dbias is None:
        dbias = torch.empty((D,), dtype=w.dtype, device=dev)
    if workspace is None:
        workspace = torch.empty(cconv_bwd_workspace_bytes(B, T, D, W, dev), dtype=torch.uint8,
                                device=dev)
    rc = _run(dev, load().cconv_bwd, _ptr(x), x.stride(0), x.stride(1), _ptr(dy), dy.stride(0),
              dy.stride(1), B, T, D, _ptr(w), _ptr(bias), _wdt(w), W, _ptr(dx), _ptr(dw),
              _ptr(dbias if want_dbias else None), _ptr(workspace),
              workspace.numel() * workspace.element_size(), _stream(stream, dev))
    _check(rc, "cconv_bwd")
    return dx, dw, (dbias if want_dbias else None)


def cconv_bwd_noalloc(x: torch.Tensor, dy: torch.Tensor, w: torch.Tensor,
                      bias: torch.Tensor | None = None, *, dx: torch.Tensor,
                      dw: torch.Tensor, dbias: torch.Tensor | None = None, stream=None):
    """cconv_bwd for callers that cannot allocate device memory at this point: every output
    must be passed in, and the partial sums use the library's fixed 8 MiB device scratch
    array instead of a workspace.  Calls that overlap on the GPU race on that array."""
    _bwd_args(x, dy, w, bias, dx, dw, dbias, True)
    B, T, D = x.shape
    dev = _device(("x", "dy", "w", "bias", "dx", "dw", "dbias"), (x, dy, w, bias, dx, dw, dbias))
    rc = _run(dev, load().cconv_bwd_noalloc, _ptr(x), x.stride(0), x.stride(1), _ptr(dy),
              dy.stride(0), dy.stride(1), B, T, D, _ptr(w), _ptr(bias), _wdt(w), w.shape[1],
              _ptr(dx), _ptr(dw), _ptr(dbias), _stream(stream, dev))
    _check(rc, "cconv_bwd_noalloc")
    return dx, dw, dbias


def _pool(state, D: int, lengths, name: str = "state"):
    """A bf16 state pool [S, D, L], contiguous, L in `lengths`; returns (S, L)."""
    _tensor(state, name)
    if state.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {state.dtype}")
    if state.dim() != 3 or state.shape[1] != D or state.shape[2] not in lengths:
        want = " or ".join(f"[S, {D}, {L}]" for L in lengths)
        raise ValueError(f"{name} must be {want}, got shape {tuple(state.shape)}")
    if not state.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return int(state.shape[0]), int(state.shape[2])


def cconv_update(x: torch.Tensor, state: torch.Tensor, w: torch.Tensor,
                 bias: torch.Tensor | None = None, state_indices: torch.Tensor | None = None,
                 *, y: torch.Tensor | None = None, status: torch.Tensor | None = None,
                 stream=None):
    """One decode step: (y [N,D], status int32[2] on the device).  state [S,D,W-1] is
    updated in place unless status[0] reports CCONV_ERR_INDEX."""
    _rows(x, "x", 2)
    N, D = x.shape
    W = _weights(w, D)
    _bias(bias, D, w)
    S, _ = _pool(state, D, (W - 1,))
    if state_indices is not None:
        _int32_vec(state_indices, N, "state_indices")
    elif S < N:
        raise ValueError(f"without state_indices row i uses slot i: state needs S >= N={N}")
    if y is not None:
        _exact(y, (N, D), torch.bfloat16, "y")
    if status is not None:
        _status(status)
    dev = _device(("x", "state", "w", "bias", "state_indices", "y", "status"),
                  (x, state, w, bias, state_indices, y, status))
    if y is None:
        y = torch.empty((N, D), dtype=torch.bfloat16, device=dev)
    if status is None:
        status = torch.empty(2, dtype=torch.int32, device=dev)
    rc = _run(dev, load().cconv_update, _ptr(x), N, D, x.stride(0), _ptr(state), S,
              _ptr(state_indices), _ptr(w), _ptr(bias), _wdt(w), W, _ptr(y), _ptr(status),
              _stream(stream, dev))
    _check(rc, "cconv_update")
    return y, status


def _act(activation) -> int:
    if activation in ("silu", "swish"):
        return CCONV_ACT_SILU
    if activation is None or activation == "none":
        return CCONV_ACT_NONE
    raise ValueError(f"activation must be 'silu' or None, got {activation!r}")


def _cu(cu_seqlens) -> int:
    """cu_seqlens: int32 [nseq + 1], contiguous, nseq >= 1; returns nseq."""
    _tensor(cu_seqlens, "cu_seqlens")
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1:
        raise TypeError("cu_seqlens must be a 1-D int32 tensor")
    if cu_seqlens.numel() < 2:
        raise ValueError("cu_seqlens must hold at least 2 entries (one sequence)")
    if not cu_seqlens.is_contiguous():
        raise ValueError("cu_seqlens must be contiguous")
    return cu_seqlens.numel() - 1


def cconv_fwd_varlen(x: torch.Tensor, cu_seqlens: torch.Tensor, w: torch.Tensor,
                     bias: torch.Tensor | None = None, *, activation="silu",
                     initial_state: torch.Tensor | None = None,
                     final_state: torch.Tensor | bool | None = None,
                     state_indices: torch.Tensor | None = None, status: torch.Tensor | None = None,
                     y: torch.Tensor | None = None, stream=None):
    """Packed-sequence forward.  x [total, D] bf16; cu_seqlens int32 [nseq+1] on the device.
    initial_state / final_state: [S, D, W-1] bf16 state arrays (final_state=True allocates
    [nseq, D, W-1]); state_indices int32 [nseq] picks each sequence's slot (then a status
    int32[2] is written on the device).  Returns (y, final_state or None, status or None)."""
    _rows(x, "x", 2)
    total, D = x.shape
    nseq = _cu(cu_seqlens)
    W = _weights(w, D)
    _bias(bias, D, w)
    act = _act(activation)
    L = W - 1
    pools = []
    if initial_state is not None:
        pools.append(_pool(initial_state, D, (L,), "initial_state")[0])
    want_final = final_state is True
    if final_state is False or final_state is True:
        final_state = None
    if final_state is not None:
        pools.append(_pool(final_state, D, (L,), "final_state")[0])
        _disjoint((("final_state", final_state),), (("x", x),))
    if state_indices is not None:
        _int32_vec(state_indices, nseq, "state_indices")
        if status is not None:
            _status(status)
    if y is not None:
        _exact(y, (total, D), torch.bfloat16, "y")
        _disjoint((("y", y),), (("x", x), ("final_state", final_state)))
    S = min(pools) if pools else nseq
    if want_final:
        S = min(S, nseq)
    if state_indices is None and (pools or want_final) and S < nseq:
        raise ValueError(f"without state_indices sequence i uses slot i: state arrays need "
                         f"at least nseq={nseq} slots")
    dev = _device(("x", "cu_seqlens", "w", "bias", "initial_state", "final_state",
                   "state_indices", "status", "y"),
                  (x, cu_seqlens, w, bias, initial_state, final_state, state_indices,
                   status if state_indices is not None else None, y))
    if want_final:
        final_state = torch.empty((nseq, D, L), dtype=torch.bfloat16, device=dev)
    if state_indices is not None and status is None:
        status = torch.empty(2, dtype=torch.int32, device=dev)
    if y is None:
        y = torch.empty((total, D), dtype=torch.bfloat16, device=dev)
    rc = _run(dev, load().cconv_fwd_varlen, _ptr(x), total, D, x.stride(0), _ptr(cu_seqlens),
              nseq, _ptr(w), _ptr(bias), _wdt(w), W, act, _ptr(initial_state), _ptr(final_state),
              _ptr(state_indices), S, _ptr(status if state_indices is not None else None),
              _ptr(y), _stream(stream, dev))
    _check(rc, "cconv_fwd_varlen")
    return y, final_state, (status if state_indices is not None else None)


def cconv_bwd_varlen_workspace_bytes(total: int, D: int, W: int, device=None) -> int:
    """Workspace cconv_bwd_varlen needs on `device` (default: the current CUDA device)."""
    n = ctypes.c_size_t(0)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    _check(_run(dev, load().cconv_bwd_varlen_workspace_bytes, total, D, W, ctypes.byref(n)),
           "cconv_bwd_varlen_workspace_bytes")
    return int(n.value)


def cconv_bwd_varlen(x: torch.Tensor, dy: torch.Tensor, cu_seqlens: torch.Tensor,
                     w: torch.Tensor, bias: torch.Tensor | None = None, *, activation="silu",
                     initial_state: torch.Tensor | None = None,
                     state_indices: torch.Tensor | None = None,
                     status: torch.Tensor | None = None, want_dbias: bool | None = None,
                     want_dinit: bool | None = None, dx: torch.Tensor | None = None,
                     dw: torch.Tensor | None = None, dbias: torch.Tensor | None = None,
                     d_initial_state: torch.Tensor | None = None,
                     workspace: torch.Tensor | None = None, stream=None):
    """Packed-sequence backward: (dx, dw, dbias or None, d_initial_state or None).
    initial_state is [nseq, D, W-1] (slot i is sequence i), or with state_indices (int32
    [nseq] on the device) a pool [S, D, W-1] whose slot state_indices[i] is sequence i's;
    the indices are checked on the device and `status` (int32[2], required with indices)
    gets the verdict.  d_initial_state is [nseq, D, W-1]."""
    _rows(x, "x", 2)
    _rows(dy, "dy", 2)
    total, D = x.shape
    if dy.shape != x.shape:
        raise ValueError(f"dy must have x's shape {tuple(x.shape)}, got {tuple(dy.shape)}")
    nseq = _cu(cu_seqlens)
    W = _weights(w, D)
    _bias(bias, D, w)
    act = _act(activation)
    L = W - 1
    S = nseq
    if state_indices is not None:
        _int32_vec(state_indices, nseq, "state_indices")
        if status is None:
            raise ValueError("status (int32[2] on the device) is required with state_indices")
        _status(status)
        if initial_state is not None:
            S = _pool(initial_state, D, (L,), "initial_state")[0]
    elif initial_state is not None:
        _exact(initial_state, (nseq, D, L), torch.bfloat16, "initial_state")
    if want_dbias is None:
        want_dbias = bias is not None or dbias is not None
    if want_dinit is None:
        want_dinit = initial_state is not None or d_initial_state is not None
    if dx is not None:
        _exact(dx, (total, D), torch.bfloat16, "dx")
        _disjoint((("dx", dx),), (("x", x), ("dy", dy)))
    if dw is not None:
        _exact(dw, (D, W), w.dtype, "dw")
    if want_dbias and dbias is not None:
        _bias(dbias, D, w, "dbias")
    if want_dinit and d_initial_state is not None:
        _exact(d_initial_state, (nseq, D, L), torch.bfloat16, "d_initial_state")
    if workspace is not None:
        _workspace(workspace)
    dev = _device(("x", "dy", "cu_seqlens", "w", "bias", "initial_state", "state_indices",
                   "status", "dx", "dw", "dbias", "d_initial_state", "workspace"),
                  (x, dy, cu_seqlens, w, bias, initial_state, state_indices,
                   status if state_indices is not None else None, dx, dw,
                   dbias if want_dbias else None, d_initial_state if want_dinit else None,
                   workspace))
    if dx is None:
        dx = torch.empty((total, D), dtype=torch.bfloat16, device=dev)
    if dw is None:
        dw = torch.empty((D, W), dtype=w.dtype, device=dev)
    if want_dbias and dbias is None:
        dbias = torch.empty((D,), dtype=w.dtype, device=dev)
    if want_dinit and d_initial_state is None:
        d_initial_state = torch.empty((nseq, D, L), dtype=torch.bfloat16, device=dev)
    if workspace is None:
        workspace = torch.empty(max(cconv_bwd_varlen_workspace_bytes(total, D, W, dev), 16),
                                dtype=torch.uint8, device=dev)
    rc = _run(dev, load().cconv_bwd_varlen,
              _ptr(x), x.stride(0), _ptr(dy), dy.stride(0), total, D, _ptr(cu_seqlens), nseq,
              _ptr(w), _ptr(bias), _wdt(w), W, act, _ptr(initial_state), _ptr(state_indices), S,
              _ptr(status if state_indices is not None else None), _ptr(dx), _ptr(dw),
              _ptr(dbias if want_dbias else None), _ptr(d_initial_state if want_dinit else None),
              _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream, dev))
    _check(rc, "cconv_bwd_varlen")
    return dx, dw, (dbias if want_dbias else None), (d_initial_state if want_dinit else None)


def cconv_update_ex(x: torch.Tensor, state: torch.Tensor, w: torch.Tensor,
                    bias: torch.Tensor | None = None, state_indices: torch.Tensor | None = None,
                    *, pad_rows: bool = False, cache_seqlens: torch.Tensor | None = None,
                    activation="silu", y: torch.Tensor | None = None,
                    status: torch.Tensor | None = None, stream=None):
    """One decode step with the variants: state [S, D, L] with L = W-1 or W; pad_rows: index
    -1 marks a padding row (no state access, y row not written); cache_seqlens int32 [N]:
    the state is a ring and the token goes to entry cache_seqlens mod L; activation 'silu'
    or None.  Returns (y [N,D], status int32[2] on the device)."""
    _rows(x, "x", 2)
    N, D = x.shape
    W = _weights(w, D)
    _bias(bias, D, w)
    act = _act(activation)
    S, L = _pool(state, D, (W - 1, W))
    if state_indices is not None:
        _int32_vec(state_indices, N, "state_indices")
    elif S < N:
        raise ValueError(f"without state_indices row i uses slot i: state needs S >= N={N}")
    if cache_seqlens is not None:
        _int32_vec(cache_seqlens, N, "cache_seqlens")
    if y is not None:
        _exact(y, (N, D), torch.bfloat16, "y")
    if status is not None:
        _status(status)
    dev = _device(("x", "state", "w", "bias", "state_indices", "cache_seqlens", "y", "status"),
                  (x, state, w, bias, state_indices, cache_seqlens, y, status))
    if y is None:
        y = torch.empty((N, D), dtype=torch.bfloat16, device=dev)
    if status is None:
        status = torch.empty(2, dtype=torch.int32, device=dev)
    rc = _run(dev, load().cconv_update_ex, _ptr(x), N, D, x.stride(0), _ptr(state), S, L,
              _ptr(state_indices), int(bool(pad_rows)), _ptr(cache_seqlens), _ptr(w), _ptr(bias),
              _wdt(w), W, act, _ptr(y), _ptr(status), _stream(stream, dev))
    _check(rc, "cconv_update_ex")
    return y, status


def _parr(ts):
    """Host array of device pointers (NULL for None)."""
    return (ctypes.c_void_p * len(ts))(*[None if t is None else t.data_ptr() for t in ts])


def _iarr(vals):
    return (ctypes.c_int64 * len(vals))(*[int(v) for v in vals])


def _problems(xs, ws, biases, name_x="x"):
    """Checks shared by the multi-problem calls; returns (n, B, T, Ds, W, biases)."""
    xs, ws = list(xs), list(ws)
    n = len(xs)
    if not 1 <= n <= 4:
        raise ValueError(f"1 to 4 problems per launch, got {n}")
    if len(ws) != n:
        raise ValueError(f"one weight per problem: {n} inputs, {len(ws)} weights")
    biases = [None] * n if biases is None else list(biases)
    if len(biases) != n:
        raise ValueError(f"one bias (or None) per problem: {n} inputs, {len(biases)} biases")
    for k, x in enumerate(xs):
        _rows(x, f"{name_x}[{k}]", 3)
    B, T = xs[0].shape[:2]
    if any(tuple(x.shape[:2]) != (B, T) for x in xs):
        raise ValueError("every problem must have the same B and T")
    Ds = [int(x.shape[2]) for x in xs]
    W = _weights(ws[0], Ds[0], "w[0]")
    for k in range(1, n):
        if _weights(ws[k], Ds[k], f"w[{k}]") != W or ws[k].dtype != ws[0].dtype:
            raise ValueError("every problem must have the same W and weight dtype")
    for k in range(n):
        _bias(biases[k], Ds[k], ws[k], f"bias[{k}]")
    return n, int(B), int(T), Ds, W, biases


def _outs(ts, n, shapes, dtypes, name):
    ts = list(ts)
    if len(ts) != n:
        raise ValueError(f"{name}: one tensor per problem, got {len(ts)} for {n}")
    for k in range(n):
        _exact(ts[k], shapes[k], dtypes[k], f"{name}[{k}]")
    return ts


def _listed(*groups):
    """Flattened (tensors, name-of-position) of named lists: groups of (prefix, list)."""
    ts, where = [], []
    for prefix, lst in groups:
        for k, t in enumerate(lst):
            ts.append(t)
            where.append((prefix, k))
    return ts, lambda i: f"{where[i][0]}[{where[i][1]}]"


def cconv_fwd_multi(xs, ws, biases=None, *, ys=None, stream=None):
    """One launch over several [B,T,D_k] problems sharing B, T, W and the weight dtype (the
    q, k, v convolutions of a layer).  Returns the list of outputs."""
    n, B, T, Ds, W, biases = _problems(xs, ws, biases)
    if ys is not None:
        ys = _outs(ys, n, [(B, T, D) for D in Ds], [torch.bfloat16] * n, "ys")
        _disjoint([(f"ys[{k}]", t) for k, t in enumerate(ys)],
                  [(f"x[{k}]", t) for k, t in enumerate(xs)])
    dev = _device(*reversed(_listed(("x", xs), ("w", ws), ("bias", biases), ("ys", ys or []))))
    if ys is None:
        ys = [torch.empty(x.shape, dtype=torch.bfloat16, device=dev) for x in xs]
    rc = _run(dev, load().cconv_fwd_multi, n, _parr(xs), _iarr(Ds),
              _iarr([x.stride(0) for x in xs]), _iarr([x.stride(1) for x in xs]), _parr(ws),
              _parr(biases), _parr(ys), B, T, _wdt(ws[0]), W, _stream(stream, dev))
    _check(rc, "cconv_fwd_multi")
    return ys


def cconv_bwd_multi_workspace_bytes(Ds, B: int, T: int, W: int, device=None) -> int:
    """Workspace cconv_bwd_multi needs on `device` (default: the current CUDA device)."""
    n = ctypes.c_size_t(0)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    _check(_run(dev, load().cconv_bwd_multi_workspace_bytes, len(Ds), _iarr(Ds), B, T, W,
                ctypes.byref(n)), "cconv_bwd_multi_workspace_bytes")
    return int(n.value)


def cconv_bwd_multi(xs, dys, ws, biases=None, *, want_dbias: bool | None = None, dxs=None,
                    dws=None, dbiases=None, workspace=None, stream=None):
    """Backward of cconv_fwd_multi: lists (dx, dw, dbias or None) per problem."""
    n, B, T, Ds, W, biases = _problems(xs, ws, biases)
    dys = list(dys)
    if len(dys) != n:
        raise ValueError(f"one dy per problem: {n} inputs, {len(dys)} gradients")
    for k in range(n):
        _rows(dys[k], f"dy[{k}]", 3)
        if dys[k].shape != xs[k].shape:
            raise ValueError(f"dy[{k}] must have x[{k}]'s shape {tuple(xs[k].shape)}, got "
                             f"{tuple(dys[k].shape)}")
    if want_dbias is None:
        want_dbias = any(b is not None for b in biases) or dbiases is not None
    wdtype = ws[0].dtype
    if dxs is not None:
        dxs = _outs(dxs, n, [(B, T, D) for D in Ds], [torch.bfloat16] * n, "dxs")
        _disjoint([(f"dxs[{k}]", t) for k, t in enumerate(dxs)],
                  [(f"x[{k}]", t) for k, t in enumerate(xs)] +
                  [(f"dy[{k}]", t) for k, t in enumerate(dys)])
    if dws is not None:
        dws = _outs(dws, n, [(D, W) for D in Ds], [wdtype] * n, "dws")
    if want_dbias and dbiases is not None:
        dbiases = _outs(dbiases, n, [(D,) for D in Ds], [wdtype] * n, "dbiases")
    if workspace is not None:
        _workspace(workspace)
    dev = _device(*reversed(_listed(("x", xs), ("dy", dys), ("w", ws), ("bias", biases),
                                    ("dxs", dxs or []), ("dws", dws or []),
                                    ("dbiases", (dbiases or []) if want_dbias else []),
                                    ("workspace", [workspace]))))
    if dxs is None:
        dxs = [torch.empty(x.shape, dtype=torch.bfloat16, device=dev) for x in xs]
    if dws is None:
        dws = [torch.empty((D, W), dtype=wdtype, device=dev) for D in Ds]
    if want_dbias and dbiases is None:
        dbiases = [torch.empty((D,), dtype=wdtype, device=dev) for D in Ds]
    if workspace is None:
        workspace = torch.empty(cconv_bwd_multi_workspace_bytes(Ds, B, T, W, dev),
                                dtype=torch.uint8, device=dev)
    rc = _run(dev, load().cconv_bwd_multi,
              n, _parr(xs), _iarr([x.stride(0) for x in xs]), _iarr([x.stride(1) for x in xs]),
              _parr(dys), _iarr([d.stride(0) for d in dys]), _iarr([d.stride(1) for d in dys]),
              _iarr(Ds), _parr(ws), _parr(biases), _parr(dxs), _parr(dws),
              _parr(dbiases) if want_dbias else None, B, T, _wdt(ws[0]), W, _ptr(workspace),
              workspace.numel() * workspace.element_size(), _stream(stream, dev))
    _check(rc, "cconv_bwd_multi")
    return dxs, dws, (dbiases if want_dbias else [None] * n)


def cconv_status_str(status: int) -> str:
    return load().cconv_status_str(status).decode()


def cconv_device_fault() -> int:
    v = ctypes.c_int32(0)
    _check(load().cconv_device_fault(ctypes.byref(v)), "cconv_device_fault")
    return int(v.value)


def describe(fn) -> list[dict]:
    """The kernels fn() would launch through this library, with their registers per thread,
    local (spill) bytes, shared memory, threads per CTA, grid size and resident CTAs per SM;
    fn runs with launches recorded instead of enqueued (nothing runs on the GPU)."""
    lib = load()
    _check(lib.cconv_describe_begin(), "cconv_describe_begin")
    try:
        fn()
    finally:
        buf = (KernelDesc * 16)()
        n = ctypes.c_int(0)
        rc = lib.cconv_describe_end(buf, 16, ctypes.byref(n))
    _check(rc, "cconv_describe_end")
    return [{f: (getattr(d, f).decode() if f == "name" else getattr(d, f))
             for f, _ in KernelDesc._fields_} for d in buf[:min(n.value, 16)]]
