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
                                     _INT, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
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
    if path is None:
        _lib = lib
    return lib


def header_functions() -> list[str]:
    """Names of the functions include/cconv.h declares (CCONV_API ... name(...))."""
    text = (_build.INCLUDE / "cconv.h").read_text()
    return re.findall(r"CCONV_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


# ---------------------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------------------

def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _wdt(w: torch.Tensor) -> int:
    if w.dtype == torch.float32:
        return CCONV_F32
    if w.dtype == torch.bfloat16:
        return CCONV_BF16
    raise TypeError(f"weight dtype must be float32 or bfloat16, got {w.dtype}")


def _check(rc: int, call: str):
    if rc != 0:
        raise CConvError(rc, call)


def _bf16_rows(t: torch.Tensor, name: str):
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    if t.dim() != 3 or t.stride(2) != 1:
        raise ValueError(f"{name} must be [B,T,D] with channel stride 1")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


# ---------------------------------------------------------------------------------------
# the three calls
# ---------------------------------------------------------------------------------------

def cconv_fwd(x: torch.Tensor, w: torch.Tensor, bias: torch.Tensor | None = None, *,
              y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y = silu(bias + causal depthwise conv(x, w)); x [B,T,D] bf16, w [D,W]."""
    _bf16_rows(x, "x")
    B, T, D = x.shape
    W = w.shape[1]
    if y is None:
        y = torch.empty((B, T, D), dtype=torch.bfloat16, device=x.device)
    rc = load().cconv_fwd(_ptr(x), B, T, D, x.stride(0), x.stride(1), _ptr(w), _ptr(bias),
                          _wdt(w), W, _ptr(y), _stream(stream))
    _check(rc, "cconv_fwd")
    return y


def cconv_bwd_workspace_bytes(B: int, T: int, D: int, W: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load().cconv_bwd_workspace_bytes(B, T, D, W, ctypes.byref(n)), "cconv_bwd_workspace_bytes")
    return int(n.value)


def cconv_bwd(x: torch.Tensor, dy: torch.Tensor, w: torch.Tensor,
              bias: torch.Tensor | None = None, *, want_dbias: bool | None = None,
              dx: torch.Tensor | None = None, dw: torch.Tensor | None = None,
              dbias: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
              stream=None):
    """(dx, dw, dbias) for upstream gradient dy; dbias is None unless wanted (default:
    when a bias is given)."""
    _bf16_rows(x, "x")
    _bf16_rows(dy, "dy")
    B, T, D = x.shape
    W = w.shape[1]
    if want_dbias is None:
        want_dbias = bias is not None or dbias is not None
    if dx is None:
        dx = torch.empty((B, T, D), dtype=torch.bfloat16, device=x.device)
    if dw is None:
        dw = torch.empty((D, W), dtype=w.dtype, device=x.device)
    if want_dbias and dbias is None:
        dbias = torch.empty((D,), dtype=w.dtype, device=x.device)
    if workspace is None:
        workspace = torch.empty(cconv_bwd_workspace_bytes(B, T, D, W), dtype=torch.uint8,
                                device=x.device)
    rc = load().cconv_bwd(_ptr(x), x.stride(0), x.stride(1), _ptr(dy), dy.stride(0), dy.stride(1),
                          B, T, D, _ptr(w), _ptr(bias), _wdt(w), W, _ptr(dx), _ptr(dw),
                          _ptr(dbias if want_dbias else None), _ptr(workspace),
                          workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "cconv_bwd")
    return dx, dw, (dbias if want_dbias else None)


def cconv_bwd_noalloc(x: torch.Tensor, dy: torch.Tensor, w: torch.Tensor,
                      bias: torch.Tensor | None = None, *, dx: torch.Tensor,
                      dw: torch.Tensor, dbias: torch.Tensor | None = None, stream=None):
    """cconv_bwd for callers that cannot allocate device memory at this point: every output
    must be passed in, and the partial sums use the library's fixed 8 MiB device scratch
    array instead of a workspace.  Calls that overlap on the GPU race on that array."""
    _bf16_rows(x, "x")
    _bf16_rows(dy, "dy")
    B, T, D = x.shape
    rc = load().cconv_bwd_noalloc(_ptr(x), x.stride(0), x.stride(1), _ptr(dy), dy.stride(0),
                                  dy.stride(1), B, T, D, _ptr(w), _ptr(bias), _wdt(w), w.shape[1],
                                  _ptr(dx), _ptr(dw), _ptr(dbias), _stream(stream))
    _check(rc, "cconv_bwd_noalloc")
    return dx, dw, dbias


def cconv_update(x: torch.Tensor, state: torch.Tensor, w: torch.Tensor,
                 bias: torch.Tensor | None = None, state_indices: torch.Tensor | None = None,
                 *, y: torch.Tensor | None = None, status: torch.Tensor | None = None,
                 stream=None):
    """One decode step: (y [N,D], status int32[2] on the device).  state [S,D,W-1] is
    updated in place unless status[0] reports CCONV_ERR_INDEX."""
    if x.dtype != torch.bfloat16 or x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be [N,D] bfloat16 with channel stride 1")
    N, D = x.shape
    W = w.shape[1]
    if state.dtype != torch.bfloat16 or not state.is_contiguous():
        raise ValueError("state must be a contiguous [S,D,W-1] bfloat16 tensor")
    S = state.shape[0]
    if y is None:
        y = torch.empty((N, D), dtype=torch.bfloat16, device=x.device)
    if status is None:
        status = torch.empty(2, dtype=torch.int32, device=x.device)
    if state_indices is not None and state_indices.dtype != torch.int32:
        raise TypeError("state_indices must be int32")
    rc = load().cconv_update(_ptr(x), N, D, x.stride(0), _ptr(state), S, _ptr(state_indices),
                             _ptr(w), _ptr(bias), _wdt(w), W, _ptr(y), _ptr(status),
                             _stream(stream))
    _check(rc, "cconv_update")
    return y, status


def _act(activation) -> int:
    if activation in ("silu", "swish"):
        return CCONV_ACT_SILU
    if activation is None or activation == "none":
        return CCONV_ACT_NONE
    raise ValueError(f"activation must be 'silu' or None, got {activation!r}")


def _packed_rows(t: torch.Tensor, name: str):
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be [total, D] with channel stride 1")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


def _cu(cu_seqlens: torch.Tensor) -> torch.Tensor:
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or not cu_seqlens.is_cuda:
        raise TypeError("cu_seqlens must be a 1-D int32 CUDA tensor")
    if not cu_seqlens.is_contiguous():
        raise ValueError("cu_seqlens must be contiguous")
    return cu_seqlens


def _state(t: torch.Tensor | None, name: str):
    if t is None:
        return
    if t.dtype != torch.bfloat16 or t.dim() != 3 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous [S, D, W-1] bfloat16 tensor")


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
    _packed_rows(x, "x")
    total, D = x.shape
    cu = _cu(cu_seqlens)
    nseq = cu.numel() - 1
    W = w.shape[1]
    _state(initial_state, "initial_state")
    if final_state is True:
        final_state = torch.empty((nseq, D, W - 1), dtype=torch.bfloat16, device=x.device)
    elif final_state is False:
        final_state = None
    _state(final_state, "final_state")
    if state_indices is not None:
        if state_indices.dtype != torch.int32:
            raise TypeError("state_indices must be int32")
        if status is None:
            status = torch.empty(2, dtype=torch.int32, device=x.device)
    pools = [t for t in (initial_state, final_state) if t is not None]
    S = pools[0].shape[0] if pools else nseq
    if y is None:
        y = torch.empty((total, D), dtype=torch.bfloat16, device=x.device)
    rc = load().cconv_fwd_varlen(_ptr(x), total, D, x.stride(0), _ptr(cu), nseq, _ptr(w),
                                 _ptr(bias), _wdt(w), W, _act(activation), _ptr(initial_state),
                                 _ptr(final_state), _ptr(state_indices), S, _ptr(status), _ptr(y),
                                 _stream(stream))
    _check(rc, "cconv_fwd_varlen")
    return y, final_state, (status if state_indices is not None else None)


def cconv_bwd_varlen_workspace_bytes(total: int, D: int, W: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load().cconv_bwd_varlen_workspace_bytes(total, D, W, ctypes.byref(n)),
           "cconv_bwd_varlen_workspace_bytes")
    return int(n.value)


def cconv_bwd_varlen(x: torch.Tensor, dy: torch.Tensor, cu_seqlens: torch.Tensor,
                     w: torch.Tensor, bias: torch.Tensor | None = None, *, activation="silu",
                     initial_state: torch.Tensor | None = None, want_dbias: bool | None = None,
                     want_dinit: bool | None = None, dx: torch.Tensor | None = None,
                     dw: torch.Tensor | None = None, dbias: torch.Tensor | None = None,
                     d_initial_state: torch.Tensor | None = None,
                     workspace: torch.Tensor | None = None, stream=None):
    """Packed-sequence backward: (dx, dw, dbias or None, d_initial_state or None)."""
    _packed_rows(x, "x")
    _packed_rows(dy, "dy")
    total, D = x.shape
    cu = _cu(cu_seqlens)
    nseq = cu.numel() - 1
    W = w.shape[1]
    _state(initial_state, "initial_state")
    if want_dbias is None:
        want_dbias = bias is not None or dbias is not None
    if want_dinit is None:
        want_dinit = initial_state is not None or d_initial_state is not None
    if dx is None:
        dx = torch.empty((total, D), dtype=torch.bfloat16, device=x.device)
    if dw is None:
        dw = torch.empty((D, W), dtype=w.dtype, device=x.device)
    if want_dbias and dbias is None:
        dbias = torch.empty((D,), dtype=w.dtype, device=x.device)
    if want_dinit and d_initial_state is None:
        d_initial_state = torch.empty((nseq, D, W - 1), dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = torch.empty(max(cconv_bwd_varlen_workspace_bytes(total, D, W), 16),
                                dtype=torch.uint8, device=x.device)
    rc = load().cconv_bwd_varlen(
        _ptr(x), x.stride(0), _ptr(dy), dy.stride(0), total, D, _ptr(cu), nseq, _ptr(w),
        _ptr(bias), _wdt(w), W, _act(activation), _ptr(initial_state), _ptr(dx), _ptr(dw),
        _ptr(dbias if want_dbias else None), _ptr(d_initial_state if want_dinit else None),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
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
    if x.dtype != torch.bfloat16 or x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be [N,D] bfloat16 with channel stride 1")
    N, D = x.shape
    W = w.shape[1]
    if state.dtype != torch.bfloat16 or state.dim() != 3 or not state.is_contiguous():
        raise ValueError("state must be a contiguous [S,D,L] bfloat16 tensor")
    S, L = state.shape[0], state.shape[2]
    if y is None:
        y = torch.empty((N, D), dtype=torch.bfloat16, device=x.device)
    if status is None:
        status = torch.empty(2, dtype=torch.int32, device=x.device)
    if state_indices is not None and state_indices.dtype != torch.int32:
        raise TypeError("state_indices must be int32")
    if cache_seqlens is not None and (cache_seqlens.dtype != torch.int32 or
                                      not cache_seqlens.is_contiguous()):
        raise TypeError("cache_seqlens must be a contiguous int32 tensor")
    rc = load().cconv_update_ex(_ptr(x), N, D, x.stride(0), _ptr(state), S, L,
                                _ptr(state_indices), int(bool(pad_rows)), _ptr(cache_seqlens),
                                _ptr(w), _ptr(bias), _wdt(w), W, _act(activation), _ptr(y),
                                _ptr(status), _stream(stream))
    _check(rc, "cconv_update_ex")
    return y, status


def _parr(ts):
    """Host array of device pointers (NULL for None)."""
    return (ctypes.c_void_p * len(ts))(*[None if t is None else t.data_ptr() for t in ts])


def _iarr(vals):
    return (ctypes.c_int64 * len(vals))(*[int(v) for v in vals])


def cconv_fwd_multi(xs, ws, biases=None, *, ys=None, stream=None):
    """One launch over several [B,T,D_k] problems sharing B, T, W and the weight dtype (the
    q, k, v convolutions of a layer).  Returns the list of outputs."""
    n = len(xs)
    for k, x in enumerate(xs):
        _bf16_rows(x, f"x[{k}]")
    B, T = xs[0].shape[:2]
    if any(x.shape[:2] != (B, T) for x in xs):
        raise ValueError("every problem must have the same B and T")
    W = ws[0].shape[1]
    if ys is None:
        ys = [torch.empty(x.shape, dtype=torch.bfloat16, device=x.device) for x in xs]
    biases = biases if biases is not None else [None] * n
    rc = load().cconv_fwd_multi(n, _parr(xs), _iarr([x.shape[2] for x in xs]),
                                _iarr([x.stride(0) for x in xs]), _iarr([x.stride(1) for x in xs]),
                                _parr(ws), _parr(biases), _parr(ys), B, T, _wdt(ws[0]), W,
                                _stream(stream))
    _check(rc, "cconv_fwd_multi")
    return ys


def cconv_bwd_multi_workspace_bytes(Ds, B: int, T: int, W: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load().cconv_bwd_multi_workspace_bytes(len(Ds), _iarr(Ds), B, T, W, ctypes.byref(n)),
           "cconv_bwd_multi_workspace_bytes")
    return int(n.value)


def cconv_bwd_multi(xs, dys, ws, biases=None, *, want_dbias: bool | None = None, dxs=None,
                    dws=None, dbiases=None, workspace=None, stream=None):
    """Backward of cconv_fwd_multi: lists (dx, dw, dbias or None) per problem."""
    n = len(xs)
    for k in range(n):
        _bf16_rows(xs[k], f"x[{k}]")
        _bf16_rows(dys[k], f"dy[{k}]")
    B, T = xs[0].shape[:2]
    W = ws[0].shape[1]
    Ds = [x.shape[2] for x in xs]
    biases = biases if biases is not None else [None] * n
    if want_dbias is None:
        want_dbias = any(b is not None for b in biases) or dbiases is not None
    if dxs is None:
        dxs = [torch.empty(x.shape, dtype=torch.bfloat16, device=x.device) for x in xs]
    if dws is None:
        dws = [torch.empty((D, W), dtype=w.dtype, device=w.device) for D, w in zip(Ds, ws)]
    if want_dbias and dbiases is None:
        dbiases = [torch.empty((D,), dtype=w.dtype, device=w.device) for D, w in zip(Ds, ws)]
    if workspace is None:
        workspace = torch.empty(cconv_bwd_multi_workspace_bytes(Ds, B, T, W), dtype=torch.uint8,
                                device=xs[0].device)
    rc = load().cconv_bwd_multi(
        n, _parr(xs), _iarr([x.stride(0) for x in xs]), _iarr([x.stride(1) for x in xs]),
        _parr(dys), _iarr([d.stride(0) for d in dys]), _iarr([d.stride(1) for d in dys]),
        _iarr(Ds), _parr(ws), _parr(biases), _parr(dxs), _parr(dws),
        _parr(dbiases) if want_dbias else None, B, T, _wdt(ws[0]), W, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "cconv_bwd_multi")
    return dxs, dws, (dbiases if want_dbias else [None] * n)


def cconv_status_str(status: int) -> str:
    return load().cconv_status_str(status).decode()


def cconv_device_fault() -> int:
    v = ctypes.c_int32(0)
    _check(load().cconv_device_fault(ctypes.byref(v)), "cconv_device_fault")
    return int(v.value)
