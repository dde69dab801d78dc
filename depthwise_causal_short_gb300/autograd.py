"""causal_conv1d: the library's calls behind one differentiable PyTorch entry point.

The keyword set follows fla's causal_conv1d as the kernel-fun 0.2.0.dev1 wheel forwards it
(kernel_fun/_common/compat.py: x, weight, bias, initial_state, output_final_state,
activation, cu_seqlens) and the return contract of that package's entry point
(kernel_fun/cconv/__init__.py: y, and the final state when asked for).  Only marshalling
and dispatch live here: the forward is one cconv_fwd or cconv_fwd_varlen call, and the
backward one cconv_bwd or cconv_bwd_varlen call.  Nothing is computed in PyTorch.

Layouts: x [B, T, D] bf16 (B = 1 with cu_seqlens, whose rows are the packed sequences);
weight [D, W] fp32 or bf16; bias [D] or None; states [N, D, W-1] bf16 (N = B, or the number
of sequences), oldest entry first, the decode pool's layout.  The final state is returned
as a constant (no gradient flows into it); gradients flow to x, weight, bias and
initial_state.
"""
from __future__ import annotations

import torch

from . import binding as cc


def _packed_cu(x: torch.Tensor, cu_seqlens: torch.Tensor | None) -> torch.Tensor:
    """cu_seqlens for the packed calls: the given one, or one sequence per batch row."""
    B, T, _ = x.shape
    if cu_seqlens is not None:
        if B != 1:
            raise ValueError("with cu_seqlens, x must be [1, total, D]")
        return cu_seqlens.to(torch.int32)
    return torch.arange(0, (B + 1) * T, T, dtype=torch.int32, device=x.device)


class _CausalConv1d(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, weight, bias, initial_state, cu_seqlens, activation, output_final_state):
        batched = cu_seqlens is None and initial_state is None and activation == "silu" \
            and not output_final_state
        final = None
        if batched:
            y = cc.cconv_fwd(x, weight, bias)
            cu = None
        else:
            if not x.is_contiguous():
                raise ValueError("the packed path needs a contiguous x")
            cu = _packed_cu(x, cu_seqlens)
            y2, final, _ = cc.cconv_fwd_varlen(x.view(-1, x.shape[2]), cu, weight, bias,
                                               activation=activation,
                                               initial_state=initial_state,
                                               final_state=bool(output_final_state))
            y = y2.view(x.shape)
        ctx.batched = batched
        ctx.activation = activation
        ctx.save_for_backward(x, weight, bias, initial_state, cu)
        if final is not None:
            ctx.mark_non_differentiable(final)
        return y, final

    @staticmethod
    def backward(ctx, dy, _dfinal):
        x, weight, bias, initial_state, cu = ctx.saved_tensors
        need_x, need_w, need_b, need_s = ctx.needs_input_grad[:4]
        dy = dy.contiguous()
        if ctx.batched:
            dx, dw, db = cc.cconv_bwd(x, dy, weight, bias, want_dbias=need_b)
            ds = None
        else:
            D = x.shape[2]
            dx, dw, db, ds = cc.cconv_bwd_varlen(
                x.view(-1, D), dy.view(-1, D), cu, weight, bias, activation=ctx.activation,
                initial_state=initial_state, want_dbias=need_b,
                want_dinit=initial_state is not None and need_s)
            dx = dx.view(x.shape)
        return (dx if need_x else None, dw if need_w else None, db if need_b else None,
                ds if need_s else None, None, None, None)


def causal_conv1d(x: torch.Tensor, weight: torch.Tensor, bias: torch.Tensor | None = None,
                  initial_state: torch.Tensor | None = None, output_final_state: bool = False,
                  activation: str | None = "silu", cu_seqlens: torch.Tensor | None = None):
    """y = act(bias + causal depthwise conv(x, weight)) per sequence; returns (y, final_state)
    with final_state None unless output_final_state.  See the module docstring for layouts."""
    if activation not in ("silu", "swish", None, "none"):
        raise ValueError(f"activation must be 'silu' or None, got {activation!r}")
    if not isinstance(x, torch.Tensor) or x.dim() != 3:
        raise ValueError("x must be a [B, T, D] tensor")
    if initial_state is not None:
        n = x.shape[0] if cu_seqlens is None else cu_seqlens.numel() - 1
        if not isinstance(initial_state, torch.Tensor) or initial_state.dim() != 3 or \
                initial_state.shape[0] != n:
            raise ValueError(f"initial_state must be [{n}, D, W-1]: one state per sequence")
    act = "silu" if activation in ("silu", "swish") else None
    return _CausalConv1d.apply(x, weight, bias, initial_state, cu_seqlens, act,
                               output_final_state)
