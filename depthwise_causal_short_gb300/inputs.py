"""Seeded synthetic inputs for the causal short convolution workloads.

This module only draws random numbers; it holds none of the convolution's arithmetic.
It is the one piece the CUDA path's tests / benchmark and the CPU oracle both use.

Recipe (every workload): a CPU ``torch.Generator`` seeded with ``seed`` (0 by default),
values drawn in fp32 and cast round-to-nearest-even to bf16 for activations, kept fp32 (or
cast to bf16) for weights and bias.  Draw order is fixed: x, dy, w, bias for the
training-shaped workloads; state, x ring, slot permutation, w, bias for the decode one.

  x, dy  ~ N(0, 1)          activations / upstream gradient, [B, T, D]
  w      ~ U(-0.5, 0.5)     depthwise taps, [D, W]
  bias   ~ U(-0.1, 0.1)     [D]
  state  ~ N(0, 1)          decode state pool, [S, D, W-1]
  state_indices              the first N entries of a random permutation of range(S)

Packed sequences (``varlen_inputs``): lengths from ``seqlen_mix`` -- log-uniform weights
over a 32x range, scaled to the requested total (a ragged mix of long and short sequences;
the caller may add empty and one-row sequences explicitly), then x, dy ~ N(0,1) [total, D],
w, bias as above, initial states ~ N(0,1) [nseq, D, W-1], drawn in that order.

The shapes follow the production call of the kernel-fun cconv package (B=16 T=8192 D=2048
W=4, bf16 x / fp32 weight; kernel-fun 0.2.0.dev1 wheel, kernel_fun/cconv/__init__.py) and
the decode batch of the cuDNN decode-update PR; there is no dataset behind either.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class FwdBwdShape:
    name: str
    B: int
    T: int
    D: int
    W: int
    bias: bool


@dataclass(frozen=True)
class DecodeShape:
    name: str
    S: int  # slots in the state pool
    N: int  # active rows per step
    D: int
    W: int
    bias: bool
    steps: int


# The training-shaped workloads: a tiny one the oracle finishes instantly, a mid-size
# multi-head one, the production-length one, and ragged edge shapes (T and D tails, W<4).
FWD_BWD_SHAPES = [
    FwdBwdShape("b1_t64_d128_w4", 1, 64, 128, 4, True),
    FwdBwdShape("b8_t1024_d2048_w4", 8, 1024, 2048, 4, True),
    FwdBwdShape("b2_t8192_d4096_w4_nobias", 2, 8192, 4096, 4, False),
    FwdBwdShape("b4_t777_d1000_w2", 4, 777, 1000, 2, True),
    FwdBwdShape("b4_t777_d1000_w3", 4, 777, 1000, 3, True),
]
PROD = FWD_BWD_SHAPES[2]

DECODE_SHAPE = DecodeShape("s512_n256_d4096_w4", S=512, N=256, D=4096, W=4, bias=True,
                           steps=1000)


def fwd_bwd_inputs(B: int, T: int, D: int, W: int, bias: bool = True,
                   wdtype: torch.dtype = torch.float32, seed: int = 0):
    """(x, dy, w, bias) on the CPU: x, dy bf16 [B,T,D]; w [D,W] and bias [D] in wdtype."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(B, T, D, generator=g).to(torch.bfloat16)
    dy = torch.randn(B, T, D, generator=g).to(torch.bfloat16)
    w = (torch.rand(D, W, generator=g) - 0.5).to(wdtype)
    b = ((torch.rand(D, generator=g) - 0.5) * 0.2).to(wdtype) if bias else None
    return x, dy, w, b


def decode_inputs(S: int, N: int, D: int, W: int, bias: bool = True, n_x: int = 8,
                  wdtype: torch.dtype = torch.float32, seed: int = 0):
    """(state [S,D,W-1] bf16, x ring [n_x,N,D] bf16, state_indices [N] int32, w, bias)."""
    g = torch.Generator().manual_seed(seed)
    state = torch.randn(S, D, W - 1, generator=g).to(torch.bfloat16)
    x = torch.randn(n_x, N, D, generator=g).to(torch.bfloat16)
    idx = torch.randperm(S, generator=g)[:N].to(torch.int32)
    w = (torch.rand(D, W, generator=g) - 0.5).to(wdtype)
    b = ((torch.rand(D, generator=g) - 0.5) * 0.2).to(wdtype) if bias else None
    return state, x, idx, w, b


def seqlen_mix(total: int, nseq: int, seed: int = 0, spread: float = 32.0) -> list[int]:
    """nseq lengths summing to total, log-uniform over a `spread`-fold range (each >= 1
    when total >= nseq)."""
    g = torch.Generator().manual_seed(seed)
    wts = torch.exp(torch.rand(nseq, generator=g, dtype=torch.float64) * float(torch.log(
        torch.tensor(spread, dtype=torch.float64))))
    raw = wts / wts.sum() * total
    lens = [max(1, int(v)) if total >= nseq else int(v) for v in raw]
    lens[-1] += total - sum(lens)
    while lens[-1] < (1 if total >= nseq else 0):   # give rows back from the longest
        k = max(range(nseq - 1), key=lambda i: lens[i])
        lens[k] -= 1
        lens[-1] += 1
    return lens


def cu_of(lengths) -> torch.Tensor:
    """int32 row offsets [0, l0, l0+l1, ...] (CPU)."""
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32)


def varlen_inputs(lengths, D: int, W: int, bias: bool = True, wdtype: torch.dtype = torch.float32,
                  seed: int = 0):
    """(x [total,D], dy [total,D] bf16, cu int32 [nseq+1], w, bias, initial state
    [nseq,D,W-1] bf16), all on the CPU."""
    g = torch.Generator().manual_seed(seed)
    cu = cu_of(lengths)
    total = int(cu[-1])
    x = torch.randn(total, D, generator=g).to(torch.bfloat16)
    dy = torch.randn(total, D, generator=g).to(torch.bfloat16)
    w = (torch.rand(D, W, generator=g) - 0.5).to(wdtype)
    b = ((torch.rand(D, generator=g) - 0.5) * 0.2).to(wdtype) if bias else None
    init = torch.randn(len(lengths), D, W - 1, generator=g).to(torch.bfloat16)
    return x, dy, cu, w, b, init
