"""Runs one library call at its benchmark workload a few times, for profilers.

    python -m depthwise_causal_short_gb300.profile_calls CALL [--calls N] [--rows-div K]

CALL is one of fwd, bwd, update, fwd_varlen, bwd_varlen, fwd_multi, bwd_multi.  The inputs
are the benchmark's (seeded, synthetic, resident on cuda:0 before the first call); two input
sets alternate so that no call reads what the previous one touched.  Nothing is timed and
nothing else is launched, so a profiler's launch list holds only the chosen call's kernels
(plus torch's own input set-up before them).  --rows-div K divides T by K (a smaller case
of the same kernels, e.g. to check how many passes a profiler's metrics take).
"""
from __future__ import annotations

import argparse

import torch

from . import _build, binding as cc, inputs

B, D, W = inputs.PROD.B, inputs.PROD.D, inputs.PROD.W
VL_NSEQ = 16
QKV_D = [D // 4, D // 4, D // 2]


def _calls(name: str, dev, T: int):
    """Returns fn(i) that issues the i-th call of `name` (T rows per batch row)."""
    if name in ("fwd", "bwd"):
        sets = []
        for k in range(2):
            x, dy, w, _ = inputs.fwd_bwd_inputs(B, T, D, W, False, seed=k)
            sets.append((x.to(dev), dy.to(dev), torch.empty_like(x, device=dev)))
        wg = w.to(dev)
        dw = torch.empty_like(wg)
        db = torch.empty(D, dtype=wg.dtype, device=dev)
        ws = torch.empty(cc.cconv_bwd_workspace_bytes(B, T, D, W), dtype=torch.uint8, device=dev)
        if name == "fwd":
            return lambda i: cc.cconv_fwd(sets[i % 2][0], wg, None, y=sets[i % 2][2])
        return lambda i: cc.cconv_bwd(sets[i % 2][0], sets[i % 2][1], wg, None, want_dbias=True,
                                      dx=sets[i % 2][2], dw=dw, dbias=db, workspace=ws)
    if name == "update":
        sh = inputs.DECODE_SHAPE
        st, xr, idx, w, b = (t.to(dev) for t in inputs.decode_inputs(sh.S, sh.N, sh.D, sh.W,
                                                                       sh.bias, n_x=8))
        y = torch.empty(sh.N, sh.D, dtype=torch.bfloat16, device=dev)
        status = torch.empty(2, dtype=torch.int32, device=dev)
        return lambda i: cc.cconv_update(xr[i % 8], st, w, b, idx, y=y, status=status)
    if name in ("fwd_varlen", "bwd_varlen"):
        lens = inputs.seqlen_mix(B * T, VL_NSEQ, seed=0)
        sets = []
        for k in range(2):
            x, dy, cu, w, _, init = inputs.varlen_inputs(lens, D, W, bias=False, seed=k)
            sets.append((x.to(dev), dy.to(dev), init.to(dev), torch.empty_like(x, device=dev)))
        cug, wg = cu.to(dev), w.to(dev)
        fin = torch.empty_like(sets[0][2])
        dinit = torch.empty_like(sets[0][2])
        dw = torch.empty_like(wg)
        db = torch.empty(D, dtype=wg.dtype, device=dev)
        ws = torch.empty(cc.cconv_bwd_varlen_workspace_bytes(B * T, D, W), dtype=torch.uint8,
                         device=dev)
        if name == "fwd_varlen":
            return lambda i: cc.cconv_fwd_varlen(sets[i % 2][0], cug, wg, None,
                                                 initial_state=sets[i % 2][2], final_state=fin,
                                                 y=sets[i % 2][3])
        return lambda i: cc.cconv_bwd_varlen(sets[i % 2][0], sets[i % 2][1], cug, wg, None,
                                             initial_state=sets[i % 2][2], want_dbias=True,
                                             dx=sets[i % 2][3], dw=dw, dbias=db,
                                             d_initial_state=dinit, workspace=ws)
    if name in ("fwd_multi", "bwd_multi"):
        sets = []
        for k in range(2):
            pr = [inputs.fwd_bwd_inputs(B, T, d, W, False, seed=10 * k + j)
                  for j, d in enumerate(QKV_D)]
            sets.append(([p[0].to(dev) for p in pr], [p[1].to(dev) for p in pr],
                         [torch.empty(B, T, d, dtype=torch.bfloat16, device=dev) for d in QKV_D]))
        ws_ = [inputs.fwd_bwd_inputs(1, 1, d, W, False, seed=j)[2].to(dev)
               for j, d in enumerate(QKV_D)]
        dws = [torch.empty_like(w) for w in ws_]
        dbs = [torch.empty(w.shape[0], dtype=w.dtype, device=dev) for w in ws_]
        work = torch.empty(cc.cconv_bwd_multi_workspace_bytes(QKV_D, B, T, W), dtype=torch.uint8,
                           device=dev)
        if name == "fwd_multi":
            return lambda i: cc.cconv_fwd_multi(sets[i % 2][0], ws_, ys=sets[i % 2][2])
        return lambda i: cc.cconv_bwd_multi(sets[i % 2][0], sets[i % 2][1], ws_, want_dbias=True,
                                            dxs=sets[i % 2][2], dws=dws, dbiases=dbs,
                                            workspace=work)
    raise SystemExit(f"unknown call {name!r}")


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("call", choices=["fwd", "bwd", "update", "fwd_varlen", "bwd_varlen",
                                     "fwd_multi", "bwd_multi"])
    ap.add_argument("--calls", type=int, default=6)
    ap.add_argument("--rows-div", type=int, default=1)
    args = ap.parse_args(argv)
    if not _build.up_to_date():
        _build.build()
    cc.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    fn = _calls(args.call, dev, inputs.PROD.T // max(1, args.rows_div))
    torch.cuda.synchronize()
    for i in range(args.calls):
        fn(i)
    torch.cuda.synchronize()
    print(f"{args.call}: {args.calls} calls done")


if __name__ == "__main__":
    main()
