"""Write the regression fixtures in this folder.  Calls only the oracle.

    python tests/golden/make_golden.py

The pages print no worked numeric example for the convolution, so these fixtures are not
pins of the oracle; they freeze its outputs on two tiny seeded cases so that any later
change to the oracle's arithmetic shows up as a diff that has to be justified.
"""
from __future__ import annotations

import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from depthwise_causal_short_gb300 import inputs  # noqa: E402


def _case_fwd_bwd():
    B, T, D, W = 1, 8, 4, 4
    x, dy, w, b = inputs.fwd_bwd_inputs(B, T, D, W, bias=True, seed=11)
    xd, dyd, wd, bd = (t.double().numpy() for t in (x, dy, w, b))
    y = oracle.fwd(xd, wd, bd)
    dx, dw, db = oracle.bwd(xd, dyd, wd, bd)
    return {
        "what": "forward + backward, B=1 T=8 D=4 W=4, bias; inputs from "
                "inputs.fwd_bwd_inputs(seed=11)",
        "source": "kernel-fun 0.2.0.dev1 wheel, kernel_fun/cconv/_kernels/strip.py "
                  "(_tap, _silu, _dsilu, _bwd4) -- definitions restated by the oracle",
        "shape": [B, T, D, W],
        "x": xd.ravel().tolist(), "dy": dyd.ravel().tolist(),
        "w": wd.ravel().tolist(), "bias": bd.ravel().tolist(),
        "y": y.ravel().tolist(), "dx": dx.ravel().tolist(),
        "dw": dw.ravel().tolist(), "dbias": db.ravel().tolist(),
    }


def _case_decode():
    S, N, D, W = 6, 3, 4, 4
    state, xr, idx, w, b = inputs.decode_inputs(S, N, D, W, bias=True, n_x=1, seed=12)
    import torch
    sb = state.view(torch.int16).numpy().view(np.uint16)
    xb = xr[0].view(torch.int16).numpy().view(np.uint16)
    status, y, new_state = oracle.update(xb, sb, idx.numpy(), w.double().numpy(),
                                         b.double().numpy())
    assert status == 0
    return {
        "what": "one decode update, S=6 N=3 D=4 W=4, bias; inputs from "
                "inputs.decode_inputs(seed=12)",
        "source": "Add experimental causal conv1d decode update - #797 "
                  "(NVIDIA/cudnn-frontend), PR summary -- restated by the oracle",
        "shape": [S, N, D, W],
        "state_bits": sb.ravel().tolist(), "x_bits": xb.ravel().tolist(),
        "state_indices": idx.tolist(), "w": w.double().numpy().ravel().tolist(),
        "bias": b.double().numpy().ravel().tolist(),
        "y": y.ravel().tolist(), "new_state_bits": new_state.ravel().tolist(),
    }


def main():
    for name, fn in (("oracle_fwd_bwd_b1_t8_d4_w4.json", _case_fwd_bwd),
                     ("oracle_decode_s6_n3_d4_w4.json", _case_decode)):
        with open(os.path.join(HERE, name), "w") as f:
            json.dump(fn(), f, indent=0)
            f.write("\n")
        print("wrote", name)


if __name__ == "__main__":
    main()
