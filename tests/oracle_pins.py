"""Pins of the fp64 oracle against facts fixed by the pages and by mathematics.

Each pin takes an ``oracle.Oracle`` handle and raises AssertionError on a mismatch, so the
same pins run against the real oracle (where all must pass) and against deliberately
broken copies of it (where at least one must fail; see test_oracle_mutants.py).

What pins what:
  fwd  - scipy.signal.lfilter (a library FIR filter with zero initial conditions) per
         channel; torch float64 grouped conv1d; W=1 elementwise; impulse and constant
         closed forms; silu(0) = 0.
  bwd  - torch float64 autograd through grouped conv1d + SiLU; central finite differences
         of L = sum(y * dy) in fp64; closed form at z = 0 (g = dy / 2).
  taps - zero-weighted padded taps reproduce the narrower width (kernel-fun 0.2.0.dev1
         wheel, cconv/_kernels/strip.py module docstring: narrow W is zero-weighted taps).
  decode - T single-token updates from a zero state reproduce every row of the full
         forward, and the final state is the last W-1 rows of x, bit for bit;
         index validation against a set-based definition, exhaustively on tiny pools;
         invalid indices leave the pool untouched ("fail closed", cuDNN decode-update PR).
"""
from __future__ import annotations

import itertools

import numpy as np
import scipy.signal
import scipy.special
import torch


def _rng(seed):
    return np.random.default_rng(seed)


def _bf16_values(rng, shape):
    """Random values exactly representable in bf16 (as float64)."""
    t = torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(torch.bfloat16)
    return t.double().numpy()


def _bf16_bits(a64):
    return torch.from_numpy(np.ascontiguousarray(a64, dtype=np.float32)).to(
        torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _silu(z):
    return z * scipy.special.expit(z)


def _close(a, b, rtol, what):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    scale = max(1.0, float(np.max(np.abs(b))) if b.size else 1.0)
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= rtol * scale, f"{what}: max err {err:.3e} > {rtol:.1e} * {scale:.3e}"


def _torch_ref(x, dy, w, bias):
    """float64 torch: grouped conv1d (cross-correlation) with W-1 left zeros + SiLU, and
    its autograd gradients."""
    B, T, D = x.shape
    W = w.shape[1]
    xt = torch.tensor(x, dtype=torch.float64).permute(0, 2, 1).contiguous().requires_grad_(True)
    wt = torch.tensor(w, dtype=torch.float64).reshape(D, 1, W).requires_grad_(True)
    bt = torch.tensor(bias, dtype=torch.float64).requires_grad_(True) if bias is not None else None
    z = torch.nn.functional.conv1d(torch.nn.functional.pad(xt, (W - 1, 0)), wt, bt, groups=D)
    y = torch.nn.functional.silu(z)
    dyt = torch.tensor(dy, dtype=torch.float64).permute(0, 2, 1)
    (y * dyt).sum().backward()
    return (y.detach().permute(0, 2, 1).numpy(), xt.grad.permute(0, 2, 1).numpy(),
            wt.grad.reshape(D, W).numpy(),
            None if bt is None else bt.grad.numpy())


# ---------------------------------------------------------------------------------------
# forward
# ---------------------------------------------------------------------------------------

def pin_fwd_lfilter(o):
    rng = _rng(1)
    for W in (1, 2, 3, 4):
        B, T, D = 2, 11, 3
        x = _bf16_values(rng, (B, T, D))
        w = rng.uniform(-0.5, 0.5, (D, W))
        bias = rng.uniform(-0.1, 0.1, D)
        y = o.fwd(x, w, bias)
        ref = np.empty_like(y)
        for b in range(B):
            for d in range(D):
                # lfilter coefficient k multiplies x[n-k]: that is w[d, W-1-k]
                z = scipy.signal.lfilter(w[d, ::-1], [1.0], x[b, :, d]) + bias[d]
                ref[b, :, d] = _silu(z)
        _close(y, ref, 1e-13, f"fwd vs lfilter W={W}")


def pin_fwd_bwd_torch(o):
    rng = _rng(2)
    for W, with_bias in ((4, True), (4, False), (3, True), (2, True), (1, True)):
        B, T, D = 3, 17, 5
        x = _bf16_values(rng, (B, T, D))
        dy = _bf16_values(rng, (B, T, D))
        w = rng.uniform(-0.5, 0.5, (D, W))
        bias = rng.uniform(-0.1, 0.1, D) if with_bias else None
        y_ref, dx_ref, dw_ref, db_ref = _torch_ref(x, dy, w, bias)
        y = o.fwd(x, w, bias)
        dx, dw, db = o.bwd(x, dy, w, bias)
        _close(y, y_ref, 1e-13, f"fwd vs torch W={W}")
        _close(dx, dx_ref, 1e-12, f"dx vs torch W={W}")
        _close(dw, dw_ref, 1e-12, f"dw vs torch W={W}")
        if with_bias:
            _close(db, db_ref, 1e-12, f"dbias vs torch W={W}")
        else:
            # dbias is sum(g) whether or not a bias was added
            y2, dx2, dw2, db2 = _torch_ref(x, dy, w, np.zeros(D))
            _close(db, db2, 1e-12, f"dbias (no bias) W={W}")


def pin_w1_elementwise(o):
    rng = _rng(3)
    B, T, D = 2, 7, 4
    x = _bf16_values(rng, (B, T, D))
    w = rng.uniform(-0.5, 0.5, (D, 1))
    bias = rng.uniform(-0.1, 0.1, D)
    y = o.fwd(x, w, bias)
    _close(y, _silu(w[:, 0] * x + bias), 1e-15, "W=1 silu(w x + b)")


def pin_impulse(o):
    # x = unit impulse at t0, bias 0  =>  z[t0 + k] = w[d, W-1-k] for k < W, else 0
    W, T, D, t0 = 4, 12, 3, 5
    w = np.array([[0.25, -0.5, 0.75, 1.0], [0.1, 0.2, 0.3, 0.4], [-1.0, 0.5, -0.25, 0.125]])
    x = np.zeros((1, T, D))
    x[0, t0, :] = 1.0
    _, z = o.fwd(x, w, None, return_z=True)
    expect = np.zeros((T, D))
    for k in range(W):
        expect[t0 + k, :] = w[:, W - 1 - k]
    _close(z[0], expect, 0.0, "impulse response")


def pin_constant(o):
    # x = c everywhere => z[t] = b + c * sum_{j >= W-1-t} w[d, j]  (fewer taps at the start)
    W, T, D, c = 4, 6, 2, 0.5
    w = np.array([[0.25, -0.5, 0.75, 1.0], [1.0, 2.0, 3.0, 4.0]])
    bias = np.array([0.125, -0.0625])
    x = np.full((1, T, D), c)
    _, z = o.fwd(x, w, bias, return_z=True)
    expect = np.empty((T, D))
    for t in range(T):
        lo = max(0, W - 1 - t)
        expect[t] = bias + c * w[:, lo:].sum(axis=1)
    _close(z[0], expect, 1e-15, "constant input")


def pin_zero_point(o):
    # x = 0, bias = 0 => z = 0 => y = silu(0) = 0 and g = dy * silu'(0) = dy / 2, so
    # dx[t] = sum_k w[d, W-1-k] dy[t+k] / 2, dw = 0, dbias = sum dy / 2.
    rng = _rng(4)
    B, T, D, W = 2, 9, 3, 4
    w = rng.uniform(-0.5, 0.5, (D, W))
    x = np.zeros((B, T, D))
    dy = _bf16_values(rng, (B, T, D))
    assert np.all(o.fwd(x, w, None) == 0.0), "silu(0) must be 0"
    dx, dw, db = o.bwd(x, dy, w, None)
    expect_dx = np.zeros_like(dx)
    for t in range(T):
        for k in range(W):
            if t + k < T:
                expect_dx[:, t, :] += w[:, W - 1 - k] * dy[:, t + k, :] / 2
    _close(dx, expect_dx, 1e-15, "dx at z=0")
    _close(dw, np.zeros_like(dw), 0.0, "dw at x=0")
    _close(db, dy.sum(axis=(0, 1)) / 2, 1e-15, "dbias at z=0")


# ---------------------------------------------------------------------------------------
# backward: finite differences
# ---------------------------------------------------------------------------------------

def pin_finite_differences(o):
    rng = _rng(5)
    B, T, D, W = 2, 6, 2, 4
    x = rng.standard_normal((B, T, D))
    dy = rng.standard_normal((B, T, D))
    w = rng.uniform(-0.5, 0.5, (D, W))
    bias = rng.uniform(-0.1, 0.1, D)
    h = 1e-6

    def loss(x_, w_, b_):
        return float(np.sum(o.fwd(x_, w_, b_) * dy))

    dx, dw, db = o.bwd(x, dy, w, bias)
    fd_dx = np.empty_like(x)
    for i in np.ndindex(x.shape):
        xp = x.copy(); xp[i] += h
        xm = x.copy(); xm[i] -= h
        fd_dx[i] = (loss(xp, w, bias) - loss(xm, w, bias)) / (2 * h)
    fd_dw = np.empty_like(w)
    for i in np.ndindex(w.shape):
        wp = w.copy(); wp[i] += h
        wm = w.copy(); wm[i] -= h
        fd_dw[i] = (loss(x, wp, bias) - loss(x, wm, bias)) / (2 * h)
    fd_db = np.empty_like(bias)
    for i in range(D):
        bp = bias.copy(); bp[i] += h
        bm = bias.copy(); bm[i] -= h
        fd_db[i] = (loss(x, w, bp) - loss(x, w, bm)) / (2 * h)
    _close(dx, fd_dx, 1e-7, "dx vs finite differences")
    _close(dw, fd_dw, 1e-7, "dw vs finite differences")
    _close(db, fd_db, 1e-7, "dbias vs finite differences")


def pin_padded_taps(o):
    rng = _rng(6)
    B, T, D = 2, 10, 3
    x = _bf16_values(rng, (B, T, D))
    dy = _bf16_values(rng, (B, T, D))
    bias = rng.uniform(-0.1, 0.1, D)
    for W in (1, 2, 3):
        w = rng.uniform(-0.5, 0.5, (D, W))
        w4 = np.concatenate([np.zeros((D, 4 - W)), w], axis=1)  # zero taps on the old side
        _close(o.fwd(x, w4, bias), o.fwd(x, w, bias), 0.0, f"padded taps fwd W={W}")
        dx4, dw4, db4 = o.bwd(x, dy, w4, bias)
        dx, dw, db = o.bwd(x, dy, w, bias)
        _close(dx4, dx, 0.0, f"padded taps dx W={W}")
        _close(dw4[:, 4 - W:], dw, 0.0, f"padded taps dw W={W}")
        _close(db4, db, 0.0, f"padded taps dbias W={W}")


# ---------------------------------------------------------------------------------------
# decode update
# ---------------------------------------------------------------------------------------

def pin_decode_matches_forward(o):
    rng = _rng(7)
    for W, T in ((4, 9), (3, 5), (2, 4), (4, 2), (1, 3)):
        B, D, S = 3, 4, 5
        x = _bf16_values(rng, (B, T, D))
        w = rng.uniform(-0.5, 0.5, (D, W))
        bias = rng.uniform(-0.1, 0.1, D)
        y_full = o.fwd(x, w, bias)
        idx = np.array([4, 0, 2], np.int32)       # sequence b lives in slot idx[b]
        state = np.zeros((S, D, W - 1), np.uint16)  # bf16 +0.0
        xb = _bf16_bits(x)
        for t in range(T):
            status, y, state = o.update(xb[:, t, :], state, idx, w, bias)
            assert status == 0
            _close(y, y_full[:, t, :], 1e-15, f"decode step {t} vs forward row W={W}")
        for b in range(B):
            expect = np.zeros((D, W - 1), np.uint16)
            for j in range(W - 1):
                t = T - (W - 1) + j          # state[..., 0] is the oldest
                if t >= 0:
                    expect[:, j] = xb[b, t, :]
            assert np.array_equal(state[idx[b]], expect), f"final state of seq {b} W={W}"
        untouched = [s for s in range(S) if s not in idx]
        assert np.all(state[untouched] == 0), "slots not named by state_indices changed"


def _validate_by_sets(idx, S):
    mask = 0
    if any(v < 0 for v in idx):
        mask |= 1
    if any(v >= S for v in idx):
        mask |= 2
    valid = [v for v in idx if 0 <= v < S]
    if len(set(valid)) != len(valid):
        mask |= 4
    return mask


def pin_validate_exhaustive(o):
    for S in range(0, 5):
        for N in range(0, 4):
            for idx in itertools.product(range(-1, S + 2), repeat=N):
                got = o.validate(np.array(idx, np.int32), S)
                assert got == _validate_by_sets(idx, S), f"validate {idx} S={S}: {got}"


def pin_update_fail_closed(o):
    rng = _rng(8)
    S, N, D, W = 6, 3, 4, 4
    state = _bf16_bits(_bf16_values(rng, (S, D, W - 1)))
    x = _bf16_bits(_bf16_values(rng, (N, D)))
    w = rng.uniform(-0.5, 0.5, (D, W))
    for idx, mask in (([0, -1, 2], 1), ([0, 6, 2], 2), ([3, 1, 3], 4), ([-5, 9, 1], 3),
                      ([7, 7, 0], 2), ([2, 2, -1], 5)):
        status, y, new_state = o.update(x, state, np.array(idx, np.int32), w, None)
        assert status == mask, f"{idx}: status {status} != {mask}"
        assert y is None
        assert np.array_equal(new_state, state), f"{idx}: pool changed on a rejected call"
    # a valid call changes exactly the named slots
    status, y, new_state = o.update(x, state, np.array([5, 0, 3], np.int32), w, None)
    assert status == 0
    changed = sorted({int(s) for s in np.nonzero(np.any(new_state != state, axis=(1, 2)))[0]})
    assert set(changed) <= {0, 3, 5}
    # NULL indices: row i -> slot i
    status, y2, st2 = o.update(x, state, None, w, None)
    assert status == 0
    for i in range(N):
        assert np.array_equal(st2[i, :, :W - 2], state[i, :, 1:]) and np.array_equal(
            st2[i, :, W - 2], x[i]), "NULL indices must update slot i"


# ---------------------------------------------------------------------------------------
# packed sequences, initial / final state, activation
# ---------------------------------------------------------------------------------------

_LENS = (5, 0, 1, 2, 7, 3)   # empty, shorter than W-1, and several-tile-free ragged lengths


def _cu_of(lens):
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)


def _torch_seq_ref(x, dy, cu, w, bias, init, act):
    """float64 torch, one sequence at a time: concatenate the W-1 initial rows (zeros when
    no state is given) in front of the sequence, grouped conv1d with no padding, then SiLU
    or nothing; autograd gives every gradient.  The final state is the last W-1 rows of the
    concatenation."""
    D, W = w.shape
    wt = torch.tensor(w).reshape(D, 1, W).requires_grad_(True)
    bt = torch.tensor(bias).requires_grad_(True) if bias is not None else None
    nseq = len(cu) - 1
    xt = torch.tensor(x).requires_grad_(True)
    it = torch.tensor(init if init is not None else np.zeros((nseq, D, W - 1))).requires_grad_(True)
    ys, fins = [], []
    for i in range(nseq):
        ext = torch.cat([it[i], xt[cu[i]:cu[i + 1]].t()], dim=1)        # [D, W-1+L]
        if cu[i + 1] > cu[i]:
            z = torch.nn.functional.conv1d(ext[None], wt, bt, groups=D)[0]   # [D, L]
            ys.append((torch.nn.functional.silu(z) if act == "silu" else z).t())
        fins.append(ext[:, ext.shape[1] - (W - 1):])
    y = torch.cat(ys, dim=0)
    (y * torch.tensor(dy)).sum().backward()
    return (y.detach().numpy(), torch.stack(fins).detach().numpy(), xt.grad.numpy(),
            wt.grad.reshape(D, W).numpy(), None if bt is None else bt.grad.numpy(),
            it.grad.numpy())


def pin_seq_torch(o):
    rng = _rng(9)
    cu = _cu_of(_LENS)
    total, D = int(cu[-1]), 3
    for W in (4, 3, 2):
        for act in ("silu", None):
            for with_init in (True, False):
                x = rng.standard_normal((total, D))
                dy = rng.standard_normal((total, D))
                w = rng.uniform(-0.7, 0.7, (D, W))
                bias = rng.uniform(-0.3, 0.3, D)
                init = rng.standard_normal((len(_LENS), D, W - 1)) if with_init else None
                ry, rfin, rdx, rdw, rdb, rdi = _torch_seq_ref(x, dy, cu, w, bias, init, act)
                y, fin = o.fwd_seq(x, cu, w, bias, init, act, want_final=True)
                dx, dw, db, di = o.bwd_seq(x, dy, cu, w, bias, init, act, want_dinit=True)
                tag = f"seq W={W} act={act} init={with_init}"
                _close(y, ry, 1e-13, tag + " y")
                _close(fin, rfin, 0.0, tag + " final state")
                _close(dx, rdx, 1e-13, tag + " dx")
                _close(dw, rdw, 1e-13, tag + " dw")
                _close(db, rdb, 1e-13, tag + " dbias")
                _close(di, rdi, 1e-13, tag + " d initial state")


def pin_seq_split_handoff(o):
    """Cutting a sequence anywhere and passing the first part's final state as the second
    part's initial state changes nothing; the gradients add up the same way."""
    rng = _rng(10)
    D, W, L = 2, 4, 11
    x = rng.standard_normal((L, D))
    dy = rng.standard_normal((L, D))
    w = rng.uniform(-0.7, 0.7, (D, W))
    bias = rng.uniform(-0.3, 0.3, D)
    init = rng.standard_normal((1, D, W - 1))
    y_all, fin_all = o.fwd_seq(x, [0, L], w, bias, init, want_final=True)
    dx_all, dw_all, db_all, di_all = o.bwd_seq(x, dy, [0, L], w, bias, init, want_dinit=True)
    for cut in (1, 2, 3, 6, 10):
        y1, f1 = o.fwd_seq(x[:cut], [0, cut], w, bias, init, want_final=True)
        y2, f2 = o.fwd_seq(x[cut:], [0, L - cut], w, bias, f1, want_final=True)
        _close(np.concatenate([y1, y2]), y_all, 1e-15, f"split at {cut}: y")
        _close(f2, fin_all, 0.0, f"split at {cut}: final state")
        dx2, dw2, db2, di2 = o.bwd_seq(x[cut:], dy[cut:], [0, L - cut], w, bias, f1,
                                       want_dinit=True)
        # the second part's initial-state gradient flows back into the first part's rows
        # (and, for rows the first part took from its own initial state, into that state)
        ext1 = np.concatenate([init[0].T, x[:cut]])            # [W-1+cut, D]
        dext = np.zeros_like(ext1)
        dext[-(W - 1):] += di2[0].T
        dy1 = dy[:cut]
        dx1, dw1, db1, di1 = o.bwd_seq(x[:cut], dy1, [0, cut], w, bias, init, want_dinit=True)
        dx_first = dx1 + dext[W - 1:]
        di_first = di1[0] + dext[:W - 1].T
        _close(np.concatenate([dx_first, dx2]), dx_all, 1e-13, f"split at {cut}: dx")
        _close(dw1 + dw2, dw_all, 1e-13, f"split at {cut}: dw")
        _close(db1 + db2, db_all, 1e-13, f"split at {cut}: dbias")
        _close(di_first[None], di_all, 1e-13, f"split at {cut}: d initial state")


def pin_seq_decode_handoff(o):
    """A packed forward's final state, put in the decode pool, continues each sequence: a
    single-token update then gives the same row as the forward over the lengthened
    sequence, and leaves the same state."""
    rng = _rng(11)
    D, W = 4, 4
    lens = (6, 1, 0, 3)
    cu = _cu_of(lens)
    x = _bf16_values(rng, (int(cu[-1]), D))
    init = _bf16_values(rng, (len(lens), D, W - 1))
    xn = _bf16_values(rng, (len(lens), D))               # the next token of each sequence
    w = rng.uniform(-0.5, 0.5, (D, W))
    bias = rng.uniform(-0.1, 0.1, D)
    _, fin = o.fwd_seq(x, cu, w, bias, init, want_final=True)
    pool = _bf16_bits(fin)                                # exact: rows of x or of init
    idx = np.arange(len(lens), dtype=np.int32)[::-1].copy()
    state = np.zeros((len(lens), D, W - 1), np.uint16)
    state[idx] = pool
    status, y_dec, state = o.update(_bf16_bits(xn), state, idx, w, bias)
    assert status == 0
    # the lengthened sequences, packed
    lens2 = tuple(n + 1 for n in lens)
    cu2 = _cu_of(lens2)
    x2 = np.concatenate([np.concatenate([x[cu[i]:cu[i + 1]], xn[i:i + 1]])
                         for i in range(len(lens))])
    y2, fin2 = o.fwd_seq(x2, cu2, w, bias, init, want_final=True)
    _close(y_dec, y2[cu2[1:] - 1], 1e-15, "decode after packed forward vs lengthened forward")
    assert np.array_equal(state[idx], _bf16_bits(fin2)), "state after the handoff step"


def pin_seq_equal_lengths_batch(o):
    """Equal lengths with no initial state are the batched [B,T,D] forward / backward."""
    rng = _rng(12)
    B, T, D, W = 3, 6, 5, 4
    x = rng.standard_normal((B, T, D))
    dy = rng.standard_normal((B, T, D))
    w = rng.uniform(-0.7, 0.7, (D, W))
    bias = rng.uniform(-0.3, 0.3, D)
    cu = np.arange(B + 1, dtype=np.int64) * T
    y = o.fwd_seq(x.reshape(B * T, D), cu, w, bias)
    _close(y.reshape(B, T, D), o.fwd(x, w, bias), 0.0, "equal lengths: y")
    dx, dw, db, _ = o.bwd_seq(x.reshape(B * T, D), dy.reshape(B * T, D), cu, w, bias)
    rdx, rdw, rdb = o.bwd(x, dy, w, bias)
    _close(dx.reshape(B, T, D), rdx, 1e-14, "equal lengths: dx")
    _close(dw, rdw, 1e-14, "equal lengths: dw")
    _close(db, rdb, 1e-14, "equal lengths: dbias")


def pin_act_none_linear(o):
    """With no activation and no bias, (x, initial state) -> y is linear, and dx does not
    depend on x."""
    rng = _rng(13)
    cu = _cu_of((4, 3))
    D, W = 3, 4
    w = rng.uniform(-0.7, 0.7, (D, W))
    x1 = rng.standard_normal((7, D))
    x2 = rng.standard_normal((7, D))
    i1 = rng.standard_normal((2, D, W - 1))
    i2 = rng.standard_normal((2, D, W - 1))
    a = 1.75
    y12 = o.fwd_seq(a * x1 + x2, cu, w, None, a * i1 + i2, None)
    _close(y12, a * o.fwd_seq(x1, cu, w, None, i1, None) + o.fwd_seq(x2, cu, w, None, i2, None),
           1e-14, "act=None linearity")
    dy = rng.standard_normal((7, D))
    dxa = o.bwd_seq(x1, dy, cu, w, None, i1, None)[0]
    dxb = o.bwd_seq(x2, dy, cu, w, None, i2, None)[0]
    _close(dxa, dxb, 0.0, "act=None: dx independent of x")


# ---------------------------------------------------------------------------------------
# general decode update: longer state, padding rows, activation
# ---------------------------------------------------------------------------------------

def pin_update_ex_state_lengths(o):
    """Single-token updates from a zero state of Ls >= W-1 entries reproduce every row of the
    forward, and leave the last Ls tokens in the state (oldest first), bit for bit."""
    rng = _rng(14)
    for W, Ls, T in ((4, 4, 9), (4, 3, 7), (3, 5, 4), (2, 2, 6), (1, 1, 3), (1, 0, 2)):
        N, D, S = 2, 3, 4
        x = _bf16_values(rng, (N, T, D))
        w = rng.uniform(-0.5, 0.5, (D, W))
        bias = rng.uniform(-0.1, 0.1, D)
        for act in ("silu", None):
            y_full = o.fwd_seq(x.reshape(N * T, D), np.arange(N + 1) * T, w, bias, None, act)
            y_full = y_full.reshape(N, T, D)
            idx = np.array([3, 1], np.int32)
            state = np.zeros((S, D, Ls), np.uint16)
            xb = _bf16_bits(x)
            for t in range(T):
                status, y, state = o.update_ex(xb[:, t, :], state, idx, w, bias, activation=act)
                assert status == 0
                _close(y, y_full[:, t, :], 1e-15, f"W={W} Ls={Ls} act={act} step {t}")
            for n in range(N):
                expect = np.zeros((D, Ls), np.uint16)
                for j in range(Ls):
                    t = T - Ls + j
                    if t >= 0:
                        expect[:, j] = xb[n, t, :]
                assert np.array_equal(state[idx[n]], expect), f"W={W} Ls={Ls}: final state"


def pin_update_ex_is_update(o):
    """Ls = W-1, no padding, SiLU: the general form is the plain decode update."""
    rng = _rng(15)
    S, N, D, W = 7, 4, 5, 4
    state = _bf16_bits(_bf16_values(rng, (S, D, W - 1)))
    x = _bf16_bits(_bf16_values(rng, (N, D)))
    w = rng.uniform(-0.5, 0.5, (D, W))
    bias = rng.uniform(-0.1, 0.1, D)
    for idx in (np.array([6, 0, 3, 2], np.int32), None, np.array([1, -1, 2, 3], np.int32)):
        a = o.update(x, state, idx, w, bias)
        b = o.update_ex(x, state, idx, w, bias)
        assert a[0] == b[0] and np.array_equal(a[2], b[2])
        if a[0] == 0:
            _close(b[1], a[1], 0.0, "update_ex vs update")


def _validate_pad_by_sets(idx, S, pad):
    live = [v for v in idx if not (pad and v == -1)]
    return _validate_by_sets(live, S)


def pin_validate_pad_exhaustive(o):
    for S in range(0, 4):
        for N in range(0, 4):
            for idx in itertools.product(range(-2, S + 2), repeat=N):
                for pad in (False, True):
                    got = o.validate_pad(np.array(idx, np.int32), S, pad)
                    assert got == _validate_pad_by_sets(idx, S, pad), f"{idx} S={S} pad={pad}"


def pin_update_ex_padding_rows(o):
    """Padding rows (index -1) read and write no state and give no output; the other rows
    are exactly the update without them."""
    rng = _rng(16)
    S, D, W, Ls = 6, 4, 4, 4
    state = _bf16_bits(_bf16_values(rng, (S, D, Ls)))
    x = _bf16_bits(_bf16_values(rng, (5, D)))
    w = rng.uniform(-0.5, 0.5, (D, W))
    idx = np.array([2, -1, 5, -1, 0], np.int32)
    status, y, st = o.update_ex(x, state, idx, w, None, pad=True)
    assert status == 0
    live = idx >= 0
    status2, y2, st2 = o.update_ex(x[live], state, idx[live], w, None)
    assert status2 == 0
    assert np.array_equal(st, st2), "padding rows changed the pool"
    _close(y[live], y2, 0.0, "rows beside padding rows")
    assert np.all(np.isnan(y[~live])), "padding rows produced output"
    # without the padding mode, -1 is a negative index and the call fails closed
    status3, y3, st3 = o.update_ex(x, state, idx, w, None, pad=False)
    assert status3 == 1 and y3 is None and np.array_equal(st3, state)


def pin_update_ring_vs_shift(o):
    """The circular-buffer form against the shifting form: T single-token steps from a zero
    state, the ring fed pos = t, give the same y at every step, and the final ring is the
    shifted state rotated by T (ring[(T - Ls + j) mod Ls] = shifted[j])."""
    rng = _rng(17)
    for W, Ls, T in ((4, 3, 9), (4, 4, 10), (3, 2, 7), (2, 1, 5), (1, 1, 4), (4, 5, 11)):
        N, D, S = 3, 2, 5
        x = _bf16_bits(_bf16_values(rng, (T, N, D)))
        w = rng.uniform(-0.5, 0.5, (D, W))
        bias = rng.uniform(-0.1, 0.1, D)
        idx = np.array([4, 0, 2], np.int32)
        ring = np.zeros((S, D, Ls), np.uint16)
        shift = np.zeros((S, D, Ls), np.uint16)
        for t in range(T):
            for act in ("silu",):
                st1, y1, ring = o.update_ring(x[t], ring, idx, np.full(N, t, np.int32), w, bias,
                                              activation=act)
                st2, y2, shift = o.update_ex(x[t], shift, idx, w, bias, activation=act)
                assert st1 == 0 and st2 == 0
                _close(y1, y2, 0.0, f"W={W} Ls={Ls} step {t}")
        for j in range(Ls):
            assert np.array_equal(ring[idx][:, :, (T - Ls + j) % Ls], shift[idx][:, :, j]), \
                f"W={W} Ls={Ls}: ring is not the rotated shifted state"


def pin_update_ring_positions(o):
    """Closed form on one slot: a ring holding known tokens, read at several positions."""
    D, W, Ls = 1, 3, 4
    w = np.array([[0.25, 0.5, 1.0]])          # taps on (older, newer, token)
    vals = np.array([1.0, 2.0, 4.0, 8.0])     # ring entries 0..3, exact in bf16
    ring = _bf16_bits(vals.reshape(1, 1, Ls))
    x = _bf16_bits(np.array([[16.0]]))
    for p in (0, 1, 2, 3, 4, 7, -1):
        h = p % Ls
        want_z = 0.25 * vals[(h - 2) % Ls] + 0.5 * vals[(h - 1) % Ls] + 16.0
        st, y, new = o.update_ring(x, ring, None, np.array([p], np.int32), w, None,
                                   activation=None)
        assert st == 0 and y[0, 0] == want_z, f"pos {p}: {y[0, 0]} != {want_z}"
        expect = ring.copy()
        expect[0, 0, h] = x[0, 0]
        assert np.array_equal(new, expect), f"pos {p}: token not at entry {h}"


ALL_PINS = [
    pin_fwd_lfilter,
    pin_fwd_bwd_torch,
    pin_w1_elementwise,
    pin_impulse,
    pin_constant,
    pin_zero_point,
    pin_finite_differences,
    pin_padded_taps,
    pin_decode_matches_forward,
    pin_validate_exhaustive,
    pin_update_fail_closed,
    pin_seq_torch,
    pin_seq_split_handoff,
    pin_seq_decode_handoff,
    pin_seq_equal_lengths_batch,
    pin_act_none_linear,
    pin_update_ex_state_lengths,
    pin_update_ex_is_update,
    pin_validate_pad_exhaustive,
    pin_update_ex_padding_rows,
    pin_update_ring_vs_shift,
    pin_update_ring_positions,
]
