"""Seeded random cases of every entry point against the oracle (GPU).

Each case draws its shape and options from a fixed-seed generator, so a failure names a
reproducible case: batched forward / backward with random B, T, D tails, widths, bias,
weight dtype and row strides; packed sequences with random length mixes (empty and short
ones included), states, activation; decode updates with random pools, state lengths,
padding rows and layouts, shifting or circular (random positions), at small batches and at
batches that take the 256-thread row-lane CTAs; several problems in one
launch; and the same three backward calls at widths of 2048 channels and more, where they
take the lockstep kernels (with ragged last strip groups and short ranges).  Sizes stay
small enough for the fp64 oracle to finish in milliseconds.
"""
import random

import numpy as np
import pytest
import torch

import depthwise_causal_short_gb300 as cc
import oracle
from depthwise_causal_short_gb300 import _build, inputs
from tests.helpers import BWD_TOL, FWD_TOL, bits, f64, oracle_bwd, oracle_fwd, rel_err

pytestmark = pytest.mark.gpu

N_CASES = 100


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    return cc.load()


def _bits64(a):
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _strided(t, pad, dev):
    """t [.., D] placed at channel offset `pad` in rows of D + 2*pad channels (pad a multiple
    of 8, so the view keeps the 16-byte base and row-stride alignment the ABI requires)."""
    if pad == 0:
        return t.to(dev)
    big = torch.zeros(*t.shape[:-1], t.shape[-1] + 2 * pad, dtype=t.dtype)
    big[..., pad:pad + t.shape[-1]] = t
    return big.to(dev)[..., pad:pad + t.shape[-1]]


@pytest.mark.parametrize("case", range(N_CASES))
def test_batched(case):
    r = random.Random(1000 + case)
    B, T = r.randint(1, 4), r.choice([1, 2, 3, 5, 17, 64, 130, 513])
    D = 8 * r.randint(1, 128)
    W = r.randint(1, 4)
    has_bias = r.random() < 0.6
    wdt = r.choice([torch.float32, torch.bfloat16])
    pad = 8 * r.randint(0, 3)
    x, dy, w, b = inputs.fwd_bwd_inputs(B, T, D, W, has_bias, wdtype=wdt, seed=case)
    dev = torch.device("cuda", 0)
    xg, dyg = _strided(x, pad, dev), _strided(dy, 0, dev)
    y = cc.cconv_fwd(xg, w.to(dev), None if b is None else b.to(dev))
    dx, dw, db = cc.cconv_bwd(xg, dyg, w.to(dev), None if b is None else b.to(dev),
                              want_dbias=True)
    torch.cuda.synchronize()
    what = f"B={B} T={T} D={D} W={W} bias={has_bias} {wdt} pad={pad}"
    assert rel_err(f64(y), oracle_fwd(x, w, b)) <= FWD_TOL, what
    rdx, rdw, rdb = oracle_bwd(x, dy, w, b, want_dbias=True)
    for name, g, ref in (("dx", dx, rdx), ("dw", dw, rdw), ("dbias", db, rdb)):
        assert rel_err(f64(g), ref) <= BWD_TOL, f"{what}: {name}"


@pytest.mark.parametrize("case", range(N_CASES))
def test_packed(case):
    r = random.Random(2000 + case)
    nseq = r.randint(1, 12)
    lens = [r.choice([0, 1, 2, 3, r.randint(4, 40), r.randint(40, 400)]) for _ in range(nseq)]
    if sum(lens) == 0:
        lens[-1] = 5
    D = 8 * r.randint(1, 100)
    W = r.randint(1, 4)
    act = r.choice(["silu", None])
    with_init = r.random() < 0.7
    x, dy, cu, w, b, init = inputs.varlen_inputs(lens, D, W, bias=r.random() < 0.5,
                                                 wdtype=r.choice([torch.float32,
                                                                  torch.bfloat16]),
                                                 seed=case)
    init = init if with_init else None
    dev = torch.device("cuda", 0)
    ig = None if init is None else init.to(dev)
    bg = None if b is None else b.to(dev)
    y, fin, _ = cc.cconv_fwd_varlen(x.to(dev), cu.to(dev), w.to(dev), bg, activation=act,
                                    initial_state=ig, final_state=True)
    dx, dw, db, di = cc.cconv_bwd_varlen(x.to(dev), dy.to(dev), cu.to(dev), w.to(dev), bg,
                                         activation=act, initial_state=ig, want_dbias=True,
                                         want_dinit=True)
    torch.cuda.synchronize()
    what = f"lens={lens} D={D} W={W} act={act} init={with_init}"
    ry, rfin = oracle.fwd_seq(f64(x), cu.numpy(), f64(w), f64(b), f64(init), act,
                              want_final=True)
    assert rel_err(f64(y), ry) <= FWD_TOL, what
    if W > 1:
        assert np.array_equal(bits(fin), _bits64(rfin)), f"{what}: final state"
    rdx, rdw, rdb, rdi = oracle.bwd_seq(f64(x), f64(dy), cu.numpy(), f64(w), f64(b), f64(init),
                                        act, want_dinit=True)
    for name, g, ref in (("dx", dx, rdx), ("dw", dw, rdw), ("dbias", db, rdb),
                         ("d_initial_state", di, rdi)):
        assert rel_err(f64(g), ref) <= BWD_TOL, f"{what}: {name}"


@pytest.mark.parametrize("case", range(N_CASES))
def test_decode(case):
    r = random.Random(3000 + case)
    W = r.randint(1, 4)
    L = W - 1 + (r.random() < 0.4)
    S = r.randint(1, 80)
    N = r.randint(1, min(S, 70))
    D = r.choice([8 * r.randint(1, 64), r.randint(1, 300)])
    pad_rows = r.random() < 0.4
    act = r.choice(["silu", None]) if (pad_rows or L == W or r.random() < 0.3) else "silu"
    g = torch.Generator().manual_seed(case)
    state = torch.randn(S, D, L, generator=g).to(torch.bfloat16)
    x = torch.randn(N, D, generator=g).to(torch.bfloat16)
    w = torch.rand(D, W, generator=g) - 0.5
    b = torch.rand(D, generator=g) - 0.5 if r.random() < 0.5 else None
    idx = torch.randperm(S, generator=g)[:N].to(torch.int32)
    if pad_rows:
        for i in range(N):
            if r.random() < 0.3:
                idx[i] = -1
    dev = torch.device("cuda", 0)
    sg = state.to(dev)
    y = torch.zeros(N, D, dtype=torch.bfloat16, device=dev)
    _, status = cc.cconv_update_ex(x.to(dev), sg, w.to(dev), None if b is None else b.to(dev),
                                   idx.to(dev), pad_rows=pad_rows, activation=act, y=y)
    torch.cuda.synchronize()
    what = f"W={W} L={L} S={S} N={N} D={D} pad={pad_rows} act={act}"
    rc, y_ref, st_ref = oracle.update_ex(bits(x), bits(state), idx.numpy(), f64(w), f64(b),
                                         pad=pad_rows, activation=act)
    assert status.tolist() == [0 if rc == 0 else -8, rc], what
    assert np.array_equal(bits(sg), st_ref), f"{what}: pool"
    live = (idx >= 0).numpy()
    assert rel_err(f64(y)[live], y_ref[live]) <= FWD_TOL, f"{what}: y"
    assert not y[torch.from_numpy(~live).to(dev)].float().any(), f"{what}: padding y written"


@pytest.mark.parametrize("case", range(N_CASES // 2))
def test_multi(case):
    r = random.Random(4000 + case)
    n = r.randint(1, 4)
    B, T = r.randint(1, 3), r.choice([1, 4, 33, 300, 900])
    W = r.randint(1, 4)
    Ds = [8 * r.randint(1, 140) for _ in range(n)]
    wdt = r.choice([torch.float32, torch.bfloat16])
    probs = [inputs.fwd_bwd_inputs(B, T, D, W, r.random() < 0.5, wdtype=wdt, seed=case * 10 + k)
             for k, D in enumerate(Ds)]
    dev = torch.device("cuda", 0)
    xs = [p[0].to(dev) for p in probs]
    dys = [p[1].to(dev) for p in probs]
    ws = [p[2].to(dev) for p in probs]
    bs = [None if p[3] is None else p[3].to(dev) for p in probs]
    ys = cc.cconv_fwd_multi(xs, ws, bs)
    dxs, dws, dbs = cc.cconv_bwd_multi(xs, dys, ws, bs, want_dbias=True)
    torch.cuda.synchronize()
    for k, (x, dy, w, b) in enumerate(probs):
        what = f"n={n} B={B} T={T} Ds={Ds} W={W} problem {k}"
        assert rel_err(f64(ys[k]), oracle_fwd(x, w, b)) <= FWD_TOL, what
        rdx, rdw, rdb = oracle_bwd(x, dy, w, b, want_dbias=True)
        for name, gt, ref in (("dx", dxs[k], rdx), ("dw", dws[k], rdw), ("dbias", dbs[k], rdb)):
            assert rel_err(f64(gt), ref) <= BWD_TOL, f"{what}: {name}"


@pytest.mark.parametrize("case", range(N_CASES // 2))
def test_decode_ring(case):
    r = random.Random(5000 + case)
    W = r.randint(1, 4)
    L = max(1, W - 1 + (r.random() < 0.4))
    S = r.randint(1, 80)
    N = r.randint(1, min(S, 70))
    D = r.choice([8 * r.randint(1, 64), r.randint(1, 300)])
    pad_rows = r.random() < 0.3
    act = r.choice(["silu", None])
    g = torch.Generator().manual_seed(case)
    state = torch.randn(S, D, L, generator=g).to(torch.bfloat16)
    x = torch.randn(N, D, generator=g).to(torch.bfloat16)
    w = torch.rand(D, W, generator=g) - 0.5
    b = torch.rand(D, generator=g) - 0.5 if r.random() < 0.5 else None
    idx = torch.randperm(S, generator=g)[:N].to(torch.int32)
    if pad_rows:
        for i in range(N):
            if r.random() < 0.3:
                idx[i] = -1
    pos = torch.tensor([r.randint(-20, 1000) for _ in range(N)], dtype=torch.int32)
    dev = torch.device("cuda", 0)
    sg = state.to(dev)
    y = torch.zeros(N, D, dtype=torch.bfloat16, device=dev)
    _, status = cc.cconv_update_ex(x.to(dev), sg, w.to(dev), None if b is None else b.to(dev),
                                   idx.to(dev), pad_rows=pad_rows, cache_seqlens=pos.to(dev),
                                   activation=act, y=y)
    torch.cuda.synchronize()
    what = f"ring W={W} L={L} S={S} N={N} D={D} pad={pad_rows} act={act}"
    rc, y_ref, st_ref = oracle.update_ring(bits(x), bits(state), idx.numpy(), pos.numpy(),
                                           f64(w), f64(b), pad=pad_rows, activation=act)
    assert status.tolist() == [0 if rc == 0 else -8, rc], what
    assert np.array_equal(bits(sg), st_ref), f"{what}: pool"
    live = (idx >= 0).numpy()
    assert rel_err(f64(y)[live], y_ref[live]) <= FWD_TOL, f"{what}: y"


_ROW_LANE_THREADS: list[int] = []  # CTA size each test_decode_row_lanes case launched with


# Batches large enough for the 256-thread decode CTAs (32 channel vectors x 8 row lanes,
# staged taps, rows split evenly over a grid sized to the SM count, one CTA per SM): random
# batch sizes and widths (partial last channel blocks included), plain, general and
# circular-buffer modes, plain and bf16 taps, padding rows.
@pytest.mark.parametrize("case", range(N_CASES // 2))
def test_decode_row_lanes(case):
    r = random.Random(9000 + case)
    W = r.randint(1, 4)
    ring = r.random() < 0.3
    L = max(1, W - 1 + (r.random() < 0.4)) if ring else W - 1 + (r.random() < 0.3)
    N = r.randint(60, 600)
    S = N + r.randint(0, 90)
    D = 8 * r.randint(8, 1024)
    pad_rows = r.random() < 0.3
    act = r.choice(["silu", None]) if (pad_rows or ring or L == W or r.random() < 0.3) else "silu"
    wdtype = r.choice([torch.float32, torch.bfloat16])
    g = torch.Generator().manual_seed(9000 + case)
    state = torch.randn(S, D, L, generator=g).to(torch.bfloat16)
    x = torch.randn(N, D, generator=g).to(torch.bfloat16)
    w = (torch.rand(D, W, generator=g) - 0.5).to(wdtype)
    b = (torch.rand(D, generator=g) - 0.5).to(wdtype) if r.random() < 0.5 else None
    idx = torch.randperm(S, generator=g)[:N].to(torch.int32)
    if pad_rows:
        for i in range(N):
            if r.random() < 0.2:
                idx[i] = -1
    pos = torch.tensor([r.randint(-20, 1000) for _ in range(N)], dtype=torch.int32)
    dev = torch.device("cuda", 0)
    sg = state.to(dev)
    y = torch.zeros(N, D, dtype=torch.bfloat16, device=dev)
    args = (x.to(dev), sg, w.to(dev), None if b is None else b.to(dev), idx.to(dev))
    kw = dict(pad_rows=pad_rows, cache_seqlens=pos.to(dev) if ring else None, activation=act,
              y=y)
    ks = cc.describe(lambda: cc.cconv_update_ex(*args, **kw))  # records, launches nothing
    _ROW_LANE_THREADS.append(ks[-1]["threads"])
    _, status = cc.cconv_update_ex(*args, **kw)
    torch.cuda.synchronize()
    what = f"W={W} L={L} S={S} N={N} D={D} ring={ring} pad={pad_rows} act={act} w={wdtype}"
    if ring:
        rc, y_ref, st_ref = oracle.update_ring(bits(x), bits(state), idx.numpy(), pos.numpy(),
                                               f64(w), f64(b), pad=pad_rows, activation=act)
    else:
        rc, y_ref, st_ref = oracle.update_ex(bits(x), bits(state), idx.numpy(), f64(w), f64(b),
                                             pad=pad_rows, activation=act)
    assert status.tolist() == [0 if rc == 0 else -8, rc], what
    assert np.array_equal(bits(sg), st_ref), f"{what}: pool"
    live = (idx >= 0).numpy()
    assert rel_err(f64(y)[live], y_ref[live]) <= FWD_TOL, f"{what}: y"
    assert not y[torch.from_numpy(~live).to(dev)].float().any(), f"{what}: padding y written"


def test_decode_row_lanes_took_the_row_lane_kernels():
    """Most of the cases above must have run on the 256-thread CTAs they are there for."""
    if len(_ROW_LANE_THREADS) < N_CASES // 2:
        pytest.skip("runs after the full set of test_decode_row_lanes cases")
    share = sum(t == 256 for t in _ROW_LANE_THREADS) / len(_ROW_LANE_THREADS)
    assert share >= 0.6, share


# Widths from 2048 channels on take the lockstep backward kernels (a producer warp streams 8
# strips per stage); these cases cover them with ragged last strip groups, rows that give
# short ranges, strided x, and every width and weight dtype.
@pytest.mark.parametrize("case", range(N_CASES // 4))
def test_lockstep_batched(case):
    r = random.Random(6000 + case)
    B, T = r.randint(1, 3), r.choice([1, 3, 17, 64, 130, 333])
    D = 8 * r.randint(256, 640)
    W = r.randint(1, 4)
    has_bias = r.random() < 0.6
    wdt = r.choice([torch.float32, torch.bfloat16])
    pad = 8 * r.randint(0, 2)
    x, dy, w, b = inputs.fwd_bwd_inputs(B, T, D, W, has_bias, wdtype=wdt, seed=6000 + case)
    dev = torch.device("cuda", 0)
    xg, dyg = _strided(x, pad, dev), _strided(dy, 0, dev)
    bg = None if b is None else b.to(dev)
    dx, dw, db = cc.cconv_bwd(xg, dyg, w.to(dev), bg, want_dbias=True)
    torch.cuda.synchronize()
    what = f"B={B} T={T} D={D} W={W} bias={has_bias} {wdt} pad={pad}"
    rdx, rdw, rdb = oracle_bwd(x, dy, w, b, want_dbias=True)
    for name, g, ref in (("dx", dx, rdx), ("dw", dw, rdw), ("dbias", db, rdb)):
        assert rel_err(f64(g), ref) <= BWD_TOL, f"{what}: {name}"


@pytest.mark.parametrize("case", range(N_CASES // 4))
def test_lockstep_packed(case):
    r = random.Random(7000 + case)
    nseq = r.randint(1, 10)
    lens = [r.choice([0, 1, 2, 3, r.randint(4, 40), r.randint(40, 300)]) for _ in range(nseq)]
    if sum(lens) == 0:
        lens[-1] = 5
    D = 8 * r.randint(256, 520)
    W = r.randint(1, 4)
    act = r.choice(["silu", None])
    with_init = r.random() < 0.7
    x, dy, cu, w, b, init = inputs.varlen_inputs(lens, D, W, bias=r.random() < 0.5,
                                                 wdtype=r.choice([torch.float32,
                                                                  torch.bfloat16]),
                                                 seed=7000 + case)
    init = init if with_init else None
    dev = torch.device("cuda", 0)
    ig = None if init is None else init.to(dev)
    bg = None if b is None else b.to(dev)
    dx, dw, db, di = cc.cconv_bwd_varlen(x.to(dev), dy.to(dev), cu.to(dev), w.to(dev), bg,
                                         activation=act, initial_state=ig, want_dbias=True,
                                         want_dinit=True)
    torch.cuda.synchronize()
    what = f"lens={lens} D={D} W={W} act={act} init={with_init}"
    rdx, rdw, rdb, rdi = oracle.bwd_seq(f64(x), f64(dy), cu.numpy(), f64(w), f64(b), f64(init),
                                        act, want_dinit=True)
    for name, g, ref in (("dx", dx, rdx), ("dw", dw, rdw), ("dbias", db, rdb),
                         ("d_initial_state", di, rdi)):
        assert rel_err(f64(g), ref) <= BWD_TOL, f"{what}: {name}"


@pytest.mark.parametrize("case", range(N_CASES // 4))
def test_lockstep_multi(case):
    r = random.Random(8000 + case)
    n = r.randint(1, 4)
    B, T = r.randint(1, 2), r.choice([1, 4, 33, 300])
    W = r.randint(1, 4)
    Ds = [8 * r.randint(113, 300) for _ in range(n)]  # each fills a group of 8 strips
    if sum(Ds) < 2048:
        Ds[0] = 2048
    wdt = r.choice([torch.float32, torch.bfloat16])
    probs = [inputs.fwd_bwd_inputs(B, T, D, W, r.random() < 0.5, wdtype=wdt,
                                   seed=8000 + case * 10 + k) for k, D in enumerate(Ds)]
    dev = torch.device("cuda", 0)
    xs = [p[0].to(dev) for p in probs]
    dys = [p[1].to(dev) for p in probs]
    ws = [p[2].to(dev) for p in probs]
    bs = [None if p[3] is None else p[3].to(dev) for p in probs]
    dxs, dws, dbs = cc.cconv_bwd_multi(xs, dys, ws, bs, want_dbias=True)
    torch.cuda.synchronize()
    for k, (x, dy, w, b) in enumerate(probs):
        what = f"n={n} B={B} T={T} Ds={Ds} W={W} problem {k}"
        rdx, rdw, rdb = oracle_bwd(x, dy, w, b, want_dbias=True)
        for name, gt, ref in (("dx", dxs[k], rdx), ("dw", dws[k], rdw), ("dbias", dbs[k], rdb)):
            assert rel_err(f64(gt), ref) <= BWD_TOL, f"{what}: {name}"
