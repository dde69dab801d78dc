"""Packed variable-length sequences with initial / final states, and activation=None (GPU).

The CUDA path (cconv_fwd_varlen / cconv_bwd_varlen through the C ABI) is compared element
by element with the fp64 oracle's packed-sequence forms: ragged length mixes that include
empty, one-row and shorter-than-the-ring sequences, every width, both activations, with and
without initial states, bias and bf16 weights, at sizes spanning many tiles and CTA ranges
and at the production row count.  Final states must equal the oracle's bit for bit (they
are copies of bf16 rows).  Also: equal lengths without states reproduce the batched calls
bit for bit (dw, dbias up to the grouping of their partial sums); the final state written in place into a decode pool through state indices
continues the sequences under cconv_update; invalid indices fail closed; no rows at all;
an ill-formed cu_seqlens is reported through the device fault word.
"""
import numpy as np
import pytest
import torch

import depthwise_causal_short_gb300 as cc
import oracle
from depthwise_causal_short_gb300 import _build, inputs
from tests.helpers import BWD_TOL, FWD_TOL, bits, f64, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    return cc.load()


def _bits64(a):
    """fp64 array of bf16-representable values -> uint16 bf16 bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _lengths(total, nseq, seed):
    """A ragged mix with an empty, a one-row and a two-row sequence in it."""
    lens = inputs.seqlen_mix(total - 3, nseq - 3, seed=seed)
    return lens[:2] + [0] + lens[2:4] + [1] + lens[4:] + [2]


def _run(x, dy, cu, w, b, init, act, want_dinit=True):
    xg, dyg, cug, wg = x.cuda(), dy.cuda(), cu.cuda(), w.cuda()
    bg = None if b is None else b.cuda()
    ig = None if init is None else init.cuda()
    y, fin, _ = cc.cconv_fwd_varlen(xg, cug, wg, bg, activation=act, initial_state=ig,
                                    final_state=True)
    dx, dw, db, di = cc.cconv_bwd_varlen(xg, dyg, cug, wg, bg, activation=act, initial_state=ig,
                                         want_dbias=True, want_dinit=want_dinit)
    torch.cuda.synchronize()
    return y, fin, dx, dw, db, di


def _check(x, dy, cu, w, b, init, act, out, what):
    y, fin, dx, dw, db, di = out
    ry, rfin = oracle.fwd_seq(f64(x), cu.numpy(), f64(w), f64(b), f64(init), act,
                              want_final=True)
    e = rel_err(f64(y), ry)
    assert e <= FWD_TOL, f"{what}: y err {e:.2e}"
    if w.shape[1] > 1:
        assert np.array_equal(bits(fin), _bits64(rfin)), f"{what}: final state differs"
    rdx, rdw, rdb, rdi = oracle.bwd_seq(f64(x), f64(dy), cu.numpy(), f64(w), f64(b), f64(init),
                                        act, want_dinit=True)
    for name, g, r in (("dx", dx, rdx), ("dw", dw, rdw), ("dbias", db, rdb),
                       ("d_initial_state", di, rdi)):
        if g is None:
            continue
        e = rel_err(f64(g), r)
        assert e <= BWD_TOL, f"{what}: {name} err {e:.2e}"


@pytest.mark.parametrize("act", ["silu", None], ids=["silu", "none"])
@pytest.mark.parametrize("W", [4, 3, 2, 1])
@pytest.mark.parametrize("with_init", [True, False], ids=["init", "zeros"])
def test_ragged_mix(W, act, with_init):
    lens = _lengths(3000, 14, seed=W)
    x, dy, cu, w, b, init = inputs.varlen_inputs(lens, 1000, W, bias=True, seed=W)
    init = init if with_init else None
    out = _run(x, dy, cu, w, b, init, act)
    _check(x, dy, cu, w, b, init, act, out, f"W={W} act={act} init={with_init}")


@pytest.mark.parametrize("lens", [[1], [2], [3], [5], [1, 1, 1, 1], [0, 4, 0], [3, 0, 0, 9],
                                  [40, 1, 2, 3, 0, 77], [257, 256, 255]],
                         ids=lambda l: "_".join(map(str, l)))
def test_short_sequences(lens):
    x, dy, cu, w, b, init = inputs.varlen_inputs(lens, 264, 4, bias=True, seed=5)
    out = _run(x, dy, cu, w, b, init, "silu")
    _check(x, dy, cu, w, b, init, "silu", out, f"lens={lens}")


@pytest.mark.parametrize("wdtype", [torch.float32, torch.bfloat16], ids=["w_f32", "w_bf16"])
def test_production_rows(wdtype):
    """The production row count (16384 = 2 x 8192) at D=4096, packed as 16 mixed lengths."""
    lens = inputs.seqlen_mix(16384, 16, seed=0)
    x, dy, cu, w, b, init = inputs.varlen_inputs(lens, 4096, 4, bias=False, wdtype=wdtype)
    out = _run(x, dy, cu, w, b, init, "silu")
    _check(x, dy, cu, w, b, init, "silu", out, f"production rows {wdtype}")


def test_equal_lengths_match_batched_bitwise():
    B, T, D, W = 2, 8192, 4096, 4
    x, dy, w, b = inputs.fwd_bwd_inputs(B, T, D, W, bias=True)
    xg, dyg, wg, bg = x.cuda(), dy.cuda(), w.cuda(), b.cuda()
    cu = inputs.cu_of([T] * B).cuda()
    y_b = cc.cconv_fwd(xg, wg, bg)
    dx_b, dw_b, db_b = cc.cconv_bwd(xg, dyg, wg, bg)
    y_v, _, _ = cc.cconv_fwd_varlen(xg.view(B * T, D), cu, wg, bg)
    dx_v, dw_v, db_v, _ = cc.cconv_bwd_varlen(xg.view(B * T, D), dyg.view(B * T, D), cu, wg, bg)
    torch.cuda.synchronize()
    assert torch.equal(y_b.view(B * T, D).view(torch.int16), y_v.view(torch.int16))
    assert torch.equal(dx_b.view(B * T, D).view(torch.int16), dx_v.view(torch.int16))
    # dw / dbias: the same fp32 terms, but the two calls may group the partial sums
    # differently (each call's grouping is fixed, so each is deterministic on its own)
    assert torch.allclose(dw_b, dw_v, rtol=1e-5, atol=1e-5 * float(dw_b.abs().max()))
    assert torch.allclose(db_b, db_v, rtol=1e-5, atol=1e-5 * float(db_b.abs().max()))


def test_strided_rows():
    lens = [300, 0, 511, 64]
    x, dy, cu, w, b, init = inputs.varlen_inputs(lens, 512, 4, bias=True, seed=2)
    big = torch.zeros(x.shape[0], 1024, dtype=torch.bfloat16)
    big[:, 256:768] = x
    bigdy = torch.zeros_like(big)
    bigdy[:, 128:640] = dy
    xg, dyg = big.cuda()[:, 256:768], bigdy.cuda()[:, 128:640]
    y, fin, _ = cc.cconv_fwd_varlen(xg, cu.cuda(), w.cuda(), b.cuda(), initial_state=init.cuda(),
                                    final_state=True)
    dx, dw, db, di = cc.cconv_bwd_varlen(xg, dyg, cu.cuda(), w.cuda(), b.cuda(),
                                         initial_state=init.cuda())
    torch.cuda.synchronize()
    _check(x, dy, cu, w, b, init, "silu", (y, fin, dx, dw, db, di), "strided rows")


def test_backward_deterministic():
    lens = inputs.seqlen_mix(20000, 9, seed=4)
    x, dy, cu, w, b, init = inputs.varlen_inputs(lens, 2048, 4, bias=True, seed=4)
    a = _run(x, dy, cu, w, b, init, "silu")
    c = _run(x, dy, cu, w, b, init, "silu")
    for u, v in zip(a[2:], c[2:]):
        assert torch.equal(u.view(torch.int16) if u.dtype == torch.bfloat16 else u,
                           v.view(torch.int16) if v.dtype == torch.bfloat16 else v)


def test_pool_in_place_and_decode_handoff():
    """Chunked prefill into a decode pool: initial and final states are the same pool, the
    slots picked by state indices; then one decode step continues every sequence."""
    D, W, S = 1024, 4, 40
    lens = [700, 1, 0, 2, 129, 3000]
    x, _, cu, w, b, _ = inputs.varlen_inputs(lens, D, W, bias=True, seed=6)
    g = torch.Generator().manual_seed(6)
    pool = torch.randn(S, D, W - 1, generator=g).to(torch.bfloat16)
    idx = torch.randperm(S, generator=g)[:len(lens)].to(torch.int32)
    xn = torch.randn(len(lens), D, generator=g).to(torch.bfloat16)
    pool_g, idx_g = pool.cuda(), idx.cuda()
    y, fin, status = cc.cconv_fwd_varlen(x.cuda(), cu.cuda(), w.cuda(), b.cuda(),
                                         initial_state=pool_g, final_state=pool_g,
                                         state_indices=idx_g)
    torch.cuda.synchronize()
    assert fin is pool_g and status.tolist() == [0, 0]
    init = pool[idx.long()]
    ry, rfin = oracle.fwd_seq(f64(x), cu.numpy(), f64(w), f64(b), f64(init), "silu",
                              want_final=True)
    assert rel_err(f64(y), ry) <= FWD_TOL
    after = pool.clone()
    after[idx.long()] = torch.from_numpy(_bits64(rfin).view(np.int16)).view(torch.bfloat16)
    assert torch.equal(pool_g.cpu().view(torch.int16), after.view(torch.int16)), "pool"
    # one decode step from the handed-off states
    yd, st = cc.cconv_update(xn.cuda(), pool_g, w.cuda(), b.cuda(), state_indices=idx_g)
    torch.cuda.synchronize()
    assert st.tolist() == [0, 0]
    lens2 = [n + 1 for n in lens]
    cu2 = inputs.cu_of(lens2)
    x2 = torch.cat([torch.cat([x[int(cu[i]):int(cu[i + 1])], xn[i:i + 1]])
                    for i in range(len(lens))])
    ry2, rfin2 = oracle.fwd_seq(f64(x2), cu2.numpy(), f64(w), f64(b), f64(init), "silu",
                                want_final=True)
    assert rel_err(f64(yd), ry2[cu2[1:].numpy() - 1]) <= FWD_TOL
    assert np.array_equal(bits(pool_g[idx_g.long()]), _bits64(rfin2)), "state after decode"


def test_dense_in_place():
    """initial_state and final_state the same dense array (no indices): the final states are
    written by the second kernel after every read of the initial ones."""
    lens = _lengths(2000, 9, seed=11)
    x, dy, cu, w, b, init = inputs.varlen_inputs(lens, 512, 4, bias=True, seed=11)
    st = init.cuda()
    y, fin, _ = cc.cconv_fwd_varlen(x.cuda(), cu.cuda(), w.cuda(), b.cuda(), initial_state=st,
                                    final_state=st)
    torch.cuda.synchronize()
    assert fin is st
    ry, rfin = oracle.fwd_seq(f64(x), cu.numpy(), f64(w), f64(b), f64(init), "silu",
                              want_final=True)
    assert rel_err(f64(y), ry) <= FWD_TOL
    assert np.array_equal(bits(st), _bits64(rfin))


@pytest.mark.parametrize("bad,mask", [([0, -1, 2], 1), ([0, 5, 2], 2), ([3, 1, 3], 4)])
def test_invalid_state_indices_fail_closed(bad, mask):
    D, W, S = 256, 4, 5
    lens = [10, 20, 30]
    x, _, cu, w, b, init = inputs.varlen_inputs(lens, D, W, seed=7)
    g = torch.Generator().manual_seed(9)
    pool = torch.randn(S, D, W - 1, generator=g).to(torch.bfloat16).cuda()
    before = pool.clone()
    y, _, status = cc.cconv_fwd_varlen(x.cuda(), cu.cuda(), w.cuda(), b.cuda(),
                                       initial_state=pool, final_state=pool,
                                       state_indices=torch.tensor(bad, dtype=torch.int32).cuda())
    torch.cuda.synchronize()
    assert status.tolist() == [-8, mask]
    assert torch.equal(pool.view(torch.int16), before.view(torch.int16)), "pool changed"


def test_no_rows():
    D, W = 64, 4
    cu = torch.zeros(4, dtype=torch.int32).cuda()
    g = torch.Generator().manual_seed(10)
    init = torch.randn(3, D, W - 1, generator=g).to(torch.bfloat16).cuda()
    w = torch.rand(D, W, generator=g).cuda()
    x = torch.empty(0, D, dtype=torch.bfloat16).cuda()
    y, fin, _ = cc.cconv_fwd_varlen(x, cu, w, initial_state=init, final_state=True)
    dx, dw, db, di = cc.cconv_bwd_varlen(x, x, cu, w, initial_state=init, want_dbias=True)
    torch.cuda.synchronize()
    assert y.shape == (0, D) and torch.equal(fin.view(torch.int16), init.view(torch.int16))
    assert not dw.any() and not db.any() and not di.float().any()


def test_ill_formed_seqlens_reported():
    """cu_seqlens that decreases and overshoots: every access stays in bounds (rows are
    clamped to the range the host planned), the result is unspecified, and the device fault
    word reports it; the next well-formed call is clean."""
    D, W = 256, 4
    x, dy, cu, w, b, init = inputs.varlen_inputs([100, 100, 100], D, W, seed=8)
    bad = torch.tensor([0, 250, 120, 999], dtype=torch.int32).cuda()
    assert cc.cconv_device_fault() == 0
    cc.cconv_fwd_varlen(x.cuda(), bad, w.cuda(), b.cuda(), initial_state=init.cuda(),
                        final_state=True)
    cc.cconv_bwd_varlen(x.cuda(), dy.cuda(), bad, w.cuda(), b.cuda(), initial_state=init.cuda())
    assert cc.cconv_device_fault() == 4
    out = _run(x, dy, cu, w, b, init, "silu")
    assert cc.cconv_device_fault() == 0
    _check(x, dy, cu, w, b, init, "silu", out, "after an ill-formed call")


def _pool_case(lens, D, W, S, seed):
    """Inputs of a packed call whose initial states live in a decode pool of S slots."""
    x, dy, cu, w, b, _ = inputs.varlen_inputs(lens, D, W, bias=True, seed=seed)
    g = torch.Generator().manual_seed(seed + 1000)
    pool = torch.randn(S, D, W - 1, generator=g).to(torch.bfloat16)
    idx = torch.randperm(S, generator=g)[:len(lens)].to(torch.int32)
    return x, dy, cu, w, b, pool, idx


@pytest.mark.parametrize("D", [256, 1024, 2048])
def test_backward_reads_initial_states_from_pool_slots(D):
    """Packed backward with each sequence's initial state picked from a decode pool by
    state_indices (the gradient path of a chunked prefill that read from the pool): against
    the oracle on the gathered states, and bit for bit against the same call on the states
    gathered into a dense array.  D = 256, 1024 and 2048 take the independent-pipeline and
    the 4- and 8-strip lockstep kernels."""
    W, S = 4, 37
    lens = [700, 1, 0, 2, 129, 3000, 64, 5]
    x, dy, cu, w, b, pool, idx = _pool_case(lens, D, W, S, seed=D)
    xg, dyg, cug, wg, bg = (t.cuda() for t in (x, dy, cu, w, b))
    status = torch.full((2,), 7, dtype=torch.int32, device="cuda")
    dx, dw, db, di = cc.cconv_bwd_varlen(xg, dyg, cug, wg, bg, initial_state=pool.cuda(),
                                         state_indices=idx.cuda(), status=status,
                                         want_dbias=True, want_dinit=True)
    dense = pool[idx.long()]
    ref = cc.cconv_bwd_varlen(xg, dyg, cug, wg, bg, initial_state=dense.cuda(), want_dbias=True,
                              want_dinit=True)
    torch.cuda.synchronize()
    assert status.tolist() == [0, 0]
    for a, r in zip((dx, dw, db, di), ref):
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                           r.view(torch.int16) if r.dtype == torch.bfloat16 else r)
    rdx, rdw, rdb, rdi = oracle.bwd_seq(f64(x), f64(dy), cu.numpy(), f64(w), f64(b), f64(dense),
                                        "silu", want_dinit=True)
    for name, g, r in (("dx", dx, rdx), ("dw", dw, rdw), ("dbias", db, rdb),
                       ("d_initial_state", di, rdi)):
        assert rel_err(f64(g), r) <= BWD_TOL, name


def _offset_copy(t):
    """t's values in a tensor that starts one element (2 bytes) into its buffer, so its data
    pointer is not 8-byte aligned."""
    buf = torch.empty(t.numel() + 1, dtype=t.dtype, device=t.device)
    v = buf[1:].view(t.shape)
    v.copy_(t)
    assert v.data_ptr() % 8 != 0
    return v


@pytest.mark.parametrize("D", [1024, 4096])
def test_unaligned_initial_states(D):
    """The backward reads W = 4 initial rings as three 8-byte words per lane when the state is
    8-byte aligned, and through 2-byte loads into the same layout otherwise.  A state that
    starts 2 bytes into its buffer (dense, and a decode pool addressed through state indices)
    must give the aligned call's results bit for bit, and the oracle's within tolerance.  The
    forward, whose states must be 16-byte aligned, refuses it with CCONV_ERR_ALIGN."""
    W, S = 4, 29
    lens = [300, 1, 0, 2, 129, 777, 3]
    x, dy, cu, w, b, pool, idx = _pool_case(lens, D, W, S, seed=D + 3)
    xg, dyg, cug, wg, bg = (t.cuda() for t in (x, dy, cu, w, b))
    dense = pool[idx.long()]
    dense_g, pool_g = dense.cuda(), pool.cuda()
    r0 = cc.cconv_bwd_varlen(xg, dyg, cug, wg, bg, initial_state=dense_g, want_dbias=True,
                             want_dinit=True)
    r1 = cc.cconv_bwd_varlen(xg, dyg, cug, wg, bg, initial_state=_offset_copy(dense_g),
                             want_dbias=True, want_dinit=True)
    status = torch.full((2,), 7, dtype=torch.int32, device="cuda")
    r2 = cc.cconv_bwd_varlen(xg, dyg, cug, wg, bg, initial_state=_offset_copy(pool_g),
                             state_indices=idx.cuda(), status=status, want_dbias=True,
                             want_dinit=True)
    torch.cuda.synchronize()
    assert status.tolist() == [0, 0]
    as_bits = lambda t: t.view(torch.int16) if t.dtype == torch.bfloat16 else t
    for a, c, r in zip(r1, r2, r0):
        assert torch.equal(as_bits(a), as_bits(r)) and torch.equal(as_bits(c), as_bits(r))
    rdx, rdw, rdb, rdi = oracle.bwd_seq(f64(x), f64(dy), cu.numpy(), f64(w), f64(b), f64(dense),
                                        "silu", want_dinit=True)
    for name, g, r in (("dx", r1[0], rdx), ("dw", r1[1], rdw), ("dbias", r1[2], rdb),
                       ("d_initial_state", r1[3], rdi)):
        assert rel_err(f64(g), r) <= BWD_TOL, name
    with pytest.raises(cc.CConvError) as e:
        cc.cconv_fwd_varlen(xg, cug, wg, bg, initial_state=_offset_copy(dense_g))
    assert e.value.status == -4


@pytest.mark.parametrize("bad,mask", [([0, -1, 2], 1), ([0, 5, 2], 2), ([3, 1, 3], 4),
                                      ([-3, 9, 1], 3)])
def test_backward_pool_indices_checked(bad, mask):
    """Invalid state indices in the packed backward: the status words report the offence as
    the forward's check does; negative and out-of-range slots read as zero initial states,
    repeated slots are read as they are."""
    D, W, S = 512, 4, 5
    lens = [10, 20, 30]
    x, dy, cu, w, b, pool, _ = _pool_case(lens, D, W, S, seed=8)
    idx = torch.tensor(bad, dtype=torch.int32)
    status = torch.zeros(2, dtype=torch.int32, device="cuda")
    dx, dw, db, di = cc.cconv_bwd_varlen(x.cuda(), dy.cuda(), cu.cuda(), w.cuda(), b.cuda(),
                                         initial_state=pool.cuda(), state_indices=idx.cuda(),
                                         status=status, want_dbias=True, want_dinit=True)
    torch.cuda.synchronize()
    assert status.tolist() == [-8, mask]
    init = torch.zeros(len(lens), D, W - 1, dtype=torch.bfloat16)
    for i, s in enumerate(bad):
        if 0 <= s < S:
            init[i] = pool[s]
    rdx, rdw, rdb, rdi = oracle.bwd_seq(f64(x), f64(dy), cu.numpy(), f64(w), f64(b), f64(init),
                                        "silu", want_dinit=True)
    for name, g, r in (("dx", dx, rdx), ("dw", dw, rdw), ("dbias", db, rdb),
                       ("d_initial_state", di, rdi)):
        assert rel_err(f64(g), r) <= BWD_TOL, name


def test_backward_pool_indices_with_no_rows():
    """No rows at all: the gradients are zero and the indices are still checked."""
    D, W, S = 64, 3, 4
    cu = torch.zeros(4, dtype=torch.int32, device="cuda")
    pool = torch.randn(S, D, W - 1).to(torch.bfloat16).cuda()
    w = torch.rand(D, W).cuda()
    x = torch.empty(0, D, dtype=torch.bfloat16).cuda()
    status = torch.zeros(2, dtype=torch.int32, device="cuda")
    dx, dw, db, di = cc.cconv_bwd_varlen(x, x, cu, w, initial_state=pool,
                                         state_indices=torch.tensor([1, 1, 0], dtype=torch.int32,
                                                                    device="cuda"),
                                         status=status, want_dbias=True)
    torch.cuda.synchronize()
    assert status.tolist() == [-8, 4]
    assert not dw.any() and not db.any() and not di.float().any()
