"""The seeded input generators (CPU): the recipe's shapes, dtypes, ranges and determinism.

Both the oracle and the CUDA path draw their inputs from `depthwise_causal_short_gb300.inputs`,
so these checks pin what every parity test and the benchmark feed in: same seed, same
bits; the stated distributions' supports; sequence mixes that sum to the requested rows;
decode slots that are distinct and in range.
"""
import pytest
import torch

from depthwise_causal_short_gb300 import inputs


def _same(a, b):
    if a is None or b is None:
        return a is None and b is None
    if a.dtype == torch.bfloat16:
        return torch.equal(a.view(torch.int16), b.view(torch.int16))
    return torch.equal(a, b)


@pytest.mark.parametrize("wdtype", [torch.float32, torch.bfloat16])
def test_fwd_bwd_inputs_recipe(wdtype):
    x, dy, w, b = inputs.fwd_bwd_inputs(2, 33, 24, 3, True, wdtype=wdtype, seed=5)
    assert x.shape == (2, 33, 24) and dy.shape == (2, 33, 24)
    assert x.dtype == torch.bfloat16 and dy.dtype == torch.bfloat16
    assert w.shape == (24, 3) and w.dtype == wdtype
    assert b.shape == (24,) and b.dtype == wdtype
    assert float(w.float().abs().max()) <= 0.5
    assert float(b.float().abs().max()) <= 0.1
    assert not torch.equal(x, dy)
    again = inputs.fwd_bwd_inputs(2, 33, 24, 3, True, wdtype=wdtype, seed=5)
    assert all(_same(u, v) for u, v in zip((x, dy, w, b), again))
    other = inputs.fwd_bwd_inputs(2, 33, 24, 3, True, wdtype=wdtype, seed=6)
    assert not _same(x, other[0])
    assert inputs.fwd_bwd_inputs(1, 4, 8, 4, False)[3] is None


def test_fwd_bwd_draw_order_is_fixed():
    """x then dy: asking for a bias draws after them and leaves x, dy, w unchanged."""
    with_b = inputs.fwd_bwd_inputs(1, 10, 16, 4, True, seed=9)
    without = inputs.fwd_bwd_inputs(1, 10, 16, 4, False, seed=9)
    for u, v in zip(with_b[:3], without[:3]):
        assert _same(u, v)


def test_decode_inputs_recipe():
    st, xr, idx, w, b = inputs.decode_inputs(40, 17, 32, 4, True, n_x=3, seed=2)
    assert st.shape == (40, 32, 3) and st.dtype == torch.bfloat16
    assert xr.shape == (3, 17, 32) and xr.dtype == torch.bfloat16
    assert idx.shape == (17,) and idx.dtype == torch.int32
    assert len(set(idx.tolist())) == 17
    assert int(idx.min()) >= 0 and int(idx.max()) < 40
    assert w.shape == (32, 4) and b.shape == (32,)
    again = inputs.decode_inputs(40, 17, 32, 4, True, n_x=3, seed=2)
    assert all(_same(u, v) for u, v in zip((st, xr, idx, w, b), again))
    st1 = inputs.decode_inputs(40, 17, 32, 1, True, n_x=1)[0]
    assert st1.shape == (40, 32, 0)


@pytest.mark.parametrize("total, nseq", [(16384, 16), (16384, 128), (100, 7), (5, 5),
                                         (3, 8), (0, 4), (1000, 1)])
def test_seqlen_mix(total, nseq):
    lens = inputs.seqlen_mix(total, nseq, seed=1)
    assert len(lens) == nseq
    assert sum(lens) == total
    assert all(n >= 0 for n in lens)
    if total >= nseq:
        assert min(lens) >= 1
    assert lens == inputs.seqlen_mix(total, nseq, seed=1)


def test_seqlen_mix_is_a_mix():
    """The bench's packing: long and short sequences, not equal splits."""
    lens = inputs.seqlen_mix(16384, 16, seed=0)
    assert max(lens) > 4 * min(lens)
    assert inputs.seqlen_mix(16384, 16, seed=1) != lens


def test_cu_of_and_varlen_inputs():
    lens = [5, 0, 1, 12]
    cu = inputs.cu_of(lens)
    assert cu.dtype == torch.int32 and cu.tolist() == [0, 5, 5, 6, 18]
    x, dy, cu2, w, b, init = inputs.varlen_inputs(lens, 16, 3, bias=False, seed=4)
    assert torch.equal(cu, cu2)
    assert x.shape == (18, 16) and dy.shape == (18, 16)
    assert x.dtype == torch.bfloat16 and init.dtype == torch.bfloat16
    assert init.shape == (4, 16, 2)
    assert w.shape == (16, 3) and b is None
    again = inputs.varlen_inputs(lens, 16, 3, bias=False, seed=4)
    assert all(_same(u, v) for u, v in zip((x, dy, cu2, w, b, init), again))
