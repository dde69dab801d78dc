"""Plant single mistakes in copies of the oracle (on the CPU) and check the pins notice.

Each mutant is a one-token change of the kind a careless restatement makes: a reversed
tap, a dropped term, a wrong sign, a wrong shift.  A pin set that passes a mutant would
not have caught that mistake in the real oracle.  Mutants that would read out of bounds
are not planted.
"""
import shutil

import pytest

import oracle
from oracle import build as oracle_build
from tests import oracle_pins

SRC = oracle_build.SOURCE.read_text()

MUTANTS = {
    "tap_reversed_fwd": ("z += w[d * W + (W - 1 - k)] * x[", "z += w[d * W + k] * x["),
    "bias_dropped": ("double z = bias ? bias[d] : 0.0;\n  for (int k = 0; k < W; ++k) {\n    if (t - k < 0)",
                     "double z = 0.0;\n  for (int k = 0; k < W; ++k) {\n    if (t - k < 0)"),
    "sigmoid_sign": ("return 1.0 / (1.0 + exp(-z));", "return 1.0 / (1.0 + exp(z));"),
    "dsilu_term_dropped": ("s * (1.0 + zz * (1.0 - s))", "s * (1.0 + (1.0 - s))"),
    "dsilu_sign": ("(1.0 - s))", "(1.0 + s))"),
    "dx_tap_reversed": ("acc += w[d * W + (W - 1 - k)] * g[", "acc += w[d * W + k] * g["),
    "dw_index_reversed": ("dw[d * W + (W - 1 - k)] += gg", "dw[d * W + k] += gg"),
    "dbias_dropped": ("if (dbias) dbias[d] += gg;", "if (dbias) dbias[d] += 0.0 * gg;"),
    "dw_lag_shifted": ("if (t - k < 0) continue;\n          dw[d * W + (W - 1 - k)] += gg * x[(b * T + (t - k)) * D + d];",
                       "if (t - k - 1 < 0) continue;\n          dw[d * W + (W - 1 - k)] += gg * x[(b * T + (t - k - 1)) * D + d];"),
    "dx_reads_the_past": ("if (t + k >= T) continue;\n          acc += w[d * W + (W - 1 - k)] * g[(b * T + (t + k)) * D + d];",
                          "if (t - k < 0) continue;\n          acc += w[d * W + (W - 1 - k)] * g[(b * T + (t - k)) * D + d];"),
    "dx_tail_dropped": ("if (t + k >= T) continue;\n          acc +=", "if (t + k >= T - 1) continue;\n          acc +="),
    "decode_no_shift": ("st[j] = window[j + 1];", "st[j] = window[j];"),
    "decode_tap_reversed": ("z += w[d * W + j] * bf16_to_double(window[j]);",
                            "z += w[d * W + (W - 1 - j)] * bf16_to_double(window[j]);"),
    "validate_no_duplicates": ("mask |= ORACLE_IDX_DUPLICATE;", "mask |= 0;"),
    "validate_range_off_by_one": ("else if (idx[i] >= S) mask |= ORACLE_IDX_OUT_OF_RANGE;",
                                  "else if (idx[i] > S) mask |= ORACLE_IDX_OUT_OF_RANGE;"),
    # packed sequences, initial / final state, activation
    "seq_boundary_leak": ("if (u >= cu[i]) return x[u * D + d];",
                          "if (u >= 0) return x[u * D + d];"),
    "seq_init_ignored": ("return init[(i * D + d) * (W - 1) + j];",
                         "return 0.0 * init[(i * D + d) * (W - 1) + j];"),
    "seq_init_reversed": ("return init[(i * D + d) * (W - 1) + j];",
                          "return init[(i * D + d) * (W - 1) + (W - 2 - j)];"),
    "seq_final_shift": ("seq_x(D, W, x, cu, init, i, cu[i + 1] - (W - 1) + j, d);",
                        "seq_x(D, W, x, cu, init, i, cu[i + 1] - W + j, d);"),
    "seq_dx_crosses_end": ("if (t + k < e) ax +=", "if (t + k < total) ax +="),
    "seq_dinit_tap_reversed": ("ai += w[d * W + (W - 1 - k)] * gs[", "ai += w[d * W + k] * gs["),
    "seq_dinit_window": ("if (u + k >= s && u + k < e) ai", "if (u + k > s && u + k < e) ai"),
    "act_none_ignored_fwd": ("y[t * D + d] = act == 0 ? silu(zs) : zs;", "y[t * D + d] = silu(zs);"),
    "act_none_ignored_bwd": ("if (act == 0) {\n          const double zv", "if (1) {\n          const double zv"),
    # general decode update
    "upd_ex_window_oldest": ("win[j] = cell[Ls - (W - 1) + j];", "win[j] = cell[j];"),
    "upd_ex_no_shift": ("cell[j] = cell[j + 1];", "cell[j] = cell[j];"),
    "upd_ex_pad_not_skipped_validate": ("if (pad && v == -1) continue;", "if (pad && v == -2) continue;"),
    "upd_ex_pad_not_skipped_update": ("if (idx && pad && idx[i] == -1) {", "if (idx && pad && idx[i] == -2) {"),
    "upd_ex_act_ignored": ("y[i * D + d] = act == 0 ? silu(zd) : zd;", "y[i * D + d] = silu(zd);"),
    "upd_ex_no_duplicates": ("if (idx[k] == v) off |= ORACLE_IDX_DUPLICATE;",
                             "if (idx[k] == v && 0) off |= ORACLE_IDX_DUPLICATE;"),
    # circular-buffer decode
    "ring_head_off_by_one": ("const int64_t head = ring_mod(pos[i], Ls);",
                             "const int64_t head = ring_mod(pos[i] + 1, Ls);"),
    "ring_window_reversed": ("ring_win[j] = ring[ring_mod(head - (W - 1) + j, Ls)];",
                             "ring_win[j] = ring[ring_mod(head - 1 - j, Ls)];"),
    "ring_token_not_stored": ("      ring[head] = x[i * D + d];\n", "      (void)0;\n"),
    "ring_mod_negative": ("return r < 0 ? r + m : r;", "return r < 0 ? 0 : r;"),
}


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    d = tmp_path_factory.mktemp("oracle_mutants")
    yield d
    shutil.rmtree(d, ignore_errors=True)


def _run_pins(o):
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(o)
        except Exception as e:  # an assertion, or the oracle refusing its own result
            failed.append(f"{pin.__name__}: {type(e).__name__}: {str(e)[:80]}")
    return failed


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, mutant_dir):
    old, new = MUTANTS[name]
    assert SRC.count(old) == 1, f"mutation site for {name} not unique in the oracle source"
    src = mutant_dir / f"{name}.c"
    src.write_text(SRC.replace(old, new))
    lib = oracle_build.build(source=src, out=mutant_dir / f"lib{name}.so", force=True)
    failed = _run_pins(oracle.Oracle(lib))
    assert failed, f"no pin catches the planted mistake {name}"
