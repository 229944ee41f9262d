"""The threaded driver of the oracle (rows split across threads, results
merged) gives exactly the single-call oracle's bits: every full-size GPU
check reassembles its reference rows through it, so a mis-merged row, layout
or output would hide behind it.  Rows of a batch never interact (page
"Recurrent operators: RNN, GRU, LSTM", Computation: every product and gate is
per batch row), so computing them one at a time must change nothing."""
import numpy as np
import pytest

import oracle
from helpers import assert_bits_equal, oracle_case
from onnx_recurrent_gb300.synth import make_case


CASES = [
    dict(op="LSTM", direction="bidirectional", layout=0, lens=("uniform", 0, 6), with_P=True),
    dict(op="LSTM", direction="reverse", layout=1, lens=None, with_P=False),
    dict(op="GRU", direction="bidirectional", layout=1, lens=("uniform", 1, 6), with_P=False),
    dict(op="RNN", direction="forward", layout=0, lens=None, with_P=False),
]


@pytest.mark.parametrize("kw", CASES, ids=[f"{c['op']}-{c['direction']}-l{c['layout']}" for c in CASES])
def test_threaded_equals_single_call(kw):
    kw = dict(kw)
    op, direction = kw.pop("op"), kw.pop("direction")
    c = make_case(op, direction, 6, 7, 5, 9, seed=13, h0_scale=0.5, c0_scale=0.5, clip=2.0, **kw)
    ref = oracle_case(c)
    got = oracle_case(c, threaded=True)
    for name, g, r in zip(("Y", "Y_h", "Y_c"), got, ref):
        if r is None:
            assert g is None
            continue
        assert_bits_equal(g, r, name)


def test_threaded_subset_leaves_other_rows_zero():
    c = make_case("LSTM", "bidirectional", 5, 6, 4, 8, seed=3, layout=0, with_P=True, h0_scale=0.5,
                  c0_scale=0.5, lens=("uniform", 1, 5))
    rows = [1, 4]
    ref = oracle_case(c)
    got = oracle_case(c, rows=rows, threaded=True)
    for name, g, r in zip(("Y", "Y_h", "Y_c"), got, ref):
        ax = 2 if name == "Y" else 1
        for n in range(c.batch):
            gs, rs = np.take(g, n, axis=ax), np.take(r, n, axis=ax)
            if n in rows:
                assert_bits_equal(gs, rs, f"{name} row {n}")
            else:
                assert not np.any(gs), f"{name} row {n} should be untouched"


def test_threaded_single_row_matches():
    c = make_case("GRU", "forward", 4, 3, 3, 5, seed=5, layout=1, linear_before_reset=1)
    ref = oracle_case(c)
    got = oracle.rnn_threaded(c.op, c.direction, c.hidden_size, c.input_size, c.X, c.W, c.R, B=c.B,
                              layout=1, linear_before_reset=1, rows=[2], threads=3)
    assert_bits_equal(got[0][2], ref[0][2], "Y row 2")
    assert_bits_equal(got[1][2], ref[1][2], "Y_h row 2")
