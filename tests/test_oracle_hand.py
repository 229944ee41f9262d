"""Hand-derived cases (tests/golden/*.json): small dyadic inputs whose every
intermediate value is exact in fp32, so the page's formulas give the outputs
exactly; each fixture carries its citation and derivation."""
import glob
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
FILES = sorted(glob.glob(os.path.join(GOLDEN, "*.json")))


def load(path):
    with open(path) as f:
        return json.load(f)


def run_fixture(fx):
    a = dict(fx["attrs"])
    ins = {k: (np.array(v, np.int32) if k == "sequence_lens" else np.array(v, np.float32))
           for k, v in fx["inputs"].items()}
    return oracle.rnn(a.pop("op"), a.pop("direction"), a.pop("hidden_size"), a.pop("input_size"),
                      ins["X"], ins["W"], ins["R"], B=ins.get("B"),
                      sequence_lens=ins.get("sequence_lens"), initial_h=ins.get("initial_h"),
                      initial_c=ins.get("initial_c"), P=ins.get("P"), **a)


@pytest.mark.parametrize("path", FILES, ids=[os.path.basename(p) for p in FILES])
def test_golden_case(path):
    fx = load(path)
    assert fx["citation"] and fx["derivation"]
    Y, Yh, Yc = run_fixture(fx)
    exp = fx["expected"]
    np.testing.assert_array_equal(Y, np.array(exp["Y"], np.float32))
    np.testing.assert_array_equal(Yh, np.array(exp["Y_h"], np.float32))
    if "Y_c" in exp:
        np.testing.assert_array_equal(Yc, np.array(exp["Y_c"], np.float32))


def test_nan_outputs_are_canonical():
    # Exact mode: every NaN written to Y, Y_h, Y_c is 0x7FC00000.
    X = np.array([[[np.nan]], [[1.0]]], np.float32)
    W = np.array([[[1.0], [1.0], [1.0], [1.0]]], np.float32)
    R = np.zeros((1, 4, 1), np.float32)
    Y, Yh, Yc = oracle.rnn("LSTM", "forward", 1, 1, X, W, R)
    for arr in (Y, Yh, Yc):
        assert np.all(arr.view(np.uint32) == 0x7FC00000)
    Y, Yh, _ = oracle.rnn("RNN", "forward", 1, 1, X, W[:, :1], R[:, :1], activations=["Relu"])
    assert np.all(Y.view(np.uint32) == 0x7FC00000)


def test_accumulation_starts_from_plus_zero():
    # Computation: one accumulator per output, k increasing from +0.  Every
    # product here is 0 * -1 = -0; from +0 each sum is +0 + -0 = +0, Relu
    # keeps it, and Y is +0 bit for bit (a sum started from -0 would stay -0
    # and Relu would pass the -0 on).
    X = np.zeros((1, 1, 1), np.float32)
    W = np.full((1, 1, 1), -1.0, np.float32)
    R = np.full((1, 1, 1), -1.0, np.float32)
    Y, Yh, _ = oracle.rnn("RNN", "forward", 1, 1, X, W, R, activations=["Relu"])
    assert Y.view(np.uint32).tolist() == [[[[0]]]] and Yh.view(np.uint32).tolist() == [[[0]]]


def test_nan_passes_through_clip():
    # Computation: clip clamps the pre-activation to [-clip, clip], a NaN
    # passing through: with Affine the NaN reaches Y (canonical in exact
    # mode), where a clamp that caught it would give the bound.
    X = np.array([[[np.nan]]], np.float32)
    W = np.ones((1, 1, 1), np.float32)
    R = np.zeros((1, 1, 1), np.float32)
    for clip in (0.5, 2.0):
        Y, Yh, _ = oracle.rnn("RNN", "forward", 1, 1, X, W, R, activations=["Affine"], alpha=[1.0], beta=[0.0],
                              clip=clip)
        assert Y.view(np.uint32).tolist() == [[[[0x7FC00000]]]] and Yh.view(np.uint32).tolist() == [[[0x7FC00000]]]


def test_bidirectional_lens_combines_both_hand_cases():
    fwd = load(os.path.join(GOLDEN, "rnn_lens_forward.json"))
    rev = load(os.path.join(GOLDEN, "rnn_lens_reverse.json"))
    bi = json.loads(json.dumps(fwd))
    bi["attrs"]["direction"] = "bidirectional"
    bi["inputs"]["W"] = fwd["inputs"]["W"] * 2
    bi["inputs"]["R"] = fwd["inputs"]["R"] * 2
    bi["inputs"]["initial_h"] = fwd["inputs"]["initial_h"] * 2
    Y, Yh, _ = run_fixture(bi)
    np.testing.assert_array_equal(Y[:, 0], np.array(fwd["expected"]["Y"], np.float32)[:, 0])
    np.testing.assert_array_equal(Y[:, 1], np.array(rev["expected"]["Y"], np.float32)[:, 0])
    np.testing.assert_array_equal(Yh[0], np.array(fwd["expected"]["Y_h"], np.float32)[0])
    np.testing.assert_array_equal(Yh[1], np.array(rev["expected"]["Y_h"], np.float32)[0])
