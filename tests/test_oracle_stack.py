"""Pins for the oracle's stacked layers (the library's reading: layer l+1's X
is layer l's Y with the directions side by side per step): hand-derived
cases (tests/golden/stack), the layer handoff against an independent
transpose/reshape formula, one layer = the single operator, layout 1 = the
transposed layout 0 stack, and the shared sequence_lens."""
import glob
import json
import os

import numpy as np
import pytest

import oracle
from onnx_recurrent_gb300.synth import make_case

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "stack")
FILES = sorted(glob.glob(os.path.join(GOLDEN, "*.json")))


def _layers(fx):
    out = []
    for L in fx["layers"]:
        L = dict(L)
        L["W"] = np.array(L["W"], np.float32)
        L["R"] = np.array(L["R"], np.float32)
        out.append(L)
    return out


@pytest.mark.parametrize("path", FILES, ids=[os.path.basename(p) for p in FILES])
def test_stack_golden(path):
    with open(path) as f:
        fx = json.load(f)
    assert fx["citation"] and fx["derivation"]
    Y, yh, _ = oracle.rnn_stack(_layers(fx), np.array(fx["X"], np.float32))
    np.testing.assert_array_equal(Y, np.array(fx["expected"]["Y"], np.float32))
    for got, exp in zip(yh, fx["expected"]["Y_h"]):
        np.testing.assert_array_equal(got, np.array(exp, np.float32))


@pytest.mark.parametrize("layout", [0, 1])
def test_stack_input_matches_transpose_reshape(layout):
    g = np.random.default_rng(1)
    if layout == 0:
        Y = g.normal(size=(4, 2, 3, 5)).astype(np.float32)
        ref = Y.transpose(0, 2, 1, 3).reshape(4, 3, 10)
    else:
        Y = g.normal(size=(3, 4, 2, 5)).astype(np.float32)
        ref = Y.reshape(3, 4, 10)
    np.testing.assert_array_equal(oracle.stack_input(Y, layout), ref)


def _case_layers(seed, layout, lens=None):
    c0 = make_case("LSTM", "bidirectional", 5, 3, 6, 7, seed=seed, layout=layout, with_P=True, h0_scale=0.5,
                   lens=lens)
    c1 = make_case("GRU", "forward", 5, 3, 14, 4, seed=seed + 1, layout=layout, h0_scale=0.5,
                   linear_before_reset=1)
    layers = []
    for c in (c0, c1):
        a = c.attrs()
        a.update(W=c.W, R=c.R, B=c.B, P=c.P, initial_h=c.initial_h, initial_c=c.initial_c)
        layers.append(a)
    return c0, c1, layers


def test_one_layer_stack_is_the_operator():
    c0, _, layers = _case_layers(3, 0)
    Y, yh, yc = oracle.rnn_stack(layers[:1], c0.X)
    Y1, Yh1, Yc1 = oracle.rnn(c0.op, c0.direction, c0.hidden_size, c0.input_size, c0.X, c0.W, c0.R, B=c0.B,
                              P=c0.P, initial_h=c0.initial_h, layout=0)
    np.testing.assert_array_equal(Y, Y1)
    np.testing.assert_array_equal(yh[0], Yh1)
    np.testing.assert_array_equal(yc[0], Yc1)


def test_layout1_stack_is_transposed_layout0_stack():
    c0, c1, l0 = _case_layers(5, 0, lens=[5, 2, 0])
    Y0, yh0, yc0 = oracle.rnn_stack(l0, c0.X, sequence_lens=c0.sequence_lens)
    l1 = []
    for L in l0:
        L = dict(L, layout=1)
        for k in ("initial_h", "initial_c"):
            if L[k] is not None:
                L[k] = np.ascontiguousarray(L[k].transpose(1, 0, 2))
        l1.append(L)
    Y1, yh1, yc1 = oracle.rnn_stack(l1, np.ascontiguousarray(c0.X.transpose(1, 0, 2)),
                                    sequence_lens=c0.sequence_lens)
    np.testing.assert_array_equal(Y1, Y0.transpose(2, 0, 1, 3))
    for a, b in zip(yh1, yh0):
        np.testing.assert_array_equal(a, b.transpose(1, 0, 2))


def test_shared_lengths_mask_every_layer():
    c0, c1, layers = _case_layers(7, 0, lens=[5, 2, 0])
    Y, yh, _ = oracle.rnn_stack(layers, c0.X, sequence_lens=c0.sequence_lens)
    assert np.all(Y[2:, :, 1] == 0) and np.all(Y[:, :, 2] == 0)
    assert np.all(yh[1][:, 2] == 0)


_STACK_INPUT = oracle.stack_input


def _stack_input_directions_swapped(Y, layout):
    Y = np.asarray(Y, np.float32)
    return _STACK_INPUT(Y[:, ::-1] if layout == 0 else Y[:, :, ::-1], layout)


def _stack_input_batch_major(Y, layout):
    Y = np.asarray(Y, np.float32)
    if layout == 0:
        S, D, N, H = Y.shape
        return np.ascontiguousarray(Y.reshape(S, N, D * H))   # the directions' planes read as rows
    return _STACK_INPUT(Y, layout)


@pytest.mark.parametrize("mistake", [_stack_input_directions_swapped, _stack_input_batch_major])
def test_planted_handoff_mistakes_are_caught(mistake, monkeypatch):
    # a plausible misreading of the handoff, planted in the oracle: the
    # golden cases or the independent transpose formula must reject it
    monkeypatch.setattr(oracle, "stack_input", mistake)
    failed = 0
    for p in FILES:
        try:
            test_stack_golden(p)
        except AssertionError:
            failed += 1
    for layout in (0, 1):
        try:
            test_stack_input_matches_transpose_reshape(layout)
        except AssertionError:
            failed += 1
    assert failed > 0
