"""Pins for the oracle's own transcendentals and its IEEE activations.

The page ("Recurrent operators: RNN, GRU, LSTM", Activations) gives the
definitions; its own polynomials are not available, so the transcendental
functions are pinned by their error against double-precision math over dense
sweeps (bounds in float32 ulps of the exact value) and by special values.
"""
import math

import numpy as np
import pytest

import oracle


def _ulps(y, ref):
    ref = np.asarray(ref, np.float64)
    sp = np.spacing(np.abs(ref.astype(np.float32))).astype(np.float64)
    return np.abs(y.astype(np.float64) - ref) / sp


def test_exp_accuracy_sweep():
    x = np.concatenate([np.linspace(-103.0, 88.72, 1_000_003),
                        np.random.default_rng(1).uniform(-6, 6, 300_000)]).astype(np.float32)
    y = oracle.exp(x)
    ref = np.exp(x.astype(np.float64))
    e = _ulps(y, ref)
    normal = ref > np.finfo(np.float32).tiny
    assert e[normal].max() <= 1.5
    # subnormal results: absolute error within one subnormal step
    sub = ~normal
    assert np.all(np.abs(y[sub].astype(np.float64) - ref[sub]) <= 2.0 ** -149)


def test_exp_special_values():
    x = np.array([0.0, -0.0, np.nan, np.inf, -np.inf, 100.0, -200.0, 88.72, 1.0], np.float32)
    y = oracle.exp(x)
    assert y[0] == 1.0 and y[1] == 1.0
    assert np.isnan(y[2])
    assert y[3] == np.inf and y[4] == 0.0 and y[5] == np.inf and y[6] == 0.0
    assert np.isfinite(y[7]) and y[7] > 3e38
    assert abs(float(y[8]) - math.e) <= np.spacing(np.float32(math.e))


def test_log_accuracy_sweep():
    x = np.concatenate([np.geomspace(1e-44, 3e38, 600_001), np.linspace(0.5, 2.0, 300_001),
                        np.linspace(1.0, 5e8, 100_001)]).astype(np.float32)
    x = x[x > 0]
    y = oracle.log(x)
    e = _ulps(y, np.log(x.astype(np.float64)))
    assert e.max() <= 2.0


def test_log_special_values():
    y = oracle.log(np.array([1.0, 0.0, np.inf, np.nan, -1.0, 2.0], np.float32))
    assert y[0] == 0.0
    assert y[1] == -np.inf and y[2] == np.inf
    assert np.isnan(y[3]) and np.isnan(y[4])
    assert abs(float(y[5]) - math.log(2)) <= np.spacing(np.float32(math.log(2)))


def test_tanh_accuracy_sweep():
    x = np.concatenate([np.linspace(-10, 10, 1_000_001), np.geomspace(1e-38, 0.6, 200_001),
                        -np.geomspace(1e-38, 0.6, 20_001)]).astype(np.float32)
    e = _ulps(oracle.tanh(x), np.tanh(x.astype(np.float64)))
    assert e.max() <= 2.5


def test_tanh_special_values():
    y = oracle.tanh(np.array([0.0, -0.0, 20.0, -20.0, np.nan, np.inf, -np.inf], np.float32))
    b = y.view(np.uint32)
    assert b[0] == 0x00000000 and b[1] == 0x80000000
    assert y[2] == 1.0 and y[3] == -1.0 and np.isnan(y[4])
    assert y[5] == 1.0 and y[6] == -1.0


def test_sigmoid_accuracy_sweep():
    x = np.linspace(-80, 80, 800_001).astype(np.float32)
    ref = 1.0 / (1.0 + np.exp(-x.astype(np.float64)))
    e = _ulps(oracle.sigmoid(x), ref)
    assert e[ref > 1e-37].max() <= 3.0
    s = oracle.sigmoid(np.array([0.0, -200.0, 200.0, np.nan], np.float32))
    assert s[0] == 0.5 and s[1] == 0.0 and s[2] == 1.0 and np.isnan(s[3])


def _a(name, xs, alpha=0.0, beta=0.0):
    return oracle.activation(name, np.array(xs, np.float32), alpha, beta)


def test_relu_points():
    y = _a("relu", [-2.0, 3.0, np.nan, -0.0, 0.0])
    assert y[0] == 0.0 and y.view(np.uint32)[0] == 0
    assert y[1] == 3.0 and np.isnan(y[2])
    assert y.view(np.uint32)[3] == 0x80000000   # -0 is not < 0: kept
    assert y.view(np.uint32)[4] == 0


def test_leaky_thresholded_points():
    assert list(_a("leakyrelu", [-2.0, 3.0], 0.5)) == [-1.0, 3.0]
    # x < 0 ? alpha*x : x: a NaN is not < 0, so it is returned; -0 likewise
    y = _a("leakyrelu", [np.nan, -0.0], 0.5)
    assert np.isnan(y[0]) and y.view(np.uint32)[1] == 0x80000000
    y = _a("thresholdedrelu", [1.0, 1.5, -3.0, np.nan], 1.0)
    assert y[0] == 0.0 and y[1] == 1.5 and y[2] == 0.0 and y[3] == 0.0


def test_hardsigmoid_affine_softsign_points():
    y = _a("hardsigmoid", [2.0, -2.0, 1.0, 10.0, np.nan], 0.25, 0.5)
    assert list(y[:4]) == [1.0, 0.0, 0.75, 1.0] and np.isnan(y[4])
    assert list(_a("affine", [3.0, -1.0], 2.0, -1.0)) == [5.0, -3.0]
    assert list(_a("softsign", [1.0, -3.0, 0.0])) == [0.5, -0.75, 0.0]


def test_softplus_points():
    y = _a("softplus", [21.0, 25.0, 0.0, -30.0, 20.0])
    assert y[0] == 21.0 and y[1] == 25.0
    assert abs(float(y[2]) - math.log(2)) <= 2 * np.spacing(np.float32(math.log(2)))
    assert y[3] == 0.0                      # 1 + e^-30 rounds to 1 in fp32
    assert abs(float(y[4]) - 20.0) <= 2 * np.spacing(np.float32(20.0))


def test_elu_scaledtanh_points():
    y = _a("elu", [-1.0, 2.0, -0.0], 1.0)
    assert abs(float(y[0]) - (math.exp(-1) - 1)) <= 3 * np.spacing(np.float32(0.63))
    assert y[1] == 2.0 and y.view(np.uint32)[2] == 0x80000000
    y = _a("scaledtanh", [2.0], 2.0, 0.5)
    assert abs(float(y[0]) - 2 * math.tanh(1.0)) <= 4 * np.spacing(np.float32(1.5))
    # ScaledTanh with beta 0 (its default) is 0 for finite inputs
    assert list(_a("scaledtanh", [5.0, -3.0], 1.0, 0.0)) == [0.0, 0.0]


@pytest.mark.parametrize("name", ["sigmoid", "tanh", "elu", "softplus", "scaledtanh"])
def test_nan_propagates_through_transcendental_activations(name):
    assert np.isnan(_a(name, [np.nan], 1.0, 1.0)[0])


def test_softplus_elu_softsign_sweeps():
    x = np.linspace(-30, 30, 600_001).astype(np.float32)
    xd = x.astype(np.float64)
    ref = np.where(xd > 20, xd, np.log1p(np.exp(xd)))
    # log(1 + exp(x)) is evaluated literally: accurate to a few ulps of
    # max(1, result), not relative to tiny results for very negative x
    y = _a("softplus", x).astype(np.float64)
    scale = np.spacing(np.maximum(np.abs(ref), 1.0).astype(np.float32)).astype(np.float64)
    assert (np.abs(y - ref) / scale).max() <= 3.0
    neg = x[x < 0]
    ref = 0.7 * np.expm1(neg.astype(np.float64))
    y = _a("elu", neg, 0.7)
    # exp(x) - 1 is evaluated literally, so the error is absolute near 0
    assert np.abs(y - ref).max() <= 2 * np.spacing(np.float32(1.0))
    ref = xd / (1 + np.abs(xd))
    assert _ulps(_a("softsign", x), ref).max() <= 2.0   # two roundings
