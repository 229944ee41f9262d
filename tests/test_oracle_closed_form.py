"""Closed forms: with Affine(1, 0) (or Relu on non-negative data) the RNN is
the linear recurrence h_t = W x_t + R h_{t-1} + Wb + Rb ("Recurrent
operators: RNN, GRU, LSTM", Computation; OpenVINO RNNCell-3, Detailed
description).  With small integers every fp32 operation is exact, so the
oracle must equal the matrix-power closed form
    h_T = R^(T+1) h0 + sum_{s<=T} R^(T-s) (W x_s + b)
computed here in exact integer arithmetic."""
import numpy as np
import pytest

import oracle


def closed_form(X, W, R, b, h0):
    """X [S, N, I] ints; W [H, I]; R [H, H]; b [H]; h0 [N, H] -> Y [S, N, H] (Python ints)."""
    S = X.shape[0]
    Wo, Ro = W.astype(object), R.astype(object)
    powers = [np.eye(R.shape[0], dtype=object)]
    for _ in range(S + 1):
        powers.append(powers[-1].dot(Ro))
    Y = np.zeros((S,) + h0.shape, dtype=object)
    for T in range(S):
        for n in range(h0.shape[0]):
            acc = powers[T + 1].dot(h0[n].astype(object))
            for s in range(T + 1):
                acc = acc + powers[T - s].dot(Wo.dot(X[s, n].astype(object)) + b.astype(object))
            Y[T, n] = acc
    return Y


@pytest.mark.parametrize("seed", range(4))
def test_affine_rnn_matches_integer_closed_form(seed):
    rng = np.random.default_rng(seed)
    S, N, I, H = 5, 3, 3, 4
    X = rng.integers(-3, 4, (S, N, I))
    W = rng.integers(-2, 3, (H, I))
    R = rng.integers(-1, 2, (H, H))
    Wb = rng.integers(-4, 5, H)
    Rb = rng.integers(-4, 5, H)
    h0 = rng.integers(-3, 4, (N, H))
    ref = closed_form(X, W, R, Wb + Rb, h0)
    assert np.abs(ref).max() < 2 ** 24
    Y, Yh, _ = oracle.rnn("RNN", "forward", H, I, X.astype(np.float32), W[None].astype(np.float32),
                          R[None].astype(np.float32),
                          B=np.concatenate([Wb, Rb])[None].astype(np.float32),
                          initial_h=h0[None].astype(np.float32), activations=["Affine"],
                          alpha=[1.0], beta=[0.0])
    np.testing.assert_array_equal(Y[:, 0], ref.astype(np.float32))
    np.testing.assert_array_equal(Yh[0], ref[-1].astype(np.float32))


def test_affine_alpha_beta_closed_form():
    # Affine(2, 1): h_t = 2 (W x_t + R h_{t-1}) + 1, i.e. the linear form with
    # W' = 2W, R' = 2R, b' = 1.
    rng = np.random.default_rng(7)
    S, N, I, H = 4, 2, 2, 3
    X = rng.integers(-2, 3, (S, N, I))
    W = rng.integers(-1, 2, (H, I))
    R = rng.integers(-1, 2, (H, H))
    h0 = rng.integers(-2, 3, (N, H))
    ref = closed_form(X, 2 * W, 2 * R, np.ones(H, dtype=np.int64), h0)
    Y, _, _ = oracle.rnn("RNN", "forward", H, I, X.astype(np.float32), W[None].astype(np.float32),
                         R[None].astype(np.float32), initial_h=h0[None].astype(np.float32),
                         activations=["Affine"], alpha=[2.0], beta=[1.0])
    np.testing.assert_array_equal(Y[:, 0], ref.astype(np.float32))


def test_relu_nonnegative_is_linear():
    rng = np.random.default_rng(3)
    S, N, I, H = 4, 2, 3, 3
    X = rng.integers(0, 3, (S, N, I))
    W = rng.integers(0, 2, (H, I))
    R = rng.integers(0, 2, (H, H))
    Wb = rng.integers(0, 3, H)
    Rb = rng.integers(0, 3, H)
    h0 = rng.integers(0, 3, (N, H))
    ref = closed_form(X, W, R, Wb + Rb, h0)
    Y, _, _ = oracle.rnn("RNN", "forward", H, I, X.astype(np.float32), W[None].astype(np.float32),
                         R[None].astype(np.float32),
                         B=np.concatenate([Wb, Rb])[None].astype(np.float32),
                         initial_h=h0[None].astype(np.float32), activations=["Relu"])
    np.testing.assert_array_equal(Y[:, 0], ref.astype(np.float32))


def test_reverse_affine_closed_form():
    # Reverse direction: the recurrence runs from t = S-1 down to 0.
    rng = np.random.default_rng(11)
    S, N, I, H = 4, 2, 2, 3
    X = rng.integers(-2, 3, (S, N, I))
    W = rng.integers(-1, 2, (H, I))
    R = rng.integers(-1, 2, (H, H))
    h0 = rng.integers(-2, 3, (N, H))
    ref = closed_form(X[::-1], W, R, np.zeros(H, dtype=np.int64), h0)[::-1]
    Y, Yh, _ = oracle.rnn("RNN", "reverse", H, I, X.astype(np.float32), W[None].astype(np.float32),
                          R[None].astype(np.float32), initial_h=h0[None].astype(np.float32),
                          activations=["Affine"])
    np.testing.assert_array_equal(Y[:, 0], ref.astype(np.float32))
    np.testing.assert_array_equal(Yh[0], ref[0].astype(np.float32))
