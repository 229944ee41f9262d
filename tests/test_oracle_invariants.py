"""Invariants of the operator that the pages fix, checked on the oracle.

Page "Recurrent operators: RNN, GRU, LSTM": reverse is the forward recurrence
on each row's time-flipped valid prefix; a bidirectional layer is two
independent directions with their own activation sets (Activations); layout 1
is the layout-0 case with every tensor transposed, sequence_lens semantics,
zero-size and omitted inputs (Choices the specification leaves open).
OpenVINO "RNNCell" (Detailed description formula) and Apple BNNS "gru(...)"
(Discussion) restate one RNN step and the GRU with the reset gate applied
after the product.
"""
import math

import numpy as np
import pytest

import oracle
from onnx_recurrent_gb300.synth import make_case, random_case, workload
from helpers import assert_bits_equal, oracle_case


def _flip_valid(X, lens, layout):
    X = X.copy()
    N = X.shape[1] if layout == 0 else X.shape[0]
    S = X.shape[0] if layout == 0 else X.shape[1]
    for n in range(N):
        L = S if lens is None else int(lens[n])
        if layout == 0:
            X[:L, n] = X[:L, n][::-1]
        else:
            X[n, :L] = X[n, :L][::-1]
    return X


@pytest.mark.parametrize("seed", range(8))
def test_reverse_is_forward_on_flipped_rows(seed):
    c = random_case(seed, direction="reverse")
    Yr, Yhr, Ycr = oracle_case(c)
    f = c.with_(direction="forward", X=_flip_valid(c.X, c.sequence_lens, c.layout))
    Yf, Yhf, Ycf = oracle_case(f)
    Yf_back = _flip_valid(Yf[:, 0] if c.layout == 0 else Yf[:, :, 0], c.sequence_lens, c.layout)
    assert_bits_equal(Yr[:, 0] if c.layout == 0 else Yr[:, :, 0], Yf_back, "Y")
    assert_bits_equal(Yhr, Yhf, "Y_h")
    if Ycr is not None:
        assert_bits_equal(Ycr, Ycf, "Y_c")


def _split_dir(c, d, direction):
    sl = slice(d, d + 1)

    def st(a):
        if a is None:
            return None
        return a[sl] if c.layout == 0 else a[:, sl]
    acts = c.activations
    k = {"RNN": 1, "GRU": 2, "LSTM": 3}[c.op]
    return c.with_(direction=direction, W=c.W[sl], R=c.R[sl],
                   B=None if c.B is None else c.B[sl], P=None if c.P is None else c.P[sl],
                   initial_h=st(c.initial_h), initial_c=st(c.initial_c)), k, acts


@pytest.mark.parametrize("seed", range(8))
def test_bidirectional_is_two_directions(seed):
    c = random_case(seed, direction="bidirectional")
    Y, Yh, Yc = oracle_case(c)
    # resolved triples per direction, applied to unidirectional runs
    res = oracle.resolve_activations(c.op, "bidirectional", c.activations, c.alpha, c.beta)
    for d, direction in ((0, "forward"), (1, "reverse")):
        u, k, _ = _split_dir(c, d, direction)
        names = [t[0] for t in res[d]]
        alpha = [t[1] for t in res[d]]
        beta = [t[2] for t in res[d]]
        # give every activation its resolved alpha and beta explicitly
        acts, al, be = [], [], []
        for nm, a, b in zip(names, alpha, beta):
            acts.append(nm)
            if nm in ("affine", "leakyrelu", "thresholdedrelu", "scaledtanh", "hardsigmoid", "elu"):
                al.append(a)
            if nm in ("affine", "scaledtanh", "hardsigmoid"):
                be.append(b)
        Yd, Yhd, Ycd = oracle_case(u.with_(activations=acts, alpha=al, beta=be))
        ysl = (slice(None), slice(d, d + 1)) if c.layout == 0 else (slice(None), slice(None), slice(d, d + 1))
        ssl = (slice(d, d + 1),) if c.layout == 0 else (slice(None), slice(d, d + 1))
        assert_bits_equal(Y[ysl], Yd, f"Y dir {d}")
        assert_bits_equal(Yh[ssl], Yhd, f"Y_h dir {d}")
        if Yc is not None:
            assert_bits_equal(Yc[ssl], Ycd, f"Y_c dir {d}")


@pytest.mark.parametrize("seed", range(8))
def test_layout1_is_transposed_layout0(seed):
    c0 = random_case(seed, layout=0)
    Y0, Yh0, Yc0 = oracle_case(c0)

    def tr(a):
        return None if a is None else np.ascontiguousarray(a.transpose(1, 0, 2))
    c1 = c0.with_(layout=1, X=tr(c0.X), initial_h=tr(c0.initial_h), initial_c=tr(c0.initial_c))
    Y1, Yh1, Yc1 = oracle_case(c1)
    assert_bits_equal(Y1, Y0.transpose(2, 0, 1, 3), "Y")
    assert_bits_equal(Yh1, Yh0.transpose(1, 0, 2), "Y_h")
    if Yc0 is not None:
        assert_bits_equal(Yc1, Yc0.transpose(1, 0, 2), "Y_c")


@pytest.mark.parametrize("op", ["RNN", "GRU", "LSTM"])
def test_resumption_through_final_states(op):
    c = make_case(op, "forward", 9, 3, 5, 6, seed=3, with_P=True, h0_scale=0.5, c0_scale=0.5)
    Y, Yh, Yc = oracle_case(c)
    s = 4
    a = c.with_(seq=s, X=c.X[:s])
    Ya, Yha, Yca = oracle_case(a)
    b = c.with_(seq=c.seq - s, X=c.X[s:], initial_h=Yha, initial_c=Yca)
    Yb, Yhb, Ycb = oracle_case(b)
    assert_bits_equal(np.concatenate([Ya, Yb]), Y, "Y")
    assert_bits_equal(Yhb, Yh, "Y_h")
    if Yc is not None:
        assert_bits_equal(Ycb, Yc, "Y_c")


@pytest.mark.parametrize("seed", range(6))
def test_sequence_lens_semantics(seed):
    c = random_case(100 + seed, lens=("uniform", 0, 6), seq=6, batch=7, h0_scale=0.5)
    c.sequence_lens[0] = 0
    c.sequence_lens[-1] = c.seq
    Y, Yh, Yc = oracle_case(c)
    for d in range(c.dirs):
        rev = c.direction == "reverse" or d == 1
        for n in range(c.batch):
            L = int(c.sequence_lens[n])
            yn = Y[:, d, n] if c.layout == 0 else Y[n, :, d]
            yh = Yh[d, n] if c.layout == 0 else Yh[n, d]
            assert np.all(yn[L:].view(np.uint32) == 0)
            if L == 0:
                assert np.all(yh.view(np.uint32) == 0)
                if Yc is not None:
                    yc = Yc[d, n] if c.layout == 0 else Yc[n, d]
                    assert np.all(yc.view(np.uint32) == 0)
            else:
                assert_bits_equal(yh, yn[0] if rev else yn[L - 1], "Y_h is the last valid step")


def test_gru_lbr_equal_when_recurrence_is_zero():
    c = make_case("GRU", "forward", 4, 3, 5, 6, seed=5, h0_scale=0.5)
    c.R[:] = 0.0
    c.B[:, 3 * 6 + 12:] = 0.0           # Rbh = 0
    Y0, Yh0, _ = oracle_case(c.with_(linear_before_reset=0))
    Y1, Yh1, _ = oracle_case(c.with_(linear_before_reset=1))
    np.testing.assert_array_equal(Y0, Y1)
    np.testing.assert_array_equal(Yh0, Yh1)


def test_gru_lbr_differ_in_general():
    c = make_case("GRU", "forward", 3, 2, 4, 5, seed=6, h0_scale=0.5)
    Y0, _, _ = oracle_case(c.with_(linear_before_reset=0))
    Y1, _, _ = oracle_case(c.with_(linear_before_reset=1))
    assert not np.array_equal(Y0, Y1)


@pytest.mark.parametrize("op", ["RNN", "GRU", "LSTM"])
def test_zero_size(op):
    c = make_case(op, "bidirectional", 0, 3, 4, 5, seed=1, h0_scale=0.5, c0_scale=0.5,
                  lens=[0, 0, 0])
    Y, Yh, Yc = oracle_case(c)
    assert Y.size == 0
    assert_bits_equal(Yh, c.initial_h, "Y_h = initial_h")
    if op == "LSTM":
        assert_bits_equal(Yc, c.initial_c, "Y_c = initial_c")
    c2 = c.with_(initial_h=None, initial_c=None)
    _, Yh2, Yc2 = oracle_case(c2)
    assert np.all(Yh2 == 0)
    c3 = make_case(op, "forward", 4, 0, 4, 5, seed=1)
    Y3, Yh3, _ = oracle_case(c3)
    assert Y3.size == 0 and Yh3.size == 0


def test_absent_and_zero_initial_state_agree():
    c = workload("rnn_fwd_s8_b1_i16_h128")
    z = workload("rnn_fwd_s8_b1_i16_h128", initial_h_zero=True)
    a = oracle_case(c)
    b = oracle_case(z)
    for x, y in zip(a[:2], b[:2]):
        assert_bits_equal(x, y)


def test_invalid_lengths_and_arguments():
    c = make_case("GRU", "forward", 4, 3, 2, 3, seed=2, lens=[1, 5, 2])
    with pytest.raises(oracle.OracleError) as e:
        oracle_case(c)
    assert e.value.status == 2
    with pytest.raises(oracle.OracleError) as e:
        oracle_case(c.with_(sequence_lens=np.array([1, -1, 2], np.int32)))
    assert e.value.status == 2
    ok = c.with_(sequence_lens=np.array([4, 0, 2], np.int32))
    oracle_case(ok)
    for bad in (dict(hidden_size=0), dict(activations=["Sigmoid"]),
                dict(activations=["Sigmoid", "NoSuchFn"]), dict(layout=2),
                dict(linear_before_reset=3)):
        with pytest.raises(oracle.OracleError) as e:
            oracle_case(ok, **bad)
        assert e.value.status == 1


# ------------------------------------------------------------ activations

def test_resolve_page_black_box_case():
    # The page's cursor case: HardSigmoid, LeakyRelu, ScaledTanh with
    # alpha [0.3, 0.2, 1.2] and beta [0.4, 0.7] (separate cursors).
    r = oracle.resolve_activations("LSTM", "forward", ["HardSigmoid", "LeakyRelu", "ScaledTanh"],
                                   [0.3, 0.2, 1.2], [0.4, 0.7])
    f32 = lambda v: float(np.float32(v))
    assert r == [[("hardsigmoid", f32(0.3), f32(0.4)), ("leakyrelu", f32(0.2), 0.0),
                  ("scaledtanh", f32(1.2), f32(0.7))]]


def test_resolve_lstm_bidi_workload():
    c = workload("lstm_bidi_s512_b128_i1024_h1024")
    r = oracle.resolve_activations(c.op, c.direction, c.activations, c.alpha, c.beta)
    f32 = lambda v: float(np.float32(v))
    assert r[0] == [("hardsigmoid", 0.25, f32(0.45)), ("leakyrelu", f32(0.05), 0.0),
                    ("scaledtanh", 1.5, f32(0.8))]
    assert [t[0] for t in r[1]] == ["sigmoid", "tanh", "tanh"]


def test_resolve_defaults_and_case_and_single_set():
    assert oracle.resolve_activations("GRU", "bidirectional") == \
        [[("sigmoid", 0.0, 0.0), ("tanh", 0.0, 0.0)]] * 2
    assert oracle.resolve_activations("RNN", "forward") == [[("tanh", 0.0, 0.0)]]
    r = oracle.resolve_activations("RNN", "bidirectional", ["leakyRELU"])
    assert r == [[("leakyrelu", float(np.float32(0.01)), 0.0)]] * 2
    r = oracle.resolve_activations("RNN", "bidirectional", ["Affine", "HardSigmoid"], [2.0], [3.0])
    assert r == [[("affine", 2.0, 3.0)], [("hardsigmoid", float(np.float32(0.2)), 0.5)]]
    r = oracle.resolve_activations("RNN", "reverse", ["Elu", "Relu"], [0.5])
    assert r == [[("elu", 0.5, 0.0)]]


def test_resolve_every_default_the_page_lists():
    # Activations: missing values take the activation's own defaults, as the
    # page lists them: LeakyRelu 0.01, ThresholdedRelu 1, Elu 1, HardSigmoid
    # 0.2 and 0.5, Affine and ScaledTanh 1 and 0.
    f32 = lambda v: float(np.float32(v))
    page = {"LeakyRelu": (f32(0.01), 0.0), "ThresholdedRelu": (1.0, 0.0), "Elu": (1.0, 0.0),
            "HardSigmoid": (f32(0.2), 0.5), "Affine": (1.0, 0.0), "ScaledTanh": (1.0, 0.0)}
    for name, (alpha, beta) in page.items():
        r = oracle.resolve_activations("RNN", "forward", [name])
        assert r == [[(name.lower(), alpha, beta)]], name
    # one of the pair given: the other keeps its default
    assert oracle.resolve_activations("RNN", "forward", ["ScaledTanh"], None, [0.5]) == \
        [[("scaledtanh", 1.0, 0.5)]]
    assert oracle.resolve_activations("RNN", "forward", ["Affine"], [3.0]) == [[("affine", 3.0, 0.0)]]


# ------------------------------------------------------ cross-statements

def _np_act(name, x):
    return {"relu": lambda v: np.maximum(v, 0), "sigmoid": lambda v: 1 / (1 + np.exp(-v)),
            "tanh": np.tanh}[name](x)


@pytest.mark.parametrize("act", ["tanh", "sigmoid", "relu"])
def test_rnncell3_one_step(act):
    # OpenVINO RNNCell-3: Ht = f(Xt*Wi^T + Ht-1*Ri^T + Wbi + Rbi), with the
    # example's shapes (X 1x16, H 1x128, W 128x16, R 128x128, B 128).
    c = make_case("RNN", "forward", 1, 1, 16, 128, seed=4, x_dist=("uniform", -1, 1),
                  h0_scale=0.5, activations=[act.capitalize()])
    Y, Yh, _ = oracle_case(c)
    X, W, R, B, h = (c.X[0].astype(np.float64), c.W[0].astype(np.float64),
                     c.R[0].astype(np.float64), c.B[0].astype(np.float64),
                     c.initial_h[0].astype(np.float64))
    ref = _np_act(act, X @ W.T + h @ R.T + (B[:128] + B[128:]))
    np.testing.assert_allclose(Yh[0], ref, rtol=0, atol=2e-6)
    np.testing.assert_array_equal(Y[0], Yh)


def test_bnns_gru_reset_after_matmul():
    # Apple BNNS gru(..., applyResetGateAfterMatMul: true): gate blocks r, n, z;
    # n = A(W_in x + b_in + (W_hn h + b_hn) * r); h' = (1 - z) * n + z * h.
    c = make_case("GRU", "forward", 3, 2, 6, 5, seed=9, h0_scale=0.5, linear_before_reset=1)
    Y, Yh, _ = oracle_case(c)
    H = 5
    W, R, B = (c.W[0].astype(np.float64), c.R[0].astype(np.float64), c.B[0].astype(np.float64))
    blk = lambda M, g: M[g * H:(g + 1) * H]          # ONNX order z=0, r=1, h=2
    Wiz, Wir, Win = blk(W, 0), blk(W, 1), blk(W, 2)
    Whz, Whr, Whn = blk(R, 0), blk(R, 1), blk(R, 2)
    biz, bir, bin_ = blk(B, 0), blk(B, 1), blk(B, 2)
    bhz, bhr, bhn = blk(B[3 * H:], 0), blk(B[3 * H:], 1), blk(B[3 * H:], 2)
    sig = lambda v: 1 / (1 + np.exp(-v))
    h = c.initial_h[0].astype(np.float64)
    for t in range(c.seq):
        x = c.X[t].astype(np.float64)
        r = sig(x @ Wir.T + bir + h @ Whr.T + bhr)
        z = sig(x @ Wiz.T + biz + h @ Whz.T + bhz)
        n = np.tanh(x @ Win.T + bin_ + (h @ Whn.T + bhn) * r)
        h = (1 - z) * n + z * h
        np.testing.assert_allclose(Y[t, 0], h, rtol=0, atol=3e-6)
    np.testing.assert_allclose(Yh[0], h, rtol=0, atol=3e-6)
