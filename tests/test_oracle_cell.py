"""Pins for the single-cell oracle (page "RNNCell", RNNCell-3):
hand-derived dyadic cases, float64 brute force within the rounding bound,
the page's default activation and clip, and the sequence operator at one
step (the summed bias given as Wb with Rb = -0, which adds nothing)."""
import glob
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "cell")
FILES = sorted(glob.glob(os.path.join(GOLDEN, "*.json")))
ACTS = ["Relu", "Sigmoid", "Tanh"]


def _draw(seed, N, I, H, w=None):
    g = np.random.default_rng(seed)
    s = 1.0 / np.sqrt(H) if w is None else w
    X = g.uniform(-1, 1, (N, I)).astype(np.float32)
    Hp = g.uniform(-0.5, 0.5, (N, H)).astype(np.float32)
    W = g.uniform(-s, s, (H, I)).astype(np.float32)
    R = g.uniform(-s, s, (H, H)).astype(np.float32)
    B = g.uniform(-0.1, 0.1, H).astype(np.float32)
    return X, Hp, W, R, B


def _f64(act, v):
    return {"relu": lambda x: np.maximum(x, 0), "sigmoid": lambda x: 1 / (1 + np.exp(-x)),
            "tanh": np.tanh}[act.lower()](v)


@pytest.mark.parametrize("path", FILES, ids=[os.path.basename(p) for p in FILES])
def test_cell_golden(path):
    with open(path) as f:
        fx = json.load(f)
    assert fx["citation"] and fx["derivation"]
    a, i = fx["attrs"], {k: np.array(v, np.float32) for k, v in fx["inputs"].items()}
    Ho = oracle.rnn_cell(a["hidden_size"], a["input_size"], i["X"], i["H"], i["W"], i["R"], i["B"],
                         activation=a["activation"], clip=a.get("clip", float("inf")))
    np.testing.assert_array_equal(Ho, np.array(fx["expected"]["Ho"], np.float32))


@pytest.mark.parametrize("seed", range(6))
def test_cell_matches_float64(seed):
    # |fp32 - exact| of each dot is at most gamma_K * sum |a||b| (K products and
    # sums, each rounded once); the activations are 1-Lipschitz and add a few ulp.
    N, I, H = 3, 5 + seed, 4 + 2 * seed
    X, Hp, W, R, B = _draw(seed, N, I, H, w=0.7)
    act = ACTS[seed % 3]
    clip = [float("inf"), 0.6][seed % 2]
    Ho = oracle.rnn_cell(H, I, X, Hp, W, R, B, activation=act, clip=clip)
    Xd, Hd, Wd, Rd, Bd = (v.astype(np.float64) for v in (X, Hp, W, R, B))
    pre = Xd @ Wd.T + Hd @ Rd.T + Bd
    ref = _f64(act, np.clip(pre, -clip, clip))
    u = 2.0 ** -24
    K = I + H + 1
    bound = (K * u / (1 - K * u)) * (np.abs(Xd) @ np.abs(Wd).T + np.abs(Hd) @ np.abs(Rd).T + np.abs(Bd)) + 4e-7
    assert np.all(np.abs(Ho - ref) <= bound), np.max(np.abs(Ho - ref) - bound)


def test_cell_default_activation_is_tanh_and_default_clip_clamps_nothing():
    X, Hp, W, R, B = _draw(11, 2, 6, 8, w=3.0)          # large pre-activations
    Ho = oracle.rnn_cell(8, 6, X, Hp, W, R, B, activation=None)
    pre = X.astype(np.float64) @ W.T.astype(np.float64) + Hp.astype(np.float64) @ R.T.astype(np.float64) + B
    assert np.max(np.abs(pre)) > 2.0
    np.testing.assert_allclose(Ho, np.tanh(pre), rtol=0, atol=1e-5)


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("clip", [None, 0.25])
def test_cell_is_the_sequence_operator_at_one_step(act, clip):
    # Sequence operator, seq 1, forward, B = [Wb | Rb] with Wb = the summed
    # bias and Rb = -0: pre = ((xw + rec) + B) + (-0) = (xw + rec) + B for
    # every value, so the two must agree bit for bit.
    N, I, H = 4, 9, 12
    X, Hp, W, R, B = _draw(5, N, I, H, w=0.9)
    Ho = oracle.rnn_cell(H, I, X, Hp, W, R, B, activation=act, clip=float("inf") if clip is None else clip)
    Bs = np.concatenate([B, np.full(H, -0.0, np.float32)])[None]
    Y, Yh, _ = oracle.rnn("RNN", "forward", H, I, X[None], W[None], R[None], B=Bs, initial_h=Hp[None],
                          activations=[act], clip=clip)
    np.testing.assert_array_equal(Ho.view(np.uint32), Yh[0].view(np.uint32))
    np.testing.assert_array_equal(Ho.view(np.uint32), Y[0, 0].view(np.uint32))


def test_cell_clip_saturates_exactly():
    X = np.array([[100.0], [-100.0]], np.float32)
    W = np.ones((1, 1), np.float32)
    R = np.zeros((1, 1), np.float32)
    Hp = np.zeros((2, 1), np.float32)
    B = np.zeros(1, np.float32)
    np.testing.assert_array_equal(oracle.rnn_cell(1, 1, X, Hp, W, R, B, "Relu", clip=2.5)[:, 0], [2.5, 0.0])
    np.testing.assert_array_equal(oracle.rnn_cell(1, 1, X, Hp, W, R, B, "Tanh", clip=2.5)[:, 0],
                                  oracle.tanh(np.array([2.5, -2.5], np.float32)))


def test_cell_nan_is_canonical():
    # the quiet NaN and a negative NaN with a payload both come out as 0x7FC00000
    for bits in (0x7FC00000, 0xFFA00001):
        X = np.array([[bits]], np.uint32).view(np.float32)
        Ho = oracle.rnn_cell(1, 1, X, np.zeros((1, 1), np.float32), np.ones((1, 1), np.float32),
                             np.ones((1, 1), np.float32), np.zeros(1, np.float32), "Relu")
        assert Ho.view(np.uint32)[0, 0] == 0x7FC00000, hex(bits)


@pytest.mark.parametrize("bad", [dict(activation="Affine"), dict(activation="LeakyRelu"),
                                 dict(activation="nope"), dict(clip=0.0), dict(clip=-1.0),
                                 dict(clip=float("nan"))])
def test_cell_rejects_what_the_page_excludes(bad):
    X, Hp, W, R, B = _draw(1, 1, 2, 3)
    kw = dict(activation="Tanh", clip=float("inf"))
    kw.update(bad)
    with pytest.raises(oracle.OracleError) as e:
        oracle.rnn_cell(3, 2, X, Hp, W, R, B, **kw)
    assert e.value.status == 1


def test_cell_empty_batch():
    X, Hp, W, R, B = _draw(1, 0, 2, 3)
    assert oracle.rnn_cell(3, 2, X, Hp, W, R, B).shape == (0, 3)
