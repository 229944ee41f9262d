"""Special values on the GPU against the oracle, bit for bit in exact mode.

Page "Recurrent operators: RNN, GRU, LSTM":
  - Exact mode: every NaN written to Y, Y_h and Y_c is 0x7FC00000;
  - Activations: Relu keeps a NaN (and -0), ThresholdedRelu is x > alpha ? x : 0,
    Softplus is x past 20, log(1 + exp(x)) below, HardSigmoid clamps
    alpha * x + beta to [0, 1], Elu is alpha * (exp(x) - 1) below 0;
  - Computation: clip clamps every gate input to [-clip, clip] and lets a
    NaN through; the bias adds are skipped when B is absent;
  - Choices the specification leaves open: a row of length 0 has final
    states +0 whatever its initial state, and Y is +0 past every row's length.

The pre-activations are placed exactly: with W = 0 and R = 0 every product
is +0 (for finite operands), so a gate's input is its bias Wb (Rb = +0), and
each hidden unit carries one edge value of the activations (exp's overflow at
89 and underflow at -110, tanh's 0.4 and 9.1 branch points, Softplus' 20,
ThresholdedRelu's alpha, the clip edges, subnormals, +-0, +-inf, NaN).  The
cell state, peepholes, initial states and X carry NaN, infinities, -0 and
subnormals in chosen places, and a second family runs random weights with
such values planted in single rows (rows never interact, so the rest stays
finite).  Every recurrent kernel runs each case: the staged kernel (one CTA,
several CTAs, streamed R) and the dataflow kernel (resident and streamed R),
and the single-cell kernel takes the same edges.  Fast mode is checked on
the same cases for NaN positions, infinity signs and the 1e-5 bound."""
import numpy as np
import pytest

import onnx_recurrent_gb300 as orc
import oracle
from gpu_helpers import gpu_case
from helpers import assert_bits_equal, oracle_case
from onnx_recurrent_gb300.synth import make_case

pytestmark = pytest.mark.gpu

F = np.float32
INF = F(np.inf)
NAN = F(np.nan)
NEG_NAN = np.array([0xFFC00000], np.uint32).view(np.float32)[0]
SNAN = np.array([0x7FA00001], np.uint32).view(np.float32)[0]


def nxt(x, toward):
    return np.nextafter(F(x), F(toward))


THRESH_ALPHA = F(1.5)

# One edge value per hidden unit (56 units: a multiple of 4, as the dataflow
# kernel's 16-byte loads want).
EDGES = np.array([
    0.0, -0.0, 1e-45, -1e-45, 1e-40, -1e-40, 1.17549435e-38, -1.17549435e-38,
    0.4, nxt(0.4, 0), nxt(0.4, 1), -0.4, 9.1, nxt(9.1, 10), nxt(9.1, 0), -9.1,
    20.0, nxt(20, 21), nxt(20, 19), -20.0, 88.72, 89.0, nxt(89, 90), 100.0,
    -87.5, -103.0, -110.0, nxt(-110, -111), -150.0, 0.5, -0.5, 1.0,
    -1.0, 2.5, -2.5, 5.0, -5.0, 3.0, nxt(3, 4), nxt(3, 0),
    -3.0, nxt(-3, -4), THRESH_ALPHA, nxt(THRESH_ALPHA, 2), nxt(THRESH_ALPHA, 1), 3e38, -3e38, INF,
    -INF, NAN, NEG_NAN, SNAN, 0.1, -0.1, 15.0, -15.0,
], np.float32)
H_EDGE = len(EDGES)
FINITE_EDGES = np.where(np.isfinite(EDGES) & (np.abs(EDGES) < 1e3), EDGES, F(0.75)).astype(np.float32)

# (unit_groups, rows_per_thread, r_resident, row_groups, kernel): the planner's
# choice, the staged kernel with one and with several CTAs, streamed R, and the
# dataflow kernel with resident and streamed R, one row per thread or a tile
# of four rows (units fastest across the lanes, rows ranked by length), and
# the dataflow kernel exchanging h inside a cluster of 4 or 7 CTAs.
KERNELS = {
    "planner": None,
    "staged-1cta": (1, 1, 1, 0, 1),
    "staged-3cta": (3, 2, 1, 0, 1),
    "staged-streamed": (2, 1, 0, 0, 1),
    "dataflow": (4, 1, 1, 1, 2),
    "dataflow-streamed": (3, 1, 0, 1, 2),
    "dataflow-wide": (3, 4, 0, 1, 2),
    "cluster": (4, 1, -1, 1, 5),
    "cluster-2rows": (7, 2, -1, 0, 5),
}

# (op, direction, activations, alpha, beta, lbr, input_forget)
OPS = {
    "rnn-relu-tanh": ("RNN", "bidirectional", ["Relu", "Tanh"], None, None, 0, 0),
    "rnn-sigmoid-affine": ("RNN", "bidirectional", ["Sigmoid", "Affine"], [-1.0], [-0.0], 0, 0),
    "rnn-leaky-thresholded": ("RNN", "bidirectional", ["LeakyRelu", "ThresholdedRelu"],
                              [0.1, float(THRESH_ALPHA)], None, 0, 0),
    "rnn-scaledtanh-hardsigmoid": ("RNN", "bidirectional", ["ScaledTanh", "HardSigmoid"],
                                   [-1.25, -0.2], [0.5, -0.0], 0, 0),
    "rnn-elu-softsign": ("RNN", "bidirectional", ["Elu", "Softsign"], [0.75], None, 0, 0),
    "rnn-softplus": ("RNN", "forward", ["Softplus"], None, None, 0, 0),
    "gru-lbr0": ("GRU", "bidirectional", None, None, None, 0, 0),
    "gru-lbr1": ("GRU", "bidirectional", None, None, None, 1, 0),
    "gru-hardsigmoid-scaledtanh": ("GRU", "reverse", ["HardSigmoid", "ScaledTanh"], [0.25, -1.0], [0.45, 0.8],
                                   0, 0),
    "lstm": ("LSTM", "bidirectional", None, None, None, 0, 0),
    "lstm-forget-coupled": ("LSTM", "forward", ["HardSigmoid", "LeakyRelu", "ScaledTanh"], [0.25, 0.05, 1.5],
                            [0.45, 0.8], 0, 1),
    "lstm-elu-softplus": ("LSTM", "reverse", ["Sigmoid", "Elu", "Softplus"], [0.5], None, 0, 0),
}


def edge_case(name, clip, seq=2, edges=EDGES, with_B=True):
    """W = R = 0; Wb[g][u] = edges rolled by 7g units (every gate sees every
    edge, in different pairings; GRU's reset gate with linear_before_reset = 0
    the finite ones only), Rb = +0; planted NaN / infinities / -0 /
    subnormals in X, the initial states and the peepholes; four rows with
    lengths [seq, 1, seq, 0] (the last row, of length 0, starts from NaN)."""
    op, direction, acts, alpha, beta, lbr, inf_ = OPS[name]
    H = len(edges)
    c = make_case(op, direction, seq, 4, 6, H, seed=71, with_P=True, h0_scale=0.5, c0_scale=0.5,
                  lens=[seq, 1, seq, 0], clip=clip, activations=acts, alpha=alpha, beta=beta,
                  linear_before_reset=lbr, input_forget=inf_, with_B=with_B)
    G, D = c.gates, c.dirs
    c.W[...] = 0.0
    c.R[...] = 0.0
    if with_B:
        c.B[...] = 0.0
        for d in range(D):
            for g in range(G):
                c.B[d, g * H:(g + 1) * H] = np.roll(edges, 7 * g + 3 * d)
            if op == "GRU" and lbr == 0:
                # the candidate's product sums r (.) h over every unit: one NaN
                # reset gate would turn the whole step to NaN, so r sees the
                # finite edges only (z and the candidate keep them all)
                fin = np.where(np.isfinite(edges), edges, F(0.75)).astype(np.float32)
                c.B[d, H:2 * H] = np.roll(fin, 7 + 3 * d)
    # X: row 1 NaN at t = 1 (past its length: must not leak), row 2 +inf at t = 0
    X = c.X
    if c.layout == 0:
        X[min(1, seq - 1), 1, 2] = NAN
        X[0, 2, 0] = INF
    # initial states: row 0 finite specials, row 3 (length 0) NaN
    h0, c0 = c.initial_h, c.initial_c
    for d in range(D):
        h0[d, 0, :8] = [-0.0, 1e-45, -1e-40, 3e38, -3e38, 0.0, -0.0, 1e-38]
        h0[d, 3, 5] = NAN
        if c0 is not None:
            c0[d, 0, :8] = [NAN, INF, -INF, -0.0, 1e-45, 3e38, -0.0, -1e-42]
            c0[d, 3, 1] = NAN
    if c.P is not None:
        for d in range(D):
            c.P[d, [9, 10, 11, 12]] = [NAN, INF, -0.0, 3e38]                  # Pi
            c.P[d, H + np.array([13, 14, 15])] = [-INF, 1e-45, -0.0]          # Po
            c.P[d, 2 * H + np.array([16, 17, 18])] = [INF, NAN, 1e-40]        # Pf
    return c


def _exact(c, launch):
    got = gpu_case(c, "exact", launch=launch)
    ref = oracle_case(c)
    for name, g, r in zip(("Y", "Y_h", "Y_c"), got, ref):
        if r is None:
            continue
        assert_bits_equal(g, r, f"{name}")
        nan = np.isnan(g)
        assert np.all(g[nan].view(np.uint32) == 0x7FC00000), f"{name}: a NaN is not 0x7FC00000"
    return got


@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("clip", [None, 3.0], ids=["noclip", "clip3"])
@pytest.mark.parametrize("name", sorted(OPS))
def test_activation_edges_bit_identical(name, clip, kernel):
    c = edge_case(name, clip)
    got = _exact(c, KERNELS[kernel])
    # the planted edges must reach the outputs: some NaN and some value that is
    # neither 0 nor NaN (a run that zeroed everything would otherwise pass)
    Y = got[0]
    assert np.isnan(Y).any() and (np.isfinite(Y) & (Y != 0)).any()


@pytest.mark.parametrize("kernel", ["planner", "staged-3cta", "dataflow-streamed"])
@pytest.mark.parametrize("name", ["rnn-sigmoid-affine", "rnn-scaledtanh-hardsigmoid", "gru-hardsigmoid-scaledtanh",
                                  "lstm-forget-coupled"])
def test_bias_absent_keeps_negative_zero(name, kernel):
    # B absent: no add can turn a -0 made by an activation (ScaledTanh or
    # Affine with a negative alpha, beta = -0) into +0; the outputs must keep
    # the oracle's signs of zero bit for bit
    c = edge_case(name, None, with_B=False)
    got = _exact(c, KERNELS[kernel])
    assert any((g.view(np.uint32) == 0x80000000).any() for g in got if g is not None) or name.startswith("lstm")


@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("name", ["rnn-relu-tanh", "rnn-elu-softsign", "gru-lbr0", "gru-lbr1", "lstm",
                                  "lstm-elu-softplus"])
def test_finite_edges_through_random_recurrence(name, kernel):
    # three steps with random R: the finite edges' outputs (saturated,
    # underflowed, subnormal) feed the next steps' products
    c = edge_case(name, 3.0, seq=3, edges=FINITE_EDGES)
    rng = np.random.default_rng(5)
    c.R[...] = rng.uniform(-0.2, 0.2, c.R.shape).astype(np.float32)
    c.W[...] = rng.uniform(-0.2, 0.2, c.W.shape).astype(np.float32)
    _exact(c, KERNELS[kernel])


def planted_rows_case(op, direction, lbr=0, layout=0, seed=3):
    """Random weights; each batch row carries one kind of special value in X
    (row 0 -0, 1 NaN, 2 +inf, 3 -inf, 4 1e30, 5 a subnormal, 6 none), the
    initial states of rows 1 and 4 carry NaN and an infinity, B and P carry
    finite extremes."""
    c = make_case(op, direction, 6, 8, 12, 40, seed=seed, layout=layout, with_P=True, h0_scale=0.5,
                  c0_scale=0.5, lens=[6, 3, 6, 5, 6, 0, 6, 2], linear_before_reset=lbr, clip=None)
    vals = [F(-0.0), NAN, INF, -INF, F(1e30), F(1e-44)]
    for n, v in enumerate(vals):
        t = 2 if n != 5 else 0
        if layout == 0:
            c.X[t, n, 3] = v
            c.X[t + 1, n, :] = v if n in (0, 5) else c.X[t + 1, n, :]
        else:
            c.X[n, t, 3] = v
            c.X[n, t + 1, :] = v if n in (0, 5) else c.X[n, t + 1, :]
    D = c.dirs
    for d in range(D):
        if layout == 0:
            c.initial_h[d, 1, 4] = NAN
            c.initial_h[d, 4, 7] = INF
            if c.initial_c is not None:
                c.initial_c[d, 1, 2] = -INF
                c.initial_c[d, 6, 0] = -0.0
        else:
            c.initial_h[1, d, 4] = NAN
            c.initial_h[4, d, 7] = INF
            if c.initial_c is not None:
                c.initial_c[1, d, 2] = -INF
                c.initial_c[6, d, 0] = -0.0
    c.B[:, 5] = 3e38
    c.B[:, 6] = -3e38
    c.B[:, 7] = -0.0
    c.B[:, 8] = 1e-42
    if c.P is not None:
        c.P[:, 3] = 1e30
        c.P[:, 4] = -0.0
    return c


PLANTED = [("RNN", "bidirectional", 0, 0), ("GRU", "forward", 0, 1), ("GRU", "bidirectional", 1, 0),
           ("LSTM", "bidirectional", 0, 1), ("LSTM", "reverse", 0, 0)]


@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("op,direction,lbr,layout", PLANTED, ids=[f"{p[0]}-{p[1]}-lbr{p[2]}-l{p[3]}" for p in PLANTED])
def test_planted_rows_bit_identical(op, direction, lbr, layout, kernel):
    c = planted_rows_case(op, direction, lbr, layout)
    got = _exact(c, KERNELS[kernel])
    # rows never interact: the row without planted values stays finite
    Y = got[0]
    row6 = Y[:, :, 6] if layout == 0 else Y[6]
    assert np.isfinite(row6).all()


def _fast_agrees(got, ref, tol=1e-5):
    for name, g, r in zip(("Y", "Y_h", "Y_c"), got, ref):
        if r is None:
            continue
        g64, r64 = g.astype(np.float64), r.astype(np.float64)
        assert np.array_equal(np.isnan(g64), np.isnan(r64)), f"{name}: NaN positions differ"
        assert np.all(g[np.isnan(g)].view(np.uint32) == 0x7FC00000), f"{name}: non-canonical NaN"
        big = ~np.isnan(r64) & (~np.isfinite(r64) | (np.abs(r64) > 1e30))
        assert np.array_equal(np.sign(g64[big]), np.sign(r64[big])), f"{name}: signs of huge values differ"
        ok = ~np.isnan(r64) & ~big
        err = np.abs(g64[ok] - r64[ok]) / np.maximum(1.0, np.abs(r64[ok]))
        assert float(err.max(initial=0.0)) <= tol, f"{name}: {float(err.max()):.3e}"


@pytest.mark.parametrize("kernel", ["planner", "staged-3cta", "dataflow"])
@pytest.mark.parametrize("name", ["rnn-relu-tanh", "rnn-elu-softsign", "rnn-softplus", "gru-lbr0", "gru-lbr1",
                                  "lstm"])
def test_fast_mode_special_values(name, kernel):
    # fast mode keeps the NaN positions (canonical) and the signs of the
    # infinities, and stays within its bound elsewhere
    c = edge_case(name, None)
    _fast_agrees(gpu_case(c, "fast", launch=KERNELS[kernel]), oracle_case(c))


# ------------------------------------------------------------- the single cell

def _cell(hidden, inp, X, Hp, W, R, B, act, clip, mode="exact"):
    import torch
    plan = orc.rnn_cell_plan_create(hidden, inp, activation=act, clip=clip)
    orc.rnn_plan_set_mode(plan, mode)
    t = [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in (X, Hp, W, R, B)]
    Ho = torch.full((X.shape[0], hidden), 7.0, device="cuda")
    orc.rnn_cell_run(plan, *t, Ho)
    orc.rnn_plan_sync(plan)
    torch.cuda.synchronize()
    orc.rnn_plan_destroy(plan)
    return Ho.cpu().numpy()


@pytest.mark.parametrize("clip", [None, 3.0], ids=["noclip", "clip3"])
@pytest.mark.parametrize("act", ["Relu", "Tanh", "Sigmoid"])
def test_cell_edges_bit_identical(act, clip):
    # RNNCell-3 (page "RNNCell"): Ho = f(clip(X.W^T + H.R^T + B)); with W = R = 0
    # the activation sees B exactly; row 1 has a NaN in X, row 2 an infinity
    H, I, N = H_EDGE, 5, 4
    X = np.random.default_rng(1).uniform(-1, 1, (N, I)).astype(np.float32)
    X[1, 2] = NAN
    X[2, 0] = INF
    Hp = np.zeros((N, H), np.float32)
    Hp[0, :6] = [-0.0, 1e-45, 3e38, -3e38, -0.0, 1e-40]
    W = np.zeros((H, I), np.float32)
    R = np.zeros((H, H), np.float32)
    B = EDGES.copy()
    got = _cell(H, I, X, Hp, W, R, B, act, clip)
    ref = oracle.rnn_cell(H, I, X, Hp, W, R, B, activation=act, clip=float("inf") if clip is None else clip)
    assert_bits_equal(got, ref, f"cell {act}")
    assert np.all(got[np.isnan(got)].view(np.uint32) == 0x7FC00000)


@pytest.mark.parametrize("act", ["Relu", "Tanh", "Sigmoid"])
def test_cell_planted_rows_bit_identical(act):
    rng = np.random.default_rng(2)
    N, I, H = 7, 33, 96
    X = rng.uniform(-1, 1, (N, I)).astype(np.float32)
    Hp = rng.uniform(-0.5, 0.5, (N, H)).astype(np.float32)
    W = rng.uniform(-0.2, 0.2, (H, I)).astype(np.float32)
    R = rng.uniform(-0.2, 0.2, (H, H)).astype(np.float32)
    B = rng.uniform(-0.1, 0.1, (H,)).astype(np.float32)
    X[0, 4], X[1, 7], X[2, 0], X[3, 1] = -0.0, NAN, INF, -INF
    Hp[4, 9], Hp[5, 2] = 1e30, 1e-44
    B[3], B[4], B[5] = 3e38, -3e38, -0.0
    got = _cell(H, I, X, Hp, W, R, B, act, None)
    ref = oracle.rnn_cell(H, I, X, Hp, W, R, B, activation=act)
    assert_bits_equal(got, ref, f"cell {act}")
    assert np.isfinite(got[6]).all()
