"""Seeded synthetic inputs for the RNN / GRU / LSTM sequence operator.

This module only draws random tensors in the shapes and distributions of the
workloads; it holds none of the operator's arithmetic.  Both the CUDA path and
the CPU oracle are fed from it.

Draw order for every case: X, W, R, B, P, initial_h, initial_c, sequence_lens
(absent tensors draw nothing).  U(a, b) is ``a + (b - a) * uniform``, N(0, 1)
the standard normal, U{a..b} uniform integers; all float tensors are float32,
lengths int32.  The generator is numpy's PCG64 (``default_rng(seed)``), so the
same seed gives the same tensors on every machine.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional, Sequence

import numpy as np

GATES = {"RNN": 1, "GRU": 3, "LSTM": 4}


@dataclass
class RNNCase:
    """One invocation of the operator: attributes plus host input tensors."""
    op: str
    direction: str
    seq: int
    batch: int
    input_size: int
    hidden_size: int
    layout: int = 0
    activations: Optional[Sequence[str]] = None
    alpha: Optional[Sequence[float]] = None
    beta: Optional[Sequence[float]] = None
    clip: Optional[float] = None
    linear_before_reset: int = 0
    input_forget: int = 0
    X: np.ndarray = None
    W: np.ndarray = None
    R: np.ndarray = None
    B: Optional[np.ndarray] = None
    P: Optional[np.ndarray] = None
    initial_h: Optional[np.ndarray] = None
    initial_c: Optional[np.ndarray] = None
    sequence_lens: Optional[np.ndarray] = None
    name: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def dirs(self) -> int:
        return 2 if self.direction == "bidirectional" else 1

    @property
    def gates(self) -> int:
        return GATES[self.op]

    def cell_steps(self) -> int:
        """seq * batch * dirs: the unit of the throughput metric."""
        return self.seq * self.batch * self.dirs

    def valid_cell_steps(self) -> int:
        if self.sequence_lens is None:
            return self.cell_steps()
        return int(np.asarray(self.sequence_lens, np.int64).sum()) * self.dirs

    def attrs(self) -> dict:
        return dict(op=self.op, direction=self.direction, hidden_size=self.hidden_size,
                    input_size=self.input_size, activations=self.activations,
                    alpha=self.alpha, beta=self.beta, clip=self.clip, layout=self.layout,
                    linear_before_reset=self.linear_before_reset,
                    input_forget=self.input_forget)

    def tensors(self) -> dict:
        return dict(X=self.X, W=self.W, R=self.R, B=self.B, sequence_lens=self.sequence_lens,
                    initial_h=self.initial_h, initial_c=self.initial_c, P=self.P)

    def with_(self, **kw) -> "RNNCase":
        return replace(self, **kw)

    def x_shape(self):
        return (self.seq, self.batch, self.input_size) if self.layout == 0 else \
            (self.batch, self.seq, self.input_size)

    def state_shape(self):
        return (self.dirs, self.batch, self.hidden_size) if self.layout == 0 else \
            (self.batch, self.dirs, self.hidden_size)

    def y_shape(self):
        return (self.seq, self.dirs, self.batch, self.hidden_size) if self.layout == 0 else \
            (self.batch, self.seq, self.dirs, self.hidden_size)


class _Draw:
    def __init__(self, seed: int):
        self.rng = np.random.default_rng(seed)

    def uniform(self, shape, lo, hi):
        u = self.rng.random(shape, dtype=np.float32)
        return (np.float32(lo) + np.float32(hi - lo) * u).astype(np.float32)

    def normal(self, shape):
        return self.rng.standard_normal(shape, dtype=np.float32)

    def ints(self, shape, lo, hi):
        return self.rng.integers(lo, hi + 1, size=shape).astype(np.int32)


def make_case(op, direction, seq, batch, input_size, hidden_size, *, seed=0, layout=0,
              x_dist=("normal",), w_scale=None, b_scale=0.1, with_B=True, with_P=False,
              p_scale=0.1, h0_scale=None, c0_scale=None, lens=None, name="", **attrs):
    """Draw one case.  ``x_dist`` is ("normal",) or ("uniform", lo, hi);
    ``w_scale`` s gives W, R ~ U(-s, s) (default 1/sqrt(hidden)); ``lens`` is
    None, ("uniform", lo, hi) or an explicit list."""
    g = GATES[op]
    D = 2 if direction == "bidirectional" else 1
    H, I, S, N = hidden_size, input_size, seq, batch
    d = _Draw(seed)
    xs = (S, N, I) if layout == 0 else (N, S, I)
    X = d.normal(xs) if x_dist[0] == "normal" else d.uniform(xs, x_dist[1], x_dist[2])
    s = (1.0 / np.sqrt(H)) if w_scale is None else w_scale
    W = d.uniform((D, g * H, I), -s, s)
    R = d.uniform((D, g * H, H), -s, s)
    B = d.uniform((D, 2 * g * H), -b_scale, b_scale) if with_B else None
    P = d.uniform((D, 3 * H), -p_scale, p_scale) if (with_P and op == "LSTM") else None
    ss = (D, N, H) if layout == 0 else (N, D, H)
    h0 = d.uniform(ss, -h0_scale, h0_scale) if h0_scale is not None else None
    c0 = d.uniform(ss, -c0_scale, c0_scale) if (c0_scale is not None and op == "LSTM") else None
    L = None
    if lens is not None:
        if isinstance(lens, tuple) and lens[0] == "uniform":
            L = d.ints((N,), lens[1], lens[2])
        else:
            L = np.asarray(lens, np.int32)
    return RNNCase(op=op, direction=direction, seq=S, batch=N, input_size=I, hidden_size=H,
                   layout=layout, X=X, W=W, R=R, B=B, P=P, initial_h=h0, initial_c=c0,
                   sequence_lens=L, name=name, **attrs)


# --------------------------------------------------------------------------
# The five workloads the operator is measured and checked on.
# --------------------------------------------------------------------------

WORKLOADS = {
    "rnn_fwd_s8_b1_i16_h128":
        "RNN forward, seq 8, batch 1, input 16, hidden 128, Tanh, layout 0",
    "lstm_fwd_s64_b32_i256_h512":
        "LSTM forward, seq 64, batch 32, input 256, hidden 512, peepholes, layout 0",
    "gru_bidi_s128_b64_i512_h1024":
        "GRU bidirectional, seq 128, batch 64, input 512, hidden 1024, layout 1, sequence_lens",
    "lstm_bidi_s512_b128_i1024_h1024":
        "LSTM bidirectional, seq 512, batch 128, input 1024, hidden 1024, clip 3, "
        "HardSigmoid/LeakyRelu/ScaledTanh forward, sequence_lens",
    "gru_rev_s4096_b4_i256_h2048":
        "GRU reverse, seq 4096, batch 4, input 256, hidden 2048, linear_before_reset 1",
}

# Shorter sequences of the same per-step shapes, for profiler captures (a few
# hundred MB on the device instead of gigabytes; every step is the same work).
PROFILE_WORKLOADS = {
    "lstm_bidi_s64_b128_i1024_h1024":
        "the LSTM bidirectional workload (batch 128, input 1024, hidden 1024, clip 3, same activations) "
        "cut to 64 steps, sequence_lens U{1..64}",
    "gru_rev_s256_b4_i256_h2048":
        "the GRU reverse workload (batch 4, input 256, hidden 2048, linear_before_reset 1) cut to 256 steps",
}


def workload(name: str, *, lbr: int = 0, initial_h_zero: bool = False) -> RNNCase:
    """Seeded inputs (seed 0) of a named workload."""
    if name == "rnn_fwd_s8_b1_i16_h128":
        c = make_case("RNN", "forward", 8, 1, 16, 128, x_dist=("uniform", -1.0, 1.0),
                      activations=["Tanh"], name=name)
        if initial_h_zero:
            c.initial_h = np.zeros(c.state_shape(), np.float32)
        return c
    if name == "lstm_fwd_s64_b32_i256_h512":
        return make_case("LSTM", "forward", 64, 32, 256, 512, with_P=True,
                         h0_scale=0.5, c0_scale=0.5, input_forget=0, name=name)
    if name == "gru_bidi_s128_b64_i512_h1024":
        c = make_case("GRU", "bidirectional", 128, 64, 512, 1024, layout=1,
                      w_scale=1.0 / 32, lens=("uniform", 0, 128), linear_before_reset=lbr,
                      name=name)
        c.sequence_lens[0] = 0
        c.sequence_lens[1] = 128
        return c
    if name == "lstm_bidi_s512_b128_i1024_h1024":
        return make_case("LSTM", "bidirectional", 512, 128, 1024, 1024, w_scale=1.0 / 32,
                         with_B=False, with_P=True, lens=("uniform", 1, 512), clip=3.0,
                         activations=["HardSigmoid", "LeakyRelu", "ScaledTanh",
                                      "Sigmoid", "Tanh", "Tanh"],
                         alpha=[0.25, 0.05, 1.5], beta=[0.45, 0.8], name=name)
    if name == "gru_rev_s4096_b4_i256_h2048":
        return make_case("GRU", "reverse", 4096, 4, 256, 2048, linear_before_reset=1,
                         h0_scale=0.5, name=name)
    if name == "lstm_bidi_s64_b128_i1024_h1024":
        return make_case("LSTM", "bidirectional", 64, 128, 1024, 1024, w_scale=1.0 / 32,
                         with_B=False, with_P=True, lens=("uniform", 1, 64), clip=3.0,
                         activations=["HardSigmoid", "LeakyRelu", "ScaledTanh",
                                      "Sigmoid", "Tanh", "Tanh"],
                         alpha=[0.25, 0.05, 1.5], beta=[0.45, 0.8], name=name)
    if name == "gru_rev_s256_b4_i256_h2048":
        return make_case("GRU", "reverse", 256, 4, 256, 2048, linear_before_reset=1,
                         h0_scale=0.5, name=name)
    raise KeyError(name)


@dataclass
class CellCase:
    """One call of the single RNN cell (RNNCell-3): attributes plus host inputs
    X [batch, input], H [batch, hidden], W [hidden, input], R [hidden, hidden],
    B [hidden] (the summed bias)."""
    batch: int
    input_size: int
    hidden_size: int
    activation: str = "Tanh"
    clip: Optional[float] = None
    X: np.ndarray = None
    H: np.ndarray = None
    W: np.ndarray = None
    R: np.ndarray = None
    B: np.ndarray = None
    name: str = ""

    def tensors(self) -> dict:
        return dict(X=self.X, H=self.H, W=self.W, R=self.R, B=self.B)


def make_cell_case(batch, input_size, hidden_size, *, seed=0, activation="Tanh", clip=None,
                   w_scale=None, name="") -> CellCase:
    """Draw order X, H, W, R, B: X ~ U(-1, 1), H ~ U(-0.5, 0.5), W and R ~ U(-s, s)
    (default s = 1/sqrt(hidden)), B ~ U(-0.1, 0.1)."""
    d = _Draw(seed)
    N, I, Hs = batch, input_size, hidden_size
    s = (1.0 / np.sqrt(Hs)) if w_scale is None else w_scale
    X = d.uniform((N, I), -1.0, 1.0)
    H = d.uniform((N, Hs), -0.5, 0.5)
    W = d.uniform((Hs, I), -s, s)
    R = d.uniform((Hs, Hs), -s, s)
    B = d.uniform((Hs,), -0.1, 0.1)
    return CellCase(N, I, Hs, activation, clip, X, H, W, R, B, name)


CELL_WORKLOADS = {
    "rnncell_b1_i16_h128": "RNNCell-3 single step, batch 1, input 16, hidden 128, Tanh (the page's example shapes)",
    "rnncell_b256_i1024_h1024": "RNNCell-3 single step, batch 256, input 1024, hidden 1024, Tanh",
}


def cell_workload(name: str) -> CellCase:
    """Seeded inputs (seed 0) of a named single-cell workload."""
    if name == "rnncell_b1_i16_h128":
        return make_cell_case(1, 16, 128, name=name)
    if name == "rnncell_b256_i1024_h1024":
        return make_cell_case(256, 1024, 1024, name=name)
    raise KeyError(name)


STACK_WORKLOADS = {
    "lstm2_fwd_s64_b32_i256_h512": "two stacked LSTM forward layers, seq 64, batch 32, input 256, hidden 512, "
                                   "peepholes (the LSTM forward workload with a second layer on top)",
    "gru2_bidi_s128_b64_i512_h1024": "two stacked GRU bidirectional layers, seq 128, batch 64, input 512, hidden "
                                     "1024, lbr 1, layout 0, sequence_lens",
    "lstm4_fwd_s256_b8_i128_h128": "four stacked LSTM forward layers, seq 256, batch 8, input 128, hidden 128, "
                                   "peepholes (small latency-bound layers)",
    "gru3_fwd_s256_b16_i256_h256": "three stacked GRU forward layers, seq 256, batch 16, input 256, hidden 256, "
                                   "lbr 1, sequence_lens",
}


def stack_workload(name: str):
    """Seeded per-layer cases (seed 0, then 1) of a named stack workload."""
    if name == "lstm2_fwd_s64_b32_i256_h512":
        a = make_case("LSTM", "forward", 64, 32, 256, 512, with_P=True, h0_scale=0.5, c0_scale=0.5, name=name)
        b = make_case("LSTM", "forward", 64, 32, 512, 512, seed=1, with_P=True, h0_scale=0.5, c0_scale=0.5)
        return [a, b]
    if name == "gru2_bidi_s128_b64_i512_h1024":
        a = make_case("GRU", "bidirectional", 128, 64, 512, 1024, w_scale=1.0 / 32, lens=("uniform", 0, 128),
                      linear_before_reset=1, name=name)
        b = make_case("GRU", "bidirectional", 128, 64, 2048, 1024, seed=1, w_scale=1.0 / 32,
                      linear_before_reset=1)
        return [a, b]
    if name == "lstm4_fwd_s256_b8_i128_h128":
        return [make_case("LSTM", "forward", 256, 8, 128, 128, seed=i, with_P=True, h0_scale=0.5, c0_scale=0.5,
                          name=name if i == 0 else "") for i in range(4)]
    if name == "gru3_fwd_s256_b16_i256_h256":
        a = make_case("GRU", "forward", 256, 16, 256, 256, lens=("uniform", 64, 256), linear_before_reset=1,
                      name=name)
        return [a] + [make_case("GRU", "forward", 256, 16, 256, 256, seed=i, linear_before_reset=1)
                      for i in (1, 2)]
    raise KeyError(name)


ACTIVATIONS = ["Relu", "Tanh", "Sigmoid", "Affine", "LeakyRelu", "ThresholdedRelu",
               "ScaledTanh", "HardSigmoid", "Elu", "Softsign", "Softplus"]


def random_case(seed: int, *, op=None, direction=None, layout=None, max_seq=7, max_batch=9,
                max_input=37, max_hidden=41, **over) -> RNNCase:
    """A small random case covering the attribute space (for parity sweeps)."""
    rng = np.random.default_rng(10_000 + seed)
    op = op or ["RNN", "GRU", "LSTM"][rng.integers(3)]
    direction = direction or ["forward", "reverse", "bidirectional"][rng.integers(3)]
    layout = int(rng.integers(2)) if layout is None else layout
    S = int(rng.integers(1, max_seq + 1))
    N = int(rng.integers(1, max_batch + 1))
    I = int(rng.integers(0, max_input + 1))
    H = int(rng.integers(1, max_hidden + 1))
    k = {"RNN": 1, "GRU": 2, "LSTM": 3}[op]
    D = 2 if direction == "bidirectional" else 1
    acts = None
    alpha = beta = None
    if rng.random() < 0.6:
        nsets = D if rng.random() < 0.7 else 1
        pool = ["Sigmoid", "Tanh", "HardSigmoid", "Softsign", "Relu", "Affine", "LeakyRelu",
                "ScaledTanh", "Elu", "Softplus", "ThresholdedRelu"]
        acts = [pool[rng.integers(len(pool))] for _ in range(k * nsets)]
        acts = [a.upper() if rng.random() < 0.2 else a for a in acts]
        if rng.random() < 0.7:
            alpha = [float(np.float32(v)) for v in rng.uniform(0.05, 1.5, int(rng.integers(0, 4)))]
            beta = [float(np.float32(v)) for v in rng.uniform(-0.5, 0.9, int(rng.integers(0, 3)))]
    clip = None
    r = rng.random()
    if r < 0.3:
        clip = float(np.float32(rng.uniform(0.5, 3.0)))
    elif r < 0.35:
        clip = 0.0
    lens = None
    if rng.random() < 0.5:
        lens = ("uniform", 0, S)
    attrs = dict(activations=acts, alpha=alpha, beta=beta, clip=clip,
                 linear_before_reset=int(rng.integers(2)) if op == "GRU" else 0,
                 input_forget=int(rng.random() < 0.3) if op == "LSTM" else 0)
    attrs.update({k2: v for k2, v in over.items() if k2 in attrs})
    gen = dict(seed=seed, layout=layout, with_B=bool(rng.random() < 0.8),
               with_P=bool(rng.random() < 0.6), h0_scale=0.5 if rng.random() < 0.6 else None,
               c0_scale=0.5 if rng.random() < 0.6 else None, lens=lens,
               w_scale=float(rng.uniform(0.2, 0.8)))
    gen.update({k2: v for k2, v in over.items() if k2 in gen})
    for k2 in ("seq", "batch", "input_size", "hidden_size"):
        if k2 in over:
            S, N, I, H = (over.get("seq", S), over.get("batch", N),
                          over.get("input_size", I), over.get("hidden_size", H))
    return make_case(op, direction, S, N, I, H, name=f"random{seed}", **gen, **attrs)
