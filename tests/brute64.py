"""Straight-line float64 re-derivation of the operator, for tiny shapes only.

Written independently of the oracle from the page "Recurrent operators: RNN,
GRU, LSTM" (Support, Computation, Activations, Choices the specification
leaves open), in pure Python with double precision and math's own
transcendentals.  It pins the oracle's wiring (indices, gate order, bias
order, peephole placement, directions, layouts, sequence_lens) up to fp32
rounding; it does not pin rounding order.
"""
import math

import numpy as np

_K = {"RNN": 1, "GRU": 2, "LSTM": 3}
_G = {"RNN": 1, "GRU": 3, "LSTM": 4}
_DEFAULTS = {"RNN": ["tanh"], "GRU": ["sigmoid", "tanh"], "LSTM": ["sigmoid", "tanh", "tanh"]}
_ALPHA0 = {"leakyrelu": 0.01, "thresholdedrelu": 1.0, "elu": 1.0, "hardsigmoid": 0.2,
           "affine": 1.0, "scaledtanh": 1.0}
_BETA0 = {"hardsigmoid": 0.5, "affine": 0.0, "scaledtanh": 0.0}


def _act(name, a, b, x):
    if name == "relu":
        return 0.0 if x < 0 else x
    if name == "tanh":
        return math.tanh(x)
    if name == "sigmoid":
        return 1.0 / (1.0 + math.exp(-x)) if x > -700 else 0.0
    if name == "affine":
        return a * x + b
    if name == "leakyrelu":
        return a * x if x < 0 else x
    if name == "thresholdedrelu":
        return x if x > a else 0.0
    if name == "scaledtanh":
        return a * math.tanh(b * x)
    if name == "hardsigmoid":
        return min(1.0, max(0.0, a * x + b))
    if name == "elu":
        return x if x >= 0 else a * (math.exp(x) - 1.0)
    if name == "softsign":
        return x / (1.0 + abs(x))
    if name == "softplus":
        return x if x > 20 else math.log(1.0 + math.exp(x))
    raise ValueError(name)


def _resolve(op, D, activations, alpha, beta):
    k = _K[op]
    names = [s.lower() for s in activations] if activations else list(_DEFAULTS[op])
    alpha = list(alpha or [])
    beta = list(beta or [])
    triples = []
    ia = ib = 0
    for nm in names:
        a = _ALPHA0.get(nm, 0.0)
        b = _BETA0.get(nm, 0.0)
        if nm in _ALPHA0:
            if ia < len(alpha):
                a = float(alpha[ia])
            ia += 1
        if nm in _BETA0:
            if ib < len(beta):
                b = float(beta[ib])
            ib += 1
        triples.append((nm, a, b))
    sets = [triples[0:k]]
    if len(triples) == 2 * k:
        sets.append(triples[k:2 * k])
    return [sets[d] if d < len(sets) else sets[0] for d in range(D)]


def run(case):
    """Return (Y, Y_h, Y_c) in float64 for an RNNCase (tiny shapes)."""
    op, H, I = case.op, case.hidden_size, case.input_size
    S, N, L0 = case.seq, case.batch, case.layout
    D = case.dirs
    G = _G[op]
    X = case.X.astype(np.float64)
    W = case.W.astype(np.float64)
    R = case.R.astype(np.float64)
    B = None if case.B is None else case.B.astype(np.float64)
    P = None if (case.P is None or op != "LSTM") else case.P.astype(np.float64)
    clip = case.clip if (case.clip is not None and case.clip > 0) else None
    acts = _resolve(op, D, case.activations, case.alpha, case.beta)

    def xrow(t, n):
        return X[t, n] if L0 == 0 else X[n, t]

    def st(arr, d, n):
        if arr is None:
            return [0.0] * H
        a = arr.astype(np.float64)
        return list(a[d, n] if L0 == 0 else a[n, d])

    def cl(v):
        return v if clip is None else min(clip, max(-clip, v))

    Y = np.zeros(case.y_shape())
    Yh = np.zeros(case.state_shape())
    Yc = np.zeros(case.state_shape()) if op == "LSTM" else None
    for d in range(D):
        rev = case.direction == "reverse" or (case.direction == "bidirectional" and d == 1)
        f = acts[d]
        for n in range(N):
            h = st(case.initial_h, d, n)
            c = st(case.initial_c if op == "LSTM" else None, d, n)
            Ln = S if case.sequence_lens is None else int(case.sequence_lens[n])
            order = range(Ln - 1, -1, -1) if rev else range(Ln)
            for t in order:
                x = xrow(t, n)

                def lin(j, hv):
                    v = sum(x[k] * W[d, j, k] for k in range(I)) + sum(hv[k] * R[d, j, k] for k in range(H))
                    return v

                def bias(j):
                    return 0.0 if B is None else B[d, j] + B[d, G * H + j]
                hn = [0.0] * H
                cn = list(c)
                if op == "RNN":
                    for u in range(H):
                        hn[u] = _act(*f[0], cl(lin(u, h) + bias(u)))
                elif op == "GRU":
                    z = [_act(*f[0], cl(lin(u, h) + bias(u))) for u in range(H)]
                    r = [_act(*f[0], cl(lin(H + u, h) + bias(H + u))) for u in range(H)]
                    for u in range(H):
                        j = 2 * H + u
                        xw = sum(x[k] * W[d, j, k] for k in range(I))
                        wb = 0.0 if B is None else B[d, j]
                        rb = 0.0 if B is None else B[d, G * H + j]
                        if case.linear_before_reset:
                            rec = sum(h[k] * R[d, j, k] for k in range(H))
                            pre = xw + r[u] * (rec + rb) + wb
                        else:
                            pre = xw + sum(r[k] * h[k] * R[d, j, k] for k in range(H)) + wb + rb
                        ht = _act(*f[1], cl(pre))
                        hn[u] = (1 - z[u]) * ht + z[u] * h[u]
                else:
                    for u in range(H):
                        pi = lin(u, h) + bias(u)
                        po = lin(H + u, h) + bias(H + u)
                        pf = lin(2 * H + u, h) + bias(2 * H + u)
                        pc = lin(3 * H + u, h) + bias(3 * H + u)
                        if P is not None:
                            pi += P[d, u] * c[u]
                            pf += P[d, 2 * H + u] * c[u]
                        i = _act(*f[0], cl(pi))
                        fg = 1 - i if case.input_forget else _act(*f[0], cl(pf))
                        ct = _act(*f[1], cl(pc))
                        cn[u] = fg * c[u] + i * ct
                        if P is not None:
                            po += P[d, H + u] * cn[u]
                        o = _act(*f[0], cl(po))
                        hn[u] = o * _act(*f[2], cn[u])
                h, c = hn, cn
                if L0 == 0:
                    Y[t, d, n] = h
                else:
                    Y[n, t, d] = h
            idx = (d, n) if L0 == 0 else (n, d)
            Yh[idx] = h if Ln > 0 else 0.0
            if Yc is not None:
                Yc[idx] = c if Ln > 0 else 0.0
    return Y, Yh, Yc
