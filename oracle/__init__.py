"""CPU oracle for the ONNX RNN / GRU / LSTM sequence operators.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The
product library never imports or links it and shares no code with it.

The arithmetic lives in ``rnn_oracle.c`` (plain single-threaded C, fp32, every
operation separately rounded, compiled with ``-ffp-contract=off``); this module
only compiles it with gcc and marshals numpy arrays through ctypes.  ctypes
releases the GIL during a call, so independent batch rows can be computed on
several threads (``rnn(..., rows=(b, e))``).
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rnn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lib = None
_lock = threading.Lock()

OPS = {"RNN": 0, "GRU": 1, "LSTM": 2}
DIRECTIONS = {"forward": 0, "reverse": 1, "bidirectional": 2}
ACT_NAMES = ["relu", "tanh", "sigmoid", "affine", "leakyrelu", "thresholdedrelu",
             "scaledtanh", "hardsigmoid", "elu", "softsign", "softplus"]


class OracleError(RuntimeError):
    def __init__(self, status: int):
        super().__init__({1: "invalid argument", 2: "invalid input"}.get(status, f"status {status}"))
        self.status = status


def build(force: bool = False) -> str:
    """Compile rnn_oracle.c into oracle/_build/liboracle.so (gcc, no FMA)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _configure(lib):
    fp = ctypes.POINTER(ctypes.c_float)
    ip = ctypes.POINTER(ctypes.c_int32)
    L = ctypes.c_long
    lib.oracle_rnn_rows.restype = ctypes.c_int
    lib.oracle_rnn_rows.argtypes = [
        ctypes.c_int, ctypes.c_int, L, L,
        ctypes.POINTER(ctypes.c_char_p), ctypes.c_int,
        fp, ctypes.c_int, fp, ctypes.c_int,
        ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        L, L, fp, fp, fp, fp, ip, fp, fp, fp, fp, fp, fp, L, L]
    lib.oracle_resolve_activations.restype = ctypes.c_int
    lib.oracle_resolve_activations.argtypes = [
        ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_char_p), ctypes.c_int,
        fp, ctypes.c_int, fp, ctypes.c_int,
        ctypes.POINTER(ctypes.c_int), fp, fp]
    for name in ("oracle_exp_n", "oracle_log_n", "oracle_tanh_n", "oracle_sigmoid_n"):
        getattr(lib, name).argtypes = [fp, fp, L]
        getattr(lib, name).restype = None
    lib.oracle_activation_n.argtypes = [ctypes.c_int, ctypes.c_float, ctypes.c_float, fp, fp, L]
    lib.oracle_activation_n.restype = None
    lib.oracle_rnn_cell.argtypes = [L, L, ctypes.c_char_p, ctypes.c_float, L, fp, fp, fp, fp, fp, fp]
    lib.oracle_rnn_cell.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _configure(ctypes.CDLL(build()))
    return _lib


def compile_variant(source_text: str, out_path: str) -> str:
    """Compile an edited copy of the oracle source (used by the test that
    plants mistakes in the oracle to show that its pins catch them)."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(source_text)
    subprocess.run(["gcc", *_CFLAGS, "-o", out_path, src], check=True)
    return out_path


def source() -> str:
    with open(_SRC) as f:
        return f.read()


@contextlib.contextmanager
def use_library(path: str):
    """Temporarily route every oracle call to another compiled copy."""
    global _lib
    _load()
    with _lock:
        saved = _lib
        _lib = _configure(ctypes.CDLL(path))
    try:
        yield
    finally:
        with _lock:
            _lib = saved


def _fptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def _f32(a):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=np.float32)


def _acts(activations):
    if not activations:
        return None, 0
    arr = (ctypes.c_char_p * len(activations))(*[s.encode() for s in activations])
    return arr, len(activations)


def _floats(vals):
    if vals is None or len(vals) == 0:
        return None, 0
    a = np.ascontiguousarray(vals, dtype=np.float32)
    return a, len(a)


def _code(table, v):
    return table[v] if isinstance(v, str) else int(v)


def rnn(op, direction, hidden_size, input_size, X, W, R, B=None, sequence_lens=None,
        initial_h=None, initial_c=None, P=None, activations=None, alpha=None, beta=None,
        clip=None, layout=0, linear_before_reset=0, input_forget=0, rows=None,
        want_y=True):
    """Run the oracle.  Returns (Y, Y_h, Y_c); Y_c is None unless op is LSTM.

    ``rows=(b, e)`` computes only batch rows b..e-1 (the other rows of the
    outputs stay zero); the result for those rows is the same as a full run.
    """
    lib = _load()
    opc = _code(OPS, op)
    dirc = _code(DIRECTIONS, direction)
    D = 2 if dirc == 2 else 1
    H = int(hidden_size)
    I = int(input_size)
    X = _f32(X)
    if layout == 0:
        S, N = X.shape[0], X.shape[1]
    else:
        N, S = X.shape[0], X.shape[1]
    W, R, B, h0, c0, P = map(_f32, (W, R, B, initial_h, initial_c, P))
    lens = None if sequence_lens is None else np.ascontiguousarray(sequence_lens, dtype=np.int32)
    yshape = (S, D, N, H) if layout == 0 else (N, S, D, H)
    sshape = (D, N, H) if layout == 0 else (N, D, H)
    Y = np.zeros(yshape, np.float32) if want_y else None
    Yh = np.zeros(sshape, np.float32)
    Yc = np.zeros(sshape, np.float32) if opc == 2 else None
    acts, nacts = _acts(activations)
    al, nal = _floats(alpha)
    be, nbe = _floats(beta)
    c = float("nan") if clip is None else float(clip)
    b, e = (0, N) if rows is None else rows
    st = lib.oracle_rnn_rows(
        opc, dirc, H, I, acts, nacts, _fptr(al), nal, _fptr(be), nbe, c, int(layout),
        int(linear_before_reset), int(input_forget), S, N,
        _fptr(X), _fptr(W), _fptr(R), _fptr(B),
        None if lens is None else lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
        _fptr(h0), _fptr(c0), _fptr(P), _fptr(Y), _fptr(Yh), _fptr(Yc), b, e)
    if st != 0:
        raise OracleError(st)
    return Y, Yh, Yc


def rnn_threaded(*args, threads=None, rows=None, **kw):
    """rnn() over the batch rows split across threads (ctypes drops the GIL).

    ``rows`` (optional) is an iterable of batch-row indices to compute; rows
    not listed stay zero in the outputs."""
    X = kw.get("X") if "X" in kw else args[4]
    layout = kw.get("layout", 0)
    N = X.shape[1] if layout == 0 else X.shape[0]
    todo = list(range(N)) if rows is None else sorted(set(int(r) for r in rows))
    if not todo:
        return rnn(*args, rows=(0, 0), **kw)
    threads = threads or min(len(todo), os.cpu_count() or 1)
    parts = [todo[i::threads] for i in range(threads)]
    results = [None] * len(todo)
    errors = []

    def work(ix):
        try:
            for r in parts[ix]:
                results[todo.index(r)] = (r, rnn(*args, rows=(r, r + 1), **kw))
        except Exception as exc:  # pragma: no cover - reported below
            errors.append(exc)

    ths = [threading.Thread(target=work, args=(i,)) for i in range(threads)]
    for t in ths:
        t.start()
    for t in ths:
        t.join()
    if errors:
        raise errors[0]
    Y, Yh, Yc = results[0][1]
    Y, Yh = (None if Y is None else Y.copy()), Yh.copy()
    Yc = None if Yc is None else Yc.copy()
    for r, (y, yh, yc) in results[1:]:
        sl = (slice(None), slice(None), r) if layout == 0 else (r,)
        sls = (slice(None), r) if layout == 0 else (r,)
        if Y is not None:
            Y[sl] = y[sl]
        Yh[sls] = yh[sls]
        if Yc is not None:
            Yc[sls] = yc[sls]
    return Y, Yh, Yc


def resolve_activations(op, direction, activations=None, alpha=None, beta=None):
    """[(name, alpha, beta) per slot] per direction, as the oracle resolves them."""
    lib = _load()
    opc = _code(OPS, op)
    dirc = _code(DIRECTIONS, direction)
    acts, nacts = _acts(activations)
    al, nal = _floats(alpha)
    be, nbe = _floats(beta)
    fn = (ctypes.c_int * 6)()
    ao = np.zeros(6, np.float32)
    bo = np.zeros(6, np.float32)
    st = lib.oracle_resolve_activations(opc, dirc, acts, nacts, _fptr(al), nal, _fptr(be), nbe,
                                        fn, _fptr(ao), _fptr(bo))
    if st != 0:
        raise OracleError(st)
    D = 2 if dirc == 2 else 1
    k = {0: 1, 1: 2, 2: 3}[opc]
    return [[(ACT_NAMES[fn[d * 3 + s]], float(ao[d * 3 + s]), float(bo[d * 3 + s]))
             for s in range(k)] for d in range(D)]


def _unary(name, x):
    lib = _load()
    x = _f32(np.asarray(x))
    y = np.empty_like(x)
    getattr(lib, name)(_fptr(x), _fptr(y), x.size)
    return y


def exp(x):
    return _unary("oracle_exp_n", x)


def log(x):
    return _unary("oracle_log_n", x)


def tanh(x):
    return _unary("oracle_tanh_n", x)


def sigmoid(x):
    return _unary("oracle_sigmoid_n", x)


def activation(name, x, alpha=0.0, beta=0.0):
    lib = _load()
    x = _f32(np.asarray(x))
    y = np.empty_like(x)
    lib.oracle_activation_n(ACT_NAMES.index(name.lower()), float(alpha), float(beta),
                            _fptr(x), _fptr(y), x.size)
    return y


def rnn_cell(hidden_size, input_size, X, H, W, R, B, activation="Tanh", clip=float("inf")):
    """One RNN cell (page "RNNCell", RNNCell-3): Ho = f(clip(X.W^T + H.R^T + B)),
    B the summed bias, in the sequence operator's rounding order.
    X [batch, I], H [batch, hidden], W [hidden, I], R [hidden, hidden], B [hidden]."""
    lib = _load()
    X, H, W, R, B = map(_f32, (X, H, W, R, B))
    N = X.shape[0]
    Ho = np.zeros((N, int(hidden_size)), np.float32)
    st = lib.oracle_rnn_cell(int(hidden_size), int(input_size),
                             None if activation is None else activation.encode(), float(clip), N,
                             _fptr(X), _fptr(H), _fptr(W), _fptr(R), _fptr(B), _fptr(Ho))
    if st != 0:
        raise OracleError(st)
    return Ho


# ------------------------------------------------------------ fp16 / bf16 I/O
#
# The operator with 2-byte activation tensors (the fp16/bf16 variants of the
# type T on the Apple BNNS page): the fp32 operator applied to the inputs
# widened exactly, each output rounded to nearest even once, a NaN output
# written as the type's canonical quiet NaN.  bf16 arrays are carried as
# their uint16 bit patterns (numpy has no bf16 type).

def widen(a, io):
    """fp16 (numpy float16) or bf16 (uint16 bits) to float32, exactly."""
    if a is None or io == "f32":
        return a
    if io == "f16":
        return np.asarray(a, np.float16).astype(np.float32)
    bits = np.asarray(a, np.uint16).astype(np.uint32) << 16
    return bits.view(np.float32)


def narrow(a, io):
    """float32 to fp16 (numpy float16) or bf16 (uint16 bits), round to nearest even."""
    if a is None or io == "f32":
        return a
    a = np.ascontiguousarray(a, np.float32)
    nan = np.isnan(a)
    if io == "f16":
        with np.errstate(over="ignore"):
            out = a.astype(np.float16)
        out.view(np.uint16)[nan] = 0x7E00
        return out
    u = a.view(np.uint32).astype(np.uint64)
    # add half an ulp of the kept part, plus one if the kept part is odd (ties to even)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    r[nan] = 0x7FC0
    return r


def rnn_io(io, op, direction, hidden_size, input_size, X, W, R, B=None, sequence_lens=None,
           initial_h=None, initial_c=None, P=None, **kw):
    """rnn() with X, initial_h, initial_c given in `io` ("f16": float16, "bf16":
    uint16 bits) and Y, Y_h, Y_c returned in it; W, R, B, P stay float32."""
    Y, Yh, Yc = rnn(op, direction, hidden_size, input_size, widen(X, io), W, R, B=B,
                    sequence_lens=sequence_lens, initial_h=widen(initial_h, io),
                    initial_c=widen(initial_c, io), P=P, **kw)
    return narrow(Y, io), narrow(Yh, io), narrow(Yc, io)


# ------------------------------------------------------------ stacked layers
#
# Layers chained by their output sequence: layer l+1 reads layer l's Y with
# the directions side by side per step (input_size of layer l+1 = dirs_l *
# hidden_l), forward units first:  layout 0  X'[t, n, d*H + u] = Y[t, d, n, u];
# layout 1  X'[n, t, d*H + u] = Y[n, t, d, u].  sequence_lens is shared.

def stack_input(Y, layout):
    """The next layer's X from a layer's Y (the rule above)."""
    Y = np.asarray(Y, np.float32)
    if layout == 0:
        S, D, N, H = Y.shape
        X = np.empty((S, N, D * H), np.float32)
        for t in range(S):
            for n in range(N):
                for d in range(D):
                    X[t, n, d * H:(d + 1) * H] = Y[t, d, n, :]
        return X
    N, S, D, H = Y.shape
    X = np.empty((N, S, D * H), np.float32)
    for n in range(N):
        for t in range(S):
            for d in range(D):
                X[n, t, d * H:(d + 1) * H] = Y[n, t, d, :]
    return X


def rnn_stack(layers, X, sequence_lens=None):
    """Run layers (dicts of rnn() keyword arguments without X and
    sequence_lens) one after another; returns (Y of the last layer, [Y_h per
    layer], [Y_c per layer])."""
    x = X
    yh, yc = [], []
    Y = None
    for L in layers:
        L = dict(L)
        args = [L.pop(k) for k in ("op", "direction", "hidden_size", "input_size")]
        W, R = L.pop("W"), L.pop("R")
        Y, h, c = rnn(*args, x, W, R, sequence_lens=sequence_lens, **L)
        yh.append(h)
        yc.append(c)
        x = stack_input(Y, L.get("layout", 0))
    return Y, yh, yc
