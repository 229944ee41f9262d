"""Thin ctypes binding of the C ABI in include/onnx_recurrent.h.

Argument marshalling only: every step of a run executes in the CUDA library.
PyTorch supplies device memory and streams.  The library must have been built
(``onnx_recurrent_gb300.build()``); there is no fallback when it is missing.
"""
from __future__ import annotations

import ctypes
import os
import re

from . import _build

OPS = {"RNN": 0, "GRU": 1, "LSTM": 2}
DIRECTIONS = {"forward": 0, "reverse": 1, "bidirectional": 2}
MODES = {"exact": 0, "fast": 1, "tf32": 2, "bf16": 3}
IO_TYPES = {"f32": 0, "f16": 1, "bf16": 2}
ACT_NAMES = ["relu", "tanh", "sigmoid", "affine", "leakyrelu", "thresholdedrelu",
             "scaledtanh", "hardsigmoid", "elu", "softsign", "softplus"]
STATUS = {0: "RNN_OK", 1: "RNN_ERR_INVALID_ARGUMENT", 2: "RNN_ERR_INVALID_INPUT",
          3: "RNN_ERR_UNSUPPORTED", 4: "RNN_ERR_CUDA", 5: "RNN_ERR_OOM", 6: "RNN_ERR_TIMEOUT"}
HEADER = os.path.join(_build.ROOT, "include", "onnx_recurrent.h")

_lib = None


class RNNError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status
        self.message = message


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load the built library (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB
    if not os.path.exists(p):
        raise RuntimeError(f"CUDA library not built ({p}); call onnx_recurrent_gb300.build()")
    lib = ctypes.CDLL(p)
    vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    fp = ctypes.POINTER(ctypes.c_float)
    ip = ctypes.POINTER(ctypes.c_int)
    lib.rnn_plan_create.argtypes = [ctypes.POINTER(vp), i32, i32, i64, i64,
                                    ctypes.POINTER(ctypes.c_char_p), i32, fp, i32, fp, i32,
                                    f32, i32, i32, i32]
    lib.rnn_run.argtypes = [vp, i64, i64] + [vp] * 11 + [vp]
    lib.rnn_run_static_scratch.argtypes = [vp, i64, i64] + [vp] * 11 + [vp]
    lib.rnn_plan_destroy.argtypes = [vp]
    lib.rnn_plan_destroy.restype = None
    lib.rnn_plan_set_mode.argtypes = [vp, i32]
    lib.rnn_plan_set_weights.argtypes = [vp, vp, vp, vp]
    lib.rnn_plan_sync.argtypes = [vp]
    lib.rnn_plan_get_activation.argtypes = [vp, i32, i32, ip, fp, fp]
    lib.rnn_plan_set_launch.argtypes = [vp, i32, i32, i32, i32, i32]
    lib.rnn_plan_get_launch.argtypes = [vp, ip, ip, ip, ip, ip, ip, ip]
    lib.rnn_plan_set_timing.argtypes = [vp, i32]
    lib.rnn_plan_last_timing.argtypes = [vp, fp, i32]
    lib.rnn_plan_timing_totals.argtypes = [vp, fp, i32, ip]
    lib.rnn_plan_debug_barrier.argtypes = [vp, i64, i32]
    lib.rnn_plan_last_launch_count.argtypes = [vp]
    lib.rnn_plan_last_launch_count.restype = i32
    lib.rnn_plan_set_io_type.argtypes = [vp, i32]
    lib.rnn_stack_create.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(vp), i32]
    lib.rnn_stack_run.argtypes = [vp, i64, i64, vp, ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(vp), vp,
                                  ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(vp), vp,
                                  ctypes.POINTER(vp), ctypes.POINTER(vp), vp]
    lib.rnn_stack_destroy.argtypes = [vp]
    lib.rnn_stack_destroy.restype = None
    lib.rnn_stack_last_launch_count.argtypes = [vp]
    lib.rnn_stack_last_launch_count.restype = i32
    lib.rnn_stack_set_wavefront.argtypes = [vp, i32]
    lib.rnn_stack_last_wavefront.argtypes = [vp]
    lib.rnn_stack_last_wavefront.restype = i32
    lib.rnn_cell_plan_create.argtypes = [ctypes.POINTER(vp), i64, i64, ctypes.c_char_p, f32]
    lib.rnn_cell_run.argtypes = [vp, i64] + [vp] * 6 + [vp]
    lib.rnn_last_error.argtypes = []
    lib.rnn_last_error.restype = ctypes.c_char_p
    for name in ("rnn_plan_create", "rnn_run", "rnn_run_static_scratch", "rnn_plan_set_mode", "rnn_plan_set_weights",
                 "rnn_plan_sync", "rnn_plan_get_activation", "rnn_plan_set_launch",
                 "rnn_plan_get_launch", "rnn_plan_set_timing", "rnn_plan_last_timing",
                 "rnn_plan_timing_totals",
                 "rnn_plan_debug_barrier", "rnn_cell_plan_create", "rnn_cell_run", "rnn_plan_set_io_type",
                 "rnn_stack_create", "rnn_stack_run", "rnn_stack_set_wavefront"):
        getattr(lib, name).restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def declared_functions() -> list[str]:
    """Names of the functions include/onnx_recurrent.h declares."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rnn_\w+)\s*\(", text)))


def rnn_last_error() -> str:
    return load().rnn_last_error().decode()


def _check(st: int):
    if st != 0:
        raise RNNError(st, rnn_last_error())


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


class Plan:
    """A plan handle plus the attributes it was created with."""

    def __init__(self, handle, op, direction, hidden_size, input_size, layout):
        self.handle = handle
        self.op = op
        self.direction = direction
        self.hidden_size = hidden_size
        self.input_size = input_size
        self.layout = layout
        self.io = "f32"          # element type of X, initial states and outputs

    @property
    def dirs(self):
        return 2 if self.direction == "bidirectional" else 1

    def __del__(self):
        try:
            if self.handle:
                rnn_plan_destroy(self)
        except Exception:
            pass


def rnn_plan_create(op, direction, hidden_size, input_size, activations=None, alpha=None,
                    beta=None, clip=None, layout=0, linear_before_reset=0, input_forget=0) -> Plan:
    lib = load()
    h = ctypes.c_void_p()
    acts = None
    nacts = 0
    if activations:
        acts = (ctypes.c_char_p * len(activations))(*[a.encode() for a in activations])
        nacts = len(activations)

    def farr(v):
        if not v:
            return None, 0
        return (ctypes.c_float * len(v))(*[float(x) for x in v]), len(v)
    al, nal = farr(alpha)
    be, nbe = farr(beta)
    c = float("nan") if clip is None else float(clip)
    st = lib.rnn_plan_create(ctypes.byref(h), OPS[op] if isinstance(op, str) else int(op),
                             DIRECTIONS[direction] if isinstance(direction, str) else int(direction),
                             int(hidden_size), int(input_size), acts, nacts, al, nal, be, nbe, c,
                             int(layout), int(linear_before_reset), int(input_forget))
    _check(st)
    return Plan(h, op, direction, int(hidden_size), int(input_size), int(layout))


def rnn_plan_destroy(plan: Plan):
    if plan.handle:
        load().rnn_plan_destroy(plan.handle)
        plan.handle = None


def rnn_plan_set_mode(plan: Plan, mode):
    _check(load().rnn_plan_set_mode(plan.handle, MODES[mode] if isinstance(mode, str) else int(mode)))


def rnn_plan_set_io_type(plan: Plan, io):
    """Element type of X, initial_h, initial_c, Y, Y_h, Y_c: "f32", "f16" or "bf16"."""
    _check(load().rnn_plan_set_io_type(plan.handle, IO_TYPES[io] if isinstance(io, str) else int(io)))
    plan.io = io if isinstance(io, str) else {v: k for k, v in IO_TYPES.items()}[int(io)]


def io_dtype(plan: Plan):
    import torch
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[plan.io]


def rnn_plan_set_weights(plan: Plan, W, R, stream=None):
    _check(load().rnn_plan_set_weights(plan.handle, _ptr(W), _ptr(R), _stream(stream)))


def rnn_plan_sync(plan: Plan):
    _check(load().rnn_plan_sync(plan.handle))


def rnn_plan_get_activation(plan: Plan, d: int, slot: int):
    fn = ctypes.c_int()
    a = ctypes.c_float()
    b = ctypes.c_float()
    _check(load().rnn_plan_get_activation(plan.handle, d, slot, ctypes.byref(fn), ctypes.byref(a),
                                          ctypes.byref(b)))
    return (ACT_NAMES[fn.value] if fn.value >= 0 else None), a.value, b.value


def rnn_plan_set_launch(plan: Plan, unit_groups=0, rows_per_thread=0, r_resident=-1,
                        row_groups=0, kernel=0):
    _check(load().rnn_plan_set_launch(plan.handle, int(unit_groups), int(rows_per_thread),
                                      int(r_resident), int(row_groups), int(kernel)))


def rnn_plan_get_launch(plan: Plan) -> dict:
    v = [ctypes.c_int() for _ in range(7)]
    _check(load().rnn_plan_get_launch(plan.handle, *[ctypes.byref(x) for x in v]))
    return dict(zip(["unit_groups", "rows_per_thread", "r_resident", "row_groups", "kernel",
                     "threads", "smem_bytes"], [x.value for x in v]))


def rnn_plan_set_timing(plan: Plan, enable=True):
    _check(load().rnn_plan_set_timing(plan.handle, int(bool(enable))))


def rnn_plan_last_timing(plan: Plan) -> dict:
    out = (ctypes.c_float * 5)()
    _check(load().rnn_plan_last_timing(plan.handle, out, 5))
    return dict(zip(["pack", "projection", "setup", "recurrence", "mask"], list(out)))


def rnn_plan_timing_totals(plan: Plan) -> tuple[dict, int]:
    """Per-kernel milliseconds summed over the runs since the last read."""
    out = (ctypes.c_float * 5)()
    runs = ctypes.c_int()
    _check(load().rnn_plan_timing_totals(plan.handle, out, 5, ctypes.byref(runs)))
    return dict(zip(["pack", "projection", "setup", "recurrence", "mask"], list(out))), runs.value


def rnn_plan_debug_barrier(plan: Plan, spin_limit_ns=0, skip_cta=-1):
    _check(load().rnn_plan_debug_barrier(plan.handle, int(spin_limit_ns), int(skip_cta)))


def rnn_plan_last_launch_count(plan: Plan) -> int:
    return int(load().rnn_plan_last_launch_count(plan.handle))


def _need(t, shape, name, dtype="float32"):
    import torch
    if t is None:
        return
    want = {"float32": torch.float32, "int32": torch.int32}.get(dtype, dtype)
    if t.dtype != want:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def shapes(plan: Plan, seq, batch):
    G = {"RNN": 1, "GRU": 3, "LSTM": 4}[plan.op] if isinstance(plan.op, str) else [1, 3, 4][plan.op]
    D, H, I = plan.dirs, plan.hidden_size, plan.input_size
    lay = plan.layout
    return dict(
        X=(seq, batch, I) if lay == 0 else (batch, seq, I),
        W=(D, G * H, I), R=(D, G * H, H), B=(D, 2 * G * H), P=(D, 3 * H),
        state=(D, batch, H) if lay == 0 else (batch, D, H),
        Y=(seq, D, batch, H) if lay == 0 else (batch, seq, D, H),
        lens=(batch,))


def rnn_run(plan: Plan, X, W, R, B=None, sequence_lens=None, initial_h=None, initial_c=None,
            P=None, Y=None, Y_h=None, Y_c=None, stream=None):
    """Run on CUDA tensors; outputs are written into Y, Y_h, Y_c (each optional)."""
    seq, batch = (X.shape[0], X.shape[1]) if plan.layout == 0 else (X.shape[1], X.shape[0])
    sh = shapes(plan, seq, batch)
    act = io_dtype(plan)
    _need(X, sh["X"], "X", act)
    _need(W, sh["W"], "W")
    _need(R, sh["R"], "R")
    _need(B, sh["B"], "B")
    _need(P, sh["P"], "P")
    _need(initial_h, sh["state"], "initial_h", act)
    _need(initial_c, sh["state"], "initial_c", act)
    _need(sequence_lens, sh["lens"], "sequence_lens", "int32")
    _need(Y, sh["Y"], "Y", act)
    _need(Y_h, sh["state"], "Y_h", act)
    _need(Y_c, sh["state"], "Y_c", act)
    st = load().rnn_run(plan.handle, int(seq), int(batch), _ptr(X), _ptr(W), _ptr(R), _ptr(B),
                        _ptr(sequence_lens), _ptr(initial_h), _ptr(initial_c), _ptr(P), _ptr(Y),
                        _ptr(Y_h), _ptr(Y_c), _stream(stream))
    _check(st)


def rnn_run_static_scratch(plan: Plan, X, W, R, B=None, sequence_lens=None, initial_h=None,
                           initial_c=None, P=None, Y=None, Y_h=None, Y_c=None, stream=None):
    """rnn_run that allocates no device memory (the library's fixed scratch array)."""
    seq, batch = (X.shape[0], X.shape[1]) if plan.layout == 0 else (X.shape[1], X.shape[0])
    sh = shapes(plan, seq, batch)
    act = io_dtype(plan)
    for t, k, n, dt in ((X, "X", "X", act), (W, "W", "W", "float32"), (R, "R", "R", "float32"),
                        (B, "B", "B", "float32"), (P, "P", "P", "float32"),
                        (initial_h, "state", "initial_h", act), (initial_c, "state", "initial_c", act),
                        (Y, "Y", "Y", act), (Y_h, "state", "Y_h", act), (Y_c, "state", "Y_c", act)):
        _need(t, sh[k], n, dt)
    _need(sequence_lens, sh["lens"], "sequence_lens", "int32")
    st = load().rnn_run_static_scratch(plan.handle, int(seq), int(batch), _ptr(X), _ptr(W), _ptr(R),
                                       _ptr(B), _ptr(sequence_lens), _ptr(initial_h),
                                       _ptr(initial_c), _ptr(P), _ptr(Y), _ptr(Y_h), _ptr(Y_c),
                                       _stream(stream))
    _check(st)


def rnn_cell_plan_create(hidden_size, input_size, activation="Tanh", clip=None) -> Plan:
    """Single RNN cell (RNNCell-3); clip None = +infinity (no clipping)."""
    h = ctypes.c_void_p()
    c = float("inf") if clip is None else float(clip)
    _check(load().rnn_cell_plan_create(ctypes.byref(h), int(hidden_size), int(input_size),
                                       None if activation is None else activation.encode(), c))
    plan = Plan(h, "RNN", "forward", int(hidden_size), int(input_size), 0)
    plan.cell = True
    return plan


def rnn_cell_run(plan: Plan, X, H, W, R, B, Ho, stream=None):
    """Ho = f(clip(X.W^T + H.R^T + B)) on CUDA tensors: X [batch, input],
    H and Ho [batch, hidden], W [hidden, input], R [hidden, hidden], B [hidden]."""
    batch = H.shape[0]
    hs, inp = plan.hidden_size, plan.input_size
    _need(X, (batch, inp), "X")
    _need(H, (batch, hs), "H")
    _need(W, (hs, inp), "W")
    _need(R, (hs, hs), "R")
    _need(B, (hs,), "B")
    _need(Ho, (batch, hs), "Ho")
    _check(load().rnn_cell_run(plan.handle, int(batch), _ptr(X), _ptr(H), _ptr(W), _ptr(R), _ptr(B),
                               _ptr(Ho), _stream(stream)))


class Stack:
    """A stack handle plus its layers' plans (kept alive with it)."""

    def __init__(self, handle, plans):
        self.handle = handle
        self.plans = list(plans)

    def __del__(self):
        try:
            if self.handle:
                rnn_stack_destroy(self)
        except Exception:
            pass


def rnn_stack_create(plans) -> Stack:
    h = ctypes.c_void_p()
    arr = (ctypes.c_void_p * len(plans))(*[p.handle for p in plans])
    _check(load().rnn_stack_create(ctypes.byref(h), arr, len(plans)))
    return Stack(h, plans)


def rnn_stack_destroy(stack: Stack):
    if stack.handle:
        load().rnn_stack_destroy(stack.handle)
        stack.handle = None


def rnn_stack_last_launch_count(stack: Stack) -> int:
    return int(load().rnn_stack_last_launch_count(stack.handle))


def rnn_stack_set_wavefront(stack: Stack, mode=1):
    """0 (or False): layer by layer; 1 (or True): the wavefront where it is
    faster; 2: the wavefront whenever the stack qualifies."""
    _check(load().rnn_stack_set_wavefront(stack.handle, int(mode)))


def rnn_stack_last_wavefront(stack: Stack) -> bool:
    return bool(load().rnn_stack_last_wavefront(stack.handle))


def rnn_stack_run(stack: Stack, X, W, R, B=None, sequence_lens=None, initial_h=None, initial_c=None, P=None,
                  Y=None, Y_h=None, Y_c=None, stream=None):
    """Per-layer arguments are lists (one entry per layer, entries may be None)."""
    plans = stack.plans
    L = len(plans)
    first = plans[0]
    seq, batch = (X.shape[0], X.shape[1]) if first.layout == 0 else (X.shape[1], X.shape[0])
    act = io_dtype(first)
    _need(X, shapes(first, seq, batch)["X"], "X", act)
    _need(sequence_lens, (batch,), "sequence_lens", "int32")

    def per_layer(v, key, name, dt):
        if v is None:
            return None
        if len(v) != L:
            raise ValueError(f"{name}: one entry per layer ({L})")
        for pl, t in zip(plans, v):
            _need(t, shapes(pl, seq, batch)[key], name, dt)
        return (ctypes.c_void_p * L)(*[None if t is None else t.data_ptr() for t in v])
    args = [per_layer(W, "W", "W", "float32"), per_layer(R, "R", "R", "float32"),
            per_layer(B, "B", "B", "float32")]
    h0 = per_layer(initial_h, "state", "initial_h", act)
    c0 = per_layer(initial_c, "state", "initial_c", act)
    Pa = per_layer(P, "P", "P", "float32")
    _need(Y, shapes(plans[-1], seq, batch)["Y"], "Y", act)
    yh = per_layer(Y_h, "state", "Y_h", act)
    yc = per_layer(Y_c, "state", "Y_c", act)
    _check(load().rnn_stack_run(stack.handle, int(seq), int(batch), _ptr(X), args[0], args[1], args[2],
                                _ptr(sequence_lens), h0, c0, Pa, _ptr(Y), yh, yc, _stream(stream)))


def run(plan: Plan, X, W, R, B=None, sequence_lens=None, initial_h=None, initial_c=None, P=None,
        stream=None, want_y=True):
    """Allocate the outputs (torch.empty on X's device) and run; returns (Y, Y_h, Y_c)."""
    import torch
    seq, batch = (X.shape[0], X.shape[1]) if plan.layout == 0 else (X.shape[1], X.shape[0])
    sh = shapes(plan, seq, batch)
    act = io_dtype(plan)
    Y = torch.empty(sh["Y"], dtype=act, device=X.device) if want_y else None
    Yh = torch.empty(sh["state"], dtype=act, device=X.device)
    is_lstm = plan.op in ("LSTM", 2)
    Yc = torch.empty(sh["state"], dtype=act, device=X.device) if is_lstm else None
    rnn_run(plan, X, W, R, B, sequence_lens, initial_h, initial_c, P, Y, Yh, Yc, stream)
    return Y, Yh, Yc
