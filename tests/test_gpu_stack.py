"""Stacked layers (rnn_stack_*) on the GPU against the oracle's rnn_stack:
bit for bit in EXACT mode for mixed operators, directions and layouts
(with and without the layout-0 bidirectional rearrangement between layers),
shared sequence_lens, absent optional outputs; the fp16 I/O stack (the
intermediate sequences stored in fp16) against a per-layer oracle chain;
a tensor-core mode within its bound."""
import numpy as np
import pytest

import onnx_recurrent_gb300 as orc
import oracle
from helpers import assert_bits_equal
from onnx_recurrent_gb300.synth import make_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    orc.build()
    oracle.build()


STACKS = {
    # (op, direction, hidden, lbr) per layer; input of layer 0; layout; lens
    "lstm_bidi_gru_fwd": ([("LSTM", "bidirectional", 24, 0), ("GRU", "forward", 16, 1)], 12, 0, ("uniform", 0, 6)),
    "gru_bidi_x3": ([("GRU", "bidirectional", 20, 0), ("GRU", "bidirectional", 20, 1), ("RNN", "reverse", 12, 0)],
                    9, 0, None),
    "layout1_mixed": ([("RNN", "bidirectional", 16, 0), ("LSTM", "forward", 32, 0), ("GRU", "reverse", 8, 0)],
                      7, 1, ("uniform", 1, 6)),
    "fwd_chain": ([("LSTM", "forward", 40, 0), ("LSTM", "forward", 40, 0)], 40, 0, None),
}
SEQ, BATCH = 6, 5


def build_stack(name, seed=0):
    spec, inp, layout, lens = STACKS[name]
    cases = []
    for i, (op, direction, hid, lbr) in enumerate(spec):
        c = make_case(op, direction, SEQ, BATCH, inp, hid, seed=seed + 17 * i, layout=layout, with_P=True,
                      h0_scale=0.5, c0_scale=0.5, lens=lens if i == 0 else None, linear_before_reset=lbr)
        cases.append(c)
        inp = c.dirs * hid
    return cases, layout


def oracle_layers(cases):
    out = []
    for c in cases:
        a = c.attrs()
        a.update(W=c.W, R=c.R, B=c.B, P=c.P, initial_h=c.initial_h, initial_c=c.initial_c)
        out.append(a)
    return out


def gpu_stack(cases, mode="exact", want_y=True, io="f32", X=None, h0=None, c0=None):
    import torch
    plans = []
    for c in cases:
        p = orc.rnn_plan_create(c.op, c.direction, c.hidden_size, c.input_size, clip=c.clip, layout=c.layout,
                                linear_before_reset=c.linear_before_reset)
        orc.rnn_plan_set_mode(p, mode)
        orc.rnn_plan_set_io_type(p, io)
        plans.append(p)
    st = orc.rnn_stack_create(plans)
    act = orc.rnn.io_dtype(plans[0])
    dev = lambda a, dt=torch.float32: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda().to(dt)
    c0_ = cases[0]
    Xd = dev(c0_.X if X is None else X, act)
    lens = None if c0_.sequence_lens is None else torch.from_numpy(c0_.sequence_lens).cuda()
    last = cases[-1]
    Y = torch.full(last.y_shape(), float("nan"), device="cuda", dtype=act) if want_y else None
    Yh = [torch.full(c.state_shape(), float("nan"), device="cuda", dtype=act) for c in cases]
    Yc = [torch.full(c.state_shape(), float("nan"), device="cuda", dtype=act) if c.op == "LSTM" else None
          for c in cases]
    orc.rnn_stack_run(st, Xd, [dev(c.W) for c in cases], [dev(c.R) for c in cases], [dev(c.B) for c in cases],
                      lens, [dev(c.initial_h if h0 is None else h0[i], act) for i, c in enumerate(cases)],
                      [dev(c.initial_c if c0 is None else c0[i], act) for i, c in enumerate(cases)],
                      [dev(c.P) for c in cases], Y, Yh, Yc)
    for p in plans:
        orc.rnn_plan_sync(p)
    torch.cuda.synchronize()
    launches = orc.rnn_stack_last_launch_count(st)
    orc.rnn_stack_destroy(st)
    host = lambda t: None if t is None else t.float().cpu().numpy()
    return host(Y), [host(t) for t in Yh], [host(t) for t in Yc], launches


@pytest.mark.parametrize("name", sorted(STACKS))
@pytest.mark.parametrize("seed", [0, 1])
def test_stack_exact_bits(name, seed):
    cases, layout = build_stack(name, seed)
    Y, yh, yc, launches = gpu_stack(cases)
    rY, ryh, ryc = oracle.rnn_stack(oracle_layers(cases), cases[0].X, sequence_lens=cases[0].sequence_lens)
    assert_bits_equal(rY, Y, f"{name} Y")
    for i, (a, b) in enumerate(zip(ryh, yh)):
        assert_bits_equal(a, b, f"{name} Y_h[{i}]")
    for i, (a, b) in enumerate(zip(ryc, yc)):
        if a is not None:
            assert_bits_equal(a, b, f"{name} Y_c[{i}]")
    assert launches >= 4 * len(cases)


def test_stack_without_output_sequence():
    cases, _ = build_stack("lstm_bidi_gru_fwd", 3)
    Y, yh, _, _ = gpu_stack(cases, want_y=False)
    assert Y is None
    _, ryh, _ = oracle.rnn_stack(oracle_layers(cases), cases[0].X, sequence_lens=cases[0].sequence_lens)
    assert_bits_equal(ryh[-1], yh[-1], "last Y_h")


def test_stack_f16_io_chain():
    # every layer reads and writes fp16: the oracle chain rounds each layer's
    # outputs once and feeds them (exactly widened) to the next layer
    cases, layout = build_stack("lstm_bidi_gru_fwd", 5)
    n16 = lambda a: None if a is None else oracle.narrow(a, "f16")
    X16 = n16(cases[0].X)
    h16 = [n16(c.initial_h) for c in cases]
    c16 = [n16(c.initial_c) for c in cases]
    Y, yh, yc, _ = gpu_stack(cases, io="f16", X=X16, h0=h16, c0=c16)
    x = X16
    for i, c in enumerate(cases):
        a = c.attrs()
        rY, rYh, rYc = oracle.rnn_io("f16", a.pop("op"), a.pop("direction"), a.pop("hidden_size"),
                                     a.pop("input_size"), x, c.W, c.R, B=c.B, sequence_lens=cases[0].sequence_lens,
                                     initial_h=h16[i], initial_c=c16[i], P=c.P, **a)
        assert np.array_equal(yh[i].astype(np.float16).view(np.uint16), rYh.view(np.uint16)), i
        x = oracle.narrow(oracle.stack_input(oracle.widen(rY, "f16"), layout), "f16")
    assert np.array_equal(Y.astype(np.float16).view(np.uint16), rY.view(np.uint16))


def test_stack_tensor_core_mode_within_tolerance():
    cases, _ = build_stack("fwd_chain", 2)
    Y, yh, _, _ = gpu_stack(cases, mode="tf32")
    rY, ryh, _ = oracle.rnn_stack(oracle_layers(cases), cases[0].X)
    assert np.max(np.abs(Y - rY)) <= 5e-3
    assert np.max(np.abs(yh[-1] - ryh[-1])) <= 5e-3
