"""Stacked layers (rnn_stack_*) on the GPU against the oracle's rnn_stack:
bit for bit in EXACT mode for mixed operators, directions and layouts
(with and without the layout-0 bidirectional rearrangement between layers),
shared sequence_lens, absent optional outputs; the fp16 I/O stack (the
intermediate sequences stored in fp16) against a per-layer oracle chain;
a tensor-core mode within its bound.

The wavefront (every layer of a unidirectional stack in one launch, layer
l+1 taking step t while layer l takes step t+1) against the oracle and
against the same stack run layer by layer: bit for bit in EXACT and in FAST
mode (both sum every product k ascending in one accumulator), over
operators, directions, layouts, GRU's two reset orders, per-layer
activations and clip, sequence_lens, 2 to 4 layers and batches that take
1, 2 and 4 rows per thread; the stacks it does not take; its bounded
waits."""
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


def gpu_stack(cases, mode="exact", want_y=True, io="f32", X=None, h0=None, c0=None, wavefront=2,
              info=None, debug=None):
    import torch
    plans = []
    for c in cases:
        p = orc.rnn_plan_create(c.op, c.direction, c.hidden_size, c.input_size, activations=c.activations,
                                alpha=c.alpha, beta=c.beta, clip=c.clip, layout=c.layout,
                                linear_before_reset=c.linear_before_reset, input_forget=c.input_forget)
        orc.rnn_plan_set_mode(p, mode)
        orc.rnn_plan_set_io_type(p, io)
        plans.append(p)
    if debug:
        orc.rnn_plan_debug_barrier(plans[0], *debug)
    st = orc.rnn_stack_create(plans)
    orc.rnn_stack_set_wavefront(st, wavefront)
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
    if info is not None:
        info["wavefront"] = orc.rnn_stack_last_wavefront(st)
        info["launch"] = orc.rnn_plan_get_launch(plans[0])
    orc.rnn_stack_destroy(st)
    for p in plans:
        orc.rnn_plan_destroy(p)
    host = lambda t: None if t is None else t.float().cpu().numpy()
    return host(Y), [host(t) for t in Yh], [host(t) for t in Yc], launches


@pytest.mark.parametrize("name", sorted(STACKS))
@pytest.mark.parametrize("seed", [0, 1])
def test_stack_exact_bits(name, seed):
    cases, layout = build_stack(name, seed)
    info = {}
    Y, yh, yc, launches = gpu_stack(cases, info=info)
    rY, ryh, ryc = oracle.rnn_stack(oracle_layers(cases), cases[0].X, sequence_lens=cases[0].sequence_lens)
    assert_bits_equal(rY, Y, f"{name} Y")
    for i, (a, b) in enumerate(zip(ryh, yh)):
        assert_bits_equal(a, b, f"{name} Y_h[{i}]")
    for i, (a, b) in enumerate(zip(ryc, yc)):
        if a is not None:
            assert_bits_equal(a, b, f"{name} Y_c[{i}]")
    # layer by layer: pack, projection, set-up, recurrence per layer; the
    # wavefront: the packs, one projection, one set-up, one recurrence
    assert launches >= (5 if info["wavefront"] else 4 * len(cases))
    assert info["wavefront"] == (name == "fwd_chain")


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


# ------------------------------------------------------------- the wavefront

# per layer (op, direction, hidden, lbr, activations, alpha, beta, clip,
# input_forget); input size of layer 0; layout; lens; batch
WAVE_STACKS = {
    "lstm_fwd_x2": ([("LSTM", "forward", 40, 0, None, None, None, None, 0),
                     ("LSTM", "forward", 40, 0, None, None, None, 2.0, 0)], 24, 0, ("uniform", 0, 7), 5),
    "lstm_rev_x3_layout1": ([("LSTM", "reverse", 36, 0, ["HardSigmoid", "LeakyRelu", "ScaledTanh"],
                              [0.25, 0.05, 1.5], [0.45, 0.8], 3.0, 0),
                             ("LSTM", "reverse", 36, 0, None, None, None, None, 1),
                             ("LSTM", "reverse", 36, 0, ["Sigmoid", "Tanh", "Softsign"], None, None, 1.5, 0)],
                            9, 1, ("uniform", 1, 7), 6),
    "gru_fwd_lbr0_x2": ([("GRU", "forward", 48, 0, None, None, None, None, 0),
                         ("GRU", "forward", 48, 0, ["HardSigmoid", "Tanh"], [0.3], [0.4], 2.5, 0)],
                        16, 0, ("uniform", 0, 7), 7),
    "gru_rev_mixed_lbr_layout1": ([("GRU", "reverse", 32, 1, None, None, None, None, 0),
                                   ("GRU", "reverse", 32, 0, None, None, None, None, 0)], 20, 1, None, 4),
    "rnn_fwd_x4": ([("RNN", "forward", 24, 0, ["Relu"], None, None, None, 0),
                    ("RNN", "forward", 24, 0, ["Tanh"], None, None, None, 0),
                    ("RNN", "forward", 24, 0, ["Affine"], [0.5], [0.1], 4.0, 0),
                    ("RNN", "forward", 24, 0, ["Elu"], [0.7], None, None, 0)], 8, 0, ("uniform", 2, 7), 3),
    "gru_fwd_wide_batch": ([("GRU", "forward", 72, 1, None, None, None, None, 0),
                            ("GRU", "forward", 72, 1, None, None, None, None, 0)], 30, 0, ("uniform", 1, 7), 37),
    # 6 units per CTA in layer 0: 130 rows take 2 rows per thread, 200 rows 4
    "lstm_fwd_batch_130": ([("LSTM", "forward", 256, 0, None, None, None, None, 0),
                            ("LSTM", "forward", 256, 0, None, None, None, None, 0)], 16, 0, ("uniform", 0, 7), 130),
    "gru_rev_batch_200": ([("GRU", "reverse", 256, 1, None, None, None, 2.0, 0),
                           ("GRU", "reverse", 256, 1, None, None, None, None, 0)], 24, 0, ("uniform", 0, 7), 200),
}
WAVE_SEQ = 7


def build_wave(name, seed=0):
    spec, inp, layout, lens, batch = WAVE_STACKS[name]
    cases = []
    for i, (op, direction, hid, lbr, acts, alpha, beta, clip, inf_) in enumerate(spec):
        c = make_case(op, direction, WAVE_SEQ, batch, inp, hid, seed=seed + 31 * i, layout=layout, with_P=True,
                      h0_scale=0.5, c0_scale=0.5, lens=lens if i == 0 else None, linear_before_reset=lbr,
                      activations=acts, alpha=alpha, beta=beta, clip=clip, input_forget=inf_)
        cases.append(c)
        inp = hid
    return cases


def _same(got, ref, what):
    Y, yh, yc = got
    rY, ryh, ryc = ref
    assert_bits_equal(rY, Y, f"{what} Y")
    for i, (a, b) in enumerate(zip(ryh, yh)):
        assert_bits_equal(a, b, f"{what} Y_h[{i}]")
    for i, (a, b) in enumerate(zip(ryc, yc)):
        if a is not None:
            assert_bits_equal(a, b, f"{what} Y_c[{i}]")


@pytest.mark.parametrize("name", sorted(WAVE_STACKS))
def test_wavefront_exact_bits(name):
    cases = build_wave(name)
    info = {}
    Y, yh, yc, _ = gpu_stack(cases, info=info)
    assert info["wavefront"], "the stack should run as one wavefront launch"
    assert info["launch"]["kernel"] == 4
    if name == "lstm_fwd_batch_130":
        assert info["launch"]["rows_per_thread"] == 2
    if name == "gru_rev_batch_200":
        assert info["launch"]["rows_per_thread"] == 4
    ref = oracle.rnn_stack(oracle_layers(cases), cases[0].X, sequence_lens=cases[0].sequence_lens)
    _same((Y, yh, yc), ref, f"{name} vs oracle")
    lY, lyh, lyc, _ = gpu_stack(cases, wavefront=0, info=info)
    assert not info["wavefront"]
    _same((Y, yh, yc), (lY, lyh, lyc), f"{name} vs layer by layer")


@pytest.mark.parametrize("name", ["lstm_fwd_x2", "gru_fwd_lbr0_x2", "rnn_fwd_x4", "lstm_fwd_batch_130"])
def test_wavefront_fast_matches_layer_by_layer(name):
    # fast mode: one fused multiply-add chain per output, k ascending, in the
    # projection GEMM and in the wavefront's own input product alike
    cases = build_wave(name, seed=3)
    info = {}
    got = gpu_stack(cases, mode="fast", info=info)[:3]
    assert info["wavefront"]
    lay = gpu_stack(cases, mode="fast", wavefront=0)[:3]
    _same(got, lay, f"{name} fast")
    rY, ryh, _ = oracle.rnn_stack(oracle_layers(cases), cases[0].X, sequence_lens=cases[0].sequence_lens)
    if name != "rnn_fwd_x4":            # Relu / Affine chains: the normwise bound of the single-layer tests
        assert np.max(np.abs(got[0] - rY)) <= 1e-5


@pytest.mark.parametrize("what", ["bidirectional", "mixed_ops", "f16_io", "tf32", "disabled", "one_layer",
                                  "large_layers"])
def test_wavefront_not_taken(what):
    if what == "bidirectional":
        cases, _ = build_stack("gru_bidi_x3")
    elif what == "mixed_ops":
        cases = [make_case("LSTM", "forward", 6, 5, 12, 16, seed=1), make_case("GRU", "forward", 6, 5, 16, 16, seed=2)]
    else:
        cases = build_wave("lstm_fwd_x2")
    if what == "one_layer":
        cases = cases[:1]
    if what == "large_layers":
        # 8 x 4 x 512 x 1024 products per step of the second layer: the automatic
        # choice (mode 1) runs such layers one after another
        cases = [make_case("LSTM", "forward", 3, 8, 64, 512, seed=1), make_case("LSTM", "forward", 3, 8, 512, 512, seed=2)]
    info = {}
    kw = {"f16_io": dict(io="f16"), "tf32": dict(mode="tf32"), "disabled": dict(wavefront=0)}.get(what, {})
    if what == "f16_io":
        n16 = lambda a: None if a is None else oracle.narrow(a, "f16")
        kw.update(X=n16(cases[0].X), h0=[n16(c.initial_h) for c in cases], c0=[n16(c.initial_c) for c in cases])
    if what == "large_layers":
        kw["wavefront"] = 1
    gpu_stack(cases, info=info, **kw)
    assert not info["wavefront"]


def test_wavefront_timeout_is_reported_and_the_device_stays_usable():
    # CTA 1 (layer 0) withholds its first arrival; every wait gives up after
    # 50 ms; the first layer's plan reports TIMEOUT, and a clean run after it
    # gives the oracle's bits
    cases = build_wave("lstm_fwd_x2")
    with pytest.raises(orc.RNNError) as e:
        gpu_stack(cases, debug=(50_000_000, 1))
    assert e.value.status == 6
    Y, yh, yc, _ = gpu_stack(cases)
    _same((Y, yh, yc), oracle.rnn_stack(oracle_layers(cases), cases[0].X, sequence_lens=cases[0].sequence_lens),
          "after timeout")
