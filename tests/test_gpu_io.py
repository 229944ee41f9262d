"""fp16 / bf16 activation I/O (rnn_plan_set_io_type) on the GPU against the
oracle's rnn_io: X, initial_h, initial_c given in the 2-byte type and Y,
Y_h, Y_c written in it, the arithmetic fp32.  EXACT mode is compared bit for
bit (the fp32 result is the oracle's, rounded once to nearest even), on the
staged and the dataflow kernels (the latter also with the in-cluster exchange), with sequence_lens, the masked tail, the
zero-size path and the static-scratch entry point; the tensor-core modes
within their bound plus one unit in the last place of the output type."""
import numpy as np
import pytest

import onnx_recurrent_gb300 as orc
import oracle
from onnx_recurrent_gb300.synth import make_case, random_case

pytestmark = pytest.mark.gpu

IOS = ["f16", "bf16"]
TC_TOL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    orc.build()
    oracle.build()


def _to_dev(a, io, torch):
    """A host array in the 2-byte type (float16, or uint16 bf16 bits) to a CUDA tensor."""
    if a is None:
        return None
    if io == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _to_host(t, io):
    if t is None:
        return None
    if io == "bf16":
        return t.view(orc_torch().int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def orc_torch():
    import torch
    return torch


def io_inputs(c, io):
    """The case's X and initial states rounded to the 2-byte type (the inputs both sides see)."""
    return {k: oracle.narrow(getattr(c, k), io) for k in ("X", "initial_h", "initial_c")}


def gpu_io(c, io, mode="exact", launch=None, static=False):
    import torch
    plan = orc.rnn_plan_create(c.op, c.direction, c.hidden_size, c.input_size, activations=c.activations,
                               alpha=c.alpha, beta=c.beta, clip=c.clip, layout=c.layout,
                               linear_before_reset=c.linear_before_reset, input_forget=c.input_forget)
    orc.rnn_plan_set_mode(plan, mode)
    orc.rnn_plan_set_io_type(plan, io)
    if launch:
        orc.rnn_plan_set_launch(plan, *launch)
    act = orc.rnn.io_dtype(plan)
    ins = io_inputs(c, io)
    X, h0, c0 = (_to_dev(ins[k], io, torch) for k in ("X", "initial_h", "initial_c"))
    f32 = {k: (None if getattr(c, k) is None else torch.from_numpy(getattr(c, k)).cuda())
           for k in ("W", "R", "B", "P", "sequence_lens")}
    Y = torch.full(c.y_shape(), float("nan"), device="cuda", dtype=act)
    Yh = torch.full(c.state_shape(), float("nan"), device="cuda", dtype=act)
    Yc = torch.full(c.state_shape(), float("nan"), device="cuda", dtype=act) if c.op == "LSTM" else None
    run = orc.rnn.rnn_run_static_scratch if static else orc.rnn_run
    run(plan, X, f32["W"], f32["R"], f32["B"], f32["sequence_lens"], h0, c0, f32["P"], Y, Yh, Yc)
    orc.rnn_plan_sync(plan)
    torch.cuda.synchronize()
    kernel = orc.rnn_plan_get_launch(plan)["kernel"]
    orc.rnn_plan_destroy(plan)
    return tuple(_to_host(t, io) for t in (Y, Yh, Yc)), kernel


def oracle_io(c, io):
    ins = io_inputs(c, io)
    a = c.attrs()
    return oracle.rnn_io(io, a.pop("op"), a.pop("direction"), a.pop("hidden_size"), a.pop("input_size"),
                         ins["X"], c.W, c.R, B=c.B, sequence_lens=c.sequence_lens, initial_h=ins["initial_h"],
                         initial_c=ins["initial_c"], P=c.P, **a)


def assert_same_bits(got, ref, what):
    for g, r, name in zip(got, ref, ("Y", "Y_h", "Y_c")):
        if r is None:
            continue
        gb, rb = np.asarray(g).view(np.uint16), np.asarray(r).view(np.uint16)
        assert gb.shape == rb.shape, (what, name)
        bad = np.argwhere(gb != rb)
        assert len(bad) == 0, f"{what} {name}: {len(bad)} of {gb.size} differ, first at {tuple(bad[0])}: " \
                              f"{hex(gb[tuple(bad[0])])} vs {hex(rb[tuple(bad[0])])}"


@pytest.mark.parametrize("io", IOS)
@pytest.mark.parametrize("seed", range(12))
def test_random_exact_io_bits(io, seed):
    c = random_case(300 + seed)
    got, _ = gpu_io(c, io)
    assert_same_bits(got, oracle_io(c, io), f"seed {seed} {io}")


@pytest.mark.parametrize("io", IOS)
@pytest.mark.parametrize("launch", [(0, 0, -1, 0, 1), (0, 0, -1, 0, 2), (3, 2, 0, 0, 1), (3, 1, 0, 2, 2),
                                    (6, 0, -1, 0, 5)],
                         ids=["staged", "dataflow", "staged-streamed", "dataflow-streamed", "cluster"])
@pytest.mark.parametrize("op", ["GRU", "LSTM"])
def test_each_kernel_writes_the_io_type(io, launch, op):
    # lengths below seq: the masked tail and the per-row freeze both write 2-byte zeros
    c = make_case(op, "bidirectional", 7, 10, 24, 72, seed=8, layout=1, with_P=True, h0_scale=0.5,
                  c0_scale=0.5, lens=[0, 5, 3, 5, 1, 2, 5, 4, 5, 5], linear_before_reset=0)
    got, kernel = gpu_io(c, io, launch=launch)
    assert kernel == launch[4]
    assert_same_bits(got, oracle_io(c, io), f"{op} {launch} {io}")


@pytest.mark.parametrize("io", IOS)
def test_static_scratch_and_zero_size_io(io):
    c = make_case("LSTM", "forward", 5, 6, 16, 40, seed=4, h0_scale=0.5, c0_scale=0.5)
    got, _ = gpu_io(c, io, static=True)
    assert_same_bits(got, oracle_io(c, io), f"static {io}")
    z = c.with_(seq=0, X=np.zeros((0, 6, 16), np.float32))
    got, _ = gpu_io(z, io)
    ins = io_inputs(c, io)
    assert np.array_equal(np.asarray(got[1]).view(np.uint16), np.asarray(ins["initial_h"]).view(np.uint16))
    assert np.array_equal(np.asarray(got[2]).view(np.uint16), np.asarray(ins["initial_c"]).view(np.uint16))


@pytest.mark.parametrize("io,mode", [("bf16", "bf16"), ("f16", "bf16"), ("bf16", "tf32"), ("f16", "fast")])
def test_fast_modes_io_within_tolerance(io, mode):
    # bf16 X straight into the bf16 tensor-core projection; fp16 X converted;
    # the recurrence on the tensor cores where the planner takes it
    c = make_case("LSTM", "bidirectional", 6, 64, 32, 96, seed=12, with_P=True, h0_scale=0.5, c0_scale=0.5,
                  lens=("uniform", 1, 6), w_scale=1.0 / np.sqrt(96))
    got, kernel = gpu_io(c, io, mode=mode)
    ins = io_inputs(c, io)
    ref = oracle.rnn(c.op, c.direction, c.hidden_size, c.input_size, oracle.widen(ins["X"], io), c.W, c.R,
                     B=c.B, sequence_lens=c.sequence_lens, initial_h=oracle.widen(ins["initial_h"], io),
                     initial_c=oracle.widen(ins["initial_c"], io), P=c.P)
    ulp = 2.0 ** (-10 if io == "f16" else -7)        # one unit in the last place at 1
    tol = (TC_TOL if mode != "fast" else 1e-5)
    for g, r in zip(got, ref):
        if r is None:
            continue
        w = oracle.widen(g, io)
        assert np.all(np.abs(w - r) <= tol + ulp * np.maximum(1.0, np.abs(r))), (io, mode, np.max(np.abs(w - r)))
    if mode != "fast":
        assert kernel == 3
