"""rnn_run_static_scratch: the entry point for callers that cannot allocate
device memory while they run (a serving runtime that gave the whole GPU's
memory to its own pool at start-up, or a latency-critical caller that cannot
afford cudaMalloc / cudaFree mid-run).  It must give the same results as
rnn_run, call after call, using only the library's fixed device array.

This file is collected last so that a failure here, under -x, comes after
every other test has run; it also passes alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import onnx_recurrent_gb300 as orc
from gpu_helpers import gpu_case
from helpers import assert_bits_equal
from onnx_recurrent_gb300.synth import make_case, workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    orc.build()
    return orc.load()


def _static_run(lib, plan, case, dev, outs):
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    st = lib.rnn_run_static_scratch(
        plan.handle, case.seq, case.batch, p(dev["X"]), p(dev["W"]), p(dev["R"]), p(dev["B"]),
        p(dev["sequence_lens"]), p(dev["initial_h"]), p(dev["initial_c"]), p(dev["P"]),
        p(outs[0]), p(outs[1]), p(outs[2]),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, orc.rnn_last_error()


CASES = {
    "lstm_fwd_s64_b32_i256_h512": lambda: workload("lstm_fwd_s64_b32_i256_h512"),
    "gru_bidi_lbr0_lens_layout1": lambda: make_case("GRU", "bidirectional", 11, 9, 20, 70, seed=3,
                                                    layout=1, lens=("uniform", 0, 11),
                                                    h0_scale=0.5, linear_before_reset=0),
    "lstm_rev_input_forget_clip": lambda: make_case("LSTM", "reverse", 7, 5, 13, 33, seed=4,
                                                    with_P=True, h0_scale=0.5, c0_scale=0.5,
                                                    input_forget=1, clip=1.5),
}


@pytest.mark.parametrize("name", list(CASES))
def test_static_scratch_matches_rnn_run_on_two_calls(lib, name):
    c = CASES[name]()
    ref = gpu_case(c, "exact")
    plan = orc.rnn_plan_create(c.op, c.direction, c.hidden_size, c.input_size,
                               activations=c.activations, alpha=c.alpha, beta=c.beta, clip=c.clip,
                               layout=c.layout, linear_before_reset=c.linear_before_reset,
                               input_forget=c.input_forget)
    dev = {k: (None if v is None else torch.from_numpy(v).cuda()) for k, v in c.tensors().items()}
    for call in range(2):
        outs = [torch.full(c.y_shape(), float("nan"), device="cuda"),
                torch.full(c.state_shape(), float("nan"), device="cuda"),
                torch.full(c.state_shape(), float("nan"), device="cuda") if c.op == "LSTM" else None]
        _static_run(lib, plan, c, dev, outs)
        torch.cuda.synchronize()
        for nm, g, r in zip(("Y", "Y_h", "Y_c"), outs, ref):
            if r is not None:
                assert_bits_equal(g.cpu().numpy(), r, f"{name} call {call} {nm}")
    orc.rnn_plan_destroy(plan)


def test_static_scratch_refuses_runs_that_do_not_fit(lib):
    c = workload("gru_bidi_s128_b64_i512_h1024")     # ~200 MB of projection scratch
    plan = orc.rnn_plan_create(c.op, c.direction, c.hidden_size, c.input_size, layout=c.layout)
    dev = {k: (None if v is None else torch.from_numpy(v).cuda()) for k, v in c.tensors().items()}
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    st = lib.rnn_run_static_scratch(plan.handle, c.seq, c.batch, p(dev["X"]), p(dev["W"]),
                                    p(dev["R"]), p(dev["B"]), p(dev["sequence_lens"]), None, None,
                                    None, None, None, None,
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 3
    assert "static scratch" in orc.rnn_last_error()
    orc.rnn_plan_destroy(plan)


def test_static_scratch_runs_inside_a_cuda_graph(lib):
    # captured once (after one call outside the capture, which looks up the
    # static array), then replayed with new inputs: the same bits as rnn_run
    c = make_case("LSTM", "forward", 6, 8, 16, 64, seed=11, with_P=True, h0_scale=0.5, c0_scale=0.5)
    plan = orc.rnn_plan_create(c.op, c.direction, c.hidden_size, c.input_size, layout=c.layout)
    dev = {k: (None if v is None else torch.from_numpy(v).cuda()) for k, v in c.tensors().items()}
    outs = [torch.empty(c.y_shape(), device="cuda"), torch.empty(c.state_shape(), device="cuda"),
            torch.empty(c.state_shape(), device="cuda")]
    _static_run(lib, plan, c, dev, outs)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            _static_run(lib, plan, c, dev, outs)
    torch.cuda.synchronize()
    g = np.random.default_rng(2)
    for rep in range(2):
        X = g.normal(size=c.X.shape).astype(np.float32)
        dev["X"].copy_(torch.from_numpy(X))
        for o in outs:
            o.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        ref = gpu_case(c.with_(X=X), "exact")
        for nm, got, r in zip(("Y", "Y_h", "Y_c"), outs, ref):
            assert_bits_equal(got.cpu().numpy(), r, f"replay {rep} {nm}")
    del graph
    orc.rnn_plan_destroy(plan)
