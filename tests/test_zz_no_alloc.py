"""rnn_run_static_scratch: the entry point for callers that cannot allocate
device memory while they run (a serving runtime that gave the whole GPU's
memory to its own pool at start-up, or a latency-critical caller that cannot
afford cudaMalloc / cudaFree mid-run).  It must give the same results as
rnn_run, call after call, using only the library's fixed device array.

This file is collected last so that a failure here, under -x, comes after
every other test has run; it also passes alone in a fresh process."""
import ctypes

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


def test_static_scratch_timeout_is_reported(lib):
    # one CTA withholds its first arrival and every wait gives up after 50 ms:
    # rnn_plan_sync reads the fixed array's status word and reports TIMEOUT;
    # the next call clears the word and gives rnn_run's bits
    c = make_case("LSTM", "forward", 5, 4, 8, 64, seed=9, h0_scale=0.5, c0_scale=0.5)
    plan = orc.rnn_plan_create(c.op, c.direction, c.hidden_size, c.input_size)
    orc.rnn_plan_set_launch(plan, 4, 1, 1, 0, 1)
    orc.rnn_plan_debug_barrier(plan, 50_000_000, 1)
    dev = {k: (None if v is None else torch.from_numpy(v).cuda()) for k, v in c.tensors().items()}
    outs = [torch.empty(c.y_shape(), device="cuda"), torch.empty(c.state_shape(), device="cuda"),
            torch.empty(c.state_shape(), device="cuda")]
    _static_run(lib, plan, c, dev, outs)
    with pytest.raises(orc.RNNError) as e:
        orc.rnn_plan_sync(plan)
    assert e.value.status == 6
    orc.rnn_plan_debug_barrier(plan, 0, -1)
    ref = gpu_case(c, "exact")
    for call in range(2):
        for o in outs:
            o.fill_(float("nan"))
        _static_run(lib, plan, c, dev, outs)
        orc.rnn_plan_sync(plan)
        for nm, g, r in zip(("Y", "Y_h", "Y_c"), outs, ref):
            assert_bits_equal(g.cpu().numpy(), r, f"after timeout, call {call} {nm}")
    orc.rnn_plan_destroy(plan)


def test_static_scratch_zero_size_takes_any_batch(lib):
    # seq 0 needs no scratch: a batch past the static limit (4096 rows) is
    # served like rnn_run (Y_h = initial_h)
    N, H = 5000, 8
    plan = orc.rnn_plan_create("GRU", "forward", H, 3)
    h0 = torch.randn(1, N, H, device="cuda")
    Yh = torch.full((1, N, H), float("nan"), device="cuda")
    X = torch.empty(0, N, 3, device="cuda")
    W = torch.zeros(1, 3 * H, 3, device="cuda")
    R = torch.zeros(1, 3 * H, H, device="cuda")
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    st = lib.rnn_run_static_scratch(plan.handle, 0, N, p(X), p(W), p(R), None, None, p(h0), None, None,
                                    None, p(Yh), None, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, orc.rnn_last_error()
    torch.cuda.synchronize()
    assert torch.equal(Yh, h0)
    orc.rnn_plan_destroy(plan)
