"""The single RNN cell (page "RNNCell", RNNCell-3) on the GPU against the
oracle's cell: bit-exact in exact mode, within the stated bounds in the fast
modes, over shapes that span several tiles with ragged edges, the page's
example shapes and a large batch; chained cells against the sequence
operator; constant weights; the zero-size and error paths."""
import numpy as np
import pytest

import onnx_recurrent_gb300 as orc
import oracle
from helpers import assert_bits_equal
from onnx_recurrent_gb300.synth import cell_workload, make_cell_case

pytestmark = pytest.mark.gpu

FAST_TOL = 1e-5
TC_TOL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    orc.build()
    oracle.build()


def _dev(c):
    import torch
    return {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in c.tensors().items()}


def gpu_cell(c, mode="exact", const_weights=False, plan=None):
    import torch
    own = plan is None
    if own:
        plan = orc.rnn_cell_plan_create(c.hidden_size, c.input_size, activation=c.activation, clip=c.clip)
        orc.rnn_plan_set_mode(plan, mode)
    t = _dev(c)
    W, R = t["W"], t["R"]
    if const_weights:
        orc.rnn_plan_set_weights(plan, W[None], R[None])
        W = R = None
    Ho = torch.full((c.batch, c.hidden_size), float("nan"), device="cuda")
    orc.rnn_cell_run(plan, t["X"], t["H"], W, R, t["B"], Ho)
    orc.rnn_plan_sync(plan)
    torch.cuda.synchronize()
    if own:
        orc.rnn_plan_destroy(plan)
    return Ho.cpu().numpy()


def oracle_cell(c):
    return oracle.rnn_cell(c.hidden_size, c.input_size, c.X, c.H, c.W, c.R, c.B,
                           activation=c.activation, clip=float("inf") if c.clip is None else c.clip)


SHAPES = [(1, 16, 128), (3, 5, 7), (9, 37, 41), (64, 256, 512), (33, 0, 20), (130, 100, 96)]


@pytest.mark.parametrize("shape", SHAPES, ids=[f"b{b}_i{i}_h{h}" for b, i, h in SHAPES])
@pytest.mark.parametrize("act", ["Tanh", "Sigmoid", "Relu"])
@pytest.mark.parametrize("clip", [None, 0.3])
def test_cell_exact_is_bit_identical(shape, act, clip):
    b, i, h = shape
    c = make_cell_case(b, i, h, seed=b + i + h, activation=act, clip=clip, w_scale=0.6)
    assert_bits_equal(oracle_cell(c), gpu_cell(c), f"cell {shape} {act} {clip}")


@pytest.mark.parametrize("shape", SHAPES[:4])
@pytest.mark.parametrize("mode,tol", [("fast", FAST_TOL), ("tf32", TC_TOL), ("bf16", TC_TOL)])
def test_cell_fast_modes_within_tolerance(shape, mode, tol):
    b, i, h = shape
    c = make_cell_case(b, i, h, seed=7 + b, activation="Tanh")
    err = np.max(np.abs(gpu_cell(c, mode) - oracle_cell(c)))
    assert err <= tol, (mode, err)


@pytest.mark.parametrize("name", ["rnncell_b1_i16_h128", "rnncell_b256_i1024_h1024"])
def test_cell_workloads_exact(name):
    c = cell_workload(name)
    assert_bits_equal(oracle_cell(c), gpu_cell(c), name)


def test_cell_constant_weights():
    c = make_cell_case(17, 24, 40, seed=3, activation="Sigmoid", clip=1.0)
    assert_bits_equal(oracle_cell(c), gpu_cell(c, const_weights=True), "constant weights")


def test_chained_cells_are_the_sequence_operator():
    # S cell calls, each fed the previous Ho, against the sequence operator's
    # oracle with B = [B | -0] over S steps: bit for bit.
    import torch
    S, N, I, H = 5, 6, 12, 24
    c = make_cell_case(N, I, H, seed=21, activation="Tanh", clip=2.0, w_scale=0.5)
    g = np.random.default_rng(5)
    Xs = g.uniform(-1, 1, (S, N, I)).astype(np.float32)
    plan = orc.rnn_cell_plan_create(H, I, activation="Tanh", clip=2.0)
    t = _dev(c)
    h = t["H"].clone()
    for s in range(S):
        out = torch.empty_like(h)
        orc.rnn_cell_run(plan, torch.from_numpy(Xs[s]).cuda(), h, t["W"], t["R"], t["B"], out)
        h = out
    orc.rnn_plan_sync(plan)
    orc.rnn_plan_destroy(plan)
    Bs = np.concatenate([c.B, np.full(H, -0.0, np.float32)])[None]
    _, Yh, _ = oracle.rnn("RNN", "forward", H, I, Xs, c.W[None], c.R[None], B=Bs, initial_h=c.H[None],
                          activations=["Tanh"], clip=2.0)
    assert_bits_equal(Yh[0], h.cpu().numpy(), "chained")


def test_cell_zero_batch_and_errors():
    import torch
    plan = orc.rnn_cell_plan_create(8, 4)
    z = torch.zeros((0, 8), device="cuda")
    orc.rnn_cell_run(plan, torch.zeros((0, 4), device="cuda"), z, torch.zeros((8, 4), device="cuda"),
                     torch.zeros((8, 8), device="cuda"), torch.zeros(8, device="cuda"), z)
    assert orc.rnn_plan_last_launch_count(plan) == 0
    seq = orc.rnn_plan_create("RNN", "forward", 8, 4)
    with pytest.raises(orc.RNNError) as e:
        orc.rnn_cell_run(seq, torch.zeros((2, 4), device="cuda"), torch.zeros((2, 8), device="cuda"),
                         torch.zeros((8, 4), device="cuda"), torch.zeros((8, 8), device="cuda"),
                         torch.zeros(8, device="cuda"), torch.zeros((2, 8), device="cuda"))
    assert e.value.status == 1
    orc.rnn_plan_destroy(seq)
    orc.rnn_plan_destroy(plan)


def test_cell_is_one_launch_and_timed_as_the_recurrence():
    import torch
    c = make_cell_case(40, 24, 72, seed=2)
    plan = orc.rnn_cell_plan_create(72, 24)
    orc.rnn_plan_set_timing(plan, True)
    t = _dev(c)
    Ho = torch.empty((40, 72), device="cuda")
    orc.rnn_cell_run(plan, t["X"], t["H"], t["W"], t["R"], t["B"], Ho)
    orc.rnn_plan_sync(plan)
    assert orc.rnn_plan_last_launch_count(plan) == 1
    assert orc.rnn_plan_last_timing(plan)["recurrence"] > 0
    orc.rnn_plan_destroy(plan)
    assert_bits_equal(oracle_cell(c), Ho.cpu().numpy(), "timed")
