"""CUDA path vs the oracle, through the C ABI.

Exact mode must be bit-identical to the oracle (page "Recurrent operators:
RNN, GRU, LSTM", Exact mode); fast mode must stay within 1e-5 absolute (scaled
by max(1, |value|) for the unbounded cell state).  Small cases cover the
attribute space and several tiles with ragged tails; forced launch geometries
(CTAs per direction, rows per thread, R resident or streamed) must all give
the same bits; the five workloads run at full size and are compared on
sampled batch rows, which the oracle computes independently (rows of a batch
never interact)."""
import numpy as np
import pytest

import onnx_recurrent_gb300 as orc
from gpu_helpers import gpu_case, row_slice
from helpers import assert_bits_equal, oracle_case
from onnx_recurrent_gb300.synth import make_case, random_case, workload

pytestmark = pytest.mark.gpu

FAST_TOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    orc.build()


def _compare_exact(case, got, ref, what=""):
    for name, g, r in zip(("Y", "Y_h", "Y_c"), got, ref):
        if r is None or g is None:
            continue
        assert_bits_equal(g, r, f"{what} {name}")


def _compare_fast(got, ref, tol=FAST_TOL):
    """|gpu - oracle| <= tol * max(1, |oracle|) elementwise: the absolute bound
    for the bounded outputs of transcendental activations, relative for the
    unbounded ones (Affine, Relu, ... and the LSTM cell).  NaNs must match;
    values past 1e30 (on their way to overflow) are only sign-checked."""
    for name, g, r in zip(("Y", "Y_h", "Y_c"), got, ref):
        if r is None or g is None:
            continue
        g64, r64 = g.astype(np.float64), r.astype(np.float64)
        assert np.array_equal(np.isnan(g64), np.isnan(r64)), f"{name}: NaN positions differ"
        big = ~np.isfinite(r64) | (np.abs(r64) > 1e30)
        big &= ~np.isnan(r64)
        assert np.array_equal(np.sign(g64[big]), np.sign(r64[big])), f"{name}: overflow signs differ"
        ok = ~np.isnan(r64) & ~big
        err = np.abs(g64[ok] - r64[ok]) / np.maximum(1.0, np.abs(r64[ok]))
        worst = float(err.max(initial=0.0))
        assert worst <= tol, f"{name}: max scaled error {worst:.3e} > {tol:.1e}"


@pytest.mark.parametrize("seed", range(80))
def test_random_small_exact_is_bit_identical(seed):
    c = random_case(seed)
    _compare_exact(c, gpu_case(c, "exact"), oracle_case(c), f"seed {seed}")


@pytest.mark.parametrize("seed", range(30))
def test_random_small_fast_within_tolerance(seed):
    # the stated fast-mode bound holds for the transcendental (default)
    # activations: Sigmoid / Tanh gates keep every value bounded
    c = random_case(seed).with_(activations=None, alpha=None, beta=None)
    _compare_fast(gpu_case(c, "fast"), oracle_case(c))


@pytest.mark.parametrize("seed", range(30))
def test_random_small_fast_any_activation_normwise(seed):
    # Unbounded activation chains (Affine, Relu, ...) amplify the one-rounding
    # difference between fused and unfused products by the recurrence's gain,
    # so the bound is normwise: max|gpu - oracle| <= 1e-4 * max(1, max|oracle|).
    c = random_case(seed)
    got, ref = gpu_case(c, "fast"), oracle_case(c)
    for name, g, r in zip(("Y", "Y_h", "Y_c"), got, ref):
        if r is None:
            continue
        g64, r64 = g.astype(np.float64), r.astype(np.float64)
        assert np.array_equal(np.isnan(g64), np.isnan(r64)), name
        fin = np.isfinite(r64) & (np.abs(r64) < 1e30)
        scale = max(1.0, float(np.abs(r64[fin]).max(initial=0.0)))
        assert float(np.abs(g64[fin] - r64[fin]).max(initial=0.0)) <= 1e-4 * scale, name


# (unit_groups, rows_per_thread, r_resident, row_groups, kernel); kernel 1 is
# the staged kernel, 2 the dataflow kernel; zeros and -1 let the planner choose.
GEOMETRIES = [
    (1, 2, 1, 0, 1), (2, 1, 1, 0, 1), (3, 2, 0, 0, 1), (5, 4, 1, 0, 1), (7, 8, 0, 0, 1),
    (13, 1, 0, 0, 1), (72, 2, 1, 0, 1), (4, 8, 1, 0, 1),
    (0, 0, -1, 0, 2), (8, 1, 1, 1, 2), (9, 2, 1, 2, 2), (5, 1, 0, 2, 2), (18, 4, 1, 1, 2),
    (3, 1, 0, 2, 2), (36, 1, 1, 2, 2), (1, 4, 0, 1, 2), (3, 2, 0, 1, 2),
    (9, 8, 0, 1, 2), (4, 8, 1, 1, 2), (6, 4, 1, 1, 2),
]


@pytest.mark.parametrize("op,direction,lbr", [("RNN", "bidirectional", 0), ("GRU", "forward", 0),
                                              ("GRU", "bidirectional", 1), ("LSTM", "reverse", 0),
                                              ("LSTM", "bidirectional", 0), ("GRU", "bidirectional", 0)])
def test_every_launch_geometry_gives_the_same_bits(op, direction, lbr):
    c = make_case(op, direction, 9, 11, 33, 72, seed=21, layout=1, with_P=True, h0_scale=0.5,
                  c0_scale=0.5, lens=("uniform", 0, 9), linear_before_reset=lbr, clip=2.0,
                  activations=None)
    ref = oracle_case(c)
    for g in GEOMETRIES:
        try:
            out = gpu_case(c, "exact", launch=g)
        except orc.RNNError as e:
            pytest.fail(f"geometry {g}: {e}")
        _compare_exact(c, out, ref, f"geometry {g}")


# Input projection through its tensor-copy loader: input sizes that are
# multiples of 4 (16-byte rows) but not of the 16-k stage, row counts
# (seq * batch) and column counts (dirs * gates * hidden) that are not
# multiples of the 128 x 128 tile, so every edge of the zero-filled boxes is
# crossed; and an input size that is not a multiple of 4 (register loader).
@pytest.mark.parametrize("op,direction,seq,batch,inp,hid", [
    ("LSTM", "forward", 7, 19, 20, 40), ("GRU", "bidirectional", 9, 15, 36, 44),
    ("RNN", "reverse", 11, 13, 260, 68), ("LSTM", "bidirectional", 5, 29, 4, 36),
    ("GRU", "forward", 6, 23, 34, 32)])
def test_projection_tile_edges(op, direction, seq, batch, inp, hid):
    c = make_case(op, direction, seq, batch, inp, hid, seed=31, with_P=True, h0_scale=0.5, c0_scale=0.5)
    _compare_exact(c, gpu_case(c, "exact"), oracle_case(c), "exact")
    ref = oracle_case(c)
    for g, r in zip(gpu_case(c, "fast"), ref):
        if g is None or r is None:
            continue
        assert float(np.abs(g.astype(np.float64) - r.astype(np.float64)).max(initial=0.0)) <= 1e-5


@pytest.mark.parametrize("op", ["RNN", "GRU", "LSTM"])
def test_hidden_not_multiple_of_four(op):
    # The dataflow kernel moves whole 16-byte groups of k, so it needs hidden
    # a multiple of 4: the planner falls back to the staged kernel, and
    # forcing the dataflow kernel is refused cleanly.
    c = make_case(op, "bidirectional", 6, 7, 9, 37, seed=8, with_P=True, h0_scale=0.5,
                  lens=("uniform", 1, 6))
    ref = oracle_case(c)
    for g in [(0, 0, -1, 0, 0), (5, 0, 0, 0, 0), (3, 2, 1, 0, 1)]:
        _compare_exact(c, gpu_case(c, "exact", launch=g), ref, f"geometry {g}")
    with pytest.raises(orc.RNNError) as e:
        gpu_case(c, "exact", launch=(0, 0, 1, 0, 2))
    assert e.value.status == 3


# Staged kernel with hidden 1024 and 16-52 units per CTA: the R slice (up to
# 245 KB) does not fit beside the rings, so its leading 32-k chunks stay in
# shared memory and the rest stream (16 bytes at a time where the slice's
# rows are whole 16-byte pieces, else 4); every split gives the same bits.
@pytest.mark.parametrize("op,lbr,launch", [("LSTM", 0, (64, 2, -1, 0, 1)), ("GRU", 0, (52, 2, -1, 0, 1)),
                                           ("GRU", 1, (52, 2, -1, 0, 1)), ("RNN", 0, (17, 2, -1, 0, 1)),
                                           ("LSTM", 0, (64, 2, 0, 0, 1))])
def test_staged_kernel_partly_resident_r(op, lbr, launch):
    c = make_case(op, "bidirectional", 5, 11, 40, 1024, seed=44, with_P=True, h0_scale=0.5, c0_scale=0.5,
                  lens=("uniform", 0, 5), linear_before_reset=lbr, clip=2.0, w_scale=1.0 / 32)
    Y, Yh, Yc, plan = gpu_case(c, "exact", launch=launch, keep_plan=True)
    got = orc.rnn_plan_get_launch(plan)
    orc.rnn_plan_destroy(plan)
    assert got["kernel"] == 1 and got["r_resident"] == 0
    _compare_exact(c, (Y, Yh, Yc), oracle_case(c), f"{op} lbr {lbr} {launch}")


# Dataflow kernel with hidden 1024 and 16-64 units per CTA: the R slice does
# not fit; r_resident 2 keeps its leading pieces resident and streams the
# rest by tensor copies (GRU with linear_before_reset 0 streams the z and r
# rows for the first product of a step and the candidate's rows for the
# second), r_resident 0 streams all of it, -1 lets the planner choose.
# Every split gives the same bits.
@pytest.mark.parametrize("op,lbr,launch", [("LSTM", 0, (64, 0, 2, 1, 2)), ("GRU", 0, (48, 0, 2, 1, 2)),
                                           ("GRU", 1, (48, 0, 2, 1, 2)), ("RNN", 0, (16, 0, 2, 1, 2)),
                                           ("LSTM", 0, (64, 0, 0, 1, 2)), ("GRU", 0, (48, 0, 0, 1, 2)),
                                           ("GRU", 1, (48, 0, -1, 1, 2))])
def test_dataflow_kernel_partly_resident_r(op, lbr, launch):
    c = make_case(op, "bidirectional", 5, 11, 40, 1024, seed=45, with_P=True, h0_scale=0.5, c0_scale=0.5,
                  lens=("uniform", 0, 5), linear_before_reset=lbr, clip=2.0, w_scale=1.0 / 32)
    Y, Yh, Yc, plan = gpu_case(c, "exact", launch=launch, keep_plan=True)
    got = orc.rnn_plan_get_launch(plan)
    orc.rnn_plan_destroy(plan)
    assert got["kernel"] == 2 and got["r_resident"] == 0
    ref = oracle_case(c)
    _compare_exact(c, (Y, Yh, Yc), ref, f"{op} lbr {lbr} {launch}")
    for g, r in zip(gpu_case(c, "fast", launch=launch), ref):
        if g is not None:
            assert float(np.abs(g.astype(np.float64) - r.astype(np.float64)).max(initial=0.0)) <= 1e-5


# Dataflow kernel with the in-cluster exchange (kernel 5): each row group of
# a direction is one thread-block cluster of 1-16 CTAs holding all of R; h
# (and r (.) h) passes through the CTAs' shared memory.  One or two rows per
# thread, one or two row groups, ragged unit splits.
@pytest.mark.parametrize("op,lbr,H,launch", [("LSTM", 0, 128, (8, 2, -1, 1, 5)), ("LSTM", 0, 256, (16, 1, -1, 2, 5)),
                                             ("LSTM", 0, 256, (8, 2, -1, 1, 5)), ("GRU", 0, 256, (9, 2, -1, 2, 5)),
                                             ("GRU", 1, 256, (16, 2, -1, 2, 5)), ("RNN", 0, 512, (12, 2, -1, 2, 5)),
                                             ("GRU", 0, 64, (1, 2, -1, 2, 5))])
def test_cluster_exchange(op, lbr, H, launch):
    c = make_case(op, "bidirectional", 7, 11, 40, H, seed=46, with_P=True, h0_scale=0.5, c0_scale=0.5,
                  lens=("uniform", 0, 7), linear_before_reset=lbr, clip=2.0)
    Y, Yh, Yc, plan = gpu_case(c, "exact", launch=launch, keep_plan=True)
    got = orc.rnn_plan_get_launch(plan)
    orc.rnn_plan_destroy(plan)
    assert got["kernel"] == 5 and got["unit_groups"] == launch[0]
    ref = oracle_case(c)
    _compare_exact(c, (Y, Yh, Yc), ref, f"{op} lbr {lbr} H {H} {launch}")
    for g, r in zip(gpu_case(c, "fast", launch=launch), ref):
        if g is not None:
            assert float(np.abs(g.astype(np.float64) - r.astype(np.float64)).max(initial=0.0)) <= 1e-5


# The in-cluster exchange across the attribute space: one direction or both,
# layouts 0 and 1, named activations with their alpha / beta, clip,
# input_forget, GRU's two products, lengths with empty rows.
@pytest.mark.parametrize("op,direction,layout,attrs", [
    ("LSTM", "forward", 1, dict(activations=["HardSigmoid", "LeakyRelu", "ScaledTanh"], alpha=[0.25, 0.05, 1.5],
                                beta=[0.45, 0.8], input_forget=1, clip=3.0)),
    ("GRU", "reverse", 0, dict(activations=["HardSigmoid", "Softsign"], alpha=[0.2], beta=[0.5],
                               linear_before_reset=0)),
    ("GRU", "bidirectional", 1, dict(linear_before_reset=1, clip=1.5)),
    ("RNN", "bidirectional", 1, dict(activations=["Relu", "Elu"], alpha=[0.7])),
])
def test_cluster_exchange_attributes(op, direction, layout, attrs):
    c = make_case(op, direction, 6, 9, 20, 96, seed=47, layout=layout, with_P=True, h0_scale=0.5,
                  c0_scale=0.5, lens=[6, 0, 3, 6, 1, 5, 6, 2, 4], **attrs)
    ref = oracle_case(c)
    for launch in [(12, 0, -1, 0, 5), (5, 2, -1, 2, 5)]:
        Y, Yh, Yc, plan = gpu_case(c, "exact", launch=launch, keep_plan=True)
        got = orc.rnn_plan_get_launch(plan)
        orc.rnn_plan_destroy(plan)
        assert got["kernel"] == 5 and got["unit_groups"] == launch[0]
        _compare_exact(c, (Y, Yh, Yc), ref, f"{op} {direction} layout {layout} {launch}")


# Gate split (GRU, linear_before_reset 1, one row per thread): three lanes per
# (unit, row), a gate column each over all k in order, the sums gathered by
# shuffles; the launch shows it as 3x the compute threads (ten groups of three
# lanes per warp).  GRU with linear_before_reset 0 (two products) does not
# split.  Both give the oracle's bits.
@pytest.mark.parametrize("lbr,threads", [(1, 6 * 32 + 32), (0, 2 * 32 + 32)])
def test_dataflow_gate_split(lbr, threads):
    c = make_case("GRU", "bidirectional", 9, 4, 20, 56, seed=48, h0_scale=0.5, lens=[9, 0, 4, 7],
                  linear_before_reset=lbr, clip=2.0)
    Y, Yh, Yc, plan = gpu_case(c, "exact", launch=(4, 1, 1, 1, 2), keep_plan=True)
    got = orc.rnn_plan_get_launch(plan)
    orc.rnn_plan_destroy(plan)
    assert got["kernel"] == 2 and got["threads"] == threads
    ref = oracle_case(c)
    _compare_exact(c, (Y, Yh, Yc), ref, f"gate split, lbr {lbr}")
    for g, r in zip(gpu_case(c, "fast", launch=(4, 1, 1, 1, 2)), ref):
        if g is not None:
            assert float(np.abs(g.astype(np.float64) - r.astype(np.float64)).max(initial=0.0)) <= 1e-5


def test_cluster_exchange_more_clusters_than_fit():
    # 16 row groups x 2 directions of 13-CTA clusters: 416 CTAs for 152 SMs;
    # clusters are independent, so the later ones run after the first finish
    c = make_case("LSTM", "bidirectional", 12, 128, 24, 256, seed=49, with_P=True, h0_scale=0.5, c0_scale=0.5,
                  lens=("uniform", 0, 12))
    Y, Yh, Yc, plan = gpu_case(c, "exact", launch=(13, 1, -1, 16, 5), keep_plan=True)
    got = orc.rnn_plan_get_launch(plan)
    orc.rnn_plan_destroy(plan)
    assert got["kernel"] == 5 and got["unit_groups"] == 13 and got["row_groups"] == 16
    _compare_exact(c, (Y, Yh, Yc), oracle_case(c), "416 CTAs in clusters of 13")


def test_cluster_exchange_refuses_streamed_r():
    c = make_case("LSTM", "forward", 3, 4, 8, 64, seed=3)
    with pytest.raises(orc.RNNError) as e:
        gpu_case(c, "exact", launch=(4, 1, 0, 1, 5))
    assert e.value.status == 3


@pytest.mark.parametrize("g", [(2, 1, 0, 0, 1), (5, 2, 1, 0, 1), (4, 1, 1, 2, 2), (3, 2, 0, 1, 2), (4, 1, -1, 1, 5)])
def test_fast_mode_is_geometry_independent(g):
    c = make_case("LSTM", "bidirectional", 6, 9, 20, 36, seed=5, with_P=True, h0_scale=0.5)
    a = gpu_case(c, "fast", launch=(1, 1, 1, 0, 1))
    b = gpu_case(c, "fast", launch=g)
    for x, y in zip(a, b):
        assert_bits_equal(x, y, "fast mode across geometries")


def test_constant_weights_path():
    c = random_case(3, op="LSTM", direction="bidirectional")
    _compare_exact(c, gpu_case(c, "exact", const_weights=True), oracle_case(c), "const")


@pytest.mark.parametrize("want", [("Y",), ("Y_h",), ("Y_c",), ("Y_h", "Y_c")])
def test_optional_outputs(want):
    c = random_case(4, op="LSTM")
    got = gpu_case(c, "exact", want=want)
    ref = oracle_case(c)
    for name, g, r in zip(("Y", "Y_h", "Y_c"), got, ref):
        if name in want:
            assert_bits_equal(g, r, name)
        else:
            assert g is None


@pytest.mark.parametrize("op", ["RNN", "GRU", "LSTM"])
def test_zero_size(op):
    c = make_case(op, "bidirectional", 0, 3, 4, 5, seed=1, h0_scale=0.5, c0_scale=0.5)
    Y, Yh, Yc = gpu_case(c)
    assert Y.size == 0
    assert_bits_equal(Yh, c.initial_h, "Y_h = initial_h")
    if op == "LSTM":
        assert_bits_equal(Yc, c.initial_c, "Y_c = initial_c")
    c2 = c.with_(initial_h=None, initial_c=None)
    _, Yh2, _ = gpu_case(c2)
    assert np.all(Yh2 == 0)


def test_invalid_lengths_write_nothing():
    import torch
    c = make_case("GRU", "forward", 4, 3, 2, 3, seed=2, lens=[1, 5, 2])
    plan = orc.rnn_plan_create("GRU", "forward", 3, 2)
    t = {k: (None if v is None else torch.from_numpy(v).cuda()) for k, v in c.tensors().items()}
    Y = torch.full(c.y_shape(), 7.0, device="cuda")
    Yh = torch.full(c.state_shape(), 7.0, device="cuda")
    with pytest.raises(orc.RNNError) as e:
        orc.rnn_run(plan, t["X"], t["W"], t["R"], t["B"], t["sequence_lens"], Y=Y, Y_h=Yh)
    assert e.value.status == 2
    torch.cuda.synchronize()
    assert bool((Y == 7.0).all()) and bool((Yh == 7.0).all())
    orc.rnn_plan_destroy(plan)


@pytest.mark.parametrize("kernel,lbr", [(1, 0), (2, 0), (2, 1), (5, 0), (5, 1)])
def test_barrier_timeout_is_reported_and_the_device_stays_usable(kernel, lbr):
    # One CTA withholds its first arrival (staged kernel), its first flag
    # (dataflow kernel) or its first arrivals on its cluster peers' barriers
    # (in-cluster exchange); every wait is bounded (50 ms here), so the grid
    # exits (a cluster only after all its CTAs have met) and the status says
    # TIMEOUT.
    op = "LSTM" if lbr == 0 else "GRU"
    c = make_case(op, "forward", 5, 4, 8, 64, seed=9, h0_scale=0.5, linear_before_reset=lbr)
    plan = orc.rnn_plan_create(op, "forward", 64, 8, linear_before_reset=lbr)
    orc.rnn_plan_set_launch(plan, 4, 1, 1, 0, kernel)
    orc.rnn_plan_debug_barrier(plan, 50_000_000, 1)
    import torch
    t = {k: (None if v is None else torch.from_numpy(v).cuda()) for k, v in c.tensors().items()}
    Yh = torch.zeros(c.state_shape(), device="cuda")
    orc.rnn_run(plan, t["X"], t["W"], t["R"], t["B"], initial_h=t["initial_h"], Y_h=Yh)
    with pytest.raises(orc.RNNError) as e:
        orc.rnn_plan_sync(plan)
    assert e.value.status == 6
    orc.rnn_plan_debug_barrier(plan, 0, -1)
    got = gpu_case(c, "exact", plan=plan)
    _compare_exact(c, got, oracle_case(c), "after timeout")
    orc.rnn_plan_destroy(plan)


def test_timing_and_launch_count():
    c = random_case(8, op="GRU", seq=5, lens=("uniform", 0, 3))
    Y, Yh, Yc, plan = gpu_case(c, "exact", keep_plan=True)
    orc.rnn_plan_set_timing(plan, True)
    gpu_case(c, "exact", plan=plan)
    tm = orc.rnn_plan_last_timing(plan)
    assert tm["recurrence"] > 0 and tm["projection"] > 0
    assert orc.rnn_plan_last_launch_count(plan) >= 4
    orc.rnn_plan_destroy(plan)


CONCURRENT = {
    # recurrent grids that fill the GPU: the staged kernel, the dataflow
    # kernel, the tensor-core kernel; and clusters of the in-cluster exchange
    "staged": (dict(op="GRU", direction="bidirectional", seq=24, batch=64, input_size=32, hidden_size=1024,
                    lens=("uniform", 1, 24)), "exact", 1),
    "dataflow": (dict(op="LSTM", direction="forward", seq=24, batch=32, input_size=32, hidden_size=512,
                      with_P=True), "exact", 2),
    "tensor_core": (dict(op="GRU", direction="bidirectional", seq=24, batch=64, input_size=32, hidden_size=512,
                         linear_before_reset=1), "tf32", 3),
    # the in-cluster exchange (the planner's choice here: 4 clusters of 16 CTAs)
    "cluster": (dict(op="LSTM", direction="forward", seq=24, batch=32, input_size=32, hidden_size=256,
                     with_P=True), "exact", 5),
}


@pytest.mark.parametrize("name", sorted(CONCURRENT))
def test_two_plans_on_two_streams(name):
    """Runs of two plans queued on two streams without host waits in between
    give the same bits as one run alone, and none of them times out: the
    recurrent kernels, which need all their CTAs resident at once, must not
    split the SMs between them."""
    import torch
    kw, mode, kernel = CONCURRENT[name]
    kw = dict(kw)
    op, direction = kw.pop("op"), kw.pop("direction")
    c = make_case(op, direction, kw.pop("seq"), kw.pop("batch"), kw.pop("input_size"), kw.pop("hidden_size"),
                  seed=31, h0_scale=0.5, **kw)
    ref = gpu_case(c, mode)
    t = {k: (None if v is None else torch.from_numpy(v).cuda()) for k, v in c.tensors().items()}
    plans, outs = [], []
    for _ in range(2):
        pl = orc.rnn_plan_create(c.op, c.direction, c.hidden_size, c.input_size, clip=c.clip,
                                 linear_before_reset=c.linear_before_reset)
        orc.rnn_plan_set_mode(pl, mode)
        orc.rnn_plan_debug_barrier(pl, 200_000_000, -1)     # a starved wait gives up after 0.2 s
        plans.append(pl)
        outs.append([torch.full(c.y_shape(), float("nan"), device="cuda"),
                     torch.full(c.state_shape(), float("nan"), device="cuda"),
                     torch.full(c.state_shape(), float("nan"), device="cuda") if c.op == "LSTM" else None])
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for _ in range(3):
        for pl, o, st in zip(plans, outs, streams):
            orc.rnn_run(pl, t["X"], t["W"], t["R"], t["B"], t["sequence_lens"], t["initial_h"], t["initial_c"],
                        t["P"], o[0], o[1], o[2], st)
    torch.cuda.synchronize()
    for pl, o in zip(plans, outs):
        assert orc.rnn_plan_get_launch(pl)["kernel"] == kernel
        orc.rnn_plan_sync(pl)
        for x, y in zip(ref, o):
            if x is not None:
                assert_bits_equal(x, y.cpu().numpy())
        orc.rnn_plan_destroy(pl)


# ------------------------------------------------------------ workloads

def _sample_rows(c, k):
    N = c.batch
    rows = {0, N - 1}
    if c.sequence_lens is not None:
        rows.add(int(np.argmax(c.sequence_lens)))
        rows.add(int(np.argmin(c.sequence_lens)))
    rng = np.random.default_rng(123)
    while len(rows) < min(k, N):
        rows.add(int(rng.integers(N)))
    return sorted(rows)


_ORACLE_ROWS = {}


def _oracle_rows(c, rows):
    """The oracle's outputs on the listed rows of a workload (row slices only),
    computed once per (workload, lbr, rows) for the exact and the fast checks."""
    key = (c.name, c.linear_before_reset, tuple(rows))
    if key not in _ORACLE_ROWS:
        ref = oracle_case(c, rows=rows, threaded=True)
        _ORACLE_ROWS[key] = (row_slice(c, rows, ref[0], "Y"), row_slice(c, rows, ref[1], "state"),
                             row_slice(c, rows, ref[2], "state"))
    return _ORACLE_ROWS[key]


def _workload_check(c, rows, mode="exact"):
    got = gpu_case(c, mode)
    rs = _oracle_rows(c, rows)
    gs = (row_slice(c, rows, got[0], "Y"), row_slice(c, rows, got[1], "state"),
          row_slice(c, rows, got[2], "state"))
    if mode == "exact":
        _compare_exact(c, gs, rs, c.name)
    else:
        _compare_fast(gs, rs)
    # at any size: Y is +0 past every row's length
    if c.sequence_lens is not None:
        Y = got[0]
        for n, L in enumerate(c.sequence_lens):
            tail = Y[L:, :, n] if c.layout == 0 else Y[n, L:]
            assert np.all(tail.view(np.uint32) == 0), f"row {n}: Y not zero past len {L}"
    return got


WORKLOAD_CASES = [("rnn_fwd_s8_b1_i16_h128", 0, 1), ("lstm_fwd_s64_b32_i256_h512", 0, 8),
                  ("gru_bidi_s128_b64_i512_h1024", 0, 6), ("gru_bidi_s128_b64_i512_h1024", 1, 6),
                  ("lstm_bidi_s512_b128_i1024_h1024", 0, 3), ("gru_rev_s4096_b4_i256_h2048", 1, 4)]


@pytest.mark.slow
@pytest.mark.parametrize("name,lbr,k", WORKLOAD_CASES, ids=[f"{w[0]}-lbr{w[1]}" for w in WORKLOAD_CASES])
def test_workload_full_size_exact(name, lbr, k):
    c = workload(name, lbr=lbr)
    _workload_check(c, _sample_rows(c, k), "exact")


@pytest.mark.slow
@pytest.mark.parametrize("name,lbr,k", WORKLOAD_CASES, ids=[f"{w[0]}-lbr{w[1]}" for w in WORKLOAD_CASES])
def test_workload_full_size_fast(name, lbr, k):
    # the same rows as the exact check (the oracle's rows are computed once);
    # the 4096-step GRU reverse workload checks all four of its rows, where
    # the fused products' rounding compounds over the most steps
    c = workload(name, lbr=lbr)
    _workload_check(c, _sample_rows(c, k), "fast")


# TF32 and BF16 modes: the input projection on the tensor cores (tcgen05),
# within 5e-3 of the oracle.  Shapes cross the 128 x 128 tile and the k-block
# edges; input sizes that are not multiples of 4 (TF32) or 8 (BF16) take the
# FP32 projection.
TC_TOL = 5e-3
TC_SHAPES = {
    "tf32": [("LSTM", "forward", 7, 19, 20, 40, 0), ("GRU", "bidirectional", 9, 15, 36, 44, 1),
             ("RNN", "reverse", 11, 13, 260, 68, 0), ("LSTM", "bidirectional", 5, 29, 4, 36, 1),
             ("GRU", "forward", 6, 23, 34, 32, 0), ("LSTM", "forward", 3, 50, 96, 136, 0)],
    "bf16": [("LSTM", "forward", 7, 19, 24, 40, 0), ("GRU", "bidirectional", 9, 15, 40, 44, 1),
             ("RNN", "reverse", 11, 13, 264, 68, 0), ("LSTM", "bidirectional", 5, 29, 8, 36, 1),
             ("GRU", "forward", 6, 23, 36, 32, 0), ("LSTM", "forward", 3, 50, 136, 136, 0)],
}


@pytest.mark.parametrize("mode,op,direction,seq,batch,inp,hid,layout",
                         [(m,) + sh for m in ("tf32", "bf16") for sh in TC_SHAPES[m]])
def test_tensor_core_modes_within_tolerance(mode, op, direction, seq, batch, inp, hid, layout):
    # weights scaled like the workloads' (1/sqrt of the longer of hidden and
    # input): bf16's 8-bit mantissas leave an error of about
    # 2^-8 * sqrt(input) * |x| * |w| in the projection, which the 5e-3 bound
    # covers at that scale
    c = make_case(op, direction, seq, batch, inp, hid, seed=41, layout=layout, with_P=True, h0_scale=0.5,
                  c0_scale=0.5, w_scale=1.0 / np.sqrt(max(hid, inp)))
    _compare_fast(gpu_case(c, mode), oracle_case(c), TC_TOL)


@pytest.mark.parametrize("mode", ["tf32", "bf16"])
def test_tensor_core_modes_differ_from_fp32_only_by_the_projection(mode):
    # a zero input projection (X = 0) leaves nothing to round: the tensor-core
    # modes and FAST must then agree bit for bit
    c = make_case("LSTM", "forward", 5, 9, 24, 32, seed=3, with_P=True, h0_scale=0.5, c0_scale=0.5)
    c.X[...] = 0.0
    for g, f in zip(gpu_case(c, mode), gpu_case(c, "fast")):
        if g is not None:
            assert_bits_equal(g, f, f"{mode} vs fast with X = 0")


@pytest.mark.slow
@pytest.mark.parametrize("mode", ["tf32", "bf16"])
@pytest.mark.parametrize("name,lbr,k", WORKLOAD_CASES[1:5], ids=[f"{w[0]}-lbr{w[1]}" for w in WORKLOAD_CASES[1:5]])
def test_workload_full_size_tensor_core_modes(name, lbr, k, mode):
    c = workload(name, lbr=lbr)
    rows = _sample_rows(c, k)
    got = gpu_case(c, mode)
    _compare_fast(tuple(row_slice(c, rows, g, kind) for g, kind in zip(got, ("Y", "state", "state"))),
                  _oracle_rows(c, rows), TC_TOL)


# The tensor-core recurrent kernel (kernel 3: fp16 operands, FP32 sums),
# chosen in the tensor-core modes for 48..128 batch rows with bounded h; on
# smaller batches it is forced through the launch override.
TC_REC_SHAPES = [
    # op, direction, seq, batch, input, hidden, layout, lbr, lens, clip, launch override
    ("LSTM", "bidirectional", 9, 64, 24, 128, 0, 0, ("uniform", 0, 9), None, None),
    ("LSTM", "forward", 7, 128, 40, 200, 1, 0, None, 2.5, None),
    ("GRU", "bidirectional", 8, 100, 16, 136, 1, 1, ("uniform", 1, 8), None, None),
    ("GRU", "reverse", 6, 48, 32, 64, 0, 1, None, None, None),
    ("RNN", "bidirectional", 10, 77, 8, 96, 0, 0, ("uniform", 0, 10), None, None),
    ("LSTM", "reverse", 5, 9, 16, 64, 0, 0, None, None, (0, 0, -1, 0, 3)),
    ("GRU", "forward", 4, 1, 8, 32, 1, 1, None, None, (3, 0, -1, 0, 3)),
    # GRU linear_before_reset = 0: the z, r product, then r (.) h exchanged and the candidate's product
    ("GRU", "bidirectional", 8, 100, 16, 136, 1, 0, ("uniform", 1, 8), None, None),
    ("GRU", "forward", 6, 64, 32, 512, 0, 0, None, 2.0, None),
    ("GRU", "reverse", 5, 48, 8, 64, 0, 0, None, None, (4, 0, -1, 0, 3)),
    ("GRU", "forward", 4, 32, 8, 168, 0, 0, ("uniform", 0, 4), None, (8, 0, -1, 0, 3)),
]


@pytest.mark.parametrize("mode", ["tf32", "bf16"])
@pytest.mark.parametrize("shape", TC_REC_SHAPES, ids=[f"{s[0]}-{s[1]}-n{s[3]}-h{s[5]}" for s in TC_REC_SHAPES])
def test_tensor_core_recurrence_within_tolerance(shape, mode):
    op, direction, seq, batch, inp, hid, layout, lbr, lens, clip, launch = shape
    c = make_case(op, direction, seq, batch, inp, hid, seed=57, layout=layout, with_P=True, h0_scale=0.5,
                  c0_scale=0.5, lens=lens, linear_before_reset=lbr, clip=clip,
                  w_scale=1.0 / np.sqrt(max(hid, inp)))
    Y, Yh, Yc, plan = gpu_case(c, mode, launch=launch, keep_plan=True)
    assert orc.rnn_plan_get_launch(plan)["kernel"] == 3
    orc.rnn_plan_destroy(plan)
    _compare_fast((Y, Yh, Yc), oracle_case(c), TC_TOL)


@pytest.mark.parametrize("what", ["hidden_not_multiple_of_8", "relu", "too_many_rows"])
def test_tensor_core_recurrence_falls_back(what):
    # cases the fp16 tensor-core kernel does not take run on the FP32 kernels
    if what == "hidden_not_multiple_of_8":
        c = make_case("GRU", "forward", 4, 64, 16, 60, seed=5, linear_before_reset=0)
    elif what == "relu":
        c = make_case("RNN", "forward", 4, 64, 16, 64, seed=5, activations=["Relu"], w_scale=0.05)
    else:
        c = make_case("LSTM", "forward", 3, 130, 16, 64, seed=5)
    Y, Yh, Yc, plan = gpu_case(c, "tf32", keep_plan=True)
    assert orc.rnn_plan_get_launch(plan)["kernel"] != 3
    orc.rnn_plan_destroy(plan)
    _compare_fast((Y, Yh, Yc), oracle_case(c), TC_TOL)


@pytest.mark.parametrize("op,lbr", [("LSTM", 0), ("GRU", 0)])
def test_tensor_core_recurrence_timeout_is_reported_and_the_device_stays_usable(op, lbr):
    # one CTA withholds its first publication: the others' bounded waits
    # (50 ms) expire, the status says TIMEOUT, and the next run is correct
    c = make_case(op, "forward", 5, 64, 8, 64, seed=9, h0_scale=0.5, linear_before_reset=lbr)
    plan = orc.rnn_plan_create(op, "forward", 64, 8, linear_before_reset=lbr)
    orc.rnn_plan_set_mode(plan, "tf32")
    orc.rnn_plan_set_launch(plan, 4, 0, -1, 0, 3)
    orc.rnn_plan_debug_barrier(plan, 50_000_000, 1)
    import torch
    t = {k: (None if v is None else torch.from_numpy(v).cuda()) for k, v in c.tensors().items()}
    Yh = torch.zeros(c.state_shape(), device="cuda")
    orc.rnn_run(plan, t["X"], t["W"], t["R"], t["B"], initial_h=t["initial_h"], Y_h=Yh)
    with pytest.raises(orc.RNNError) as e:
        orc.rnn_plan_sync(plan)
    assert e.value.status == 6
    orc.rnn_plan_debug_barrier(plan, 0, -1)
    got = gpu_case(c, "tf32", plan=plan)
    _compare_fast(got, oracle_case(c), TC_TOL)
    orc.rnn_plan_destroy(plan)


def test_rnn_workload_absent_and_zero_initial_state():
    a = gpu_case(workload("rnn_fwd_s8_b1_i16_h128"))
    b = gpu_case(workload("rnn_fwd_s8_b1_i16_h128", initial_h_zero=True))
    for x, y in zip(a[:2], b[:2]):
        assert_bits_equal(x, y)
