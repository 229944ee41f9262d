"""The C-ABI library without a GPU: it builds, loads and exports every symbol
include/onnx_recurrent.h declares; plan creation validates the attributes and
resolves activations exactly as the oracle does; rnn_run rejects bad sizes and
the scratch limit ("Recurrent operators: RNN, GRU, LSTM", Limits) before any
device work."""
import ctypes

import numpy as np
import pytest

import onnx_recurrent_gb300 as orc
import oracle
from onnx_recurrent_gb300 import rnn as rb
from onnx_recurrent_gb300.synth import random_case, workload


@pytest.fixture(scope="module")
def lib():
    orc.build()
    return orc.load()


def test_exports_every_declared_symbol(lib):
    names = rb.declared_functions()
    assert "rnn_plan_create" in names and "rnn_run" in names and "rnn_plan_destroy" in names
    for n in names:
        assert hasattr(lib, n), n


def test_plan_create_and_destroy_without_gpu(lib):
    p = orc.rnn_plan_create("LSTM", "bidirectional", 8, 4)
    orc.rnn_plan_destroy(p)
    orc.rnn_plan_destroy(p)   # idempotent in the binding


@pytest.mark.parametrize("kw", [dict(hidden_size=0), dict(hidden_size=-3), dict(input_size=-1),
                                dict(layout=2), dict(linear_before_reset=2), dict(input_forget=5),
                                dict(activations=["Sigmoid"]),
                                dict(activations=["Sigmoid", "Tanh", "NoSuch"]),
                                dict(op=7), dict(direction=9)])
def test_plan_create_rejects(lib, kw):
    args = dict(op="LSTM", direction="forward", hidden_size=4, input_size=3)
    args.update(kw)
    with pytest.raises(rb.RNNError) as e:
        orc.rnn_plan_create(**args)
    assert e.value.status == 1
    assert orc.rnn_last_error()


def _resolved_lib(case):
    p = orc.rnn_plan_create(case.op, case.direction, case.hidden_size, case.input_size,
                            activations=case.activations, alpha=case.alpha, beta=case.beta)
    k = {"RNN": 1, "GRU": 2, "LSTM": 3}[case.op]
    out = [[orc.rnn_plan_get_activation(p, d, s) for s in range(k)] for d in range(case.dirs)]
    orc.rnn_plan_destroy(p)
    return out


@pytest.mark.parametrize("seed", range(40))
def test_activation_resolution_matches_oracle(lib, seed):
    c = random_case(seed)
    ref = oracle.resolve_activations(c.op, c.direction, c.activations, c.alpha, c.beta)
    got = _resolved_lib(c)
    assert got == ref


def test_activation_resolution_workload(lib):
    c = workload("lstm_bidi_s512_b128_i1024_h1024")
    assert _resolved_lib(c) == oracle.resolve_activations(c.op, c.direction, c.activations,
                                                          c.alpha, c.beta)


def test_run_rejects_sizes_and_scratch_limit_before_device_work(lib):
    p = orc.rnn_plan_create("LSTM", "bidirectional", 1024, 1024)
    fake = ctypes.c_void_p(0x1000)
    st = lib.rnn_run(p.handle, -1, 4, fake, fake, fake, None, None, None, None, None, None, None,
                     None, None)
    assert st == 1
    # per direction: S*N*G*H + 4*N*H + G*H*(I+H) >= 2^30 floats -> Unsupported
    st = lib.rnn_run(p.handle, 4096, 128, fake, fake, fake, None, None, None, None, None, None,
                     None, None, None)
    assert st == 3 and "2^30" in orc.rnn_last_error()
    orc.rnn_plan_destroy(p)


def test_set_launch_validation(lib):
    p = orc.rnn_plan_create("GRU", "forward", 16, 8)
    with pytest.raises(rb.RNNError):
        orc.rnn_plan_set_launch(p, 4, 3, -1)
    with pytest.raises(rb.RNNError):
        orc.rnn_plan_set_launch(p, 4, 1, 3)
    with pytest.raises(rb.RNNError):
        orc.rnn_plan_set_launch(p, 4, 1, -2)
    orc.rnn_plan_set_launch(p, 4, 1, 2)      # partly resident (dataflow kernel)
    orc.rnn_plan_set_launch(p, 4, 2, 0)
    orc.rnn_plan_set_launch(p, 16, 2, -1, 2, 5)   # in-cluster exchange
    for bad in [(4, 1, -1, 0, 4), (4, 4, -1, 0, 5), (17, 1, -1, 0, 5), (4, 1, -1, 0, 6)]:
        with pytest.raises(rb.RNNError):
            orc.rnn_plan_set_launch(p, *bad)
    with pytest.raises(rb.RNNError):
        orc.rnn_plan_set_mode(p, 9)
    orc.rnn_plan_set_mode(p, "fast")
    orc.rnn_plan_destroy(p)


def test_product_does_not_import_or_link_the_oracle():
    import os
    import re
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    pkg = os.path.join(root, "onnx_recurrent_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".cpp", ".h")):
                with open(os.path.join(dirpath, f)) as fh:
                    text = fh.read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
                assert "rnn_oracle" not in text and "liboracle" not in text, f


# ------------------------------------------------------------ single cell

@pytest.mark.parametrize("act", ["Relu", "sigmoid", "TANH", None])
def test_cell_plan_create_resolves_the_page_activations(lib, act):
    p = orc.rnn_cell_plan_create(16, 8, activation=act, clip=2.0)
    name, _, _ = orc.rnn_plan_get_activation(p, 0, 0)
    assert name == ("tanh" if act is None else act.lower())
    orc.rnn_plan_destroy(p)


@pytest.mark.parametrize("kw", [dict(activation="Affine"), dict(activation="LeakyRelu"),
                                dict(activation="NoSuch"), dict(clip=0.0), dict(clip=-2.0),
                                dict(clip=float("nan")), dict(hidden_size=0), dict(input_size=-1)])
def test_cell_plan_create_rejects(lib, kw):
    args = dict(hidden_size=4, input_size=3, activation="Tanh", clip=None)
    args.update(kw)
    with pytest.raises(rb.RNNError) as e:
        orc.rnn_cell_plan_create(**args)
    assert e.value.status == 1


def test_cell_run_checks_before_device_work(lib):
    seq_plan = orc.rnn_plan_create("RNN", "forward", 4, 3)
    cell = orc.rnn_cell_plan_create(4, 3)
    nul = ctypes.c_void_p()
    st = lib.rnn_cell_run(seq_plan.handle, 2, nul, nul, nul, nul, nul, nul, nul)
    assert st == 1 and "cell" in orc.rnn_last_error()
    st = lib.rnn_cell_run(cell.handle, 2, nul, nul, nul, nul, nul, nul, nul)
    assert st == 1
    st = lib.rnn_cell_run(cell.handle, -1, nul, nul, nul, nul, nul, nul, nul)
    assert st == 1
    assert lib.rnn_cell_run(cell.handle, 0, nul, nul, nul, nul, nul, nul, nul) == 0   # batch 0: nothing read
    orc.rnn_plan_destroy(seq_plan)
    orc.rnn_plan_destroy(cell)


# ------------------------------------------------------------ fp16 / bf16 I/O

def test_io_type_validation(lib):
    p = orc.rnn_plan_create("GRU", "forward", 8, 4)
    for io in ("f16", "bf16", "f32"):
        orc.rnn_plan_set_io_type(p, io)
    with pytest.raises(rb.RNNError) as e:
        orc.rnn_plan_set_io_type(p, 7)
    assert e.value.status == 1
    orc.rnn_plan_destroy(p)
    cell = orc.rnn_cell_plan_create(8, 4)
    with pytest.raises(rb.RNNError) as e:
        orc.rnn_plan_set_io_type(cell, "f16")
    assert e.value.status == 3
    orc.rnn_plan_set_io_type(cell, "f32")
    orc.rnn_plan_destroy(cell)


# ------------------------------------------------------------ stacked layers

def test_stack_create_validation(lib):
    a = orc.rnn_plan_create("LSTM", "bidirectional", 8, 4)
    b = orc.rnn_plan_create("GRU", "forward", 5, 16)       # 2 * 8 inputs: chains
    c = orc.rnn_plan_create("GRU", "forward", 5, 15)       # does not
    d = orc.rnn_plan_create("GRU", "forward", 5, 16, layout=1)
    st = orc.rnn_stack_create([a, b])
    orc.rnn_stack_destroy(st)
    for bad in ([a, c], [a, d], [a, orc.rnn_cell_plan_create(5, 16)]):
        with pytest.raises(rb.RNNError) as e:
            orc.rnn_stack_create(bad)
        assert e.value.status == 1
    orc.rnn_plan_set_io_type(b, "f16")
    with pytest.raises(rb.RNNError) as e:
        orc.rnn_stack_create([a, b])
    assert e.value.status == 1 and "io" in orc.rnn_last_error()
    with pytest.raises(rb.RNNError):
        orc.rnn_stack_create([])
