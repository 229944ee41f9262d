"""Shared test helpers: run an RNNCase through the oracle."""
import numpy as np

import oracle


def oracle_case(case, rows=None, threaded=False, **over):
    a = case.attrs()
    a.update(over)
    t = case.tensors()
    args = (a.pop("op"), a.pop("direction"), a.pop("hidden_size"), a.pop("input_size"),
            t.pop("X"), t.pop("W"), t.pop("R"))
    if threaded:
        return oracle.rnn_threaded(*args, rows=rows, **t, **a)
    if rows is not None:
        return oracle.rnn(*args, rows=rows, **t, **a)
    return oracle.rnn(*args, **t, **a)


def bits(a):
    return np.ascontiguousarray(a, np.float32).view(np.uint32)


def assert_bits_equal(a, b, what=""):
    a = np.ascontiguousarray(a, np.float32)
    b = np.ascontiguousarray(b, np.float32)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    ba, bb = a.view(np.uint32), b.view(np.uint32)
    if not np.array_equal(ba, bb):
        idx = np.argwhere(ba != bb)
        i = tuple(idx[0])
        raise AssertionError(f"{what}: {len(idx)} of {a.size} values differ; first at {i}: "
                             f"{a[i]!r} ({ba[i]:#010x}) vs {b[i]!r} ({bb[i]:#010x})")
