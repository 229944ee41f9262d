"""Pins for the oracle's fp16/bf16 activation I/O (the operator's type T in
its 2-byte variants, Apple BNNS page): widening is exact, narrowing rounds
to nearest with ties to even, overflow goes to infinity, NaN becomes the
type's canonical quiet NaN.  Expected bit patterns are worked out by hand
from the formats (fp16: 1 sign, 5 exponent, 10 fraction bits; bf16: the
upper 16 bits of fp32)."""
import numpy as np
import pytest

import oracle

F16_CASES = [
    # value, expected fp16 bits, why
    (1.0, 0x3C00, "exact"),
    (1.0 + 2.0 ** -11, 0x3C00, "halfway between 1 and 1 + 2^-10: ties to even (1)"),
    (1.0 + 3 * 2.0 ** -11, 0x3C02, "halfway between 1 + 2^-10 and 1 + 2^-9: ties to even"),
    (1.0 + 2.0 ** -11 + 2.0 ** -20, 0x3C01, "just above halfway: rounds up"),
    (65504.0, 0x7BFF, "largest finite"),
    (65520.0, 0x7C00, "halfway between 65504 and 2^16: ties to even, which overflows to infinity"),
    (2.0 ** -24, 0x0001, "smallest subnormal"),
    (2.0 ** -25, 0x0000, "half the smallest subnormal: ties to even (0)"),
    (3 * 2.0 ** -26, 0x0001, "above half the smallest subnormal"),
    (-0.0, 0x8000, "negative zero keeps its sign"),
    (-2.5, 0xC100, "exact negative"),
    (float("inf"), 0x7C00, "infinity"),
    (float("nan"), 0x7E00, "canonical quiet NaN"),
]

BF16_CASES = [
    (1.0, 0x3F80, "exact"),
    (1.0 + 2.0 ** -8, 0x3F80, "halfway between 1 and 1 + 2^-7: ties to even (1)"),
    (1.0 + 3 * 2.0 ** -8, 0x3F82, "halfway between 1 + 2^-7 and 1 + 2^-6: ties to even"),
    (1.0 + 2.0 ** -8 + 2.0 ** -20, 0x3F81, "just above halfway: rounds up"),
    (-0.0, 0x8000, "negative zero"),
    (2.0 ** -133, 0x0001, "smallest bf16 subnormal (exact in fp32)"),
    (3.3895313892515355e38, 0x7F7F, "largest finite bf16"),
    (3.4e38, 0x7F80, "past the halfway point above the largest finite: infinity"),
    (float("-inf"), 0xFF80, "negative infinity"),
    (float("nan"), 0x7FC0, "canonical quiet NaN"),
]


@pytest.mark.parametrize("v,bits,why", F16_CASES, ids=[c[2] for c in F16_CASES])
def test_narrow_f16(v, bits, why):
    got = oracle.narrow(np.array([v], np.float32), "f16").view(np.uint16)[0]
    assert got == bits, (why, hex(got))


@pytest.mark.parametrize("v,bits,why", BF16_CASES, ids=[c[2] for c in BF16_CASES])
def test_narrow_bf16(v, bits, why):
    got = oracle.narrow(np.array([v], np.float32), "bf16")[0]
    assert got == bits, (why, hex(got))


def test_widen_is_exact_and_inverts_narrow():
    # every bf16 pattern widens to the fp32 whose upper half it is; every
    # finite fp16 value survives a round trip
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    w = oracle.widen(bits, "bf16")
    assert np.array_equal(w.view(np.uint32) >> 16, bits.astype(np.uint32))
    assert np.array_equal(w.view(np.uint32) & 0xFFFF, np.zeros(1 << 16, np.uint32))
    back = oracle.narrow(w, "bf16")
    finite = ~np.isnan(w)
    assert np.array_equal(back[finite], bits[finite])
    h = bits.view(np.float16)
    wh = oracle.widen(h, "f16")
    fin = np.isfinite(wh)
    assert np.array_equal(oracle.narrow(wh, "f16").view(np.uint16)[fin], bits[fin])
    assert wh[0x3C00] == 1.0 and wh[0x0001] == 2.0 ** -24 and wh[0x7BFF] == 65504.0


@pytest.mark.parametrize("io", ["f16", "bf16"])
def test_rnn_io_is_the_fp32_operator_rounded(io):
    # the hand case of the two-step Affine RNN (W = 2, R = 0.5, clip 2.5):
    # outputs 2 and -2.5 are exact in both 2-byte types
    X = np.array([[[1.0]], [[-10.0]]], np.float32)
    Xio = oracle.narrow(X, io)
    Y, Yh, _ = oracle.rnn_io(io, "RNN", "forward", 1, 1, Xio, np.full((1, 1, 1), 2.0, np.float32),
                             np.full((1, 1, 1), 0.5, np.float32), activations=["Affine"], clip=2.5)
    assert np.array_equal(oracle.widen(Y, io).ravel(), [2.0, -2.5])
    assert np.array_equal(oracle.widen(Yh, io).ravel(), [-2.5])


@pytest.mark.parametrize("io", ["f16", "bf16"])
def test_rnn_io_rounds_once(io):
    # a random case: the 2-byte outputs are the fp32 operator's outputs
    # (on the widened inputs) rounded once, and within half an ulp of them
    g = np.random.default_rng(3)
    X = g.normal(size=(4, 3, 5)).astype(np.float32)
    W = g.uniform(-0.5, 0.5, (1, 4 * 6, 5)).astype(np.float32)
    R = g.uniform(-0.5, 0.5, (1, 4 * 6, 6)).astype(np.float32)
    h0 = g.uniform(-0.5, 0.5, (1, 3, 6)).astype(np.float32)
    Xio, h0io = oracle.narrow(X, io), oracle.narrow(h0, io)
    Y, Yh, Yc = oracle.rnn_io(io, "LSTM", "forward", 6, 5, Xio, W, R, initial_h=h0io)
    Y32, Yh32, Yc32 = oracle.rnn("LSTM", "forward", 6, 5, oracle.widen(Xio, io), W, R,
                                 initial_h=oracle.widen(h0io, io))
    ulp = 2.0 ** (-11 if io == "f16" else -8)
    for a, b in ((Y, Y32), (Yh, Yh32), (Yc, Yc32)):
        wa = oracle.widen(a, io)
        assert np.all(np.abs(wa - b) <= ulp * np.abs(b) + 1e-30)
        assert np.array_equal(np.asarray(a).view(np.uint16), np.asarray(oracle.narrow(b, io)).view(np.uint16))
