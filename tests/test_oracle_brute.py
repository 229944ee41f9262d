"""Oracle vs a straight-line float64 re-derivation on tiny random shapes
covering op x direction x layout x lbr x input_forget x clip x activations x
sequence_lens x optional inputs.  Agreement within fp32 rounding pins the
wiring (indices, gate and bias order, peephole placement, directions, layouts,
masking) independently of the oracle's code."""
import numpy as np
import pytest

from brute64 import run as brute
from onnx_recurrent_gb300.synth import random_case
from helpers import oracle_case


@pytest.mark.parametrize("seed", range(60))
def test_oracle_matches_float64_brute_force(seed):
    c = random_case(seed, max_seq=3, max_batch=3, max_input=4, max_hidden=4)
    Y, Yh, Yc = oracle_case(c)
    rY, rYh, rYc = brute(c)
    tol = 2e-5 * max(1.0, float(np.abs(rY).max(initial=0)), float(np.abs(rYh).max(initial=0)))
    np.testing.assert_allclose(Y, rY, rtol=0, atol=tol)
    np.testing.assert_allclose(Yh, rYh, rtol=0, atol=tol)
    if Yc is not None:
        ctol = 2e-5 * max(1.0, float(np.abs(rYc).max(initial=0)))
        np.testing.assert_allclose(Yc, rYc, rtol=0, atol=ctol)
