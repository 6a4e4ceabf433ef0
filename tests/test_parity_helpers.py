"""CPU checks of the parity tests' own reference helpers (tests/gpu_util.py).

The GPU tests hold decode output rows to the oracle's single-token steps with
the conv output and the rule's output rounded to the activation dtype.  That
reference is composed here from the oracle's functions; with no rounding it
must be the oracle's own layer step exactly, and its rounding must be
round-to-nearest-even onto the dtype's values.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import oracle_step_in_activation_dtype, rounded_to


@pytest.fixture(scope="module", autouse=True)
def _oracle_built():
    oracle.build()


@pytest.mark.parametrize("shape", [W.TINY, W.GDNShape(H_k=1, H_v=3, d_k=32, d_v=32)], ids=["tiny", "r3"])
def test_composed_step_without_rounding_is_the_oracle_step(shape):
    B = 3
    dec = W.decode_inputs(shape, torch.float32, B, 2, seed=71)
    p = W.layer_inputs(shape, torch.float32, [4] * B, seed=72, init_state=True)
    f = W.to_f64
    S, cs = f(p["S0"]), f(p["conv_state0"])
    S2, cs2 = S, cs
    for t in range(2):
        step = (f(dec["qkv"][t]), f(dec["z"][t]), f(dec["a"][t]), f(dec["b"][t]), f(p["conv_w"]),
                f(p["A_log"]), f(p["dt_bias"]), f(p["norm_w"]))
        out, S, cs, _ = oracle.layer_decode_step(*step, shape.H_k, shape.H_v, shape.d_k, shape.d_v, S, cs)
        out2, S2, cs2 = oracle_step_in_activation_dtype(*step, shape, S2, cs2, lambda x: x)
        assert np.array_equal(out, out2) and np.array_equal(S, S2) and np.array_equal(cs, cs2)


def test_composed_step_rounds_the_activations():
    # with bf16 rounding the step differs from the exact one, but only by
    # about the rounding of y and o (a few 1e-3 relative, not more)
    shape = W.GDNShape(H_k=1, H_v=2, d_k=32, d_v=32)
    dec = W.decode_inputs(shape, torch.float32, 4, 1, seed=73)
    p = W.layer_inputs(shape, torch.float32, [4] * 4, seed=74, init_state=True)
    f = W.to_f64
    step = (f(dec["qkv"][0]), f(dec["z"][0]), f(dec["a"][0]), f(dec["b"][0]), f(p["conv_w"]),
            f(p["A_log"]), f(p["dt_bias"]), f(p["norm_w"]))
    S, cs = f(p["S0"]), f(p["conv_state0"])
    exact, _, _, _ = oracle.layer_decode_step(*step, shape.H_k, shape.H_v, shape.d_k, shape.d_v, S, cs)
    rounded, _, _ = oracle_step_in_activation_dtype(*step, shape, S, cs, rounded_to(torch.bfloat16))
    e = np.linalg.norm(rounded - exact) / np.linalg.norm(exact)
    assert 1e-4 < e < 2e-2


def test_rounded_to_bf16_is_nearest_even():
    r = rounded_to(torch.bfloat16)
    ulp = 2.0 ** -7  # bf16 spacing in [1, 2); 2 ulp in [2, 4)
    x = np.array([1.0, 1.0 + ulp / 2, 1.0 + 3 * ulp / 2, 1.0 + ulp / 4, -3.0 - 1.5 * ulp, -3.0 - 0.75 * ulp])
    want = np.array([1.0, 1.0, 1.0 + 2 * ulp, 1.0, -3.0 - 2 * ulp, -3.0])
    assert np.array_equal(r(x), want)
