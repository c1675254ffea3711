"""Pins of the oracle's SwiGLU step (O8), from the mathematics of the gated
unit (Shazeer, "GLU Variants Improve Transformer", 2020: silu(g) * u with
silu(g) = g * sigmoid(g)), not from a retyped formula:
  - silu(g) - silu(-g) = g, since sigmoid(g) + sigmoid(-g) = 1 (catches a
    sign error on g);
  - silu(0) = 0, silu(g) -> g for large g and -> 0 for very negative g;
  - sigmoid(ln 3) = 3/4, so silu(ln 3) = 0.75 ln 3 (catches sigmoid(-g) in
    place of sigmoid(g), a plain sigmoid gate, and gate and up swapped);
  - h is linear in u: doubling u doubles h exactly;
  - the bf16 output is the fp64 value rounded once (the rounding itself is
    pinned with the other bf16 tests)."""
import math

import numpy as np

import oracle
from dit_convrot_linear_gb300 import synth


def test_silu_odd_part_is_the_identity():
    rng = np.random.default_rng(0)
    g = rng.normal(0, 3.0, 2000)
    one = np.ones_like(g)
    d = oracle.swiglu_f64(g, one) - oracle.swiglu_f64(-g, one)
    assert np.max(np.abs(d - g) / np.maximum(np.abs(g), 1e-300)) < 1e-14


def test_silu_special_values():
    g = np.array([0.0, math.log(3.0), 40.0, -40.0, 1e-8])
    h = oracle.swiglu_f64(g, np.ones_like(g))
    assert h[0] == 0.0
    assert abs(h[1] - 0.75 * math.log(3.0)) < 1e-15
    assert h[2] == 40.0                                   # e^-40 below half an ulp of 1
    assert abs(h[3]) < 1e-15
    # near 0, sigmoid(x) = 1/2 + x/4 + O(x^3)
    assert abs(h[4] - 1e-8 * (0.5 + 0.25e-8)) < 1e-23


def test_swiglu_is_linear_in_up():
    rng = np.random.default_rng(1)
    g = rng.normal(0, 2.0, 500)
    u = rng.normal(0, 2.0, 500)
    assert np.array_equal(oracle.swiglu_f64(g, 2.0 * u), 2.0 * oracle.swiglu_f64(g, u))


def test_swiglu_bf16_is_one_rounding_of_the_fp64_value():
    G = synth.tensor("oracle/swiglu/g", 5, 96, 1.5, 0.0, 1.0)
    U = synth.tensor("oracle/swiglu/u", 5, 96, 1.0, 0.0, 1.0)
    H = oracle.swiglu_bf16(G, U)
    ref = oracle.round_bf16(oracle.swiglu_f64(oracle.bf16_to_f64(G), oracle.bf16_to_f64(U)))
    assert np.array_equal(H, ref)


def test_swiglu_quant_act_is_the_rotation_of_h():
    G = synth.tensor("oracle/swiglu/g2", 3, 544, 1.5, 0.0, 1.0)
    U = synth.tensor("oracle/swiglu/u2", 3, 544, 1.0, 0.0, 1.0)
    q1, s1 = oracle.swiglu_quant_act(G, U)
    q2, s2 = oracle.rotate_quant_act(oracle.swiglu_bf16(G, U))
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2)
