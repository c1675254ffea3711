"""Pins of the oracle's modulated layer norm (O11), from the mathematics of a
layer norm and of the adaptive modulation LN(x) (1 + scale) + shift (Peebles
and Xie, "Scalable Diffusion Models with Transformers", 2023), and from an
independent library routine, not from a retyped formula:
  - a worked row: x = (0, 2, 4, 6) has mean 3 and biased variance 5 (by
    hand), so h = (-3, -1, 1, 3) / sqrt(5 + eps) (catches the unbiased
    variance, eps outside the square root, the mean not subtracted);
  - with no modulation, h equals torch's layer_norm in fp64 (a library
    routine with its own code), and its bf16 rounding bit for bit;
  - with no modulation and eps = 0, every row has mean 0 and mean square 1,
    and h is unchanged by x -> a x + b (a > 0) and negated by x -> -x;
  - scale = -1 gives h = shift exactly, whatever x (catches x * scale + shift
    and shift and scale swapped); scale = c, shift = 0 gives (1 + c) LN(x);
  - a constant row has h = shift exactly (no division by a zero variance);
  - the bf16 output is the fp64 value rounded once, and the fused operand is
    the rotation and quantisation of that bf16 row."""
import math

import numpy as np
import pytest

import oracle
from dit_convrot_linear_gb300 import synth


def _zeros(K):
    return np.zeros(K, dtype=np.float32)


def test_worked_row():
    x = np.array([[0.0, 2.0, 4.0, 6.0]])
    for eps in (0.0, 1.0, 0.25):
        h = oracle.modnorm_f64(x, np.zeros(4), np.zeros(4), eps)[0]
        ref = np.array([-3.0, -1.0, 1.0, 3.0]) / math.sqrt(5.0 + eps)
        assert np.max(np.abs(h - ref)) < 1e-15


def test_matches_torch_layer_norm():
    torch = pytest.importorskip("torch")
    for K, eps in ((512, 1e-6), (3072, 1e-6), (4096 + 32, 1e-5)):
        X = synth.tensor(f"oracle/modnorm/ln{K}", 6, K, 1.0, 0.002, 40.0)
        xf = oracle.bf16_to_f64(X)
        ref = torch.nn.functional.layer_norm(torch.from_numpy(xf), (K,), eps=eps).numpy()
        h = oracle.modnorm_f64(xf, np.zeros(K), np.zeros(K), eps)
        assert np.max(np.abs(h - ref)) < 1e-12
        H = oracle.modnorm_bf16(X, _zeros(K), _zeros(K), np.float32(eps))
        # eps travels as fp32: the routine gets the same value
        ref32 = torch.nn.functional.layer_norm(torch.from_numpy(xf), (K,),
                                               eps=float(np.float32(eps))).numpy()
        assert np.array_equal(H, oracle.round_bf16(ref32))


def test_moments_and_invariances():
    X = synth.tensor("oracle/modnorm/mom", 5, 768, 2.0, 0.01, 10.0)
    x = oracle.bf16_to_f64(X)
    z = np.zeros(768)
    h = oracle.modnorm_f64(x, z, z, 0.0)
    assert np.max(np.abs(h.mean(axis=1))) < 1e-14
    assert np.max(np.abs((h * h).mean(axis=1) - 1.0)) < 1e-13
    h2 = oracle.modnorm_f64(3.5 * x + 100.0, z, z, 0.0)
    assert np.max(np.abs(h2 - h)) < 1e-11
    h3 = oracle.modnorm_f64(-x, z, z, 0.0)
    assert np.max(np.abs(h3 + h)) < 1e-14


def test_modulation_special_values():
    K = 544
    X = synth.tensor("oracle/modnorm/mod", 4, K, 1.0, 0.0, 1.0)
    x = oracle.bf16_to_f64(X)
    rng = np.random.default_rng(3)
    shift = rng.normal(0.0, 0.5, K)
    z = np.zeros(K)
    # scale = -1: the norm is multiplied by zero, so h is the shift exactly
    h = oracle.modnorm_f64(x, shift, -np.ones(K), 1e-6)
    assert np.array_equal(h, np.broadcast_to(shift, h.shape))
    # scale = c, shift = 0: (1 + c) LN(x); shift alone adds to every row
    ln = oracle.modnorm_f64(x, z, z, 1e-6)
    c = rng.uniform(-0.5, 0.5, K)
    assert np.max(np.abs(oracle.modnorm_f64(x, z, c, 1e-6) - (1.0 + c) * ln)) < 1e-14
    assert np.max(np.abs(oracle.modnorm_f64(x, shift, z, 1e-6) - (ln + shift))) < 1e-14


def test_constant_row_gives_the_shift():
    K = 256
    rng = np.random.default_rng(4)
    shift = rng.normal(0.0, 0.5, K).astype(np.float32)
    scale = rng.normal(0.0, 0.5, K).astype(np.float32)
    X = np.full((3, K), oracle.f64_to_bf16(1.375), dtype=np.uint16)
    X[1] = 0
    X[2] = oracle.f64_to_bf16(-96.0)
    H = oracle.modnorm_bf16(X, shift, scale, np.float32(1e-6))
    assert np.array_equal(H, np.tile(oracle.round_bf16(shift.astype(np.float64)), (3, 1)))


def test_bf16_is_one_rounding_of_the_fp64_value():
    K = 896
    X = synth.tensor("oracle/modnorm/b16", 4, K, 1.0, 0.01, 20.0)
    rng = np.random.default_rng(5)
    shift = rng.normal(0.0, 0.5, K).astype(np.float32)
    scale = rng.normal(0.0, 0.3, K).astype(np.float32)
    H = oracle.modnorm_bf16(X, shift, scale, np.float32(1e-6))
    ref = oracle.round_bf16(oracle.modnorm_f64(oracle.bf16_to_f64(X), shift.astype(np.float64),
                                               scale.astype(np.float64), float(np.float32(1e-6))))
    assert np.array_equal(H, ref)


def test_modnorm_quant_act_is_the_rotation_of_h():
    K = 3072 + 64
    X = synth.tensor("oracle/modnorm/q", 3, K, 1.0, 0.002, 40.0)
    rng = np.random.default_rng(6)
    shift = rng.normal(0.0, 0.5, K).astype(np.float32)
    scale = rng.normal(0.0, 0.3, K).astype(np.float32)
    q1, s1 = oracle.modnorm_quant_act(X, shift, scale, 1e-6)
    q2, s2 = oracle.rotate_quant_act(oracle.modnorm_bf16(X, shift, scale, 1e-6))
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2)
