"""Pins of the oracle's block-scaled weights (O9) and their A16 product (O10).

Block scales are the GGML formats' shared scale per block (Q8_0 and Q4_0,
32 wide) and kvad's own q8 with an fp32 scale per 32 weights (kvad-gpu
internals, "Quantised weights on the GPU"); on the rotated weights they are
the way back to 4-bit accuracy, which the rotation alone improves less than
8-bit's (tensai docs, "画像生成" / Image generation, section "幅とメモリ").

Each pin checks the oracle against a separate fact: the per-row quantiser as
the one-block special case, brute force with exact summation, a dense fp64
matmul of the dequantised weights, per-element error bounds, blocks of wildly
different magnitude, and the distance to the unquantised product.
"""
import math

import numpy as np
import pytest
import scipy.linalg

import oracle
from dit_convrot_linear_gb300 import synth

WD = (0.02, 0.01, 20.0)     # decode weights: N(0, 0.02), 1% columns x20


def dequant(codes, scales, G):
    """codes [R, K] times each column's block scale, fp64."""
    return codes.astype(np.float64) * np.repeat(scales.astype(np.float64), G, axis=1)


def test_one_block_per_row_is_the_per_row_quantiser():
    V = oracle.rotate_rows(synth.tensor("pinb/one", 16, 512, *WD))
    for qmax in (127, 7):
        cb, sb = oracle.quantize_blocks(V, qmax, 512)
        cr, sr = oracle.quantize_rows(V, qmax)
        assert np.array_equal(cb, cr) and np.array_equal(sb[:, 0], sr)


@pytest.mark.parametrize("qmax,G", [(127, 32), (7, 32), (7, 64), (127, 256)])
def test_block_quantiser_error_bound_range_and_scale(qmax, G):
    V = oracle.rotate_rows(synth.tensor(f"pinb/q{qmax}_{G}", 24, 1024, *WD))
    codes, s = oracle.quantize_blocks(V, qmax, G)
    assert s.shape == (24, 1024 // G)
    blocks = np.abs(V).reshape(24, 1024 // G, G)
    amax = blocks.max(axis=2)
    assert np.array_equal(s, (amax / qmax).astype(np.float32))
    cb = np.abs(codes.astype(np.int64)).reshape(24, 1024 // G, G)
    assert np.all(cb.max(axis=2) == qmax)                 # every block reaches qmax
    s64 = np.repeat(s.astype(np.float64), G, axis=1)
    err = np.abs(V - codes * s64)
    assert np.all(err <= s64 * (0.5 + 1e-6))


def test_blocks_scale_independently():
    # Block b of the row holds values of magnitude 10^(b - 6): with one scale
    # per row every block but the last would round to zero; with a scale per
    # block each reaches qmax and is reproduced to s_b / 2.
    rng = np.random.default_rng(11)
    nb, G = 10, 32
    V = np.concatenate([10.0 ** (b - 6) * rng.uniform(-1, 1, G) for b in range(nb)])[None, :]
    codes, s = oracle.quantize_blocks(V, 127, G)
    for b in range(nb):
        blk = slice(b * G, (b + 1) * G)
        assert s[0, b] == np.float32(np.abs(V[0, blk]).max() / 127)
        assert np.abs(codes[0, blk]).max() == 127
        assert np.all(np.abs(V[0, blk] - codes[0, blk] * np.float64(s[0, b])) <= np.float64(s[0, b]) * 0.5000001)


def test_block_quantiser_ties_to_even_in_a_later_block():
    # block 0: scale 1/8 (amax 127/8); block 1: scale 1/64 exactly with the
    # half-integer multiples of it rounding to even codes.
    b0 = np.full(32, 127 / 8.0)
    b1 = np.zeros(32)
    b1[:6] = [127 / 64, 0.5 / 64, 1.5 / 64, 2.5 / 64, -0.5 / 64, -1.5 / 64]
    codes, s = oracle.quantize_blocks(np.concatenate([b0, b1])[None, :], 127, 32)
    assert s[0, 0] == np.float32(1 / 8) and s[0, 1] == np.float32(1 / 64)
    assert np.all(codes[0, :32] == 127)
    assert codes[0, 32:38].tolist() == [127, 0, 2, 2, 0, -2]


def test_zero_block_has_zero_scale_and_codes():
    V = np.zeros((1, 96))
    V[0, 40] = 1.0
    codes, s = oracle.quantize_blocks(V, 7, 32)
    assert s[0, 0] == 0 and s[0, 2] == 0 and s[0, 1] == np.float32(1 / 7)
    assert np.all(codes[0, :32] == 0) and np.all(codes[0, 64:] == 0) and codes[0, 40] == 7


def test_block_width_must_divide_k():
    with pytest.raises(ValueError):
        oracle.quantize_blocks(np.zeros((1, 96)), 127, 64)


def test_blocked_product_brute_force():
    rng = np.random.default_rng(12)
    M, N, K, G = 2, 3, 128, 32
    X = synth.tensor("pinb/bfx", M, K, 1.0)
    Wq = rng.integers(-127, 128, size=(N, K), dtype=np.int8)
    sw = rng.uniform(0.001, 0.1, size=(N, K // G)).astype(np.float32)
    Y = oracle.linear_a16_blocked(X, Wq, sw, G)
    xf = oracle.bf16_to_f64(X)
    for m in range(M):
        for n in range(N):
            ref = math.fsum(float(sw[n, k // G]) * float(Wq[n, k]) * xf[m, k] for k in range(K))
            assert abs(Y[m, n] - ref) <= 1e-12 * max(1.0, abs(ref))


@pytest.mark.parametrize("rotate", [True, False])
def test_blocked_product_equals_dense_dequantised_matmul(rotate):
    W = synth.tensor("pinb/dd/w", 64, 1024, *WD)
    X = synth.tensor("pinb/dd/x", 4, 1024, 1.0, 0.002, 40.0)
    for bits, G in ((8, 32), (4, 64)):
        Wq, sw = oracle.quantize_weights_blocked(W, bits, G, rotate)
        c = oracle.weight_codes(Wq, bits, 1024)
        Xa = oracle.rotate_act_bf16(X) if rotate else X
        Y = oracle.linear_a16_blocked(Xa, c, sw, G)
        ref = oracle.bf16_to_f64(Xa) @ dequant(c, sw, G).T
        assert np.max(np.abs(Y - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_uniform_block_scales_reduce_to_the_per_row_product():
    X = oracle.rotate_act_bf16(synth.tensor("pinb/u/x", 3, 512, 1.0))
    rng = np.random.default_rng(13)
    Wq = rng.integers(-7, 8, size=(5, 512), dtype=np.int8)
    sw = np.linspace(0.01, 0.05, 5).astype(np.float32)
    Yb = oracle.linear_a16_blocked(X, Wq, np.repeat(sw[:, None], 512 // 32, axis=1), 32)
    Yr = oracle.linear_a16(X, Wq, sw)
    assert np.max(np.abs(Yb - Yr)) <= 1e-12 * np.max(np.abs(Yr))


def test_rotated_blocked_product_is_within_the_quantisation_bound():
    # X W^T = (X H)(W H)^T; the blocked product differs from it by the weight
    # rounding (at most s_b / 2 per code, times |x''|) and the bf16 rounding
    # of x' (at most 2^-9 |x'| per element, times |v|).
    W = synth.tensor("pinb/bd/w", 48, 896, *WD)
    X = synth.tensor("pinb/bd/x", 3, 896, 1.0, 0.002, 40.0)
    exact = oracle.matmul_f64(synth.bf16_to_f32(X), synth.bf16_to_f32(W))
    Xr = oracle.rotate_rows(X)
    V = oracle.rotate_rows(W)
    xb = oracle.bf16_to_f64(oracle.round_bf16(Xr))
    for bits, G in ((8, 32), (4, 32), (4, 128)):
        Wq, sw = oracle.quantize_weights_blocked(W, bits, G)
        Y = oracle.linear_blocked(X, W, bits, G)
        s64 = np.repeat(sw.astype(np.float64), G, axis=1)
        bound = (np.abs(xb) @ (s64 / 2).T + 2.0 ** -9 * (np.abs(Xr) @ np.abs(V).T)
                 + 1e-9 * np.abs(exact).max())
        assert np.all(np.abs(Y - exact) <= bound)
        # and the bound is not vacuous: the error uses a fair share of it
        assert np.abs(Y - exact).max() >= 1e-3 * bound.max()


def test_group_scales_recover_4_bit_accuracy():
    # On weights with outlier columns (the decode workload's), per-block
    # scales on the rotated weights cut the 4-bit error, measured in the
    # original basis, below the per-row scale's, and smaller blocks cut it
    # further; the unrotated 32-wide 8-bit blocks beat one unrotated scale
    # per row.
    W = synth.tensor("pinb/acc", 128, 896, *WD)
    V0 = synth.bf16_to_f32(W).astype(np.float64)
    H = {n: scipy.linalg.hadamard(n) / math.sqrt(n) for n in (256, 128)}

    def back(D):
        return np.concatenate([D[:, g:g + w] @ H[w] for g, w in
                               ((0, 256), (256, 256), (512, 256), (768, 128))], axis=1)

    R = oracle.rotate_rows(W)
    c, s = oracle.quantize_rows(R, 7)
    row_err = np.linalg.norm(V0 - back(c * s[:, None].astype(np.float64)))
    errs = {}
    for G in (128, 64, 32):
        cb, sb = oracle.quantize_blocks(R, 7, G)
        errs[G] = np.linalg.norm(V0 - back(dequant(cb, sb, G)))
    assert errs[128] < row_err and errs[64] < errs[128] and errs[32] < errs[64]
    assert errs[32] < 0.8 * row_err
    c8, s8 = oracle.quantize_rows(V0, 127)
    cq, sq = oracle.quantize_blocks(V0, 127, 32)
    assert (np.linalg.norm(V0 - dequant(cq, sq, 32))
            < np.linalg.norm(V0 - c8 * s8[:, None].astype(np.float64)))
