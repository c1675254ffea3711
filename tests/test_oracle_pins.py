"""Pins of the CPU oracle against what the pages and mathematics fix.

None of these re-types the oracle's formula: each checks it against a separate
fact — an independent construction, a closed form, an invariant, a library
routine or brute force on tiny inputs.

The method (tensai docs, "画像生成" / Image generation, sections "チェックポイント
の入手" and "幅とメモリ"): rotate weights by a Hadamard matrix every 256 input
columns, quantise with one scale per row; the matrix is orthogonal, so rotating
the input the same way leaves the product unchanged.
"""
import fractions
import math
import os

import numpy as np
import pytest
import scipy.linalg

import oracle
from dit_convrot_linear_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits_of(values):
    """bf16 bits of values that are exactly representable in bf16."""
    f = np.asarray(values, dtype=np.float32)
    bits = f.view(np.uint32)
    assert np.all(bits & 0xFFFF == 0), "value not exact in bf16"
    return (bits >> 16).astype(np.uint16)


def butterfly_f64(v):
    """In-place fast Walsh-Hadamard butterfly (natural order), unnormalised."""
    v = np.array(v, dtype=np.float64)
    n = v.size
    h = 1
    while h < n:
        for i in range(0, n, 2 * h):
            a = v[i:i + h].copy()
            b = v[i + h:i + 2 * h].copy()
            v[i:i + h] = a + b
            v[i + h:i + 2 * h] = a - b
        h *= 2
    return v


# --------------------------------------------------------------- Hadamard

@pytest.mark.parametrize("n", [2, 4, 32, 64, 128, 256])
def test_sylvester_matches_scipy(n):
    # scipy.linalg.hadamard builds Sylvester's matrix by its own recursion.
    assert np.array_equal(oracle.sylvester(n), scipy.linalg.hadamard(n))


@pytest.mark.parametrize("n", [32, 64, 128, 256])
def test_sylvester_recursion_and_orthogonality(n):
    H = oracle.sylvester(n).astype(np.int64)
    half = oracle.sylvester(n // 2).astype(np.int64)
    assert np.array_equal(H, np.block([[half, half], [half, -half]]))
    assert np.array_equal(H, H.T)
    assert np.array_equal(H @ H.T, n * np.eye(n, dtype=np.int64))


def test_normalised_h256_is_exactly_orthogonal():
    c = oracle.hadamard_norm(256)
    assert c == 1.0 / 16.0
    H = oracle.sylvester(256).astype(np.float64) * c
    assert np.array_equal(H @ H.T, np.eye(256))


@pytest.mark.parametrize("n", [32, 64, 128])
def test_tail_norms(n):
    c = oracle.hadamard_norm(n)
    # the correctly rounded 1/sqrt(n): |c - 1/sqrt(n)| <= half an ulp of c,
    # checked in exact rational arithmetic (c^2 n - 1 changes sign across it)
    C = fractions.Fraction(c)
    half_ulp = fractions.Fraction(np.spacing(c)) / 2
    lo, hi = C - half_ulp, C + half_ulp
    assert lo * lo * n <= 1 <= hi * hi * n
    assert abs(c * c * n - 1.0) <= 2 * np.finfo(np.float64).eps
    H = oracle.sylvester(n).astype(np.float64) * c
    assert np.allclose(H @ H.T, np.eye(n), atol=4e-16, rtol=0)


def test_group_layout():
    assert [oracle.group_width(896, g) for g in (0, 256, 512, 768)] == [256, 256, 256, 128]
    assert oracle.group_width(4864, 4608) == 256
    assert oracle.group_width(32, 0) == 32
    for K in (256, 512, 896, 3072, 4096, 4864, 12288, 32, 64, 128, 288):
        assert oracle.valid_k(K)
    for K in (0, 16, 100, 200, 257, 300, 896 + 16):
        assert not oracle.valid_k(K)


# --------------------------------------------------------------- rotation

def test_rotation_of_unit_vectors_gives_columns():
    # H . e_j is column j of H: every entry is +-1/16.
    X = np.zeros((256, 256), dtype=np.float32)
    np.fill_diagonal(X, 1.0)
    R = oracle.rotate_rows(bf16_bits_of(X))
    H = scipy.linalg.hadamard(256) / 16.0
    assert np.array_equal(R, H.T)   # row j of R = H e_j = column j of H


def test_rotation_of_ones_is_16_e0():
    X = np.ones((1, 512), dtype=np.float32)
    R = oracle.rotate_rows(bf16_bits_of(X))
    expect = np.zeros(512)
    expect[0] = expect[256] = 16.0
    assert np.array_equal(R[0], expect)


def test_rotation_tail_group_uses_its_own_h():
    # K = 256 + 128: the tail of ones maps to sqrt(128) e_0 of the tail group.
    X = np.zeros((1, 384), dtype=np.float32)
    X[0, 256:] = 1.0
    R = oracle.rotate_rows(bf16_bits_of(X))[0]
    assert np.all(R[:256] == 0)
    assert abs(R[256] - math.sqrt(128)) < 1e-12
    assert np.all(np.abs(R[257:]) < 1e-12)


def test_explicit_product_equals_butterfly_exactly():
    # On bf16 data whose sums are exact in fp64, the explicit product (the
    # oracle) and an fp64 butterfly (written here) agree bit for bit.
    X = synth.tensor("pin/butterfly", 8, 896, 1.0, 0.01, 25.0)
    R = oracle.rotate_rows(X)
    V = synth.bf16_to_f32(X).astype(np.float64)
    for r in range(8):
        for g0 in (0, 256, 512, 768):
            n = oracle.group_width(896, g0)
            ref = butterfly_f64(V[r, g0:g0 + n]) * oracle.hadamard_norm(n)
            assert np.array_equal(R[r, g0:g0 + n], ref)


def test_rotation_honours_row_stride():
    X = synth.tensor("pin/stride", 5, 640, 1.0)
    R_full = oracle.rotate_rows(X[:, :512])
    R_view = oracle.rotate_rows(X, K=512)   # same rows read through ld = 640
    assert np.array_equal(R_full, R_view)


SHAPES = [(256, 512), (4864, 896), (896, 4864), (12288, 4096), (4096, 12288),
          (12288, 3072), (3072, 12288), (9216, 3072), (24576, 3072)]


@pytest.mark.parametrize("N,K", SHAPES)
def test_rotation_leaves_the_product_unchanged(N, K):
    # (W H)(H x) = W x in fp64 to 1e-10 relative: H is orthogonal and symmetric.
    rows = min(N, 64)
    W = synth.tensor(f"pin/inv/W{N}x{K}", rows, K, 0.02, 0.01, 20.0)
    X = synth.tensor(f"pin/inv/X{K}", 3, K, 1.0, 0.002, 40.0)
    plain = oracle.matmul_f64(synth.bf16_to_f32(X), synth.bf16_to_f32(W))
    rotated = oracle.matmul_f64(oracle.rotate_rows(X), oracle.rotate_rows(W))
    rel = np.linalg.norm(rotated - plain) / np.linalg.norm(plain)
    assert rel <= 1e-10


# --------------------------------------------------------------- quantiser

@pytest.mark.parametrize("qmax", [127, 7])
def test_quantiser_error_bound_and_range(qmax):
    V = oracle.rotate_rows(synth.tensor("pin/q", 64, 896, 0.02, 0.01, 20.0))
    codes, s = oracle.quantize_rows(V, qmax)
    assert codes.min() >= -qmax and codes.max() <= qmax
    assert np.all(np.abs(codes).max(axis=1) == qmax)   # every row reaches qmax
    s64 = np.broadcast_to(s.astype(np.float64)[:, None], V.shape)
    err = np.abs(V - codes.astype(np.float64) * s64)
    clamped = np.abs(codes) == qmax
    assert np.all(err[~clamped] <= s64[~clamped] / 2)
    # clamped entries stay within the fp32 rounding of the scale
    assert np.all(err[clamped] <= s64[clamped] * (0.5 + 1e-6))


def test_quantiser_scale_is_fp32_of_fp64_ratio():
    V = np.array([[-2.54, 1.0, 0.25, 0.0]])
    codes, s = oracle.quantize_rows(V, 127)
    assert s[0] == np.float32(2.54 / 127)
    expect = np.rint(V[0] / np.float64(s[0])).clip(-127, 127)
    assert np.array_equal(codes[0], expect.astype(np.int8))
    assert codes[0, 0] == -127


def test_quantiser_ties_to_even():
    # scale 1/64 exactly (amax = 127/64): codes of k + 1/2 round to even k.
    V = np.array([[127 / 64, 0.5 / 64, 1.5 / 64, 2.5 / 64, -0.5 / 64, -1.5 / 64]])
    codes, s = oracle.quantize_rows(V, 127)
    assert s[0] == np.float32(1 / 64)
    assert codes[0].tolist() == [127, 0, 2, 2, 0, -2]


def test_zero_row():
    codes, s = oracle.quantize_rows(np.zeros((2, 256)), 127)
    assert np.all(codes == 0) and np.all(s == 0)


def test_hadamard_rows_closed_form():
    # W row n = row n of Hs_256 => W' = 16 e_n => code 127 at n, 0 elsewhere;
    # x = ones => x' = 16 e_0 => acc = 127 * 127 at n = 0, else 0.
    fixture = open(os.path.join(GOLDEN, "hadamard_rows_closed_form.txt")).read()
    expect = dict(line.split("=", 1) for line in fixture.splitlines()
                  if "=" in line and not line.startswith("#"))
    H = scipy.linalg.hadamard(256).astype(np.float32)
    Wq, sw = oracle.quantize_weights(bf16_bits_of(H[:4]), 8)
    Xq, sx = oracle.rotate_quant_act(bf16_bits_of(np.ones((2, 256), np.float32)))
    assert np.all(sw == np.float32(float(expect["weight_scale"])))
    assert np.all(sx == np.float32(float(expect["act_scale"])))
    want_w = np.zeros((4, 256), np.int8)
    want_w[np.arange(4), np.arange(4)] = int(expect["weight_code_diag"])
    assert np.array_equal(Wq, want_w)
    want_x = np.zeros((2, 256), np.int8)
    want_x[:, 0] = int(expect["act_code_0"])
    assert np.array_equal(Xq, want_x)
    acc, Y = oracle.linear_a8(Xq, sx, Wq, sw)
    assert acc[:, 0].tolist() == [int(expect["acc_n0"])] * 2
    assert np.all(acc[:, 1:] == 0)
    assert abs(Y[0, 0] - float(expect["y_n0_approx"])) < 1e-3


# --------------------------------------------------------------- int4 packing

def test_int4_pack_layout():
    codes = np.array([[1, -1, 7, -7, 0, -8]], dtype=np.int8)
    packed = oracle.pack_int4(codes)
    assert packed.tolist() == [[0xF1, 0x97, 0x80]]
    assert np.array_equal(oracle.unpack_int4(packed, 6), codes)


def test_int4_weights_round_trip():
    W = synth.tensor("pin/w4", 16, 512, 0.015, 0.005, 30.0)
    packed, s4 = oracle.quantize_weights(W, 4)
    codes = oracle.unpack_int4(packed, 512)
    assert codes.min() >= -7 and codes.max() <= 7
    ref_codes, ref_s = oracle.quantize_rows(oracle.rotate_rows(W), 7)
    assert np.array_equal(codes, ref_codes) and np.array_equal(s4, ref_s)


# --------------------------------------------------------------- products

def test_a8_product_brute_force():
    rng = np.random.default_rng(1)
    Xq = rng.integers(-127, 128, size=(2, 256), dtype=np.int8)
    Wq = rng.integers(-127, 128, size=(4, 256), dtype=np.int8)
    sx = np.array([0.5, 0.25], np.float32)
    sw = np.array([1.0, 2.0, 0.125, 3.0], np.float32)
    acc, Y = oracle.linear_a8(Xq, sx, Wq, sw)
    for m in range(2):
        for n in range(4):
            s = sum(int(Xq[m, k]) * int(Wq[n, k]) for k in range(256))
            assert acc[m, n] == s
            assert Y[m, n] == float(sx[m]) * float(sw[n]) * s


def test_a8_extreme_accumulator_fits_int32():
    K = 12288
    Xq = np.full((1, K), 127, np.int8)
    Wq = np.full((1, K), -127, np.int8)
    acc, _ = oracle.linear_a8(Xq, np.ones(1, np.float32), Wq, np.ones(1, np.float32))
    assert acc[0, 0] == -127 * 127 * K


def test_a16_product_brute_force():
    X = synth.tensor("pin/a16x", 3, 288, 1.0)
    Xr = oracle.rotate_act_bf16(X)
    Wq = np.random.default_rng(2).integers(-7, 8, size=(5, 288), dtype=np.int8)
    sw = np.linspace(0.1, 0.5, 5).astype(np.float32)
    Y = oracle.linear_a16(Xr, Wq, sw)
    xf = oracle.bf16_to_f64(Xr)
    for m in range(3):
        for n in range(5):
            ref = float(sw[n]) * math.fsum(float(Wq[n, k]) * xf[m, k] for k in range(288))
            assert abs(Y[m, n] - ref) <= 1e-12 * max(1.0, abs(ref))


def test_pairs_match_dense():
    X = synth.tensor("pin/pairs/x", 6, 512, 1.0, 0.002, 40.0)
    W = synth.tensor("pin/pairs/w", 40, 512, 0.02, 0.01, 20.0)
    Wq, sw = oracle.quantize_weights(W, 8)
    Xq, sx = oracle.rotate_quant_act(X)
    acc, Y = oracle.linear_a8(Xq, sx, Wq, sw)
    pm = np.array([0, 5, 3, 2]); pn = np.array([39, 0, 17, 2])
    acc_p, Y_p = oracle.linear_a8_pairs(Xq, sx, Wq, sw, pm, pn)
    assert np.array_equal(acc_p, acc[pm, pn]) and np.array_equal(Y_p, Y[pm, pn])
    Xr = oracle.rotate_act_bf16(X)
    Ya = oracle.linear_a16(Xr, Wq, sw)
    assert np.array_equal(oracle.linear_a16_pairs(Xr, Wq, sw, pm, pn), Ya[pm, pn])


# --------------------------------------------------------------- bf16 rounding

def test_bf16_rounding_matches_exact_nearest():
    # brute force against exact rational arithmetic on random doubles
    rng = np.random.default_rng(3)
    vals = np.concatenate([rng.normal(size=400) * 10.0 ** rng.integers(-30, 30, 400),
                           [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8),
                            1.0 + 2 ** -8 + 2 ** -40, 2.0 ** -133 * 1.5, 3.0e38]])
    for v in vals:
        b = oracle.f64_to_bf16(v)
        got = oracle.bf16_to_f64(np.array([b], np.uint16))[0]
        # neighbours of the result in bf16
        lo = oracle.bf16_to_f64(np.array([b - 1 if b & 0x7FFF else b], np.uint16))[0]
        hi = oracle.bf16_to_f64(np.array([b + 1], np.uint16))[0]
        fv, fg = fractions.Fraction(v), fractions.Fraction(got)
        for nb in (lo, hi):
            if math.isfinite(nb) and nb != got:
                d_nb, d_g = abs(fractions.Fraction(nb) - fv), abs(fg - fv)
                assert d_g < d_nb or (d_g == d_nb and (b & 1) == 0), (v, got, nb)


def test_bf16_rounding_matches_torch_on_fp32_values():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(4)
    f = (rng.normal(size=2000) * 100).astype(np.float32)
    ours = oracle.round_bf16(f.astype(np.float64))
    theirs = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, theirs)


# --------------------------------------------------------------- properties

def test_rotation_reduces_quantisation_error_with_outliers():
    # The few outlier columns that set a row's scale get spread over their
    # group (tensai docs, section "幅とメモリ"): the dequantisation error of
    # rotated 8-bit and 4-bit weights, measured in the original basis, is below
    # that of the same weights quantised without rotation.
    W = synth.tensor("pin/spread", 128, 896, 0.02, 0.01, 20.0)
    V = synth.bf16_to_f32(W).astype(np.float64)
    H = {n: scipy.linalg.hadamard(n) / math.sqrt(n) for n in (256, 128)}
    for qmax in (127, 7):
        c0, s0 = oracle.quantize_rows(V, qmax)
        plain_err = np.linalg.norm(V - c0 * s0[:, None].astype(np.float64))
        R = oracle.rotate_rows(W)
        c1, s1 = oracle.quantize_rows(R, qmax)
        D = c1 * s1[:, None].astype(np.float64)
        back = np.concatenate([D[:, g:g + w] @ H[w] for g, w in
                               ((0, 256), (256, 256), (512, 256), (768, 128))], axis=1)
        rot_err = np.linalg.norm(V - back)
        assert rot_err < plain_err


def test_oracle_is_deterministic():
    W = synth.tensor("pin/det", 32, 896, 0.02, 0.01, 20.0)
    a = oracle.quantize_weights(W, 8)
    b = oracle.quantize_weights(W, 8)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
