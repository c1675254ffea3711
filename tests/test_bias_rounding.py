"""The rounding argument behind the bf16 bar of the products that sum the
weight codes with their bias (the grouped decode product and the split-K
product): they add (q + B) x' in fp32, B = 8 for int4 and 128 for int8 codes,
and take off B times the sum of x' at the end.  The pages fix fp32 sums, not
their order or form, so the bar is the exact value's bf16 step or, for
outputs near zero, 2^-20 of sum_k |q_k + B| |x'_k|.

This CPU test emulates that arithmetic with numpy float32 (products exact in
fp32; partial sums of 16 products, as one MMA step, then a running fp32 sum
over the steps; the bias term taken off with one rounding) on the shapes and
value distributions of the GPU tests, and checks that its error against the
exact sum stays well inside the bar, while one wrong code would not."""
import numpy as np
import pytest

from dit_convrot_linear_gb300 import synth

pytestmark = pytest.mark.filterwarnings("ignore")


def _codes(rng, n, k, bits):
    qmax = 7 if bits == 4 else 127
    w = rng.normal(0.0, 1.0, (n, k))
    s = np.abs(w).max(axis=1, keepdims=True) / qmax
    return np.clip(np.rint(w / s), -qmax - (1 if bits == 4 else 0), qmax).astype(np.int64)


def _biased_sum_f32(q, x, B):
    """fp32 emulation: 16-term partial sums (one MMA's k16), a running fp32
    sum over them, then fma(sum, 1, -B * S) with S the fp32 sum of x."""
    n, k = q.shape
    terms = ((q + B).astype(np.float32) * x.astype(np.float32)[None, :])      # exact products
    acc = np.zeros(n, dtype=np.float32)
    for k0 in range(0, k, 16):
        part = np.zeros(n, dtype=np.float32)
        for j in range(k0, min(k0 + 16, k)):
            part = (part + terms[:, j]).astype(np.float32)
        acc = (acc + part).astype(np.float32)
    S = np.float32(0.0)
    for v in x.astype(np.float32):
        S = np.float32(S + v)
    return (acc.astype(np.float64) - np.float64(np.float32(B * S))).astype(np.float32)


@pytest.mark.parametrize("bits,n,k", [(4, 512, 896), (4, 256, 4864), (8, 512, 896), (8, 256, 4864)])
def test_biased_fp32_sums_stay_inside_the_bar(bits, n, k):
    rng = np.random.default_rng(bits * 1000 + k)
    q = _codes(rng, n, k, bits)
    # x' as the A16 operand: bf16-valued, N(0, 1) with a few outlier columns
    x = synth.tensor(f"cpu/bias/x{k}", 1, k, 1.0, 0.005, 30.0)[0]
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    B = 8 if bits == 4 else 128
    exact = q.astype(np.float64) @ xf
    got = _biased_sum_f32(q, xf, B).astype(np.float64)
    mag = np.abs(q + B).astype(np.float64) @ np.abs(xf)
    err = np.abs(got - exact)
    # well inside the bar (2^-20 of the magnitude), by at least 4x
    assert np.all(err <= 2.0 ** -22 * mag)
    # while a single wrong code (off by one at the largest |x'|) moves the
    # sum by far more than the bar allows, so the bar still catches it
    assert np.abs(xf).max() > 100 * (2.0 ** -20 * mag).max()
