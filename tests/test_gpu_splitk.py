"""GPU parity of the split-K A16 product (tq_linear in mode W4A16 / W8A16 for
up to 16 token rows over a matrix of at least 2^24 weights): clusters of CTAs
along K, each CTA rotating its own run of the input's groups, codes widened
with their bias into fp16 subnormals, mma.sync with the tokens as the N side,
partial sums added over the cluster in rank order.

Shapes: the batched-decode projections of an 8B-class model (K = 4096 ->
N = 12288 and K = 12288 -> N = 4096; kvad-gpu internals, "Numbers") at 1, 8
and 16 tokens in full, and ragged ones: N not a multiple of the 256-row tile,
K with a partial last group (tails of 32, 64 and 128), runs of groups that do
not divide evenly over a cluster, 8- and 4-bit weights.

Bars: fp32 Y within relative L2 1e-4 of the oracle's O6 on the GPU's own bf16
rotation and on the oracle's rotation; bf16 Y within one bf16 step of the
exact value, or, for outputs near zero, within the rounding of fp32 sums of
the biased terms (2^-20 of sw sum_k |q + B| |x'_k|, B = 8 or 128: the
product sums the codes plus their bias and takes off B times the sum of x');
the same bytes on every run.
"""
import numpy as np
import pytest

import oracle
from dit_convrot_linear_gb300 import synth
from helpers import REL_L2_Y, bf16_bits, bf16_ulp_diff, rel_l2, to_dev_bf16, to_np

pytestmark = pytest.mark.gpu

WB = (0.015, 0.005, 30.0)   # batched-decode weights: N(0, 0.015), 0.5% columns x30


def _setup(tq, M, N, K, bits, tag, xd=(1.0, 0.0, 1.0)):
    W = synth.tensor(f"gpu/splitk/{tag}/w{N}x{K}", N, K, *WB)
    Xb = synth.tensor(f"gpu/splitk/{tag}/x{M}x{K}", M, K, *xd)
    codes, sw = tq.quantize_weights(to_dev_bf16(W), bits)
    c = to_np(codes)
    wc = oracle.weight_codes(c.view(np.int8) if bits == 8 else c.view(np.uint8), bits, K)
    return Xb, to_dev_bf16(Xb), codes, sw, wc


def _bf16_close(got_bits, xr, wc, sw, bits):
    ref = oracle.linear_a16(xr, wc, sw)
    B = 8.0 if bits == 4 else 128.0
    one_ulp = bf16_ulp_diff(got_bits, oracle.round_bf16(ref)) <= 1
    mag = (np.abs(oracle.bf16_to_f64(xr)) @ np.abs(wc.astype(np.float64) + B).T) * sw.astype(np.float64)[None, :]
    a = np.abs(ref)
    step = np.exp2(np.floor(np.log2(np.where(a > 0, a, 2.0 ** -133))) - 7)
    near = np.abs(oracle.bf16_to_f64(got_bits) - ref) <= step + 2.0 ** -20 * mag
    return bool(np.all(one_ulp | near)), float(one_ulp.mean())


@pytest.mark.parametrize("M", [1, 8, 16])
@pytest.mark.parametrize("N,K", [(12288, 4096), (4096, 12288)])
def test_splitk_full_size(tq, M, N, K):
    Xb, X, codes, sw, wc = _setup(tq, M, N, K, 4, "full")
    Y = to_np(tq.linear(X, codes, sw, N, 4, "W4A16"))
    assert tq.device_status() == 0
    ref = oracle.linear_a16(bf16_bits(tq.rotate_act_bf16(X)), wc, to_np(sw))
    assert rel_l2(Y, ref) <= REL_L2_Y
    assert rel_l2(Y, oracle.linear_a16(oracle.rotate_act_bf16(Xb), wc, to_np(sw))) <= REL_L2_Y
    # every row of every token: no tile, run or cluster share left out
    assert np.all(np.isfinite(Y))
    rows = np.linalg.norm(Y - ref, axis=1) / np.linalg.norm(ref, axis=1)
    assert rows.max() <= 4 * REL_L2_Y


@pytest.mark.parametrize("M,N,K,bits", [
    (5, 4096 + 77, 4096 + 32, 4),    # ragged rows (a partial last tile), K tail of 32
    (3, 6000, 4096 + 64, 8),         # 8-bit, K tail of 64 (half a stage of 8-bit codes)
    (9, 8192, 2304 + 128, 4),        # 9 tokens: two groups of 8 MMA columns, K tail of 128
    (2, 16384, 1024, 8),             # short K: runs of two groups
    (1, 4096, 16384, 4),             # the longest K
    (16, 4352, 5120, 8),             # 16 tokens, 8-bit, 20 groups over the cluster
    (7, 1100, 16384, 4),             # few row tiles, long K
])
def test_splitk_ragged_shapes(tq, M, N, K, bits):
    mode = "W8A16" if bits == 8 else "W4A16"
    Xb, X, codes, sw, wc = _setup(tq, M, N, K, bits, "rag")
    Y = to_np(tq.linear(X, codes, sw, N, bits, mode))
    assert tq.device_status() == 0
    ref = oracle.linear_a16(bf16_bits(tq.rotate_act_bf16(X)), wc, to_np(sw))
    assert rel_l2(Y, ref) <= REL_L2_Y
    assert rel_l2(Y, oracle.linear_a16(oracle.rotate_act_bf16(Xb), wc, to_np(sw))) <= REL_L2_Y


@pytest.mark.parametrize("bits", [4, 8])
def test_splitk_bf16_output_strided_input(tq, bits):
    """bf16 Y into a padded buffer, from a strided view of a wider input with
    outlier channels (0.2% of columns x40)."""
    import torch
    M, N, K = 8, 4096, 12288
    W = synth.tensor(f"gpu/splitk/bf{bits}/w", N, K, *WB)
    big = synth.tensor(f"gpu/splitk/bf{bits}/x", M, K + 64, 1.0, 0.002, 40.0)
    codes, sw = tq.quantize_weights(to_dev_bf16(W), bits)
    c = to_np(codes)
    wc = oracle.weight_codes(c.view(np.int8) if bits == 8 else c.view(np.uint8), bits, K)
    X = to_dev_bf16(big)[:, 8:8 + K]
    Yfull = torch.full((M, N + 8), 5.0, dtype=torch.bfloat16, device="cuda")
    Y = Yfull[:, :N]
    tq.linear(X, codes, sw, N, bits, "W8A16" if bits == 8 else "W4A16", Y=Y, out="bf16")
    assert tq.device_status() == 0
    ok, frac = _bf16_close(bf16_bits(Y), bf16_bits(tq.rotate_act_bf16(X)), wc, to_np(sw), bits)
    assert ok and frac >= 0.999
    assert torch.all(Yfull[:, N:] == 5.0)


def test_splitk_deterministic_and_rows_of_zeros(tq):
    """Two calls give the same bytes; a token row of zeros gives zeros (its
    rotation is zero, and so is its sum of x', so the bias cancels exactly)."""
    M, N, K = 6, 12288, 4096
    Xb, X, codes, sw, wc = _setup(tq, M, N, K, 4, "det")
    X[2].zero_()
    a = to_np(tq.linear(X, codes, sw, N, 4, "W4A16"))
    b = to_np(tq.linear(X, codes, sw, N, 4, "W4A16"))
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    assert np.all(a[2] == 0)
    ref = oracle.linear_a16(bf16_bits(tq.rotate_act_bf16(X)), wc, to_np(sw))
    assert rel_l2(a, ref) <= REL_L2_Y


def test_splitk_back_to_back_dependent_calls(tq):
    """Each call's input is the previous call's output (bf16), launched back
    to back on one stream: the weight copies of a call start while the one
    before still runs, its input is read only after that one has finished."""
    import torch
    N = K = 4096 + 256
    M = 4
    W = synth.tensor("gpu/splitk/dep/w", N, K, *WB)
    codes, sw = tq.quantize_weights(to_dev_bf16(W), 4)
    c = to_np(codes)
    wc = oracle.weight_codes(c.view(np.uint8), 4, K)
    x0 = synth.tensor("gpu/splitk/dep/x", M, K, 1.0)
    ys = [to_dev_bf16(x0)] + [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    for i in range(4):
        tq.linear(ys[i], codes, sw, N, 4, "W4A16", Y=ys[i + 1], out="bf16")
    torch.cuda.synchronize()
    assert tq.device_status() == 0
    for i in range(4):   # each step against the oracle on the input it actually read
        ok, frac = _bf16_close(bf16_bits(ys[i + 1]), bf16_bits(tq.rotate_act_bf16(ys[i])), wc, to_np(sw), 4)
        assert ok and frac >= 0.999
