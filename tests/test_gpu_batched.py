"""GPU parity of the batched A16 product on the tensor cores (tq_linear in
mode W4A16 / W8A16 with its workspace): 8B-class projections (K = 4096 ->
N = 12288 and K = 12288 -> N = 4096, 4-bit weights N(0, 0.015) with 0.5% of
columns x30) at M = 1, 8, 32 and 64 token rows, the batched-decode sizes the
pages' decode/prefill discussion spans (kvad-gpu internals, "Numbers" and
"Quantised weights on the GPU").  One or two tokens over these matrices
stream through the CUDA cores (one token only when N >= K; else the small
decode kernel), three and more run on the tensor cores.

The operand is the A16 one (the rotated row rounded to bf16); the kernel holds
it as fp16 times a power of two per token, which is the same value exactly,
and sums in fp32.  Bar: fp32 Y within relative L2 1e-4 of the oracle's O6 on
the GPU's own bf16 rotation (and on the oracle's rotation), bf16 Y within one
bf16 ulp of the oracle's value rounded to bf16.  The same call without a
workspace runs the CUDA-core kernels, which must agree to the same bar.
"""
import ctypes

import numpy as np
import pytest

import oracle
from dit_convrot_linear_gb300 import synth
from helpers import REL_L2_Y, bf16_bits, bf16_ulp_diff, rel_l2, to_dev_bf16, to_np

pytestmark = pytest.mark.gpu

WB = (0.015, 0.005, 30.0)


def _setup(tq, M, N, K, bits, tag):
    W = synth.tensor(f"gpu/batched/{tag}/w{N}x{K}", N, K, *WB)
    Xb = synth.tensor(f"gpu/batched/{tag}/x{M}x{K}", M, K, 1.0)
    codes, sw = tq.quantize_weights(to_dev_bf16(W), bits)
    return Xb, to_dev_bf16(Xb), codes, sw


def _codes(codes, bits, K):
    c = to_np(codes)
    return oracle.weight_codes(c.view(np.int8) if bits == 8 else c.view(np.uint8), bits, K)


def _no_workspace(tq, X, codes, sw, N, bits, out="f32"):
    """The same call through the C ABI with no workspace (CUDA-core kernels)."""
    import torch
    M, K = X.shape
    Y = torch.empty((M, N), dtype=torch.float32 if out == "f32" else torch.bfloat16, device="cuda")
    rc = tq.lib().tq_linear(X.data_ptr(), M, K, X.stride(0), codes.data_ptr(), sw.data_ptr(), N, bits,
                            0 if bits == 8 else 1, Y.data_ptr(), 0 if out == "f32" else 1, Y.stride(0),
                            None, 0, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    return Y


@pytest.mark.parametrize("M", [1, 2, 3, 8, 32, 64])
@pytest.mark.parametrize("N,K", [(12288, 4096), (4096, 12288)])
def test_batched_w4a16_full_size_sampled(tq, M, N, K):
    Xb, X, codes, sw = _setup(tq, M, N, K, 4, "full")
    assert (tq.linear_workspace_bytes(M, K, N, 4, "W4A16") > 0) == (M > 2)
    Y = to_np(tq.linear(X, codes, sw, N, 4, "W4A16"))
    rng = np.random.default_rng(M * 7 + N)
    pm = np.concatenate([rng.integers(0, M, 3000), [0, M - 1]])
    pn = np.concatenate([rng.integers(0, N, 3000), [N - 1, 0]])
    wc = _codes(codes, 4, K)
    Xr = bf16_bits(tq.rotate_act_bf16(X))
    ref = oracle.linear_a16_pairs(Xr, wc, to_np(sw), pm, pn)
    assert rel_l2(Y[pm, pn], ref) <= REL_L2_Y
    ref2 = oracle.linear_a16_pairs(oracle.rotate_act_bf16(Xb), wc, to_np(sw), pm, pn)
    assert rel_l2(Y[pm, pn], ref2) <= REL_L2_Y
    assert tq.device_status() == 0


@pytest.mark.parametrize("M,N,K,bits", [
    (13, 300, 896, 8),          # K tail of 128, 2 row tiles
    (64, 257, 12288, 4),        # ragged rows (the last tile one row), long K
    (33, 1000, 4096 + 32, 4),   # K tail of 32 (half a K step), 48 token columns
    (16, 4096, 4096, 8),        # 8-bit weights
    (2, 12288, 4096 + 64, 8),   # two tokens: streaming, 8-bit, a K tail of 64
    (1, 9000, 4096 + 32, 4),    # one token, N >= K: streaming, ragged N, a K tail of 32
    (3, 4096, 12288, 4),        # three tokens, N < K: tensor cores
])
def test_batched_matches_the_oracle_and_the_cuda_core_path(tq, M, N, K, bits):
    mode = "W8A16" if bits == 8 else "W4A16"
    Xb, X, codes, sw = _setup(tq, M, N, K, bits, "mix")
    Y = to_np(tq.linear(X, codes, sw, N, bits, mode))
    ref = oracle.linear_a16(bf16_bits(tq.rotate_act_bf16(X)), _codes(codes, bits, K), to_np(sw))
    assert rel_l2(Y, ref) <= REL_L2_Y
    Y0 = to_np(_no_workspace(tq, X, codes, sw, N, bits))
    assert rel_l2(Y0, ref) <= REL_L2_Y
    assert rel_l2(Y, Y0) <= REL_L2_Y
    assert tq.device_status() == 0


def test_batched_bf16_output_strided(tq):
    """bf16 output into a padded buffer from a strided input view."""
    import torch
    M, N, K = 32, 4096, 4096
    W = synth.tensor("gpu/batched/bf/w", N, K, *WB)
    big = synth.tensor("gpu/batched/bf/x", M, K + 64, 1.0)
    codes, sw = tq.quantize_weights(to_dev_bf16(W), 4)
    X = to_dev_bf16(big)[:, 8:8 + K]
    Yfull = torch.full((M, N + 8), 5.0, dtype=torch.bfloat16, device="cuda")
    Y = Yfull[:, :N]
    tq.linear(X, codes, sw, N, 4, "W4A16", Y=Y, out="bf16")
    ref = oracle.linear_a16(oracle.rotate_act_bf16(np.ascontiguousarray(big[:, 8:8 + K])),
                            _codes(codes, 4, K), to_np(sw))
    assert bf16_ulp_diff(bf16_bits(Y), oracle.round_bf16(ref)).max() <= 1
    assert torch.all(Yfull[:, N:] == 5.0)
    assert tq.device_status() == 0


def test_batched_deterministic_and_rows_of_zeros(tq):
    """Two calls give the same bytes; a token row of zeros gives zeros (its
    factor is 2^0 and every code product is 0)."""
    M, N, K = 24, 12288, 4096
    Xb, X, codes, sw = _setup(tq, M, N, K, 4, "det")
    X[5].zero_()
    a = to_np(tq.linear(X, codes, sw, N, 4, "W4A16"))
    b = to_np(tq.linear(X, codes, sw, N, 4, "W4A16"))
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    assert np.all(a[5] == 0)
