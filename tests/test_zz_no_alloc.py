"""tq_linear_a8_static: the W8A8 product for callers that cannot allocate.

Plugins whose host application owns every device allocation, and services
that reserve all device memory at start-up, have no workspace to hand to
tq_linear; tq_linear_a8_static uses a fixed array inside the library instead.
These tests call it through the C ABI and check it, on two calls in a row with
different inputs (so a stale scratch would show), against tq_linear (the
workspace entry point) and against the oracle's product (O5) on the GPU's own
int8 codes, within the fp32 bar of the parity tests; a bf16 case is held to
one bf16 ulp of the oracle.  The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest

import oracle
from dit_convrot_linear_gb300 import synth
from helpers import REL_L2_Y, bf16_bits, bf16_ulp_diff, rel_l2, to_dev_bf16, to_np

pytestmark = pytest.mark.gpu

WORKSPACE = 7
OUT = {"f32": 0, "bf16": 1}


def _static_call(tq, X, codes, sw, N, bits, Y, out="f32"):
    import torch
    M, K = X.shape
    return tq.lib().tq_linear_a8_static(
        ctypes.c_void_p(X.data_ptr()), M, K, X.stride(0), ctypes.c_void_p(codes.data_ptr()),
        ctypes.c_void_p(sw.data_ptr()), N, bits, ctypes.c_void_p(Y.data_ptr()), OUT[out], Y.stride(0),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _oracle_y(tq, X, codes, sw, N, bits):
    """O5 on the GPU's own int8 codes and token scales for X."""
    K = X.shape[1]
    Xq, sx = tq.rotate_quant_act(X)
    c = to_np(codes)
    wc = oracle.weight_codes(c.view(np.int8) if bits == 8 else c.view(np.uint8), bits, K)
    return oracle.linear_a8(to_np(Xq), to_np(sx), wc, to_np(sw), want_acc=False)[1]


@pytest.mark.parametrize("M,N,K,bits", [(200, 300, 3072, 8), (1024, 512, 3072, 4)])
def test_static_scratch_matches_workspace_entry(tq, M, N, K, bits):
    import torch
    W = synth.tensor(f"noalloc/w{N}x{K}", N, K, 0.02, 0.01, 20.0)
    codes, sw = tq.quantize_weights(to_dev_bf16(W), bits)
    for call in range(2):   # two calls in a row, different activations
        X = to_dev_bf16(synth.tensor(f"noalloc/x{call}/{M}x{K}", M, K, 1.0, 0.002, 40.0))
        ref = to_np(tq.linear(X, codes, sw, N, bits, "W8A8"))
        Y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        assert _static_call(tq, X, codes, sw, N, bits, Y) == 0
        got = to_np(Y)
        assert np.all(np.isfinite(got))
        assert rel_l2(got, ref) <= REL_L2_Y
        assert rel_l2(got, _oracle_y(tq, X, codes, sw, N, bits)) <= REL_L2_Y
    assert tq.device_status() == 0


def test_static_scratch_tail_strided_bf16(tq):
    """A row length with a 32-column tail group, X read through a strided
    view (row stride above K), Y written as bf16 into a padded buffer: each
    output within one bf16 ulp of the oracle's value rounded to bf16, the
    padding untouched, on two calls in a row."""
    import torch
    M, N, K = 130, 200, 3072 + 32
    W = synth.tensor("noalloc/tail/w", N, K, 0.02, 0.01, 20.0)
    codes, sw = tq.quantize_weights(to_dev_bf16(W), 8)
    for call in range(2):
        big = to_dev_bf16(synth.tensor(f"noalloc/tail/x{call}", M, K + 64, 1.0, 0.002, 40.0))
        X = big[:, 8:8 + K]                     # offset 16 bytes, row stride K + 64
        assert X.stride(0) == K + 64
        Yfull = torch.full((M, N + 24), 3.0, dtype=torch.bfloat16, device="cuda")
        Y = Yfull[:, :N]
        assert _static_call(tq, X, codes, sw, N, 8, Y, out="bf16") == 0
        ref = _oracle_y(tq, X, codes, sw, N, 8)
        assert bf16_ulp_diff(bf16_bits(Y), oracle.round_bf16(ref)).max() <= 1
        assert torch.all(Yfull[:, N:] == 3.0)
    assert tq.device_status() == 0


def test_static_scratch_refuses_oversize_calls(tq):
    import torch
    K = 12288
    M = (16 << 20) // K + 1       # codes alone exceed the 16 MiB array
    X = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    codes = torch.zeros((64, K), dtype=torch.int8, device="cuda")
    sw = torch.ones(64, dtype=torch.float32, device="cuda")
    Y = torch.zeros((M, 64), dtype=torch.float32, device="cuda")
    assert _static_call(tq, X, codes, sw, 64, 8, Y) == WORKSPACE
