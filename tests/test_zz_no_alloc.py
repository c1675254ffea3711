"""tq_linear_a8_static: the W8A8 product for callers that cannot allocate.

Plugins whose host application owns every device allocation, and services
that reserve all device memory at start-up, have no workspace to hand to
tq_linear; tq_linear_a8_static uses a fixed array inside the library instead.
These tests call it through the C ABI and check it against tq_linear (the
workspace entry point) within the fp32 tolerance of the parity tests, on two
calls in a row with different inputs, so a stale scratch would show.  The file
is named to be collected last.
"""
import ctypes

import numpy as np
import pytest

from dit_convrot_linear_gb300 import synth
from helpers import REL_L2_Y, rel_l2, to_dev_bf16, to_np

pytestmark = pytest.mark.gpu

WORKSPACE = 7


def _static_call(tq, X, codes, sw, N, bits, Y):
    import torch
    M, K = X.shape
    return tq.lib().tq_linear_a8_static(
        ctypes.c_void_p(X.data_ptr()), M, K, X.stride(0), ctypes.c_void_p(codes.data_ptr()),
        ctypes.c_void_p(sw.data_ptr()), N, bits, ctypes.c_void_p(Y.data_ptr()), 0, Y.stride(0),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


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
