"""A bounded device wait that runs out: the expiry path of the decode product.

Every device-side wait of the library is bounded; when one runs out the
kernel records the failure in the library's status word, skips the work that
needed the data, lets its own copies in flight land (waiting again, with the
full limit) and returns, so the CUDA context stays usable and
tq_device_status reports TQ_ERR_DEVICE_TIMEOUT.  To take that path on
purpose, the test builds a copy of the library whose decode kernel expects
16 bytes that no copy brings (its barrier's phase then never completes) and
whose operand wait is about 1 ms instead of 2 s.  Nothing traps or spins
without a limit: the operand wait gives up after 2e6 cycles, the final wait
for copies after 4e9 (about 2 s); every copy the kernel issued has landed by
then.  After the expired call, a call of the product library on the same
context must succeed and be correct.
"""
import ctypes

import numpy as np
import pytest

import oracle
from dit_convrot_linear_gb300 import synth
from helpers import REL_L2_Y, rel_l2, to_dev_bf16, to_np

pytestmark = pytest.mark.gpu

TIMEOUT = 9


@pytest.fixture(scope="module")
def expiring_lib():
    from dit_convrot_linear_gb300 import build, tq
    path = build.build_variant("wait_expiry", ["TQ_TEST_UNSET_BYTES=16", "TQ_TEST_WAIT_CYCLES=2000000"],
                               ["k_gemv_small.cu"])
    L = ctypes.CDLL(path)
    for name in ("tq_linear", "tq_device_status"):
        res, args = tq.SIGNATURES[name]
        fn = getattr(L, name)
        fn.restype, fn.argtypes = res, args
    return L


def test_expired_wait_is_reported_and_the_context_stays_usable(tq, expiring_lib):
    import torch
    M, N, K = 1, 4864, 896            # the decode gate projection (small decode kernel)
    W = synth.tensor("gpu/expiry/w", N, K, 0.02, 0.01, 20.0)
    X = to_dev_bf16(synth.tensor("gpu/expiry/x", M, K, 1.0))
    codes, sw = tq.quantize_weights(to_dev_bf16(W), 8)
    assert tq.device_status() == 0
    s = torch.cuda.current_stream().cuda_stream
    Y = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    L = expiring_lib
    rc = L.tq_linear(X.data_ptr(), M, K, X.stride(0), codes.data_ptr(), sw.data_ptr(), N, 8, 0,
                     Y.data_ptr(), 0, Y.stride(0), None, 0, s)
    assert rc == 0                                  # launched; the wait runs out on the device
    assert L.tq_device_status(s) == TIMEOUT         # reported ...
    assert L.tq_device_status(s) == 0               # ... once: reading clears it
    assert torch.all(Y == 0)                        # nothing written by the expired call
    # the product library on the same context: a normal call succeeds and is right
    Y2 = to_np(tq.linear(X, codes, sw, N, 8, "W8A16"))
    assert tq.device_status() == 0
    ref = oracle.linear_a16(oracle.rotate_act_bf16(synth.tensor("gpu/expiry/x", M, K, 1.0)),
                            to_np(codes), to_np(sw))
    assert rel_l2(Y2, ref) <= REL_L2_Y
