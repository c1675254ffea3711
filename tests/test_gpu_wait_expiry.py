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


@pytest.fixture(scope="module")
def splitk_expiring_lib():
    """A copy whose split-K product expects 16 bytes more than its copies
    bring on every stage, its operand waits limited to 2e6 cycles."""
    from dit_convrot_linear_gb300 import build, tq
    path = build.build_variant("splitk_expiry", ["TQ_TEST_UNSET_BYTES=16", "TQ_TEST_WAIT_CYCLES=2000000"],
                               ["k_gemv_splitk.cu"])
    L = ctypes.CDLL(path)
    for name in ("tq_linear", "tq_device_status"):
        res, args = tq.SIGNATURES[name]
        fn = getattr(L, name)
        fn.restype, fn.argtypes = res, args
    return L


def test_split_k_expired_wait_is_reported_and_the_cluster_stores_nothing(tq, splitk_expiring_lib):
    """Every CTA of every cluster gives up its wait (no stage completes);
    each still reaches both cluster barriers, none stores, the status is
    reported once, and the product library then runs the same call right."""
    import torch
    M, N, K = 8, 4096, 12288          # the batched down projection at eight tokens (split-K)
    W = synth.tensor("gpu/expiry/skw", N, K, 0.015, 0.005, 30.0)
    Xh = synth.tensor("gpu/expiry/skx", M, K, 1.0)
    X = to_dev_bf16(Xh)
    codes, sw = tq.quantize_weights(to_dev_bf16(W), 4)
    assert tq.device_status() == 0
    s = torch.cuda.current_stream().cuda_stream
    Y = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    L = splitk_expiring_lib
    rc = L.tq_linear(X.data_ptr(), M, K, X.stride(0), codes.data_ptr(), sw.data_ptr(), N, 4, 1,
                     Y.data_ptr(), 0, Y.stride(0), None, 0, s)
    assert rc == 0
    assert L.tq_device_status(s) == TIMEOUT
    assert L.tq_device_status(s) == 0
    assert torch.all(Y == 0)
    Y2 = to_np(tq.linear(X, codes, sw, N, 4, "W4A16"))
    assert tq.device_status() == 0
    c = to_np(codes)
    ref = oracle.linear_a16(oracle.rotate_act_bf16(Xh), oracle.weight_codes(c.view(np.uint8), 4, K), to_np(sw))
    assert rel_l2(Y2, ref) <= REL_L2_Y


@pytest.fixture(scope="module")
def chain_expiring_lib():
    """A copy whose chained plans wait for one item more than the previous
    call has (so the wait between calls cannot end), every wait of the
    grouped kernel limited to 2e6 cycles."""
    from dit_convrot_linear_gb300 import build, tq
    path = build.build_variant("chain_expiry", ["TQ_TEST_CHAIN_WAIT_EXTRA=1", "TQ_TEST_WAIT_CYCLES=2000000"],
                               ["k_gemv_grouped.cu"])
    L = ctypes.CDLL(path)
    for name in ("tq_chain_bytes", "tq_chain_create", "tq_grouped_run", "tq_grouped_destroy",
                 "tq_device_status"):
        res, args = tq.SIGNATURES[name]
        fn = getattr(L, name)
        fn.restype, fn.argtypes = res, args
    return L


def test_chained_plan_expired_wait_is_reported(tq, chain_expiring_lib):
    """Two dependent calls through the test copy: the first (nothing to wait
    for) completes and is right; the second's wait for the first runs out on
    every CTA that has its items, which stop; the status reports the expiry
    once; the product library then runs the same chain correctly."""
    import torch
    L = chain_expiring_lib
    M, K0, N0, N1 = 1, 512, 256, 128
    x = synth.tensor("gpu/cexp/x", M, K0, 1.0)
    X = to_dev_bf16(x)
    c0, s0 = tq.quantize_weights(to_dev_bf16(synth.tensor("gpu/cexp/w0", N0, K0, 0.02, 0.01, 20.0)), 8)
    c1, s1 = tq.quantize_weights(to_dev_bf16(synth.tensor("gpu/cexp/w1", N1, N0, 0.02, 0.01, 20.0)), 8)
    Y0 = torch.zeros((M, N0), dtype=torch.bfloat16, device="cuda")
    Y1 = torch.zeros((M, N1), dtype=torch.bfloat16, device="cuda")
    recs = [tq.ChainCall(tq.A16Call(X.data_ptr(), K0, c0.data_ptr(), s0.data_ptr(), Y0.data_ptr(), N0, M, N0, K0),
                         None, 0),
            tq.ChainCall(tq.A16Call(Y0.data_ptr(), N0, c1.data_ptr(), s1.data_ptr(), Y1.data_ptr(), N1, M, N1, N0),
                         None, 0)]
    arr = (tq.ChainCall * 2)(*recs)
    need = ctypes.c_size_t(0)
    assert L.tq_chain_bytes(ctypes.addressof(arr), 2, 8, ctypes.byref(need)) == 0
    buf = torch.empty(need.value, dtype=torch.uint8, device="cuda")
    h = ctypes.c_void_p(None)
    assert L.tq_chain_create(ctypes.addressof(arr), 2, 8, 1, buf.data_ptr(), need.value, ctypes.byref(h)) == 0
    assert tq.device_status() == 0
    s = torch.cuda.current_stream().cuda_stream
    assert L.tq_grouped_run(h, s) == 0              # launched; the second call's wait runs out
    assert L.tq_device_status(s) == TIMEOUT
    assert L.tq_device_status(s) == 0
    L.tq_grouped_destroy(h)
    assert torch.all(Y1 == 0)                       # the second call wrote nothing
    ref0 = oracle.linear_a16(oracle.rotate_act_bf16(x), to_np(c0), to_np(s0))
    assert rel_l2(Y0.float().cpu().numpy(), ref0) <= 2.0 ** -8     # the first call is done (bf16 out)
    # the product library on the same context
    plan = tq.ChainPlan([(X, c0, s0, N0, Y0), (Y0, c1, s1, N1, Y1)], 8, out="bf16")
    plan.run()
    assert tq.device_status() == 0
    y0 = Y0.view(torch.int16).cpu().numpy().view(np.uint16)
    ref1 = oracle.linear_a16(oracle.rotate_act_bf16(y0), to_np(c1), to_np(s1))
    assert rel_l2(Y1.float().cpu().numpy(), ref1) <= 2.0 ** -8
