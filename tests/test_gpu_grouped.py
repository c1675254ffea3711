"""GPU parity of the grouped A16 product (tq_grouped_*) against the CPU oracle.

Each call of a plan computes what tq_linear computes in an A16 mode, so the
bars are tq_linear's: fp32 Y within relative L2 1e-4 of the oracle (on the
GPU's own rotated operand and on the oracle's), bf16 Y within 1 bf16 ulp, and
the same bytes on every run.
"""
import numpy as np
import pytest

import oracle
from dit_convrot_linear_gb300 import synth
from helpers import REL_L2_Y, bf16_bits, bf16_ulp_diff, rel_l2, to_dev_bf16, to_np

pytestmark = pytest.mark.gpu

WD = (0.02, 0.01, 20.0)     # decode weights: N(0, 0.02), 1% columns x20
WB = (0.015, 0.005, 30.0)   # batched-decode weights: N(0, 0.015), 0.5% columns x30


def weights(tq, name, N, K, bits):
    W = synth.tensor(name, N, K, *(WD if bits == 8 else WB))
    codes, sw = tq.quantize_weights(to_dev_bf16(W), bits)
    c = to_np(codes)
    Wc = oracle.weight_codes(c.view(np.int8) if bits == 8 else c.view(np.uint8), bits, K)
    return codes, sw, Wc


def build(tq, bits, shapes, out="f32", tag=""):
    """Calls of the given (M, N, K) with fresh inputs; returns the plan, the
    device outputs and, per call, (X as numpy, device X, codes as numpy, sw)."""
    import torch
    calls, host = [], []
    for i, (M, N, K) in enumerate(shapes):
        codes, sw, Wc = weights(tq, f"gpu/grp{tag}/w{i}_{N}x{K}", N, K, bits)
        X = synth.tensor(f"gpu/grp{tag}/x{i}_{M}x{K}", M, K, 1.0, 0.0, 1.0)
        Xd = to_dev_bf16(X)
        Y = torch.full((M, N), float("nan"), dtype=torch.float32 if out == "f32" else torch.bfloat16,
                       device="cuda")
        calls.append((Xd, codes, sw, N, Y))
        host.append((X, Xd, Wc, to_np(sw)))
    return tq.GroupedPlan(calls, bits, out), calls, host


def check_call(tq, Y, X, Xd, Wc, sw):
    Yn = to_np(Y)
    ref_gpu = oracle.linear_a16(bf16_bits(tq.rotate_act_bf16(Xd)), Wc, sw)
    ref_orc = oracle.linear_a16(oracle.rotate_act_bf16(X), Wc, sw)
    assert rel_l2(Yn, ref_gpu) <= REL_L2_Y
    assert rel_l2(Yn, ref_orc) <= REL_L2_Y


SHAPES8 = [(1, 4864, 896), (1, 896, 4864), (2, 300, 4096 + 32), (3, 77, 288), (8, 100, 896),
           (1, 17, 32), (5, 1000, 2304 + 64), (1, 5000, 512), (1, 40, 6400)]
SHAPES4 = [(1, 4864, 896), (1, 896, 4864), (2, 77, 4096 + 128), (1, 21, 2304 + 32),
           (8, 257, 896), (4, 300, 544), (1, 33, 10752)]


@pytest.mark.parametrize("bits,shapes", [(8, SHAPES8), (4, SHAPES4)])
def test_grouped_mixed_shapes(tq, bits, shapes):
    plan, calls, host = build(tq, bits, shapes, tag=f"m{bits}")
    plan.run()
    assert tq.device_status() == 0
    for (_, _, _, _, Y), (X, Xd, Wc, sw) in zip(calls, host):
        check_call(tq, Y, X, Xd, Wc, sw)


def test_grouped_matches_tq_linear_to_rounding(tq):
    shapes = [(1, 4864, 896), (1, 896, 4864), (2, 300, 4096 + 32)]
    plan, calls, host = build(tq, 8, shapes, tag="lin")
    plan.run()
    for (Xd, codes, sw, N, Y) in calls:
        ref = to_np(tq.linear(Xd, codes, sw, N, 8, "W8A16"))
        assert rel_l2(to_np(Y), ref) <= 1e-5


def test_grouped_many_calls_wrap_the_ring(tq):
    """240 calls over four weight sets: every CTA takes many items, so each
    shared-memory stage is reused many times."""
    import torch
    sets = [weights(tq, f"gpu/grpmany/w{j}", N, K, 8)
            for j, (N, K) in enumerate([(4864, 896), (4864, 896), (896, 4864), (1000, 2304 + 64)])]
    shp = [(4864, 896), (4864, 896), (896, 4864), (1000, 2304 + 64)]
    calls, host = [], []
    for i in range(240):
        j = i % 4
        N, K = shp[j]
        codes, sw, Wc = sets[j]
        X = synth.tensor(f"gpu/grpmany/x{i}", 1, K, 1.0, 0.0, 1.0)
        Xd = to_dev_bf16(X)
        Y = torch.full((1, N), float("nan"), dtype=torch.float32, device="cuda")
        calls.append((Xd, codes, sw, N, Y))
        host.append((X, Xd, Wc, to_np(sw)))
    plan = tq.GroupedPlan(calls, 8)
    plan.run()
    assert tq.device_status() == 0
    for i in (0, 1, 2, 3, 117, 238, 239):
        check_call(tq, calls[i][4], *host[i])
    # every output written (no item skipped)
    for c in calls:
        assert torch.isfinite(c[4]).all()


@pytest.mark.parametrize("bits", [4, 8])
def test_grouped_bf16_output_within_one_ulp_or_fp32_rounding(tq, bits):
    """bf16 Y against the oracle's O6 on the GPU's own rotated operand: within
    one bf16 step of the exact value, or, for outputs near zero, within the
    rounding of the fp32 sums.  The product sums the codes with their bias B
    (q + 8 or q + 128, then takes off B times the sum of x'), so its fp32
    partial sums reach sw sum_k |q_nk + B| |x'_k|, and so does their rounding
    error, times a few units of 2^-24: the bar allows 2^-20 of that sum.  It
    stays near 1e-4 of a typical output, while one wrong code, scale or index
    moves Y by about 1e-2 of it."""
    plan, calls, host = build(tq, bits, [(1, 4864, 896), (8, 1000, 2304 + 128)], out="bf16", tag=f"b{bits}")
    plan.run()
    B = 8.0 if bits == 4 else 128.0
    for (_, _, _, _, Y), (X, Xd, Wc, sw) in zip(calls, host):
        xr = bf16_bits(tq.rotate_act_bf16(Xd))
        ref = oracle.linear_a16(xr, Wc, sw)
        got = bf16_bits(Y)
        one_ulp = bf16_ulp_diff(got, oracle.round_bf16(ref)) <= 1
        mag = (np.abs(oracle.bf16_to_f64(xr)) @ np.abs(Wc.astype(np.float64) + B).T) * sw.astype(np.float64)[None, :]
        a = np.abs(ref)
        step = np.exp2(np.floor(np.log2(np.where(a > 0, a, 2.0 ** -133))) - 7)
        near = np.abs(oracle.bf16_to_f64(got) - ref) <= step + 2.0 ** -20 * mag
        assert np.all(one_ulp | near)
        assert one_ulp.mean() >= 0.999     # the rest are outputs near zero


def test_grouped_deterministic_and_graph_replay(tq):
    import torch
    plan, calls, host = build(tq, 8, [(1, 4864, 896), (1, 896, 4864), (3, 500, 1024)], tag="det")
    plan.run()
    first = [to_np(c[4]).copy() for c in calls]
    plan.run()
    for a, c in zip(first, calls):
        assert np.array_equal(a.view(np.uint32), to_np(c[4]).view(np.uint32))
    for c in calls:
        c[4].fill_(float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            plan.run()
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    for a, c in zip(first, calls):
        assert np.array_equal(a.view(np.uint32), to_np(c[4]).view(np.uint32))
    # the two launches of run() on their own
    for c in calls:
        c[4].fill_(float("nan"))
    plan.rotate()
    plan.product()
    for a, c in zip(first, calls):
        assert np.array_equal(a.view(np.uint32), to_np(c[4]).view(np.uint32))


def test_grouped_strided_input_padded_output_and_empty_calls(tq):
    import torch
    M, N, K = 3, 300, 896
    big = synth.tensor("gpu/grpview/x", M, K + 64, 1.0, 0.0, 1.0)
    codes, sw, Wc = weights(tq, "gpu/grpview/w", N, K, 8)
    Xd = to_dev_bf16(big)[:, 8:8 + K]
    Yfull = torch.full((M, N + 28), 7.0, dtype=torch.float32, device="cuda")
    Y = Yfull[:, :N]
    X0 = to_dev_bf16(synth.tensor("gpu/grpview/x0", 1, K, 1.0, 0.0, 1.0))[:0]
    Y0 = torch.empty((0, N), dtype=torch.float32, device="cuda")
    plan = tq.GroupedPlan([(X0, codes, sw, N, Y0), (Xd, codes, sw, N, Y)], 8)
    assert plan.weight_bytes == N * K + 4 * N
    plan.run()
    ref = oracle.linear_a16(oracle.rotate_act_bf16(np.ascontiguousarray(big[:, 8:8 + K])), Wc, to_np(sw))
    assert rel_l2(to_np(Y), ref) <= REL_L2_Y
    assert torch.all(Yfull[:, N:] == 7.0)          # the stride padding is untouched


def test_grouped_decode_workload_sampled(tq):
    """The decode workload's launch configuration: 1000 M = 1 calls cycling
    gate, up, down (896 -> 4864 -> 896); sampled calls against the oracle."""
    import torch
    w = synth.DECODE
    sets = []
    for L in range(2):
        row = []
        for p in w.projs:
            Wd = to_dev_bf16(w.weight(L, p))
            codes, sw = tq.quantize_weights(Wd, 8)
            row.append((codes, sw))
        sets.append(row)
    calls, xs = [], []
    for i in range(1000):
        p = w.projs[i % 3]
        codes, sw = sets[(i // 3) % 2][i % 3]
        X = w.activation(i, p, 1)
        Xd = to_dev_bf16(X)
        Y = torch.full((1, p.N), float("nan"), dtype=torch.float32, device="cuda")
        calls.append((Xd, codes, sw, p.N, Y))
        xs.append((X, Xd))
    plan = tq.GroupedPlan(calls, 8)
    plan.run()
    assert tq.device_status() == 0
    for i in (0, 1, 2, 500, 997, 998, 999):
        Xd, codes, sw, N, Y = calls[i]
        K = Xd.shape[1]
        c = to_np(codes)
        Wc = oracle.weight_codes(c.view(np.int8), 8, K)
        check_call(tq, Y, xs[i][0], Xd, Wc, to_np(sw))


def test_grouped_activation_scales_far_from_one(tq):
    """The product's fp16 operand is x' times a per-token power of two: token
    rows of very large, very small and mixed magnitude (and a zero row) give
    the oracle's result."""
    import torch
    K, N = 896, 300
    codes, sw, Wc = weights(tq, "gpu/grpscale/w", N, K, 8)
    base = oracle.bf16_to_f64(synth.tensor("gpu/grpscale/x", 4, K, 1.0, 0.0, 1.0))
    base[1] *= 2.0 ** 100                     # beyond fp16 range before scaling
    base[2] *= 2.0 ** -100                    # below fp16's smallest normal
    base[3] = 0.0
    X = oracle.round_bf16(base)
    Xd = to_dev_bf16(X)
    Y = torch.full((4, N), float("nan"), dtype=torch.float32, device="cuda")
    plan = tq.GroupedPlan([(Xd, codes, sw, N, Y)], 8)
    plan.run()
    Yn = to_np(Y)
    ref = oracle.linear_a16(oracle.rotate_act_bf16(X), Wc, to_np(sw))
    for m in range(3):
        assert rel_l2(Yn[m], ref[m]) <= REL_L2_Y, m
    assert np.all(Yn[3] == 0.0)
