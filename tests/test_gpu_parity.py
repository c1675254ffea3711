"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Bars (fixed before any kernel ran):
  - weight codes and scales: bit-exact;
  - A8 activation codes: at most 0.1% differ, each by at most 1 (fp32 FWHT
    summation order); token scales within 2^-20 relative;
  - A16 bf16 operands: at most 0.1% differ, each by at most 1 ulp;
  - int32 accumulators: bit-exact given the GPU's own int8 operands;
  - fp32 Y: relative L2 <= 1e-4 against the oracle on the GPU's own operands;
    bf16 Y: within 1 bf16 ulp of the oracle's value rounded to bf16.
"""
import numpy as np
import pytest

import oracle
from dit_convrot_linear_gb300 import synth
from helpers import (CODE_FLIP_FRAC, REL_L2_Y, SCALE_REL, ULP_FLIP_FRAC, act_trailer, bf16_bits,
                     bf16_ulp_diff, check_codes_close, parity_report, rel_l2, untile_codes,
                     to_dev_bf16, to_np)

pytestmark = pytest.mark.gpu

WD = (0.02, 0.01, 20.0)     # decode / DiT weights: N(0, 0.02), 1% columns x20
WB = (0.015, 0.005, 30.0)   # batched-decode / chain weights
XD = (1.0, 0.002, 40.0)     # DiT activations: 0.2% channels x40


def wgen(name, N, K, d=WD):
    return synth.tensor(name, N, K, *d)


def xgen(name, M, K, d=(1.0, 0.0, 1.0)):
    return synth.tensor(name, M, K, *d)


def gpu_weights(tq, W, bits):
    codes, sw = tq.quantize_weights(to_dev_bf16(W), bits)
    return codes, sw


def codes_np(codes, bits, K):
    c = to_np(codes)
    return oracle.weight_codes(c.view(np.int8) if bits == 8 else c.view(np.uint8), bits, K)


# ------------------------------------------------------------------ weights

W_CASES = [
    ("tiny", 256, 512, 8), ("tiny", 256, 512, 4),
    ("gate", 4864, 896, 8), ("gate", 4864, 896, 4),
    ("down", 896, 4864, 8), ("down", 896, 4864, 4),
    ("tail32", 40, 288, 8), ("tail64", 33, 320, 4), ("k32", 17, 32, 4),
    ("k64", 9, 64, 8), ("k128", 5, 128, 4), ("ragged", 1001, 4096 + 128, 4),
]


@pytest.mark.parametrize("name,N,K,bits", W_CASES)
def test_weights_bit_exact(tq, name, N, K, bits):
    W = wgen(f"gpu/w/{name}", N, K)
    codes, sw = gpu_weights(tq, W, bits)
    ref_codes, ref_s = oracle.quantize_weights(W, bits)
    got = to_np(codes)
    assert np.array_equal(got.view(np.uint8), ref_codes.view(np.uint8))
    assert np.array_equal(to_np(sw).view(np.uint32), ref_s.view(np.uint32))


@pytest.mark.parametrize("N,K,bits", [(12288, 4096, 4), (4096, 12288, 4), (12288, 3072, 8),
                                      (3072, 12288, 8), (24576, 3072, 4)])
def test_weights_full_size_sampled_rows(tq, N, K, bits):
    W = wgen(f"gpu/wbig/{N}x{K}", N, K, WB if bits == 4 else WD)
    codes, sw = gpu_weights(tq, W, bits)
    rows = np.unique(np.concatenate([[0, N - 1], np.random.default_rng(N).integers(0, N, 62)]))
    ref_codes, ref_s = oracle.quantize_weights(W[rows], bits)
    got = to_np(codes)[rows]
    assert np.array_equal(got.view(np.uint8), ref_codes.view(np.uint8))
    assert np.array_equal(to_np(sw)[rows].view(np.uint32), ref_s.view(np.uint32))


def test_weights_strided_source(tq):
    import torch
    W = wgen("gpu/w/strided", 64, 896 + 64)
    Wd = to_dev_bf16(W)[:, :896]          # row stride 960 elements
    assert Wd.stride(0) == 960
    codes, sw = tq.quantize_weights(Wd, 8)
    ref_codes, ref_s = oracle.quantize_weights(np.ascontiguousarray(W[:, :896]), 8)
    assert np.array_equal(to_np(codes), ref_codes)
    assert np.array_equal(to_np(sw), ref_s)
    del torch


def test_weights_zero_row(tq):
    W = wgen("gpu/w/zero", 8, 512)
    W[3] = 0
    codes, sw = gpu_weights(tq, W, 8)
    assert to_np(sw)[3] == 0 and np.all(to_np(codes)[3] == 0)


# ------------------------------------------------------------------ activations

X_CASES = [
    ("tiny", 4, 512, (1.0, 0.0, 25.0), (3, 300)),
    ("dit_up", 64, 3072, XD, None), ("dit_down", 16, 12288, XD, None),
    ("k896", 7, 896, XD, None), ("k32", 3, 32, XD, None), ("k4864", 5, 4864, XD, None),
    ("long", 2, 65536, XD, None), ("k4160", 9, 4096 + 64, XD, None),
]


@pytest.mark.parametrize("name,M,K,d,ch", X_CASES)
def test_activation_codes(tq, name, M, K, d, ch):
    X = synth.tensor(f"gpu/x/{name}", M, K, d[0], d[1], d[2], channels=ch)
    Xq, sx = tq.rotate_quant_act(to_dev_bf16(X))
    rq, rs = oracle.rotate_quant_act(X)
    check_codes_close(to_np(Xq), rq)
    assert np.all(np.abs(to_np(sx).astype(np.float64) - rs) <= SCALE_REL * np.abs(rs))


def test_activation_bf16_rotation(tq):
    for K in (512, 896, 4864, 12288, 96 + 256 - 96):
        X = xgen(f"gpu/xr/{K}", 6, K, XD)
        Xr = tq.rotate_act_bf16(to_dev_bf16(X))
        ref = oracle.rotate_act_bf16(X)
        d = bf16_ulp_diff(bf16_bits(Xr), ref)
        assert d.max() <= 1
        assert np.count_nonzero(d) <= ULP_FLIP_FRAC * d.size


def test_activation_strided_offset_view(tq):
    # The pages' offset-view lesson (kvad-gpu internals): a product must read
    # its input rows where the view starts, not from the buffer start.
    K = 896
    big = xgen("gpu/x/view", 9, K + 64, XD)
    Xd = to_dev_bf16(big)[:, 8:8 + K]       # offset 16 bytes, row stride K + 64
    Xq, sx = tq.rotate_quant_act(Xd)
    rq, rs = oracle.rotate_quant_act(np.ascontiguousarray(big[:, 8:8 + K]))
    check_codes_close(to_np(Xq), rq)


# ------------------------------------------------------------------ A16 product

A16_CASES = [
    (4, 256, 512, 8), (1, 4864, 896, 8), (1, 896, 4864, 8), (1, 4864, 896, 4),
    (1, 896, 4864, 4), (8, 1000, 4096 + 128, 4), (13, 300, 896, 8), (32, 512, 4096, 4),
    (64, 257, 12288, 4), (3, 77, 32, 8), (5, 100, 288, 4), (64, 4096, 4096, 8),
    # eight-row decode kernel: M <= 2, ragged rows, K with a partial last block
    (2, 300, 4096 + 32, 8), (2, 77, 4096 + 128, 4), (1, 40, 2304 + 64, 8), (1, 21, 2304 + 32, 4),
]


@pytest.mark.parametrize("M,N,K,bits", A16_CASES)
def test_a16_product(tq, M, N, K, bits):
    mode = "W8A16" if bits == 8 else "W4A16"
    X = xgen(f"gpu/a16/x{M}x{K}", M, K)
    W = wgen(f"gpu/a16/w{N}x{K}", N, K, WD if bits == 8 else WB)
    codes, sw = gpu_weights(tq, W, bits)
    Xd = to_dev_bf16(X)
    Y = to_np(tq.linear(Xd, codes, sw, N, bits, mode))
    Wc = codes_np(codes, bits, K)
    # oracle on the GPU's own operands (its bf16 rotation and codes)
    Xr = bf16_bits(tq.rotate_act_bf16(Xd))
    ref = oracle.linear_a16(Xr, Wc, to_np(sw))
    rep = parity_report(Y, ref)
    assert rep["rel_l2"] <= REL_L2_Y, rep
    # and on the oracle's own rotation of the same input
    ref2 = oracle.linear_a16(oracle.rotate_act_bf16(X), Wc, to_np(sw))
    assert rel_l2(Y, ref2) <= REL_L2_Y


def test_a16_strided_offset_input_and_padded_output(tq):
    import torch
    M, N, K = 5, 300, 896
    big = xgen("gpu/a16/view", M, K + 64)
    W = wgen("gpu/a16/vw", N, K)
    codes, sw = gpu_weights(tq, W, 8)
    Xd = to_dev_bf16(big)[:, 8:8 + K]
    Yfull = torch.full((M, N + 28), 7.0, dtype=torch.float32, device="cuda")
    Y = Yfull[:, :N]
    tq.linear(Xd, codes, sw, N, 8, "W8A16", Y=Y)
    ref = oracle.linear_a16(oracle.rotate_act_bf16(np.ascontiguousarray(big[:, 8:8 + K])),
                            to_np(codes), to_np(sw))
    assert rel_l2(to_np(Y), ref) <= REL_L2_Y
    assert torch.all(Yfull[:, N:] == 7.0)       # the stride padding is untouched


def test_a16_bf16_output_within_one_ulp(tq):
    M, N, K = 8, 1000, 4096
    X = xgen("gpu/a16b/x", M, K)
    W = wgen("gpu/a16b/w", N, K, WB)
    codes, sw = gpu_weights(tq, W, 4)
    Xd = to_dev_bf16(X)
    Yb = tq.linear(Xd, codes, sw, N, 4, "W4A16", out="bf16")
    ref = oracle.linear_a16(bf16_bits(tq.rotate_act_bf16(Xd)), codes_np(codes, 4, K), to_np(sw))
    assert bf16_ulp_diff(bf16_bits(Yb), oracle.round_bf16(ref)).max() <= 1


def test_a16_deterministic(tq):
    M, N, K = 1, 896, 4864
    X = to_dev_bf16(xgen("gpu/det/x", M, K))
    codes, sw = gpu_weights(tq, wgen("gpu/det/w", N, K), 8)
    a = to_np(tq.linear(X, codes, sw, N, 8, "W8A16"))
    b = to_np(tq.linear(X, codes, sw, N, 8, "W8A16"))
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


# ------------------------------------------------------------------ A8 product

A8_CASES = [
    (4, 256, 512, 8), (130, 200, 896, 8), (130, 200, 896, 4), (257, 300, 4096 + 32, 8),
    (64, 1024, 12288, 4), (1, 64, 256, 8), (300, 129, 3072, 4),
]


@pytest.mark.parametrize("M,N,K,bits", A8_CASES)
def test_a8_product(tq, M, N, K, bits):
    X = xgen(f"gpu/a8/x{M}x{K}", M, K, XD)
    W = wgen(f"gpu/a8/w{N}x{K}", N, K, WD if bits == 8 else WB)
    codes, sw = gpu_weights(tq, W, bits)
    Xd = to_dev_bf16(X)
    Xq, sx = tq.rotate_quant_act(Xd)
    acc = to_np(tq.linear_q8(Xq, sx, codes, sw, N, bits, out="i32"))
    ref_acc, ref_Y = oracle.linear_a8(to_np(Xq), to_np(sx), codes_np(codes, bits, K), to_np(sw))
    assert np.array_equal(acc, ref_acc)
    Y = to_np(tq.linear_q8(Xq, sx, codes, sw, N, bits))
    assert rel_l2(Y, ref_Y) <= REL_L2_Y
    Y2 = to_np(tq.linear(Xd, codes, sw, N, bits, "W8A8"))
    assert np.array_equal(Y.view(np.uint32), Y2.view(np.uint32))


@pytest.mark.parametrize("M,N,K,bits", [(300, 129, 3072, 8), (257, 300, 4096 + 32, 4), (1, 64, 288, 8),
                                          (600, 512, 12288, 8)])
def test_tiled_operand_matches_int8_path(tq, M, N, K, bits):
    """The tiled activation operand carries the same codes and scales as
    tq_rotate_quant_act and gives the same exact int32 sums.  The buffer is
    filled with 0xFF first (fp16 NaN) so that padding it fails to zero, or a
    pad row leaking into real rows, would show."""
    import torch
    X = to_dev_bf16(xgen(f"gpu/tiled/x{M}x{K}", M, K, XD))
    codes, sw = gpu_weights(tq, wgen(f"gpu/tiled/w{N}x{K}", N, K, WD if bits == 8 else WB), bits)
    At = torch.full((tq.act_tiled_bytes(M, K),), 0xFF, dtype=torch.uint8, device="cuda")
    At, sxt = tq.rotate_quant_act_tiled(X, At=At)
    Xq, sx = tq.rotate_quant_act(X)
    assert np.array_equal(to_np(sxt).view(np.uint32), to_np(sx).view(np.uint32))
    acc_t = to_np(tq.linear_tiled(At, sxt, M, K, codes, sw, N, bits, out="i32"))
    acc = to_np(tq.linear_q8(Xq, sx, codes, sw, N, bits, out="i32"))
    assert np.array_equal(acc_t, acc)
    # the tests' decoding of the tiled layout gives the same codes
    assert np.array_equal(untile_codes(At, M, K), to_np(Xq).astype(np.int64))
    ref_acc, _ = oracle.linear_a8(to_np(Xq), to_np(sx), codes_np(codes, bits, K), to_np(sw))
    assert np.array_equal(acc_t, ref_acc)


@pytest.mark.parametrize("M,N,K,bits", [(300, 129, 3072, 8), (257, 300, 4096 + 32, 4), (1, 64, 288, 8),
                                         (513, 520, 2304 + 64, 8), (64, 256, 12288, 4)])
def test_tiled_weights_match_the_converting_product(tq, M, N, K, bits):
    """Weights widened once into fp16 tiles (tq_tile_weights) give the same
    exact int32 sums as the product that widens them itself, and the oracle's.
    The tile buffer is filled with 0xFF first (fp16 NaN), so padding that was
    not zeroed, or a pad row reaching an output, would show."""
    import torch
    X = to_dev_bf16(xgen(f"gpu/tt/x{M}x{K}", M, K, XD))
    codes, sw = gpu_weights(tq, wgen(f"gpu/tt/w{N}x{K}", N, K, WD if bits == 8 else WB), bits)
    At, sx = tq.rotate_quant_act_tiled(X)
    Wt = torch.full((tq.weights_tiled_bytes(N, K),), 0xFF, dtype=torch.uint8, device="cuda")
    tq.tile_weights(codes, N, K, bits, Wt=Wt)
    acc_tt = to_np(tq.linear_tt(At, sx, M, K, Wt, sw, N, bits, out="i32"))
    acc_t = to_np(tq.linear_tiled(At, sx, M, K, codes, sw, N, bits, out="i32"))
    assert np.array_equal(acc_tt, acc_t)
    Xq, sxq = tq.rotate_quant_act(X)
    ref_acc, ref_Y = oracle.linear_a8(to_np(Xq), to_np(sxq), codes_np(codes, bits, K), to_np(sw))
    assert np.array_equal(acc_tt, ref_acc)
    Y = to_np(tq.linear_tt(At, sx, M, K, Wt, sw, N, bits))
    assert rel_l2(Y, ref_Y) <= REL_L2_Y
    assert tq.device_status() == 0


@pytest.mark.parametrize("M,N,K,bits", [(300, 129, 3072, 8), (257, 300, 4096 + 32, 4), (64, 256, 12288, 8)])
def test_tiled_trailers_hold_the_largest_row_sums_of_squares(tq, M, N, K, bits):
    """The product's exactness bound reads, after the tiles, the activation
    rows' and the weight rows' largest sum of codes squared (word 6 of the
    activation trailer, word 0 of the weights'): both equal the maximum over
    the real rows computed from the codes themselves."""
    X = to_dev_bf16(xgen(f"gpu/trail/x{M}x{K}", M, K, XD))
    codes, sw = gpu_weights(tq, wgen(f"gpu/trail/w{N}x{K}", N, K, WD if bits == 8 else WB), bits)
    At, sx = tq.rotate_quant_act_tiled(X)
    a = untile_codes(At, M, K).astype(np.int64)
    at_tr = act_trailer(tq, At, M, K)
    def window_max(v, j):          # largest sum over an aligned run of 2^j 1024-column windows
        L = 1024 << j
        pad = np.zeros((v.shape[0], -v.shape[1] % L), dtype=np.int64)
        return int(np.concatenate([v, pad], axis=1).reshape(v.shape[0], -1, L).sum(axis=2).max())
    assert int(at_tr[6]) == int((a * a).sum(axis=1).max())
    # words 0..5: the |code| row sums, whole and per aligned window; 7..11 the squares per window
    assert int(at_tr[0]) == int(np.abs(a).sum(axis=1).max())
    for j in range(5):
        assert int(at_tr[1 + j]) == window_max(np.abs(a), j)
        assert int(at_tr[7 + j]) == window_max(a * a, j)
    Wt = tq.tile_weights(codes, N, K, bits)
    w = codes_np(codes, bits, K).astype(np.int64)
    wt_tr = to_np(Wt[tq.weights_tiled_bytes(N, K) - 256:]).view(np.uint32)
    assert int(wt_tr[0]) == int((w * w).sum(axis=1).max())
    for j in range(5):
        assert int(wt_tr[1 + j]) == window_max(w * w, j)


@pytest.mark.parametrize("N,K", [(12288, 3072), (3072, 12288)])
def test_tiled_weights_dit_m4032_sampled(tq, N, K):
    """The DiT projections at full size through the both-tiled product, in the
    launch configuration the bench times; sampled outputs against the oracle."""
    M = 4032
    X = xgen(f"gpu/ttdit/x{K}", M, K, XD)
    W = wgen(f"gpu/ttdit/w{N}x{K}", N, K)
    codes, sw = gpu_weights(tq, W, 8)
    At, sx = tq.rotate_quant_act_tiled(to_dev_bf16(X))
    Wt = tq.tile_weights(codes, N, K, 8)
    acc = to_np(tq.linear_tt(At, sx, M, K, Wt, sw, N, 8, out="i32"))
    Y = to_np(tq.linear_tt(At, sx, M, K, Wt, sw, N, 8))
    rng = np.random.default_rng(7)
    rows = np.sort(rng.choice(M, 24, replace=False))
    Xq, sxq = tq.rotate_quant_act(to_dev_bf16(X))
    pm = rng.integers(0, len(rows), 400)
    pn = rng.integers(0, N, 400)
    ref_acc, ref_Y = oracle.linear_a8_pairs(to_np(Xq)[rows], to_np(sxq)[rows], to_np(codes), to_np(sw), pm, pn)
    assert np.array_equal(acc[rows[pm], pn], ref_acc)
    assert rel_l2(Y[rows[pm], pn], ref_Y) <= REL_L2_Y


@pytest.mark.parametrize("M,N,K,bits,parts", [
    (300, 129, 3072, 8, "bgr32"), (257, 300, 4096 + 32, 4, "bgr16"), (64, 256, 512, 8, "b"),
    (130, 200, 896, 8, "g"), (513, 520, 2304 + 64, 8, "r16")])
def test_tiled_weights_fused_epilogue(tq, M, N, K, bits, parts):
    """Y = R + gate * (product + bias) in the product's epilogue, against the
    oracle's product with the same formula in fp64 (fp32 and bf16 residuals)."""
    import torch
    X = to_dev_bf16(xgen(f"gpu/epi/x{M}x{K}", M, K, XD))
    codes, sw = gpu_weights(tq, wgen(f"gpu/epi/w{N}x{K}", N, K, WD if bits == 8 else WB), bits)
    At, sx = tq.rotate_quant_act_tiled(X)
    Wt = tq.tile_weights(codes, N, K, bits)
    rng = np.random.default_rng(M + N)
    bias = torch.from_numpy(rng.normal(0, 2.0, N).astype(np.float32)).cuda() if "b" in parts else None
    gate = torch.from_numpy(rng.normal(0, 1.0, N).astype(np.float32)).cuda() if "g" in parts else None
    R = None
    if "r" in parts:
        Rn = rng.normal(0, 30.0, (M, N)).astype(np.float32)
        R = torch.from_numpy(Rn).cuda()
        if parts.endswith("16"):
            R = R.to(torch.bfloat16)
    Y = tq.linear_tt_ex(At, sx, M, K, Wt, sw, N, bits, bias=bias, gate=gate, residual=R)
    Xq, sxq = tq.rotate_quant_act(X)
    _, Y0 = oracle.linear_a8(to_np(Xq), to_np(sxq), codes_np(codes, bits, K), to_np(sw))
    b = to_np(bias).astype(np.float64) if bias is not None else 0.0
    g = to_np(gate).astype(np.float64) if gate is not None else 1.0
    r = to_np(R.float()).astype(np.float64) if R is not None else 0.0
    ref = r + g * (Y0 + b)
    assert rel_l2(to_np(Y), ref) <= REL_L2_Y
    assert tq.device_status() == 0


def test_tiled_weights_epilogue_in_place_bf16(tq):
    """The residual stream updated in place (R is Y, bf16): each output within
    one bf16 ulp of the oracle's value rounded to bf16."""
    import torch
    M, N, K = 260, 384, 3072
    X = to_dev_bf16(xgen("gpu/epiip/x", M, K, XD))
    codes, sw = gpu_weights(tq, wgen("gpu/epiip/w", N, K), 8)
    At, sx = tq.rotate_quant_act_tiled(X)
    Wt = tq.tile_weights(codes, N, K, 8)
    rng = np.random.default_rng(5)
    gate = torch.from_numpy(rng.normal(0, 1.0, N).astype(np.float32)).cuda()
    R = torch.from_numpy(rng.normal(0, 30.0, (M, N)).astype(np.float32)).cuda().to(torch.bfloat16)
    r = to_np(R.float()).astype(np.float64)
    tq.linear_tt_ex(At, sx, M, K, Wt, sw, N, 8, Y=R, out="bf16", gate=gate, residual=R)
    Xq, sxq = tq.rotate_quant_act(X)
    _, Y0 = oracle.linear_a8(to_np(Xq), to_np(sxq), to_np(codes), to_np(sw))
    ref = r + to_np(gate).astype(np.float64) * Y0
    assert bf16_ulp_diff(bf16_bits(R), oracle.round_bf16(ref)).max() <= 1


@pytest.mark.parametrize("M,K", [(300, 3072), (257, 4096 + 32), (5, 544), (64, 12288), (130, 896)])
def test_swiglu_fused_operand(tq, M, K):
    """The down projection's operand made from gate and up in one pass: codes
    and token scales against the oracle's SwiGLU (O8) then quantiser (O4), to
    the activation-code bar; and the tiled form's own layout decodes to the
    same codes as the unfused route (the oracle's bf16 h through
    tq_rotate_quant_act_tiled), the two differing only where h does."""
    import torch
    G = xgen(f"gpu/swiglu/g{M}x{K}", M, K, (1.5, 0.0, 1.0))
    U = xgen(f"gpu/swiglu/u{M}x{K}", M, K, XD)
    # gate and up as the two halves of one fused gate/up output row
    GU = np.concatenate([G, U], axis=1)
    GUd = to_dev_bf16(GU)
    At, sx = tq.swiglu_quant_act_tiled(GUd[:, :K], GUd[:, K:])
    codes = untile_codes(At, M, K)
    rq, rs = oracle.swiglu_quant_act(G, U)
    check_codes_close(codes, rq, frac=CODE_FLIP_FRAC)
    assert np.max(np.abs(to_np(sx).astype(np.float64) / np.where(rs == 0, 1, rs) - 1)) <= SCALE_REL
    H = oracle.swiglu_bf16(G, U)
    At2, sx2 = tq.rotate_quant_act_tiled(to_dev_bf16(H))
    check_codes_close(codes, untile_codes(At2, M, K), frac=CODE_FLIP_FRAC)
    assert tq.device_status() == 0


def test_swiglu_fused_operand_full_size_sampled(tq):
    """The DiT down projection's operand at the size the bench times (M = 4032,
    K = 12288), from gate and up in one pass: sampled token rows against the
    oracle's SwiGLU then quantiser on the same rows, and the trailer's exact
    row sums on them."""
    M, K = 4032, 12288
    G = xgen("gpu/swfull/g", M, K, (1.5, 0.0, 1.0))
    U = xgen("gpu/swfull/u", M, K, XD)
    At, sx = tq.swiglu_quant_act_tiled(to_dev_bf16(G), to_dev_bf16(U))
    assert tq.device_status() == 0
    rows = np.sort(np.random.default_rng(11).choice(M, 24, replace=False))
    codes = untile_codes(At, M, K, rows=rows)
    rq, rs = oracle.swiglu_quant_act(G[rows], U[rows])
    check_codes_close(codes, rq, frac=CODE_FLIP_FRAC)
    assert np.max(np.abs(to_np(sx)[rows].astype(np.float64) / np.where(rs == 0, 1, rs) - 1)) <= SCALE_REL
    tr = act_trailer(tq, At, M, K)
    assert int(tr[0]) >= int(np.abs(codes).sum(axis=1).max())     # a maximum over all rows
    assert int(tr[6]) >= int((codes * codes).sum(axis=1).max())


def test_swiglu_fused_operand_feeds_the_product(tq):
    """gate/up -> fused SwiGLU operand -> both-tiled down product, against the
    oracle's int32 sums on the same codes (exact) and its Y."""
    M, N, K = 260, 300, 4096
    G = xgen("gpu/swiglu2/g", M, K, (1.5, 0.0, 1.0))
    U = xgen("gpu/swiglu2/u", M, K, XD)
    codes_w, sw = gpu_weights(tq, wgen("gpu/swiglu2/w", N, K), 8)
    At, sx = tq.swiglu_quant_act_tiled(to_dev_bf16(G), to_dev_bf16(U))
    Wt = tq.tile_weights(codes_w, N, K, 8)
    acc = to_np(tq.linear_tt(At, sx, M, K, Wt, sw, N, 8, out="i32"))
    xq = untile_codes(At, M, K).astype(np.int8)
    ref_acc, ref_Y = oracle.linear_a8(xq, to_np(sx), to_np(codes_w), to_np(sw))
    assert np.array_equal(acc, ref_acc)
    Y = to_np(tq.linear_tt(At, sx, M, K, Wt, sw, N, 8))
    assert rel_l2(Y, ref_Y) <= REL_L2_Y


@pytest.mark.parametrize("bits", [8, 4])
def test_tiled_operand_flat_rows(tq, bits):
    """Rows whose rotation is flat (one nonzero per 256-group, so every rotated
    value of a group is equal): all codes are +-127, the row norms are as large
    as they can be, and the product must fall back from one fp32 accumulation
    per tile to exact chunks (8-bit weights) and still be exact."""
    import torch
    M, N, K = 300, 129, 3072
    X = np.zeros((M, K), np.float32)
    rng = np.random.default_rng(bits)
    mag = rng.choice([0.5, 0.75, 1.0, 1.5, 2.0], size=(M, 1)).astype(np.float32)   # exact in bf16
    X[:, ::256] = rng.choice([-1.0, 1.0], size=(M, K // 256)).astype(np.float32) * mag
    Xd = to_dev_bf16((X.view(np.uint32) >> 16).astype(np.uint16))
    codes, sw = gpu_weights(tq, wgen(f"gpu/flat/w{bits}", N, K, WD if bits == 8 else WB), bits)
    At, sxt = tq.rotate_quant_act_tiled(Xd)
    Xq, sx = tq.rotate_quant_act(Xd)
    assert np.all(np.abs(to_np(Xq).astype(np.int32)) == 127)
    acc_t = to_np(tq.linear_tiled(At, sxt, M, K, codes, sw, N, bits, out="i32"))
    ref_acc, _ = oracle.linear_a8(to_np(Xq), to_np(sx), codes_np(codes, bits, K), to_np(sw))
    assert np.array_equal(acc_t, ref_acc)


def test_a8_extreme_accumulators(tq):
    import torch
    K = 12288
    Xq = torch.full((3, K), 127, dtype=torch.int8, device="cuda")
    Xq[1] = -127
    Wq = torch.full((5, K), -127, dtype=torch.int8, device="cuda")
    ones = torch.ones(5, dtype=torch.float32, device="cuda")
    acc = to_np(tq.linear_q8(Xq, ones[:3], Wq, ones, 5, 8, out="i32"))
    assert np.all(acc[0] == -127 * 127 * K) and np.all(acc[1] == 127 * 127 * K)


def test_a8_bf16_output_within_one_ulp(tq):
    M, N, K = 200, 300, 3072
    X = xgen("gpu/a8b/x", M, K, XD)
    codes, sw = gpu_weights(tq, wgen("gpu/a8b/w", N, K), 8)
    Xq, sx = tq.rotate_quant_act(to_dev_bf16(X))
    Yb = tq.linear_q8(Xq, sx, codes, sw, N, 8, out="bf16")
    _, ref = oracle.linear_a8(to_np(Xq), to_np(sx), to_np(codes), to_np(sw))
    assert bf16_ulp_diff(bf16_bits(Yb), oracle.round_bf16(ref)).max() <= 1


def test_a8_deterministic(tq):
    M, N, K = 300, 500, 3072
    X = to_dev_bf16(xgen("gpu/det8/x", M, K, XD))
    codes, sw = gpu_weights(tq, wgen("gpu/det8/w", N, K), 8)
    a = to_np(tq.linear(X, codes, sw, N, 8, "W8A8"))
    b = to_np(tq.linear(X, codes, sw, N, 8, "W8A8"))
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


# ------------------------------------------------------------------ full sizes

@pytest.mark.parametrize("N,K", [(12288, 3072), (3072, 12288)])
def test_dit_m4032_sampled(tq, N, K):
    """The DiT workload at full size (M = 4032, W8A8), in the bench's launch
    configuration, checked on sampled outputs the oracle computes one by one."""
    M = 4032
    X = xgen(f"gpu/dit/x{K}", M, K, XD)
    codes, sw = gpu_weights(tq, wgen(f"gpu/dit/w{N}x{K}", N, K), 8)
    Xd = to_dev_bf16(X)
    Y = to_np(tq.linear(Xd, codes, sw, N, 8, "W8A8"))
    Xq, sx = tq.rotate_quant_act(Xd)
    rng = np.random.default_rng(K)
    rows = np.unique(np.concatenate([[0, M - 1], rng.integers(0, M, 30)]))
    rq, rs = oracle.rotate_quant_act(X[rows])
    check_codes_close(to_np(Xq)[rows], rq, frac=CODE_FLIP_FRAC)
    pm = np.concatenate([rng.integers(0, M, 2000), [0, M - 1, M - 1]])
    pn = np.concatenate([rng.integers(0, N, 2000), [0, N - 1, 0]])
    acc, refY = oracle.linear_a8_pairs(to_np(Xq), to_np(sx), to_np(codes), to_np(sw), pm, pn)
    assert rel_l2(Y[pm, pn], refY) <= REL_L2_Y


@pytest.mark.parametrize("N,K", [(12288, 4096), (4096, 12288)])
def test_batched_m64_full(tq, N, K):
    M = 64
    X = xgen(f"gpu/b64/x{K}", M, K)
    codes, sw = gpu_weights(tq, wgen(f"gpu/b64/w{N}x{K}", N, K, WB), 4)
    Xd = to_dev_bf16(X)
    Y = to_np(tq.linear(Xd, codes, sw, N, 4, "W4A16"))
    ref = oracle.linear_a16(bf16_bits(tq.rotate_act_bf16(Xd)), codes_np(codes, 4, K), to_np(sw))
    assert rel_l2(Y, ref) <= REL_L2_Y


def test_empty_calls(tq):
    import torch
    X = torch.empty((0, 512), dtype=torch.bfloat16, device="cuda")
    codes, sw = gpu_weights(tq, wgen("gpu/empty/w", 16, 512), 8)
    Y = tq.linear(X, codes, sw, 16, 8, "W8A16")
    assert Y.shape == (0, 16)
    Y = tq.linear(to_dev_bf16(xgen("gpu/empty/x", 2, 512)), codes, sw, 0, 8, "W8A8")
    assert Y.shape == (2, 0)


def test_binding_refuses_buffers_smaller_than_their_sizes(tq):
    """The C ABI sees only pointers, so the binding checks that each tensor is
    as large, and of the type, that the call will read or write."""
    import torch
    M, N, K = 8, 256, 512
    X = to_dev_bf16(xgen("gpu/guard/x", M, K, XD))
    codes, sw = gpu_weights(tq, wgen("gpu/guard/w", N, K), 8)
    Xq, sx = tq.rotate_quant_act(X)
    with pytest.raises(ValueError):    # an fp32 product into a bf16 buffer
        tq.linear_q8(Xq, sx, codes, sw, N, 8, Y=torch.empty(M, N, dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(ValueError):    # too few rows
        tq.linear(X, codes, sw, N, 8, "W8A8", Y=torch.empty(M - 1, N, device="cuda"))
    with pytest.raises(ValueError):    # weights for fewer rows than N
        tq.linear(X, codes[: N // 2], sw, N, 8, "W8A16")
    with pytest.raises(ValueError):    # tiled operand smaller than its size
        At, sxt = tq.rotate_quant_act_tiled(X)
        tq.linear_tiled(At[:100], sxt, M, K, codes, sw, N, 8)
    assert tq.device_status() == 0


def test_device_status_clean(tq):
    assert tq.device_status() == 0
