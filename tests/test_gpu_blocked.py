"""GPU parity of the block-scaled weights (tq_quantize_weights_blocked) and
their decode product (tq_linear_blocked) against the CPU oracle (O9, O10).

Bars: codes and block scales bit-exact (the quantiser's fp64 arithmetic is
the oracle's); fp32 Y within relative L2 1e-4 of the oracle on the GPU's
codes, both with the oracle's rotated operand and with the GPU's own; bf16 Y
within 1 bf16 ulp of the oracle's value rounded.
"""
import numpy as np
import pytest

import oracle
from dit_convrot_linear_gb300 import synth
from helpers import REL_L2_Y, bf16_bits, bf16_ulp_diff, rel_l2, to_dev_bf16, to_np

pytestmark = pytest.mark.gpu

WD = (0.02, 0.01, 20.0)     # decode weights: N(0, 0.02), 1% columns x20
XD = (1.0, 0.002, 40.0)     # activations: N(0, 1), 0.2% columns x40


def gpu_blocked(tq, W, bits, G, rotate):
    codes, sw = tq.quantize_weights_blocked(to_dev_bf16(W), bits, G, rotate)
    c = to_np(codes)
    return codes, sw, oracle.weight_codes(c.view(np.int8) if bits == 8 else c.view(np.uint8), bits,
                                          W.shape[1])


QSHAPES = [(64, 896, 8, 32, 1), (64, 896, 4, 32, 1), (33, 1024, 4, 64, 1), (17, 4096 + 128, 8, 128, 0),
           (40, 512, 4, 256, 1), (5, 32, 8, 32, 0), (5, 32, 4, 32, 1), (24, 4864, 4, 64, 1),
           (24, 4864, 8, 32, 0), (9, 2304 + 64, 4, 32, 0)]


@pytest.mark.parametrize("N,K,bits,G,rotate", QSHAPES)
def test_blocked_quantiser_is_bit_exact(tq, N, K, bits, G, rotate):
    W = synth.tensor(f"gpu/blkq/{N}x{K}", N, K, *WD)
    codes, sw, _ = gpu_blocked(tq, W, bits, G, rotate)
    rq, rs = oracle.quantize_weights_blocked(W, bits, G, bool(rotate))
    assert np.array_equal(to_np(codes).view(np.uint8), rq.view(np.uint8))
    assert np.array_equal(to_np(sw).view(np.uint32), rs.view(np.uint32))


def check_product(tq, X, Wc, sw, G, rotate, Y):
    Xa_orc = oracle.rotate_act_bf16(X) if rotate else X
    ref = oracle.linear_a16_blocked(Xa_orc, Wc, to_np(sw), G)
    assert rel_l2(to_np(Y), ref) <= REL_L2_Y
    if rotate:
        Xd = to_dev_bf16(X)
        ref_gpu = oracle.linear_a16_blocked(bf16_bits(tq.rotate_act_bf16(Xd)), Wc, to_np(sw), G)
        assert rel_l2(to_np(Y), ref_gpu) <= REL_L2_Y
    return ref


PSHAPES = [(1, 4864, 896, 8, 32, 1), (1, 896, 4864, 4, 32, 1), (2, 300, 4096 + 32, 8, 32, 0),
           (3, 77, 1024, 4, 64, 1), (5, 129, 2304, 8, 256, 1), (8, 100, 896, 4, 128, 1),
           (8, 257, 896, 8, 32, 0), (4, 33, 10752, 4, 32, 1), (1, 40, 32, 8, 32, 1), (7, 11, 4864, 8, 64, 0)]


@pytest.mark.parametrize("M,N,K,bits,G,rotate", PSHAPES)
def test_blocked_product_matches_the_oracle(tq, M, N, K, bits, G, rotate):
    W = synth.tensor(f"gpu/blkp/w{N}x{K}", N, K, *WD)
    X = synth.tensor(f"gpu/blkp/x{M}x{K}", M, K, *XD)
    codes, sw, Wc = gpu_blocked(tq, W, bits, G, rotate)
    Y = tq.linear_blocked(to_dev_bf16(X), codes, sw, N, bits, G, bool(rotate))
    assert tq.device_status() == 0
    check_product(tq, X, Wc, sw, G, rotate, Y)


def test_blocked_product_bf16_output_within_one_ulp(tq):
    M, N, K = 3, 500, 2304
    W = synth.tensor("gpu/blkb/w", N, K, *WD)
    X = synth.tensor("gpu/blkb/x", M, K, *XD)
    for bits, G, rotate in ((8, 32, 0), (4, 64, 1)):
        codes, sw, Wc = gpu_blocked(tq, W, bits, G, rotate)
        Y = tq.linear_blocked(to_dev_bf16(X), codes, sw, N, bits, G, bool(rotate), out="bf16")
        Xa = bf16_bits(tq.rotate_act_bf16(to_dev_bf16(X))) if rotate else X
        ref = oracle.linear_a16_blocked(Xa, Wc, to_np(sw), G)
        assert bf16_ulp_diff(bf16_bits(Y), oracle.round_bf16(ref)).max() <= 1


def test_blocked_strided_input_padded_output_zero_rows(tq):
    import torch
    M, N, K = 3, 200, 1024
    big = synth.tensor("gpu/blkv/x", M, K + 64, *XD)
    W = synth.tensor("gpu/blkv/w", N, K, *WD)
    W[7] = 0                                          # a zero row: scales 0, codes 0, Y 0
    codes, sw, Wc = gpu_blocked(tq, W, 4, 32, 1)
    assert torch.all(sw[7] == 0)
    Xd = to_dev_bf16(big)[:, 8:8 + K]
    Yfull = torch.full((M, N + 24), 7.0, dtype=torch.float32, device="cuda")
    Y = Yfull[:, :N]
    tq.linear_blocked(Xd, codes, sw, N, 4, 32, True, Y=Y)
    check_product(tq, np.ascontiguousarray(big[:, 8:8 + K]), Wc, sw, 32, 1, Y)
    assert torch.all(Y[:, 7] == 0)
    assert torch.all(Yfull[:, N:] == 7.0)             # the stride padding is untouched
    # empty calls launch nothing and touch nothing
    Y0 = torch.full((0, N), 1.0, device="cuda")
    tq.linear_blocked(Xd[:0], codes, sw, N, 4, 32, True, Y=Y0)
    tq.linear_blocked(Xd, codes, sw, 0, 4, 32, True, Y=Yfull[:, :0])
    assert torch.all(Yfull[:, N:] == 7.0)


def test_blocked_large_stream_sampled(tq):
    """A weight matrix larger than L2 (16384 x 16384 int8, 268 MB): sampled
    rows against the oracle on the GPU's codes."""
    import torch
    N, K = 16384, 16384
    Wh = synth.tensor("gpu/blkl/w", N, K, *WD)
    Wd = to_dev_bf16(Wh)
    X = synth.tensor("gpu/blkl/x", 1, K, *XD)
    for bits, G, rotate in ((8, 32, 0), (4, 64, 1)):
        codes, sw = tq.quantize_weights_blocked(Wd, bits, G, rotate)
        Y = to_np(tq.linear_blocked(to_dev_bf16(X), codes, sw, N, bits, G, bool(rotate)))
        rows = np.array([0, 1, 4095, 8191, 12000, 16383])
        sel = torch.as_tensor(rows, device="cuda")
        c = to_np(codes[sel])
        Wc = oracle.weight_codes(c.view(np.int8) if bits == 8 else c.view(np.uint8), bits, K)
        Xa = oracle.rotate_act_bf16(X) if rotate else X
        ref = oracle.linear_a16_blocked(Xa, Wc, to_np(sw[sel]), G)
        assert rel_l2(Y[:, rows], ref) <= REL_L2_Y
        # the quantiser on the same sampled rows
        rq, rs = oracle.quantize_weights_blocked(Wh[rows], bits, G, bool(rotate))
        assert np.array_equal(c.view(np.uint8), rq.view(np.uint8))
        assert np.array_equal(to_np(sw[sel]).view(np.uint32), rs.view(np.uint32))
        del codes, sw
    assert tq.device_status() == 0


def test_blocked_product_refuses_rows_beyond_shared_memory(tq):
    import torch
    K, N = 8192, 64                                   # 8 tokens x 8192 x 4 B = 256 KB > 227 KB
    W = torch.zeros((N, K), dtype=torch.bfloat16, device="cuda")
    codes, sw = tq.quantize_weights_blocked(W, 8, 32, True)
    X = torch.zeros((8, K), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(RuntimeError, match="TQ_ERR_SHAPE"):
        tq.linear_blocked(X, codes, sw, N, 8, 32, True)
    Y = tq.linear_blocked(X[:4], codes, sw, N, 8, 32, True)   # 4 tokens: 128 KB fits
    assert torch.all(Y == 0)


def test_blocked_product_graph_replay_is_deterministic(tq):
    import torch
    M, N, K = 2, 4864, 896
    W = synth.tensor("gpu/blkg/w", N, K, *WD)
    X = to_dev_bf16(synth.tensor("gpu/blkg/x", M, K, *XD))
    codes, sw, _ = gpu_blocked(tq, W, 4, 32, 1)
    Y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    tq.linear_blocked(X, codes, sw, N, 4, 32, True, Y=Y)
    first = to_np(Y).copy()
    Y.fill_(float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            tq.linear_blocked(X, codes, sw, N, 4, 32, True, Y=Y, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(first.view(np.uint32), to_np(Y).view(np.uint32))


# int4 on matrices that fill the GPU (the two-rows-a-warp variants and their
# last, ragged row pair), K with a partial last group, one to eight tokens,
# both formats, fp32 and bf16 outputs
TC4 = [(1, 4864, 896, 32, 1), (2, 5000, 2304 + 32, 32, 1), (3, 4870, 1024, 64, 0), (8, 4864, 896, 128, 1),
       (5, 4900, 544, 32, 1), (4, 4880, 2304 + 64, 32, 0), (1, 6000, 4096, 256, 1), (6, 4864, 2304, 32, 0),
       (1, 7297, 896, 32, 1), (2, 8001, 544, 32, 0)]


@pytest.mark.parametrize("M,N,K,G,rotate", [(1, 7297, 896, 32, 0), (2, 8001, 2304 + 64, 64, 1)])
def test_blocked_int8_two_rows_a_warp_ragged(tq, M, N, K, G, rotate):
    """N large enough for two rows a warp, and odd: the last warp's second row
    is past N (loads nothing, stores nothing)."""
    W = synth.tensor(f"gpu/blk2r/w{N}x{K}", N, K, *WD)
    X = synth.tensor(f"gpu/blk2r/x{M}x{K}", M, K, *XD)
    codes, sw, Wc = gpu_blocked(tq, W, 8, G, rotate)
    Y = tq.linear_blocked(to_dev_bf16(X), codes, sw, N, 8, G, bool(rotate))
    assert tq.device_status() == 0
    check_product(tq, X, Wc, sw, G, rotate, Y)


@pytest.mark.parametrize("M,N,K,G,rotate", TC4)
def test_blocked_int4_full_width_matches_the_oracle(tq, M, N, K, G, rotate):
    W = synth.tensor(f"gpu/blkfw/w{N}x{K}", N, K, 0.015, 0.005, 30.0)
    X = synth.tensor(f"gpu/blkfw/x{M}x{K}", M, K, *XD)
    codes, sw, Wc = gpu_blocked(tq, W, 4, G, rotate)
    Y = tq.linear_blocked(to_dev_bf16(X), codes, sw, N, 4, G, bool(rotate))
    assert tq.device_status() == 0
    check_product(tq, X, Wc, sw, G, rotate, Y)
    Yb = tq.linear_blocked(to_dev_bf16(X), codes, sw, N, 4, G, bool(rotate), out="bf16")
    Xa = bf16_bits(tq.rotate_act_bf16(to_dev_bf16(X))) if rotate else X
    ref = oracle.linear_a16_blocked(Xa, Wc, to_np(sw), G)
    assert bf16_ulp_diff(bf16_bits(Yb), oracle.round_bf16(ref)).max() <= 1


@pytest.mark.parametrize("bits", [8, 4])
def test_one_block_per_row_is_the_per_row_format(tq, bits):
    """With G = K (one block a row) and the rotation, the blocked quantiser is
    the per-row one: the same codes and scales bit for bit, and the blocked
    product agrees with the per-row A16 product to rounding."""
    M, N, K = 3, 700, 256
    W = synth.tensor(f"gpu/blkrow/w{bits}", N, K, *WD)
    X = to_dev_bf16(synth.tensor(f"gpu/blkrow/x{bits}", M, K, *XD))
    cb, sb = tq.quantize_weights_blocked(to_dev_bf16(W), bits, K, True)
    cr, sr = tq.quantize_weights(to_dev_bf16(W), bits)
    assert np.array_equal(to_np(cb).view(np.uint8), to_np(cr).view(np.uint8))
    assert np.array_equal(to_np(sb)[:, 0].view(np.uint32), to_np(sr).view(np.uint32))
    Yb = to_np(tq.linear_blocked(X, cb, sb, N, bits, K, True))
    Yr = to_np(tq.linear(X, cr, sr, N, bits, "W8A16" if bits == 8 else "W4A16"))
    assert rel_l2(Yb, Yr) <= 1e-5
