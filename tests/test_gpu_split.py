"""GPU checks of the both-tiled product with split tiles (tq_linear_tt_split).

When a product's 256 x 256 output tiles leave the last wave of CTA pairs
mostly idle, the K steps of the last waves are shared by every pair: a pair
holding part of a tile stores its exact int32 partial sums, and the pair
holding the tile's last K step adds them.  Integer sums do not depend on the
order of addition, so every output must be bit-identical to the unsplit
product (and its int32 sums equal to the oracle's), whatever the split.  The
shapes cover a tile shared by every pair (one tile, 192 K steps), the DiT
block chain's down projection (48 tiles, long K), chunked accumulation (8-bit
weights over 12288 columns), ragged sizes with a K tail, bf16 output, the
fused epilogue in place, products whose whole waves stay whole and whose last
wave is split (the DiT down projection), and shapes the library leaves
unsplit (short K), which must be unchanged too.  The workspace's flags must be zero again after each
call, so the same workspace serves the next call.
"""
import numpy as np
import pytest

import oracle
from dit_convrot_linear_gb300 import synth
from helpers import REL_L2_Y, rel_l2, to_dev_bf16, to_np, untile_codes

pytestmark = pytest.mark.gpu

WD = (0.02, 0.01, 20.0)
WB = (0.015, 0.005, 30.0)
XD = (1.0, 0.002, 40.0)


def _flags_zero(ws):
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    nflag = (sms // 2) * 2 * 12          # [pairs][2 CTAs][12 drain warps] words
    return bool(torch.all(ws.view(torch.int32)[:nflag] == 0).item())


def _operands(tq, M, N, K, bits, tag):
    X = to_dev_bf16(synth.tensor(f"gpu/split/{tag}/x{M}x{K}", M, K, *XD))
    W = synth.tensor(f"gpu/split/{tag}/w{N}x{K}", N, K, *(WD if bits == 8 else WB))
    codes, sw = tq.quantize_weights(to_dev_bf16(W), bits)
    At, sx = tq.rotate_quant_act_tiled(X)
    Wt = tq.tile_weights(codes, N, K, bits)
    return At, sx, codes, sw, Wt


SHAPES = [
    (64, 256, 12288, 8),       # one tile, its 192 K steps over every pair
    (1024, 3072, 12288, 4),    # chain down projection: 48 tiles, long K (split)
    (1024, 3072, 12288, 8),    # the same with 8-bit weights: chunked exact accumulation
    (257, 300, 12288 + 32, 8), # ragged rows and columns, a K tail, 4 tiles split
    (1024, 3072, 3072, 4),     # chain out projection: short K, left whole
    (4032, 3072, 12288, 8),    # DiT down: 192 tiles, two whole waves, the last wave's 40 split
    (900, 5400, 12288 + 32, 8),  # 88 tiles: one whole wave, 12 split; ragged, a K tail
    (1024, 5120, 8192, 4),     # 80 tiles: one whole wave, 4 split over every pair
]


@pytest.mark.parametrize("M,N,K,bits", SHAPES)
def test_split_matches_unsplit_bit_for_bit(tq, M, N, K, bits):
    import torch
    At, sx, codes, sw, Wt = _operands(tq, M, N, K, bits, "eq")
    ws = tq.split_workspace()
    acc = to_np(tq.linear_tt(At, sx, M, K, Wt, sw, N, bits, out="i32"))
    for call in range(2):          # the same workspace twice in a row
        acc_s = to_np(tq.linear_tt(At, sx, M, K, Wt, sw, N, bits, out="i32", split=ws))
        assert np.array_equal(acc_s, acc), f"call {call}"
        assert _flags_zero(ws)
    Y = to_np(tq.linear_tt(At, sx, M, K, Wt, sw, N, bits))
    Ys = to_np(tq.linear_tt(At, sx, M, K, Wt, sw, N, bits, split=ws))
    assert np.array_equal(Ys.view(np.uint32), Y.view(np.uint32))
    Yb = tq.linear_tt(At, sx, M, K, Wt, sw, N, bits, out="bf16")
    Ybs = tq.linear_tt(At, sx, M, K, Wt, sw, N, bits, out="bf16", split=ws)
    assert torch.equal(Ybs.view(torch.int16), Yb.view(torch.int16))
    assert _flags_zero(ws)
    # and the int32 sums against the oracle on sampled pairs
    rng = np.random.default_rng(M + N + K)
    pm = np.concatenate([rng.integers(0, M, 600), [0, M - 1]])
    pn = np.concatenate([rng.integers(0, N, 600), [N - 1, 0]])
    xq = untile_codes(At, M, K).astype(np.int8)
    wc = oracle.weight_codes(to_np(codes), bits, K)
    ref_acc, ref_Y = oracle.linear_a8_pairs(xq, to_np(sx), wc, to_np(sw), pm, pn)
    assert np.array_equal(acc_s[pm, pn], ref_acc)
    assert rel_l2(Ys[pm, pn], ref_Y) <= REL_L2_Y
    assert tq.device_status() == 0


def test_split_epilogue_in_place(tq):
    """The gated residual fused into the split product, updating a bf16
    residual stream in place: the same bytes as the unsplit product."""
    import torch
    M, N, K, bits = 1024, 3072, 12288, 4
    At, sx, codes, sw, Wt = _operands(tq, M, N, K, bits, "epi")
    rng = np.random.default_rng(9)
    gate = torch.from_numpy(rng.normal(0, 1.0, N).astype(np.float32)).cuda()
    bias = torch.from_numpy(rng.normal(0, 2.0, N).astype(np.float32)).cuda()
    R0 = torch.from_numpy(rng.normal(0, 30.0, (M, N)).astype(np.float32)).cuda().to(torch.bfloat16)
    R1, R2 = R0.clone(), R0.clone()
    ws = tq.split_workspace()
    tq.linear_tt_ex(At, sx, M, K, Wt, sw, N, bits, Y=R1, out="bf16", gate=gate, bias=bias, residual=R1)
    tq.linear_tt_ex(At, sx, M, K, Wt, sw, N, bits, Y=R2, out="bf16", gate=gate, bias=bias, residual=R2,
                    split=ws)
    assert torch.equal(R1.view(torch.int16), R2.view(torch.int16))
    assert _flags_zero(ws)
    assert tq.device_status() == 0


def test_split_chain_projections_full(tq):
    """The chain's gate+up (384 tiles: the last, nearly empty wave split) and
    QKV (144 tiles, left whole) through the split entry point: the same int32
    sums as without it."""
    ws = None
    for (M, N, K) in [(1024, 24576, 3072), (1024, 9216, 3072)]:
        At, sx, codes, sw, Wt = _operands(tq, M, N, K, 4, "chain")
        if ws is None:
            ws = tq.split_workspace()
        a = to_np(tq.linear_tt(At, sx, M, K, Wt, sw, N, 4, out="i32"))
        b = to_np(tq.linear_tt(At, sx, M, K, Wt, sw, N, 4, out="i32", split=ws))
        assert np.array_equal(a, b)
        assert _flags_zero(ws)
    assert tq.device_status() == 0


def test_split_deterministic(tq):
    M, N, K, bits = 4032, 3072, 12288, 8
    At, sx, codes, sw, Wt = _operands(tq, M, N, K, bits, "det")
    ws = tq.split_workspace()
    a = to_np(tq.linear_tt(At, sx, M, K, Wt, sw, N, bits, split=ws))
    b = to_np(tq.linear_tt(At, sx, M, K, Wt, sw, N, bits, split=ws))
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
