"""GPU parity at the shapes of one DiT block's projection chain: 4-bit weights
with int8 activations, M = 1024 token rows (a 512 x 512 image), the four
projections QKV 3072 -> 9216, out 3072 -> 3072, gate+up 3072 -> 24576 and
down 12288 -> 3072 (tensai docs "画像生成", section "幅とメモリ": 32 blocks,
1024 tokens at 512 x 512, 4-bit weights with -q4; TensorFold PR #948,
"Receipts": the projections are most of a forward).

At these sizes the product runs its persistent schedule over many tiles per
CTA pair with the 4-bit codes widened on the way in (converting product) or
once at set-up (both tiled), and the out and down projections leave most CTA
pairs without a second tile.  Weights follow the batched-decode recipe
(N(0, 0.015), 0.5% of columns x30), activations the DiT recipe (N(0, 1), 0.2%
of channels x40).

Bars: int32 sums bit-exact against the oracle (O5) on the GPU's own int8
codes, fp32 Y within relative L2 1e-4.  Large shapes are checked on sampled
(m, n) pairs the oracle computes one by one; the out projection, whose tiles
cover only part of the GPU, is checked in full.
"""
import numpy as np
import pytest

import oracle
from dit_convrot_linear_gb300 import synth
from helpers import REL_L2_Y, rel_l2, to_dev_bf16, to_np, untile_codes

pytestmark = pytest.mark.gpu

M = 1024
WB = (0.015, 0.005, 30.0)
XD = (1.0, 0.002, 40.0)
CHAIN = {p.name: (p.N, p.K) for p in synth.CHAIN.projs}


def _pairs(N, seed, n=1500):
    rng = np.random.default_rng(seed)
    pm = np.concatenate([rng.integers(0, M, n), [0, M - 1, M - 1, 0]])
    pn = np.concatenate([rng.integers(0, N, n), [0, N - 1, 0, N - 1]])
    return pm, pn


def _setup(tq, name):
    N, K = CHAIN[name]
    W = synth.tensor(f"gpu/chain/{name}/w", N, K, *WB)
    X = to_dev_bf16(synth.tensor(f"gpu/chain/{name}/x", M, K, *XD))
    codes, sw = tq.quantize_weights(to_dev_bf16(W), 4)
    return N, K, X, codes, sw


@pytest.mark.parametrize("name", ["qkv", "out", "gateup", "down"])
def test_chain_projection_w4a8(tq, name):
    """Converting product (int8 codes and the tiled activation operand) and
    the both-tiled product at the chain's shape: the same exact int32 sums,
    equal to the oracle's on sampled pairs, and Y within the fp32 bar."""
    N, K, X, codes, sw = _setup(tq, name)
    Xq, sx = tq.rotate_quant_act(X)
    At, sxt = tq.rotate_quant_act_tiled(X)
    Wt = tq.tile_weights(codes, N, K, 4)
    acc_q8 = to_np(tq.linear_q8(Xq, sx, codes, sw, N, 4, out="i32"))
    acc_t = to_np(tq.linear_tiled(At, sxt, M, K, codes, sw, N, 4, out="i32"))
    acc_tt = to_np(tq.linear_tt(At, sxt, M, K, Wt, sw, N, 4, out="i32"))
    assert np.array_equal(acc_t, acc_q8)
    assert np.array_equal(acc_tt, acc_q8)
    xq, s_x, wc, s_w = to_np(Xq), to_np(sx), oracle.weight_codes(to_np(codes), 4, K), to_np(sw)
    pm, pn = _pairs(N, N + K)
    ref_acc, ref_Y = oracle.linear_a8_pairs(xq, s_x, wc, s_w, pm, pn)
    assert np.array_equal(acc_tt[pm, pn], ref_acc)
    Y = to_np(tq.linear(X, codes, sw, N, 4, "W8A8"))
    Ytt = to_np(tq.linear_tt(At, sxt, M, K, Wt, sw, N, 4))
    assert rel_l2(Y[pm, pn], ref_Y) <= REL_L2_Y
    assert rel_l2(Ytt[pm, pn], ref_Y) <= REL_L2_Y
    assert np.array_equal(Y.view(np.uint32), Ytt.view(np.uint32))
    assert tq.device_status() == 0


def test_chain_out_projection_full(tq):
    """The out projection (48 tiles of 256 x 256 on the GPU's CTA pairs),
    every output against the oracle."""
    N, K, X, codes, sw = _setup(tq, "out")
    At, sx = tq.rotate_quant_act_tiled(X)
    Wt = tq.tile_weights(codes, N, K, 4)
    acc = to_np(tq.linear_tt(At, sx, M, K, Wt, sw, N, 4, out="i32"))
    Y = to_np(tq.linear_tt(At, sx, M, K, Wt, sw, N, 4))
    xq = untile_codes(At, M, K).astype(np.int8)
    ref_acc, ref_Y = oracle.linear_a8(xq, to_np(sx), oracle.weight_codes(to_np(codes), 4, K), to_np(sw))
    assert np.array_equal(acc, ref_acc)
    assert rel_l2(Y, ref_Y) <= REL_L2_Y


def test_chain_down_from_gate_and_up(tq):
    """gate+up product (bf16 out, the two halves of one [M, 24576] output) ->
    the SwiGLU operand made from its halves in one pass -> down product, as
    the block runs them; the down sums against the oracle on the operand's
    own codes, and those codes against the oracle's SwiGLU and quantiser on
    the same gate/up values."""
    import torch
    Ngu, Kgu, X, cgu, sgu = _setup(tq, "gateup")
    Nd, Kd = CHAIN["down"]
    assert Ngu == 2 * Kd
    Wd = synth.tensor("gpu/chain/down/w", Nd, Kd, *WB)
    cd, sd = tq.quantize_weights(to_dev_bf16(Wd), 4)
    At, sx = tq.rotate_quant_act_tiled(X)
    GU = tq.linear_tt(At, sx, M, Kgu, tq.tile_weights(cgu, Ngu, Kgu, 4), sgu, Ngu, 4, out="bf16")
    Ad, sxd = tq.swiglu_quant_act_tiled(GU[:, :Kd], GU[:, Kd:])
    Wtd = tq.tile_weights(cd, Nd, Kd, 4)
    acc = to_np(tq.linear_tt(Ad, sxd, M, Kd, Wtd, sd, Nd, 4, out="i32"))
    Y = to_np(tq.linear_tt(Ad, sxd, M, Kd, Wtd, sd, Nd, 4))
    rows = np.sort(np.random.default_rng(3).choice(M, 32, replace=False))
    codes = untile_codes(Ad, M, Kd, rows=rows)
    gu = GU.view(torch.int16).cpu().numpy().view(np.uint16)
    rq, rs = oracle.swiglu_quant_act(np.ascontiguousarray(gu[rows, :Kd]),
                                     np.ascontiguousarray(gu[rows, Kd:]))
    d = np.abs(codes - rq.astype(np.int64))
    assert d.max() <= 1 and np.count_nonzero(d) <= 1e-3 * d.size
    pm = np.random.default_rng(4).integers(0, len(rows), 1500)
    pn = np.random.default_rng(5).integers(0, Nd, 1500)
    ref_acc, ref_Y = oracle.linear_a8_pairs(codes.astype(np.int8), to_np(sxd)[rows],
                                            oracle.weight_codes(to_np(cd), 4, Kd), to_np(sd), pm, pn)
    assert np.array_equal(acc[rows[pm], pn], ref_acc)
    assert rel_l2(Y[rows[pm], pn], ref_Y) <= REL_L2_Y
    assert tq.device_status() == 0
