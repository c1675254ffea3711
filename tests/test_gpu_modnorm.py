"""GPU parity of the modulated layer norm fused with the rotation and the
per-token quantiser (tq_modnorm_quant_act_tiled), against the oracle's O11
(fp64 norm, rounded to bf16) then O1+O2+O4.

The kernel computes the norm in fp32 (the pages keep norms in fp32) and rounds
h to bf16, so an h whose exact value lies within the fp32 error of a bf16
rounding boundary may round the other way.  The bars follow from that:
  - "near-tie" elements are those whose fp64 h lies within
    2^-17 (|h - shift| + |shift| + |mu| rstd |1 + scale|) of a bf16 rounding
    boundary: several times the fp32 error of the mean, the variance, rsqrtf
    and the fused multiply-add, a few parts in 10^7 of the terms h adds (their
    sum may cancel, so the error is bounded by the terms, not by |h|);
  - a row whose largest rotated value lies in a group with no near-tie
    element has its token scale within 2^-20 of the oracle's (the bar of the
    plain rotation); every row's scale is within 2^-8 (one flipped h_k moves
    each rotated value of its group by ulp(h_k) / 16 at most);
  - codes of groups with no near-tie element, in rows whose scale met the
    strict bar, follow the plain rotation's bar (at most 0.1% differ, each by
    at most 1); every code is within 2 of the oracle's;
  - where a whole row has no near-tie element, its codes equal, bit for bit,
    those of the unfused GPU route (the oracle's bf16 h through
    tq_rotate_quant_act_tiled): the two share the transform and quantiser.
"""
import zlib

import numpy as np
import pytest

import oracle
from dit_convrot_linear_gb300 import synth
from helpers import (CODE_FLIP_FRAC, REL_L2_Y, SCALE_REL, act_trailer, check_codes_close, rel_l2,
                     to_dev_bf16, to_np, untile_codes)

pytestmark = pytest.mark.gpu

XD = (1.0, 0.002, 40.0)     # DiT block inputs: 0.2% of channels x40
EPS = 1e-6
NEAR_REL = 2.0 ** -17
SCALE_LOOSE = 2.0 ** -8


def _modulation(K, tag):
    rng = np.random.default_rng(zlib.crc32(f"modnorm/{tag}/{K}".encode()))
    shift = rng.normal(0.0, 0.5, K).astype(np.float32)
    scale = rng.normal(0.0, 0.3, K).astype(np.float32)
    return shift, scale


def _dev_f32(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def _near_ties(X, shift, scale):
    """Boolean [M, K]: the fp64 h lies within NEAR_REL times the size of its
    terms of a bf16 rounding boundary (the midpoint of two neighbouring bf16
    values)."""
    sh = shift.astype(np.float64)
    x = oracle.bf16_to_f64(X)
    h = oracle.modnorm_f64(x, sh, scale.astype(np.float64), float(np.float32(EPS)))
    a = np.abs(h)
    # the terms of h, and the rounding of the mean carried through rstd
    # (window only: the expected values come from the oracle alone)
    rstd = 1.0 / np.sqrt(x.var(axis=1, keepdims=True) + EPS)
    mu_term = np.abs(x.mean(axis=1, keepdims=True)) * rstd * np.abs(1.0 + scale.astype(np.float64))
    size = np.abs(h - sh) + np.abs(sh) + mu_term
    nz = a > 0
    e = np.floor(np.log2(np.where(nz, a, 1.0)))
    ulp = np.exp2(e - 7)
    lo = np.floor(a / ulp) * ulp
    dist = np.abs(a - (lo + ulp / 2))
    return nz & (dist <= NEAR_REL * size)


def _check(tq, X, shift, scale, At, sx, rows=None):
    M, K = X.shape
    rows = np.arange(M) if rows is None else np.asarray(rows)
    Xr = X[rows]
    codes = untile_codes(At, M, K, rows=rows)
    rq, rs = oracle.modnorm_quant_act(Xr, shift, scale, EPS)
    got_s = to_np(sx)[rows].astype(np.float64)
    near = _near_ties(Xr, shift, scale)
    G = (K + 255) // 256
    gid = np.arange(K) // 256
    near_g = np.stack([near[:, gid == g].any(axis=1) for g in range(G)], axis=1)
    # the oracle's largest rotated value picks the group that sets the scale
    v = oracle.rotate_rows(oracle.modnorm_bf16(Xr, shift, scale, EPS))
    gmax = gid[np.argmax(np.abs(v), axis=1)]
    strict = ~near_g[np.arange(len(rows)), gmax]
    rel = np.where(rs == 0, np.abs(got_s), np.abs(got_s / np.where(rs == 0, 1, rs) - 1))
    assert np.all(rel <= SCALE_LOOSE), f"scale off by {rel.max()}"
    assert np.all(rel[strict] <= SCALE_REL), f"strict rows: scale off by {rel[strict].max()}"
    assert np.max(np.abs(codes - rq)) <= 2
    clean = strict[:, None] & ~near_g[:, gid]
    check_codes_close(codes[clean], rq[clean], frac=CODE_FLIP_FRAC)
    # rows without any near tie: the unfused GPU route gives the same bytes
    whole = ~near.any(axis=1)
    if whole.any():
        H = oracle.modnorm_bf16(Xr[whole], shift, scale, EPS)
        At2, sx2 = tq.rotate_quant_act_tiled(to_dev_bf16(H))
        assert np.array_equal(untile_codes(At2, int(whole.sum()), K), codes[whole])
        assert np.array_equal(to_np(sx2), to_np(sx)[rows[whole]])
    return {"strict_rows": float(strict.mean()), "near_frac": float(near.mean())}


SHAPES = [(300, 3072), (257, 4096 + 32), (5, 544), (64, 12288), (130, 896), (1024, 3072),
          (3, 16384), (3, 16384 - 128), (9, 32)]


@pytest.mark.parametrize("M,K", SHAPES)
def test_modnorm_fused_operand(tq, M, K):
    X = synth.tensor(f"gpu/modnorm/x{M}x{K}", M, K, *XD)
    shift, scale = _modulation(K, "shapes")
    At, sx = tq.modnorm_quant_act_tiled(to_dev_bf16(X), _dev_f32(shift), _dev_f32(scale), EPS)
    assert tq.device_status() == 0
    _check(tq, X, shift, scale, At, sx)


def test_modnorm_strided_rows_and_special_rows(tq):
    """X read through a strided view (row stride above K, offset start); a
    constant row and a zero row (variance 0: h is the shift), a row with a
    large mean (100 + N(0, 1): the two-pass variance keeps its spread), a
    row of one outlier; no modulation (a plain layer norm) in a second call."""
    M, K = 40, 3072 + 64
    big = synth.tensor("gpu/modnorm/strided", M, K + 72, *XD)
    big[0, :] = oracle.f64_to_bf16(1.375)
    big[1, :] = 0
    rng = np.random.default_rng(12)
    for k in range(K + 72):
        big[2, k] = oracle.f64_to_bf16(100.0 + rng.normal())
    big[3, :] = 0
    big[3, 8 + 777] = oracle.f64_to_bf16(-3.0)
    Xd = to_dev_bf16(big)[:, 8:8 + K]
    X = np.ascontiguousarray(big[:, 8:8 + K])
    for tag in ("mod", "plain"):
        shift, scale = _modulation(K, "strided")
        if tag == "plain":
            shift, scale = np.zeros(K, np.float32), np.zeros(K, np.float32)
        At, sx = tq.modnorm_quant_act_tiled(Xd, _dev_f32(shift), _dev_f32(scale), EPS)
        assert tq.device_status() == 0
        _check(tq, X, shift, scale, At, sx)
        # variance 0: the codes are those of the rotated shift
        codes = untile_codes(At, M, K, rows=[0, 1])
        ref = oracle.rotate_quant_act(np.tile(oracle.round_bf16(shift.astype(np.float64)), (2, 1)))[0]
        if tag == "plain":
            assert np.all(codes == 0) and np.all(to_np(sx)[:2] == 0)
        else:
            assert np.max(np.abs(codes - ref)) <= 1


def test_modnorm_fused_operand_full_size_sampled(tq):
    """The DiT up projection's operand at the size the bench times (M = 4032,
    K = 3072): sampled token rows against the oracle, and the trailer's exact
    row sums on them."""
    M, K = 4032, 3072
    X = synth.tensor("gpu/modnorm/full", M, K, *XD)
    shift, scale = _modulation(K, "full")
    At, sx = tq.modnorm_quant_act_tiled(to_dev_bf16(X), _dev_f32(shift), _dev_f32(scale), EPS)
    assert tq.device_status() == 0
    rows = np.sort(np.random.default_rng(13).choice(M, 48, replace=False))
    _check(tq, X, shift, scale, At, sx, rows=rows)
    codes = untile_codes(At, M, K, rows=rows)
    tr = act_trailer(tq, At, M, K)
    assert int(tr[0]) >= int(np.abs(codes).sum(axis=1).max())
    assert int(tr[6]) >= int((codes * codes).sum(axis=1).max())


def test_modnorm_operand_feeds_the_product(tq):
    """block input -> fused modulated-norm operand -> both-tiled QKV-shaped
    product (4-bit weights), against the oracle's int32 sums on the same codes
    (exact) and its Y."""
    M, N, K = 260, 576, 3072
    X = synth.tensor("gpu/modnorm/prod/x", M, K, *XD)
    shift, scale = _modulation(K, "prod")
    W = synth.tensor("gpu/modnorm/prod/w", N, K, 0.015, 0.005, 30.0)
    codes_w, sw = tq.quantize_weights(to_dev_bf16(W), 4)
    At, sx = tq.modnorm_quant_act_tiled(to_dev_bf16(X), _dev_f32(shift), _dev_f32(scale), EPS)
    Wt = tq.tile_weights(codes_w, N, K, 4)
    acc = to_np(tq.linear_tt(At, sx, M, K, Wt, sw, N, 4, out="i32"))
    xq = untile_codes(At, M, K).astype(np.int8)
    wc = oracle.weight_codes(to_np(codes_w).view(np.uint8), 4, K)
    ref_acc, ref_Y = oracle.linear_a8(xq, to_np(sx), wc, to_np(sw))
    assert np.array_equal(acc, ref_acc)
    Y = to_np(tq.linear_tt(At, sx, M, K, Wt, sw, N, 4))
    assert rel_l2(Y, ref_Y) <= REL_L2_Y
    assert tq.device_status() == 0


def test_modnorm_deterministic(tq):
    import torch
    M, K = 1024, 3072
    X = to_dev_bf16(synth.tensor("gpu/modnorm/det", M, K, *XD))
    shift, scale = _modulation(K, "det")
    a = tq.modnorm_quant_act_tiled(X, _dev_f32(shift), _dev_f32(scale), EPS)
    b = tq.modnorm_quant_act_tiled(X, _dev_f32(shift), _dev_f32(scale), EPS)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
