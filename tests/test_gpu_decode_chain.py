"""GPU parity of a dependent decode chain (M = 1): gate (896 -> 4864) then
down (4864 -> 896) through three layer sets, each call's input the previous
call's bf16 output, in one CUDA graph as the bench runs it.  Every call is
checked against the oracle's O6 on the GPU's own input for that call (so a
rounding difference in one call does not travel into the next one's check):
bf16 Y within a16_close's bar (one bf16 step, plus one x' rounding flip).  Both
weight formats; the per-call kernels release the next launch before their
dependency wait, so this also checks that no call reads its input before the
previous call has written it."""
import numpy as np
import pytest

import oracle
from dit_convrot_linear_gb300 import synth
from helpers import REL_L2_Y, bf16_bits, bf16_ulp_diff, rel_l2, to_dev_bf16, to_np

pytestmark = pytest.mark.gpu

WD = (0.02, 0.01, 20.0)


def a16_close(got_bits, x_bits, wc, sw):
    """bf16 Y of an A16 product against the oracle's O6 on the same input,
    element by element: |Y - ref| at most one bf16 step of ref (the fp32 sum
    may round to the other neighbour) plus the most that one flip of an x'
    rounding can move it (the kernel rotates in fp32: an x'_j within its
    rounding error of a bf16 tie may round the other way, moving Y_n by one
    bf16 step of x'_j times |q_nj| s_n).  A wrong index, scale or operand
    moves Y by its own size.  Returns the worst excess (<= 0 passes)."""
    xr = oracle.rotate_act_bf16(x_bits)
    ref = oracle.linear_a16(xr, wc, sw)
    got = oracle.bf16_to_f64(got_bits)
    xa = np.abs(oracle.bf16_to_f64(xr)).max(axis=1, keepdims=True)
    flip = 2.0 ** -8 * xa * np.abs(wc).max(axis=1)[None, :].astype(np.float64) * sw.astype(np.float64)[None, :]
    a = np.abs(ref)
    step = np.exp2(np.floor(np.log2(np.where(a > 0, a, 2.0 ** -133))) - 7)
    return float(np.max(np.abs(got - ref) - step - flip)), ref


def swiglu_down_close(got_bits, ref):
    """bf16 Y of a decode product of a SwiGLU input against the oracle's
    value on the same gate and up rows.  The kernel's h may differ from the
    oracle's by one bf16 step where h lies within its silu error (under 2^-19
    relative) of a rounding tie, a few elements a row; each such flip moves
    Y_n by about 2^-8 |h_k| |w_nk|, together well under 2^-9 of Y's RMS.  The
    bar: a relative L2 error of 2^-8 (the bf16 output rounding alone gives up
    to 2^-9), and every element within one bf16 step plus 2^-7 of the RMS."""
    got = oracle.bf16_to_f64(got_bits)
    a = np.abs(ref)
    step = np.exp2(np.floor(np.log2(np.where(a > 0, a, 2.0 ** -133))) - 7)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    return rel_l2(got, ref) <= 2.0 ** -8 and bool(np.all(np.abs(got - ref) <= step + 2.0 ** -7 * rms)), got


@pytest.mark.parametrize("bits", [8, 4])
def test_dependent_chain_each_call_against_the_oracle(tq, bits):
    import torch
    mode = "W8A16" if bits == 8 else "W4A16"
    shapes = [(4864, 896), (896, 4864)] * 3
    weights = []
    for i, (N, K) in enumerate(shapes):
        codes, sw = tq.quantize_weights(to_dev_bf16(synth.tensor(f"gpu/dchain/w{i}", N, K, *WD)), bits)
        weights.append((N, K, codes, (sw / 8.0).contiguous()))      # keeps the chain's values O(1)
    x0 = to_dev_bf16(synth.tensor("gpu/dchain/x", 1, 896, 1.0))
    ins = [torch.empty((1, K), dtype=torch.bfloat16, device="cuda") for (N, K, _, _) in weights]
    outs = [torch.empty((1, N), dtype=torch.bfloat16, device="cuda") for (N, K, _, _) in weights]
    bufs = [torch.empty((1, 4864), dtype=torch.bfloat16, device="cuda"),
            torch.empty((1, 896), dtype=torch.bfloat16, device="cuda")]

    def run():
        x = x0
        for i, (N, K, codes, sw) in enumerate(weights):
            y = bufs[i % 2]
            ins[i].copy_(x)
            tq.linear(x, codes, sw, N, bits, mode, Y=y, out="bf16")
            outs[i].copy_(y)
            x = y
    run()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            run()
    torch.cuda.current_stream().wait_stream(s)
    for o in outs:
        o.zero_()
    g.replay()
    torch.cuda.synchronize()
    for i, (N, K, codes, sw) in enumerate(weights):
        xb = bf16_bits(ins[i])
        assert np.any(xb != 0)
        c = to_np(codes)
        wc = oracle.weight_codes(c.view(np.int8) if bits == 8 else c.view(np.uint8), bits, K)
        worst, _ = a16_close(bf16_bits(outs[i]), xb, wc, to_np(sw))
        assert worst <= 0, f"call {i}: {worst}"
        if i > 0:   # the chain: this call's input is the previous call's output
            assert np.array_equal(xb, bf16_bits(outs[i - 1]))
    assert tq.device_status() == 0


# ---- the decode product of a SwiGLU input (tq_linear_swiglu)

TIE_WINDOW = 2.0 ** -16


def _near_ties(h):
    """Boolean: the fp64 h lies within TIE_WINDOW |h| of a bf16 rounding
    boundary (the midpoint of two neighbouring bf16 values).  The kernel's
    silu uses the hardware's approximate exponential and division, a relative
    error under 2^-19 for the gate values here, so only such h may round to
    the other bf16 neighbour than the exact value does."""
    a = np.abs(h)
    nz = a > 0
    e = np.floor(np.log2(np.where(nz, a, 1.0)))
    ulp = np.exp2(e - 7)
    mid = np.floor(a / ulp) * ulp + ulp / 2
    return nz & (np.abs(a - mid) <= TIE_WINDOW * a)


def _swiglu_inputs(tag, M, K):
    """Seeded gate and up rows, with each up value whose h = silu(g) u lies
    near a bf16 rounding tie moved by one bf16 step (an input choice made with
    the oracle alone), so the kernel's h must equal the oracle's bit for bit."""
    G = synth.tensor(f"gpu/dswiglu/g/{tag}", M, K, 1.5, 0.0, 1.0)
    U = synth.tensor(f"gpu/dswiglu/u/{tag}", M, K, 1.0, 0.002, 40.0)
    g = oracle.bf16_to_f64(G)
    for _ in range(16):
        near = _near_ties(oracle.swiglu_f64(g, oracle.bf16_to_f64(U)))
        if not near.any():
            return G, U
        U[near] = U[near] + 1          # one step away from zero in magnitude
    raise AssertionError("could not move every h off a rounding tie")


SWIGLU_CASES = [  # M, N, K, bits, out
    (1, 896, 4864, 8, "bf16"),       # the decode down projection (eight-row kernel)
    (1, 896, 4864, 4, "f32"),
    (2, 896, 4864, 4, "bf16"),
    (8, 896, 4864, 8, "f32"),        # 16-row fragments, three groups a warp
    (3, 300, 2048 + 32, 8, "f32"),   # a ragged 32-wide last group
    (2, 4864, 896, 4, "f32"),        # one group a warp, fragments in registers
    (5, 1000, 4096 + 128, 4, "bf16"),
]


@pytest.mark.parametrize("M,N,K,bits,out", SWIGLU_CASES)
def test_swiglu_decode_product(tq, M, N, K, bits, out):
    """Y of h = bf16(silu(G) U), G and U the two halves of one gate/up row
    (strided views): against the oracle's O8 then O6 (f32 Y to REL_L2_Y, bf16
    Y within a16_close's bar), and equal bit for
    bit to the unfused route (the oracle's h through tq_linear, the same
    decode kernel without the SwiGLU prologue)."""
    import torch
    mode = "W8A16" if bits == 8 else "W4A16"
    G, U = _swiglu_inputs(f"{M}x{N}x{K}b{bits}", M, K)
    GU = to_dev_bf16(np.concatenate([G, U], axis=1))
    codes, sw = tq.quantize_weights(to_dev_bf16(synth.tensor(f"gpu/dswiglu/w{N}x{K}", N, K, *WD)), bits)
    Y = tq.linear_swiglu(GU[:, :K], GU[:, K:], codes, sw, N, bits, mode, out=out)
    H = oracle.swiglu_bf16(G, U)
    Y0 = tq.linear(to_dev_bf16(H), codes, sw, N, bits, mode, out=out)
    assert tq.device_status() == 0
    assert torch.equal(Y.view(torch.int16) if out == "bf16" else Y, Y0.view(torch.int16) if out == "bf16" else Y0)
    c = to_np(codes)
    wc = oracle.weight_codes(c.view(np.int8) if bits == 8 else c.view(np.uint8), bits, K)
    ref = oracle.linear_a16(oracle.rotate_act_bf16(H), wc, to_np(sw))
    if out == "bf16":
        assert a16_close(bf16_bits(Y), H, wc, to_np(sw))[0] <= 0
    else:
        assert rel_l2(to_np(Y), ref) <= REL_L2_Y


def test_swiglu_decode_product_padded_rows_and_output_stride(tq):
    """Gate and up from separate buffers with row strides above K, Y written
    into a wider matrix: the columns past N stay untouched."""
    import torch
    M, N, K, bits = 2, 640, 1024 + 64, 8
    G, U = _swiglu_inputs("strided", M, K)
    Gd = to_dev_bf16(np.pad(G, ((0, 0), (0, 40))))[:, :K]
    Ud = to_dev_bf16(np.pad(U, ((0, 0), (16, 24))))[:, 16:16 + K]
    codes, sw = tq.quantize_weights(to_dev_bf16(synth.tensor("gpu/dswiglu/ws", N, K, *WD)), bits)
    Yw = torch.full((M, N + 24), 7.0, dtype=torch.float32, device="cuda")
    tq.linear_swiglu(Gd, Ud, codes, sw, N, bits, "W8A16", Y=Yw[:, :N])
    assert tq.device_status() == 0
    ref = oracle.linear_a16(oracle.rotate_act_bf16(oracle.swiglu_bf16(G, U)), to_np(codes), to_np(sw))
    assert rel_l2(to_np(Yw[:, :N]), ref) <= REL_L2_Y
    assert torch.all(Yw[:, N:] == 7.0)


@pytest.mark.parametrize("bits", [8, 4])
def test_ffn_layer_chain_each_call_against_the_oracle(tq, bits):
    """Three gated FFN layers at decode (M = 1) in one CUDA graph, as the
    bench runs them: gate+up as one product over the stacked rows (9728 x
    896, bf16 out), then the down product of the SwiGLU of its two halves
    (896 x 4864), its output the next layer's input.  Each call against the
    oracle on the GPU's own input for that call.  The gate+up calls: within
    a16_close's bar.  The down calls: swiglu_down_close's bar."""
    import torch
    mode = "W8A16" if bits == 8 else "W4A16"
    K, F = 896, 4864
    def weights(name, N, Kw, post):
        # row scales over the RMS row norm, so a call keeps its input's RMS
        # (times post: 1 / 0.596, the RMS of silu(z) z' for standard normals,
        # for the down rows)
        W = synth.tensor(name, N, Kw, *WD)
        gain = np.sqrt(np.mean(np.sum(oracle.bf16_to_f64(W) ** 2, axis=1)))
        c, s = tq.quantize_weights(to_dev_bf16(W), bits)
        return c, (s * float(post / gain)).contiguous()
    layers = []
    for L in range(3):
        gc, gs = weights(f"gpu/ffn/gu{L}", 2 * F, K, 1.0)
        dc, ds = weights(f"gpu/ffn/d{L}", K, F, 1.0 / 0.596)
        layers.append((gc, gs, dc, ds))
    x0 = to_dev_bf16(synth.tensor("gpu/ffn/x", 1, K, 1.0))
    gu = torch.empty((1, 2 * F), dtype=torch.bfloat16, device="cuda")
    bufs = [torch.empty((1, K), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    rec_x = [torch.empty((1, K), dtype=torch.bfloat16, device="cuda") for _ in layers]
    rec_gu = [torch.empty((1, 2 * F), dtype=torch.bfloat16, device="cuda") for _ in layers]
    rec_y = [torch.empty((1, K), dtype=torch.bfloat16, device="cuda") for _ in layers]

    def run():
        x = x0
        for L, (gc, gs, dc, ds) in enumerate(layers):
            y = bufs[L % 2]
            rec_x[L].copy_(x)
            tq.linear(x, gc, gs, 2 * F, bits, mode, Y=gu, out="bf16")
            rec_gu[L].copy_(gu)
            tq.linear_swiglu(gu[:, :F], gu[:, F:], dc, ds, K, bits, mode, Y=y, out="bf16")
            rec_y[L].copy_(y)
            x = y
    run()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            run()
    torch.cuda.current_stream().wait_stream(s)
    for r in rec_x + rec_gu + rec_y:
        r.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert tq.device_status() == 0

    def wcodes(c, Kc):
        c = to_np(c)
        return oracle.weight_codes(c.view(np.int8) if bits == 8 else c.view(np.uint8), bits, Kc)
    for L, (gc, gs, dc, ds) in enumerate(layers):
        xb, gub, yb = bf16_bits(rec_x[L]), bf16_bits(rec_gu[L]), bf16_bits(rec_y[L])
        if L > 0:
            assert np.array_equal(xb, bf16_bits(rec_y[L - 1]))
        worst, _ = a16_close(gub, xb, wcodes(gc, K), to_np(gs))
        assert worst <= 0, f"layer {L} gate+up: {worst}"
        h = oracle.swiglu_bf16(gub[:, :F], gub[:, F:])
        assert np.count_nonzero(h) > F // 2
        ref_y = oracle.linear_a16(oracle.rotate_act_bf16(h), wcodes(dc, F), to_np(ds))
        good, got = swiglu_down_close(yb, ref_y)
        assert good, f"layer {L} down"
        assert 0.05 < np.sqrt(np.mean(got ** 2)) < 50.0     # the chain stays O(1)


# ---- chained plans: the dependent calls in one launch (tq_chain_create)

def _ffn_weights(tq, bits, L, tag):
    """A gated FFN layer's weights, gate and up stacked (9728 x 896) and down
    (896 x 4864), row scales normalised as in the per-call chain test."""
    K, F = 896, 4864

    def weights(name, N, Kw, post):
        W = synth.tensor(name, N, Kw, *WD)
        gain = np.sqrt(np.mean(np.sum(oracle.bf16_to_f64(W) ** 2, axis=1)))
        c, s = tq.quantize_weights(to_dev_bf16(W), bits)
        return c, (s * float(post / gain)).contiguous()
    gc, gs = weights(f"gpu/{tag}/gu{L}", 2 * F, K, 1.0)
    dc, ds = weights(f"gpu/{tag}/d{L}", K, F, 1.0 / 0.596)
    return gc, gs, dc, ds


def _wcodes(c, bits, Kc):
    c = to_np(c)
    return oracle.weight_codes(c.view(np.int8) if bits == 8 else c.view(np.uint8), bits, Kc)


def _check_ffn_layer(bits, L, x, gu, y, gc, gs, dc, ds, F):
    """One layer's two calls against the oracle on the GPU's own inputs
    (the bars of test_ffn_layer_chain_each_call_against_the_oracle)."""
    K = x.shape[1]
    worst, _ = a16_close(gu, x, _wcodes(gc, bits, K), to_np(gs))
    assert worst <= 0, f"layer {L} gate+up: {worst}"
    h = oracle.swiglu_bf16(gu[:, :F], gu[:, F:])
    ref_y = oracle.linear_a16(oracle.rotate_act_bf16(h), _wcodes(dc, bits, F), to_np(ds))
    good, got = swiglu_down_close(y, ref_y)
    assert good, f"layer {L} down"
    return got


@pytest.mark.parametrize("bits", [8, 4])
def test_chained_plan_ffn_layers(tq, bits):
    """Eight gated FFN layers at decode (M = 1) as one chained plan, 16
    dependent calls in one launch: gate+up, then the down product of the
    SwiGLU of its halves, its output the next layer's input.  Each call
    against the oracle on the GPU's own input; a second run and a CUDA-graph
    replay give the same bytes."""
    import torch
    K, F, layers = 896, 4864, 8
    x0_bits = synth.tensor("gpu/cplan/x", 1, K, 1.0)
    x0 = to_dev_bf16(x0_bits)
    # down row scales so that the oracle's output of each layer has RMS 1
    # (h = silu(g) u is quadratic in the layer input: without this the chain's
    # values grow as a double exponential); the chain run on the oracle alone
    ws, xr = [], x0_bits
    for L in range(layers):
        gc, gs, dc, ds = _ffn_weights(tq, bits, L, "cplan")
        gu_r = oracle.round_bf16(oracle.linear_a16(oracle.rotate_act_bf16(xr), _wcodes(gc, bits, K), to_np(gs)))
        y_r = oracle.linear_a16(oracle.rotate_act_bf16(oracle.swiglu_bf16(gu_r[:, :F], gu_r[:, F:])),
                                _wcodes(dc, bits, F), to_np(ds))
        r = float(np.sqrt(np.mean(y_r ** 2)))
        ws.append((gc, gs, dc, (ds / r).contiguous()))
        xr = oracle.round_bf16(y_r / r)
    gus = [torch.empty((1, 2 * F), dtype=torch.bfloat16, device="cuda") for _ in range(layers)]
    ys = [torch.empty((1, K), dtype=torch.bfloat16, device="cuda") for _ in range(layers)]
    calls, x = [], x0
    for L, (gc, gs, dc, ds) in enumerate(ws):
        calls.append((x, gc, gs, 2 * F, gus[L]))
        calls.append((gus[L][:, :F], dc, ds, K, ys[L], gus[L][:, F:]))
        x = ys[L]
    plan = tq.ChainPlan(calls, bits, out="bf16")
    plan.run()
    assert tq.device_status() == 0
    first = [bf16_bits(t).copy() for t in gus + ys]
    x = bf16_bits(x0)
    for L, (gc, gs, dc, ds) in enumerate(ws):
        got = _check_ffn_layer(bits, L, x, bf16_bits(gus[L]), bf16_bits(ys[L]), gc, gs, dc, ds, F)
        assert 0.5 < np.sqrt(np.mean(got ** 2)) < 2.0
        x = bf16_bits(ys[L])
    for t in gus + ys:
        t.zero_()
    plan.run()
    assert all(np.array_equal(a, bf16_bits(t)) for a, t in zip(first, gus + ys))
    for t in gus + ys:
        t.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            plan.run(stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for t in gus + ys:
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert tq.device_status() == 0
    assert all(np.array_equal(a, bf16_bits(t)) for a, t in zip(first, gus + ys))
    # a run with another input: every call must read this run's values, never
    # the last run's (the counters start from zero each run).  The input differs in
    # 16 signs, which changes every later value by far more than the bars
    # while keeping the chain's scale (h is quadratic in the input: a new
    # random input would drift from the calibrated scale layer by layer)
    x2 = x0_bits.copy()
    x2[0, :16] ^= 0x8000
    x0.copy_(to_dev_bf16(x2))
    g.replay()
    torch.cuda.synchronize()
    assert tq.device_status() == 0
    x = bf16_bits(x0)
    for L, (gc, gs, dc, ds) in enumerate(ws):
        _check_ffn_layer(bits, L, x, bf16_bits(gus[L]), bf16_bits(ys[L]), gc, gs, dc, ds, F)
        x = bf16_bits(ys[L])


@pytest.mark.parametrize("bits", [8, 4])
def test_chained_plan_mixed_calls(tq, bits):
    """Three-token calls of mixed shapes (ragged last groups, 8- and 16-row
    items, the row and tile forms), each input the output of the call before
    or of one further back, bf16 out; each call against the oracle on its
    GPU input (a16_close's bar)."""
    import torch
    mode_shapes = [(640, 1024 + 32), (2080, 640), (1024 + 32, 2080), (3000, 1024 + 32), (640, 2080)]
    # (N, K): call c reads Y of call c - 1, except the last, which reads call 1's
    M = 3
    x0 = to_dev_bf16(synth.tensor("gpu/cmix/x", M, 1024 + 32, 1.0))
    weights, ys, calls = [], [], []
    srcs = [None, 0, 1, 2, 1]
    for c, (N, K) in enumerate(mode_shapes):
        W = synth.tensor(f"gpu/cmix/w{c}", N, K, *WD)
        gain = np.sqrt(np.mean(np.sum(oracle.bf16_to_f64(W) ** 2, axis=1)))
        codes, sw = tq.quantize_weights(to_dev_bf16(W), bits)
        sw = (sw / float(gain)).contiguous()
        weights.append((codes, sw, N, K))
        ys.append(torch.empty((M, N), dtype=torch.bfloat16, device="cuda"))
    for c, (codes, sw, N, K) in enumerate(weights):
        X = x0 if srcs[c] is None else ys[srcs[c]][:, :K]
        calls.append((X, codes, sw, N, ys[c]))
    plan = tq.ChainPlan(calls, bits, out="bf16")
    plan.run()
    assert tq.device_status() == 0
    for c, (codes, sw, N, K) in enumerate(weights):
        xb = bf16_bits(x0) if srcs[c] is None else bf16_bits(ys[srcs[c]])[:, :K]
        worst, _ = a16_close(bf16_bits(ys[c]), xb, _wcodes(codes, bits, K), to_np(sw))
        assert worst <= 0, f"call {c}: {worst}"


def test_chained_plan_f32_outputs(tq):
    """A chained plan writing fp32 (its inputs then come from outside the
    plan): two independent calls and one that reuses the first's input, each
    against the oracle to REL_L2_Y."""
    import torch
    M = 2
    shapes = [(896, 4096), (4864, 896), (1000, 4096)]
    xs = [to_dev_bf16(synth.tensor(f"gpu/cf32/x{i}", M, K, 1.0)) for i, (_, K) in enumerate(shapes)]
    xs[2] = xs[0]
    calls, keep = [], []
    for i, (N, K) in enumerate(shapes):
        codes, sw = tq.quantize_weights(to_dev_bf16(synth.tensor(f"gpu/cf32/w{i}", N, K, *WD)), 8)
        Y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        calls.append((xs[i], codes, sw, N, Y))
        keep.append((codes, sw, Y))
    plan = tq.ChainPlan(calls, 8, out="f32")
    plan.run()
    assert tq.device_status() == 0
    for i, ((N, K), (codes, sw, Y)) in enumerate(zip(shapes, keep)):
        ref = oracle.linear_a16(oracle.rotate_act_bf16(bf16_bits(xs[i])), to_np(codes), to_np(sw))
        assert rel_l2(to_np(Y), ref) <= REL_L2_Y, f"call {i}"


def test_chained_plan_refuses_split_phases(tq):
    import torch
    codes, sw = tq.quantize_weights(to_dev_bf16(synth.tensor("gpu/cph/w", 256, 512, *WD)), 8)
    X = to_dev_bf16(synth.tensor("gpu/cph/x", 1, 512, 1.0))
    Y = torch.empty((1, 256), dtype=torch.float32, device="cuda")
    plan = tq.ChainPlan([(X, codes, sw, 256, Y)], 8)
    with pytest.raises(tq.TQError):
        plan.rotate()
    with pytest.raises(tq.TQError):
        plan.product()
    plan.run()
    ref = oracle.linear_a16(oracle.rotate_act_bf16(bf16_bits(X)), to_np(codes), to_np(sw))
    assert rel_l2(to_np(Y), ref) <= REL_L2_Y


@pytest.mark.parametrize("bits", [8, 4])
def test_chained_plan_eight_tokens(tq, bits):
    """Eight-token calls (the most a chained call takes): three dependent
    calls, the middle one with a ragged last group for 8-bit weights
    (K = 1024 + 32), each against the oracle on its GPU input."""
    import torch
    M = 8
    shapes = [(1056 if bits == 8 else 1024, 1024), (512, 1056 if bits == 8 else 1024), (300, 512)]
    x0b = synth.tensor(f"gpu/c8/x{bits}", M, 1024, 1.0)
    x0 = to_dev_bf16(x0b)
    calls, keep, x = [], [], x0
    for c, (N, K) in enumerate(shapes):
        W = synth.tensor(f"gpu/c8/w{bits}/{c}", N, K, *WD)
        gain = np.sqrt(np.mean(np.sum(oracle.bf16_to_f64(W) ** 2, axis=1)))
        codes, sw = tq.quantize_weights(to_dev_bf16(W), bits)
        sw = (sw / float(gain)).contiguous()
        Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        calls.append((x, codes, sw, N, Y))
        keep.append((codes, sw, Y, K))
        x = Y
    plan = tq.ChainPlan(calls, bits, out="bf16")
    plan.run()
    assert tq.device_status() == 0
    xb = x0b
    for c, (codes, sw, Y, K) in enumerate(keep):
        worst, _ = a16_close(bf16_bits(Y), xb, _wcodes(codes, bits, K), to_np(sw))
        assert worst <= 0, f"call {c}: {worst}"
        xb = bf16_bits(Y)
