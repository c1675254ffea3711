"""GPU parity of a dependent decode chain (M = 1): gate (896 -> 4864) then
down (4864 -> 896) through three layer sets, each call's input the previous
call's bf16 output, in one CUDA graph as the bench runs it.  Every call is
checked against the oracle's O6 on the GPU's own input for that call (so a
rounding difference in one call does not travel into the next one's check):
bf16 Y within one bf16 ulp of the oracle's value rounded to bf16.  Both
weight formats; the per-call kernels release the next launch before their
dependency wait, so this also checks that no call reads its input before the
previous call has written it."""
import numpy as np
import pytest

import oracle
from dit_convrot_linear_gb300 import synth
from helpers import bf16_bits, bf16_ulp_diff, to_dev_bf16, to_np

pytestmark = pytest.mark.gpu

WD = (0.02, 0.01, 20.0)


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
        ref = oracle.linear_a16(oracle.rotate_act_bf16(xb), wc, to_np(sw))
        d = bf16_ulp_diff(bf16_bits(outs[i]), oracle.round_bf16(ref))
        assert d.max() <= 1, f"call {i}: {d.max()} ulp"
        if i > 0:   # the chain: this call's input is the previous call's output
            assert np.array_equal(xb, bf16_bits(outs[i - 1]))
    assert tq.device_status() == 0
