"""C-ABI checks that need no GPU: the library builds, loads, exports every
symbol the header declares, and refuses bad arguments on the host, by name,
before any launch (TensorFold PR #948 review follow-up: sizes and overflowing
products are refused by name before device work; kvad-gpu internals: widths the
format cannot take are refused up front)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tq.h")

OK, NULL, SHAPE, BITS, MODE, OVERFLOW, ALIGN, WORKSPACE, CUDA, TIMEOUT, DEVICE = range(11)
FAKE = 0x10000          # 16-byte aligned, never dereferenced by a refused call
S0 = None               # default stream


@pytest.fixture(scope="module")
def L():
    from dit_convrot_linear_gb300 import build, tq
    build.build()
    return tq.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tq_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("tq_quantize_weights", "tq_rotate_quant_act", "tq_linear",
                     "tq_linear_q8", "tq_linear_workspace_bytes", "tq_status_str"):
        assert required in names


def test_library_exports_every_declared_symbol(L):
    from dit_convrot_linear_gb300 import tq
    for name in declared_functions():
        assert hasattr(L, name), f"{name} declared in tq.h but not exported"
        assert name in tq.SIGNATURES, f"{name} has no binding"


def test_status_strings(L):
    for s in range(11):
        assert L.tq_status_str(s).decode().startswith(
            ["TQ_OK", "TQ_ERR_NULL", "TQ_ERR_SHAPE", "TQ_ERR_BITS", "TQ_ERR_MODE",
             "TQ_ERR_OVERFLOW", "TQ_ERR_ALIGN", "TQ_ERR_WORKSPACE", "TQ_ERR_CUDA",
             "TQ_ERR_DEVICE_TIMEOUT", "TQ_ERR_DEVICE"][s])


def qw(L, W=FAKE, N=16, K=256, ldw=256, bits=8, group=256, codes=FAKE, scales=FAKE):
    return L.tq_quantize_weights(W, N, K, ldw, bits, group, codes, scales, S0)


def test_quantize_weights_refusals(L):
    assert qw(L, bits=5) == BITS
    assert qw(L, group=128) == SHAPE
    assert qw(L, K=300, ldw=304) == SHAPE            # 300 = 256 + 44: no valid tail
    assert qw(L, K=16, ldw=16) == SHAPE
    assert qw(L, K=65536 + 256, ldw=65536 + 256) == SHAPE
    assert qw(L, N=-1) == SHAPE
    assert qw(L, ldw=128) == SHAPE                   # stride shorter than a row
    assert qw(L, W=0) == NULL
    assert qw(L, codes=0) == NULL
    assert qw(L, W=FAKE + 2) == ALIGN
    assert qw(L, ldw=260) == ALIGN
    assert qw(L, codes=FAKE + 8) == ALIGN
    assert qw(L, N=2 ** 62, ldw=2 ** 20, K=256) == OVERFLOW
    assert qw(L, N=0) == OK                          # empty: nothing launched


def lin(L, X=FAKE, M=4, K=512, ldx=512, W=FAKE, sw=FAKE, N=256, bits=8, mode=0,
        Y=FAKE, yt=0, ldy=256, ws=0, wsb=0):
    return L.tq_linear(X, M, K, ldx, W, sw, N, bits, mode, Y, yt, ldy, ws, wsb, S0)


def test_linear_refusals(L):
    assert lin(L, mode=7) == MODE
    assert lin(L, yt=2) == MODE                      # int32 output only for tq_linear_q8
    assert lin(L, bits=3) == BITS
    assert lin(L, mode=0, bits=4) == MODE            # W8A16 needs 8-bit weights
    assert lin(L, mode=1, bits=8) == MODE
    assert lin(L, M=65, mode=0) == SHAPE             # A16 kernel takes M <= 64
    assert lin(L, K=200, ldx=200) == SHAPE
    assert lin(L, X=0) == NULL
    assert lin(L, W=0) == NULL
    assert lin(L, Y=0) == NULL
    assert lin(L, ldy=100) == SHAPE
    assert lin(L, ldx=520 + 4) == ALIGN
    assert lin(L, X=FAKE + 16) != ALIGN              # a 16-byte offset view is fine
    assert lin(L, ldy=257) != ALIGN                  # any row stride >= N is fine
    assert lin(L, Y=FAKE + 2) == ALIGN               # fp32 output must be 4-byte aligned
    assert lin(L, Y=FAKE + 2, yt=1) != ALIGN         # bf16 output: 2-byte alignment
    assert lin(L, mode=2, ws=0, wsb=0) == WORKSPACE
    need = L.tq_linear_workspace_bytes(4, 512, 256, 8, 2)
    assert need >= 4 * 512 + 16
    assert lin(L, mode=2, ws=FAKE, wsb=need - 1) == WORKSPACE
    assert lin(L, mode=2, ws=FAKE + 16, wsb=need) == ALIGN
    assert lin(L, M=0) == OK and lin(L, N=0) == OK
    assert lin(L, M=2 ** 62, ldx=2 ** 10, K=512, mode=2, ws=FAKE, wsb=2 ** 62) == OVERFLOW


def test_workspace_is_zero_for_a16(L):
    assert L.tq_linear_workspace_bytes(64, 4096, 12288, 4, 1) == 0
    assert L.tq_linear_workspace_bytes(4032, 12288, 3072, 8, 2) >= 4032 * 12288 + 4032 * 4


def test_linear_q8_refusals(L):
    f = L.tq_linear_q8
    assert f(FAKE, FAKE, 4, 512, FAKE, FAKE, 256, 8, FAKE, 5, 256, S0) == MODE
    assert f(0, FAKE, 4, 512, FAKE, FAKE, 256, 8, FAKE, 0, 256, S0) == NULL
    assert f(FAKE, 0, 4, 512, FAKE, FAKE, 256, 8, FAKE, 0, 256, S0) == NULL
    assert f(FAKE, FAKE, 4, 500, FAKE, FAKE, 256, 8, FAKE, 0, 256, S0) == SHAPE
    assert f(FAKE, FAKE, 4, 512, FAKE, FAKE, 256, 6, FAKE, 0, 256, S0) == BITS
    assert f(FAKE + 1, FAKE, 4, 512, FAKE, FAKE, 256, 8, FAKE, 0, 256, S0) == ALIGN


def test_tiled_refusals(L):
    assert L.tq_act_tiled_bytes(4, 16384 + 256) == 0          # above TQ_MAX_K_TILED
    assert L.tq_act_tiled_bytes(4, 500) == 0
    need = L.tq_act_tiled_bytes(300, 3072)
    assert need == 4 * 48 * 16384 + 256  # rows padded to two 256-row tile pairs, 48 K steps; trailer
    r = L.tq_rotate_quant_act_tiled
    assert r(FAKE, 4, 16384 + 256, 16384 + 256, FAKE, 1 << 30, FAKE, S0) == SHAPE
    assert r(FAKE, 4, 512, 512, 0, 1 << 20, FAKE, S0) == NULL
    assert r(FAKE, 4, 512, 512, FAKE, 100, FAKE, S0) == WORKSPACE
    assert r(FAKE, 4, 512, 512, FAKE + 16, 1 << 20, FAKE, S0) == ALIGN
    f = L.tq_linear_tiled
    assert f(FAKE, FAKE, 4, 512, FAKE, FAKE, 256, 8, FAKE, 5, 256, S0) == MODE
    assert f(0, FAKE, 4, 512, FAKE, FAKE, 256, 8, FAKE, 0, 256, S0) == NULL
    assert f(FAKE, FAKE, 4, 16384 + 256, FAKE, FAKE, 256, 8, FAKE, 0, 256, S0) == SHAPE
    assert f(FAKE + 16, FAKE, 4, 512, FAKE, FAKE, 256, 8, FAKE, 0, 256, S0) == ALIGN


def test_rotate_refusals(L):
    assert L.tq_rotate_quant_act(FAKE, 4, 96, 96, FAKE, FAKE, S0) == SHAPE
    assert L.tq_rotate_quant_act(FAKE, 4, 512, 512, 0, FAKE, S0) == NULL
    assert L.tq_rotate_quant_act(FAKE, 4, 512, 512, FAKE + 3, FAKE, S0) == ALIGN
    assert L.tq_rotate_act_bf16(FAKE, 4, 512, 512, 0, S0) == NULL
    assert L.tq_rotate_act_bf16(FAKE, 0, 512, 512, 0, S0) == OK


def test_valid_call_without_a_gpu_reports_no_device(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert qw(L) == DEVICE
