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
def lib_loaded():
    from dit_convrot_linear_gb300 import build, tq
    build.build()
    return tq.load()


@pytest.fixture(scope="module")
def L(lib_loaded):
    """The library for the refusal checks.  These pass fake device addresses
    (FAKE): a call that no host check refuses would launch a kernel on them,
    so with a GPU visible they do not run at all (they test the host logic,
    on a machine without a GPU, where such a call stops at the device query)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("refusal checks use fake device addresses: run them where no GPU is visible")
    return lib_loaded


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tq_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("tq_quantize_weights", "tq_rotate_quant_act", "tq_linear",
                     "tq_linear_q8", "tq_linear_workspace_bytes", "tq_status_str"):
        assert required in names


def test_library_exports_every_declared_symbol(lib_loaded):
    L = lib_loaded
    from dit_convrot_linear_gb300 import tq
    for name in declared_functions():
        assert hasattr(L, name), f"{name} declared in tq.h but not exported"
        assert name in tq.SIGNATURES, f"{name} has no binding"


def test_status_strings(lib_loaded):
    L = lib_loaded
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


def test_a16_workspace_is_the_tensor_core_operand(L):
    """A16 modes: the optional workspace holds the x' tiles of the tensor-core
    product ([ceil(K/64)] tiles of M rounded up to 16 rows x 64 fp16, then the
    token factors), for more than 8 tokens, or for weights of at least 2^24
    codes with 3 to 8 tokens; 0 for one or two tokens (they stream through
    the CUDA cores) and for decode-sized products, which need none."""
    assert L.tq_linear_workspace_bytes(64, 4096, 12288, 4, 1) == 64 * 64 * 64 * 2 + 256
    assert L.tq_linear_workspace_bytes(13, 896, 300, 8, 0) == 14 * 16 * 64 * 2 + 256
    assert L.tq_linear_workspace_bytes(3, 4096, 12288, 4, 1) == 64 * 16 * 64 * 2 + 256
    assert L.tq_linear_workspace_bytes(2, 4096, 12288, 4, 1) == 0     # two tokens: streaming
    assert L.tq_linear_workspace_bytes(2, 12288, 4096, 4, 1) == 0
    assert L.tq_linear_workspace_bytes(1, 4096, 12288, 4, 1) == 0     # one token: a CUDA-core kernel
    assert L.tq_linear_workspace_bytes(1, 896, 4864, 8, 0) == 0          # decode: none
    assert L.tq_linear_workspace_bytes(8, 4096, 1000, 4, 1) == 0
    assert L.tq_linear_workspace_bytes(64, 16384 + 256, 256, 8, 0) == 0   # K above the tiled limit
    assert L.tq_linear_workspace_bytes(4032, 12288, 3072, 8, 2) >= 4032 * 12288 + 4032 * 4
    # an A16 call without a workspace is not refused (the CUDA-core kernels run)
    import torch
    if not torch.cuda.is_available():
        assert lin(L, M=13, K=896, ldx=896, N=300, ldy=300, mode=0, bits=8, ws=0, wsb=0) == DEVICE


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
    assert need == 4 * 48 * 16384 + 2048  # rows padded to two 256-row tile pairs, 48 K steps; trailer
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


# ------------------------------------------------------------------ grouped plans

def gcalls(n=1, **kw):
    from dit_convrot_linear_gb300.tq import A16Call
    d = dict(X=FAKE, ldx=896, Wq=FAKE, sw=FAKE, Y=FAKE, ldy=4864, M=1, N=4864, K=896)
    d.update(kw)
    return [A16Call(**d) for _ in range(n)]


def gbytes(L, calls, bits=8):
    from dit_convrot_linear_gb300 import tq
    arr = (tq.A16Call * max(len(calls), 1))(*calls)
    out = ctypes.c_size_t(0)
    rc = L.tq_grouped_bytes(ctypes.addressof(arr), len(calls), bits, ctypes.byref(out))
    return rc, out.value


def gcreate(L, calls, bits=8, ytype=0, dmem=FAKE, dbytes=1 << 20):
    from dit_convrot_linear_gb300 import tq
    arr = (tq.A16Call * max(len(calls), 1))(*calls)
    h = ctypes.c_void_p(None)
    rc = L.tq_grouped_create(ctypes.addressof(arr), len(calls), bits, ytype, dmem, dbytes,
                             ctypes.byref(h))
    return rc, h


def test_grouped_refusals(L):
    assert gbytes(L, gcalls(), bits=5)[0] == BITS
    assert gbytes(L, gcalls(M=9))[0] == SHAPE             # above TQ_MAX_M_GROUPED
    assert gbytes(L, gcalls(K=96))[0] == SHAPE            # K not 256q + {0, 32, 64, 128}
    assert gbytes(L, gcalls(X=0))[0] == NULL
    assert gbytes(L, gcalls(sw=0))[0] == NULL
    assert gbytes(L, gcalls(X=FAKE + 2))[0] == ALIGN
    assert gbytes(L, gcalls(ldx=900))[0] == ALIGN          # row stride not a multiple of 8
    assert gbytes(L, gcalls(ldy=100))[0] == SHAPE          # ldy < N
    assert gbytes(L, gcalls(Wq=FAKE + 8))[0] == ALIGN
    assert gbytes(L, gcalls(K=12288, ldx=12288))[0] == SHAPE      # 8 rows + x' exceed a stage
    assert gbytes(L, gcalls(M=8, K=4864, ldx=4864))[0] == SHAPE   # x' of 8 tokens too long
    assert gbytes(L, gcalls(K=16384, ldx=16384), bits=4)[0] == SHAPE
    assert gbytes(L, gcalls(K=9728, ldx=9728))[0] == OK           # the longest 8-bit K for M = 1
    assert gbytes(L, gcalls(K=9760, ldx=9760))[0] == SHAPE
    assert gbytes(L, gcalls(K=16128, ldx=16128), bits=4)[0] == OK  # and 4-bit
    assert gbytes(L, gcalls(K=16160, ldx=16160), bits=4)[0] == SHAPE
    # an empty call is skipped before its pointers are looked at
    assert gbytes(L, gcalls(M=0, X=0, Wq=0)) == (OK, 0)
    assert gbytes(L, []) == (OK, 0)
    assert L.tq_grouped_bytes(FAKE, -1, 8, ctypes.byref(ctypes.c_size_t(0))) == SHAPE
    # create: the call checks, then the buffer, all before any device work
    assert gcreate(L, gcalls(M=9))[0] == SHAPE
    assert gcreate(L, gcalls(), ytype=2)[0] == MODE        # i32 is not an A16 output
    assert gcreate(L, gcalls(), dbytes=100)[0] == WORKSPACE
    assert gcreate(L, gcalls(), dmem=0)[0] == WORKSPACE
    assert gcreate(L, gcalls(), dmem=FAKE + 16)[0] == ALIGN
    assert L.tq_grouped_create(FAKE, 1, 8, 0, FAKE, 1 << 20, None) == NULL
    assert L.tq_grouped_run(None, S0) == NULL
    assert L.tq_grouped_rotate(None, S0) == NULL
    assert L.tq_grouped_product(None, S0) == NULL
    assert L.tq_grouped_weight_bytes(None) == 0
    L.tq_grouped_destroy(None)


def test_grouped_bytes_count_tables_and_rotated_inputs(L):
    # M = 1, K = 896, N = 4864, 8-bit: items of 96 rows (960-byte shared rows,
    # 1792 bytes of x' per item, a 96 KB stage) -> 51 items of 128 bytes (6528,
    # rounded to 6656); one 40-byte call record and one 128-byte tensor map
    # (rows of 7 chunks of 128 bytes: the tile form), each rounded to 256; x'
    # of 896 fp16 and a 64-byte tail (the token scales and sums of x')
    assert gbytes(L, gcalls()) == (OK, 256 + 6656 + 256 + 896 * 2 + 64)
    # two tokens, K = 544 (x' padded to 640 columns), N = 100, 4-bit: two
    # items of 64 rows, tile form
    calls = gcalls(M=2, N=100, K=544, ldx=544, ldy=100)
    assert gbytes(L, calls, bits=4) == (OK, 256 + 256 + 256 + 2 * 640 * 2 + 64)
    # long rows (K = 4864: 38 chunks, items of 16 rows) stay in the row form:
    # no tensor map; 56 items of 128 bytes
    calls = gcalls(N=896, K=4864, ldx=4864, ldy=896)
    assert gbytes(L, calls) == (OK, 256 + 7168 + 4864 * 2 + 64)


def test_grouped_create_without_a_gpu_reports_no_device(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert gcreate(L, gcalls())[0] == DEVICE


def test_tiled_weights_refusals_and_size(L):
    # rows padded to 256, columns to 64: ceil(300/256)*2 row tiles x 48 column tiles x 16 KB
    assert L.tq_weights_tiled_bytes(300, 3072) == 4 * 48 * 16384 + 256   # tiles, then a trailer
    assert L.tq_weights_tiled_bytes(256, 32) == 2 * 1 * 16384 + 256
    assert L.tq_weights_tiled_bytes(1, 96) == 0                 # K not a valid row length
    assert L.tq_weights_tiled_bytes(1, 16384 + 256) == 0        # above TQ_MAX_K_TILED
    assert L.tq_tile_weights(FAKE, 16, 256, 5, FAKE, 1 << 20, S0) == BITS
    assert L.tq_tile_weights(FAKE, 16, 96, 8, FAKE, 1 << 20, S0) == SHAPE
    assert L.tq_tile_weights(0, 16, 256, 8, FAKE, 1 << 20, S0) == NULL
    assert L.tq_tile_weights(FAKE, 16, 256, 8, FAKE, 100, S0) == WORKSPACE
    assert L.tq_tile_weights(FAKE, 16, 256, 8, FAKE + 16, 1 << 20, S0) == ALIGN
    assert L.tq_tile_weights(FAKE, 0, 256, 8, 0, 0, S0) == OK      # empty
    tt = lambda **k: L.tq_linear_tt(*[k.get(n, d) for n, d in (
        ("At", FAKE), ("sx", FAKE), ("M", 4), ("K", 512), ("Wt", FAKE), ("sw", FAKE), ("N", 256),
        ("bits", 8), ("Y", FAKE), ("ytype", 0), ("ldy", 256), ("s", S0))])
    assert tt(bits=3) == BITS
    assert tt(ytype=7) == MODE
    assert tt(K=96) == SHAPE
    assert tt(Wt=0) == NULL
    assert tt(At=FAKE + 16) == ALIGN
    assert tt(Wt=FAKE + 16) == ALIGN
    assert tt(ldy=100) == SHAPE
    assert tt(M=0) == OK


def test_split_refusals(L):
    """tq_linear_tt_split checks what tq_linear_tt does, and its workspace;
    without a device the workspace size is 0 and a valid call reports it."""
    sp = lambda **k: L.tq_linear_tt_split(*[k.get(n, d) for n, d in (
        ("At", FAKE), ("sx", FAKE), ("M", 4), ("K", 512), ("Wt", FAKE), ("sw", FAKE), ("N", 256),
        ("bits", 8), ("epi", None), ("Y", FAKE), ("ytype", 0), ("ldy", 256), ("ws", FAKE),
        ("wsb", 1 << 30), ("s", S0))])
    assert sp(bits=3) == BITS
    assert sp(ytype=7) == MODE
    assert sp(K=96) == SHAPE
    assert sp(Wt=0) == NULL
    assert sp(At=FAKE + 16) == ALIGN
    assert sp(ldy=100) == SHAPE
    assert sp(M=0) == OK
    import torch
    if not torch.cuda.is_available():
        assert L.tq_split_workspace_bytes() == 0
        assert sp() == DEVICE
        assert sp(ws=None, wsb=0) == DEVICE


def test_epilogue_refusals(L):
    from dit_convrot_linear_gb300 import tq
    Y = 0x100000
    def ex(epi, ytype=0, ldy=256):
        e = ctypes.addressof(epi) if epi is not None else None
        return L.tq_linear_tt_ex(FAKE, FAKE, 4, 512, FAKE, FAKE, 256, 8, e, Y, ytype, ldy, S0)
    E = lambda **k: tq.Epilogue(k.get("bias", 0), k.get("gate", 0), k.get("residual", 0),
                                k.get("ldr", 256), k.get("rtype", 0))
    assert ex(E(bias=FAKE), ytype=2) == MODE                   # no epilogue on raw int32 sums
    assert ex(E(residual=FAKE, rtype=7)) == MODE
    assert ex(E(bias=FAKE + 2)) == ALIGN
    assert ex(E(gate=FAKE + 1)) == ALIGN
    assert ex(E(residual=FAKE, ldr=100)) == SHAPE             # ldr < N
    assert ex(E(residual=FAKE + 2, rtype=0)) == ALIGN          # fp32 residual on a 2-byte boundary
    assert ex(E(residual=Y, ldr=512)) == SHAPE                 # the same buffer with another stride
    assert ex(E(residual=Y, rtype=1)) == SHAPE                 # ... or another type
    assert ex(E(residual=Y + 64)) == SHAPE                     # a partial overlap
    import torch
    if not torch.cuda.is_available():
        assert ex(E(residual=Y)) == DEVICE                     # in place: accepted on the host
        assert ex(E(bias=FAKE, gate=FAKE)) == DEVICE
        assert ex(None) == DEVICE


def test_swiglu_quant_refusals(L):
    sq = lambda **k: L.tq_swiglu_quant_act_tiled(*[k.get(n, d) for n, d in (
        ("G", FAKE), ("ldg", 1024), ("U", FAKE + 1024), ("ldu", 1024), ("M", 4), ("K", 512),
        ("At", FAKE), ("at", 1 << 30), ("sx", FAKE), ("s", S0))])
    assert sq(K=96) == SHAPE
    assert sq(K=16384 + 256) == SHAPE                 # above TQ_MAX_K_TILED
    assert sq(G=0) == NULL
    assert sq(U=0) == NULL
    assert sq(ldu=500) == SHAPE                       # ldu < K
    assert sq(U=FAKE + 2) == ALIGN
    assert sq(ldg=1028) == ALIGN                      # stride not a multiple of 8
    assert sq(At=0) == NULL
    assert sq(at=100) == WORKSPACE
    assert sq(At=FAKE + 16) == ALIGN
    assert sq(M=0) == OK


def test_blocked_refusals(L):
    qb = lambda **k: L.tq_quantize_weights_blocked(*[k.get(n, d) for n, d in (
        ("W", FAKE), ("N", 16), ("K", 896), ("ldw", 896), ("bits", 4), ("G", 32), ("rot", 1),
        ("codes", FAKE), ("scales", FAKE), ("s", S0))])
    assert qb(bits=2) == BITS
    assert qb(rot=2) == MODE
    for G in (16, 48, 512, 0, -32):
        assert qb(G=G) == SHAPE                       # block widths 32, 64, 128, 256 only
    assert qb(G=256) == SHAPE                          # 896 = 3 x 256 + 128: 256 does not divide K
    assert qb(G=128) == DEVICE and qb(G=64, rot=0) == DEVICE
    assert qb(K=96, ldw=96) == SHAPE                   # not a valid row length
    assert qb(N=-1) == SHAPE
    assert qb(W=0) == NULL and qb(codes=0) == NULL and qb(scales=0) == NULL
    assert qb(W=FAKE + 2) == ALIGN and qb(ldw=900) == ALIGN
    assert qb(codes=FAKE + 8) == ALIGN and qb(scales=FAKE + 2) == ALIGN
    assert qb(N=2 ** 62, ldw=2 ** 20) == OVERFLOW
    assert qb(N=0) == OK
    lb = lambda **k: L.tq_linear_blocked(*[k.get(n, d) for n, d in (
        ("X", FAKE), ("M", 1), ("K", 896), ("ldx", 896), ("W", FAKE), ("sw", FAKE), ("G", 32),
        ("N", 4864), ("bits", 8), ("rot", 0), ("Y", FAKE), ("yt", 0), ("ldy", 4864), ("s", S0))])
    assert lb() == DEVICE                              # every check passes; no GPU here
    assert lb(bits=3) == BITS
    assert lb(rot=-1) == MODE and lb(yt=2) == MODE     # no int32 output
    assert lb(M=9) == SHAPE and lb(M=-1) == SHAPE      # TQ_MAX_M_BLOCKED = 8
    assert lb(G=256) == SHAPE and lb(G=24) == SHAPE
    assert lb(K=300, ldx=304) == SHAPE
    assert lb(X=0) == NULL and lb(W=0) == NULL and lb(sw=0) == NULL and lb(Y=0) == NULL
    assert lb(ldx=900) == ALIGN and lb(W=FAKE + 4) == ALIGN and lb(Y=FAKE + 2) == ALIGN
    assert lb(Y=FAKE + 2, yt=1) == DEVICE              # bf16 output: 2-byte alignment
    assert lb(ldy=100) == SHAPE
    assert lb(M=0) == OK and lb(N=0) == OK


def test_modnorm_quant_refusals(L):
    import ctypes
    mq = lambda **k: L.tq_modnorm_quant_act_tiled(*[k.get(n, d) for n, d in (
        ("X", FAKE), ("M", 4), ("K", 512), ("ldx", 512), ("shift", FAKE), ("scale", FAKE + 4096),
        ("eps", ctypes.c_float(1e-6)), ("At", FAKE), ("at", 1 << 30), ("sx", FAKE), ("s", S0))])
    assert mq(K=96) == SHAPE
    assert mq(K=16384 + 256) == SHAPE                 # above TQ_MAX_K_TILED
    assert mq(X=0) == NULL
    assert mq(shift=0) == NULL
    assert mq(scale=0) == NULL
    assert mq(ldx=500) == SHAPE                       # ldx < K
    assert mq(ldx=1028) == ALIGN                      # stride not a multiple of 8
    assert mq(shift=FAKE + 4) == ALIGN                # modulation vectors 16-byte aligned
    assert mq(scale=FAKE + 8) == ALIGN
    assert mq(eps=ctypes.c_float(-1e-6)) == MODE
    assert mq(eps=ctypes.c_float(float("nan"))) == MODE
    assert mq(eps=ctypes.c_float(float("inf"))) == MODE
    assert mq(At=0) == NULL
    assert mq(at=100) == WORKSPACE
    assert mq(At=FAKE + 16) == ALIGN
    assert mq(M=0) == OK
    assert mq(M=0, eps=ctypes.c_float(-1.0)) == MODE  # eps is checked even for an empty call


def test_linear_swiglu_refusals(L):
    sg = lambda **k: L.tq_linear_swiglu(*[k.get(n, d) for n, d in (
        ("G", FAKE), ("ldg", 1024), ("U", FAKE + 1024), ("ldu", 1024), ("M", 1), ("K", 512),
        ("W", FAKE), ("sw", FAKE), ("N", 256), ("bits", 8), ("mode", 0), ("Y", FAKE), ("yt", 0),
        ("ldy", 256), ("s", S0))])
    assert sg(mode=2) == MODE                         # A16 modes only: the input is bf16
    assert sg(mode=1) == MODE                         # W4A16 needs 4-bit weights
    assert sg(bits=5) == BITS
    assert sg(yt=2) == MODE
    assert sg(M=9) == SHAPE                           # the decode kernels take M <= 8
    assert sg(K=200, ldg=200, ldu=200) == SHAPE
    assert sg(G=0) == NULL
    assert sg(U=0) == NULL
    assert sg(W=0) == NULL
    assert sg(Y=0) == NULL
    assert sg(ldu=500) == SHAPE                       # ldu < K
    assert sg(ldg=1028) == ALIGN
    assert sg(U=FAKE + 8) == ALIGN                    # each half 16-byte aligned
    assert sg(M=0) == OK and sg(N=0) == OK
    assert sg(M=0, mode=2) == MODE                    # the mode is checked even for an empty call


# ------------------------------------------------------------------ chained plans

def ccalls(n=1, U=0, ldu=0, **kw):
    from dit_convrot_linear_gb300.tq import ChainCall
    return [ChainCall(c, U, ldu) for c in gcalls(n, **kw)]


def cbytes(L, calls, bits=8):
    from dit_convrot_linear_gb300 import tq
    arr = (tq.ChainCall * max(len(calls), 1))(*calls)
    out = ctypes.c_size_t(0)
    rc = L.tq_chain_bytes(ctypes.addressof(arr), len(calls), bits, ctypes.byref(out))
    return rc, out.value


def test_chain_refusals(L):
    from dit_convrot_linear_gb300 import tq
    assert cbytes(L, ccalls(), bits=5)[0] == BITS
    assert cbytes(L, ccalls(M=9))[0] == SHAPE
    assert cbytes(L, ccalls(X=0))[0] == NULL
    assert cbytes(L, ccalls(U=FAKE + 8, ldu=896))[0] == ALIGN      # up rows 16-byte aligned
    assert cbytes(L, ccalls(U=FAKE, ldu=500))[0] == SHAPE          # ldu < K
    assert cbytes(L, ccalls(U=FAKE, ldu=900))[0] == ALIGN
    assert cbytes(L, ccalls(U=FAKE + 4096, ldu=896))[0] == OK
    # the longest rows: the rotated input must fit the launch's own buffer
    # (K = 8960 at M = 1, 8- or 4-bit weights)
    assert cbytes(L, ccalls(K=8960, ldx=8960))[0] == OK
    assert cbytes(L, ccalls(K=8992, ldx=8992))[0] == SHAPE
    assert cbytes(L, ccalls(K=8960, ldx=8960), bits=4)[0] == OK
    assert cbytes(L, ccalls(K=8992, ldx=8992), bits=4)[0] == SHAPE
    assert cbytes(L, ccalls(M=8, K=1024, ldx=1024), bits=4)[0] == OK
    assert cbytes(L, ccalls(M=8, K=1024 + 64, ldx=1088), bits=4)[0] == SHAPE   # x' of 8 tokens too long
    assert cbytes(L, ccalls(M=0, X=0, Wq=0)) == (OK, 0)
    assert L.tq_chain_bytes(FAKE, -1, 8, ctypes.byref(ctypes.c_size_t(0))) == SHAPE
    arr = (tq.ChainCall * 1)(*ccalls())
    h = ctypes.c_void_p(None)
    assert L.tq_chain_create(ctypes.addressof(arr), 1, 8, 2, FAKE, 1 << 20, ctypes.byref(h)) == MODE
    assert L.tq_chain_create(ctypes.addressof(arr), 1, 8, 0, FAKE, 100, ctypes.byref(h)) == WORKSPACE
    assert L.tq_chain_create(ctypes.addressof(arr), 1, 8, 0, FAKE + 16, 1 << 20, ctypes.byref(h)) == ALIGN
    assert L.tq_chain_create(ctypes.addressof(arr), 1, 8, 0, FAKE, 1 << 20, None) == NULL


def test_chain_bytes_count_the_most_items(L):
    """Sizes need no device: every call counted with items of 8 rows (the
    most a plan can have), every short-row call with a tensor map; no x'
    workspace, a call record of 48 bytes and a counter of 4 per call."""
    # a gated FFN layer at decode: gate+up 9728 x 896 (1216 items, tile
    # form), down 896 x 4864 with the SwiGLU of the halves (112 items, rows)
    gu = ccalls(N=9728, ldy=9728)
    down = ccalls(N=896, K=4864, ldx=9728, ldy=896, U=FAKE + 4864 * 2, ldu=9728)
    items = -(-(1216 + 112) * 128 // 256) * 256
    assert cbytes(L, gu + down) == (OK, items + 256 + 256 + 256)
