"""CPU oracle for the rotated low-bit linear projection (numpy front end).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke``
and by the benchmark's CPU-baseline leg, never by the product path.  It shares
no code with the CUDA library: the arithmetic is the plain C in
``tq_oracle.c`` (explicit fp64 Hadamard products, nearest-even rounding, int64
code products), compiled here with gcc.

Every function takes and returns numpy arrays; bf16 tensors travel as their
``uint16`` bit patterns.  Step names (O1..O11) are those of ``tq_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tq_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libtq_oracle.so")
_CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
           "-ffp-contract=off"]
_lock = threading.Lock()
_lib = None

QMAX = {8: 127, 4: 7}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into ``oracle/libtq_oracle.so``."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    try:
        subprocess.run(["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return _LIB_PATH


_P = ctypes.c_void_p
_I = ctypes.c_int64
_SIGS = {
    "or_sylvester": (ctypes.c_int, [ctypes.c_int, _P]),
    "or_hadamard_norm": (ctypes.c_double, [ctypes.c_int]),
    "or_group_width": (ctypes.c_int, [_I, _I]),
    "or_valid_k": (ctypes.c_int, [_I]),
    "or_f64_to_bf16": (ctypes.c_uint16, [ctypes.c_double]),
    "or_bf16_to_f64": (ctypes.c_double, [ctypes.c_uint16]),
    "or_round_bf16": (ctypes.c_int, [_P, _I, _P]),
    "or_rotate_rows": (ctypes.c_int, [_P, _I, _I, _I, _P, ctypes.c_int]),
    "or_quantize_rows": (ctypes.c_int, [_P, _I, _I, ctypes.c_int, _P, _P]),
    "or_pack_int4": (ctypes.c_int, [_P, _I, _I, _P]),
    "or_unpack_int4": (ctypes.c_int, [_P, _I, _I, _P]),
    "or_linear_a8": (ctypes.c_int, [_P, _P, _I, _I, _P, _P, _I, _P, _P, ctypes.c_int]),
    "or_linear_a8_pairs": (ctypes.c_int, [_P, _P, _I, _I, _P, _P, _I, _P, _P, _I,
                                          _P, _P, ctypes.c_int]),
    "or_linear_a16": (ctypes.c_int, [_P, _I, _I, _P, _P, _I, _P, ctypes.c_int]),
    "or_linear_a16_pairs": (ctypes.c_int, [_P, _I, _I, _P, _P, _I, _P, _P, _I, _P,
                                           ctypes.c_int]),
    "or_matmul_f64": (ctypes.c_int, [_P, _I, _I, _P, _I, _P, ctypes.c_int]),
    "or_swiglu_f64": (ctypes.c_int, [_P, _P, _I, _P]),
    "or_swiglu_bf16": (ctypes.c_int, [_P, _I, _P, _I, _I, _I, _P]),
    "or_modnorm_f64": (ctypes.c_int, [_P, _I, _P, _P, ctypes.c_double, _P]),
    "or_modnorm_bf16": (ctypes.c_int, [_P, _I, _I, _I, _P, _P, ctypes.c_float, _P]),
    "or_quantize_blocks": (ctypes.c_int, [_P, _I, _I, _I, ctypes.c_int, _P, _P]),
    "or_linear_a16_blocked": (ctypes.c_int, [_P, _I, _I, _P, _P, _I, _I, _P, ctypes.c_int]),
}


def _bind(path: str):
    L = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


class using:
    """Context manager: route this module's calls to another build of the
    oracle (tests use it to plant mistakes in a copy of the C source)."""

    def __init__(self, so_path: str):
        self.path = so_path

    def __enter__(self):
        global _lib
        L = _bind(self.path)
        lib()
        with _lock:
            self.saved, _lib = _lib, L
        return L

    def __exit__(self, *exc):
        global _lib
        with _lock:
            _lib = self.saved
        return False


def compile_variant(src_text: str, out_dir: str, name: str) -> str:
    """Compile C source text with the oracle's flags into out_dir/name.so."""
    src = os.path.join(out_dir, name + ".c")
    so = os.path.join(out_dir, name + ".so")
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", *_CFLAGS, src, "-o", so, "-lm"], check=True)
    return so


def source() -> str:
    with open(_SRC) as f:
        return f.read()


_threads = None


def threads() -> int:
    """Threads the oracle runs on: every host core, unless set_threads chose."""
    return _threads or max(1, os.cpu_count() or 1)


def set_threads(n=None):
    """Run the oracle on n threads (None: every host core again)."""
    global _threads
    _threads = None if n is None else max(1, int(n))


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


# ---------------------------------------------------------------- definitions

def sylvester(n: int) -> np.ndarray:
    """Hs_n[i][j] = (-1)^popcount(i & j) as int8 [n, n]."""
    H = np.empty((n, n), dtype=np.int8)
    _check(lib().or_sylvester(n, H.ctypes.data), "sylvester")
    return H


def hadamard_norm(n: int) -> float:
    return float(lib().or_hadamard_norm(n))


def group_width(K: int, g0: int) -> int:
    return int(lib().or_group_width(K, g0))


def valid_k(K: int) -> bool:
    return bool(lib().or_valid_k(K))


def f64_to_bf16(x: float) -> int:
    return int(lib().or_f64_to_bf16(float(x)))


def bf16_to_f64(b) -> np.ndarray:
    """O1: exact widening of bf16 bit patterns."""
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def round_bf16(v: np.ndarray) -> np.ndarray:
    """O4': nearest bf16 (ties to even) of fp64 values, one rounding."""
    v = _c(v, np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _check(lib().or_round_bf16(v.ctypes.data, v.size, out.ctypes.data), "round_bf16")
    return out


# ---------------------------------------------------------------- steps

def rotate_rows(X: np.ndarray, K: int | None = None) -> np.ndarray:
    """O1+O2: group-wise Hadamard rotation of bf16 rows, fp64 [R, K].

    ``X`` is a 2-D uint16 array; its first ``K`` columns are the rows (the
    rest of each row, if any, is stride padding and is not read)."""
    X = np.asarray(X, dtype=np.uint16)
    if X.ndim != 2 or X.strides[1] != 2 or X.strides[0] % 2:
        X = _c(X, np.uint16)
    R, ld = X.shape[0], X.strides[0] // 2
    K = X.shape[1] if K is None else K
    out = np.empty((R, K), dtype=np.float64)
    _check(lib().or_rotate_rows(X.ctypes.data, R, K, ld, out.ctypes.data,
                                threads()), "rotate_rows")
    return out


def quantize_rows(V: np.ndarray, qmax: int):
    """O3/O4: per-row symmetric quantisation -> (int8 codes [R,K], fp32 [R])."""
    V = _c(V, np.float64)
    R, K = V.shape
    codes = np.empty((R, K), dtype=np.int8)
    scales = np.empty(R, dtype=np.float32)
    _check(lib().or_quantize_rows(V.ctypes.data, R, K, qmax, codes.ctypes.data,
                                  scales.ctypes.data), "quantize_rows")
    return codes, scales


def pack_int4(codes: np.ndarray) -> np.ndarray:
    """O7: [R, K] int8 codes in [-8, 7] -> [R, K/2] bytes, low nibble = even k."""
    codes = _c(codes, np.int8)
    R, K = codes.shape
    out = np.empty((R, K // 2), dtype=np.uint8)
    _check(lib().or_pack_int4(codes.ctypes.data, R, K, out.ctypes.data), "pack_int4")
    return out


def unpack_int4(packed: np.ndarray, K: int) -> np.ndarray:
    packed = _c(packed, np.uint8)
    R = packed.shape[0]
    out = np.empty((R, K), dtype=np.int8)
    _check(lib().or_unpack_int4(packed.ctypes.data, R, K, out.ctypes.data),
           "unpack_int4")
    return out


def quantize_weights(W: np.ndarray, bits: int):
    """O1-O3 (+O7 for 4 bits): bf16 W [N, K] -> (codes, fp32 row scales).

    codes are int8 [N, K] for 8 bits, packed uint8 [N, K/2] for 4 bits."""
    codes, scales = quantize_rows(rotate_rows(W), QMAX[bits])
    return (codes if bits == 8 else pack_int4(codes)), scales


def rotate_quant_act(X: np.ndarray, K: int | None = None):
    """O1+O2+O4: bf16 X [M, K] -> (int8 codes [M, K], fp32 token scales [M])."""
    return quantize_rows(rotate_rows(X, K), 127)


def rotate_act_bf16(X: np.ndarray, K: int | None = None) -> np.ndarray:
    """O1+O2+O4': bf16 X [M, K] -> rotated bf16 bits [M, K]."""
    return round_bf16(rotate_rows(X, K))


def weight_codes(Wq: np.ndarray, bits: int, K: int) -> np.ndarray:
    """int8 codes [N, K] from either storage form (O7 unpack for 4 bits)."""
    return _c(Wq, np.int8) if bits == 8 else unpack_int4(Wq, K)


def linear_a8(Xq, sx, Wcodes, sw, want_acc: bool = True):
    """O5: (int32 acc [M,N] or None, fp64 Y [M,N])."""
    Xq, Wcodes = _c(Xq, np.int8), _c(Wcodes, np.int8)
    sx, sw = _c(sx, np.float32), _c(sw, np.float32)
    M, K = Xq.shape
    N = Wcodes.shape[0]
    acc = np.empty((M, N), dtype=np.int32) if want_acc else None
    Y = np.empty((M, N), dtype=np.float64)
    _check(lib().or_linear_a8(Xq.ctypes.data, sx.ctypes.data, M, K,
                              Wcodes.ctypes.data, sw.ctypes.data, N,
                              acc.ctypes.data if want_acc else None,
                              Y.ctypes.data, threads()), "linear_a8")
    return acc, Y


def linear_a8_pairs(Xq, sx, Wcodes, sw, pm, pn):
    """O5 at listed (m, n) pairs -> (int32 acc [P], fp64 Y [P])."""
    Xq, Wcodes = _c(Xq, np.int8), _c(Wcodes, np.int8)
    sx, sw = _c(sx, np.float32), _c(sw, np.float32)
    pm, pn = _c(pm, np.int64), _c(pn, np.int64)
    M, K = Xq.shape
    N = Wcodes.shape[0]
    acc = np.empty(pm.size, dtype=np.int32)
    Y = np.empty(pm.size, dtype=np.float64)
    _check(lib().or_linear_a8_pairs(Xq.ctypes.data, sx.ctypes.data, M, K,
                                    Wcodes.ctypes.data, sw.ctypes.data, N,
                                    pm.ctypes.data, pn.ctypes.data, pm.size,
                                    acc.ctypes.data, Y.ctypes.data, threads()),
           "linear_a8_pairs")
    return acc, Y


def linear_a16(Xr, Wcodes, sw):
    """O6: fp64 Y [M, N] from rotated bf16 activations and weight codes."""
    Xr, Wcodes, sw = _c(Xr, np.uint16), _c(Wcodes, np.int8), _c(sw, np.float32)
    M, K = Xr.shape
    N = Wcodes.shape[0]
    Y = np.empty((M, N), dtype=np.float64)
    _check(lib().or_linear_a16(Xr.ctypes.data, M, K, Wcodes.ctypes.data,
                               sw.ctypes.data, N, Y.ctypes.data, threads()),
           "linear_a16")
    return Y


def linear_a16_pairs(Xr, Wcodes, sw, pm, pn):
    Xr, Wcodes, sw = _c(Xr, np.uint16), _c(Wcodes, np.int8), _c(sw, np.float32)
    pm, pn = _c(pm, np.int64), _c(pn, np.int64)
    M, K = Xr.shape
    N = Wcodes.shape[0]
    Y = np.empty(pm.size, dtype=np.float64)
    _check(lib().or_linear_a16_pairs(Xr.ctypes.data, M, K, Wcodes.ctypes.data,
                                     sw.ctypes.data, N, pm.ctypes.data,
                                     pn.ctypes.data, pm.size, Y.ctypes.data,
                                     threads()), "linear_a16_pairs")
    return Y


def swiglu_f64(g, u) -> np.ndarray:
    """O8 in fp64: silu(g) * u, silu(g) = g / (1 + e^-g)."""
    g, u = _c(g, np.float64), _c(u, np.float64)
    h = np.empty(g.shape, dtype=np.float64)
    _check(lib().or_swiglu_f64(g.ctypes.data, u.ctypes.data, g.size, h.ctypes.data), "swiglu_f64")
    return h


def swiglu_bf16(G: np.ndarray, U: np.ndarray) -> np.ndarray:
    """O8: bf16 G, U [M, K] -> bf16 bits of silu(G) * U [M, K]."""
    G, U = _c(G, np.uint16), _c(U, np.uint16)
    M, K = G.shape
    H = np.empty((M, K), dtype=np.uint16)
    _check(lib().or_swiglu_bf16(G.ctypes.data, K, U.ctypes.data, K, M, K, H.ctypes.data), "swiglu_bf16")
    return H


def swiglu_quant_act(G: np.ndarray, U: np.ndarray):
    """O8 then O1+O2+O4: the down projection's A8 operand from gate and up."""
    return rotate_quant_act(swiglu_bf16(G, U))


def modnorm_f64(x, shift, scale, eps: float) -> np.ndarray:
    """O11 in fp64 on rows x [R, K] (fp64 values): (x - mu) / sqrt(var + eps)
    * (1 + scale) + shift, mu and var the row's mean and biased variance."""
    x = _c(np.atleast_2d(x), np.float64)
    sh, sc = _c(shift, np.float64), _c(scale, np.float64)
    R, K = x.shape
    if sh.shape != (K,) or sc.shape != (K,):
        raise ValueError("shift and scale must have K entries")
    h = np.empty_like(x)
    for r in range(R):
        _check(lib().or_modnorm_f64(x[r].ctypes.data, K, sh.ctypes.data, sc.ctypes.data, float(eps),
                                    h[r].ctypes.data), "modnorm_f64")
    return h


def modnorm_bf16(X: np.ndarray, shift, scale, eps: float) -> np.ndarray:
    """O11: bf16 X [M, K], fp32 shift and scale [K] -> bf16 bits of the
    modulated layer norm [M, K]."""
    X = _c(X, np.uint16)
    M, K = X.shape
    sh, sc = _c(shift, np.float32), _c(scale, np.float32)
    if sh.shape != (K,) or sc.shape != (K,):
        raise ValueError("shift and scale must have K entries")
    H = np.empty((M, K), dtype=np.uint16)
    _check(lib().or_modnorm_bf16(X.ctypes.data, K, M, K, sh.ctypes.data, sc.ctypes.data,
                                 float(np.float32(eps)), H.ctypes.data), "modnorm_bf16")
    return H


def modnorm_quant_act(X: np.ndarray, shift, scale, eps: float):
    """O11 then O1+O2+O4: a QKV or gate/up projection's A8 operand from the
    block input X and its modulation."""
    return rotate_quant_act(modnorm_bf16(X, shift, scale, eps))


def quantize_blocks(V: np.ndarray, qmax: int, G: int):
    """O9: symmetric quantisation with one scale per block of G columns ->
    (int8 codes [R, K], fp32 scales [R, K/G])."""
    V = _c(V, np.float64)
    R, K = V.shape
    codes = np.empty((R, K), dtype=np.int8)
    scales = np.empty((R, K // G if G else 0), dtype=np.float32)
    _check(lib().or_quantize_blocks(V.ctypes.data, R, K, G, qmax, codes.ctypes.data,
                                    scales.ctypes.data), "quantize_blocks")
    return codes, scales


def quantize_weights_blocked(W: np.ndarray, bits: int, G: int, rotate: bool = True):
    """O1 (+O2 when rotate) + O9 (+O7 for 4 bits): bf16 W [N, K] -> (codes,
    fp32 block scales [N, K/G]); codes as in quantize_weights."""
    V = rotate_rows(W) if rotate else bf16_to_f64(W)
    codes, scales = quantize_blocks(V, QMAX[bits], G)
    return (codes if bits == 8 else pack_int4(codes)), scales


def linear_a16_blocked(X, Wcodes, sw, G: int):
    """O10: fp64 Y [M, N] from bf16 activations X (already rotated and
    rounded when the weights were rotated) and block-scaled weight codes."""
    X, Wcodes, sw = _c(X, np.uint16), _c(Wcodes, np.int8), _c(sw, np.float32)
    M, K = X.shape
    N = Wcodes.shape[0]
    Y = np.empty((M, N), dtype=np.float64)
    _check(lib().or_linear_a16_blocked(X.ctypes.data, M, K, Wcodes.ctypes.data, sw.ctypes.data,
                                       G, N, Y.ctypes.data, threads()), "linear_a16_blocked")
    return Y


def linear_blocked(X, W, bits: int, G: int, rotate: bool = True):
    """The whole block-scaled decode projection from bf16 inputs (O1-O2, O9,
    O4' when rotated, O10). Returns fp64 Y [M, N]."""
    Wq, sw = quantize_weights_blocked(W, bits, G, rotate)
    K = W.shape[1]
    Xa = rotate_act_bf16(X) if rotate else _c(X, np.uint16)
    return linear_a16_blocked(Xa, weight_codes(Wq, bits, K), sw, G)


def matmul_f64(A, B):
    """Plain fp64 Y = A . B^T (A [M, K], B [N, K])."""
    A, B = _c(A, np.float64), _c(B, np.float64)
    M, K = A.shape
    N = B.shape[0]
    Y = np.empty((M, N), dtype=np.float64)
    _check(lib().or_matmul_f64(A.ctypes.data, M, K, B.ctypes.data, N,
                               Y.ctypes.data, threads()), "matmul_f64")
    return Y


def linear(X, W, bits: int, mode: str):
    """The whole projection from bf16 inputs, as the oracle defines it.

    mode "A8" (W8A8 / W4A8) or "A16" (W8A16 / W4A16).  Returns fp64 Y [M, N]."""
    Wq, sw = quantize_weights(W, bits)
    K = np.asarray(W).shape[1]
    codes = weight_codes(Wq, bits, K)
    if mode == "A8":
        Xq, sx = rotate_quant_act(X)
        return linear_a8(Xq, sx, codes, sw, want_acc=False)[1]
    return linear_a16(rotate_act_bf16(X), codes, sw)
