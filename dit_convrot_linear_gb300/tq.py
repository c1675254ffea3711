"""Python binding of ``libtq.so`` (the C ABI of ``include/tq.h``).

Argument marshalling only: every step of the projection runs in the CUDA
library.  Tensors are PyTorch device tensors (PyTorch provides memory and
streams); the functions pass their pointers, sizes and the current stream to
the C entry points of the same names and raise ``TQError`` on any status other
than ``TQ_OK``.  There is no fallback: if the library is missing, ``load()``
raises.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtq.so")

TQ_OK = 0
STATUS = {0: "TQ_OK", 1: "TQ_ERR_NULL", 2: "TQ_ERR_SHAPE", 3: "TQ_ERR_BITS",
          4: "TQ_ERR_MODE", 5: "TQ_ERR_OVERFLOW", 6: "TQ_ERR_ALIGN",
          7: "TQ_ERR_WORKSPACE", 8: "TQ_ERR_CUDA", 9: "TQ_ERR_DEVICE_TIMEOUT",
          10: "TQ_ERR_DEVICE"}
MODES = {"W8A16": 0, "W4A16": 1, "W8A8": 2}
OUT = {"f32": 0, "bf16": 1, "i32": 2}

# exported symbol -> (restype, argtypes)
_P, _I, _Z, _C = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int
SIGNATURES = {
    "tq_status_str": (ctypes.c_char_p, [_C]),
    "tq_last_cuda_error": (_C, []),
    "tq_version": (_C, []),
    "tq_quantize_weights": (_C, [_P, _I, _I, _I, _C, _C, _P, _P, _P]),
    "tq_rotate_quant_act": (_C, [_P, _I, _I, _I, _P, _P, _P]),
    "tq_rotate_act_bf16": (_C, [_P, _I, _I, _I, _P, _P]),
    "tq_linear_workspace_bytes": (_Z, [_I, _I, _I, _C, _C]),
    "tq_linear": (_C, [_P, _I, _I, _I, _P, _P, _I, _C, _C, _P, _C, _I, _P, _Z, _P]),
    "tq_linear_q8": (_C, [_P, _P, _I, _I, _P, _P, _I, _C, _P, _C, _I, _P]),
    "tq_device_status": (_C, [_P]),
    "tq_linear_a8_static": (_C, [_P, _I, _I, _I, _P, _P, _I, _C, _P, _C, _I, _P]),
    "tq_act_tiled_bytes": (_Z, [_I, _I]),
    "tq_rotate_quant_act_tiled": (_C, [_P, _I, _I, _I, _P, _Z, _P, _P]),
    "tq_linear_tiled": (_C, [_P, _P, _I, _I, _P, _P, _I, _C, _P, _C, _I, _P]),
    "tq_swiglu_quant_act_tiled": (_C, [_P, _I, _P, _I, _I, _I, _P, _Z, _P, _P]),
    "tq_modnorm_quant_act_tiled": (_C, [_P, _I, _I, _I, _P, _P, ctypes.c_float, _P, _Z, _P, _P]),
    "tq_linear_swiglu": (_C, [_P, _I, _P, _I, _I, _I, _P, _P, _I, _C, _C, _P, _C, _I, _P]),
    "tq_weights_tiled_bytes": (_Z, [_I, _I]),
    "tq_tile_weights": (_C, [_P, _I, _I, _C, _P, _Z, _P]),
    "tq_linear_tt": (_C, [_P, _P, _I, _I, _P, _P, _I, _C, _P, _C, _I, _P]),
    "tq_linear_tt_ex": (_C, [_P, _P, _I, _I, _P, _P, _I, _C, _P, _P, _C, _I, _P]),
    "tq_split_workspace_bytes": (_Z, []),
    "tq_linear_tt_split": (_C, [_P, _P, _I, _I, _P, _P, _I, _C, _P, _P, _C, _I, _P, _Z, _P]),
    "tq_grouped_bytes": (_C, [_P, _I, _C, ctypes.POINTER(ctypes.c_size_t)]),
    "tq_grouped_create": (_C, [_P, _I, _C, _C, _P, _Z, ctypes.POINTER(ctypes.c_void_p)]),
    "tq_grouped_run": (_C, [_P, _P]),
    "tq_grouped_rotate": (_C, [_P, _P]),
    "tq_grouped_product": (_C, [_P, _P]),
    "tq_grouped_weight_bytes": (_I, [_P]),
    "tq_grouped_destroy": (None, [_P]),
    "tq_chain_bytes": (_C, [_P, _I, _C, ctypes.POINTER(ctypes.c_size_t)]),
    "tq_chain_create": (_C, [_P, _I, _C, _C, _P, _Z, ctypes.POINTER(ctypes.c_void_p)]),
    "tq_quantize_weights_blocked": (_C, [_P, _I, _I, _I, _C, _C, _C, _P, _P, _P]),
    "tq_linear_blocked": (_C, [_P, _I, _I, _I, _P, _P, _C, _I, _C, _C, _P, _C, _I, _P]),
}


class Epilogue(ctypes.Structure):
    """``tq_epilogue``: Y = R + gate * (product + bias)."""
    _fields_ = [("bias", _P), ("gate", _P), ("residual", _P), ("ldr", _I), ("rtype", _C)]


class A16Call(ctypes.Structure):
    """``tq_a16_call``: one call of a grouped plan."""
    _fields_ = [("X", _P), ("ldx", _I), ("Wq", _P), ("sw", _P), ("Y", _P), ("ldy", _I),
                ("M", _I), ("N", _I), ("K", _I)]


class ChainCall(ctypes.Structure):
    """``tq_chain_call``: one call of a chained plan (U NULL, or the up rows)."""
    _fields_ = [("call", A16Call), ("U", _P), ("ldu", _I)]

_lib = None


class TQError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        name = STATUS.get(status, str(status))
        extra = ""
        if status == 8 and _lib is not None:
            extra = f" (cuda error {_lib.tq_last_cuda_error()})"
        super().__init__(f"{where}: {name}{extra}")


def load(path: str = LIB_PATH):
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "dit_convrot_linear_gb300.build.build()")
        import torch  # noqa: F401  (load PyTorch's CUDA runtime first)
        L = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def lib():
    return load()


def _stream(stream=None) -> int:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def _check(rc: int, where: str):
    if rc != TQ_OK:
        raise TQError(rc, where)


# ---- host-side checks of what the C ABI cannot see: tensor sizes and types.
# A call with a buffer smaller than its sizes say would write or read past it
# on the device, so the binding refuses it before the call.

def _dt(name):
    import torch
    return {"f32": torch.float32, "bf16": torch.bfloat16, "i32": torch.int32,
            "i8": torch.int8, "u8": torch.uint8}[name]


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def _req(t, what: str, dtype=None, rows: int = None, cols: int = None, nbytes: int = None,
         dense: bool = False):
    if t is None:
        raise ValueError(f"{what} is required")
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{what} is {t.dtype}, expected {dtype}")
    if rows is not None:
        if t.dim() != 2 or t.shape[0] < rows or t.shape[1] < cols or (t.numel() and t.stride(1) != 1):
            raise ValueError(f"{what} must be a row-major [>= {rows}, >= {cols}] matrix, got "
                             f"shape {tuple(t.shape)} strides {t.stride()}")
        if dense and t.numel() and t.stride(0) != cols:
            raise ValueError(f"{what} must be dense (row stride {cols})")
    if nbytes is not None and _nbytes(t) < nbytes:
        raise ValueError(f"{what} holds {_nbytes(t)} bytes, needs {nbytes}")


def _weights(Wq, sw, N: int, K: int, bits: int):
    _req(Wq, "Wq", nbytes=N * K * bits // 8)
    _req(sw, "sw", dtype=_dt("f32"), nbytes=4 * N)


def status_str(s: int) -> str:
    return lib().tq_status_str(s).decode()


def version() -> int:
    return lib().tq_version()


def quantize_weights(W, bits: int, codes=None, scales=None, stream=None):
    """bf16 W [N, K] (row stride W.stride(0)) -> (codes, fp32 scales [N])."""
    import torch
    N, K = W.shape
    if codes is None:
        codes = torch.empty((N, K if bits == 8 else K // 2),
                            dtype=torch.int8 if bits == 8 else torch.uint8, device=W.device)
    if scales is None:
        scales = torch.empty(N, dtype=torch.float32, device=W.device)
    _req(W, "W", dtype=torch.bfloat16, rows=N, cols=K)
    _req(codes, "codes", nbytes=N * K * bits // 8)
    _req(scales, "scales", dtype=torch.float32, nbytes=4 * N)
    _check(lib().tq_quantize_weights(_ptr(W), N, K, W.stride(0), bits, 256, _ptr(codes),
                                     _ptr(scales), _stream(stream)), "tq_quantize_weights")
    return codes, scales


def quantize_weights_blocked(W, bits: int, G: int, rotate: bool = True, codes=None, scales=None,
                             stream=None):
    """bf16 W [N, K] -> (codes, fp32 block scales [N, K / G]): one scale per
    block of G columns, of the rotated row (rotate) or of W as it is."""
    import torch
    N, K = W.shape
    if codes is None:
        codes = torch.empty((N, K if bits == 8 else K // 2),
                            dtype=torch.int8 if bits == 8 else torch.uint8, device=W.device)
    if scales is None:
        scales = torch.empty((N, K // G if G > 0 else 0), dtype=torch.float32, device=W.device)
    _req(W, "W", dtype=torch.bfloat16, rows=N, cols=K)
    _req(codes, "codes", nbytes=N * K * bits // 8)
    if G > 0:
        _req(scales, "scales", dtype=torch.float32, nbytes=4 * N * (K // G))
    _check(lib().tq_quantize_weights_blocked(_ptr(W), N, K, W.stride(0), bits, G, int(rotate), _ptr(codes),
                                             _ptr(scales), _stream(stream)), "tq_quantize_weights_blocked")
    return codes, scales


def linear_blocked(X, Wq, sw, N: int, bits: int, G: int, rotate: bool = True, Y=None, out: str = "f32",
                   stream=None):
    """Y [M, N] = the block-scaled decode product of bf16 X [M, K] (M <= 8)
    with (Wq, sw) from quantize_weights_blocked (same G and rotate)."""
    import torch
    M, K = X.shape
    if out not in ("f32", "bf16"):
        raise ValueError("tq_linear_blocked writes f32 or bf16")
    if Y is None:
        Y = torch.empty((M, N), dtype=_dt(out), device=X.device)
    _req(X, "X", dtype=torch.bfloat16, rows=M, cols=K)
    _req(Wq, "Wq", nbytes=N * K * bits // 8)
    if G > 0:
        _req(sw, "sw", dtype=torch.float32, nbytes=4 * N * (K // G))
    _req(Y, "Y", dtype=_dt(out), rows=M, cols=N)
    _check(lib().tq_linear_blocked(_ptr(X), M, K, X.stride(0), _ptr(Wq), _ptr(sw), G, N, bits, int(rotate),
                                   _ptr(Y), OUT[out], Y.stride(0), _stream(stream)), "tq_linear_blocked")
    return Y


def rotate_quant_act(X, Xq=None, sx=None, stream=None):
    import torch
    M, K = X.shape
    if Xq is None:
        Xq = torch.empty((M, K), dtype=torch.int8, device=X.device)
    if sx is None:
        sx = torch.empty(M, dtype=torch.float32, device=X.device)
    _req(X, "X", dtype=torch.bfloat16, rows=M, cols=K)
    _req(Xq, "Xq", dtype=torch.int8, rows=M, cols=K, dense=True)
    _req(sx, "sx", dtype=torch.float32, nbytes=4 * M)
    _check(lib().tq_rotate_quant_act(_ptr(X), M, K, X.stride(0), _ptr(Xq), _ptr(sx),
                                     _stream(stream)), "tq_rotate_quant_act")
    return Xq, sx


def rotate_act_bf16(X, Xr=None, stream=None):
    import torch
    M, K = X.shape
    if Xr is None:
        Xr = torch.empty((M, K), dtype=torch.bfloat16, device=X.device)
    _req(X, "X", dtype=torch.bfloat16, rows=M, cols=K)
    _req(Xr, "Xr", dtype=torch.bfloat16, rows=M, cols=K, dense=True)
    _check(lib().tq_rotate_act_bf16(_ptr(X), M, K, X.stride(0), _ptr(Xr), _stream(stream)),
           "tq_rotate_act_bf16")
    return Xr


def linear_workspace_bytes(M: int, K: int, N: int, bits: int, mode: str) -> int:
    return int(lib().tq_linear_workspace_bytes(M, K, N, bits, MODES[mode]))


def linear(X, Wq, sw, N: int, bits: int, mode: str, Y=None, out: str = "f32",
           workspace=None, stream=None):
    """Y [M, N] = the rotated low-bit product of bf16 X [M, K] with (Wq, sw)."""
    import torch
    M, K = X.shape
    if out not in ("f32", "bf16"):
        raise ValueError("tq_linear writes f32 or bf16")
    if Y is None:
        Y = torch.empty((M, N), dtype=_dt(out), device=X.device)
    _req(X, "X", dtype=torch.bfloat16, rows=M, cols=K)
    _weights(Wq, sw, N, K, bits)
    _req(Y, "Y", dtype=_dt(out), rows=M, cols=N)
    need = linear_workspace_bytes(M, K, N, bits, mode)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=X.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().tq_linear(_ptr(X), M, K, X.stride(0), _ptr(Wq), _ptr(sw), N, bits,
                           MODES[mode], _ptr(Y), OUT[out], Y.stride(0), _ptr(workspace),
                           ws_bytes, _stream(stream)), "tq_linear")
    return Y


def linear_swiglu(G, U, Wq, sw, N: int, bits: int, mode: str, Y=None, out: str = "f32", stream=None):
    """Y [M, N] = the decode product (A16, M <= 8) of h = bf16(silu(G) * U):
    G and U bf16 [M, K] with any row stride (for example the two halves of a
    fused gate+up output)."""
    import torch
    M, K = G.shape
    if tuple(U.shape) != (M, K):
        raise ValueError(f"U is {tuple(U.shape)}, expected {(M, K)}")
    if out not in ("f32", "bf16"):
        raise ValueError("tq_linear_swiglu writes f32 or bf16")
    if Y is None:
        Y = torch.empty((M, N), dtype=_dt(out), device=G.device)
    _req(G, "G", dtype=torch.bfloat16, rows=M, cols=K)
    _req(U, "U", dtype=torch.bfloat16, rows=M, cols=K)
    _weights(Wq, sw, N, K, bits)
    _req(Y, "Y", dtype=_dt(out), rows=M, cols=N)
    _check(lib().tq_linear_swiglu(_ptr(G), G.stride(0), _ptr(U), U.stride(0), M, K, _ptr(Wq), _ptr(sw), N, bits,
                                  MODES[mode], _ptr(Y), OUT[out], Y.stride(0), _stream(stream)),
           "tq_linear_swiglu")
    return Y


def linear_q8(Xq, sx, Wq, sw, N: int, bits: int, Y=None, out: str = "f32", stream=None):
    import torch
    M, K = Xq.shape
    if Y is None:
        Y = torch.empty((M, N), dtype=_dt(out), device=Xq.device)
    _req(Xq, "Xq", dtype=torch.int8, rows=M, cols=K, dense=True)
    if out != "i32":
        _req(sx, "sx", dtype=torch.float32, nbytes=4 * M)
    _weights(Wq, sw, N, K, bits)
    _req(Y, "Y", dtype=_dt(out), rows=M, cols=N)
    _check(lib().tq_linear_q8(_ptr(Xq), _ptr(sx), M, K, _ptr(Wq), _ptr(sw), N, bits, _ptr(Y),
                              OUT[out], Y.stride(0), _stream(stream)), "tq_linear_q8")
    return Y


def act_tiled_bytes(M: int, K: int) -> int:
    return int(lib().tq_act_tiled_bytes(M, K))


def rotate_quant_act_tiled(X, At=None, sx=None, stream=None):
    """Rotation + per-token int8 quantisation written in the A8 product's own
    operand form (fp16 codes, tiled); returns (At, sx) for linear_tiled."""
    import torch
    M, K = X.shape
    need = act_tiled_bytes(M, K)
    if At is None:
        At = torch.empty(max(need, 1), dtype=torch.uint8, device=X.device)
    if sx is None:
        sx = torch.empty(M, dtype=torch.float32, device=X.device)
    _req(X, "X", dtype=torch.bfloat16, rows=M, cols=K)
    _req(At, "At", nbytes=need)
    _req(sx, "sx", dtype=torch.float32, nbytes=4 * M)
    _check(lib().tq_rotate_quant_act_tiled(_ptr(X), M, K, X.stride(0), _ptr(At), _nbytes(At),
                                           _ptr(sx), _stream(stream)), "tq_rotate_quant_act_tiled")
    return At, sx


def modnorm_quant_act_tiled(X, shift, scale, eps=1e-6, At=None, sx=None, stream=None):
    """A QKV or gate/up projection's input from the block input X (bf16
    [M, K], any row stride) and its modulation (fp32 shift and scale [K]):
    bf16((X - mean) / sqrt(var + eps) * (1 + scale) + shift) per row, rotated
    and quantised into the tiled operand.  Returns (At, sx) for linear_tiled /
    linear_tt."""
    import torch
    M, K = X.shape
    need = act_tiled_bytes(M, K)
    if At is None:
        At = torch.empty(max(need, 1), dtype=torch.uint8, device=X.device)
    if sx is None:
        sx = torch.empty(M, dtype=torch.float32, device=X.device)
    _req(X, "X", dtype=torch.bfloat16, rows=M, cols=K)
    _req(shift, "shift", dtype=torch.float32, nbytes=4 * K)
    _req(scale, "scale", dtype=torch.float32, nbytes=4 * K)
    _req(At, "At", nbytes=need)
    _req(sx, "sx", dtype=torch.float32, nbytes=4 * M)
    _check(lib().tq_modnorm_quant_act_tiled(_ptr(X), M, K, X.stride(0), _ptr(shift), _ptr(scale), float(eps),
                                            _ptr(At), _nbytes(At), _ptr(sx), _stream(stream)),
           "tq_modnorm_quant_act_tiled")
    return At, sx


def swiglu_quant_act_tiled(G, U, At=None, sx=None, stream=None):
    """The down projection's input from gate G and up U (bf16 [M, K], any row
    stride): bf16(silu(G) * U), rotated and quantised into the tiled operand.
    Returns (At, sx) for linear_tiled / linear_tt."""
    import torch
    M, K = G.shape
    if tuple(U.shape) != (M, K):
        raise ValueError(f"U is {tuple(U.shape)}, expected {(M, K)}")
    need = act_tiled_bytes(M, K)
    if At is None:
        At = torch.empty(max(need, 1), dtype=torch.uint8, device=G.device)
    if sx is None:
        sx = torch.empty(M, dtype=torch.float32, device=G.device)
    _req(G, "G", dtype=torch.bfloat16, rows=M, cols=K)
    _req(U, "U", dtype=torch.bfloat16, rows=M, cols=K)
    _req(At, "At", nbytes=need)
    _req(sx, "sx", dtype=torch.float32, nbytes=4 * M)
    _check(lib().tq_swiglu_quant_act_tiled(_ptr(G), G.stride(0), _ptr(U), U.stride(0), M, K, _ptr(At),
                                           _nbytes(At), _ptr(sx), _stream(stream)),
           "tq_swiglu_quant_act_tiled")
    return At, sx


def linear_tiled(At, sx, M: int, K: int, Wq, sw, N: int, bits: int, Y=None, out: str = "f32",
                 stream=None):
    import torch
    if Y is None:
        Y = torch.empty((M, N), dtype=_dt(out), device=At.device)
    _req(At, "At", nbytes=act_tiled_bytes(M, K))
    if out != "i32":
        _req(sx, "sx", dtype=torch.float32, nbytes=4 * M)
    _weights(Wq, sw, N, K, bits)
    _req(Y, "Y", dtype=_dt(out), rows=M, cols=N)
    _check(lib().tq_linear_tiled(_ptr(At), _ptr(sx), M, K, _ptr(Wq), _ptr(sw), N, bits, _ptr(Y),
                                 OUT[out], Y.stride(0), _stream(stream)), "tq_linear_tiled")
    return Y


def weights_tiled_bytes(N: int, K: int) -> int:
    return int(lib().tq_weights_tiled_bytes(N, K))


def tile_weights(Wq, N: int, K: int, bits: int, Wt=None, stream=None):
    """The codes of ``quantize_weights`` widened once into the A8 product's
    operand form (fp16 tiles) for ``linear_tt``."""
    import torch
    need = weights_tiled_bytes(N, K)
    if Wt is None:
        Wt = torch.empty(max(need, 1), dtype=torch.uint8, device=Wq.device)
    _req(Wq, "Wq", nbytes=N * K * bits // 8)
    _req(Wt, "Wt", nbytes=need)
    _check(lib().tq_tile_weights(_ptr(Wq), N, K, bits, _ptr(Wt), _nbytes(Wt), _stream(stream)),
           "tq_tile_weights")
    return Wt


def split_workspace_bytes() -> int:
    return int(lib().tq_split_workspace_bytes())


def split_workspace(device="cuda"):
    """A zeroed split workspace for ``linear_tt(..., split=ws)`` (one per
    stream; every completed call leaves it zeroed)."""
    import torch
    return torch.zeros(split_workspace_bytes(), dtype=torch.uint8, device=device)


def linear_tt(At, sx, M: int, K: int, Wt, sw, N: int, bits: int, Y=None, out: str = "f32",
              split=None, stream=None):
    """The A8 product with both operands tiled (``rotate_quant_act_tiled`` and
    ``tile_weights``).  ``split``: a workspace from ``split_workspace()`` lets
    the product split the K steps of its last waves of tiles over every CTA
    pair (tq_linear_tt_split)."""
    import torch
    if Y is None:
        Y = torch.empty((M, N), dtype=_dt(out), device=At.device)
    _req(At, "At", nbytes=act_tiled_bytes(M, K))
    if out != "i32":
        _req(sx, "sx", dtype=torch.float32, nbytes=4 * M)
    _req(Wt, "Wt", nbytes=weights_tiled_bytes(N, K))
    _req(sw, "sw", dtype=torch.float32, nbytes=4 * N)
    _req(Y, "Y", dtype=_dt(out), rows=M, cols=N)
    if split is not None:
        _req(split, "split", nbytes=split_workspace_bytes())
        _check(lib().tq_linear_tt_split(_ptr(At), _ptr(sx), M, K, _ptr(Wt), _ptr(sw), N, bits, None, _ptr(Y),
                                        OUT[out], Y.stride(0), _ptr(split), _nbytes(split), _stream(stream)),
               "tq_linear_tt_split")
        return Y
    _check(lib().tq_linear_tt(_ptr(At), _ptr(sx), M, K, _ptr(Wt), _ptr(sw), N, bits, _ptr(Y),
                              OUT[out], Y.stride(0), _stream(stream)), "tq_linear_tt")
    return Y


def linear_tt_ex(At, sx, M: int, K: int, Wt, sw, N: int, bits: int, Y=None, out: str = "f32",
                 bias=None, gate=None, residual=None, split=None, stream=None):
    """``linear_tt`` with the fused epilogue Y = residual + gate * (product + bias)
    (each optional; ``residual`` may be ``Y`` itself)."""
    import torch
    if out not in ("f32", "bf16"):
        raise ValueError("the epilogue writes f32 or bf16")
    if Y is None:
        Y = torch.empty((M, N), dtype=_dt(out), device=At.device)
    _req(At, "At", nbytes=act_tiled_bytes(M, K))
    _req(sx, "sx", dtype=torch.float32, nbytes=4 * M)
    _req(Wt, "Wt", nbytes=weights_tiled_bytes(N, K))
    _req(sw, "sw", dtype=torch.float32, nbytes=4 * N)
    _req(Y, "Y", dtype=_dt(out), rows=M, cols=N)
    if bias is not None:
        _req(bias, "bias", dtype=torch.float32, nbytes=4 * N)
    if gate is not None:
        _req(gate, "gate", dtype=torch.float32, nbytes=4 * N)
    rtype, ldr = 0, 0
    if residual is not None:
        if residual.dtype not in (torch.float32, torch.bfloat16):
            raise ValueError("residual must be float32 or bfloat16")
        _req(residual, "residual", dtype=residual.dtype, rows=M, cols=N)
        rtype = OUT["f32" if residual.dtype == torch.float32 else "bf16"]
        ldr = residual.stride(0)
    epi = Epilogue(_ptr(bias), _ptr(gate), _ptr(residual), ldr, rtype)
    if split is not None:
        _req(split, "split", nbytes=split_workspace_bytes())
        _check(lib().tq_linear_tt_split(_ptr(At), _ptr(sx), M, K, _ptr(Wt), _ptr(sw), N, bits,
                                        ctypes.addressof(epi), _ptr(Y), OUT[out], Y.stride(0), _ptr(split),
                                        _nbytes(split), _stream(stream)), "tq_linear_tt_split")
        return Y
    _check(lib().tq_linear_tt_ex(_ptr(At), _ptr(sx), M, K, _ptr(Wt), _ptr(sw), N, bits,
                                 ctypes.addressof(epi), _ptr(Y), OUT[out], Y.stride(0),
                                 _stream(stream)), "tq_linear_tt_ex")
    return Y


def linear_a8_static(X, Wq, sw, N: int, bits: int, Y, out: str = "f32", stream=None):
    """The W8A8 / W4A8 product using the library's fixed device scratch
    instead of a workspace (for callers that may not allocate device memory).
    ``Y`` must be given; nothing is allocated."""
    import torch
    M, K = X.shape
    if out not in ("f32", "bf16"):
        raise ValueError("tq_linear_a8_static writes f32 or bf16")
    _req(X, "X", dtype=torch.bfloat16, rows=M, cols=K)
    _weights(Wq, sw, N, K, bits)
    _req(Y, "Y", dtype=_dt(out), rows=M, cols=N)
    _check(lib().tq_linear_a8_static(_ptr(X), M, K, X.stride(0), _ptr(Wq), _ptr(sw), N, bits,
                                     _ptr(Y), OUT[out], Y.stride(0), _stream(stream)),
           "tq_linear_a8_static")
    return Y


def device_status(stream=None) -> int:
    """Synchronise and return the library's device status (0 = TQ_OK)."""
    return int(lib().tq_device_status(_stream(stream)))


def grouped_bytes(calls, bits: int) -> int:
    """Device bytes a plan of these ``A16Call`` records needs."""
    arr = (A16Call * max(len(calls), 1))(*calls)
    out = ctypes.c_size_t(0)
    _check(lib().tq_grouped_bytes(ctypes.addressof(arr), len(calls), bits, ctypes.byref(out)),
           "tq_grouped_bytes")
    return int(out.value)


def chain_bytes(calls, bits: int) -> int:
    """Device bytes a chained plan of these ``ChainCall`` records needs."""
    arr = (ChainCall * max(len(calls), 1))(*calls)
    out = ctypes.c_size_t(0)
    _check(lib().tq_chain_bytes(ctypes.addressof(arr), len(calls), bits, ctypes.byref(out)), "tq_chain_bytes")
    return int(out.value)


class GroupedPlan:
    """Independent A16 calls run as one pass over their weights
    (``tq_grouped_create`` / ``tq_grouped_run``).

    ``calls`` is a list of ``(X, Wq, sw, N, Y)``: bf16 X [M, K] (M <= 8), the
    codes and row scales of ``quantize_weights`` with ``bits``, and Y [M, N] of
    dtype ``out``.  The plan keeps references to every tensor (their addresses
    are in its tables) and owns the device buffer of its tables."""

    def __init__(self, calls, bits: int, out: str = "f32"):
        import torch
        if out not in ("f32", "bf16"):
            raise ValueError("a grouped plan writes f32 or bf16")
        recs, keep, dev = [], [], None
        for (X, Wq, sw, N, Y) in calls:
            M, K = X.shape
            _req(X, "X", dtype=torch.bfloat16, rows=M, cols=K)
            _weights(Wq, sw, N, K, bits)
            _req(Y, "Y", dtype=_dt(out), rows=M, cols=N)
            dev = X.device if dev is None else dev
            recs.append(A16Call(_ptr(X), X.stride(0), _ptr(Wq), _ptr(sw), _ptr(Y), Y.stride(0),
                                M, N, K))
            keep.extend([X, Wq, sw, Y])
        need = grouped_bytes(recs, bits)
        self.buffer = torch.empty(max(need, 1), dtype=torch.uint8,
                                  device=dev if dev is not None else "cuda")
        arr = (A16Call * max(len(recs), 1))(*recs)
        h = ctypes.c_void_p(None)
        _check(lib().tq_grouped_create(ctypes.addressof(arr), len(recs), bits, OUT[out],
                                       _ptr(self.buffer), _nbytes(self.buffer), ctypes.byref(h)),
               "tq_grouped_create")
        self._h = h
        self._keep = keep
        self.bits = bits
        self.ncalls = len(recs)

    def run(self, stream=None):
        if self._h is None:
            raise ValueError("the plan is closed")
        _check(lib().tq_grouped_run(self._h, _stream(stream)), "tq_grouped_run")

    def rotate(self, stream=None):
        """The first launch of run(): every call's input rotation."""
        if self._h is None:
            raise ValueError("the plan is closed")
        _check(lib().tq_grouped_rotate(self._h, _stream(stream)), "tq_grouped_rotate")

    def product(self, stream=None):
        """The second launch of run(): the products, from the rotated inputs."""
        if self._h is None:
            raise ValueError("the plan is closed")
        _check(lib().tq_grouped_product(self._h, _stream(stream)), "tq_grouped_product")

    @property
    def weight_bytes(self) -> int:
        return int(lib().tq_grouped_weight_bytes(self._h)) if self._h is not None else 0

    def close(self):
        if getattr(self, "_h", None) is not None and _lib is not None:
            _lib.tq_grouped_destroy(self._h)
        self._h = None

    def __del__(self):
        self.close()


class ChainPlan(GroupedPlan):
    """Dependent A16 calls run in order in one launch (``tq_chain_create``,
    run with ``tq_grouped_run``): call c may read any earlier call's Y.

    ``calls`` is a list of ``(X, Wq, sw, N, Y)`` or ``(X, Wq, sw, N, Y, U)``:
    as ``GroupedPlan``'s, U (bf16 [M, K], any row stride) making the call's
    input the SwiGLU of X and U."""

    def __init__(self, calls, bits: int, out: str = "f32"):
        import torch
        if out not in ("f32", "bf16"):
            raise ValueError("a chained plan writes f32 or bf16")
        recs, keep, dev = [], [], None
        for c in calls:
            X, Wq, sw, N, Y = c[:5]
            U = c[5] if len(c) > 5 else None
            M, K = X.shape
            _req(X, "X", dtype=torch.bfloat16, rows=M, cols=K)
            if U is not None:
                if tuple(U.shape) != (M, K):
                    raise ValueError(f"U is {tuple(U.shape)}, expected {(M, K)}")
                _req(U, "U", dtype=torch.bfloat16, rows=M, cols=K)
            _weights(Wq, sw, N, K, bits)
            _req(Y, "Y", dtype=_dt(out), rows=M, cols=N)
            dev = X.device if dev is None else dev
            recs.append(ChainCall(A16Call(_ptr(X), X.stride(0), _ptr(Wq), _ptr(sw), _ptr(Y), Y.stride(0),
                                          M, N, K),
                                  _ptr(U), U.stride(0) if U is not None else 0))
            keep.extend([X, Wq, sw, Y] + ([U] if U is not None else []))
        need = chain_bytes(recs, bits)
        self.buffer = torch.empty(max(need, 1), dtype=torch.uint8,
                                  device=dev if dev is not None else "cuda")
        arr = (ChainCall * max(len(recs), 1))(*recs)
        h = ctypes.c_void_p(None)
        _check(lib().tq_chain_create(ctypes.addressof(arr), len(recs), bits, OUT[out],
                                     _ptr(self.buffer), _nbytes(self.buffer), ctypes.byref(h)),
               "tq_chain_create")
        self._h = h
        self._keep = keep
        self.bits = bits
        self.ncalls = len(recs)

