"""Seeded synthetic inputs for the rotated low-bit linear projection.

Input generation only: no rotation, quantisation or product lives here.  The
CUDA path's harness and the CPU oracle's tests both draw their bf16 tensors from
this module, so both sides see identical inputs.  The arithmetic of the draw is
in ``synth.c`` (SplitMix64 counters -> Box-Muller normals -> scale -> outlier
columns -> nearest-even bf16).  Tensors come back as numpy ``uint16`` arrays of
bf16 bit patterns.

Workload shapes follow the pages: the decode FFN of a Qwen2.5-0.5B-sized model
(896 wide, kvad-gpu internals, "Quantised weights on the GPU"), the 8B-class
batched-decode projections, and the DiT projections of Qwen-Image at 1344x768
(4,032 image rows; TensorFold PR #948, "Receipts").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``synth.c`` into ``libsynth.so`` beside it (gcc, no -march)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    try:
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                        _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.synth_key.restype = ctypes.c_uint64
            lib.synth_key.argtypes = [ctypes.c_char_p, ctypes.c_uint64]
            lib.synth_fill_bf16.restype = ctypes.c_int
            lib.synth_fill_bf16.argtypes = [
                ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64, ctypes.c_double,
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p,
                ctypes.c_int]
            lib.synth_choose_columns.restype = ctypes.c_int
            lib.synth_choose_columns.argtypes = [
                ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]
            _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def key(name: str, seed: int = 0) -> int:
    return int(_load().synth_key(name.encode(), seed & 0xFFFFFFFFFFFFFFFF))


def choose_columns(name: str, cols: int, count: int, seed: int = 0) -> np.ndarray:
    """``count`` distinct seeded column indices of ``[0, cols)``, ascending."""
    out = np.zeros(max(count, 1), dtype=np.int64)
    rc = _load().synth_choose_columns(key(name, seed), cols, count,
                                      out.ctypes.data)
    if rc:
        raise ValueError(f"choose_columns({name!r}, {cols}, {count}) failed: {rc}")
    return out[:count].copy()


def normal_bf16(name: str, rows: int, cols: int, sigma: float,
                outlier_cols=(), mult: float = 1.0, seed: int = 0) -> np.ndarray:
    """bf16 bits [rows, cols]: N(0, sigma), listed columns multiplied by ``mult``."""
    out = np.empty((rows, cols), dtype=np.uint16)
    oc = np.ascontiguousarray(np.asarray(outlier_cols, dtype=np.int64))
    rc = _load().synth_fill_bf16(key(name, seed), rows, cols, float(sigma),
                                 oc.ctypes.data if oc.size else None, oc.size,
                                 float(mult), out.ctypes.data, _threads())
    if rc:
        raise ValueError(f"normal_bf16({name!r}) failed: {rc}")
    return out


def outlier_count(k: int, frac: float) -> int:
    """round(frac * k) columns, the count each workload's outlier share names."""
    return int(round(frac * k))


def tensor(name: str, rows: int, cols: int, sigma: float, frac: float = 0.0,
           mult: float = 1.0, channels=None, seed: int = 0) -> np.ndarray:
    """A weight or activation tensor with seeded outlier columns.

    ``channels`` fixes the outlier columns explicitly; otherwise
    ``round(frac * cols)`` columns are drawn from the key ``name + '/cols'``.
    """
    if channels is None:
        n = outlier_count(cols, frac)
        channels = choose_columns(name + "/cols", cols, n, seed) if n else ()
    return normal_bf16(name, rows, cols, sigma, channels, mult, seed)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (for harness use)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------
# Workload recipes
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class Dist:
    sigma: float
    frac: float = 0.0       # share of outlier columns
    mult: float = 1.0       # their multiplier
    channels: tuple = None  # explicit outlier columns, overrides frac


@dataclass(frozen=True)
class Proj:
    name: str
    N: int   # out features
    K: int   # in features


@dataclass(frozen=True)
class Workload:
    name: str
    projs: tuple
    M: tuple
    bits: tuple
    modes: tuple
    wdist: Dist
    xdist: Dist
    layers: int = 1
    notes: str = ""
    extra: dict = field(default_factory=dict)

    def weight(self, layer: int, proj: Proj, seed: int = 0) -> np.ndarray:
        d = self.wdist
        return tensor(f"{self.name}/L{layer}/{proj.name}/W", proj.N, proj.K,
                      d.sigma, d.frac, d.mult, d.channels, seed)

    def activation(self, call: int, proj: Proj, M: int, seed: int = 0) -> np.ndarray:
        d = self.xdist
        return tensor(f"{self.name}/call{call}/{proj.name}/X{M}", M, proj.K,
                      d.sigma, d.frac, d.mult, d.channels, seed)


# Tiny check: X [4,512] N(0,1) with channels 3 and 300 x25; W [256,512]
# N(0,0.02) with 1% of columns x20; 8-bit weights, fp32 output.
TINY = Workload(
    name="tiny", projs=(Proj("proj", 256, 512),), M=(4,), bits=(8,),
    modes=("W8A16",), wdist=Dist(0.02, 0.01, 20.0),
    xdist=Dist(1.0, mult=25.0, channels=(3, 300)))

# Decode, M=1: Qwen2.5-0.5B-like FFN (896 wide), gate/up 896->4864 and
# down 4864->896; weights N(0,0.02) + 1% columns x20; X N(0,1).
DECODE = Workload(
    name="decode", projs=(Proj("gate", 4864, 896), Proj("up", 4864, 896),
                          Proj("down", 896, 4864)),
    M=(1,), bits=(8, 4), modes=("W8A16", "W4A16"),
    wdist=Dist(0.02, 0.01, 20.0), xdist=Dist(1.0), layers=24,
    notes="1000 seeded calls cycling gate, up, down through the layers")

# Batched decode W4A16, M in {1,8,32,64}: 8B-class projections 4096->12288
# and 12288->4096; weights N(0,0.015) with 0.5% of columns x30.
BATCHED = Workload(
    name="batched", projs=(Proj("up", 12288, 4096), Proj("down", 4096, 12288)),
    M=(1, 8, 32, 64), bits=(4,), modes=("W4A16",),
    wdist=Dist(0.015, 0.005, 30.0), xdist=Dist(1.0))

# DiT projections W8A8 at M=4032 (1344x768 latent / 16): FFN up 3072->12288
# and down 12288->3072; activations N(0,1) with 0.2% of channels x40;
# weights as the decode workload (N(0,0.02), 1% of columns x20).
DIT = Workload(
    name="dit", projs=(Proj("up", 12288, 3072), Proj("down", 3072, 12288)),
    M=(4032,), bits=(8,), modes=("W8A8",),
    wdist=Dist(0.02, 0.01, 20.0), xdist=Dist(1.0, 0.002, 40.0))

# One DiT block's projection chain, 4-bit weights / int8 activations, M=1024
# (512x512), 32 blocks: QKV 3072->9216, out 3072->3072, gate+up 3072->2x12288,
# down 12288->3072.  Weights as the batched workload, activations as DIT.
CHAIN = Workload(
    name="chain", projs=(Proj("qkv", 9216, 3072), Proj("out", 3072, 3072),
                         Proj("gateup", 24576, 3072), Proj("down", 3072, 12288)),
    M=(1024,), bits=(4,), modes=("W8A8",),
    wdist=Dist(0.015, 0.005, 30.0), xdist=Dist(1.0, 0.002, 40.0), layers=32)

WORKLOADS = {w.name: w for w in (TINY, DECODE, BATCHED, DIT, CHAIN)}
