"""Test helpers: moving bf16 bit patterns between numpy and torch, and the
parity statistics (max |diff|, relative L2, worst row) used by every test."""
import numpy as np

# Fixed tolerances of the comparison (see the design notes):
REL_L2_Y = 1e-4          # floating outputs vs the oracle on the same operands
CODE_FLIP_FRAC = 1e-3    # A8 codes: at most 0.1% differ, each by at most 1
SCALE_REL = 2.0 ** -20   # A8 token scales
ULP_FLIP_FRAC = 1e-3     # A16 bf16 operands: at most 0.1% differ, by 1 ulp


def to_dev_bf16(bits, device="cuda"):
    import torch
    a = np.ascontiguousarray(bits, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)


def bf16_bits(t):
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_np(t):
    return t.detach().cpu().numpy()


def rel_l2(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def parity_report(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    d = np.abs(got - ref)
    rows = np.linalg.norm(got - ref, axis=-1) / np.maximum(np.linalg.norm(ref, axis=-1), 1e-300)
    return {"max_abs": float(d.max()) if d.size else 0.0,
            "rel_l2": rel_l2(got, ref),
            "worst_row": float(rows.max()) if rows.size else 0.0}


def bf16_ulp_diff(a_bits, b_bits):
    """|difference| in bf16 units in the last place (sign-magnitude order)."""
    def key(b):
        b = np.asarray(b, dtype=np.int64)
        return np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)
    return np.abs(key(a_bits) - key(b_bits))


def check_codes_close(got, ref, frac=CODE_FLIP_FRAC):
    got = np.asarray(got, dtype=np.int32)
    ref = np.asarray(ref, dtype=np.int32)
    d = np.abs(got - ref)
    assert d.max(initial=0) <= 1, f"a code differs by {d.max()}"
    flips = np.count_nonzero(d)
    assert flips <= frac * d.size, f"{flips} of {d.size} codes differ"
    return flips


def untile_codes(At, M, K, rows=None):
    """Codes [M, K] (int) from a tiled activation operand (test decoding of the
    library's private layout: fp16 codes in 128-row x 64-column tiles, tile
    (mt, kt) at halfword (mt * ceil(K/64) + kt) * 8192, core matrix (r/8, k/8)
    of 64 halfwords at ((r/8) * 8 + k/8) * 64, element (r%8, k%8) at
    (r%8) * 8 + k%8).  With `rows`, only those rows, in that order."""
    import torch
    KT = (K + 63) // 64
    h = At.view(torch.uint8)[: ((M + 255) // 256) * 2 * KT * 16384].view(torch.float16).cpu().numpy()
    m = (np.arange(M) if rows is None else np.asarray(rows))[:, None]
    k = np.arange(K)[None, :]
    idx = ((m // 128) * KT + k // 64) * 8192 + (((m % 128) // 8) * 8 + (k % 64) // 8) * 64 + (m % 8) * 8 + k % 8
    return h[idx].astype(np.int64)


def act_trailer(tq, At, M, K):
    """The 12 bounds of a tiled activation operand's trailer (the library's
    private layout, decoded for tests): after the tiles, 16 copies 128 bytes
    apart of 12 32-bit words; bound j is the maximum over the copies."""
    start = tq.act_tiled_bytes(M, K) - 2048
    raw = to_np(At[start:start + 2048]).view(np.uint32).reshape(16, 32)
    return raw[:, :12].max(axis=0).astype(np.int64)
