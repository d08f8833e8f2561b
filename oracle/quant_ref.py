"""ORACLE -- test infrastructure, not part of the product.

Plain numpy (fp64) definition of the activation quantiser that produces the
W4A4 operator's activation inputs.  "SVDQuant W4A4 on Blackwell" §1 says the
operator is the compute-bound half of SVDQuant (the other half produces its
activation inputs), §2 gives the tensors it writes (act, ascales,
lora_act_in) and §3.1 their formats (two E2M1 codes per byte, one FP8-E4M3
scale per 16 K elements, single-level scaling); §3.3 calls LA the LoRA-down
activation.  The page does not spell the quantiser out; this is the plain
NVFP4 reading, per group of 16 consecutive k in a row m:

    amax  = max |x[m, k]|                                   (over the group)
    sbyte = E4M3 nearest value to amax / 6, ties to the even byte,
            saturating at 448 (byte 0x7E); s = its value
    code  = E2M1 nearest value to x / s, ties to the even code, saturating at
            6; every code of the group is 0 when s == 0; a code of magnitude 0
            is stored as +0 (code 0)
    lora_act_in[m, r] = sum_k x[m, k] * lora_down[r, k]

Rounding decisions are taken on fp64 quotients.  For 16-bit x they are the
decisions of the exact quotients: a tie point is exactly representable and a
quotient that is not on it lies at least 2^-11 (relative) away, far beyond
fp64's 2^-53.  Only tests/, the package's smoke check and bench.py's
CPU-baseline leg may import this module.
"""

from __future__ import annotations

import numpy as np

from .prepack_ref import _decode16, pack_scales
from .svdq_ref import _np_bytes, e4m3

# E2M1 magnitudes by code 0..7 (OCP Microscaling formats, FP4 E2M1)
E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e4m3_values() -> np.ndarray:
    """Values of the finite non-negative E4M3 bytes 0x00..0x7E, ascending."""
    return np.array([e4m3(b) for b in range(0x7F)], dtype=np.float64)


_E4M3 = None


def _e4m3_table() -> np.ndarray:
    global _E4M3
    if _E4M3 is None:
        _E4M3 = e4m3_values()
    return _E4M3


def round_to_table(q, table: np.ndarray) -> np.ndarray:
    """Index of the entry of an ascending table nearest to each q >= 0; a tie
    goes to the even index; q beyond the last entry gives the last index."""
    q = np.asarray(q, dtype=np.float64)
    hi = np.clip(np.searchsorted(table, q, side="left"), 0, len(table) - 1)
    lo = np.clip(hi - 1, 0, len(table) - 1)
    d_lo = q - table[lo]
    d_hi = table[hi] - q
    pick = np.where(d_hi < d_lo, hi, lo)
    pick = np.where(d_hi == d_lo, np.where(hi % 2 == 0, hi, lo), pick)
    pick = np.where(q >= table[-1], len(table) - 1, pick)
    return pick.astype(np.int64)


def round_e4m3(q) -> np.ndarray:
    """E4M3 byte nearest to q >= 0 (ties to even, saturating at 448)."""
    return round_to_table(q, _e4m3_table()).astype(np.uint8)


def round_e2m1(q) -> np.ndarray:
    """E2M1 code of q: magnitude nearest to |q| (ties to even, saturating at
    6), sign bit 3 set only for a negative q of non-zero magnitude."""
    q = np.asarray(q, dtype=np.float64)
    mag = round_to_table(np.abs(q), E2M1_VALUES)
    sign = (q < 0) & (mag > 0)
    return (mag | (sign.astype(np.int64) << 3)).astype(np.uint8)


def decode_x(x, M: int, K: int, half: bool = False) -> np.ndarray:
    """fp64 values of 16-bit x [M, K] (bf16 bits, or IEEE fp16 with half)."""
    bits = _np_bytes(x, np.uint16).reshape(M, K)
    return _decode16(bits, half).astype(np.float64)


def quantize_act(x, M: int, K: int, half: bool = False, packed: bool = False):
    """(act uint8 [M, K/2], ascales) of 16-bit x [M, K]; ascales is uint8
    [K/16, M], or uint32 [K/64, M] words (byte g = group 4s + g) with packed."""
    if K % 16:
        raise ValueError("K must be a multiple of 16")
    X = decode_x(x, M, K, half).reshape(M, K // 16, 16)
    amax = np.abs(X).max(axis=2)
    sbyte = round_e4m3(amax / 6.0)
    s = _e4m3_table()[sbyte]
    with np.errstate(divide="ignore", invalid="ignore"):
        Q = np.where(s[..., None] > 0, X / np.where(s > 0, s, 1.0)[..., None], 0.0)
    codes = round_e2m1(Q).reshape(M, K)
    act = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    ascales = np.ascontiguousarray(sbyte.T)
    if packed:
        if K % 64:
            raise ValueError("packed scales need K a multiple of 64")
        return act, pack_scales(ascales, M, K)
    return act, ascales


def lora_down(x, ld, M: int, K: int, R: int, half: bool = False) -> np.ndarray:
    """fp64 [M, R]: sum_k x[m, k] * lora_down[r, k] (lora_down 16-bit [R, K])."""
    X = decode_x(x, M, K, half)
    L = decode_x(ld, R, K, half)
    return X @ L.T
