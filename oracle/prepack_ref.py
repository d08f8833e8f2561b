"""ORACLE -- test infrastructure, not part of the product.

Plain numpy definitions of the weight-side prepack ("SVDQuant W4A4 on
Blackwell" §3.1 block scales fed per 64-wide MMA step; §6.3 LoRA folded into
the main accumulator, with the weight-side factors settled offline): what a
prepacked weight holds, element by element.  Only tests/, the package's smoke
check and bench.py's CPU-baseline leg may import this module.

- packed weight scales: uint32 [K/64][N]; word (s, n) carries the four group
  scales of column n that one K=64 step uses, byte g (bits 8g .. 8g+7) =
  wscales[4s + g][n].
- LU': 16-bit [N][R]; LU'[n, r] = round16(fp32(LU[n, r]) * rcp32(wc[n])) where
  rcp32 is the correctly rounded fp32 reciprocal, the product is one fp32
  rounding and round16 is round-to-nearest-even into the I/O type (bf16, or
  IEEE fp16 for the fp16 variant).  A zero wcscale gives LU' = 0 (the
  operator's output is wc * (...) there, so the LoRA term cannot be carried;
  the reading requires wc != 0).  No wcscale (None) means wc = 1: LU' = LU.
"""

from __future__ import annotations

import numpy as np

from .svdq_ref import _np_bytes


def pack_scales(scales, rows: int, K: int) -> np.ndarray:
    """Any scale tensor [K/16][rows] (activations or weights) as uint32
    [K/64][rows]: word (s, r) byte g = scales[4s + g][r]."""
    if K % 64:
        raise ValueError("K must be a multiple of 64")
    w = _np_bytes(scales, np.uint8).reshape(K // 16, rows).astype(np.uint32)
    out = np.zeros((K // 64, rows), dtype=np.uint32)
    for g in range(4):
        out |= w[g::4, :] << np.uint32(8 * g)
    return out


def prepack_wscales(wscales, N: int, K: int) -> np.ndarray:
    """uint32 [K/64][N]: word (s, n) byte g = wscales[4s + g][n]."""
    return pack_scales(wscales, N, K)


def _decode16(bits: np.ndarray, half: bool) -> np.ndarray:
    """Exact fp32 values of bf16 (upper half of an fp32) or IEEE fp16 bits."""
    bits = np.asarray(bits, dtype=np.uint16)
    if half:
        return bits.view(np.float16).astype(np.float32)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _round16(x: np.ndarray, half: bool) -> np.ndarray:
    """fp32 -> 16-bit bits, round to nearest, ties to even (finite inputs)."""
    x = np.asarray(x, dtype=np.float32)
    if half:
        return x.astype(np.float16).view(np.uint16)
    b = x.view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def prepack_lora_up(lora_up, wcscale, N: int, R: int, half: bool = False) -> np.ndarray:
    """16-bit bits [N][R] of LU' = round16(fp32(LU) * rcp32(wc))."""
    lu = _decode16(_np_bytes(lora_up, np.uint16).reshape(N, R), half)
    if wcscale is None:
        return _round16(lu, half)
    wc = _decode16(_np_bytes(wcscale, np.uint16).reshape(N), half)
    with np.errstate(divide="ignore"):
        inv = np.where(wc != 0, np.float32(1.0) / np.where(wc != 0, wc, np.float32(1.0)),
                       np.float32(0.0)).astype(np.float32)
    prod = (lu * inv[:, None]).astype(np.float32)
    return _round16(prod, half)
