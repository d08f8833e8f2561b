"""Pins for the oracle's weight-side prepack (no GPU).

The packed scale words are pinned by a hand-worked example and by reading
them back as bytes through numpy's own reshape/transpose; LU' is pinned by
exact rational arithmetic with a rounding routine written here from the
definition of the binary formats, by library fp32 arithmetic and conversion,
and by the cases where it is exact (wcscale a power of two, or absent).
"""

import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from nvfp4_w4a4_quantized_gb300 import synth


def test_packed_words_worked_example():
    # K = 64 (four groups), N = 2; scale byte of group g, column n = 10 g + n
    ws = np.array([[10 * g + n for n in range(2)] for g in range(4)], dtype=np.uint8)
    pk = oracle.prepack_wscales(ws, N=2, K=64)
    # column 0 holds bytes 0, 10, 20, 30 (group 0 lowest); column 1 bytes 1, 11, 21, 31
    assert pk.shape == (1, 2) and pk.dtype == np.uint32
    assert int(pk[0, 0]) == 0x1E140A00
    assert int(pk[0, 1]) == 0x1F150B01


@pytest.mark.parametrize("N,K", [(16, 64), (48, 320), (272, 3072)])
def test_packed_words_are_group_scales_read_back_as_bytes(N, K):
    rng = np.random.default_rng(N + K)
    ws = rng.integers(0, 256, size=(K // 16, N), dtype=np.uint8)
    pk = oracle.prepack_wscales(ws, N=N, K=K)
    assert pk.shape == (K // 64, N)
    by = pk.astype("<u4").view(np.uint8).reshape(K // 64, N, 4)  # [step][n][byte]
    back = np.transpose(by, (0, 2, 1)).reshape(K // 16, N)       # [step*4 + byte][n]
    assert np.array_equal(back, ws)


def test_packed_words_reject_ragged_k():
    with pytest.raises(ValueError):
        oracle.prepack_wscales(np.zeros((2, 16), np.uint8), N=16, K=32)


# --------------------------------------------------------------------------
# exact rounding into a binary format, from its definition

def _round_fraction(x: Fraction, p: int, emin: int) -> Fraction:
    """Nearest value with a p-bit significand (exponent >= emin; below it the
    quantum stays 2^(emin-p+1)), ties to the even significand."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, emin)
    quantum = Fraction(2) ** (e - p + 1)
    n = a / quantum
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * fl * quantum


def _fmt(half):
    return (11, -14) if half else (8, -126)


def _bits_value(bits: int, half: bool) -> Fraction:
    return Fraction(oracle.f16_value(bits) if half else oracle.bf16_value(bits))


def _edge_inputs(N, R, half, seed):
    inp = synth.make_inputs(16, N, 64, R, seed=seed, half=half)
    lu, wc = inp["lora_up"].clone(), inp["wcscale"].clone()
    dt = torch.float16 if half else torch.bfloat16
    tiny = 2.0 ** -20 if half else 2.0 ** -130  # subnormal in the 16-bit type
    lu[0, 0] = tiny
    lu[0, 1] = -3 * tiny
    lu[1, :] = torch.tensor([0.0, -0.0, 1.0, -1.0] * (R // 4), dtype=dt)[:R]
    wc[0] = 3.0
    wc[1] = 0.75
    wc[2] = 1e-3
    wc[3] = 7.0
    return lu, wc


@pytest.mark.parametrize("half", [False, True])
def test_lu_prime_exact_rationals(half):
    N, R = 24, 16
    lu, wc = _edge_inputs(N, R, half, seed=5)
    got = oracle.prepack_lora_up(lu, wc, N, R, half=half)
    p, emin = _fmt(half)
    lub = lu.view(torch.int16).numpy().view(np.uint16)
    wcb = wc.view(torch.int16).numpy().view(np.uint16)
    for n in range(N):
        w = _bits_value(int(wcb[n]), half)
        inv = _round_fraction(1 / w, 24, -126)
        for r in range(R):
            x = _bits_value(int(lub[n, r]), half)
            want = _round_fraction(_round_fraction(x * inv, 24, -126), p, emin)
            have = _bits_value(int(got[n, r]), half)
            assert have == want, (n, r, float(have), float(want))


@pytest.mark.parametrize("half", [False, True])
def test_lu_prime_matches_library_fp32(half):
    N, R = 300, 32
    inp = synth.make_inputs(16, N, 64, R, seed=9, half=half)
    lu, wc = inp["lora_up"], inp["wcscale"]
    dt = torch.float16 if half else torch.bfloat16
    lib = (lu.float() * torch.reciprocal(wc.float())[:, None]).to(dt)
    got = oracle.prepack_lora_up(lu, wc, N, R, half=half)
    assert np.array_equal(got, lib.view(torch.int16).numpy().view(np.uint16))


def test_lu_prime_power_of_two_is_exact_and_none_is_identity():
    N, R = 32, 16
    inp = synth.make_inputs(16, N, 64, R, seed=3)
    lu = inp["lora_up"]
    e = torch.arange(N) % 5 - 2  # wc = 2^-2 .. 2^2
    wc = torch.pow(2.0, e.float()).to(torch.bfloat16)
    got = oracle.prepack_lora_up(lu, wc, N, R)
    want = (lu.double() * torch.pow(2.0, -e.double())[:, None])
    vals = torch.from_numpy(got.view(np.int16)).view(torch.bfloat16).double()
    assert torch.equal(vals, want)
    ident = oracle.prepack_lora_up(lu, None, N, R)
    assert np.array_equal(ident, lu.view(torch.int16).numpy().view(np.uint16))


def test_lu_prime_zero_wcscale_gives_zero():
    N, R = 16, 8
    inp = synth.make_inputs(16, N, 64, R, seed=4)
    wc = inp["wcscale"].clone()
    wc[5] = 0.0
    got = oracle.prepack_lora_up(inp["lora_up"], wc, N, R)
    assert not (got[5] & 0x7FFF).any()  # +0 or -0 (the sign of LU times zero)
    assert got[4].any()
    assert math.isfinite(oracle.bf16_value(int(got[4, 0])))


@pytest.mark.parametrize("rows,K", [(16, 64), (272, 1088), (4096, 3072)])
def test_packed_activation_scales_read_back_as_bytes(rows, K):
    # the same word layout for activation scales [K/16][M]
    rng = np.random.default_rng(rows + K + 1)
    sc = rng.integers(0, 256, size=(K // 16, rows), dtype=np.uint8)
    pk = oracle.pack_scales(sc, rows, K)
    by = pk.astype("<u4").view(np.uint8).reshape(K // 64, rows, 4)
    assert np.array_equal(np.transpose(by, (0, 2, 1)).reshape(K // 16, rows), sc)
