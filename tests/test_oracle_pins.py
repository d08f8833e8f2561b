"""Pins for the CPU oracle (no GPU).

Each test ties the oracle to something other than itself: the published
value tables of the element formats, a library FP8 conversion, a hand-worked
example, exact rational brute force on tiny shapes, dequantize-then-matmul
through a library matmul, closed forms and invariants.  Together they are
chosen so that a dropped term, a wrong sign, a wrong nibble/scale index or a
transposed operand in the oracle fails at least one of them.
"""

import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from nvfp4_w4a4_quantized_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                rows.append(line.split())
    return rows


# --------------------------------------------------------------------------
# independent decoders used only by the pins (not the oracle's code)

def e2m1_bits_fraction(code: int) -> Fraction:
    """E2M1 from its bit fields: 1 sign, 2 exponent (bias 1), 1 mantissa."""
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    v = Fraction(m, 2) if e == 0 else Fraction(2) ** (e - 1) * (1 + Fraction(m, 2))
    return -v if s else v


def e4m3_library(byte_arr: np.ndarray) -> np.ndarray:
    """FP8-E4M3 through torch's float8_e4m3fn conversion (a library routine)."""
    t = torch.from_numpy(np.ascontiguousarray(byte_arr, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def bf16_library(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


def nibbles(packed: np.ndarray) -> np.ndarray:
    """[rows, K/2] bytes -> [rows, K] codes, element k in the low nibble of
    byte k/2 for even k (the packed-FP4 reading the kernel hardware uses)."""
    lo = packed & 0xF
    hi = packed >> 4
    out = np.empty((packed.shape[0], packed.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = lo
    out[:, 1::2] = hi
    return out


E2M1_GOLDEN = {int(c): float(v) for c, v in _read_table("e2m1_values.txt")}


def dequant(packed, scales):
    """Dense fp64 dequantised matrix [rows, K] from packed codes and [K/16, rows] scales."""
    codes = nibbles(packed.numpy())
    vals = np.vectorize(lambda c: E2M1_GOLDEN[int(c)])(codes).astype(np.float64)
    sc = e4m3_library(scales.numpy())          # [K/16, rows]
    return vals * np.repeat(sc.T, 16, axis=1)


# --------------------------------------------------------------------------
# element formats

def test_e2m1_table_matches_published_values():
    for code, v in E2M1_GOLDEN.items():
        got = oracle.e2m1(code)
        assert got == v and math.copysign(1, got) == math.copysign(1, v), code


def test_e2m1_table_matches_bit_fields():
    for code in range(16):
        assert Fraction(oracle.e2m1(code)) == e2m1_bits_fraction(code)


def test_e4m3_exhaustive_against_library():
    lib = e4m3_library(np.arange(256, dtype=np.uint8))
    for b in range(256):
        got = oracle.e4m3(b)
        if math.isnan(lib[b]):
            assert math.isnan(got), hex(b)
        else:
            assert got == lib[b], hex(b)


def test_e4m3_published_points():
    for b, v in _read_table("e4m3_points.txt"):
        got = oracle.e4m3(int(b, 16))
        if v == "nan":
            assert math.isnan(got)
        else:
            assert got == float(v), b


def test_bf16_decode_and_round_against_library():
    g = torch.Generator().manual_seed(7)
    x = torch.randn(20000, generator=g, dtype=torch.float32) * torch.exp(
        torch.randn(20000, generator=g) * 20)
    x = torch.cat([x, torch.tensor([0.0, -0.0, 1.0, 3.0e38, -3.4e38, 1e-40, 1.5, 1.00390625,
                                    1.01171875, 9.2e-41, float("inf")])])
    want = x.to(torch.bfloat16)
    bits = want.view(torch.int16).numpy().astype(np.uint16)
    for xi, wi, bi in zip(x.tolist(), want.to(torch.float64).tolist(), bits.tolist()):
        assert oracle.round_bf16_bits(xi) == bi, (xi, hex(bi))
        assert oracle.bf16_value(bi) == wi


# --------------------------------------------------------------------------
# the operator

def _golden_example():
    rows = {r[0]: r[1:] for r in _read_table("worked_example.txt")}
    M, N, K, R = (int(rows[k][0]) for k in "MNKR")
    hexbytes = lambda name: np.frombuffer(bytes.fromhex("".join(rows[name])), dtype=np.uint8)
    hexu16 = lambda name: np.array([int(h, 16) for h in rows[name]], dtype=np.uint16)
    inp = dict(act=hexbytes("act").reshape(M, K // 2), wgt=hexbytes("wgt").reshape(N, K // 2),
               ascales=hexbytes("ascales").reshape(K // 16, M),
               wscales=hexbytes("wscales").reshape(K // 16, N),
               lora_act_in=np.array([float(v) for v in rows["lora_act_in"]], np.float32).reshape(M, R),
               lora_up=hexu16("lora_up").reshape(N, R), wcscale=hexu16("wcscale"), bias=hexu16("bias"))
    main = np.array([float(v) for v in rows["main"]]).reshape(M, N)
    y = np.array([float(v) for v in rows["y"]]).reshape(M, N)
    return inp, (M, N, K, R), main, y


def test_hand_worked_example():
    inp, (M, N, K, R), main_want, y_want = _golden_example()
    y, main = oracle.forward(inp, M, N, K, R, want_main=True)
    assert np.array_equal(main, main_want)
    assert np.array_equal(y, y_want)


def _bruteforce(inp, M, N, K, R):
    """Exact rational evaluation of the operator definition."""
    codes_a = nibbles(inp["act"].numpy())
    codes_w = nibbles(inp["wgt"].numpy())
    sa = e4m3_library(inp["ascales"].numpy())
    sw = e4m3_library(inp["wscales"].numpy())
    la = inp["lora_act_in"].numpy().astype(np.float64)
    lu = bf16_library(inp["lora_up"])
    wc = bf16_library(inp["wcscale"])
    bi = bf16_library(inp["bias"])
    y = [[None] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for g in range(K // 16):
                s = sum(e2m1_bits_fraction(int(codes_a[m, k])) * e2m1_bits_fraction(int(codes_w[n, k]))
                        for k in range(16 * g, 16 * g + 16))
                acc += Fraction(sa[g, m]) * Fraction(sw[g, n]) * s
            lora = sum((Fraction(la[m, r]) * Fraction(lu[n, r]) for r in range(R)), Fraction(0))
            y[m][n] = Fraction(wc[n]) * acc + Fraction(bi[n]) + lora
    return y


@pytest.mark.parametrize("M,N,K,R,seed", [
    (1, 1, 16, 0, 11), (3, 2, 32, 0, 12), (5, 4, 64, 0, 13), (2, 5, 48, 1, 14),
    (4, 3, 32, 2, 15), (5, 5, 64, 16, 16), (3, 4, 16, 3, 17)])
def test_exact_bruteforce_tiny(M, N, K, R, seed):
    inp = synth.make_inputs(M, N, K, R, seed)
    y = oracle.forward(inp, M, N, K, R)
    exact = _bruteforce(inp, M, N, K, R)
    la = inp["lora_act_in"].numpy().astype(np.float64)
    lu = bf16_library(inp["lora_up"])
    for m in range(M):
        for n in range(N):
            if R == 0:
                assert Fraction(y[m, n]) == exact[m][n]
            else:
                mag = float(np.abs(la[m] * lu[n]).sum()) + abs(float(exact[m][n]))
                assert abs(Fraction(y[m, n]) - exact[m][n]) <= Fraction(2) ** -50 * Fraction(mag)


@pytest.mark.parametrize("M,N,K,seed", [(37, 29, 256, 21), (16, 48, 512, 22), (64, 8, 3072, 23)])
def test_main_equals_dequantize_then_matmul(M, N, K, seed):
    inp = synth.make_inputs(M, N, K, 0, seed)
    _, main = oracle.forward(inp, M, N, K, 0, want_main=True)
    a = dequant(inp["act"], inp["ascales"])
    w = dequant(inp["wgt"], inp["wscales"])
    # every product and partial sum is a dyadic rational needing < 53 bits,
    # so the library matmul is exact whatever its summation order
    assert np.array_equal(main, a @ w.T)


def test_affine_and_lora_terms():
    M, N, K, R = 9, 13, 64, 16
    inp = synth.make_inputs(M, N, K, R, 31)
    y = oracle.forward(inp, M, N, K, R)
    _, main = oracle.forward(inp, M, N, K, R, want_main=True)
    la = inp["lora_act_in"].numpy().astype(np.float64)
    lu = bf16_library(inp["lora_up"])
    wc = bf16_library(inp["wcscale"])
    bi = bf16_library(inp["bias"])
    want = wc[None, :] * main + bi[None, :] + la @ lu.T
    assert np.allclose(y, want, rtol=1e-13, atol=1e-13)
    # LoRA is not multiplied by wcscale: dropping the affine leaves main + lora
    bare = dict(inp, wcscale=None, bias=None)
    y0 = oracle.forward(bare, M, N, K, R)
    assert np.allclose(y0, main + la @ lu.T, rtol=1e-13, atol=1e-13)
    # R = 0 removes exactly the LoRA term
    y_nolora = oracle.forward(inp, M, N, K, 0)
    assert np.allclose(y - y_nolora, la @ lu.T, rtol=1e-12, atol=1e-12)


def test_closed_form_all_ones():
    M, N, K = 6, 10, 128
    inp = synth.make_inputs(M, N, K, 0, 41)
    inp["act"][:] = 0x22          # every element code 2 = 1.0
    inp["wgt"][:] = 0x22
    inp["ascales"][:] = 0x38      # every scale 1.0
    inp["wscales"][:] = 0x38
    y, main = oracle.forward(inp, M, N, K, 0, want_main=True)
    assert np.all(main == K)
    wc = bf16_library(inp["wcscale"])
    bi = bf16_library(inp["bias"])
    assert np.array_equal(y, np.broadcast_to(wc * K + bi, (M, N)))


@pytest.mark.parametrize("k0", [0, 1, 15, 16, 17, 63, 64, 255])
def test_one_hot(k0):
    M, N, K = 5, 7, 256
    inp = synth.make_inputs(M, N, K, 0, 50 + k0)
    m0 = 3
    w = dequant(inp["wgt"], inp["wscales"])
    wc = bf16_library(inp["wcscale"])
    bi = bf16_library(inp["bias"])
    sa = e4m3_library(inp["ascales"].numpy())
    for code in range(16):
        inp["act"][:] = 0
        inp["act"][m0, k0 // 2] = code << (4 * (k0 & 1))
        y = oracle.forward(inp, M, N, K, 0)
        want = np.broadcast_to(bi, (M, N)).copy()
        want[m0] = E2M1_GOLDEN[code] * sa[k0 // 16, m0] * w[:, k0] * wc + bi
        assert np.array_equal(y, want), (k0, code)


def test_identity():
    M = N = K = 64
    inp = synth.make_inputs(M, N, K, 0, 61)
    inp["act"][:] = 0
    for m in range(M):
        inp["act"][m, m // 2] = 2 << (4 * (m & 1))   # a(m, m) = 1.0
    inp["ascales"][:] = 0x38
    y = oracle.forward(inp, M, N, K, 0)
    w = dequant(inp["wgt"], inp["wscales"])
    wc = bf16_library(inp["wcscale"])
    bi = bf16_library(inp["bias"])
    assert np.array_equal(y, w.T * wc[None, :] + bi[None, :])


def test_operand_swap_symmetry():
    M, N, K = 11, 6, 96
    inp = synth.make_inputs(M, N, K, 0, 71)
    _, main = oracle.forward(inp, M, N, K, 0, want_main=True)
    sw = dict(act=inp["wgt"], wgt=inp["act"], ascales=inp["wscales"], wscales=inp["ascales"])
    _, main_t = oracle.forward(sw, N, M, K, 0, want_main=True)
    assert np.array_equal(main, main_t.T)


def test_scale_exponent_linearity():
    M, N, K = 7, 9, 160
    inp = synth.make_inputs(M, N, K, 0, 81)
    _, main = oracle.forward(inp, M, N, K, 0, want_main=True)
    up = dict(inp, ascales=inp["ascales"] + 8)     # exponent field + 1: every scale x2
    _, main2 = oracle.forward(up, M, N, K, 0, want_main=True)
    assert np.array_equal(main2, 2 * main)
    # changing a single group's scale changes only that group's contribution
    g0 = 3
    one = inp["ascales"].clone()
    one[g0] += 8
    _, main3 = oracle.forward(dict(inp, ascales=one), M, N, K, 0, want_main=True)
    a = dequant(inp["act"], inp["ascales"])
    w = dequant(inp["wgt"], inp["wscales"])
    grp = a[:, 16 * g0:16 * g0 + 16] @ w[:, 16 * g0:16 * g0 + 16].T
    assert np.array_equal(main3 - main, grp)


def test_row_subset_matches_full():
    M, N, K, R = 20, 12, 64, 8
    inp = synth.make_inputs(M, N, K, R, 91)
    y = oracle.forward(inp, M, N, K, R)
    rows = [19, 0, 7, 7, 3]
    ys = oracle.forward(inp, M, N, K, R, rows=rows)
    assert np.array_equal(ys, y[rows])


def test_rejects_bad_arguments():
    inp = synth.make_inputs(4, 4, 32, 0, 1)
    with pytest.raises(ValueError):
        oracle.forward(inp, 4, 4, 32, 0, rows=[4])


def test_nibble_order_invariance():
    """Swapping the two nibbles of every byte of BOTH operands permutes the
    products inside each 16-element scale group, so y is unchanged: the
    within-byte order is a convention act and wgt must merely share."""
    M, N, K, R = 9, 7, 128, 4
    inp = synth.make_inputs(M, N, K, R, 101)
    y = oracle.forward(inp, M, N, K, R)
    swap = lambda t: ((t & 0xF) << 4) | (t >> 4)
    y2 = oracle.forward(dict(inp, act=swap(inp["act"]), wgt=swap(inp["wgt"])), M, N, K, R)
    assert np.array_equal(y, y2)
    # swapping only one operand does change it
    y3 = oracle.forward(dict(inp, act=swap(inp["act"])), M, N, K, R)
    assert not np.array_equal(y, y3)


# --------------------------------------------------------------------------
# the fp16 input/output variant (lora_up, wcscale, bias in IEEE binary16)

def test_f16_decode_exhaustive_against_library():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    lib = torch.from_numpy(bits.view(np.int16)).view(torch.float16).to(torch.float64).numpy()
    for b in range(0, 65536):
        got = oracle.f16_value(b)
        if math.isnan(lib[b]):
            assert math.isnan(got), hex(b)
        else:
            assert got == lib[b] and math.copysign(1, got) == math.copysign(1, lib[b]), hex(b)


@pytest.mark.parametrize("M,N,K,R,seed", [(3, 2, 32, 0, 41), (2, 5, 48, 1, 42), (5, 4, 64, 16, 43)])
def test_exact_bruteforce_tiny_half(M, N, K, R, seed):
    inp = synth.make_inputs(M, N, K, R, seed, half=True)
    y = oracle.forward(inp, M, N, K, R)
    # the rational brute force reads the fp16 values through the library
    as_frac = lambda t: [Fraction(v) for v in t.to(torch.float64).flatten().tolist()]
    a = nibbles(inp["act"].numpy())
    w = nibbles(inp["wgt"].numpy())
    sa = e4m3_library(inp["ascales"].numpy())
    sw = e4m3_library(inp["wscales"].numpy())
    wc, bi = as_frac(inp["wcscale"]), as_frac(inp["bias"])
    lu = as_frac(inp["lora_up"])
    la = inp["lora_act_in"].numpy().astype(np.float64)
    for m in range(M):
        for n in range(N):
            main = Fraction(0)
            for g in range(K // 16):
                s = sum(e2m1_bits_fraction(int(a[m, k])) * e2m1_bits_fraction(int(w[n, k]))
                        for k in range(16 * g, 16 * g + 16))
                main += Fraction(float(sa[g, m])) * Fraction(float(sw[g, n])) * s
            lora = sum(Fraction(float(la[m, r])) * lu[n * R + r] for r in range(R))
            exact = wc[n] * main + bi[n] + lora
            mag = abs(exact) + sum(abs(Fraction(float(la[m, r])) * lu[n * R + r]) for r in range(R))
            assert abs(Fraction(y[m, n]) - exact) <= Fraction(2) ** -50 * (mag + 1), (m, n)


def test_half_and_bf16_agree_on_shared_values():
    # values exactly representable in both formats give the same y
    M, N, K, R = 7, 9, 64, 16
    inp = synth.make_inputs(M, N, K, R, 44)
    g = torch.Generator().manual_seed(45)
    shared = lambda shape: (torch.randint(-64, 64, shape, generator=g).to(torch.float32) / 64.0)
    lu, wc, bi = shared((N, R)), shared((N,)) + 2.0, shared((N,))
    y_b = oracle.forward(dict(inp, lora_up=lu.to(torch.bfloat16), wcscale=wc.to(torch.bfloat16),
                              bias=bi.to(torch.bfloat16)), M, N, K, R)
    y_h = oracle.forward(dict(inp, lora_up=lu.to(torch.float16), wcscale=wc.to(torch.float16),
                              bias=bi.to(torch.float16)), M, N, K, R)
    assert np.array_equal(y_b, y_h)
    # and different fp16 values do change it (the dtype switch is live)
    y_h2 = oracle.forward(dict(inp, lora_up=(lu * 1.0009765625).to(torch.float16),
                               wcscale=wc.to(torch.float16), bias=bi.to(torch.float16)),
                          M, N, K, R)
    assert not np.array_equal(y_h, y_h2)
