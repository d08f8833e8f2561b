"""Pins of the activation-quantiser oracle (oracle/quant_ref.py) against
things other than itself: a hand-worked example, the format definitions'
closed forms, torch's own float8 conversion and exact rational arithmetic.

The quantiser reading: per 16-group, s = E4M3(amax / 6), code = E2M1(x / s),
both nearest-even and saturating ("SVDQuant W4A4 on Blackwell" §1-§3.1 name
the producer and its output formats; OCP Microscaling Formats v1.0 §5.3 the
element encodings).
"""

import os
from fractions import Fraction

import numpy as np
import torch

from oracle import quant_ref as q

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "quant_example.txt")


def _bits(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.bfloat16)


def _codes(act: np.ndarray) -> np.ndarray:
    M, H = act.shape
    c = np.zeros((M, 2 * H), np.uint8)
    c[:, 0::2] = act & 15
    c[:, 1::2] = act >> 4
    return c


def _value(code: np.ndarray) -> np.ndarray:
    v = q.E2M1_VALUES[code & 7]
    return np.where(code & 8, -v, v)


def test_golden_worked_example():
    rows, want_s, want_c = {}, {}, {}
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        head, xs, sb, cs = line.split("|")
        r, g = map(int, head.split())
        rows[(r, g)] = [float(v) for v in xs.split()]
        want_s[(r, g)] = int(sb, 16)
        want_c[(r, g)] = [int(c, 16) for c in cs.split()]
    M, G = 2, 4
    x = torch.tensor([sum((rows[(r, g)] for g in range(G)), []) for r in range(M)])
    xb = _bits(x)
    assert torch.equal(xb.float(), x)
    act, asc = q.quantize_act(xb, M, 16 * G)
    codes = _codes(act)
    for (r, g), s in want_s.items():
        assert asc[g, r] == s, (r, g)
        assert list(codes[r, 16 * g:16 * g + 16]) == want_c[(r, g)], (r, g)


def test_e4m3_table_round_trip_and_ties():
    t = q.e4m3_values()
    assert t[0x38] == 1.0 and t[0x7E] == 448.0 and t[0x01] == 2.0 ** -9
    assert np.all(np.diff(t) > 0)
    assert np.array_equal(q.round_e4m3(t), np.arange(0x7F, dtype=np.uint8))
    mid = (t[:-1] + t[1:]) / 2
    want = np.arange(0x7E)
    want = np.where(want % 2 == 0, want, want + 1)  # the even one of b, b + 1
    assert np.array_equal(q.round_e4m3(mid), want.astype(np.uint8))
    # just off the ties: the nearer neighbour
    eps = np.diff(t) * 1e-6
    assert np.array_equal(q.round_e4m3(mid - eps), np.arange(0x7E, dtype=np.uint8))
    assert np.array_equal(q.round_e4m3(mid + eps), np.arange(1, 0x7F, dtype=np.uint8))
    # saturation and flush
    assert np.all(q.round_e4m3([448.0, 463.9, 464.0, 500.0, 1e30]) == 0x7E)
    assert np.all(q.round_e4m3([0.0, 2.0 ** -11, 2.0 ** -10]) == 0)


def test_e4m3_rounding_matches_torch_float8():
    g = torch.Generator().manual_seed(5)
    v = torch.cat([torch.rand(20000, generator=g) * 448,
                   torch.rand(20000, generator=g) * 2.0 ** -5,
                   torch.exp2(torch.rand(20000, generator=g) * 17 - 10)]).clamp(max=448)
    want = v.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q.round_e4m3(v.double().numpy()), want)


def test_e2m1_rounding_closed_forms():
    vals = q.E2M1_VALUES
    assert np.array_equal(q.round_e2m1(vals), np.arange(8, dtype=np.uint8))
    assert np.array_equal(q.round_e2m1(-vals[1:]), np.arange(9, 16, dtype=np.uint8))
    ties = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    assert list(q.round_e2m1(ties)) == [0, 2, 2, 4, 4, 6, 6]
    assert list(q.round_e2m1([-t for t in ties])) == [0, 10, 10, 12, 12, 14, 14]
    assert list(q.round_e2m1([6.0, 7.0, 1e9, -1e9, -0.0, -1e-30])) == [7, 7, 7, 15, 0, 0]


def test_e2m1_rounding_against_exact_rationals():
    rng = np.random.default_rng(6)
    qs = np.concatenate([rng.uniform(-7, 7, 3000), rng.integers(-28, 29, 500) / 4.0])
    exact = [Fraction(v).limit_denominator(1 << 40) for v in qs]
    grid = [Fraction(v) for v in (0, 0.5, 1, 1.5, 2, 3, 4, 6)]
    got = q.round_e2m1(qs)
    for v, e, c in zip(qs, exact, got):
        a = abs(e)
        d = [abs(a - gv) for gv in grid]
        best = min(d)
        cands = [i for i, di in enumerate(d) if di == best]
        mag = cands[0] if len(cands) == 1 else [i for i in cands if i % 2 == 0][0]
        want = mag | (8 if (e < 0 and mag > 0) else 0)
        assert c == want, (v, c, want)


def test_representable_groups_come_back_exactly():
    # x = code value * s with amax = 6 s: quantising returns s's byte and the codes
    rng = np.random.default_rng(7)
    t = q.e4m3_values()
    M, K = 8, 256
    x = np.zeros((M, K))
    want_codes = rng.integers(0, 16, size=(M, K)).astype(np.uint8)
    want_s = rng.integers(0x20, 0x58, size=(M, K // 16)).astype(np.uint8)
    for m in range(M):
        for g in range(K // 16):
            cg = want_codes[m, 16 * g:16 * g + 16]
            cg[0] = 7  # one element at +6 fixes amax = 6 s
            x[m, 16 * g:16 * g + 16] = _value(cg) * t[want_s[m, g]]
    want_codes = np.where((want_codes & 7) == 0, 0, want_codes).astype(np.uint8)  # +0
    xb = torch.tensor(x, dtype=torch.float32).to(torch.bfloat16)
    assert np.array_equal(xb.double().numpy(), x)
    act, asc = q.quantize_act(xb, M, K)
    assert np.array_equal(asc.T, want_s)
    assert np.array_equal(_codes(act), want_codes)


def test_power_of_two_scaling_and_sign_symmetry():
    g = torch.Generator().manual_seed(8)
    M, K = 16, 512
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    act, asc = q.quantize_act(x, M, K)
    act2, asc2 = q.quantize_act((x.float() * 4).to(torch.bfloat16), M, K)
    assert np.array_equal(act2, act)
    assert np.array_equal(asc2.astype(int), asc.astype(int) + 16)  # exponent field + 2
    actn, ascn = q.quantize_act(-x, M, K)
    assert np.array_equal(ascn, asc)
    c, cn = _codes(act), _codes(actn)
    assert np.array_equal(cn, np.where((c & 7) == 0, 0, c ^ 8))


def test_dequantised_error_bound():
    # |x - value(code) s| is at most half the E2M1 gap at x / s, or the
    # saturation distance above 6; a normal s is within 1/16 (relative) of
    # amax / 6, so no |x| / s exceeds 6 / (1 - 1/16)
    g = torch.Generator().manual_seed(9)
    M, K = 32, 1024
    x = (torch.randn(M, K, generator=g) * torch.exp2(torch.randint(-8, 8, (M, 1), generator=g))
         ).to(torch.bfloat16)
    act, asc = q.quantize_act(x, M, K)
    s = q.e4m3_values()[asc.T].repeat(16, axis=1)
    X = x.double().numpy()
    deq = _value(_codes(act)) * s
    r = np.abs(X) / s
    half_gap = np.where(r < 2, 0.25, np.where(r < 4, 0.5, 1.0))
    bound = np.where(r <= 6, half_gap * s, np.abs(X) - 6 * s)
    assert np.all(np.abs(X - deq) <= bound * (1 + 1e-12))
    normal = s >= 2.0 ** -6
    assert np.all(r[normal] <= 6 * 16 / 15 + 1e-12)


def test_packed_scales_are_the_pack_of_the_raw_ones():
    g = torch.Generator().manual_seed(10)
    M, K = 48, 384
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    act, asc = q.quantize_act(x, M, K)
    act_p, words = q.quantize_act(x, M, K, packed=True)
    assert np.array_equal(act_p, act)
    assert words.dtype == np.uint32 and words.shape == (K // 64, M)
    for s in range(K // 64):
        for gg in range(4):
            assert np.array_equal((words[s] >> np.uint32(8 * gg)) & np.uint32(255), asc[4 * s + gg])


def test_fp16_input_matches_bf16_where_values_agree():
    # values exact in both formats quantise identically
    g = torch.Generator().manual_seed(11)
    M, K = 16, 256
    x = (torch.randint(-64, 65, (M, K), generator=g).float() / 8)
    a1, s1 = q.quantize_act(x.to(torch.bfloat16), M, K)
    a2, s2 = q.quantize_act(x.to(torch.float16), M, K, half=True)
    assert np.array_equal(a1, a2) and np.array_equal(s1, s2)


def test_lora_down_brute_force_and_identity():
    g = torch.Generator().manual_seed(12)
    M, K, R = 3, 64, 5
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    ld = (torch.randn(R, K, generator=g) * 0.1).to(torch.bfloat16)
    got = q.lora_down(x, ld, M, K, R)
    xf = [[Fraction(float(v)) for v in row] for row in x.float().tolist()]
    lf = [[Fraction(float(v)) for v in row] for row in ld.float().tolist()]
    for m in range(M):
        for r in range(R):
            exact = sum(a * b for a, b in zip(xf[m], lf[r]))
            assert abs(got[m, r] - float(exact)) <= 1e-14 * max(1.0, abs(float(exact)))
    eye = torch.eye(64).to(torch.bfloat16)
    x2 = torch.randn(7, 64, generator=g).to(torch.bfloat16)
    assert np.array_equal(q.lora_down(x2, eye, 7, 64, 64), x2.double().numpy())
