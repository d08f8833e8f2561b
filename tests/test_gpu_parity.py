"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Bar (the operator's acceptance tolerance, bf16 output with fp32
accumulation): |y_gpu - y_ref| <= 2^-7 |y_ref| + 1e-3 rms(y_ref) per element.
Structural cases (LoRA-only, affine, one-hot, identity, closed form) use
bounds derived for them because at the workload distributions the LoRA and
bias terms sit far below the acceptance tolerance.
"""

import numpy as np
import pytest
import torch

from gpu_util import oracle_y, parity, run_gpu, sample_rows
from nvfp4_w4a4_quantized_gb300 import synth

pytestmark = pytest.mark.gpu

# every kernel instantiation: single CTA with 128- or 256-wide tiles, and a
# CTA pair issuing 256-row MMAs on 256 x 256 tiles
CONFIGS = [dict(cta_group=1, tile_n=128), dict(cta_group=1, tile_n=256),
           dict(cta_group=2, tile_n=256)]
CFG_IDS = ["cg1_n128", "cg1_n256", "cg2_n256"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from nvfp4_w4a4_quantized_gb300 import build
    build.build()
    import oracle
    oracle.build()


def full_check(M, N, K, R, seed, options=None, inp=None):
    inp = inp if inp is not None else synth.make_inputs(M, N, K, R, seed)
    y = run_gpu(inp, M, N, K, R, options=options)
    ref = oracle_y(inp, M, N, K, R)
    return parity(y, ref)


@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_tiny_workload_full_matrix(cfg):
    w = synth.TINY
    full_check(w.M, w.N, w.K, w.R, w.seed, options=cfg)


@pytest.mark.parametrize("M,N,K,R", [
    (272, 144, 320, 20),     # ragged M, N and a partial last K block; R not a multiple of 16
    (16, 16, 64, 1),         # smallest legal shape
    (400, 528, 1088, 100),   # several tiles, ragged everywhere, four 32-rank LoRA items
    (128, 256, 256, 0),      # no LoRA
    (384, 512, 768, 64),     # exact multiples, one full LoRA block
    (256, 272, 512, 128),    # maximum rank
    (144, 400, 192, 3),      # K below one full block, odd rank (scalar LoRA loads)
])
@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_ragged_and_edge_shapes(M, N, K, R, cfg):
    full_check(M, N, K, R, seed=M + N + K + R, options=cfg)


@pytest.mark.parametrize("cfg,max_ctas", [(CONFIGS[0], 1), (CONFIGS[1], 1), (CONFIGS[2], 2),
                                          (CONFIGS[0], 5), (CONFIGS[1], 3), (CONFIGS[2], 6)])
def test_persistent_many_tiles_per_cta(cfg, max_ctas):
    # >= 12 tiles per CTA (pair): pipeline phases must survive tile boundaries
    # and the accumulator must restart at every tile.
    M, N, K, R = 1024, 768, 512, 32
    full_check(M, N, K, R, seed=5, options=dict(cfg, max_ctas=max_ctas))


@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_accumulator_restarts_per_tile(cfg):
    # neighbouring tiles differ in magnitude by 2^8: a leaked accumulator shows
    M, N, K, R = 1024, 512, 512, 16
    inp = synth.make_inputs(M, N, K, R, 6)
    inp["ascales"][:, :256] = 0x58   # 2^4
    inp["ascales"][:, 256:] = 0x18   # 2^-4  (rows of the later M tiles)
    full_check(M, N, K, R, 6, options=dict(cfg, max_ctas=2), inp=inp)


@pytest.mark.parametrize("wc_value", [0.5, 2.0])
@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_lora_only(wc_value, cfg):
    # act codes all zero: y = bias + lora_act_in @ lora_up, and LoRA must not
    # be multiplied by wcscale.  Bound: 2^-7 sum_r |la*lu| (bf16 operands, fp32
    # sums) + 2^-8 |y| (bf16 output) + 1e-6.
    M, N, K, R = 256, 384, 256, 32
    inp = synth.make_inputs(M, N, K, R, 7)
    inp["act"][:] = 0
    inp["wcscale"][:] = wc_value
    y = run_gpu(inp, M, N, K, R, options=cfg)
    ref = oracle_y(inp, M, N, K, R)
    la = inp["lora_act_in"].double().numpy()
    lu = inp["lora_up"].double().numpy()
    mag = np.abs(la) @ np.abs(lu).T
    parity(y, ref, rel=2.0 ** -8, rms_frac=0.0, extra=2.0 ** -7 * mag + 1e-6)


@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_affine_wcscale_and_bias(cfg):
    M, N, K = 256, 256, 512
    inp = synth.make_inputs(M, N, K, 0, 8)
    inp["wcscale"][:] = 2.0
    inp["ascales"][:] = 0x18       # 2^-4: main of order 1, comparable to bias
    inp["wscales"][:] = 0x18
    y = run_gpu(inp, M, N, K, 0, options=cfg)
    ref = oracle_y(inp, M, N, K, 0)
    parity(y, ref, rel=2.0 ** -8, rms_frac=1e-4)


@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
@pytest.mark.parametrize("R", [16, 20])
def test_null_wcscale_and_bias(cfg, R):
    M, N, K = 256, 256, 256
    inp = synth.make_inputs(M, N, K, R, 9)
    inp["wcscale"] = None
    inp["bias"] = None
    full_check(M, N, K, R, 9, inp=inp, options=cfg)


def test_one_hot_rows():
    """One nonzero act element per row at distinct (row quadrant, k) positions:
    y[m, :] = e2m1(c) * ascale * wgt_deq[:, k0] * wcscale + bias, every other
    row = bias.  Pins nibble order, scale-group indexing and the scale layout
    in tensor memory for every lane quadrant and both 128-row halves of B."""
    M, N, K = 256, 256, 1024
    inp = synth.make_inputs(M, N, K, 0, 10)
    inp["act"][:] = 0
    rng = np.random.default_rng(10)
    ks = [0, 1, 14, 15, 16, 17, 63, 64, 65, 127, 128, 255, 256, 257, 511, 512, 767, 1023]
    for m in range(0, M, 3):
        k0 = ks[(m // 3) % len(ks)]
        code = int(rng.integers(1, 16))
        inp["act"][m, k0 // 2] = code << (4 * (k0 & 1))
    for cfg in CONFIGS:
        y = run_gpu(inp, M, N, K, 0, options=cfg)
        ref = oracle_y(inp, M, N, K, 0)
        parity(y, ref, rel=2.0 ** -8, rms_frac=0.0, extra=1e-6)


@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_identity(cfg):
    M = N = K = 256
    inp = synth.make_inputs(M, N, K, 0, 12)
    inp["act"][:] = 0
    for m in range(M):
        inp["act"][m, m // 2] |= 2 << (4 * (m & 1))   # a(m, m) = 1.0
    inp["ascales"][:] = 0x38
    y = run_gpu(inp, M, N, K, 0, options=cfg)
    ref = oracle_y(inp, M, N, K, 0)
    parity(y, ref, rel=2.0 ** -8, rms_frac=0.0, extra=1e-6)


def test_closed_form_all_ones():
    M, N, K = 128, 256, 3072
    inp = synth.make_inputs(M, N, K, 0, 13)
    inp["act"][:] = 0x22
    inp["wgt"][:] = 0x22
    inp["ascales"][:] = 0x38
    inp["wscales"][:] = 0x38
    y = run_gpu(inp, M, N, K, 0)
    wc = inp["wcscale"].double().numpy()
    bi = inp["bias"].double().numpy()
    ref = np.broadcast_to(wc * K + bi, (M, N))
    parity(y, ref, rel=2.0 ** -8, rms_frac=0.0, extra=1e-6)


def test_subnormal_scales():
    # E4M3 subnormal scale bytes (0x01 = 2^-9 .. 0x07) on both sides
    M, N, K, R = 128, 256, 256, 0
    inp = synth.make_inputs(M, N, K, R, 14)
    g = torch.Generator().manual_seed(14)
    inp["ascales"] = torch.randint(1, 8, inp["ascales"].shape, generator=g, dtype=torch.uint8)
    inp["wscales"][::2] = torch.randint(1, 8, inp["wscales"][::2].shape, generator=g,
                                        dtype=torch.uint8)
    full_check(M, N, K, R, 14, inp=inp)


def test_repeatable_and_output_fully_written():
    w = synth.TINY
    inp = synth.make_inputs(w.M, w.N, w.K, w.R, 3)
    y1 = run_gpu(inp, w.M, w.N, w.K, w.R)
    y2 = run_gpu(inp, w.M, w.N, w.K, w.R)
    assert np.array_equal(y1, y2)


# ------------------------------------------------------------ full-size workloads
@pytest.mark.parametrize("cfg", [None] + CONFIGS, ids=["default"] + CFG_IDS)
@pytest.mark.parametrize("w", [synth.ATTN_PROJ, synth.MLP_UP, synth.MLP_DOWN], ids=lambda w: w.name)
def test_workload_sampled_rows(w, cfg):
    inp = synth.make_workload_inputs(w)
    y = run_gpu(inp, w.M, w.N, w.K, w.R, options=cfg)
    rows = sample_rows(w.M, 40, seed=w.seed)
    ref = oracle_y(inp, w.M, w.N, w.K, w.R, rows=rows)
    parity(y[rows], ref)


@pytest.mark.parametrize("w", [synth.ATTN_PROJ, synth.MLP_UP, synth.MLP_DOWN], ids=lambda w: w.name)
def test_workload_full_matrix(w):
    # every element of the full-size workload, in the launch configuration the
    # bench times (the oracle takes 2 to 10 s of host time per workload)
    inp = synth.make_workload_inputs(w)
    y = run_gpu(inp, w.M, w.N, w.K, w.R)
    parity(y, oracle_y(inp, w.M, w.N, w.K, w.R))


def sweep_rows(M):
    """Every 8th row, plus every row of the first and of the last 256-row
    tile row (all lane quadrants and both CTAs of a pair at both ends)."""
    rows = set(range(0, M, 8)) | set(range(0, min(256, M))) | set(range(max(0, M - 256), M))
    return np.array(sorted(rows), dtype=np.int64)


@pytest.mark.parametrize("w", synth.sweep_workloads(), ids=lambda w: w.name)
def test_sweep_rows(w):
    # the full matrix where the oracle is quick (M <= 4096), else every 8th
    # row plus the first and last tile rows
    inp = synth.make_workload_inputs(w)
    y = run_gpu(inp, w.M, w.N, w.K, w.R)
    if w.M <= 4096:
        parity(y, oracle_y(inp, w.M, w.N, w.K, w.R))
    else:
        rows = sweep_rows(w.M)
        parity(y[rows], oracle_y(inp, w.M, w.N, w.K, w.R, rows=rows))


# ------------------------------------------------------------ dense calibration
@pytest.mark.parametrize("cfg", [None] + CONFIGS, ids=["default"] + CFG_IDS)
def test_dense_calibration_full_matrix(cfg):
    """The dense calibration variant of the attention projection: R = 0, no
    wcscale and no bias (1 and 0), through the same kernel -- the block-scaled
    product alone, every element against the oracle."""
    w = synth.ATTN_PROJ
    inp = synth.make_workload_inputs(w)
    inp["wcscale"] = None
    inp["bias"] = None
    inp["lora_act_in"] = None
    inp["lora_up"] = None
    full_check(w.M, w.N, w.K, 0, w.seed, options=cfg, inp=inp)
