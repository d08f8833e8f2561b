"""Weight-side prepack ("SVDQuant W4A4 on Blackwell" §3.1 scale words per
64-wide MMA step, §6.3 LU' = LU / wcscale sharing the main accumulator)
through the C ABI.

The prepack kernel's outputs are bytes and 16-bit values whose rounding both
sides take in fp32, so they must match the oracle's prepack bit for bit.  The
prepacked operator computes the same operator: it meets the acceptance bound
against the oracle evaluated on the ORIGINAL weights, and - the scale words
and LU' being what the fused kernel otherwise builds per call - it is bit
identical to the unpacked call in the same launch configuration.
"""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import (oracle_y, parity, prepack_gpu, run_gpu, run_gpu_prepacked, sample_rows)
from nvfp4_w4a4_quantized_gb300 import binding, synth

pytestmark = pytest.mark.gpu

CONFIGS = [dict(cta_group=1, tile_n=128), dict(cta_group=1, tile_n=256),
           dict(cta_group=2, tile_n=256)]
CFG_IDS = ["cg1_n128", "cg1_n256", "cg2_n256"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from nvfp4_w4a4_quantized_gb300 import build
    build.build()
    oracle.build()


def _u16(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _edge_weights(inp, half):
    """Subnormal, signed-zero, exact and zero-wcscale entries in the LoRA weights."""
    lu, wc = inp["lora_up"].clone(), inp["wcscale"].clone()
    tiny = 2.0 ** -20 if half else 2.0 ** -130
    lu.view(-1)[:4] = torch.tensor([tiny, -3 * tiny, 0.0, -0.0], dtype=lu.dtype)
    wc[0], wc[1], wc[2], wc[3], wc[5] = 3.0, 0.75, 1e-3, 7.0, 0.0
    return dict(inp, lora_up=lu, wcscale=wc)


@pytest.mark.parametrize("N,K,R", [(16, 64, 1), (272, 320, 20), (528, 1088, 100),
                                   (3072, 3072, 32), (12288, 3072, 128)])
@pytest.mark.parametrize("half", [False, True], ids=["bf16", "fp16"])
@pytest.mark.parametrize("wc_kind", ["synthetic", "edge", "none"])
def test_prepack_kernel_bit_exact(N, K, R, half, wc_kind):
    inp = synth.make_inputs(16, N, K, R, seed=N + K + R, half=half)
    if wc_kind == "edge":
        inp = _edge_weights(inp, half)
    elif wc_kind == "none":
        inp["wcscale"] = None
    binding.svdq_read_device_status(clear=True)
    d = prepack_gpu(inp, R)
    torch.cuda.synchronize()
    # a zero wcscale (edge weights, column 5) has no LU' = LU / wcscale: the
    # prepack writes 0 there and records it in the device status word
    code, site, _ = binding.svdq_read_device_status(clear=True)
    if wc_kind == "edge" and R > 0 and N > 5:
        assert (code, site) == (binding.SVDQ_ERR_WCSCALE_ZERO, 5)
    else:
        assert code == 0, (code, site)
    wpk = d["wscales"].cpu().numpy().view(np.uint32)
    assert np.array_equal(wpk, oracle.prepack_wscales(inp["wscales"], N, K))
    want = oracle.prepack_lora_up(inp["lora_up"], inp["wcscale"], N, R, half=half)
    assert np.array_equal(_u16(d["lora_up"]), want)


def test_prepack_without_lora():
    N, K = 256, 512
    inp = synth.make_inputs(16, N, K, 0, seed=1)
    d = prepack_gpu(inp, 0)
    torch.cuda.synchronize()
    assert d["lora_up"] is None
    assert np.array_equal(d["wscales"].cpu().numpy().view(np.uint32),
                          oracle.prepack_wscales(inp["wscales"], N, K))


@pytest.mark.parametrize("half", [False, True], ids=["bf16", "fp16"])
@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_tiny_workload_full_matrix_prepacked(cfg, half):
    w = synth.TINY
    inp = synth.make_inputs(w.M, w.N, w.K, w.R, w.seed, half=half)
    y = run_gpu_prepacked(inp, w.M, w.N, w.K, w.R, options=cfg)
    parity(y, oracle_y(inp, w.M, w.N, w.K, w.R))


@pytest.mark.parametrize("M,N,K,R", [
    (272, 144, 320, 20),     # ragged, partial K block, R not a multiple of 8 (direct LoRA loads)
    (400, 528, 1088, 100),   # several tiles, several LoRA blocks
    (256, 272, 512, 128),    # maximum rank, TMA LoRA rows
    (256, 256, 256, 0),      # no LoRA
])
@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_prepacked_matches_oracle_and_unpacked_bitwise(M, N, K, R, cfg):
    inp = synth.make_inputs(M, N, K, R, seed=M + N + K + R + 2)
    y_p = run_gpu_prepacked(inp, M, N, K, R, options=cfg)
    parity(y_p, oracle_y(inp, M, N, K, R))
    y_u = run_gpu(inp, M, N, K, R, options=cfg)
    assert np.array_equal(y_p, y_u), "prepacked and per-call packing differ"


@pytest.mark.parametrize("wc_value", [0.5, 2.0])
@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_lora_only_prepacked(wc_value, cfg):
    # act codes all zero: y = bias + lora_act_in @ lora_up, LoRA NOT scaled
    # by wcscale, through the pre-divided LU'.  Bound as for the per-call
    # route: 2^-7 sum_r |la*lu| (bf16 operands, fp32 sums) + 2^-8 |y| + 1e-6.
    M, N, K, R = 256, 384, 256, 32
    inp = synth.make_inputs(M, N, K, R, 7)
    inp["act"][:] = 0
    inp["wcscale"][:] = wc_value
    y = run_gpu_prepacked(inp, M, N, K, R, options=cfg)
    la = inp["lora_act_in"].double().numpy()
    lu = inp["lora_up"].double().numpy()
    mag = np.abs(la) @ np.abs(lu).T
    parity(y, oracle_y(inp, M, N, K, R), rel=2.0 ** -8, rms_frac=0.0,
           extra=2.0 ** -7 * mag + 1e-6)


@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_null_wcscale_and_bias_prepacked(cfg):
    M, N, K, R = 256, 256, 256, 16
    inp = synth.make_inputs(M, N, K, R, 9)
    inp["wcscale"] = None
    inp["bias"] = None
    y = run_gpu_prepacked(inp, M, N, K, R, options=cfg)
    parity(y, oracle_y(inp, M, N, K, R))


@pytest.mark.parametrize("half", [False, True], ids=["bf16", "fp16"])
def test_attn_proj_sampled_rows_prepacked(half):
    # the full attention-projection workload in the default launch configuration
    w = synth.ATTN_PROJ
    inp = synth.make_inputs(w.M, w.N, w.K, w.R, w.seed, half=half)
    y = run_gpu_prepacked(inp, w.M, w.N, w.K, w.R)
    rows = sample_rows(w.M, 40, seed=w.seed)
    parity(y[rows], oracle_y(inp, w.M, w.N, w.K, w.R, rows=rows))
