"""The fp16 input/output variant (lora_up, wcscale, bias and y in IEEE fp16;
"SVDQuant W4A4 on Blackwell" §8 measures fp16 alongside bf16) against the
oracle, through the C ABI.  Same acceptance bound as the bf16 operator:
|y_gpu - y_ref| <= 2^-7 |y_ref| + 1e-3 rms(y_ref); fp16's finer rounding
only tightens what the GPU can reach."""

import numpy as np
import pytest
import torch

from gpu_util import oracle_y, parity, run_gpu, sample_rows
from nvfp4_w4a4_quantized_gb300 import synth

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
    import oracle
    oracle.build()


def full_check(M, N, K, R, seed, options=None, inp=None):
    inp = inp if inp is not None else synth.make_inputs(M, N, K, R, seed, half=True)
    assert inp["wcscale"] is None or inp["wcscale"].dtype == torch.float16
    y = run_gpu(inp, M, N, K, R, options=options)
    return parity(y, oracle_y(inp, M, N, K, R))


@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_tiny_workload_full_matrix_fp16(cfg):
    w = synth.TINY
    full_check(w.M, w.N, w.K, w.R, w.seed, options=cfg)


@pytest.mark.parametrize("M,N,K,R", [
    (272, 144, 320, 20),     # ragged, partial K block, R not a multiple of 8 (direct LoRA loads)
    (400, 528, 1088, 100),   # several tiles, two LoRA blocks
    (256, 272, 512, 128),    # maximum rank, TMA LoRA rows
])
@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_ragged_shapes_fp16(M, N, K, R, cfg):
    full_check(M, N, K, R, seed=M + N + K + R + 1, options=cfg)


@pytest.mark.parametrize("wc_value", [0.5, 2.0])
@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_lora_only_fp16(wc_value, cfg):
    # act codes all zero: y = bias + lora_act_in @ lora_up, LoRA not scaled
    # by wcscale.  Bound: 2^-10 sum_r |la*lu| (fp16 operands, fp32 sums)
    # + 2^-11 |y| (fp16 output) + 1e-6, doubled for the LU / wc division.
    M, N, K, R = 256, 384, 256, 32
    inp = synth.make_inputs(M, N, K, R, 7, half=True)
    inp["act"][:] = 0
    inp["wcscale"][:] = wc_value
    y = run_gpu(inp, M, N, K, R, options=cfg)
    ref = oracle_y(inp, M, N, K, R)
    la = inp["lora_act_in"].double().numpy()
    lu = inp["lora_up"].double().numpy()
    mag = np.abs(la) @ np.abs(lu).T
    parity(y, ref, rel=2.0 ** -10, rms_frac=0.0, extra=2.0 ** -9 * mag + 1e-6)


@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_affine_fp16(cfg):
    M, N, K = 256, 256, 512
    inp = synth.make_inputs(M, N, K, 0, 8, half=True)
    inp["wcscale"][:] = 2.0
    inp["ascales"][:] = 0x18
    inp["wscales"][:] = 0x18
    y = run_gpu(inp, M, N, K, 0, options=cfg)
    parity(y, oracle_y(inp, M, N, K, 0), rel=2.0 ** -10, rms_frac=1e-4)


@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_null_wcscale_and_bias_fp16(cfg):
    M, N, K, R = 256, 256, 256, 16
    inp = synth.make_inputs(M, N, K, R, 9, half=True)
    inp["wcscale"] = None
    inp["bias"] = None
    full_check(M, N, K, R, 9, inp=inp, options=cfg)


def test_fp16_and_bf16_agree_on_shared_values():
    # lora_up / wcscale / bias exactly representable in both types: the two
    # variants differ only by the output rounding (and LoRA operand rounding)
    M, N, K, R = 256, 256, 512, 32
    inp = synth.make_inputs(M, N, K, R, 10)
    g = torch.Generator().manual_seed(11)
    shared = lambda shape: torch.randint(-64, 64, shape, generator=g).to(torch.float32) / 64.0
    lu, wc, bi = shared((N, R)), shared((N,)) + 2.0, shared((N,))
    y_b = run_gpu(dict(inp, lora_up=lu.to(torch.bfloat16), wcscale=wc.to(torch.bfloat16),
                       bias=bi.to(torch.bfloat16)), M, N, K, R)
    y_h = run_gpu(dict(inp, lora_up=lu.to(torch.float16), wcscale=wc.to(torch.float16),
                       bias=bi.to(torch.float16)), M, N, K, R)
    ref = oracle_y(dict(inp, lora_up=lu.to(torch.bfloat16), wcscale=wc.to(torch.bfloat16),
                        bias=bi.to(torch.bfloat16)), M, N, K, R)
    parity(y_b, ref)
    parity(y_h, ref)
    # fp16 keeps 3 more mantissa bits: its error is no larger than bf16's
    assert np.abs(y_h - ref).max() <= np.abs(y_b - ref).max()


@pytest.mark.parametrize("cfg", [None, CONFIGS[2]], ids=["default", "cg2_n256"])
def test_attn_proj_sampled_rows_fp16(cfg):
    w = synth.ATTN_PROJ
    inp = synth.make_inputs(w.M, w.N, w.K, w.R, w.seed, half=True)
    y = run_gpu(inp, w.M, w.N, w.K, w.R, options=cfg)
    rows = sample_rows(w.M, 40, seed=w.seed)
    parity(y[rows], oracle_y(inp, w.M, w.N, w.K, w.R, rows=rows))
