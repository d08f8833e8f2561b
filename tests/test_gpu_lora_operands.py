"""LoRA operands the shared accumulator cannot carry, through the C ABI.

The kernel accumulates LA @ LU' with LU' = LU / wcscale into the main
accumulator and multiplies the sum by wcscale in the epilogue ("SVDQuant W4A4
on Blackwell" §2: LoRA is not scaled by wcscale; §6.3: LoRA shares the
accumulator).  A column with wcscale == 0 has no LU', and a tiny wcscale can
push LU' past the 16-bit range.  The header states what happens then: that
column's LoRA term is lost (zero wcscale) or infinite (overflow), every other
column is exact to the usual bound, and the launch records the condition
with the column in the device status word.  These tests check all three
parts on the per-call and the prepacked routes.
"""

import numpy as np
import pytest
import torch

from gpu_util import oracle_y, parity, prepack_gpu, run_gpu, to_device
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
    import oracle
    oracle.build()
    binding.svdq_read_device_status(clear=True)


def _run_prepacked(inp, M, N, K, R, options=None):
    """Prepack (which records the status) and the prepacked call; status is
    read by the caller."""
    d = prepack_gpu(inp, R)
    half = inp["wcscale"].dtype == torch.float16
    out = torch.full((M, N), float("nan"), dtype=torch.float16 if half else torch.bfloat16,
                     device="cuda")
    binding.svdq_w4a4_gemm_prepacked(d["act"], d["wgt"], d["ascales"], d["wscales"],
                                     d["lora_act_in"], d["lora_up"], d["wcscale"], d["bias"],
                                     out, options=options)
    torch.cuda.synchronize()
    return out.to(torch.float64).cpu().numpy()


def _others_match(y, ref, bad):
    keep = np.ones(y.shape[1], dtype=bool)
    keep[list(bad)] = False
    parity(y[:, keep], ref[:, keep])


@pytest.mark.parametrize("route", ["per_call", "prepacked"])
@pytest.mark.parametrize("R", [32, 20])   # TMA-staged and direct-load LoRA rows
@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_zero_wcscale_drops_that_column_and_is_reported(cfg, R, route):
    M, N, K = 256, 384, 512
    inp = synth.make_inputs(M, N, K, R, seed=71)
    bad = (5, 130, N - 1)
    for n in bad:
        inp["wcscale"][n] = 0.0
    binding.svdq_read_device_status(clear=True)
    if route == "per_call":
        y = run_gpu(inp, M, N, K, R, options=cfg, check_status=False)
    else:
        y = _run_prepacked(inp, M, N, K, R, options=cfg)
    code, site, _ = binding.svdq_read_device_status(clear=True)
    assert code == binding.SVDQ_ERR_WCSCALE_ZERO
    assert site in bad
    # main * 0 + bias, with the LoRA term dropped: exactly bias
    bias = inp["bias"].double().numpy()
    for n in bad:
        assert np.array_equal(y[:, n], np.full(M, bias[n]))
    _others_match(y, oracle_y(inp, M, N, K, R), bad)


@pytest.mark.parametrize("route", ["per_call", "prepacked"])
@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_fp16_lu_overflow_is_reported(cfg, route):
    M, N, K, R = 256, 256, 256, 32
    inp = synth.make_inputs(M, N, K, R, seed=72, half=True)
    # 2^-24, the smallest fp16 subnormal: |LU / wcscale| ~ 0.05 * 2^24 > 65504
    inp["wcscale"][7] = 2.0 ** -24
    inp["lora_up"][7, :] = 0.05
    binding.svdq_read_device_status(clear=True)
    opts = dict(cfg, io_dtype=binding.SVDQ_IO_FP16)
    if route == "per_call":
        d = to_device(inp)
        out = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        binding.svdq_w4a4_gemm(d["act"], d["wgt"], d["ascales"], d["wscales"], d["lora_act_in"],
                               d["lora_up"], d["wcscale"], d["bias"], out, options=opts)
        torch.cuda.synchronize()
        y = out.double().cpu().numpy()
    else:
        y = _run_prepacked(inp, M, N, K, R, options=opts)
    code, site, _ = binding.svdq_read_device_status(clear=True)
    assert code == binding.SVDQ_ERR_LU_OVERFLOW
    assert site == 7
    assert not np.all(np.isfinite(y[:, 7]))
    _others_match(y, oracle_y(inp, M, N, K, R), (7,))


def test_zero_wcscale_without_lora_is_exact_and_silent():
    # R = 0: nothing is divided, so a zero wcscale is an ordinary column (y = bias)
    M, N, K, R = 256, 256, 512, 0
    inp = synth.make_inputs(M, N, K, R, seed=73)
    inp["wcscale"][3] = 0.0
    binding.svdq_read_device_status(clear=True)
    y = run_gpu(inp, M, N, K, R)
    parity(y, oracle_y(inp, M, N, K, R))
