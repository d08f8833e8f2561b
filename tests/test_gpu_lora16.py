"""The operator with 16-bit LoRA activations (svdq_options_t.lora_act_16bit):
lora_act_in holds the 16-bit values the tensor cores take, and the kernel
carries 64 ranks per LoRA ring item instead of 32.

The result must match the CPU oracle on those values within the acceptance
bound, and must equal bit for bit the fp32 route's result on the same values
(the fp32 route rounds LA to the same 16-bit numbers), on every tile
configuration, per call and prepacked, unsplit and split-K, bf16 and fp16,
for R below, at and above one 64-rank item and for ragged tiles.
"""

import numpy as np
import pytest
import torch

from gpu_util import oracle_y, parity, prepack_gpu, sample_rows, to_device
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


def _inputs(M, N, K, R, seed, half=False):
    inp = synth.make_inputs(M, N, K, R, seed=seed, half=half)
    h16 = torch.float16 if half else torch.bfloat16
    # the LoRA activation as the 16-bit values both routes feed the tensor cores
    inp["lora_act_in"] = inp["lora_act_in"].to(h16).to(torch.float32)
    return inp, h16


def _run(inp, M, N, K, R, opts, h16, la16, prepacked=False, split=False):
    d = prepack_gpu(inp, R) if prepacked else to_device(inp)
    o = dict(opts)
    if h16 == torch.float16:
        o["io_dtype"] = binding.SVDQ_IO_FP16
    la = d["lora_act_in"]
    if la16:
        o["lora_act_16bit"] = 1
        la = la.to(h16)
    out = torch.full((M, N), float("nan"), dtype=h16, device="cuda")
    args = (d["act"], d["wgt"], d["ascales"], d["wscales"], la, d["lora_up"], d["wcscale"],
            d["bias"], out)
    if split:
        o["k_splits"] = -1
        nbytes = binding.svdq_workspace_size(M, N, K, R, options=o)
        ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device="cuda")
        binding.svdq_w4a4_gemm_split(*args, ws, options=o, weights_prepacked=prepacked)
    elif prepacked:
        binding.svdq_w4a4_gemm_prepacked(*args, options=o)
    else:
        binding.svdq_w4a4_gemm(*args, options=o)
    torch.cuda.synchronize()
    code, site, _ = binding.svdq_read_device_status(clear=True)
    assert code == 0, f"device status {code} at wait site {site}"
    return out.double().cpu().numpy()


@pytest.mark.parametrize("route", ["per_call", "prepacked"])
@pytest.mark.parametrize("R", [8, 40, 64, 72, 128])
@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_matches_oracle_and_fp32_route(cfg, R, route):
    M, N, K = 272, 400, 1088  # ragged tiles in both directions, partial last K block
    inp, h16 = _inputs(M, N, K, R, seed=60 + R)
    y16 = _run(inp, M, N, K, R, cfg, h16, la16=True, prepacked=route == "prepacked")
    y32 = _run(inp, M, N, K, R, cfg, h16, la16=False, prepacked=route == "prepacked")
    assert np.array_equal(y16, y32)
    parity(y16, oracle_y(inp, M, N, K, R))


def test_lora_only_isolates_the_term():
    # all act codes 0: y = bias + LA @ LU exactly what the LoRA term contributes
    M, N, K, R = 256, 512, 512, 128
    inp, h16 = _inputs(M, N, K, R, seed=61)
    inp["act"].zero_()
    y = _run(inp, M, N, K, R, dict(cta_group=2, tile_n=256), h16, la16=True)
    ref = oracle_y(inp, M, N, K, R)
    la = inp["lora_act_in"].double().numpy()
    lu = inp["lora_up"].double().numpy()
    extra = 2.0 ** -7 * (np.abs(la) @ np.abs(lu).T)
    parity(y, ref, extra=extra)


def test_fp16_and_split_k():
    M, N, K, R = 256, 3072, 12288, 128  # the planner splits this shape
    inp, h16 = _inputs(M, N, K, R, seed=62, half=True)
    inp["ascales"] = inp["ascales"] - 24  # fp16 outputs stay in range at K = 12288
    assert binding.svdq_query_plan(M, N, K, R, options=dict(
        io_dtype=binding.SVDQ_IO_FP16, lora_act_16bit=1, k_splits=-1))["k_splits"] > 1
    y16 = _run(inp, M, N, K, R, {}, h16, la16=True, split=True)
    y32 = _run(inp, M, N, K, R, {}, h16, la16=False, split=True)
    assert np.array_equal(y16, y32)
    rows = sample_rows(M, 32, seed=3)
    parity(y16[rows], oracle_y(inp, M, N, K, R, rows=rows))


def test_plan_and_rejections():
    p32 = binding.svdq_query_plan(4096, 3072, 12288, 128)
    p16 = binding.svdq_query_plan(4096, 3072, 12288, 128, options=dict(lora_act_16bit=1))
    assert (p32["lora_blocks"], p16["lora_blocks"]) == (4, 2)
    # 16-bit LoRA rows go through TMA: R must keep them 16-byte strided
    inp, h16 = _inputs(256, 256, 256, 20, seed=63)
    d = to_device(inp)
    out = torch.empty((256, 256), dtype=h16, device="cuda")
    rc = binding.svdq_w4a4_gemm(d["act"], d["wgt"], d["ascales"], d["wscales"],
                                d["lora_act_in"].to(h16), d["lora_up"], d["wcscale"], d["bias"],
                                out, options=dict(lora_act_16bit=1), check=False)
    assert rc == binding.SVDQ_ERR_BAD_OPTION
