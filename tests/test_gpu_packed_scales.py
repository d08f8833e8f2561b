"""Activation scales in the word layout (svdq_options_t.act_scales_packed and
svdq_pack_scales) through the C ABI.

The words are the scales the kernel otherwise builds from the raw rows, so
every route — per-call or prepacked weights, unsplit or split-K — must give
the oracle's result within the acceptance bound and the raw-layout call's
result bit for bit.
"""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import oracle_y, parity, prepack_gpu, run_gpu, run_gpu_prepacked, sample_rows, \
    to_device
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


def _run(inp, M, N, K, R, cfg, prepacked=False, workspace=None):
    """The operator with packed activation scales; y as float64 numpy."""
    d = prepack_gpu(inp, R) if prepacked else to_device(inp)
    d["ascales"] = binding.svdq_pack_scales(d["ascales"])
    opts = dict(cfg or {}, act_scales_packed=1)
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    args = (d["act"], d["wgt"], d["ascales"], d["wscales"], d["lora_act_in"] if R else None,
            d["lora_up"] if R else None, d.get("wcscale"), d.get("bias"), out)
    if workspace is not None:
        binding.svdq_w4a4_gemm_split(*args, workspace, options=opts,
                                     weights_prepacked=prepacked)
    elif prepacked:
        binding.svdq_w4a4_gemm_prepacked(*args, options=opts)
    else:
        binding.svdq_w4a4_gemm(*args, options=opts)
    torch.cuda.synchronize()
    code, site, _ = binding.svdq_read_device_status(clear=True)
    assert code == 0, f"device status {code} at wait site {site}"
    return out.double().cpu().numpy()


@pytest.mark.parametrize("rows,K", [(16, 64), (272, 1088), (4096, 3072), (12288, 12288)])
def test_pack_scales_bit_exact(rows, K):
    sc = torch.randint(0, 256, (K // 16, rows), dtype=torch.uint8,
                       generator=torch.Generator().manual_seed(rows + K))
    pk = binding.svdq_pack_scales(sc.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(pk.cpu().numpy().view(np.uint32), oracle.pack_scales(sc, rows, K))


@pytest.mark.parametrize("M,N,K,R", [(256, 256, 256, 32), (272, 144, 1088, 20),
                                     (400, 528, 1088, 100)])
@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_packed_act_scales_match_oracle_and_raw_layout(M, N, K, R, cfg):
    inp = synth.make_inputs(M, N, K, R, seed=M + N + K + R + 7)
    y = _run(inp, M, N, K, R, cfg)
    parity(y, oracle_y(inp, M, N, K, R))
    assert np.array_equal(y, run_gpu(inp, M, N, K, R, options=cfg))
    yp = _run(inp, M, N, K, R, cfg, prepacked=True)
    parity(yp, oracle_y(inp, M, N, K, R))
    assert np.array_equal(yp, run_gpu_prepacked(inp, M, N, K, R, options=cfg))


@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_packed_act_scales_split_k(cfg):
    M, N, K, R = 256, 384, 2048, 32
    inp = synth.make_inputs(M, N, K, R, seed=61)
    ws = torch.zeros(binding.svdq_workspace_size(M, N, K, R, options=dict(cfg, k_splits=4)),
                     dtype=torch.uint8, device="cuda")
    y = _run(inp, M, N, K, R, dict(cfg, k_splits=4), workspace=ws)
    parity(y, oracle_y(inp, M, N, K, R))


def test_attn_proj_fully_packed_sampled_rows():
    w = synth.ATTN_PROJ
    inp = synth.make_inputs(w.M, w.N, w.K, w.R, w.seed)
    y = _run(inp, w.M, w.N, w.K, w.R, None, prepacked=True)
    rows = sample_rows(w.M, 40, seed=w.seed)
    parity(y[rows], oracle_y(inp, w.M, w.N, w.K, w.R, rows=rows))
