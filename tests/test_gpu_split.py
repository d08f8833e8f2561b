"""Split-K (svdq_w4a4_gemm_split) against the oracle through the C ABI.

Each output tile's K range is divided between clusters; all but the last
split store fp32 partial tiles and raise a per-launch flag, the last adds
them to its accumulator and applies the epilogue.  Same acceptance bound as
the unsplit operator (the K parts are summed in fp32, in another order).
"""

import numpy as np
import pytest
import torch

from gpu_util import oracle_y, parity, run_gpu, run_gpu_split, sample_rows
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


@pytest.mark.parametrize("M,N,K,R,splits", [
    (256, 384, 1024, 32, 2),    # four K blocks, two splits, LoRA on split 0
    (256, 384, 1024, 32, 4),    # one K block per split
    (272, 144, 1088, 20, 3),    # ragged M/N, partial last K block, direct LoRA loads
    (256, 512, 2048, 0, 5),     # no LoRA, uneven split sizes
    (256, 256, 3072, 128, 8),   # maximum rank and split count
])
@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_forced_splits_full_matrix(M, N, K, R, splits, cfg):
    inp = synth.make_inputs(M, N, K, R, seed=M + N + K + R + splits)
    y, _ = run_gpu_split(inp, M, N, K, R, options=dict(cfg, k_splits=splits))
    parity(y, oracle_y(inp, M, N, K, R))


def test_planner_split_small_m_sampled_rows():
    # 256 x 3072 x 12288 R128: the planner splits each of its 48 tiles in three
    M, N, K, R = 256, 3072, 12288, 128
    plan = binding.svdq_query_plan(M, N, K, R, options=dict(k_splits=-1))
    assert plan["k_splits"] > 1
    inp = synth.make_inputs(M, N, K, R, seed=4)
    y, _ = run_gpu_split(inp, M, N, K, R)
    rows = sample_rows(M, 40, seed=4)
    ref = oracle_y(inp, M, N, K, R, rows=rows)
    parity(y[rows], ref)
    # the unsplit launch agrees within the same bound
    y1 = run_gpu(inp, M, N, K, R)
    parity(y, y1)


def test_consecutive_calls_share_the_workspace():
    # the second call must see only its own partials (each completed call
    # leaves its flags lowered)
    M, N, K, R = 256, 384, 1024, 16
    cfg = dict(cta_group=1, tile_n=128, k_splits=4)
    a = synth.make_inputs(M, N, K, R, seed=21)
    b = synth.make_inputs(M, N, K, R, seed=22)
    ya, ws = run_gpu_split(a, M, N, K, R, options=cfg)
    yb, _ = run_gpu_split(b, M, N, K, R, options=cfg, workspace=ws)
    ya2, _ = run_gpu_split(a, M, N, K, R, options=cfg, workspace=ws)
    parity(ya, oracle_y(a, M, N, K, R))
    parity(yb, oracle_y(b, M, N, K, R))
    assert np.array_equal(ya, ya2)


@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_split_fp16_and_prepacked(cfg):
    M, N, K, R = 256, 384, 1536, 32
    inp = synth.make_inputs(M, N, K, R, seed=31, half=True)
    y, _ = run_gpu_split(inp, M, N, K, R, options=dict(cfg, k_splits=3))
    parity(y, oracle_y(inp, M, N, K, R))
    inp = synth.make_inputs(M, N, K, R, seed=32)
    y, _ = run_gpu_split(inp, M, N, K, R, options=dict(cfg, k_splits=3), prepacked=True)
    parity(y, oracle_y(inp, M, N, K, R))


def test_workspace_errors():
    M, N, K, R = 256, 384, 1024, 16
    inp = synth.make_inputs(M, N, K, R, seed=5)
    d = {k: v.cuda() for k, v in inp.items()}
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    args = (d["act"], d["wgt"], d["ascales"], d["wscales"], d["lora_act_in"], d["lora_up"],
            d["wcscale"], d["bias"], out)
    cfg = dict(cta_group=1, tile_n=128, k_splits=2)
    # a forced split on an entry point without a workspace
    assert binding.svdq_w4a4_gemm(*args, options=cfg, check=False) == binding.SVDQ_ERR_WORKSPACE
    # a workspace smaller than the plan needs
    need = binding.svdq_workspace_size(M, N, K, R, options=cfg)
    small = torch.zeros(need // 2, dtype=torch.uint8, device="cuda")
    assert binding.svdq_w4a4_gemm_split(*args, small, options=cfg, check=False) == \
        binding.SVDQ_ERR_WORKSPACE
    torch.cuda.synchronize()


@pytest.mark.parametrize("cfg", [CONFIGS[0], CONFIGS[2]], ids=[CFG_IDS[0], CFG_IDS[2]])
def test_graph_replay_with_new_inputs(cfg):
    """A split launch captured once in a CUDA graph and replayed on new inputs
    copied into the same buffers: every replay must fold only its own
    partials (the flags are lowered by each launch, nothing per call is baked
    into the graph).  Each replay is compared with the unsplit operator on
    the same inputs."""
    M, N, K, R = 256, 512, 2048, 32
    opts = dict(cfg, k_splits=4)
    seeds = (61, 62, 63)
    sets = [synth.make_inputs(M, N, K, R, seed=s) for s in seeds]
    d = {k: v.cuda() for k, v in sets[0].items()}
    nbytes = binding.svdq_workspace_size(M, N, K, R, options=opts)
    ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device="cuda")
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    args = (d["act"], d["wgt"], d["ascales"], d["wscales"], d["lora_act_in"], d["lora_up"],
            d["wcscale"], d["bias"], out, ws)
    # warm the library's one-time set-up outside the capture
    binding.svdq_w4a4_gemm_split(*args, options=opts)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        binding.svdq_w4a4_gemm_split(*args, options=opts, stream=torch.cuda.current_stream())
    for s, inp in zip(seeds, sets):
        for k, v in inp.items():
            d[k].copy_(v)
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        code, site, _ = binding.svdq_read_device_status(clear=True)
        assert code == 0, f"device status {code} at wait site {site} (seed {s})"
        y = out.double().cpu().numpy()
        ref = run_gpu(inp, M, N, K, R)
        parity(y, ref)
        rows = sample_rows(M, 16, seed=s)
        parity(y[rows], oracle_y(inp, M, N, K, R, rows=rows))
