"""The allocation-free split-K entry point, svdq_w4a4_gemm_split_noalloc.

It serves callers that cannot allocate device memory -- code running while a
serving engine has reserved the whole device for its own memory pool, or in
a runtime that forbids cudaMalloc after start-up -- and therefore have no
workspace to hand to svdq_w4a4_gemm_split.  The split-K partial tiles then
live in the library's built-in scratch array.  These tests call it through
the C ABI and compare its output with the existing entry point's
(svdq_w4a4_gemm, or svdq_w4a4_gemm_prepacked for prepacked weights, in the
same 16-bit I/O type) under the operator's acceptance bound, on two calls in
a row with different inputs, check sampled rows against the CPU oracle, and
check the size limit.  This file is collected last, so a failure here leaves
every other test already run.
"""

import ctypes

import pytest
import torch

from gpu_util import oracle_y, parity, prepack_gpu, sample_rows, to_device
from nvfp4_w4a4_quantized_gb300 import binding, build, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    import oracle
    oracle.build()
    return binding.load()


def _noalloc(lib, d, out, M, N, K, R, options=None, prepacked=0):
    opts = binding.SvdqOptions(**options) if options else None
    args = [d["act"].data_ptr(), d["wgt"].data_ptr(), d["ascales"].data_ptr(),
            d["wscales"].data_ptr(), d["lora_act_in"].data_ptr() if R else None,
            d["lora_up"].data_ptr() if R else None, d["wcscale"].data_ptr(),
            d["bias"].data_ptr(), out.data_ptr(), M, N, K, R]
    stream = torch.cuda.current_stream().cuda_stream
    return lib.svdq_w4a4_gemm_split_noalloc(*args, ctypes.byref(opts) if opts else None,
                                            prepacked, stream)


@pytest.mark.parametrize("half", [False, True], ids=["bf16", "fp16"])
@pytest.mark.parametrize("prepacked", [0, 1], ids=["raw_weights", "prepacked_weights"])
def test_two_calls_in_a_row_match_the_existing_entry_point(lib, prepacked, half):
    # the MLP-down projection at 256 tokens: the planner splits its 48 tiles
    M, N, K, R = 256, 3072, 12288, 128
    opts = dict(io_dtype=binding.SVDQ_IO_FP16 if half else binding.SVDQ_IO_BF16)
    plan = binding.svdq_query_plan(M, N, K, R, options=dict(opts, k_splits=-1))
    assert plan["k_splits"] > 1
    assert 0 < plan["workspace_bytes"] <= binding.SVDQ_NOALLOC_SCRATCH_BYTES
    out_dtype = torch.float16 if half else torch.bfloat16
    for seed in (41, 42):
        inp = synth.make_inputs(M, N, K, R, seed=seed, half=half)
        if half:
            # at K = 12288 the workload's outputs reach past fp16's 65504: scale
            # the activations by 2^-3 (exponent field - 3; every drawn scale
            # byte has an exponent field >= 3)
            inp["ascales"] = inp["ascales"] - 24
        d = prepack_gpu(inp, R) if prepacked else to_device(inp)
        out = torch.full((M, N), float("nan"), dtype=out_dtype, device="cuda")
        assert _noalloc(lib, d, out, M, N, K, R, options=opts, prepacked=prepacked) == \
            binding.SVDQ_OK
        ref = torch.full((M, N), float("nan"), dtype=out_dtype, device="cuda")
        gemm = binding.svdq_w4a4_gemm_prepacked if prepacked else binding.svdq_w4a4_gemm
        gemm(d["act"], d["wgt"], d["ascales"], d["wscales"], d["lora_act_in"], d["lora_up"],
             d["wcscale"], d["bias"], ref, options=opts)
        torch.cuda.synchronize()
        code, site, _ = binding.svdq_read_device_status(clear=True)
        assert code == 0, f"device status {code} at wait site {site}"
        y = out.double().cpu().numpy()
        parity(y, ref.double().cpu().numpy())
        rows = sample_rows(M, 24, seed=seed)
        parity(y[rows], oracle_y(inp, M, N, K, R, rows=rows))


def test_plans_beyond_the_scratch_are_rejected(lib):
    # 19 tiles x 8 splits of a 128 x 256 tile: 19 * 7 fp32 partials > 16 MiB
    M, N, K, R = 2432, 256, 2048, 0
    opts = dict(cta_group=1, tile_n=256, k_splits=8)
    need = binding.svdq_workspace_size(M, N, K, R, options=opts)
    assert need > binding.SVDQ_NOALLOC_SCRATCH_BYTES
    inp = synth.make_inputs(M, N, K, R, seed=43)
    d = to_device(inp)
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(lib, d, out, M, N, K, R, options=opts) == binding.SVDQ_ERR_SCRATCH_LIMIT
