"""A bounded wait inside the kernel runs out and is reported, not hung on.

svdq_options_t.debug_fault = 1 makes the MMA issuers wait on a barrier that
no role ever arrives on, with a 50 ms limit: the kernel must end by itself,
record SVDQ_ERR_TIMEOUT and the wait site in the device status word, and leave
the CUDA context usable -- the next, normal call must match the oracle.
"""

import pytest
import torch

from gpu_util import oracle_y, parity, run_gpu, to_device
from nvfp4_w4a4_quantized_gb300 import binding, synth

pytestmark = pytest.mark.gpu

# The issuers' accumulator wait (the one debug_fault replaces) and the
# epilogue's wait for an accumulator that is never filled start together with
# the same limit; whichever expires first records the status.
SITES = {2, 8}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from nvfp4_w4a4_quantized_gb300 import build
    build.build()
    import oracle
    oracle.build()


@pytest.mark.parametrize("cfg", [dict(cta_group=2, tile_n=256), dict(cta_group=1, tile_n=128)],
                         ids=["cg2_n256", "cg1_n128"])
def test_expired_wait_is_reported_and_context_survives(cfg):
    M, N, K, R = 256, 256, 512, 32
    inp = synth.make_inputs(M, N, K, R, seed=71)
    d = to_device(inp)
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    binding.svdq_read_device_status(clear=True)
    rc = binding.svdq_w4a4_gemm(d["act"], d["wgt"], d["ascales"], d["wscales"],
                                d["lora_act_in"], d["lora_up"], d["wcscale"], d["bias"], out,
                                options=dict(cfg, debug_fault=1, timeout_ms=50), check=False)
    assert rc == binding.SVDQ_OK  # the launch itself is fine
    torch.cuda.synchronize()      # returns: the kernel gave up after its limit
    code, site, _ = binding.svdq_read_device_status(clear=True)
    assert code == binding.SVDQ_ERR_TIMEOUT
    assert site in SITES
    # the context is still usable and the status word was cleared
    y = run_gpu(inp, M, N, K, R, options=cfg)
    parity(y, oracle_y(inp, M, N, K, R))
