"""Bit-reproducibility through the C ABI: the same call on the same inputs gives
the same output bits every time.

Every MMA accumulates in fp32, so the order in which ring items reach the
tensor core decides the last bits of the result.  By default the two MMA
issuer threads take turns, so that order is the ring order on every call,
whatever the timing of the loads: LoRA items built from direct loads (R not a
multiple of 8), tile starts after an epilogue (every stage of the ring ready
at once), full-size shapes with several waves of tiles.  With
svdq_options_t.relaxed_order the issuers run freely: the bits may change from
call to call, the result stays within the acceptance bound.
"""

import numpy as np
import pytest
import torch

from gpu_util import oracle_y, parity, prepack_gpu, run_gpu, run_gpu_prepacked, run_gpu_split
from nvfp4_w4a4_quantized_gb300 import binding, synth

pytestmark = pytest.mark.gpu

CONFIGS = [dict(cta_group=1, tile_n=128), dict(cta_group=1, tile_n=256),
           dict(cta_group=2, tile_n=256)]
CFG_IDS = ["cg1_n128", "cg1_n256", "cg2_n256"]
REPEATS = 12


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import oracle
    from nvfp4_w4a4_quantized_gb300 import build
    build.build()
    oracle.build()


@pytest.mark.parametrize("M,N,K,R", [(400, 528, 1088, 100), (1024, 1536, 3072, 32),
                                     (512, 768, 2048, 128), (4096, 3072, 3072, 32)])
@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_repeated_calls_bit_identical(M, N, K, R, cfg):
    inp = synth.make_inputs(M, N, K, R, seed=M + N + K + R)
    first = run_gpu(inp, M, N, K, R, options=cfg)
    for _ in range(REPEATS - 1):
        y = run_gpu(inp, M, N, K, R, options=cfg)
        assert np.array_equal(y, first), \
            f"{int((y != first).sum())} of {y.size} outputs differ between repeated calls"


def _packed_scales(inp, M, N, K, R, cfg):
    """Prepacked weights and activation scales in the word layout."""
    d = prepack_gpu(inp, R)
    d["ascales"] = binding.svdq_pack_scales(d["ascales"])
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    binding.svdq_w4a4_gemm_prepacked(d["act"], d["wgt"], d["ascales"], d["wscales"],
                                     d["lora_act_in"], d["lora_up"], d.get("wcscale"),
                                     d.get("bias"), out, options=dict(cfg, act_scales_packed=1))
    torch.cuda.synchronize()
    code, site, _ = binding.svdq_read_device_status(clear=True)
    assert code == 0, f"device status {code} at wait site {site}"
    return out.double().cpu().numpy()


ROUTES = {
    "prepacked": lambda inp, M, N, K, R, cfg: run_gpu_prepacked(inp, M, N, K, R, options=cfg),
    "packed_scales": _packed_scales,
    "split_k3": lambda inp, M, N, K, R, cfg: run_gpu_split(inp, M, N, K, R,
                                                           options=dict(cfg, k_splits=3))[0],
    "fp16": lambda inp, M, N, K, R, cfg: run_gpu(inp, M, N, K, R, options=cfg),
}


@pytest.mark.parametrize("route", list(ROUTES))
@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_every_route_bit_identical(route, cfg):
    # 4096 = 16 K blocks: three K splits of 5-6 blocks; 8 to 32 tiles per config
    M, N, K, R = 512, 1024, 4096, 64
    inp = synth.make_inputs(M, N, K, R, seed=11, half=(route == "fp16"))
    first = ROUTES[route](inp, M, N, K, R, cfg)
    for _ in range(5):
        y = ROUTES[route](inp, M, N, K, R, cfg)
        assert np.array_equal(y, first), \
            f"{int((y != first).sum())} of {y.size} outputs differ between repeated calls"


@pytest.mark.parametrize("M,N,K,R", [(400, 528, 1088, 100), (512, 768, 2048, 128)])
@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_relaxed_order_within_bound(M, N, K, R, cfg):
    inp = synth.make_inputs(M, N, K, R, seed=M + N + K + R + 1)
    ref = oracle_y(inp, M, N, K, R)
    for _ in range(4):
        parity(run_gpu(inp, M, N, K, R, options=dict(cfg, relaxed_order=1)), ref)


@pytest.mark.parametrize("route", ["prepacked", "packed_scales", "split_k3"])
@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_relaxed_order_routes_within_bound(route, cfg):
    M, N, K, R = 512, 1024, 4096, 64
    inp = synth.make_inputs(M, N, K, R, seed=13)
    ref = oracle_y(inp, M, N, K, R)
    for _ in range(2):
        parity(ROUTES[route](inp, M, N, K, R, dict(cfg, relaxed_order=1)), ref)


def test_concurrent_calls_from_two_threads_on_two_streams():
    # the library is thread-safe and calls on different streams are independent:
    # two host threads, each on its own stream, issue the operator and the
    # activation quantiser on different shapes (different plans, tensor maps and
    # one-time set-up) at once; every output equals the serial call's bits
    import threading

    from gpu_util import to_device

    shapes = [(512, 768, 1024, 32), (384, 512, 2048, 128)]
    devs = [to_device(synth.make_inputs(*s, seed=90 + i)) for i, s in enumerate(shapes)]
    xs = [synth.make_activations(M, K, R, seed=95 + i) for i, (M, N, K, R) in enumerate(shapes)]
    xs = [(a["x"].cuda(), a["lora_down"].cuda()) for a in xs]

    def gemm(i, out, stream=None):
        d = devs[i]
        binding.svdq_w4a4_gemm(d["act"], d["wgt"], d["ascales"], d["wscales"], d["lora_act_in"],
                               d["lora_up"], d["wcscale"], d["bias"], out, stream=stream)

    def quant(i, stream=None):
        return binding.svdq_quantize_act(*xs[i], stream=stream)

    refs = []
    for i, (M, N, K, R) in enumerate(shapes):
        out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        gemm(i, out)
        refs.append((out, quant(i)))
    torch.cuda.synchronize()
    results, errors = [None, None], []

    def worker(i):
        try:
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            M, N, K, R = shapes[i]
            got = []
            with torch.cuda.stream(s):
                for _ in range(8):
                    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
                    gemm(i, out, stream=s)
                    got.append((out, quant(i, stream=s)))
            s.synchronize()
            results[i] = got
        except Exception as e:  # re-raised in the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    code, site, _ = binding.svdq_read_device_status(clear=True)
    assert code == 0, (code, site)
    for i in range(2):
        ref_out, ref_q = refs[i]
        for out, qo in results[i]:
            assert torch.equal(out, ref_out)
            for a, b in zip(qo, ref_q):
                assert torch.equal(a, b)
