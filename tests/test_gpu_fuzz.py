"""Randomised (fixed-seed) sweep of shapes and launch options through the C
ABI, against the CPU oracle.

The operator: M, N, K, R and every route drawn at random -- tile and CTA
group, ring depth, grid cap, per-call or prepacked weights, raw or packed
activation scales, 16-bit or fp32 LoRA activations, split-K with the
planner's or a forced split count, bit-reproducible or relaxed issue order,
bf16 or fp16 I/O, wcscale / bias present or absent -- checked on sampled rows (every 128-row tile edge and
lane quadrant plus random rows) under the acceptance bound.  The activation
quantiser: random M, K, R, input type and scale layout, codes and scales bit
for bit, lora_act_in within its fp32 bound.  Each case is independent; a
failure names its seed.
"""

import numpy as np
import pytest
import torch

from gpu_util import oracle_y, parity, prepack_gpu, sample_rows, to_device
from nvfp4_w4a4_quantized_gb300 import binding, synth
from oracle import quant_ref as q

pytestmark = pytest.mark.gpu

GEMM_CASES = 96
QUANT_CASES = 48


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from nvfp4_w4a4_quantized_gb300 import build
    build.build()
    import oracle
    oracle.build()
    binding.svdq_read_device_status(clear=True)


def _gemm_case(seed):
    rng = np.random.default_rng(1000 + seed)
    M = int(rng.integers(1, 160)) * 16
    N = int(rng.integers(1, 72)) * 16
    K = int(rng.integers(1, 48)) * 64
    R = int(rng.choice([0, 1, 7, 16, 20, 32, 40, 64, 100, 128]))
    half = bool(rng.random() < 0.25)
    cfg = [dict(), dict(cta_group=1, tile_n=128), dict(cta_group=1, tile_n=256),
           dict(cta_group=2, tile_n=256)][int(rng.integers(0, 4))]
    opts = dict(cfg)
    if rng.random() < 0.3:
        opts["stages"] = int(rng.integers(2, 6))
    if rng.random() < 0.2:
        opts["max_ctas"] = int(rng.integers(1, 40))
    if rng.random() < 0.3:
        opts["relaxed_order"] = 1
    route = str(rng.choice(["per_call", "prepacked", "split"]))
    packed_act = bool(rng.random() < 0.3)
    affine = str(rng.choice(["both", "none", "wc_only", "bias_only"]))
    forced_split = int(rng.integers(2, 5)) if route == "split" and rng.random() < 0.5 else -1
    la16 = bool(R % 8 == 0 and R > 0 and rng.random() < 0.4)
    return M, N, K, R, half, opts, route, packed_act, affine, forced_split, la16


@pytest.mark.parametrize("seed", range(GEMM_CASES))
def test_operator_random_shapes_and_routes(seed):
    M, N, K, R, half, opts, route, packed_act, affine, forced_split, la16 = _gemm_case(seed)
    if route == "split":
        # a forced split needs a K block per part
        if forced_split > 0 and forced_split > -(-K // 256):
            forced_split = -1
        opts = dict(opts, k_splits=forced_split)
    if half:
        opts["io_dtype"] = binding.SVDQ_IO_FP16
    # a forced depth, grid cap or split count the planner cannot honour is
    # rejected with SVDQ_ERR_BAD_OPTION before anything runs: drop it
    for drop in ((), ("stages",), ("stages", "max_ctas"), ("stages", "max_ctas", "k_splits")):
        o = {key: v for key, v in opts.items() if key not in drop}
        if "k_splits" in drop:
            o["k_splits"] = -1
        try:
            binding.svdq_query_plan(M, N, K, R, options=o)
        except binding.SvdqError as e:
            assert e.status == binding.SVDQ_ERR_BAD_OPTION, (seed, e.status)
            continue
        opts = o
        break
    inp = synth.make_inputs(M, N, K, R, seed=2000 + seed, half=half)
    if half:
        inp["ascales"] = inp["ascales"] - 8  # keep fp16 outputs in range at long K
    if affine in ("none", "bias_only"):
        inp["wcscale"] = None
    if affine in ("none", "wc_only"):
        inp["bias"] = None
    if R == 0:
        inp["lora_act_in"] = None
        inp["lora_up"] = None
    h16 = torch.float16 if half else torch.bfloat16
    if la16:
        # 16-bit LoRA activations: the oracle sees the same (rounded) values
        inp["lora_act_in"] = inp["lora_act_in"].to(h16).to(torch.float32)
    d = prepack_gpu(inp, R) if route == "prepacked" or (route == "split" and seed % 2) \
        else to_device(inp)
    prepacked = route == "prepacked" or (route == "split" and seed % 2 == 1)
    if packed_act:
        d["ascales"] = binding.svdq_pack_scales(d["ascales"])
        opts["act_scales_packed"] = 1
    la_in = d["lora_act_in"] if R else None
    if la16:
        opts["lora_act_16bit"] = 1
        la_in = la_in.to(h16)
    out = torch.full((M, N), float("nan"), dtype=h16, device="cuda")
    args = (d["act"], d["wgt"], d["ascales"], d["wscales"], la_in,
            d["lora_up"] if R else None, d.get("wcscale"), d.get("bias"), out)
    if route == "split":
        nbytes = binding.svdq_workspace_size(M, N, K, R, options=opts)
        ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device="cuda")
        binding.svdq_w4a4_gemm_split(*args, ws, options=opts, weights_prepacked=prepacked)
    elif prepacked:
        binding.svdq_w4a4_gemm_prepacked(*args, options=opts)
    else:
        binding.svdq_w4a4_gemm(*args, options=opts)
    torch.cuda.synchronize()
    code, site, _ = binding.svdq_read_device_status(clear=True)
    assert code == 0, f"seed {seed}: device status {code} at wait site {site}"
    rows = sample_rows(M, 24, seed=seed)
    y = out.double().cpu().numpy()[rows]
    parity(y, oracle_y(inp, M, N, K, R, rows=rows))


@pytest.mark.parametrize("seed", range(QUANT_CASES))
def test_quantiser_random_shapes(seed):
    rng = np.random.default_rng(3000 + seed)
    M = int(rng.integers(1, 400)) * 16
    K = int(rng.integers(1, 80)) * 64
    R = int(rng.choice([0, 1, 5, 16, 24, 32, 48, 64, 96, 128]))
    half = bool(rng.random() < 0.35)
    packed = bool(rng.random() < 0.4)
    a = synth.make_activations(M, K, R, seed=4000 + seed, half=half)
    x, ld = a["x"], (a["lora_down"] if R else None)
    act, asc, la = binding.svdq_quantize_act(x.cuda(), ld.cuda() if R else None,
                                             scales_packed=packed)
    torch.cuda.synchronize()
    code, site, _ = binding.svdq_read_device_status(clear=True)
    assert code == 0, f"seed {seed}: device status {code} at wait site {site}"
    want_act, want_asc = q.quantize_act(x, M, K, half=half, packed=packed)
    np.testing.assert_array_equal(act.cpu().numpy(), want_act)
    got_asc = asc.cpu().numpy()
    np.testing.assert_array_equal(got_asc.view(np.uint32) if packed else got_asc, want_asc)
    if R:
        rows = sample_rows(M, 32, seed=seed)
        xr = x[torch.from_numpy(rows)]
        ref = q.lora_down(xr, ld, len(rows), K, R, half)
        mag = np.abs(q.decode_x(xr, len(rows), K, half)) @ np.abs(q.decode_x(ld, R, K, half)).T
        err = np.abs(la.double().cpu().numpy()[rows] - ref)
        assert np.all(err <= K * 2.0 ** -22 * mag + 1e-30), f"seed {seed}"
