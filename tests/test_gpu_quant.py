"""GPU parity of the activation quantiser (svdq_quantize_act) against the CPU
oracle (oracle/quant_ref.py), through the C ABI.

Codes and scale bytes are integer results: bit-exact.  lora_act_in is an fp32
contraction of 16-bit products: within the worst-case fp32 accumulation bound
K * 2^-22 * sum_k |x ld| (exact products, at most K roundings of a running
sum, with a factor 4 for the tensor core's internal order and the fixed-order
addition of the cluster's partials).
"""

import numpy as np
import pytest
import torch

from gpu_util import oracle_y, parity, sample_rows, to_device
from nvfp4_w4a4_quantized_gb300 import binding, synth
from oracle import quant_ref as q

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from nvfp4_w4a4_quantized_gb300 import build
    build.build()
    import oracle
    oracle.build()
    binding.svdq_read_device_status(clear=True)


def _run(x, ld, packed=False):
    xd = x.cuda()
    ldd = ld.cuda() if ld is not None else None
    M, K = x.shape
    act = torch.full((M, K // 2), 0xAA, dtype=torch.uint8, device="cuda")
    shape = (K // 64, M) if packed else (K // 16, M)
    dt = torch.int32 if packed else torch.uint8
    asc = torch.full(shape, -1 if packed else 0xAA, dtype=dt, device="cuda")
    la = None
    if ld is not None:
        la = torch.full((M, ld.shape[0]), float("nan"), dtype=torch.float32, device="cuda")
    binding.svdq_quantize_act(xd, ldd, act=act, ascales=asc, lora_act_in=la,
                              scales_packed=packed)
    torch.cuda.synchronize()
    code, site, block = binding.svdq_read_device_status(clear=True)
    assert code == 0, f"device status {code} at wait site {site}, CTA {block}"
    out_asc = asc.cpu().numpy()
    if packed:
        out_asc = out_asc.view(np.uint32)
    return act.cpu().numpy(), out_asc, (la.double().cpu().numpy() if la is not None else None)


def _check_la(la, x, ld, half):
    M, K = x.shape
    R = ld.shape[0]
    ref = q.lora_down(x, ld, M, K, R, half)
    mag = np.abs(q.decode_x(x, M, K, half)) @ np.abs(q.decode_x(ld, R, K, half)).T
    assert np.all(np.isfinite(la)), "unwritten lora_act_in element"
    bound = K * 2.0 ** -22 * mag + 1e-30
    err = np.abs(la - ref)
    assert np.all(err <= bound), float((err / bound).max())


def _case(M, K, R, half, seed, packed=False):
    d = synth.make_activations(M, K, R, seed, half=half)
    x, ld = d["x"], (d["lora_down"] if R else None)
    act, asc, la = _run(x, ld, packed)
    want_act, want_asc = q.quantize_act(x, M, K, half=half, packed=packed)
    np.testing.assert_array_equal(act, want_act)
    np.testing.assert_array_equal(asc, want_asc)
    if R:
        _check_la(la, x, ld, half)


@pytest.mark.parametrize("half", [False, True], ids=["bf16", "fp16"])
@pytest.mark.parametrize("R", [0, 16, 20, 32, 128])
def test_ragged_rows_several_tiles(R, half):
    # 272 rows = two full 128-row tiles and a 16-row tail; 10 K chunks
    _case(272, 640, R, half, seed=20 + R)


@pytest.mark.parametrize("M,K,want_splits", [(16, 12288, 8), (4096, 512, 4), (9728, 256, 2),
                                             (19456, 128, 1), (2432, 128, 2)])
def test_every_cluster_split(M, K, want_splits):
    plan = binding.svdq_quantize_query(M, K, 32)
    assert plan["splits"] == want_splits, plan
    _case(M, K, 32, False, seed=30)


@pytest.mark.parametrize("packed", [False, True], ids=["raw_scales", "packed_scales"])
def test_attention_projection_activations(packed):
    # x of the 4096 x 3072 x 3072 projection, R = 32, full tensors
    _case(4096, 3072, 32, False, seed=40, packed=packed)


def test_mlp_down_activations_sampled():
    # x of the 4096 x 3072 x 12288 projection (R = 128): codes and scales in
    # full, lora_act_in on sampled rows (the fp64 product of every row is slow)
    M, K, R = 4096, 12288, 128
    d = synth.make_activations(M, K, R, 41)
    act, asc, la = _run(d["x"], d["lora_down"])
    want_act, want_asc = q.quantize_act(d["x"], M, K)
    np.testing.assert_array_equal(act, want_act)
    np.testing.assert_array_equal(asc, want_asc)
    rows = np.array(sorted({0, 1, 127, 128, 2047, 4095} | set(range(3, 4096, 97))))
    _check_la(la[rows], d["x"][rows], d["lora_down"], False)


def test_edge_values():
    # the hand-worked groups, zero and huge and tiny groups, negative zeros,
    # subnormal x and exact E2M1 ties, in a 128-row tile with zero padding
    rows = []
    for line in open(__file__.replace("test_gpu_quant.py", "golden/quant_example.txt")):
        if line.startswith("#") or not line.strip():
            continue
        rows.append([float(v) for v in line.split("|")[1].split()])
    M, K = 128, 128
    x = torch.zeros(M, K)
    x[0, :64] = torch.tensor(sum(rows[0:4], []))
    x[1, :64] = torch.tensor(sum(rows[4:8], []))
    x[2, :64] = 60000.0                      # amax / 6 far beyond 448: saturated scale
    x[2, 64:] = torch.linspace(-3e4, 3e4, 64)
    x[3, :] = -0.0                           # negative zeros: +0 codes, zero scale
    x[4, :] = 2.0 ** -130                    # bf16 subnormals: zero scale
    x[5, :] = (torch.arange(K) % 16 - 8) * 0.25   # ties at every quarter
    x[6, :16] = 1e-3
    x[6, 16:32] = torch.tensor([6.0] + [0.25 * i for i in range(15)])
    xb = x.to(torch.bfloat16)
    act, asc, _ = _run(xb, None)
    want_act, want_asc = q.quantize_act(xb, M, K)
    np.testing.assert_array_equal(act, want_act)
    np.testing.assert_array_equal(asc, want_asc)


def test_same_bits_every_call():
    d = synth.make_activations(1024, 3072, 64, 42)
    a1 = _run(d["x"], d["lora_down"])
    a2 = _run(d["x"], d["lora_down"])
    for u, v in zip(a1, a2):
        assert np.array_equal(u, v)


def test_empty_and_rejected_calls():
    x = torch.zeros(0, 64, dtype=torch.bfloat16, device="cuda")
    act, asc, la = binding.svdq_quantize_act(x)
    assert act.shape == (0, 32)
    lib = binding.load()
    xb = torch.zeros(16, 64, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(16 * 64, dtype=torch.uint8, device="cuda")
    h = torch.cuda.current_stream().cuda_stream
    assert lib.svdq_quantize_act(xb.data_ptr(), None, 16, 64, 0, 0, 0, 0, out.data_ptr(),
                                 out.data_ptr() + 1, None, h) == binding.SVDQ_ERR_MISALIGNED
    assert lib.svdq_quantize_act(xb.data_ptr(), None, 16, 64, 4, 0, 0, 0, out.data_ptr(),
                                 out.data_ptr(), None, h) == binding.SVDQ_ERR_INVALID_ARG
    assert lib.svdq_quantize_act(xb.data_ptr(), None, 8, 64, 0, 0, 0, 0, out.data_ptr(),
                                 out.data_ptr(), None, h) == binding.SVDQ_ERR_UNSUPPORTED_SHAPE


@pytest.mark.parametrize("packed", [False, True], ids=["raw_scales", "packed_scales"])
def test_quantise_then_gemm(packed):
    # x -> svdq_quantize_act -> svdq_w4a4_gemm on the GPU, against the oracle's
    # quantiser, LoRA-down and operator on the CPU
    M, N, K, R = 512, 768, 1024, 32
    d = synth.make_activations(M, K, R, 43)
    w = synth.make_inputs(M, N, K, R, seed=44)
    dd = to_device(w)
    act, asc, la = binding.svdq_quantize_act(d["x"].cuda(), d["lora_down"].cuda(),
                                             scales_packed=packed)
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    binding.svdq_w4a4_gemm(act, dd["wgt"], asc, dd["wscales"], la, dd["lora_up"],
                           dd["wcscale"], dd["bias"], out,
                           options=dict(act_scales_packed=1) if packed else None)
    torch.cuda.synchronize()
    code, site, _ = binding.svdq_read_device_status(clear=True)
    assert code == 0, (code, site)
    ref_act, ref_asc = q.quantize_act(d["x"], M, K)
    ref_la = q.lora_down(d["x"], d["lora_down"], M, K, R).astype(np.float32)
    inp = dict(w, act=torch.from_numpy(ref_act), ascales=torch.from_numpy(ref_asc),
               lora_act_in=torch.from_numpy(ref_la))
    parity(out.double().cpu().numpy(), oracle_y(inp, M, N, K, R))


@pytest.mark.parametrize("half", [False, True], ids=["bf16", "fp16"])
@pytest.mark.parametrize("M,K,R", [(272, 640, 20), (4096, 3072, 32), (2432, 1024, 128),
                                   (19456, 128, 64)])
def test_lora_act_16bit_is_the_rounded_fp32_result(M, K, R, half):
    # the 16-bit LoRA-down output is the fp32 output rounded to nearest even
    # (same sum, same order: one CTA per tile and every cluster split)
    d = synth.make_activations(M, K, R, 50 + R, half=half)
    x, ld = d["x"].cuda(), d["lora_down"].cuda()
    _, _, la32 = binding.svdq_quantize_act(x, ld)
    _, _, la16 = binding.svdq_quantize_act(x, ld, lora_act_16bit=True)
    torch.cuda.synchronize()
    code, site, _ = binding.svdq_read_device_status(clear=True)
    assert code == 0, (code, site)
    assert la16.dtype == x.dtype
    assert torch.equal(la16, la32.to(x.dtype))


def test_layer_in_a_cuda_graph():
    # x -> svdq_quantize_act (packed scales, 16-bit LoRA activations) ->
    # svdq_w4a4_gemm_prepacked, captured once in a CUDA graph and replayed on new
    # x copied into the same buffer: every replay gives the eager calls' bits,
    # and sampled rows match the oracle's quantiser and operator
    M, N, K, R = 512, 768, 1024, 32
    w = synth.make_inputs(M, N, K, R, seed=70)
    dd = to_device(w)
    wpk, lup = binding.svdq_prepack_weights(dd["wscales"], dd["lora_up"], dd["wcscale"])
    ld = synth.make_activations(M, K, R, 71)["lora_down"]
    xs = [synth.make_activations(M, K, R, 72 + i)["x"] for i in range(3)]
    x_buf, ld_d = xs[0].cuda(), ld.cuda()
    act = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
    apk = torch.empty((K // 64, M), dtype=torch.int32, device="cuda")
    la = torch.empty((M, R), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    opts = dict(act_scales_packed=1, lora_act_16bit=1)

    def layer(stream):
        binding.svdq_quantize_act(x_buf, ld_d, act=act, ascales=apk, lora_act_in=la,
                                  scales_packed=True, lora_act_16bit=True, stream=stream)
        binding.svdq_w4a4_gemm_prepacked(act, dd["wgt"], apk, wpk, la, lup, dd["wcscale"],
                                         dd["bias"], out, stream=stream, options=opts)

    layer(torch.cuda.current_stream())  # the library's one-time set-up, outside the capture
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        layer(torch.cuda.current_stream())
    for i, x in enumerate(xs):
        x_buf.copy_(x)
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        code, site, _ = binding.svdq_read_device_status(clear=True)
        assert code == 0, f"device status {code} at wait site {site} (input {i})"
        y_graph = out.clone()
        out.fill_(float("nan"))
        layer(torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert torch.equal(y_graph, out), f"graph replay {i} differs from the eager calls"
        ref_act, ref_asc = q.quantize_act(x, M, K)
        ref_la = q.lora_down(x, ld, M, K, R)
        inp = dict(w, act=torch.from_numpy(ref_act), ascales=torch.from_numpy(ref_asc),
                   lora_act_in=torch.from_numpy(ref_la).to(torch.bfloat16).to(torch.float32))
        rows = np.array(sorted({0, 127, 128, 255, 256, 511} | set(range(5, M, 37))))
        parity(y_graph.double().cpu().numpy()[rows], oracle_y(inp, M, N, K, R, rows=rows))


@pytest.mark.parametrize("half", [False, True], ids=["bf16", "fp16"])
@pytest.mark.parametrize("M,N,K,R", [(272, 400, 640, 0), (272, 400, 640, 20), (512, 768, 1024, 32),
                                     (384, 512, 3072, 128)])
def test_linear_is_the_two_calls(M, N, K, R, half):
    # svdq_w4a4_linear (one call from 16-bit x) gives the bits of svdq_quantize_act
    # + svdq_w4a4_gemm_prepacked, and sampled rows match the oracle's quantiser
    # and operator
    h16 = torch.float16 if half else torch.bfloat16
    w = synth.make_inputs(M, N, K, R, seed=80 + R, half=half)
    a = synth.make_activations(M, K, R, 81 + R, half=half)
    dd = to_device(w)
    wpk, lup = binding.svdq_prepack_weights(dd["wscales"], dd["lora_up"] if R else None,
                                            dd["wcscale"])
    x, ld = a["x"].cuda(), (a["lora_down"].cuda() if R else None)
    out = torch.full((M, N), float("nan"), dtype=h16, device="cuda")
    binding.svdq_w4a4_linear(x, ld, dd["wgt"], wpk, lup if R else None, dd["wcscale"], dd["bias"],
                             out)
    la16 = R > 0 and R % 8 == 0
    act, apk, la = binding.svdq_quantize_act(x, ld, scales_packed=True, lora_act_16bit=la16)
    ref = torch.full((M, N), float("nan"), dtype=h16, device="cuda")
    binding.svdq_w4a4_gemm_prepacked(act, dd["wgt"], apk, wpk, la, lup if R else None,
                                     dd["wcscale"], dd["bias"], ref,
                                     options=dict(act_scales_packed=1, lora_act_16bit=int(la16),
                                                  io_dtype=int(half)))
    torch.cuda.synchronize()
    code, site, _ = binding.svdq_read_device_status(clear=True)
    assert code == 0, (code, site)
    assert torch.equal(out, ref)
    ref_act, ref_asc = q.quantize_act(a["x"], M, K, half=half)
    inp = dict(w, act=torch.from_numpy(ref_act), ascales=torch.from_numpy(ref_asc))
    if R:
        ref_la = torch.from_numpy(q.lora_down(a["x"], a["lora_down"], M, K, R, half))
        inp["lora_act_in"] = (ref_la.to(h16) if la16 else ref_la).to(torch.float32)
    else:
        inp["lora_act_in"] = None
        inp["lora_up"] = None
    rows = sample_rows(M, 24, seed=R)
    parity(out.double().cpu().numpy()[rows], oracle_y(inp, M, N, K, R, rows=rows))


def test_linear_rejects_a_small_workspace():
    M, N, K, R = 256, 256, 256, 32
    x = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    wgt = torch.zeros(N, K // 2, dtype=torch.uint8, device="cuda")
    wpk = torch.zeros(K // 64, N, dtype=torch.int32, device="cuda")
    lup = torch.zeros(N, R, dtype=torch.bfloat16, device="cuda")
    ld = torch.zeros(R, K, dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(binding.svdq_linear_workspace_size(M, K, R) - 256, dtype=torch.uint8,
                     device="cuda")
    rc = binding.svdq_w4a4_linear(x, ld, wgt, wpk, lup, None, None, out, workspace=ws,
                                  check=False)
    assert rc == binding.SVDQ_ERR_WORKSPACE


def test_linear_in_a_cuda_graph():
    # one svdq_w4a4_linear call captured in a CUDA graph and replayed on new x
    # copied into the same buffer: each replay gives the eager call's bits
    M, N, K, R = 512, 768, 1024, 40
    w = synth.make_inputs(M, N, K, R, seed=74)
    dd = to_device(w)
    wpk, lup = binding.svdq_prepack_weights(dd["wscales"], dd["lora_up"], dd["wcscale"])
    ld = synth.make_activations(M, K, R, 75)["lora_down"].cuda()
    xs = [synth.make_activations(M, K, R, 76 + i)["x"] for i in range(3)]
    x_buf = xs[0].cuda()
    ws = torch.empty(binding.svdq_linear_workspace_size(M, K, R), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")

    def layer(stream):
        binding.svdq_w4a4_linear(x_buf, ld, dd["wgt"], wpk, lup, dd["wcscale"], dd["bias"], out,
                                 workspace=ws, stream=stream)

    layer(torch.cuda.current_stream())  # the library's one-time set-up, outside the capture
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        layer(torch.cuda.current_stream())
    for i, x in enumerate(xs):
        x_buf.copy_(x)
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        code, site, _ = binding.svdq_read_device_status(clear=True)
        assert code == 0, (code, site, i)
        y_graph = out.clone()
        out.fill_(float("nan"))
        layer(torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert torch.equal(y_graph, out), f"graph replay {i} differs from the eager call"
