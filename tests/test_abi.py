"""The C-ABI library without a GPU: it loads, exports every symbol that
include/svdq.h declares, validates arguments on the host, and plans
launches (pipeline-depth solver, tensor-memory budget, persistent grid)."""

import ctypes
import os
import re
import subprocess

import pytest
import torch

from nvfp4_w4a4_quantized_gb300 import binding, build
from nvfp4_w4a4_quantized_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "svdq.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(svdq_\w+)\s*\(", text)))


def test_header_declares_the_binding_symbols():
    assert declared_functions() == sorted(binding.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (svdq_\w+)$", out, flags=re.M))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_status_strings(lib):
    for code in range(0, -13, -1):
        s = binding.status_string(code)
        assert s.startswith("SVDQ_")
    assert binding.status_string(-99) == "SVDQ_ERR_UNKNOWN"
    assert binding.svdq_version() == binding.ABI_VERSION


def test_abi_version_matches_header(lib):
    import re
    src = open(os.path.join(os.path.dirname(__file__), "..", "include", "svdq.h")).read()
    assert int(re.search(r"#define SVDQ_ABI_VERSION (\d+)", src).group(1)) == binding.ABI_VERSION
    assert "#define SVDQ_MAX_MN (1LL << 24)" in src and binding.SVDQ_MAX_MN == 1 << 24
    assert "#define SVDQ_MAX_K (1LL << 20)" in src and binding.SVDQ_MAX_K == 1 << 20
    assert "#define SVDQ_MAX_RANK 128" in src and binding.SVDQ_MAX_RANK == 128


# ---------------------------------------------------------------- validation
A = 1 << 20  # fake, 16-byte aligned addresses: validation never dereferences


def call(lib, M=256, N=256, K=256, R=32, ptrs=None, opts=None, prepacked=False):
    p = dict(act=A, wgt=A, ascales=A, wscales=A, la=A, lu=A, wc=A, bias=A, out=A)
    p.update(ptrs or {})
    args = [p["act"], p["wgt"], p["ascales"], p["wscales"], p["la"], p["lu"], p["wc"], p["bias"],
            p["out"], M, N, K, R]
    if prepacked:
        o = binding.SvdqOptions(**(opts or {}))
        return lib.svdq_w4a4_gemm_prepacked(*args, ctypes.byref(o) if opts else None, None)
    if opts is None:
        return lib.svdq_w4a4_gemm(*args, None)
    o = binding.SvdqOptions(**opts)
    return lib.svdq_w4a4_gemm_ex(*args, ctypes.byref(o), None)


@pytest.mark.parametrize("kw,expect", [
    (dict(ptrs=dict(act=None)), binding.SVDQ_ERR_INVALID_ARG),
    (dict(ptrs=dict(out=None)), binding.SVDQ_ERR_INVALID_ARG),
    (dict(ptrs=dict(la=None)), binding.SVDQ_ERR_INVALID_ARG),
    (dict(ptrs=dict(lu=None)), binding.SVDQ_ERR_INVALID_ARG),
    (dict(M=-16), binding.SVDQ_ERR_INVALID_ARG),
    (dict(K=0), binding.SVDQ_ERR_INVALID_ARG),
    (dict(R=-1), binding.SVDQ_ERR_INVALID_ARG),
    (dict(M=24), binding.SVDQ_ERR_UNSUPPORTED_SHAPE),
    (dict(N=40), binding.SVDQ_ERR_UNSUPPORTED_SHAPE),
    (dict(K=96), binding.SVDQ_ERR_UNSUPPORTED_SHAPE),
    (dict(R=129), binding.SVDQ_ERR_UNSUPPORTED_SHAPE),
    (dict(K=(1 << 20) + 64), binding.SVDQ_ERR_UNSUPPORTED_SHAPE),
    (dict(M=(1 << 24) + 16), binding.SVDQ_ERR_UNSUPPORTED_SHAPE),
    (dict(ptrs=dict(act=A + 8)), binding.SVDQ_ERR_MISALIGNED),
    (dict(ptrs=dict(wscales=A + 1)), binding.SVDQ_ERR_MISALIGNED),
    (dict(ptrs=dict(out=A + 2)), binding.SVDQ_ERR_MISALIGNED),
    (dict(ptrs=dict(bias=A + 2)), binding.SVDQ_ERR_MISALIGNED),
    (dict(opts=dict(tile_n=64)), binding.SVDQ_ERR_BAD_OPTION),
    (dict(opts=dict(stages=1)), binding.SVDQ_ERR_BAD_OPTION),
    (dict(opts=dict(stages=9)), binding.SVDQ_ERR_BAD_OPTION),
    (dict(opts=dict(debug_fault=2)), binding.SVDQ_ERR_BAD_OPTION),
    (dict(opts=dict(k_splits=9)), binding.SVDQ_ERR_BAD_OPTION),
    (dict(opts=dict(k_splits=-2)), binding.SVDQ_ERR_BAD_OPTION),
    (dict(opts=dict(act_scales_packed=2)), binding.SVDQ_ERR_BAD_OPTION),
    (dict(opts=dict(relaxed_order=2)), binding.SVDQ_ERR_BAD_OPTION),
    (dict(opts=dict(relaxed_order=-1)), binding.SVDQ_ERR_BAD_OPTION),
    (dict(opts=dict(io_dtype=2)), binding.SVDQ_ERR_BAD_OPTION),
    (dict(opts=dict(cta_group=3)), binding.SVDQ_ERR_BAD_OPTION),
    (dict(opts=dict(cta_group=2, tile_n=128)), binding.SVDQ_ERR_BAD_OPTION),
])
@pytest.mark.parametrize("prepacked", [False, True], ids=["per_call", "prepacked"])
def test_host_validation(lib, kw, expect, prepacked):
    assert call(lib, prepacked=prepacked, **kw) == expect


def prepack(lib, N=256, K=256, R=32, io=0, ptrs=None):
    p = dict(ws=A, lu=A, wc=A, wpk=A, lup=A)
    p.update(ptrs or {})
    return lib.svdq_prepack_weights(p["ws"], p["lu"], p["wc"], N, K, R, io, p["wpk"], p["lup"],
                                    None)


@pytest.mark.parametrize("kw,expect", [
    (dict(io=2), binding.SVDQ_ERR_BAD_OPTION),
    (dict(io=-1), binding.SVDQ_ERR_BAD_OPTION),
    (dict(N=-16), binding.SVDQ_ERR_INVALID_ARG),
    (dict(K=0), binding.SVDQ_ERR_INVALID_ARG),
    (dict(R=-1), binding.SVDQ_ERR_INVALID_ARG),
    (dict(N=40), binding.SVDQ_ERR_UNSUPPORTED_SHAPE),
    (dict(K=96), binding.SVDQ_ERR_UNSUPPORTED_SHAPE),
    (dict(R=129), binding.SVDQ_ERR_UNSUPPORTED_SHAPE),
    (dict(ptrs=dict(ws=None)), binding.SVDQ_ERR_INVALID_ARG),
    (dict(ptrs=dict(wpk=None)), binding.SVDQ_ERR_INVALID_ARG),
    (dict(ptrs=dict(lu=None)), binding.SVDQ_ERR_INVALID_ARG),
    (dict(ptrs=dict(lup=None)), binding.SVDQ_ERR_INVALID_ARG),
    (dict(ptrs=dict(ws=A + 8)), binding.SVDQ_ERR_MISALIGNED),
    (dict(ptrs=dict(lup=A + 2)), binding.SVDQ_ERR_MISALIGNED),
    (dict(ptrs=dict(wc=A + 4)), binding.SVDQ_ERR_MISALIGNED),
])
def test_prepack_host_validation(lib, kw, expect):
    assert prepack(lib, **kw) == expect


def test_prepack_empty_and_rank_zero(lib):
    assert prepack(lib, N=0) == binding.SVDQ_OK
    # R == 0 needs no LoRA pointers (N == 0 keeps it off the device)
    assert prepack(lib, N=0, R=0, ptrs=dict(lu=None, lup=None, wc=None)) == binding.SVDQ_OK


def test_rank_zero_needs_no_lora_pointers(lib):
    # R == 0 with NULL LoRA pointers passes validation; the empty M makes it a no-op
    assert call(lib, M=0, R=0, ptrs=dict(la=None, lu=None)) == binding.SVDQ_OK


def test_empty_product_is_a_no_op(lib):
    assert call(lib, M=0) == binding.SVDQ_OK
    assert call(lib, N=0) == binding.SVDQ_OK


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_no_device_is_reported(lib):
    assert call(lib) == binding.SVDQ_ERR_UNSUPPORTED_DEVICE
    assert call(lib, prepacked=True) == binding.SVDQ_ERR_UNSUPPORTED_DEVICE
    assert prepack(lib) == binding.SVDQ_ERR_UNSUPPORTED_DEVICE


# ---------------------------------------------------------------- planner
SMS = 152


@pytest.mark.parametrize("w", [synth.TINY, synth.ATTN_PROJ, synth.MLP_UP, synth.MLP_DOWN]
                         + synth.sweep_workloads(), ids=lambda w: w.name)
def test_plan_budgets(lib, w):
    plan = binding.svdq_query_plan(w.M, w.N, w.K, w.R, sm_count=SMS)
    assert plan["tmem_cols_used"] <= plan["tmem_cols"] == 512
    assert plan["smem_bytes"] <= 232448
    assert plan["num_acc_stage"] == (1 if plan["tile_n"] == 256 else 2)
    cg = plan["cta_group"]
    assert plan["tile_m"] == 128 * cg
    # a LoRA ring item (LA', LU', raw LA, wcscale, both operands split across
    # a pair) fits inside one stage, so LoRA never costs pipeline depth
    assert plan["lora_block_bytes"] <= plan["stage_bytes"]
    assert plan["lora_blocks"] == -(-w.R // 32)
    assert plan["k_blocks"] == -(-w.K // 256)
    assert plan["kblocks_per_stage"] in (1, 2)
    # pipeline depth: never silently clamped below 4 K blocks in flight
    assert plan["num_ab_stage"] * plan["kblocks_per_stage"] >= 4
    assert plan["num_ab_stage"] >= 2
    tiles = -(-w.M // plan["tile_m"]) * -(-w.N // plan["tile_n"])
    assert plan["num_tiles"] == tiles
    # balanced persistent grid: the rounds of the full grid on the fewest clusters
    rounds = -(-tiles // (SMS // cg))
    assert plan["grid"] == cg * -(-tiles // rounds)
    assert plan["grid"] <= SMS


@pytest.mark.parametrize("cg,tn", [(1, 128), (1, 256), (2, 256)])
def test_plan_each_tile_config(lib, cg, tn):
    p = binding.svdq_query_plan(4096, 3072, 3072, 32, options=dict(cta_group=cg, tile_n=tn),
                                sm_count=SMS)
    assert (p["cta_group"], p["tile_n"], p["tile_m"]) == (cg, tn, 128 * cg)
    # per-CTA stage, per K block: A rows 128 x 128 B, B rows (tile_n / cg) x 128 B,
    # raw scale boxes 16 x 128 and 16 x tile_n
    kbi = p["kblocks_per_stage"]
    assert kbi == 1
    assert p["stage_bytes"] == kbi * (128 * 128 + (tn // cg) * 128 + 16 * 128 + 16 * tn)
    assert p["num_ab_stage"] * kbi >= 3
    sf_cols = kbi * 4 * (4 + 4 * (tn // 128))
    assert p["smem_bytes"] + p["stage_bytes"] > 232448 or p["num_ab_stage"] == 8 or \
        p["tmem_cols_used"] + sf_cols > 512   # the solver took all it could


def test_plan_depth_independent_of_rank(lib):
    depths = {binding.svdq_query_plan(4096, 3072, 12288, R, sm_count=SMS)["num_ab_stage"]
              for R in (0, 16, 32, 64, 128)}
    assert len(depths) == 1


def test_plan_options(lib):
    p = binding.svdq_query_plan(4096, 3072, 3072, 32, options=dict(tile_n=128, stages=3,
                                                                  max_ctas=7), sm_count=SMS)
    assert (p["tile_n"], p["cta_group"], p["num_ab_stage"], p["grid"]) == (128, 1, 3, 7)
    p = binding.svdq_query_plan(4096, 3072, 3072, 32, options=dict(cta_group=2, max_ctas=7),
                                sm_count=SMS)
    assert p["grid"] == 6          # whole CTA pairs only
    with pytest.raises(binding.SvdqError):
        binding.svdq_query_plan(4096, 3072, 3072, 32, options=dict(tile_n=256, stages=8),
                                sm_count=SMS)
    # small problems fall back to single-CTA tiles
    assert binding.svdq_query_plan(128, 3072, 3072, 32, sm_count=SMS)["cta_group"] == 1


def test_lora_stage_bytes_match_the_pages_probe(lib):
    # "SVDQuant W4A4 on Blackwell" §7.4: 2-CTA, R=128, 16-bit LoRA operands,
    # mma tile (256, 128): per-CTA la_one = 32768 B and lu_one = 16384 B.
    tot, la, lu = binding.svdq_lora_stage_bytes(256, 128, 128, 2, 2)
    assert (la, lu, tot) == (32768, 16384, 49152)
    # single CTA: nothing is split
    assert binding.svdq_lora_stage_bytes(128, 256, 32, 2, 1)[1:] == (8192, 16384)
    with pytest.raises(binding.SvdqError):
        binding.svdq_lora_stage_bytes(255, 128, 128, 2, 2)


# ---------------------------------------------------------------- split-K planning
def test_split_plan_small_m_long_k(lib):
    # 256 x 3072 x 12288: 48 single-CTA 128x128 tiles fill under a third of
    # 152 SMs and 48 K blocks leave 16 per split
    plan = binding.svdq_query_plan(256, 3072, 12288, 128, options=dict(k_splits=-1),
                                   sm_count=SMS)
    assert (plan["cta_group"], plan["tile_n"]) == (1, 128)
    assert plan["k_splits"] == 3 and plan["num_units"] == 144 and plan["grid"] == 144
    slots = 48 * 2 * 1
    partial = slots * 128 * 128 * 4
    assert plan["workspace_bytes"] == partial + slots * 8 * 4  # one flag per epilogue warp
    assert binding.svdq_workspace_size(256, 3072, 12288, 128, sm_count=SMS) == \
        plan["workspace_bytes"]
    # the default plan (entry points without a workspace) never splits
    plain = binding.svdq_query_plan(256, 3072, 12288, 128, sm_count=SMS)
    assert plain["k_splits"] == 1 and plain["workspace_bytes"] == 0


@pytest.mark.parametrize("M,N,K", [(4096, 3072, 3072), (1024, 12288, 3072), (256, 256, 256),
                                   (256, 3072, 3072)])
def test_split_plan_declines(lib, M, N, K):
    # enough tiles for half the clusters, or fewer than 2 x 8 K blocks: no split
    plan = binding.svdq_query_plan(M, N, K, 32, options=dict(k_splits=-1), sm_count=SMS)
    assert plan["k_splits"] == 1 and plan["workspace_bytes"] == 0
    assert binding.svdq_workspace_size(M, N, K, 32, sm_count=SMS) == 0


def test_split_plan_forced_and_rejected(lib):
    plan = binding.svdq_query_plan(256, 384, 1024, 16, options=dict(k_splits=2, cta_group=1,
                                                                   tile_n=128), sm_count=SMS)
    assert plan["k_splits"] == 2 and plan["num_units"] == 2 * plan["num_tiles"]
    # more splits than K blocks, or more units than clusters: rejected
    with pytest.raises(binding.SvdqError) as e:
        binding.svdq_query_plan(256, 384, 512, 16, options=dict(k_splits=3), sm_count=SMS)
    assert e.value.status == binding.SVDQ_ERR_BAD_OPTION
    with pytest.raises(binding.SvdqError) as e:
        binding.svdq_query_plan(4096, 3072, 3072, 32, options=dict(k_splits=2), sm_count=SMS)
    assert e.value.status == binding.SVDQ_ERR_BAD_OPTION


@pytest.mark.parametrize("args,expect", [
    ((A, 40, 256, A), binding.SVDQ_ERR_UNSUPPORTED_SHAPE),
    ((A, 256, 96, A), binding.SVDQ_ERR_UNSUPPORTED_SHAPE),
    ((A, -16, 256, A), binding.SVDQ_ERR_INVALID_ARG),
    ((None, 256, 256, A), binding.SVDQ_ERR_INVALID_ARG),
    ((A, 256, 256, None), binding.SVDQ_ERR_INVALID_ARG),
    ((A + 4, 256, 256, A), binding.SVDQ_ERR_MISALIGNED),
    ((A, 0, 256, A), binding.SVDQ_OK),
])
def test_pack_scales_host_validation(lib, args, expect):
    assert lib.svdq_pack_scales(*args, None) == expect


@pytest.mark.parametrize("M,N", [(256, 256), (1024, 3072), (4096, 3072), (4096, 12288),
                                 (16384, 12288), (2816, 2816), (4352, 3840)])
def test_plan_balanced_grid(lib, M, N):
    # the full grid's number of rounds, on the fewest clusters that keep it
    plan = binding.svdq_query_plan(M, N, 3072, 32, options=dict(cta_group=2), sm_count=SMS)
    units, cg = plan["num_units"], plan["cta_group"]
    clusters = plan["grid"] // cg
    full = min(units, SMS // cg)
    rounds = -(-units // full)
    assert -(-units // clusters) == rounds
    assert clusters == 1 or -(-units // (clusters - 1)) > rounds


@pytest.mark.parametrize("args,expect", [
    ((A, None, 0, 64, 0, 0, 0, 0, A, A, None), binding.SVDQ_OK),
    ((None, None, 0, 64, 8, 0, 0, 0, None, None, None), binding.SVDQ_OK),
    ((A, None, 40, 64, 0, 0, 0, 0, A, A, None), binding.SVDQ_ERR_UNSUPPORTED_SHAPE),
    ((A, None, 32, 96, 0, 0, 0, 0, A, A, None), binding.SVDQ_ERR_UNSUPPORTED_SHAPE),
    ((A, A, 32, 64, 129, 0, 0, 0, A, A, A), binding.SVDQ_ERR_UNSUPPORTED_SHAPE),
    ((A, None, -16, 64, 0, 0, 0, 0, A, A, None), binding.SVDQ_ERR_INVALID_ARG),
    ((A, None, 32, 0, 0, 0, 0, 0, A, A, None), binding.SVDQ_ERR_INVALID_ARG),
    ((None, None, 32, 64, 0, 0, 0, 0, A, A, None), binding.SVDQ_ERR_INVALID_ARG),
    ((A, None, 32, 64, 0, 0, 0, 0, None, A, None), binding.SVDQ_ERR_INVALID_ARG),
    ((A, None, 32, 64, 8, 0, 0, 0, A, A, A), binding.SVDQ_ERR_INVALID_ARG),
    ((A, A, 32, 64, 8, 0, 0, 0, A, A, None), binding.SVDQ_ERR_INVALID_ARG),
    ((A, None, 32, 64, 0, 2, 0, 0, A, A, None), binding.SVDQ_ERR_BAD_OPTION),
    ((A, None, 32, 64, 0, 0, 2, 0, A, A, None), binding.SVDQ_ERR_BAD_OPTION),
    ((A, None, 32, 64, 0, 0, 0, 2, A, A, None), binding.SVDQ_ERR_BAD_OPTION),
    ((A + 8, None, 32, 64, 0, 0, 0, 0, A, A, None), binding.SVDQ_ERR_MISALIGNED),
    ((A, A + 2, 32, 64, 8, 0, 0, 0, A, A, A), binding.SVDQ_ERR_MISALIGNED),
])
def test_quantize_host_validation(lib, args, expect):
    # rejected before any device call (the addresses are fake); the one valid
    # call is empty (M = 0) and launches nothing
    assert lib.svdq_quantize_act(*args, None) == expect


@pytest.mark.parametrize("M,K,R,splits", [(16, 12288, 32, 8), (256, 3072, 32, 8),
                                          (1024, 3072, 32, 8), (4096, 3072, 32, 4),
                                          (4096, 12288, 128, 4), (9728, 3072, 16, 2),
                                          (16384, 3072, 32, 1), (65536, 3072, 128, 1),
                                          (4096, 64, 32, 1), (4096, 128, 0, 2)])
def test_quantize_plan(lib, M, K, R, splits):
    plan = binding.svdq_quantize_query(M, K, R, sm_count=SMS)
    tiles = -(-M // 128)
    assert plan["splits"] == splits
    assert plan["grid"] == tiles * splits
    # a split never leaves a CTA without K chunks, and the grid fits the SMs when split
    assert splits <= K // 64 and (splits == 1 or plan["grid"] <= SMS)
    assert 3 <= plan["stages"] <= 10
    r16 = -(-R // 16) * 16
    stage = 128 * 128 + 128 * r16
    # the cluster's partials reuse the stages
    assert plan["stages"] * stage >= 128 * (r16 + 4) * 4
    assert plan["smem_bytes"] >= plan["stages"] * stage
    assert plan["smem_bytes"] <= 232448


@pytest.mark.parametrize("M,K,R", [(0, 64, 0), (16, 64, 0), (4096, 3072, 32), (4096, 12288, 128),
                                   (272, 640, 20), (16, 128, 8)])
def test_linear_workspace_size(lib, M, K, R):
    # act [M][K/2], scale words [K/64][M], lora_act_in [M][R] (16-bit when R % 8 == 0,
    # else fp32), each padded to 256 bytes
    pad = lambda b: -(-b // 256) * 256
    la = 0 if R == 0 else M * R * (2 if R % 8 == 0 else 4)
    assert binding.svdq_linear_workspace_size(M, K, R) == pad(M * K // 2) + pad(M * K // 16) + pad(la)


@pytest.mark.parametrize("M,K,R,expect", [(-16, 64, 0, binding.SVDQ_ERR_INVALID_ARG),
                                          (16, 0, 0, binding.SVDQ_ERR_INVALID_ARG),
                                          (24, 64, 0, binding.SVDQ_ERR_UNSUPPORTED_SHAPE),
                                          (16, 96, 0, binding.SVDQ_ERR_UNSUPPORTED_SHAPE),
                                          (16, 64, 129, binding.SVDQ_ERR_UNSUPPORTED_SHAPE)])
def test_linear_workspace_size_rejects(lib, M, K, R, expect):
    assert lib.svdq_linear_workspace_size(M, K, R) == expect


@pytest.mark.parametrize("N,ws_off,ws_bytes,expect", [
    (64, 0, 1024, binding.SVDQ_ERR_WORKSPACE),    # too small
    (64, 16, 1 << 20, binding.SVDQ_ERR_WORKSPACE),  # not 256-byte aligned
    (72, 0, 1 << 20, binding.SVDQ_ERR_UNSUPPORTED_SHAPE),
    (-16, 0, 1 << 20, binding.SVDQ_ERR_INVALID_ARG),
])
def test_linear_host_validation(lib, N, ws_off, ws_bytes, expect):
    # rejected before any device call (the addresses are fake)
    M, K, R = 32, 128, 0
    rc = lib.svdq_w4a4_linear(A, None, A, A, None, None, None, A, M, N, K, R, None, A + ws_off,
                              ws_bytes, None)
    assert rc == expect
