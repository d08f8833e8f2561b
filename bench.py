"""Throughput of the W4A4 NVFP4 + LoRA linear operator on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--dense] [--fp16] [--prepacked] [--split]
                    [--packed-scales] [--relaxed-order]

One step is one operator call (the whole path: scale relayout, LoRA operand
prep, LoRA + block-scaled MMAs, fused affine epilogue) over one synthetic
input batch.  The default workload is the 4096 x 3072 x 3072, R=32
attention-projection shape.  Prints one JSON line (rank 0).

TFLOPS counts 2MNK + 2MNR.  Device time comes from CUDA events around each
launch on the launching stream, with L2 flushed (a 256 MiB memset, outside
the events) before every timed launch.  `e2e` times the same call through
the public API with every step's inputs copied from pinned host memory and
its result copied back inside the timed region, steps pipelined over three
streams as a serving loop runs them (`serial_value`: one step at a time).  `--impl reference` times the
CPU oracle on bounded row samples of the same workload.  `--dense` runs the
calibration variant of the workload: the same shape through the same kernel
with R = 0 and no wcscale / bias, so the difference to the default run is
the cost of the LoRA term and the affine epilogue.  `--fp16` runs the fp16
input/output variant (lora_up, wcscale, bias and y in IEEE fp16).
`--prepacked` prepacks the weights once before timing (packed scale words,
LU' = LU / wcscale, as at weight-load time) and times the prepacked call.
`--packed-scales` additionally hands the activation scales over in the
kernel's word layout (as an activation quantiser could write them; packed
once before timing) and implies `--prepacked`.
`--split` times the split-K entry point (workspace allocated once, before
timing; the planner decides the split, e.g. on mlp_down_256x3072x12288_r128).
Calls are bit-reproducible by default (the MMA issuers take turns);
`--relaxed-order` times svdq_options_t.relaxed_order = 1 instead.
A default run (no route flag) also records, under `routes`, the prepacked,
prepacked + packed-scale, relaxed-order and quantiser-format (packed scales +
16-bit LoRA activations, `lora_act_16bit`) routes of the same workload, timed
the same way (flushed L2, per-launch events, 10 launches each), and under
`per_shape` every benchmark workload timed the same way: the tiny case, the
attention projection, MLP-up and MLP-down, each on the default route, the
dense calibration variant (R = 0, no wcscale / bias), the prepacked +
packed-scale route and that route with 16-bit LoRA activations, and the
24-case token-count sweep (default route, plus
the split-K entry point where the planner splits); then the activation
quantiser on the production activations (GB/s against the measured HBM copy
bandwidth) and the whole layer from 16-bit activations (svdq_w4a4_linear:
quantiser with packed scales + prepacked operator, in one event pair).  The headline `value` is
the attention projection, the configuration the metric is quoted on.
`--no-per-shape` skips that section.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

NOMINAL_FP4_OVER_BF16 = 13.5 / 2.25      # dense fp4 / bf16 tensor throughput, nominal
FALLBACK_BF16_TFLOPS = 1900.0
METRIC_PEAK_TFLOPS = 10000.0           # the dense NVFP4 peak the metric is quoted against
L2_FLUSH_BYTES = 256 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="attn_proj_4096x3072x3072_r32")
    ap.add_argument("--dense", action="store_true",
                    help="calibration variant: R = 0, no wcscale, no bias")
    ap.add_argument("--fp16", action="store_true",
                    help="fp16 input/output variant (lora_up, wcscale, bias, y in fp16)")
    ap.add_argument("--prepacked", action="store_true",
                    help="weights prepacked once (svdq_prepack_weights); time the prepacked call")
    ap.add_argument("--packed-scales", action="store_true",
                    help="activation scales in the word layout (implies --prepacked)")
    ap.add_argument("--split", action="store_true",
                    help="time svdq_w4a4_gemm_split (planner-chosen split-K)")
    ap.add_argument("--relaxed-order", action="store_true",
                    help="relaxed_order = 1: MMA issue order free, output bits may vary")
    ap.add_argument("--tile-n", type=int, default=0)
    ap.add_argument("--stages", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-per-shape", action="store_true",
                    help="skip the per-shape section of a default run")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def _code_only(src: str) -> str:
    """C++ source without comments and with whitespace collapsed (string
    literals in these files hold no comment markers)."""
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def kernel_source_hash() -> str:
    """Identifies the kernel code the committed ncu counters were taken on;
    comment edits do not change it."""
    h = hashlib.sha256()
    for rel in ("nvfp4_w4a4_quantized_gb300/csrc/svdq_kernel.cuh",
                "nvfp4_w4a4_quantized_gb300/csrc/ptx.cuh",
                "nvfp4_w4a4_quantized_gb300/csrc/svdq_api.cu"):
        with open(os.path.join(ROOT, rel)) as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def committed_traffic(workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        ent = rec.get(workload)
        if ent and ent.get("kernel_source_hash") == kernel_source_hash():
            return float(ent["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi SM clock / throttle sampling during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"svdq_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            # wait for the first sample, so that sampling covers the warm-up
            # and timed steps that follow
            t0 = time.time()
            while time.time() - t0 < 3.0 and os.path.getsize(self.path) == 0:
                time.sleep(0.05)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None:
            return None
        try:
            rows = [ln.split(",") for ln in open(self.path).read().strip().splitlines()]
        except Exception:
            return None
        sm, mx, reasons = [], 0.0, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 7:
                continue
            try:
                sm.append(float(r[0]))
                mx = max(mx, float(r[1]))
            except ValueError:
                continue
            for nm, v in zip(names, r[3:7]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def max_over_ranks(x: float, dist=None, device="cpu") -> float:
    """The largest per-rank value over all ranks of the process group (the
    job's step time is its slowest rank's); `x` itself without a group."""
    if dist is None:
        return float(x)
    import torch

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank: float, world: int, ms: float) -> float:
    """Whole-job throughput: every rank runs its own full problem (weak
    scaling), so the job does world x the work in the slowest rank's time."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


def workload_inputs(synth, w, dense: bool, half: bool = False):
    """The workload's seeded inputs; the dense calibration variant drops
    wcscale and bias (the operator then uses 1 and 0) and has R = 0; the fp16
    variant draws the same values rounded to fp16."""
    inp = synth.make_inputs(w.M, w.N, w.K, w.R, w.seed, half=half)
    if dense:
        inp.pop("wcscale")
        inp.pop("bias")
    return inp


def oracle_sample(w, inp, target_s=12.0, max_rows=None):
    """Time the oracle on a bounded row sample; returns (tflops, rows, seconds, threads)."""
    import numpy as np

    import oracle

    oracle.build()
    rows_all = np.arange(w.M, dtype=np.int64)
    n = 8
    t = 0.0
    while True:
        rows = rows_all[:n]
        t0 = time.perf_counter()
        oracle.forward(inp, w.M, w.N, w.K, w.R, rows=rows)
        t = time.perf_counter() - t0
        if t >= target_s or n >= (max_rows or w.M):
            break
        n = min(max_rows or w.M, max(n + 1, int(n * min(8.0, 1.2 * target_s / max(t, 1e-3)))))
    flops = 2.0 * n * w.N * (w.K + w.R)
    return flops / t / 1e12, n, t, oracle.num_threads()


def run_reference(args, w, rank):
    if rank != 0:
        return
    from nvfp4_w4a4_quantized_gb300 import synth

    inp = workload_inputs(synth, w, args.dense, args.fp16)
    per_step_target = max(1.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    _, rows, _, threads = oracle_sample(w, inp, target_s=per_step_target)
    import numpy as np

    import oracle

    sel = np.arange(rows, dtype=np.int64)
    for _ in range(args.warmup):
        oracle.forward(inp, w.M, w.N, w.K, w.R, rows=sel[: max(1, rows // 4)])
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.forward(inp, w.M, w.N, w.K, w.R, rows=sel)
        times.append(time.perf_counter() - t0)
    t = statistics.mean(times)
    flops = 2.0 * rows * w.N * (w.K + w.R)
    val = flops / t / 1e12
    line = {
        "impl": "reference", "metric": "W4A4+LoRA GEMM TFLOPS (2MNK+2MNR)", "value": val,
        "unit": "TFLOPS", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "R": w.R,
                   "parallelism": "single process, OpenMP over output rows"},
        "cpu_baseline": {"value": val, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
                         "sample": f"first {rows} of {w.M} output rows per step (all N columns)"},
        "e2e": {"value": val, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def time_flushed(call, flush, stream, n_warm, n_timed, torch, dev):
    """Per-launch CUDA-event times (ms) of `call`, with the L2 flushed by a
    memset outside each event pair."""
    for _ in range(n_warm):
        flush.zero_()
        call()
    t = []
    for _ in range(n_timed):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        t.append(e0.elapsed_time(e1))
    return t


def shape_entry(flops, ms, fp4_peak, plan=None):
    mean = statistics.mean(ms)
    tf = flops / (mean * 1e-3) / 1e12
    e = {"ms_mean": mean, "ms_median": statistics.median(ms), "ms_min": min(ms),
         "launches": len(ms), "tflops": tf, "mfu_vs_10pf": tf / METRIC_PEAK_TFLOPS,
         "frac": tf / fp4_peak}
    if plan is not None:
        e["plan"] = {"tile": [plan["tile_m"], plan["tile_n"]], "stages": plan["num_ab_stage"],
                     "grid": plan["grid"], "k_splits": plan["k_splits"]}
    return e


def run_per_shape(pkg, synth, torch, dev, stream, flush, fp4_peak):
    """Every benchmark workload on one GPU, timed like the headline figure
    (L2 flushed before each launch, one event pair per launch)."""
    res = {}
    prod = [synth.TINY, synth.ATTN_PROJ, synth.MLP_UP, synth.MLP_DOWN]
    for w in prod:
        inp = synth.make_workload_inputs(w)
        d = {k: v.to(dev) for k, v in inp.items()}
        out = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=dev)
        plan = pkg.svdq_query_plan(w.M, w.N, w.K, w.R)

        def call(dd=d, r=w.R, wc=True):
            pkg.svdq_w4a4_gemm(dd["act"], dd["wgt"], dd["ascales"], dd["wscales"],
                               dd["lora_act_in"] if r else None, dd["lora_up"] if r else None,
                               dd["wcscale"] if wc else None, dd["bias"] if wc else None, out,
                               stream=stream)
        e = shape_entry(float(w.flops), time_flushed(call, flush, stream, 3, 10, torch, dev),
                        fp4_peak, plan)
        e.update({"M": w.M, "N": w.N, "K": w.K, "R": w.R})
        # dense calibration: the same shape and kernel, R = 0, no wcscale / bias
        dense_flops = 2.0 * w.M * w.N * w.K
        e["dense"] = shape_entry(dense_flops, time_flushed(lambda: call(r=0, wc=False), flush,
                                                           stream, 3, 10, torch, dev), fp4_peak)
        # weights prepacked once, activation scales in the word layout
        wpk, lup = pkg.svdq_prepack_weights(d["wscales"], d["lora_up"], d["wcscale"])
        apk = pkg.svdq_pack_scales(d["ascales"])
        torch.cuda.synchronize(dev)
        o2 = dict(act_scales_packed=1)

        def call_pk():
            pkg.svdq_w4a4_gemm_prepacked(d["act"], d["wgt"], apk, wpk, d["lora_act_in"], lup,
                                         d["wcscale"], d["bias"], out, stream=stream, options=o2)
        e["prepacked_packed_scales"] = shape_entry(
            float(w.flops), time_flushed(call_pk, flush, stream, 3, 10, torch, dev), fp4_peak)
        # ... and the quantiser's formats: packed scales and 16-bit LA
        la16 = d["lora_act_in"].to(torch.bfloat16)
        o3 = dict(act_scales_packed=1, lora_act_16bit=1)

        def call_q():
            pkg.svdq_w4a4_gemm_prepacked(d["act"], d["wgt"], apk, wpk, la16, lup, d["wcscale"],
                                         d["bias"], out, stream=stream, options=o3)
        e["prepacked_packed_scales_lora16"] = shape_entry(
            float(w.flops), time_flushed(call_q, flush, stream, 3, 10, torch, dev), fp4_peak)
        res[w.name] = e
        del d, out, wpk, lup, apk
    sweep = []
    for w in synth.sweep_workloads():
        inp = synth.make_workload_inputs(w)
        d = {k: v.to(dev) for k, v in inp.items()}
        out = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=dev)
        plan = pkg.svdq_query_plan(w.M, w.N, w.K, w.R)

        def call(dd=d):
            pkg.svdq_w4a4_gemm(dd["act"], dd["wgt"], dd["ascales"], dd["wscales"],
                               dd["lora_act_in"], dd["lora_up"], dd["wcscale"], dd["bias"], out,
                               stream=stream)
        e = shape_entry(float(w.flops), time_flushed(call, flush, stream, 2, 5, torch, dev),
                        fp4_peak, plan)
        e.update({"name": w.name, "M": w.M, "N": w.N, "K": w.K, "R": w.R})
        wsz = pkg.svdq_workspace_size(w.M, w.N, w.K, w.R, options=dict(k_splits=-1))
        if wsz > 0:
            ws = torch.zeros(wsz, dtype=torch.uint8, device=dev)
            splan = pkg.svdq_query_plan(w.M, w.N, w.K, w.R, options=dict(k_splits=-1))

            def call_split(dd=d):
                pkg.svdq_w4a4_gemm_split(dd["act"], dd["wgt"], dd["ascales"], dd["wscales"],
                                         dd["lora_act_in"], dd["lora_up"], dd["wcscale"],
                                         dd["bias"], out, ws, stream=stream,
                                         options=dict(k_splits=-1))
            e["split"] = shape_entry(float(w.flops), time_flushed(call_split, flush, stream, 2, 5,
                                                                  torch, dev), fp4_peak, splan)
            del ws
        sweep.append(e)
        del d, out
    tfs = sorted(max(s["tflops"], s.get("split", {}).get("tflops", 0.0)) for s in sweep)
    res["sweep"] = {"cases": sweep, "tflops_min": tfs[0], "tflops_median": statistics.median(tfs),
                    "tflops_max": tfs[-1],
                    "how": "svdq_w4a4_gemm per case (and svdq_w4a4_gemm_split where the planner "
                           "splits; the summary takes the faster), 2 warm-up + 5 timed flushed "
                           "launches"}
    res.update(run_quantize_shapes(pkg, synth, torch, dev, stream, flush, fp4_peak))
    code, site, _ = pkg.svdq_read_device_status(clear=True)
    if code != 0:
        raise RuntimeError(f"device status {code} at wait site {site} in the per-shape runs")
    return res


def quant_bytes(M, K, R):
    """Algorithmic HBM bytes of one quantiser call: x and lora_down read once,
    codes, scales and lora_act_in written once."""
    return 2 * M * K + 2 * R * K + M * K // 2 + M * K // 16 + 4 * M * R


def run_quantize_shapes(pkg, synth, torch, dev, stream, flush, fp4_peak):
    """The activation quantiser on the production activations (HBM-bound:
    GB/s against the measured copy bandwidth), and the whole layer from 16-bit
    activations: quantiser (packed scales) + prepacked operator, one event pair."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            hbm, hbm_src = float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        hbm, hbm_src = 6800.0, "fallback"
    quant = {}
    for name, M, K, R in (("x_4096x3072_r32", 4096, 3072, 32),
                          ("x_4096x12288_r128", 4096, 12288, 128)):
        a = synth.make_activations(M, K, R, seed=7)
        x, ld = a["x"].to(dev), a["lora_down"].to(dev)
        nbytes = quant_bytes(M, K, R)
        e = {"M": M, "K": K, "R": R, "bytes": nbytes, "plan": pkg.svdq_quantize_query(M, K, R)}
        for packed in (False, True):
            outs = pkg.svdq_quantize_act(x, ld, scales_packed=packed)
            ms = time_flushed(lambda: pkg.svdq_quantize_act(x, ld, *outs, scales_packed=packed,
                                                            stream=stream),
                              flush, stream, 3, 10, torch, dev)
            mean = statistics.mean(ms)
            gbs = nbytes / (mean * 1e-3) / 1e9
            e["packed_scales" if packed else "raw_scales"] = {
                "ms_mean": mean, "ms_median": statistics.median(ms), "ms_min": min(ms),
                "gbs": gbs, "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm,
                                         "unit": "GB/s", "frac": gbs / hbm,
                                         "peak_source": f"{hbm_src} copy bandwidth"}}
            del outs
        quant[name] = e
        del x, ld
    layer = {}
    for w in (synth.ATTN_PROJ, synth.MLP_UP, synth.MLP_DOWN):
        inp = synth.make_workload_inputs(w)
        d = {k: v.to(dev) for k, v in inp.items()}
        a = synth.make_activations(w.M, w.K, w.R, seed=w.seed + 100)
        x, ld = a["x"].to(dev), a["lora_down"].to(dev)
        wpk, lup = pkg.svdq_prepack_weights(d["wscales"], d["lora_up"], d["wcscale"])
        ws = torch.empty(pkg.svdq_linear_workspace_size(w.M, w.K, w.R), dtype=torch.uint8,
                         device=dev)
        out = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=dev)

        def call_layer():
            pkg.svdq_w4a4_linear(x, ld, d["wgt"], wpk, lup, d["wcscale"], d["bias"], out,
                                 workspace=ws, stream=stream)
        e = shape_entry(float(w.flops), time_flushed(call_layer, flush, stream, 3, 10, torch,
                                                     dev), fp4_peak)
        e["how"] = ("svdq_w4a4_linear: svdq_quantize_act (packed scales, 16-bit LA) + "
                    "svdq_w4a4_gemm_prepacked (act_scales_packed, lora_act_16bit), one event "
                    "pair; tflops counts the operator's 2MNK + 2MNR")
        layer[w.name] = e
        del d, x, ld, wpk, lup, ws, out
    return {"quantize": quant, "layer_from_16bit_x": layer}


def run_ours(args, w, rank, world, local_rank):
    import torch

    import nvfp4_w4a4_quantized_gb300 as pkg
    from nvfp4_w4a4_quantized_gb300 import build, synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    build.build()
    pkg.load()
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if dist is not None:
            dist.barrier()

    inp = workload_inputs(synth, w, args.dense, args.fp16)
    d = {k: v.to(dev) for k, v in inp.items()}
    if args.packed_scales:
        args.prepacked = True
    if args.prepacked:
        # once per weight load, outside every timed region
        wpk, lup = pkg.svdq_prepack_weights(d["wscales"], d["lora_up"] if w.R else None,
                                            d.get("wcscale"))
        d = dict(d, wscales=wpk, lora_up=lup)
        if args.packed_scales:
            d["ascales"] = pkg.svdq_pack_scales(d["ascales"])
        torch.cuda.synchronize(dev)
    # what the end-to-end call copies from the host each step (the packed
    # weights when prepacked)
    host_src = {k: v.cpu() for k, v in d.items() if v is not None} if args.prepacked else inp
    gemm = pkg.svdq_w4a4_gemm_prepacked if args.prepacked else pkg.svdq_w4a4_gemm
    if args.split:
        wsz = pkg.svdq_workspace_size(w.M, w.N, w.K, w.R,
                                      options=dict(io_dtype=1 if args.fp16 else 0))
        workspace = torch.zeros(max(wsz, 256), dtype=torch.uint8, device=dev)

        def gemm(*a, options=None, **kw):
            return pkg.svdq_w4a4_gemm_split(*a, workspace, options=options,
                                            weights_prepacked=args.prepacked, **kw)
    out_dtype = torch.float16 if args.fp16 else torch.bfloat16
    out = torch.empty((w.M, w.N), dtype=out_dtype, device=dev)
    opts = dict(tile_n=args.tile_n, stages=args.stages,
                act_scales_packed=1 if args.packed_scales else 0,
                relaxed_order=1 if args.relaxed_order else 0)
    plan = pkg.svdq_query_plan(w.M, w.N, w.K, w.R,
                               options=dict(opts, k_splits=-1) if args.split else opts)
    stream = torch.cuda.current_stream(dev)

    def step(o=out, dd=d, s=None):
        gemm(dd["act"], dd["wgt"], dd["ascales"], dd["wscales"], dd.get("lora_act_in"),
             dd.get("lora_up"), dd.get("wcscale"), dd.get("bias"), o,
             stream=stream if s is None else s, options=opts)

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local_rank) as clk:
        # warm-up right before the timed steps: an idle GPU lowers its clock,
        # and the sampler's start-up leaves it idle for a moment
        for _ in range(max(3, args.warmup)):
            flush.zero_()
            step()
        torch.cuda.synchronize(dev)
        code, site, _ = pkg.svdq_read_device_status(clear=True)
        if code != 0:
            raise RuntimeError(f"device status {code} at wait site {site} during warm-up")
        barrier()
        torch.cuda.synchronize(dev)
        t_wall0 = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        t_wall = time.perf_counter() - t_wall0
    ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms_mean = max_over_ranks(statistics.mean(ms), dist, dev)
    code, site, _ = pkg.svdq_read_device_status(clear=True)
    if code != 0:
        raise RuntimeError(f"device status {code} at wait site {site} in the timed region")

    # secondary: hot L2, a CUDA graph of 20 back-to-back launches (per-launch mean)
    hot = None
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=torch.cuda.Stream(dev)):
            cap = torch.cuda.current_stream(dev)
            for _ in range(20):
                gemm(d["act"], d["wgt"], d["ascales"], d["wscales"], d.get("lora_act_in"),
                     d.get("lora_up"), d.get("wcscale"), d.get("bias"), out, stream=cap,
                     options=opts)
        g.replay()
        torch.cuda.synchronize(dev)
        h0, h1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        h0.record(stream)
        for _ in range(5):
            g.replay()
        h1.record(stream)
        torch.cuda.synchronize(dev)
        hot_ms = h0.elapsed_time(h1) / 100.0
        hot = {"ms_per_launch": hot_ms, "value": job_tflops(float(w.flops), world, hot_ms),
               "unit": "TFLOPS", "how": "CUDA graph of 20 launches, replayed 5x, L2 not flushed"}
    except Exception as exc:  # capture is optional; report why it was skipped
        hot = {"skipped": f"{type(exc).__name__}: {exc}"[:200]}
    code, site, _ = pkg.svdq_read_device_status(clear=True)
    if code != 0:
        raise RuntimeError(f"device status {code} at wait site {site} in the hot-L2 graph")

    # secondary: back-to-back launches (no flush kernel between them) over
    # rotating input sets whose total is over twice the L2 size, one event pair
    b2b = None
    try:
        per_set = sum(v.numel() * v.element_size() for v in d.values() if v is not None)
        per_set += out.numel() * out.element_size()
        nsets = max(2, -(-(2 * L2_FLUSH_BYTES) // per_set))
        if nsets * per_set <= (8 << 30):
            sets = [({k: (v.clone() if v is not None else None) for k, v in d.items()},
                     torch.empty_like(out)) for _ in range(nsets)]
            for dd_, oo_ in sets:
                step(oo_, dd_)
            torch.cuda.synchronize(dev)
            b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            nb = max(args.steps, 2 * nsets)
            b0.record(stream)
            for i in range(nb):
                step(sets[i % nsets][1], sets[i % nsets][0])
            b1.record(stream)
            torch.cuda.synchronize(dev)
            b_ms = b0.elapsed_time(b1) / nb
            b2b = {"ms_per_launch": b_ms, "value": job_tflops(float(w.flops), world, b_ms),
                   "unit": "TFLOPS",
                   "how": f"{nb} launches back to back over {nsets} input sets "
                          f"({nsets * per_set / 2**20:.0f} MiB > 2x L2), one event pair"}
            del sets
    except Exception as exc:
        b2b = {"skipped": f"{type(exc).__name__}: {exc}"[:200]}
    code, site, _ = pkg.svdq_read_device_status(clear=True)
    if code != 0:
        raise RuntimeError(f"device status {code} at wait site {site} in the back-to-back run")

    # secondary: the same workload through the other routes of the same operator
    # (weights prepacked once, activation scales in the word layout, relaxed
    # issue order), timed like the primary figure: L2 flushed, one event pair
    # per launch, mean of 10 after 3 warm-up launches.  Default runs only.
    routes = None
    plain = not (args.dense or args.fp16 or args.prepacked or args.split or args.packed_scales
                 or args.relaxed_order)
    if plain:
        routes = {}
        try:
            wpk, lup = pkg.svdq_prepack_weights(d["wscales"], d["lora_up"] if w.R else None,
                                                d.get("wcscale"))
            apk = pkg.svdq_pack_scales(d["ascales"])
            torch.cuda.synchronize(dev)
            la = d.get("lora_act_in")
            la16 = la.to(out.dtype) if la is not None and w.R % 8 == 0 else None
            cases = {"prepacked": (d["ascales"], la, {}),
                     "prepacked_packed_scales": (apk, la, dict(act_scales_packed=1)),
                     "prepacked_packed_scales_relaxed_order": (apk, la, dict(act_scales_packed=1,
                                                                             relaxed_order=1))}
            if la16 is not None:
                # the formats the activation quantiser writes: packed scales,
                # 16-bit LA (64-rank LoRA items)
                cases["prepacked_packed_scales_lora16"] = (
                    apk, la16, dict(act_scales_packed=1, lora_act_16bit=1))
            for name, (asc, la_in, extra) in cases.items():
                o2 = dict(opts, **extra)

                def call():
                    pkg.svdq_w4a4_gemm_prepacked(d["act"], d["wgt"], asc, wpk, la_in,
                                                 lup, d.get("wcscale"), d.get("bias"), out,
                                                 stream=stream, options=o2)
                for _ in range(3):
                    flush.zero_()
                    call()
                t = []
                for _ in range(10):
                    flush.zero_()
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    call()
                    e1.record(stream)
                    torch.cuda.synchronize(dev)
                    t.append(e0.elapsed_time(e1))
                r_ms = statistics.mean(t)
                routes[name] = {"ms_per_launch": r_ms,
                                "value": job_tflops(float(w.flops), world, r_ms), "unit": "TFLOPS"}
        except Exception as exc:
            routes = {"skipped": f"{type(exc).__name__}: {exc}"[:200]}
        code, site, _ = pkg.svdq_read_device_status(clear=True)
        if code != 0:
            raise RuntimeError(f"device status {code} at wait site {site} in the route timings")

    # end to end through the public call: pinned host inputs -> device -> op ->
    # host.  Every step copies its inputs in and its result out inside the
    # timed region.  Steps are pipelined as a serving loop would run them: three
    # buffer sets and three streams (host->device, operator, device->host), so
    # step i+1's inputs travel while step i computes and step i-1's result
    # returns.  The serial form (copy in, call, copy out, wait) is kept as
    # `serial_value`.
    host = {k: v.pin_memory() for k, v in host_src.items()}
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = out.numel() * out.element_size()
    nbuf = 3
    dsets = [{k: torch.empty_like(v, device=dev) for k, v in host_src.items()} for _ in range(nbuf)]
    douts = [torch.empty_like(out) for _ in range(nbuf)]
    houts = [torch.empty((w.M, w.N), dtype=out_dtype).pin_memory() for _ in range(nbuf)]
    s_in, s_op, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev = {n: [torch.cuda.Event() for _ in range(nbuf)] for n in ("in", "op", "out")}
    used = [False] * nbuf

    def e2e_step(i):
        b = i % nbuf
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(ev["op"][b])        # the operator has read set b
            for k in host:
                dsets[b][k].copy_(host[k], non_blocking=True)
            ev["in"][b].record(s_in)
        s_op.wait_event(ev["in"][b])
        if used[b]:
            s_op.wait_event(ev["out"][b])           # set b's result has been read back
        step(douts[b], dsets[b], s=s_op)
        ev["op"][b].record(s_op)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["op"][b])
            houts[b].copy_(douts[b], non_blocking=True)
            ev["out"][b].record(s_out)
        used[b] = True

    n_e2e = max(args.e2e_steps, 2 * nbuf)
    for i in range(nbuf):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for i in range(n_e2e):
        e2e_step(nbuf + i)
    torch.cuda.synchronize(dev)
    e_ms_mean = max_over_ranks((time.perf_counter() - t0) * 1e3 / n_e2e, dist, dev)
    # serial: one step at a time
    e_ms = []
    for i in range(args.e2e_steps + 2):
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for k in host:
            dsets[0][k].copy_(host[k], non_blocking=True)
        step(douts[0], dsets[0])
        houts[0].copy_(douts[0], non_blocking=True)
        torch.cuda.synchronize(dev)
        if i >= 2:
            e_ms.append((time.perf_counter() - t0) * 1e3)
    e_ms_serial = max_over_ranks(statistics.mean(e_ms), dist, dev)
    code, site, _ = pkg.svdq_read_device_status(clear=True)
    if code != 0:
        raise RuntimeError(f"device status {code} at wait site {site} in the end-to-end run")

    flops = float(w.flops)
    tflops_kernel = job_tflops(flops, 1, ms_mean)
    value = job_tflops(flops, world, ms_mean)
    e2e_value = job_tflops(flops, world, e_ms_mean)
    bf16_peak, peak_src = load_peaks()
    fp4_peak = bf16_peak * NOMINAL_FP4_OVER_BF16
    traffic = committed_traffic(w.name)

    per_shape = None
    if plain and rank == 0 and not args.no_per_shape:
        with ClockSampler(local_rank) as clk2:
            try:
                per_shape = run_per_shape(pkg, synth, torch, dev, stream, flush, fp4_peak)
            except Exception as exc:
                per_shape = {"skipped": f"{type(exc).__name__}: {exc}"[:300]}
        if isinstance(per_shape, dict):
            per_shape["clocks"] = clk2.summary()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, rows, secs, threads = oracle_sample(w, inp, target_s=12.0)
        cpu = {"value": v, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
               "sample": f"first {rows} of {w.M} output rows, all {w.N} columns "
                         f"({secs:.1f} s, fp64, OpenMP over rows)"}

    if rank == 0:
        line = {
            "metric": "W4A4+LoRA GEMM TFLOPS (2MNK+2MNR)",
            "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_mean, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4", "data": "synthetic",
            "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "R": w.R,
                       "l2": "flushed: 256 MiB memset before every timed launch",
                       "parallelism": f"replicas x{world} (independent problems, no collective)",
                       "tile": [plan["tile_m"], plan["tile_n"]], "stages": plan["num_ab_stage"],
                       "grid": plan["grid"], "k_splits": plan["k_splits"],
                       "mma_order": "relaxed" if args.relaxed_order else
                                    "ring order (bit-reproducible)"},
            "mfu_vs_10pf": tflops_kernel / METRIC_PEAK_TFLOPS,
            "ms_per_step_min": min(ms), "ms_per_step_median": statistics.median(ms),
            "wall_s_timed_region": t_wall,
            "roofline": {"bound": "tensor", "achieved": tflops_kernel, "peak": fp4_peak,
                         "unit": "TFLOP/s", "frac": tflops_kernel / fp4_peak,
                         "traffic": traffic,
                         "peak_source": f"{peak_src} bf16 burst {bf16_peak:.1f} TFLOP/s x nominal "
                                        f"fp4/bf16 ratio {NOMINAL_FP4_OVER_BF16:g}"},
            "e2e": {"value": e2e_value, "unit": "TFLOPS", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e_ms_mean,
                    "how": f"{n_e2e} steps pipelined over {nbuf} buffer sets and 3 streams "
                           "(copy in, operator, copy out; pinned host memory); wall clock",
                    "serial_value": job_tflops(flops, world, e_ms_serial),
                    "serial_ms_per_step": e_ms_serial},
            "gpu_launches": args.steps,
            "cpu_baseline": cpu,
            "clocks": clk.summary(),
            "hot_l2": hot,
            "back_to_back_cold": b2b,
            "routes": routes,
            "per_shape": per_shape,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.warmup < 3:
        args.warmup = 3
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus if args.gpus else 1)))
    if "WORLD_SIZE" not in os.environ:
        world = 1
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    from nvfp4_w4a4_quantized_gb300 import synth

    w = synth.WORKLOADS[args.workload]
    if (args.dense or args.fp16 or args.prepacked or args.split or args.packed_scales
            or args.relaxed_order):
        import dataclasses

        if args.dense:
            w = dataclasses.replace(w, name=w.name + "_dense", R=0)
        if args.fp16:
            w = dataclasses.replace(w, name=w.name + "_fp16")
        if args.packed_scales:
            w = dataclasses.replace(w, name=w.name + "_packed_scales")
        elif args.prepacked:
            w = dataclasses.replace(w, name=w.name + "_prepacked")
        if args.split:
            w = dataclasses.replace(w, name=w.name + "_split")
        if args.relaxed_order:
            w = dataclasses.replace(w, name=w.name + "_relaxed_order")
    if args.impl == "reference":
        run_reference(args, w, rank)
    else:
        run_ours(args, w, rank, world, local_rank)


if __name__ == "__main__":
    main()
