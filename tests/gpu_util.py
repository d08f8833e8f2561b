"""Shared helpers for the GPU parity tests: run the CUDA path through the C
ABI and compare it element by element with the CPU oracle."""

import numpy as np
import torch

import oracle
from nvfp4_w4a4_quantized_gb300 import binding

NAN_BF16 = 0x7FC0


def to_device(inp, device="cuda"):
    return {k: (None if v is None else v.to(device)) for k, v in inp.items()}


def run_gpu(inp, M, N, K, R, options=None, check_status=True):
    """Run the CUDA path on `inp` (CPU tensors) and return y as float64 numpy.

    `out` is pre-filled with NaN so an element the kernel fails to write is
    caught by the finiteness check."""
    d = to_device(inp)
    # the 16-bit I/O type follows the inputs (fp16 lora_up / wcscale / bias
    # select the fp16 variant)
    half = any(isinstance(inp.get(k), torch.Tensor) and inp[k].dtype == torch.float16
               for k in ("lora_up", "wcscale", "bias"))
    out = torch.full((M, N), float("nan"), dtype=torch.float16 if half else torch.bfloat16,
                     device="cuda")
    la = d["lora_act_in"] if R > 0 else None
    lu = d["lora_up"] if R > 0 else None
    binding.svdq_w4a4_gemm(d["act"], d["wgt"], d["ascales"], d["wscales"], la, lu,
                           d.get("wcscale"), d.get("bias"), out, options=options)
    torch.cuda.synchronize()
    if check_status:
        code, site, block = binding.svdq_read_device_status(clear=True)
        assert code == 0, f"device status {code} at wait site {site}, CTA {block}"
    return out.to(torch.float64).cpu().numpy()


def parity(y_gpu, y_ref, rel=2.0 ** -7, rms_frac=1e-3, extra=None):
    """The acceptance bound |y_gpu - y_ref| <= 2^-7 |y_ref| + 1e-3 rms(y_ref),
    per element (plus an optional per-element allowance).  Returns the worst
    ratio |delta| / bound (<= 1 passes)."""
    assert y_gpu.shape == y_ref.shape
    assert np.all(np.isfinite(y_gpu)), "non-finite output (unwritten element?)"
    rms = float(np.sqrt(np.mean(y_ref ** 2))) if y_ref.size else 0.0
    bound = rel * np.abs(y_ref) + rms_frac * rms
    if extra is not None:
        bound = bound + extra
    bound = np.maximum(bound, 1e-30)
    ratio = np.abs(y_gpu - y_ref) / bound
    worst = float(ratio.max()) if ratio.size else 0.0
    if worst > 1.0:
        i = np.unravel_index(np.argmax(ratio), ratio.shape)
        raise AssertionError(f"parity fails at {i}: gpu={y_gpu[i]!r} ref={y_ref[i]!r} "
                             f"ratio={worst:.3g}; {int((ratio > 1).sum())} of {ratio.size} fail")
    return worst


def sample_rows(M, count=48, seed=0):
    """Rows spanning every 128-row tile edge, every 32-lane quadrant, plus random rows."""
    rng = np.random.default_rng(seed)
    fixed = {0, 31, 32, 63, 64, 95, 96, 127, M - 1, M - 128 if M > 128 else 0}
    rows = set(r for r in fixed if 0 <= r < M)
    while len(rows) < min(count, M):
        rows.add(int(rng.integers(0, M)))
    return np.array(sorted(rows), dtype=np.int64)


def oracle_y(inp, M, N, K, R, rows=None):
    return oracle.forward(inp, M, N, K, R, rows=rows)


def prepack_gpu(inp, R):
    """Prepack the weight side of `inp` (CPU tensors) on the GPU; returns the
    device inputs with wscales / lora_up replaced by their packed forms."""
    d = to_device(inp)
    wpk, lup = binding.svdq_prepack_weights(d["wscales"], d["lora_up"] if R > 0 else None,
                                            d.get("wcscale"))
    return dict(d, wscales=wpk, lora_up=lup)


def run_gpu_prepacked(inp, M, N, K, R, options=None):
    """The prepacked route: svdq_prepack_weights, then svdq_w4a4_gemm_prepacked
    (both on the GPU); y as float64 numpy."""
    d = prepack_gpu(inp, R)
    half = any(isinstance(inp.get(k), torch.Tensor) and inp[k].dtype == torch.float16
               for k in ("lora_up", "wcscale", "bias"))
    out = torch.full((M, N), float("nan"), dtype=torch.float16 if half else torch.bfloat16,
                     device="cuda")
    binding.svdq_w4a4_gemm_prepacked(d["act"], d["wgt"], d["ascales"], d["wscales"],
                                     d["lora_act_in"] if R > 0 else None, d["lora_up"],
                                     d.get("wcscale"), d.get("bias"), out, options=options)
    torch.cuda.synchronize()
    code, site, block = binding.svdq_read_device_status(clear=True)
    assert code == 0, f"device status {code} at wait site {site}, CTA {block}"
    return out.to(torch.float64).cpu().numpy()


def run_gpu_split(inp, M, N, K, R, options=None, prepacked=False, workspace=None):
    """The split-K entry point (svdq_w4a4_gemm_split) on `inp` (CPU tensors);
    allocates a zero-filled workspace of the planned size unless one is given.
    Returns (y as float64 numpy, workspace)."""
    d = prepack_gpu(inp, R) if prepacked else to_device(inp)
    half = any(isinstance(inp.get(k), torch.Tensor) and inp[k].dtype == torch.float16
               for k in ("lora_up", "wcscale", "bias"))
    opts = dict(options or {})
    if half:
        opts["io_dtype"] = binding.SVDQ_IO_FP16
    if workspace is None:
        nbytes = binding.svdq_workspace_size(M, N, K, R, options=opts)
        workspace = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device="cuda")
    out = torch.full((M, N), float("nan"), dtype=torch.float16 if half else torch.bfloat16,
                     device="cuda")
    binding.svdq_w4a4_gemm_split(d["act"], d["wgt"], d["ascales"], d["wscales"],
                                 d["lora_act_in"] if R > 0 else None,
                                 d["lora_up"] if R > 0 else None, d.get("wcscale"),
                                 d.get("bias"), out, workspace, options=opts,
                                 weights_prepacked=prepacked)
    torch.cuda.synchronize()
    code, site, block = binding.svdq_read_device_status(clear=True)
    assert code == 0, f"device status {code} at wait site {site}, CTA {block}"
    return out.to(torch.float64).cpu().numpy(), workspace
