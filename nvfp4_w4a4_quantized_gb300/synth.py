"""Seeded synthetic inputs for the SVDQuant W4A4 linear operator.

This module only draws input bytes and floats; it holds none of the
operator's arithmetic (no decoding, no products, no sums).  Both the CUDA
path and the CPU oracle are fed from it, so each side sees the same inputs.

Shapes and dtypes follow the operator definition in "SVDQuant W4A4 on
Blackwell" (§2): act [M, K/2] and wgt [N, K/2] hold two E2M1 nibbles per
byte; ascales [K/16, M] and wscales [K/16, N] hold one FP8-E4M3 scale per 16
K elements; the LoRA residual has rank R.

Distributions (the benchmark workloads' recipe):
  act, wgt       uint8 uniform over 0..255  (both nibbles uniform over 16 codes)
  ascales/wscales E4M3 byte ((u + 7) << 3) | i, u ~ U{-4..2}, i ~ U{0..7}
                 i.e. the value 2^u * (1 + i/8)
  lora_act_in    fp32 N(0, 1)            [M, R]
  lora_up        bf16 N(0, 0.05)         [N, R]
  wcscale        bf16 U(0.5, 2)          [N]
  bias           bf16 N(0, 0.1)          [N]
drawn in exactly that order from one seeded CPU torch.Generator.

Activations for the activation quantiser (make_activations), drawn in this
order from their own seeded generator:
  channel scale  2^u per input channel k, u ~ U{-2..2} (the per-channel
                 magnitudes smoothing leaves in activations)
  x              16-bit N(0, 1) * channel scale   [M, K]
  lora_down      16-bit N(0, 1/K)                 [R, K]
"""

from __future__ import annotations

import dataclasses
from typing import Dict, List

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """One operator shape with its seed. Shapes are written M x N x K."""

    name: str
    M: int
    N: int
    K: int
    R: int
    seed: int

    @property
    def flops(self) -> int:
        """Counted work: 2MNK for the main contraction plus 2MNR for LoRA."""
        return 2 * self.M * self.N * self.K + 2 * self.M * self.N * self.R


# The five benchmark workloads.  The token-count sweep expands to 24 cases.
TINY = Workload("tiny_256x256x256_r32", 256, 256, 256, 32, 0)
ATTN_PROJ = Workload("attn_proj_4096x3072x3072_r32", 4096, 3072, 3072, 32, 1)
MLP_UP = Workload("mlp_up_4096x12288x3072_r32", 4096, 12288, 3072, 32, 2)
MLP_DOWN = Workload("mlp_down_4096x3072x12288_r128", 4096, 3072, 12288, 128, 3)
# The MLP-down projection at 256 tokens: few tiles, long K (the split-K case).
MLP_DOWN_SMALL_M = Workload("mlp_down_256x3072x12288_r128", 256, 3072, 12288, 128, 5)


def sweep_workloads() -> List[Workload]:
    """Token-count sweep: M in {256,1024,4096,16384} x (N,K) in
    {(3072,3072),(12288,3072)} x R in {16,32,128}, all seeded with 4."""
    out = []
    for M in (256, 1024, 4096, 16384):
        for (N, K) in ((3072, 3072), (12288, 3072)):
            for R in (16, 32, 128):
                out.append(Workload(f"sweep_{M}x{N}x{K}_r{R}", M, N, K, R, 4))
    return out


WORKLOADS: Dict[str, Workload] = {
    w.name: w for w in [TINY, ATTN_PROJ, MLP_UP, MLP_DOWN, MLP_DOWN_SMALL_M] + sweep_workloads()
}


def scale_bytes(shape, g: torch.Generator) -> torch.Tensor:
    """E4M3 scale bytes 2^u * (1 + i/8), u ~ U{-4..2}, i ~ U{0..7}.

    The byte is assembled from its exponent field (u + 7, bias 7) and its
    3-bit mantissa field; the sign bit is 0.
    """
    u = torch.randint(-4, 3, shape, generator=g, dtype=torch.int32)
    i = torch.randint(0, 8, shape, generator=g, dtype=torch.int32)
    return (((u + 7) << 3) | i).to(torch.uint8)


def make_inputs(M: int, N: int, K: int, R: int, seed: int,
                half: bool = False) -> Dict[str, torch.Tensor]:
    """Draw one set of operator inputs as contiguous CPU tensors.

    Returns a dict with keys act, wgt, ascales, wscales, lora_act_in,
    lora_up, wcscale, bias (see the module docstring for layouts).  With
    ``half`` the same draws are rounded to fp16 instead of bf16 for lora_up,
    wcscale and bias (the fp16 input/output variant).
    """
    h16 = torch.float16 if half else torch.bfloat16
    if K % 16:
        raise ValueError("K must be a multiple of 16")
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    act = torch.randint(0, 256, (M, K // 2), generator=g, dtype=torch.uint8)
    wgt = torch.randint(0, 256, (N, K // 2), generator=g, dtype=torch.uint8)
    ascales = scale_bytes((K // 16, M), g)
    wscales = scale_bytes((K // 16, N), g)
    lora_act_in = torch.randn((M, R), generator=g, dtype=torch.float32)
    lora_up = (torch.randn((N, R), generator=g, dtype=torch.float32) * 0.05).to(h16)
    wcscale = (torch.rand((N,), generator=g, dtype=torch.float32) * 1.5 + 0.5).to(h16)
    bias = (torch.randn((N,), generator=g, dtype=torch.float32) * 0.1).to(h16)
    return dict(act=act.contiguous(), wgt=wgt.contiguous(), ascales=ascales.contiguous(),
                wscales=wscales.contiguous(), lora_act_in=lora_act_in.contiguous(),
                lora_up=lora_up.contiguous(), wcscale=wcscale.contiguous(), bias=bias.contiguous())


def make_workload_inputs(w: Workload) -> Dict[str, torch.Tensor]:
    return make_inputs(w.M, w.N, w.K, w.R, w.seed)


def make_activations(M: int, K: int, R: int, seed: int,
                     half: bool = False) -> Dict[str, torch.Tensor]:
    """16-bit activations x [M, K] and the LoRA down-projection [R, K] (bf16,
    or fp16 with ``half``) as contiguous CPU tensors (module docstring)."""
    h16 = torch.float16 if half else torch.bfloat16
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    chan = torch.exp2(torch.randint(-2, 3, (K,), generator=g).to(torch.float32))
    x = (torch.randn((M, K), generator=g, dtype=torch.float32) * chan).to(h16)
    lora_down = (torch.randn((R, K), generator=g, dtype=torch.float32) * K ** -0.5).to(h16)
    return dict(x=x.contiguous(), lora_down=lora_down.contiguous())
