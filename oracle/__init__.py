"""ORACLE -- test infrastructure, not part of the product.

A plain CPU reference of the SVDQuant W4A4 linear operator in fp64
("SVDQuant W4A4 on Blackwell" §2, §3.1), of the weight-side prepack and of
the activation quantiser that produces the operator's activation inputs.
Only tests/, the package's smoke check and bench.py's CPU-baseline leg may
import it.
"""

from . import quant_ref  # noqa: F401
from .prepack_ref import pack_scales, prepack_lora_up, prepack_wscales  # noqa: F401
from .svdq_ref import (bf16_value, build, e2m1, e4m3, f16_value, forward,  # noqa: F401
                       num_threads, round_bf16_bits)
