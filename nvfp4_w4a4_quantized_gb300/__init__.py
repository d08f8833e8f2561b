"""GB300 (sm_103a) SVDQuant W4A4 linear-layer operator.

    y = scaled_mma(act4, wgt4) * wcscale + bias + lora_act_in @ lora_up

The operator, and the activation quantiser that produces its activation
inputs from 16-bit activations, run in the CUDA library ``libsvdq.so`` (C ABI:
include/svdq.h); this package holds its build script, a ctypes binding with the
same entry point names, and the seeded synthetic input generator.
"""

from .binding import (SVDQ_ERR_BAD_OPTION, SVDQ_ERR_INVALID_ARG, SVDQ_ERR_MISALIGNED,  # noqa: F401
                      SVDQ_ERR_TIMEOUT, SVDQ_ERR_UNSUPPORTED_DEVICE, SVDQ_ERR_UNSUPPORTED_SHAPE,
                      SVDQ_OK, SvdqError, SvdqOptions, load, status_string, svdq_lora_stage_bytes,
                      svdq_pack_scales, svdq_prepack_weights, svdq_query_plan, svdq_read_device_status,
                      svdq_quantize_act, svdq_quantize_query, svdq_version, svdq_w4a4_gemm,
                      svdq_w4a4_gemm_prepacked, svdq_w4a4_gemm_split, svdq_w4a4_linear,
                      svdq_linear_workspace_size, svdq_workspace_size)
