"""ctypes binding of the C ABI in include/svdq.h.

Argument marshalling only: every step of the operator runs in the CUDA
library.  If ``libsvdq.so`` is missing or fails to load, importing the
entry points raises -- there is no fallback of any kind.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libsvdq.so")
# include/svdq.h SVDQ_ABI_VERSION the structs below mirror
ABI_VERSION = 701
# include/svdq.h size limits
SVDQ_MAX_MN = 1 << 24
SVDQ_MAX_K = 1 << 20
SVDQ_MAX_RANK = 128

SVDQ_OK = 0
SVDQ_ERR_INVALID_ARG = -1
SVDQ_ERR_UNSUPPORTED_SHAPE = -2
SVDQ_ERR_MISALIGNED = -3
SVDQ_ERR_UNSUPPORTED_DEVICE = -4
SVDQ_ERR_LAUNCH = -5
SVDQ_ERR_CUDA = -6
SVDQ_ERR_TIMEOUT = -7
SVDQ_ERR_BAD_OPTION = -8
SVDQ_ERR_WORKSPACE = -9
SVDQ_ERR_SCRATCH_LIMIT = -10
SVDQ_ERR_WCSCALE_ZERO = -11
SVDQ_ERR_LU_OVERFLOW = -12
SVDQ_NOALLOC_SCRATCH_BYTES = 16 << 20

SVDQ_IO_BF16 = 0
SVDQ_IO_FP16 = 1

# Every symbol include/svdq.h declares.
EXPORTED = ("svdq_w4a4_gemm", "svdq_w4a4_gemm_ex", "svdq_prepack_weights", "svdq_pack_scales",
            "svdq_w4a4_gemm_prepacked", "svdq_w4a4_gemm_split", "svdq_w4a4_gemm_split_noalloc",
            "svdq_workspace_size",
            "svdq_query_plan", "svdq_lora_stage_bytes", "svdq_read_device_status",
            "svdq_status_string", "svdq_version", "svdq_quantize_act", "svdq_quantize_query",
            "svdq_w4a4_linear", "svdq_linear_workspace_size")


class SvdqOptions(ctypes.Structure):
    _fields_ = [("tile_n", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("max_ctas", ctypes.c_int32), ("timeout_ms", ctypes.c_int32),
                ("debug_fault", ctypes.c_int32), ("cta_group", ctypes.c_int32),
                ("io_dtype", ctypes.c_int32), ("k_splits", ctypes.c_int32),
                ("act_scales_packed", ctypes.c_int32), ("relaxed_order", ctypes.c_int32),
                ("lora_act_16bit", ctypes.c_int32)]


class SvdqPlan(ctypes.Structure):
    _fields_ = [("tile_m", ctypes.c_int32), ("tile_n", ctypes.c_int32), ("tile_k", ctypes.c_int32),
                ("cta_group", ctypes.c_int32), ("num_ab_stage", ctypes.c_int32),
                ("num_acc_stage", ctypes.c_int32), ("stage_bytes", ctypes.c_int32),
                ("lora_block_bytes", ctypes.c_int32), ("lora_blocks", ctypes.c_int32),
                ("k_blocks", ctypes.c_int32), ("smem_bytes", ctypes.c_int32),
                ("tmem_cols", ctypes.c_int32), ("tmem_cols_used", ctypes.c_int32),
                ("threads", ctypes.c_int32), ("num_tiles", ctypes.c_int64),
                ("grid", ctypes.c_int32), ("sm_count", ctypes.c_int32),
                ("kblocks_per_stage", ctypes.c_int32), ("k_splits", ctypes.c_int32),
                ("num_units", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class SvdqError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})" if what else
                         f"{status_string(status)} ({status})")


_lock = threading.Lock()
_lib = None


def load(path: Optional[str] = None):
    """Load libsvdq.so (raises OSError/RuntimeError if it is absent)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"CUDA library not built: {p} (run nvfp4_w4a4_quantized_gb300.build)")
        # the CUDA runtime must be the one torch uses when both are in-process
        try:
            import torch  # noqa: F401
        except ImportError:  # pragma: no cover
            pass
        lib = ctypes.CDLL(p, mode=ctypes.RTLD_GLOBAL)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
        lib.svdq_w4a4_gemm.restype = ctypes.c_int
        lib.svdq_w4a4_gemm.argtypes = [vp] * 9 + [i64] * 4 + [vp]
        lib.svdq_w4a4_gemm_ex.restype = ctypes.c_int
        lib.svdq_w4a4_gemm_ex.argtypes = [vp] * 9 + [i64] * 4 + [ctypes.POINTER(SvdqOptions), vp]
        lib.svdq_prepack_weights.restype = ctypes.c_int
        lib.svdq_prepack_weights.argtypes = [vp] * 3 + [i64] * 3 + [i32] + [vp] * 3
        lib.svdq_pack_scales.restype = ctypes.c_int
        lib.svdq_pack_scales.argtypes = [vp, i64, i64, vp, vp]
        lib.svdq_w4a4_gemm_prepacked.restype = ctypes.c_int
        lib.svdq_w4a4_gemm_prepacked.argtypes = ([vp] * 9 + [i64] * 4 +
                                                 [ctypes.POINTER(SvdqOptions), vp])
        lib.svdq_w4a4_gemm_split.restype = ctypes.c_int
        lib.svdq_w4a4_gemm_split.argtypes = ([vp] * 9 + [i64] * 4 +
                                             [ctypes.POINTER(SvdqOptions), i32, vp, i64, vp])
        lib.svdq_w4a4_gemm_split_noalloc.restype = ctypes.c_int
        lib.svdq_w4a4_gemm_split_noalloc.argtypes = ([vp] * 9 + [i64] * 4 +
                                                     [ctypes.POINTER(SvdqOptions), i32, vp])
        lib.svdq_workspace_size.restype = i64
        lib.svdq_workspace_size.argtypes = [i64] * 4 + [ctypes.POINTER(SvdqOptions), i32]
        lib.svdq_query_plan.restype = ctypes.c_int
        lib.svdq_query_plan.argtypes = [i64] * 4 + [ctypes.POINTER(SvdqOptions), i32,
                                                    ctypes.POINTER(SvdqPlan)]
        lib.svdq_lora_stage_bytes.restype = i64
        lib.svdq_lora_stage_bytes.argtypes = [i64] * 5 + [ctypes.POINTER(i64)] * 2
        lib.svdq_read_device_status.restype = ctypes.c_int
        lib.svdq_read_device_status.argtypes = [ctypes.POINTER(i32)] * 3 + [ctypes.c_int]
        lib.svdq_status_string.restype = ctypes.c_char_p
        lib.svdq_status_string.argtypes = [ctypes.c_int]
        lib.svdq_version.restype = ctypes.c_int
        lib.svdq_version.argtypes = []
        lib.svdq_quantize_act.restype = ctypes.c_int
        lib.svdq_quantize_act.argtypes = [vp, vp] + [i64] * 3 + [i32] * 3 + [vp] * 4
        lib.svdq_quantize_query.restype = ctypes.c_int
        lib.svdq_quantize_query.argtypes = [i64] * 3 + [i32] + [ctypes.POINTER(i32)] * 4
        lib.svdq_w4a4_linear.restype = ctypes.c_int
        lib.svdq_w4a4_linear.argtypes = [vp] * 8 + [i64] * 4 + [ctypes.POINTER(SvdqOptions), vp,
                                                               i64, vp]
        lib.svdq_linear_workspace_size.restype = i64
        lib.svdq_linear_workspace_size.argtypes = [i64] * 3
        # the ctypes structs here mirror include/svdq.h at ABI_VERSION
        if lib.svdq_version() // 100 != ABI_VERSION // 100:
            raise RuntimeError(f"{p} has ABI version {lib.svdq_version()}, this binding "
                               f"expects {ABI_VERSION}: rebuild the library")
        if path is None:
            _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().svdq_status_string(int(status)).decode()


def _opts(options) -> Optional[SvdqOptions]:
    if options is None:
        return None
    if isinstance(options, SvdqOptions):
        return options
    o = SvdqOptions()
    for k, v in dict(options).items():
        setattr(o, k, int(v))
    return o


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream_handle(stream, device) -> int:
    import torch

    if stream is None:
        stream = torch.cuda.current_stream(device)
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(name, t, dt):
    if t.dtype != dt or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name}: expected contiguous CUDA {dt}, got {t.dtype} "
                         f"on {t.device} (contiguous={t.is_contiguous()})")


def svdq_w4a4_gemm(act, wgt, ascales, wscales, lora_act_in, lora_up, wcscale, bias, out,
                   stream=None, options=None, check: bool = True) -> int:
    """y = scaled_mma(act4, wgt4) * wcscale + bias + lora_act_in @ lora_up into ``out``.

    Tensors are CUDA torch tensors with the layouts of include/svdq.h
    (act uint8 [M, K/2], wgt uint8 [N, K/2], ascales uint8 [K/16, M],
    wscales uint8 [K/16, N], lora_act_in fp32 [M, R], lora_up bf16 [N, R],
    wcscale/bias bf16 [N] or None, out bf16 [M, N]).  An fp16 ``out`` selects
    the fp16 variant: lora_up, wcscale and bias must then be fp16 too.
    Asynchronous on
    ``stream`` (default: torch's current stream).  Raises SvdqError on a
    non-zero status when ``check``; returns the status otherwise.
    """
    return _gemm(act, wgt, ascales, wscales, lora_act_in, lora_up, wcscale, bias, out, stream,
                 options, check, prepacked=False)


def svdq_w4a4_gemm_prepacked(act, wgt, ascales, wscales_packed, lora_act_in, lora_up_packed,
                             wcscale, bias, out, stream=None, options=None,
                             check: bool = True) -> int:
    """svdq_w4a4_gemm on prepacked weights (see svdq_prepack_weights):
    wscales_packed int32 [K/64, N] scale words, lora_up_packed LU' [N, R];
    ``wcscale`` must be the one LU' was packed with."""
    return _gemm(act, wgt, ascales, wscales_packed, lora_act_in, lora_up_packed, wcscale, bias,
                 out, stream, options, check, prepacked=True)


def svdq_w4a4_gemm_split(act, wgt, ascales, wscales, lora_act_in, lora_up, wcscale, bias, out,
                         workspace, stream=None, options=None, weights_prepacked: bool = False,
                         check: bool = True) -> int:
    """The operator with split-K for shapes that leave most SMs idle (see
    include/svdq.h).  ``workspace`` is a zero-filled CUDA uint8 tensor of at
    least svdq_workspace_size(...) bytes, reused across calls (calls sharing
    it must not overlap on the GPU).  With ``weights_prepacked`` the weights
    come from svdq_prepack_weights."""
    return _gemm(act, wgt, ascales, wscales, lora_act_in, lora_up, wcscale, bias, out, stream,
                 options, check, prepacked=weights_prepacked, workspace=workspace)


def svdq_workspace_size(M: int, N: int, K: int, R: int, options=None, sm_count: int = 0) -> int:
    """Bytes of workspace svdq_w4a4_gemm_split needs (0: the plan does not split)."""
    opts = _opts(options)
    n = load().svdq_workspace_size(M, N, K, R, ctypes.byref(opts) if opts else None, sm_count)
    if n < 0:
        raise SvdqError(int(n), "svdq_workspace_size")
    return int(n)


def _gemm(act, wgt, ascales, wscales, lora_act_in, lora_up, wcscale, bias, out, stream, options,
          check, prepacked, workspace=None):
    import torch

    M, kh = act.shape
    N = wgt.shape[0]
    K = 2 * kh
    R = 0 if lora_act_in is None else int(lora_act_in.shape[1])
    h16 = torch.float16 if out.dtype == torch.float16 else torch.bfloat16
    ws_dt = torch.int32 if prepacked else torch.uint8
    ws_shape = (K // 64, N) if prepacked else (K // 16, N)
    act_packed = bool(_opts(options) and _opts(options).act_scales_packed)
    # lora_act_in as 16-bit values in the I/O type (lora_act_16bit) or fp32
    la_dt = h16 if (_opts(options) and _opts(options).lora_act_16bit) else torch.float32
    as_dt = torch.int32 if act_packed else torch.uint8
    as_shape = (K // 64, M) if act_packed else (K // 16, M)
    for name, t, dt in (("act", act, torch.uint8), ("wgt", wgt, torch.uint8),
                        ("ascales", ascales, as_dt), ("wscales", wscales, ws_dt),
                        ("lora_act_in", lora_act_in, la_dt),
                        ("lora_up", lora_up if R else None, h16), ("wcscale", wcscale, h16),
                        ("bias", bias, h16), ("out", out, h16)):
        if t is not None:
            _check(name, t, dt)
    if tuple(wgt.shape) != (N, kh) or tuple(ascales.shape) != as_shape or \
            tuple(wscales.shape) != ws_shape or tuple(out.shape) != (M, N):
        raise ValueError("inconsistent operand shapes")
    if R and (lora_up is None or tuple(lora_up.shape) != (N, R)):
        raise ValueError("lora_up must be [N, R]")
    for name, t in (("wcscale", wcscale), ("bias", bias)):
        if t is not None and tuple(t.shape) != (N,):
            raise ValueError(f"{name} must be [N]")
    lib = load()
    h = _stream_handle(stream, act.device)
    opts = _opts(options)
    if h16 == torch.float16:
        opts = opts if opts is not None else SvdqOptions()
        opts.io_dtype = SVDQ_IO_FP16
    args = [_ptr(act), _ptr(wgt), _ptr(ascales), _ptr(wscales), _ptr(lora_act_in),
            _ptr(lora_up), _ptr(wcscale), _ptr(bias), _ptr(out), M, N, K, R]
    with torch.cuda.device(act.device):
        if workspace is not None:
            if workspace.dtype != torch.uint8 or not workspace.is_cuda or \
                    not workspace.is_contiguous():
                raise ValueError("workspace: expected a contiguous CUDA uint8 tensor")
            rc = lib.svdq_w4a4_gemm_split(*args, ctypes.byref(opts) if opts else None,
                                          1 if prepacked else 0, workspace.data_ptr(),
                                          workspace.numel(), h)
        elif prepacked:
            rc = lib.svdq_w4a4_gemm_prepacked(*args, ctypes.byref(opts) if opts else None, h)
        elif opts is None:
            rc = lib.svdq_w4a4_gemm(*args, h)
        else:
            rc = lib.svdq_w4a4_gemm_ex(*args, ctypes.byref(opts), h)
    if check and rc != SVDQ_OK:
        raise SvdqError(rc, "svdq_w4a4_gemm_split" if workspace is not None else
                        "svdq_w4a4_gemm_prepacked" if prepacked else "svdq_w4a4_gemm")
    return rc


def svdq_pack_scales(scales, packed=None, stream=None, check: bool = True):
    """Scale tensor uint8 [K/16, rows] -> uint32 words [K/64, rows] (returned
    as int32; allocated here unless given): the layout act_scales_packed
    expects for ascales and svdq_prepack_weights writes for wscales."""
    import torch

    _check("scales", scales, torch.uint8)
    G, rows = scales.shape
    K = 16 * G
    if K % 64:
        raise ValueError("K must be a multiple of 64")
    if packed is None:
        packed = torch.empty((K // 64, rows), dtype=torch.int32, device=scales.device)
    _check("packed", packed, torch.int32)
    h = _stream_handle(stream, scales.device)
    with torch.cuda.device(scales.device):
        rc = load().svdq_pack_scales(_ptr(scales), rows, K, _ptr(packed), h)
    if check and rc != SVDQ_OK:
        raise SvdqError(rc, "svdq_pack_scales")
    return packed


def svdq_prepack_weights(wscales, lora_up, wcscale, wscales_packed=None, lora_up_packed=None,
                         stream=None, check: bool = True):
    """Weight-side prepack on the GPU: returns (wscales_packed int32 [K/64, N],
    lora_up_packed [N, R] or None).  Output tensors are allocated here unless
    given.  lora_up / wcscale are bf16, or fp16 for the fp16 variant."""
    import torch

    G, N = wscales.shape
    K = 16 * G
    R = 0 if lora_up is None else int(lora_up.shape[1])
    h16 = lora_up.dtype if lora_up is not None else (
        wcscale.dtype if wcscale is not None else torch.bfloat16)
    if h16 not in (torch.bfloat16, torch.float16):
        raise ValueError("lora_up / wcscale must be bf16 or fp16")
    _check("wscales", wscales, torch.uint8)
    if lora_up is not None:
        _check("lora_up", lora_up, h16)
        if tuple(lora_up.shape) != (N, R):
            raise ValueError("lora_up must be [N, R]")
    if wcscale is not None:
        _check("wcscale", wcscale, h16)
        if tuple(wcscale.shape) != (N,):
            raise ValueError("wcscale must be [N]")
    if K % 64:
        raise ValueError("K must be a multiple of 64")
    if wscales_packed is None:
        wscales_packed = torch.empty((K // 64, N), dtype=torch.int32, device=wscales.device)
    _check("wscales_packed", wscales_packed, torch.int32)
    if R and lora_up_packed is None:
        lora_up_packed = torch.empty((N, R), dtype=h16, device=wscales.device)
    if R:
        _check("lora_up_packed", lora_up_packed, h16)
    io = SVDQ_IO_FP16 if h16 == torch.float16 else SVDQ_IO_BF16
    lib = load()
    h = _stream_handle(stream, wscales.device)
    with torch.cuda.device(wscales.device):
        rc = lib.svdq_prepack_weights(_ptr(wscales), _ptr(lora_up) if R else None,
                                      _ptr(wcscale), N, K, R, io, _ptr(wscales_packed),
                                      _ptr(lora_up_packed) if R else None, h)
    if check and rc != SVDQ_OK:
        raise SvdqError(rc, "svdq_prepack_weights")
    return wscales_packed, (lora_up_packed if R else None)


def svdq_query_plan(M: int, N: int, K: int, R: int, options=None, sm_count: int = 0) -> dict:
    plan = SvdqPlan()
    opts = _opts(options)
    rc = load().svdq_query_plan(M, N, K, R, ctypes.byref(opts) if opts else None, sm_count,
                                ctypes.byref(plan))
    if rc != SVDQ_OK:
        raise SvdqError(rc, "svdq_query_plan")
    return plan.as_dict()


def svdq_lora_stage_bytes(tile_m: int, tile_n: int, R: int, elem_bytes: int, cta_group: int):
    la, lu = ctypes.c_int64(), ctypes.c_int64()
    tot = load().svdq_lora_stage_bytes(tile_m, tile_n, R, elem_bytes, cta_group,
                                       ctypes.byref(la), ctypes.byref(lu))
    if tot < 0:
        raise SvdqError(int(tot), "svdq_lora_stage_bytes")
    return int(tot), int(la.value), int(lu.value)


def svdq_read_device_status(clear: bool = True):
    code, site, block = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    rc = load().svdq_read_device_status(ctypes.byref(code), ctypes.byref(site),
                                        ctypes.byref(block), 1 if clear else 0)
    if rc != SVDQ_OK:
        raise SvdqError(rc, "svdq_read_device_status")
    return int(code.value), int(site.value), int(block.value)


def svdq_version() -> int:
    return int(load().svdq_version())


def svdq_quantize_act(x, lora_down=None, act=None, ascales=None, lora_act_in=None,
                      scales_packed: bool = False, lora_act_16bit: bool = False, stream=None,
                      check: bool = True):
    """The operator's activation inputs from 16-bit activations x [M, K]
    (bf16 or fp16): returns (act uint8 [M, K/2], ascales uint8 [K/16, M] or
    int32 words [K/64, M] with ``scales_packed``, lora_act_in [M, R] or None:
    fp32, or x's 16-bit type with ``lora_act_16bit``).  lora_down is [R, K] in
    x's type, or None for R = 0.  Outputs are allocated here unless given.
    Asynchronous on ``stream``."""
    import torch

    if x.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("x must be bf16 or fp16")
    _check("x", x, x.dtype)
    M, K = x.shape
    R = 0 if lora_down is None else int(lora_down.shape[0])
    if R:
        _check("lora_down", lora_down, x.dtype)
        if tuple(lora_down.shape) != (R, K):
            raise ValueError("lora_down must be [R, K]")
    dev = x.device
    if act is None:
        act = torch.empty((M, K // 2), dtype=torch.uint8, device=dev)
    sc_dt, sc_shape = (torch.int32, (K // 64, M)) if scales_packed else (torch.uint8, (K // 16, M))
    if ascales is None:
        ascales = torch.empty(sc_shape, dtype=sc_dt, device=dev)
    la_dt = x.dtype if lora_act_16bit else torch.float32
    if R and lora_act_in is None:
        lora_act_in = torch.empty((M, R), dtype=la_dt, device=dev)
    _check("act", act, torch.uint8)
    _check("ascales", ascales, sc_dt)
    if tuple(act.shape) != (M, K // 2) or tuple(ascales.shape) != sc_shape:
        raise ValueError("inconsistent output shapes")
    if R:
        _check("lora_act_in", lora_act_in, la_dt)
        if tuple(lora_act_in.shape) != (M, R):
            raise ValueError("lora_act_in must be [M, R]")
    io = SVDQ_IO_FP16 if x.dtype == torch.float16 else SVDQ_IO_BF16
    h = _stream_handle(stream, dev)
    with torch.cuda.device(dev):
        rc = load().svdq_quantize_act(_ptr(x), _ptr(lora_down) if R else None, M, K, R, io,
                                      1 if scales_packed else 0, 1 if lora_act_16bit else 0,
                                      _ptr(act), _ptr(ascales),
                                      _ptr(lora_act_in) if R else None, h)
    if check and rc != SVDQ_OK:
        raise SvdqError(rc, "svdq_quantize_act")
    return act, ascales, (lora_act_in if R else None)


def svdq_quantize_query(M: int, K: int, R: int, sm_count: int = 0) -> dict:
    """The quantiser's launch: K splits per row tile, CTAs, stages, smem bytes."""
    v = [ctypes.c_int32() for _ in range(4)]
    rc = load().svdq_quantize_query(M, K, R, sm_count, *[ctypes.byref(t) for t in v])
    if rc != SVDQ_OK:
        raise SvdqError(rc, "svdq_quantize_query")
    return dict(zip(("splits", "grid", "stages", "smem_bytes"), (int(t.value) for t in v)))


def svdq_linear_workspace_size(M: int, K: int, R: int) -> int:
    """Workspace bytes svdq_w4a4_linear needs for x [M, K] and rank R."""
    n = int(load().svdq_linear_workspace_size(M, K, R))
    if n < 0:
        raise SvdqError(n, "svdq_linear_workspace_size")
    return n


def svdq_w4a4_linear(x, lora_down, wgt, wscales_packed, lora_up_packed, wcscale, bias, out,
                     workspace=None, stream=None, options=None, check: bool = True) -> int:
    """The whole layer from 16-bit activations x [M, K] (bf16 or fp16):
    svdq_quantize_act (packed scales, 16-bit LoRA-down product when R % 8 == 0)
    then svdq_w4a4_gemm_prepacked, into ``out`` [M, N] of x's type.
    lora_down [R, K] in x's type or None; wgt uint8 [N, K/2]; wscales_packed /
    lora_up_packed from svdq_prepack_weights; ``workspace`` a uint8 CUDA tensor
    of at least svdq_linear_workspace_size bytes (allocated here if None)."""
    import torch

    if x.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("x must be bf16 or fp16")
    _check("x", x, x.dtype)
    _check("out", out, x.dtype)
    M, K = x.shape
    N = int(out.shape[1])
    R = 0 if lora_down is None else int(lora_down.shape[0])
    if R:
        _check("lora_down", lora_down, x.dtype)
        if tuple(lora_down.shape) != (R, K):
            raise ValueError("lora_down must be [R, K]")
    _check("wgt", wgt, torch.uint8)
    _check("wscales_packed", wscales_packed, torch.int32)
    for name, t in (("lora_up_packed", lora_up_packed if R else None), ("wcscale", wcscale),
                    ("bias", bias)):
        if t is not None:
            _check(name, t, x.dtype)
    if tuple(wgt.shape) != (N, K // 2) or tuple(out.shape) != (M, N):
        raise ValueError("inconsistent shapes")
    need = svdq_linear_workspace_size(M, K, R)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
    _check("workspace", workspace, torch.uint8)
    o = _opts(options)
    o = SvdqOptions() if o is None else SvdqOptions.from_buffer_copy(o)
    o.io_dtype = SVDQ_IO_FP16 if x.dtype == torch.float16 else SVDQ_IO_BF16
    h = _stream_handle(stream, x.device)
    with torch.cuda.device(x.device):
        rc = load().svdq_w4a4_linear(_ptr(x), _ptr(lora_down) if R else None, _ptr(wgt),
                                     _ptr(wscales_packed), _ptr(lora_up_packed) if R else None,
                                     _ptr(wcscale), _ptr(bias), _ptr(out), M, N, K, R,
                                     ctypes.byref(o), _ptr(workspace), workspace.numel(), h)
    if check and rc != SVDQ_OK:
        raise SvdqError(rc, "svdq_w4a4_linear")
    return rc
