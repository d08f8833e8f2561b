"""ORACLE loader -- test infrastructure, not part of the product.

Builds and loads ``libsvdq_oracle.so`` (plain C, fp64; see svdq_oracle.c for
the definition it evaluates, "SVDQuant W4A4 on Blackwell" §2 and §3.1) and
exposes it to Python.  Only tests/, the package's smoke check and bench.py's
CPU-baseline leg may import this module.  It imports nothing from the
product package.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Dict, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "svdq_oracle.c")
_LIB = os.path.join(_HERE, "libsvdq_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP over output rows)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            d, i64, u8p = ctypes.c_double, ctypes.c_int64, ctypes.c_void_p
            lib.svdq_oracle_e2m1.restype = d
            lib.svdq_oracle_e2m1.argtypes = [ctypes.c_int]
            lib.svdq_oracle_e4m3.restype = d
            lib.svdq_oracle_e4m3.argtypes = [ctypes.c_int]
            lib.svdq_oracle_bf16.restype = d
            lib.svdq_oracle_bf16.argtypes = [ctypes.c_uint16]
            lib.svdq_oracle_f16.restype = d
            lib.svdq_oracle_f16.argtypes = [ctypes.c_uint16]
            lib.svdq_oracle_round_bf16.restype = ctypes.c_uint16
            lib.svdq_oracle_round_bf16.argtypes = [d]
            lib.svdq_oracle_num_threads.restype = ctypes.c_int
            lib.svdq_oracle_forward.restype = ctypes.c_int
            lib.svdq_oracle_forward.argtypes = [u8p] * 8 + [i64] * 4 + [u8p, i64, u8p, u8p]
            lib.svdq_oracle_forward_io.restype = ctypes.c_int
            lib.svdq_oracle_forward_io.argtypes = ([u8p] * 8 + [i64] * 4 +
                                                   [u8p, i64, u8p, u8p, ctypes.c_int])
            _lib = lib
    return _lib


def e2m1(code: int) -> float:
    return _load().svdq_oracle_e2m1(int(code))


def e4m3(byte: int) -> float:
    return _load().svdq_oracle_e4m3(int(byte))


def bf16_value(bits: int) -> float:
    return _load().svdq_oracle_bf16(int(bits) & 0xFFFF)


def f16_value(bits: int) -> float:
    return _load().svdq_oracle_f16(int(bits) & 0xFFFF)


def round_bf16_bits(x: float) -> int:
    return int(_load().svdq_oracle_round_bf16(float(x)))


def num_threads() -> int:
    return int(_load().svdq_oracle_num_threads())


def _np_bytes(t, dtype):
    """Contiguous numpy view of a CPU torch tensor (or array) with the given
    storage dtype; bf16 tensors are viewed as their uint16 bits."""
    if t is None:
        return None
    try:
        import torch

        if isinstance(t, torch.Tensor):
            t = t.detach().contiguous().cpu()
            if t.dtype in (torch.bfloat16, torch.float16):
                t = t.view(torch.int16)
            t = t.numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(t).view(dtype))


def forward(inputs: Dict[str, object], M: int, N: int, K: int, R: int,
            rows: Optional[Sequence[int]] = None, want_main: bool = False,
            half_io: Optional[bool] = None):
    """Evaluate y (fp64) for the requested rows (all rows when None).

    ``inputs`` holds act, wgt, ascales, wscales, lora_act_in, lora_up,
    wcscale, bias (CPU torch tensors or numpy arrays; wcscale/bias may be
    None).  lora_up, wcscale and bias are bf16, or IEEE fp16 when
    ``half_io`` (by default taken from the tensors' dtype).  Returns
    y [len(rows), N] float64, and main [len(rows), N] when want_main is set.
    """
    if half_io is None:
        half_io = False
        try:
            import torch

            for key in ("lora_up", "wcscale", "bias"):
                t = inputs.get(key)
                if isinstance(t, torch.Tensor) and t.dtype == torch.float16:
                    half_io = True
        except ImportError:  # pragma: no cover
            pass
    lib = _load()
    act = _np_bytes(inputs["act"], np.uint8)
    wgt = _np_bytes(inputs["wgt"], np.uint8)
    asc = _np_bytes(inputs["ascales"], np.uint8)
    wsc = _np_bytes(inputs["wscales"], np.uint8)
    la = _np_bytes(inputs.get("lora_act_in"), np.float32) if R > 0 else None
    lu = _np_bytes(inputs.get("lora_up"), np.uint16) if R > 0 else None
    wc = _np_bytes(inputs.get("wcscale"), np.uint16)
    bi = _np_bytes(inputs.get("bias"), np.uint16)
    assert act.size == M * K // 2 and wgt.size == N * K // 2
    assert asc.size == (K // 16) * M and wsc.size == (K // 16) * N
    if R > 0:
        assert la.size == M * R and lu.size == N * R
    if rows is None:
        rows_arr = None
        nrows = M
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = rows_arr.size
    y = np.empty((nrows, N), dtype=np.float64)
    mo = np.empty((nrows, N), dtype=np.float64) if want_main else None

    def p(a):
        return None if a is None else a.ctypes.data_as(ctypes.c_void_p)

    rc = lib.svdq_oracle_forward_io(p(act), p(wgt), p(asc), p(wsc), p(la), p(lu), p(wc), p(bi),
                                    M, N, K, R, p(rows_arr), nrows, p(y), p(mo),
                                    1 if half_io else 0)
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return (y, mo) if want_main else y
