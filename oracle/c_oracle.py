"""ctypes loader for the C oracle (awq_oracle_c.c).

TEST INFRASTRUCTURE ONLY, like the numpy oracle: the tests use it to check the two oracles
against each other.  It is compiled in place with gcc on first use (or by the build step),
and it shares no code with the numpy oracle or with the CUDA library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "awq_oracle_c.c")
LIB = os.path.join(HERE, "_awq_oracle_c.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle to oracle/_awq_oracle_c.so (portable C, OpenMP over rows)."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, SRC, "-lm"],
                       check=True, capture_output=True, text=True)
        os.replace(tmp, LIB)
    return LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.awq_oracle_widen_f16.argtypes = [vp, vp, i64]
        lib.awq_oracle_widen_f16.restype = None
        lib.awq_oracle_dequant_f32.argtypes = [vp, vp, vp, i64, i64, i64, i32, vp]
        lib.awq_oracle_dequant_f32.restype = i32
        lib.awq_oracle_gemm_f64.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i32, vp]
        lib.awq_oracle_gemm_f64.restype = i32
        _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def widen_f16(h: np.ndarray) -> np.ndarray:
    """fp16 -> fp32 by the C oracle's own binary16 decoding."""
    h = _c(np.asarray(h).view(np.uint16), np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    _load().awq_oracle_widen_f16(_p(h), _p(out), h.size)
    return out


def dequant_f32(qweight, qzeros, scales, group_size, bits=4) -> np.ndarray:
    qw, qz = _c(qweight, np.int32), _c(qzeros, np.int32)
    sc = _c(np.asarray(scales, dtype=np.float16).view(np.uint16), np.uint16)
    K, N = qw.shape[0], qw.shape[1] * (32 // bits)
    w = np.empty((K, N), dtype=np.float32)
    if _load().awq_oracle_dequant_f32(_p(qw), _p(qz), _p(sc), K, N, group_size, bits, _p(w)):
        raise ValueError("invalid shape")
    return w


def gemm(x, qweight, qzeros, scales, bias, group_size, bits=4) -> np.ndarray:
    xx = _c(np.asarray(x, dtype=np.float16).view(np.uint16), np.uint16)
    qw, qz = _c(qweight, np.int32), _c(qzeros, np.int32)
    sc = _c(np.asarray(scales, dtype=np.float16).view(np.uint16), np.uint16)
    b = None if bias is None else _c(np.asarray(bias, dtype=np.float16).view(np.uint16), np.uint16)
    M, K = xx.shape
    N = qw.shape[1] * (32 // bits)
    y = np.empty((M, N), dtype=np.float64)
    if _load().awq_oracle_gemm_f64(_p(xx), _p(qw), _p(qz), _p(sc), _p(b), M, K, N, group_size, bits,
                                   _p(y)):
        raise ValueError("invalid shape")
    return y
