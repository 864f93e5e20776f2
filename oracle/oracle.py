"""ctypes marshalling for the C oracle in ``qmm_oracle.c`` (test infrastructure).

Array conventions (numpy):
  codes   uint8  [N, K]          one code per byte (int8 bit pattern for bits=8)
  packed  uint32 [N, K*bits/32]  little-endian packing, see qmm_oracle.c
  scales  uint16 [N, K/group]    IEEE binary16 bit patterns
  biases  uint16 [N, K/group]    binary16 bit patterns (bits=4 only, else None)
  x       float32 [M, K] (qmm_f32x) or uint16 bfloat16 bit patterns (qmm_bf16x)
  y       float64 [M, N]
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# -ffp-contract=off: no fused multiply-add, every written operation rounds once.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread"]


def lib_path() -> str:
    return _LIB


def build(force: bool = False) -> str:
    """Compile qmm_oracle.c into liboracle.so next to it (gcc, no GPU needed)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
            lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_half_to_double.restype = ctypes.c_double
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_double.restype = ctypes.c_double
            lib.oracle_pack.argtypes = [vp, vp, i64, i64, i32]
            lib.oracle_unpack.argtypes = [vp, vp, i64, i64, i32]
            lib.oracle_dequant.argtypes = [vp, vp, vp, vp, i64, i64, i32, i32]
            lib.oracle_qmm_f32x.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, i32, i32]
            lib.oracle_qmm_bf16x.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, i32, i32]
            lib.oracle_qmm_sampled.argtypes = [vp, i32, vp, vp, vp, vp, vp, i64, vp,
                                               i64, i64, i64, i32, i32]
            lib.oracle_quantize_affine4.argtypes = [vp, i64, vp, vp, vp]
            lib.oracle_float_to_half.argtypes = [ctypes.c_float]
            lib.oracle_float_to_half.restype = ctypes.c_uint16
            lib.oracle_quantize_affine4_f32.argtypes = [vp, i64, i64, i32, vp, vp, vp]
            for f in ("oracle_pack", "oracle_unpack", "oracle_dequant", "oracle_qmm_f32x",
                      "oracle_qmm_bf16x", "oracle_qmm_sampled", "oracle_quantize_affine4"):
                getattr(lib, f).restype = i32
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _arr(a, dtype):
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return a


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"{what}: oracle rejected the arguments (rc={rc})")


def half_to_double(h: int) -> float:
    return _load().oracle_half_to_double(int(h))


def bf16_to_double(b: int) -> float:
    return _load().oracle_bf16_to_double(int(b))


def pack(codes: np.ndarray, bits: int) -> np.ndarray:
    codes = _arr(codes, np.uint8)
    N, K = codes.shape
    out = np.empty((N, K * bits // 32), dtype=np.uint32)
    _check(_load().oracle_pack(_ptr(codes), _ptr(out), N, K, bits), "pack")
    return out


def unpack(packed: np.ndarray, N: int, K: int, bits: int) -> np.ndarray:
    packed = _arr(packed, np.uint32)
    out = np.empty((N, K), dtype=np.uint8)
    _check(_load().oracle_unpack(_ptr(packed), _ptr(out), N, K, bits), "unpack")
    return out


def dequant(packed, scales, biases, N, K, bits, group) -> np.ndarray:
    packed = _arr(packed, np.uint32)
    scales = _arr(scales, np.uint16)
    biases = None if biases is None else _arr(biases, np.uint16)
    w = np.empty((N, K), dtype=np.float64)
    _check(_load().oracle_dequant(_ptr(packed), _ptr(scales), _ptr(biases), _ptr(w),
                                  N, K, bits, group), "dequant")
    return w


def _threads(nthreads):
    if nthreads is None:
        try:
            return max(1, len(os.sched_getaffinity(0)))
        except AttributeError:
            return max(1, os.cpu_count() or 1)
    return int(nthreads)


def qmm_f32x(x, packed, scales, biases, N, K, bits, group, nthreads=None) -> np.ndarray:
    """y[M, N] (float64) for float32 activations x[M, K]."""
    x = _arr(x, np.float32)
    M = x.shape[0]
    packed = _arr(packed, np.uint32)
    scales = _arr(scales, np.uint16)
    biases = None if biases is None else _arr(biases, np.uint16)
    y = np.empty((M, N), dtype=np.float64)
    _check(_load().oracle_qmm_f32x(_ptr(x), _ptr(packed), _ptr(scales), _ptr(biases), _ptr(y),
                                   M, N, K, bits, group, _threads(nthreads)), "qmm_f32x")
    return y


def qmm_bf16x(x_bf16, packed, scales, biases, N, K, bits, group, nthreads=None) -> np.ndarray:
    """y[M, N] (float64) for bfloat16 activations given as uint16 bit patterns."""
    x = _arr(x_bf16, np.uint16)
    M = x.shape[0]
    packed = _arr(packed, np.uint32)
    scales = _arr(scales, np.uint16)
    biases = None if biases is None else _arr(biases, np.uint16)
    y = np.empty((M, N), dtype=np.float64)
    _check(_load().oracle_qmm_bf16x(_ptr(x), _ptr(packed), _ptr(scales), _ptr(biases), _ptr(y),
                                    M, N, K, bits, group, _threads(nthreads)), "qmm_bf16x")
    return y


def qmm_sampled(x, packed, scales, biases, ms, ns, N, K, bits, group) -> np.ndarray:
    """y[ms[i], ns[i]] for the listed outputs only; x is float32 or bf16 (uint16)."""
    if x.dtype == np.uint16:
        is_bf16 = 1
    elif x.dtype == np.float32:
        is_bf16 = 0
    else:
        raise TypeError("x must be float32 or bfloat16 bit patterns (uint16)")
    x = np.ascontiguousarray(x)
    M = x.shape[0]
    ms = _arr(np.asarray(ms, dtype=np.int64), np.int64)
    ns = _arr(np.asarray(ns, dtype=np.int64), np.int64)
    if ms.shape != ns.shape:
        raise ValueError("ms and ns differ in length")
    packed = _arr(packed, np.uint32)
    scales = _arr(scales, np.uint16)
    biases = None if biases is None else _arr(biases, np.uint16)
    out = np.empty(ms.shape, dtype=np.float64)
    _check(_load().oracle_qmm_sampled(_ptr(x), is_bf16, _ptr(packed), _ptr(scales), _ptr(biases),
                                      _ptr(ms), _ptr(ns), ms.size, _ptr(out), M, N, K, bits, group),
           "qmm_sampled")
    return out


def quantize_affine4(w):
    """(codes uint8, scale float, min float) of one block, see qmm_oracle.c."""
    w = _arr(np.asarray(w, dtype=np.float64), np.float64)
    q = np.empty(w.shape, dtype=np.uint8)
    s = ctypes.c_double()
    mn = ctypes.c_double()
    _check(_load().oracle_quantize_affine4(_ptr(w), w.size, _ptr(q), ctypes.addressof(s),
                                           ctypes.addressof(mn)), "quantize_affine4")
    return q, s.value, mn.value


def float_to_half(f: float) -> int:
    """binary16 bit pattern of float32 f, round to nearest even (qmm_oracle.c)."""
    return int(_load().oracle_float_to_half(ctypes.c_float(f)))


def quantize_affine4_f32(w, group):
    """(codes uint8 [N,K], scales uint16 [N,K/group], biases uint16) of float32 w [N,K]:
    the stored-format INT4 affine quantizer of qmm_oracle.c."""
    w = _arr(np.asarray(w, dtype=np.float32), np.float32)
    N, K = w.shape
    codes = np.empty((N, K), dtype=np.uint8)
    sc = np.empty((N, K // group), dtype=np.uint16)
    bi = np.empty((N, K // group), dtype=np.uint16)
    _check(_load().oracle_quantize_affine4_f32(_ptr(w), N, K, group, _ptr(codes), _ptr(sc), _ptr(bi)),
           "quantize_affine4_f32")
    return codes, sc, bi
