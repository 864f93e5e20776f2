"""Python binding of libqmm.so (the C ABI in include/qmm.h).

Argument marshalling only: every function checks tensor devices, dtypes and
shapes, then passes raw device pointers, sizes and the current CUDA stream to
the library.  All arithmetic runs in the library's CUDA kernels; if the
library is missing, the first call raises instead of computing anything
another way.

Tensor conventions (all CUDA, contiguous):
  codes   torch.uint8  [N, K]           one code per byte (int8 bit pattern for bits=8)
  packed  torch.int32  [N, K*bits/32]   32-bit code words (bit patterns)
  scales  torch.float16 [N, K/group]
  biases  torch.float16 [N, K/group]    bits=4 only, else None
  x       torch.float32 [M, K] (gemv) or torch.bfloat16 [M, K] (gemm)
  y       torch.float32 [M, N]
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqmm.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "qmm.h")

QMM_OK = 0
STATUS = {0: "QMM_OK", -1: "QMM_ERR_ARG", -2: "QMM_ERR_SHAPE", -3: "QMM_ERR_ALIGN",
          -4: "QMM_ERR_UNSUPPORTED", -5: "QMM_ERR_CUDA", -6: "QMM_ERR_DEVICE_TIMEOUT"}

_lock = threading.Lock()
_lib = None


class QmmError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_status_string(status)}")


def declared_symbols() -> list[str]:
    """Names of the entry points declared in include/qmm.h."""
    text = open(HEADER_PATH).read()
    return sorted(set(re.findall(r"\b(qmm_[a-z_0-9]+)\s*\(", text)))


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it first (python -m quantized_weight_gb300.build)")
            L = ctypes.CDLL(LIB_PATH)
            i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
            L.qmm_pack.argtypes = [vp, vp, i64, i64, i32, vp]
            L.qmm_unpack.argtypes = [vp, vp, i64, i64, i32, vp]
            L.qmm_dequant.argtypes = [vp, vp, vp, vp, i64, i64, i32, i32, vp]
            L.qmm_gemv.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, i32, vp]
            L.qmm_gemm.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, i32, vp]
            L.qmm_quantize.argtypes = [vp, vp, vp, vp, i64, i64, i32, vp]
            L.qmm_gather_dequant.argtypes = [vp, i64, vp, vp, vp, vp, i64, i64, i32, i32, vp]
            L.qmm_gemv_argmax_workspace_size.argtypes = [i64, i64]
            L.qmm_gemv_argmax_workspace_size.restype = ctypes.c_size_t
            L.qmm_gemv_argmax.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i32, i32, vp, ctypes.c_size_t, vp]
            L.qmm_gemv_argmax_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i32, i32, vp]
            L.qmm_check.argtypes = [vp]
            L.qmm_test_timeout_next_decode.argtypes = [i64]
            L.qmm_status_string.argtypes = [i32]
            L.qmm_status_string.restype = ctypes.c_char_p
            L.qmm_abi_version.argtypes = []
            for f in ("qmm_pack", "qmm_unpack", "qmm_dequant", "qmm_gemv", "qmm_gemm", "qmm_quantize",
                      "qmm_gather_dequant", "qmm_gemv_argmax", "qmm_gemv_argmax_noalloc", "qmm_check",
                      "qmm_test_timeout_next_decode", "qmm_abi_version"):
                getattr(L, f).restype = i32
            _lib = L
    return _lib


def _status_string(status: int) -> str:
    try:
        return lib().qmm_status_string(int(status)).decode()
    except Exception:
        return STATUS.get(int(status), str(status))


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def _need(t, name, dtype, shape=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _call(what, rc):
    if rc != QMM_OK:
        raise QmmError(rc, what)


def pack(codes: torch.Tensor, bits: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    N, K = codes.shape
    _need(codes, "codes", torch.uint8)
    if out is None:
        out = torch.empty((N, K * bits // 32), dtype=torch.int32, device=codes.device)
    _need(out, "out", torch.int32, (N, K * bits // 32))
    _call("qmm_pack", lib().qmm_pack(_ptr(codes), _ptr(out), N, K, bits, _stream(stream)))
    return out


def unpack(packed: torch.Tensor, N: int, K: int, bits: int, out=None, stream=None) -> torch.Tensor:
    _need(packed, "packed", torch.int32, (N, K * bits // 32))
    if out is None:
        out = torch.empty((N, K), dtype=torch.uint8, device=packed.device)
    _need(out, "out", torch.uint8, (N, K))
    _call("qmm_unpack", lib().qmm_unpack(_ptr(packed), _ptr(out), N, K, bits, _stream(stream)))
    return out


def _coeffs(scales, biases, N, K, bits, group):
    _need(scales, "scales", torch.float16, (N, K // group))
    if bits == 4:
        _need(biases, "biases", torch.float16, (N, K // group))
    elif biases is not None:
        raise ValueError("biases must be None unless bits == 4")


def dequant(packed, scales, biases, N, K, bits, group, out=None, stream=None) -> torch.Tensor:
    _need(packed, "packed", torch.int32, (N, K * bits // 32))
    _coeffs(scales, biases, N, K, bits, group)
    if out is None:
        out = torch.empty((N, K), dtype=torch.float32, device=packed.device)
    _need(out, "out", torch.float32, (N, K))
    _call("qmm_dequant", lib().qmm_dequant(_ptr(packed), _ptr(scales), _ptr(biases), _ptr(out),
                                           N, K, bits, group, _stream(stream)))
    return out


def gemv(x, packed, scales, biases, N, bits, group, out=None, stream=None) -> torch.Tensor:
    """Decode product y[M, N] = x[M, K] . dequant(W)^T, float32 x, 1 <= M <= 8."""
    M, K = x.shape
    _need(x, "x", torch.float32)
    _need(packed, "packed", torch.int32, (N, K * bits // 32))
    _coeffs(scales, biases, N, K, bits, group)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    _need(out, "out", torch.float32, (M, N))
    _call("qmm_gemv", lib().qmm_gemv(_ptr(x), _ptr(packed), _ptr(scales), _ptr(biases), _ptr(out),
                                     M, N, K, bits, group, _stream(stream)))
    return out


def gemm(x, packed, scales, biases, N, bits, group, out=None, stream=None) -> torch.Tensor:
    """Prefill product y[M, N] = x[M, K] . dequant(W)^T, bfloat16 x, any M, bits 4 / 8 / 1."""
    M, K = x.shape
    _need(x, "x", torch.bfloat16)
    _need(packed, "packed", torch.int32, (N, K * bits // 32))
    _coeffs(scales, biases, N, K, bits, group)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    _need(out, "out", torch.float32, (M, N))
    _call("qmm_gemm", lib().qmm_gemm(_ptr(x), _ptr(packed), _ptr(scales), _ptr(biases), _ptr(out),
                                     M, N, K, bits, group, _stream(stream)))
    return out


def argmax_workspace(M: int, N: int, device="cuda") -> torch.Tensor:
    """A zeroed work area for gemv_argmax (reusable: every call leaves it ready)."""
    n = int(lib().qmm_gemv_argmax_workspace_size(M, N))
    return torch.zeros(((n + 15) // 16 * 16,), dtype=torch.uint8, device=device)


def gemv_argmax(x, packed, scales, biases, N, bits, group, workspace, idx=None, val=None, stream=None):
    """Greedy head: (idx int32 [M], val float32 [M]) of argmax_n (x . dequant(W)^T)[m, n]."""
    M, K = x.shape
    _need(x, "x", torch.float32)
    _need(packed, "packed", torch.int32, (N, K * bits // 32))
    _coeffs(scales, biases, N, K, bits, group)
    _need(workspace, "workspace", torch.uint8)
    if idx is None:
        idx = torch.empty((M,), dtype=torch.int32, device=x.device)
    if val is None:
        val = torch.empty((M,), dtype=torch.float32, device=x.device)
    _need(idx, "idx", torch.int32, (M,))
    _need(val, "val", torch.float32, (M,))
    _call("qmm_gemv_argmax", lib().qmm_gemv_argmax(_ptr(x), _ptr(packed), _ptr(scales), _ptr(biases), _ptr(idx),
                                                   _ptr(val), M, N, K, bits, group, _ptr(workspace),
                                                   workspace.numel(), _stream(stream)))
    return idx, val


def gemv_argmax_noalloc(x, packed, scales, biases, N, bits, group, idx=None, val=None, stream=None):
    """gemv_argmax for one token with the library's static work area (no workspace argument)."""
    M, K = x.shape
    if M != 1:
        raise ValueError("gemv_argmax_noalloc takes one token (M == 1)")
    _need(x, "x", torch.float32)
    _need(packed, "packed", torch.int32, (N, K * bits // 32))
    _coeffs(scales, biases, N, K, bits, group)
    if idx is None:
        idx = torch.empty((1,), dtype=torch.int32, device=x.device)
    if val is None:
        val = torch.empty((1,), dtype=torch.float32, device=x.device)
    _need(idx, "idx", torch.int32, (1,))
    _need(val, "val", torch.float32, (1,))
    _call("qmm_gemv_argmax_noalloc", lib().qmm_gemv_argmax_noalloc(
        _ptr(x), _ptr(packed), _ptr(scales), _ptr(biases), _ptr(idx), _ptr(val), N, K, bits, group, _stream(stream)))
    return idx, val


def quantize(w, group=64, out=None, stream=None):
    """INT4 affine quantization of float32 w [N, K]: (packed int32 [N, K/8],
    scales float16 [N, K/group], biases float16 [N, K/group])."""
    N, K = w.shape
    _need(w, "w", torch.float32)
    if out is None:
        out = (torch.empty((N, K // 8), dtype=torch.int32, device=w.device),
               torch.empty((N, K // group), dtype=torch.float16, device=w.device),
               torch.empty((N, K // group), dtype=torch.float16, device=w.device))
    packed, scales, biases = out
    _need(packed, "packed", torch.int32, (N, K // 8))
    _need(scales, "scales", torch.float16, (N, K // group))
    _need(biases, "biases", torch.float16, (N, K // group))
    _call("qmm_quantize", lib().qmm_quantize(_ptr(w), _ptr(packed), _ptr(scales), _ptr(biases), N, K, group,
                                             _stream(stream)))
    return packed, scales, biases


def gather_dequant(ids, packed, scales, biases, N, K, bits, group, out=None, stream=None) -> torch.Tensor:
    """out[t, :] = dequant(W[ids[t], :]); int32 ids [T]; an id outside [0, N) gives a NaN row."""
    _need(ids, "ids", torch.int32)
    T = ids.numel()
    _need(packed, "packed", torch.int32, (N, K * bits // 32))
    _coeffs(scales, biases, N, K, bits, group)
    if out is None:
        out = torch.empty((T, K), dtype=torch.float32, device=packed.device)
    _need(out, "out", torch.float32, (T, K))
    _call("qmm_gather_dequant", lib().qmm_gather_dequant(_ptr(ids), T, _ptr(packed), _ptr(scales), _ptr(biases),
                                                         _ptr(out), N, K, bits, group, _stream(stream)))
    return out


def test_timeout_next_decode(limit_ns: int) -> None:
    """Test hook: the next tensor-core decode launch makes one wait that runs
    out after limit_ns; it writes no output and the next check() raises
    QMM_ERR_DEVICE_TIMEOUT."""
    _call("qmm_test_timeout_next_decode", lib().qmm_test_timeout_next_decode(int(limit_ns)))


def check(stream=None) -> None:
    """Synchronize the stream and raise if a kernel failed or a device wait timed out."""
    _call("qmm_check", lib().qmm_check(_stream(stream)))
