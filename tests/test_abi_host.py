"""Host-side checks of the C ABI: the library builds, loads without a GPU,
exports every entry point include/qmm.h declares, and rejects bad arguments
before touching any device memory (no call here reaches a kernel)."""
import ctypes

import pytest

from quantized_weight_gb300 import build as qbuild
from quantized_weight_gb300 import qmm

OK, ARG, SHAPE, ALIGN, UNSUP = 0, -1, -2, -3, -4
FAKE = 0x10000          # never dereferenced: every call below fails validation first
MIS = 0x10004           # not 16-byte aligned
ODD = 0x10002           # not even 4-byte aligned


@pytest.fixture(scope="module")
def L():
    qbuild.build()
    return qmm.lib()


def test_exports_every_declared_symbol(L):
    names = qmm.declared_symbols()
    assert {"qmm_pack", "qmm_unpack", "qmm_dequant", "qmm_gemv", "qmm_gemm", "qmm_check",
            "qmm_status_string", "qmm_abi_version", "qmm_quantize", "qmm_gather_dequant", "qmm_gemv_argmax",
            "qmm_gemv_argmax_workspace_size"} <= set(names)
    for n in names:
        assert hasattr(L, n), f"{n} declared in qmm.h but not exported"
    assert L.qmm_abi_version() == 1


def test_status_strings(L):
    for code, name in qmm.STATUS.items():
        assert L.qmm_status_string(code).decode().startswith(name)
    assert L.qmm_status_string(12345).decode() == "unknown qmm status"


def gemv(L, x=FAKE, c=FAKE, s=FAKE, b=FAKE, y=FAKE, M=1, N=64, K=128, bits=4, g=64):
    return L.qmm_gemv(x, c, s, b, y, M, N, K, bits, g, None)


def gemm(L, x=FAKE, c=FAKE, s=FAKE, b=FAKE, y=FAKE, M=1, N=64, K=128, bits=4, g=64):
    return L.qmm_gemm(x, c, s, b, y, M, N, K, bits, g, None)


def test_gemv_validation(L):
    assert gemv(L, bits=3) == UNSUP
    assert gemv(L, g=48) == UNSUP
    assert gemv(L, M=9) == SHAPE
    assert gemv(L, M=-1) == SHAPE
    assert gemv(L, K=100) == SHAPE                 # K % 32
    assert gemv(L, K=96, g=64) == SHAPE            # K % group
    assert gemv(L, bits=1, b=None, K=96, g=32) == SHAPE   # Q1 needs K % 128
    assert gemv(L, x=None) == ARG
    assert gemv(L, y=None) == ARG
    assert gemv(L, b=None) == ARG                  # INT4 needs biases
    assert gemv(L, bits=8, b=FAKE) == ARG          # INT8 takes no biases
    assert gemv(L, bits=1, b=FAKE, K=128, g=128) == ARG
    assert gemv(L, x=MIS) == ALIGN
    assert gemv(L, c=MIS) == ALIGN
    assert gemv(L, s=MIS) == ALIGN
    assert gemv(L, y=MIS) == ALIGN
    # empty problems are valid no-ops
    assert gemv(L, M=0) == OK
    assert gemv(L, N=0) == OK


def test_gemm_validation(L):
    assert gemm(L, bits=2, b=None) == UNSUP
    assert gemm(L, bits=8, b=FAKE) == ARG          # INT8 takes no biases
    assert gemm(L, bits=1, b=None, K=192) == SHAPE  # Q1 prefill needs K % 128
    assert gemm(L, g=16) == UNSUP
    assert gemm(L, K=32) == SHAPE
    assert gemm(L, K=96) == SHAPE
    assert gemm(L, K=192, g=128) == SHAPE
    assert gemm(L, M=-3) == SHAPE
    assert gemm(L, x=None) == ARG
    assert gemm(L, b=None) == ARG
    assert gemm(L, x=MIS) == ALIGN
    assert gemm(L, y=MIS) == ALIGN
    assert gemm(L, M=0) == OK
    assert gemm(L, N=0) == OK


def test_pack_dequant_validation(L):
    assert L.qmm_pack(FAKE, FAKE, 4, 33, 4, None) == SHAPE
    assert L.qmm_pack(FAKE, FAKE, 4, 64, 2, None) == UNSUP
    assert L.qmm_pack(None, FAKE, 4, 64, 4, None) == ARG
    assert L.qmm_pack(MIS, FAKE, 4, 64, 4, None) == ALIGN
    assert L.qmm_pack(FAKE, FAKE, 0, 64, 4, None) == OK
    assert L.qmm_unpack(FAKE, None, 4, 64, 4, None) == ARG
    assert L.qmm_dequant(FAKE, FAKE, None, FAKE, 4, 64, 4, 64, None) == ARG
    assert L.qmm_dequant(FAKE, FAKE, None, FAKE, 4, 64, 8, 96, None) == UNSUP
    assert L.qmm_dequant(FAKE, FAKE, None, FAKE, 4, 96, 8, 64, None) == SHAPE


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(qmm, "_lib", None)
    monkeypatch.setattr(qmm, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        qmm.lib()


def argmax(L, x=FAKE, c=FAKE, s=FAKE, b=FAKE, i=FAKE, v=FAKE, M=1, N=64, K=128, bits=4, g=64, ws=FAKE,
           nbytes=1 << 20):
    return L.qmm_gemv_argmax(x, c, s, b, i, v, M, N, K, bits, g, ws, nbytes, None)


def test_timeout_hook_validation(L):
    assert L.qmm_test_timeout_next_decode(999) == ARG            # out of [1 us, 100 ms]
    assert L.qmm_test_timeout_next_decode(100_000_001) == ARG
    assert L.qmm_test_timeout_next_decode(-5) == ARG


def test_argmax_validation(L):
    need = L.qmm_gemv_argmax_workspace_size(2, 1000)
    assert need >= 2 * 1000 * 4 + 16
    assert L.qmm_gemv_argmax_workspace_size(-1, 5) == 0
    assert argmax(L, bits=3) == UNSUP
    assert argmax(L, M=0) == SHAPE                 # a greedy head needs at least one token
    assert argmax(L, M=9) == SHAPE
    assert argmax(L, N=0) == SHAPE
    assert argmax(L, K=0) == SHAPE
    assert argmax(L, i=None) == ARG
    assert argmax(L, ws=None) == ARG
    assert argmax(L, b=None) == ARG
    assert argmax(L, ws=MIS) == ALIGN
    assert argmax(L, i=ODD) == ALIGN               # idx and val need only 4-byte alignment
    assert argmax(L, v=ODD) == ALIGN
    assert argmax(L, M=2, x=MIS, i=ODD) == ALIGN
    assert argmax(L, M=2, N=1000, nbytes=need - 1) == SHAPE   # workspace too small


def test_quantize_gather_validation(L):
    assert L.qmm_quantize(FAKE, FAKE, FAKE, FAKE, 4, 64, 16, None) == UNSUP
    assert L.qmm_quantize(FAKE, FAKE, FAKE, FAKE, 4, 96, 64, None) == SHAPE
    assert L.qmm_quantize(FAKE, FAKE, FAKE, None, 4, 64, 64, None) == ARG
    assert L.qmm_quantize(MIS, FAKE, FAKE, FAKE, 4, 64, 64, None) == ALIGN
    assert L.qmm_quantize(FAKE, FAKE, FAKE, FAKE, 0, 64, 64, None) == OK
    assert L.qmm_gather_dequant(FAKE, -1, FAKE, FAKE, FAKE, FAKE, 4, 64, 4, 64, None) == SHAPE
    assert L.qmm_gather_dequant(FAKE, 3, FAKE, FAKE, None, FAKE, 4, 64, 4, 64, None) == ARG
    assert L.qmm_gather_dequant(FAKE, 3, FAKE, FAKE, FAKE, FAKE, 4, 64, 8, 64, None) == ARG
    assert L.qmm_gather_dequant(MIS, 3, FAKE, FAKE, FAKE, FAKE, 4, 64, 4, 64, None) == ALIGN
    assert L.qmm_gather_dequant(FAKE, 0, FAKE, FAKE, FAKE, FAKE, 4, 64, 4, 64, None) == OK
