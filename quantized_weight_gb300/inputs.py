"""Seeded synthetic inputs for the quantized matrix product.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests.  It draws random numbers and casts them to the storage types
(binary16, bfloat16, bytes); it holds none of the product's arithmetic: no
packing, no dequantization, no accumulation.

Draw order for one workload, from ``numpy.random.default_rng(seed)``:
codes, then scales, then biases (INT4 only), then x.

Distributions (the workloads the pages' models imply, with synthetic values):
  INT4 affine, group 64 : codes uniform in 0..15; scales binary16 of
                          U[0.001, 0.02]; bias = binary16(-8*scale + N(0, 1e-3))
                          with the standard deviation read as 1e-3
  INT8 symmetric, g 64  : codes uniform in -127..127; scales binary16 of U[1e-4, 5e-3]
  Q1 sign, group 128    : bits Bernoulli(0.5); scales binary16 of U[0.005, 0.05]
  x                     : float32 N(0, 1) (cast from float64, round to nearest);
                          the prefill contraction takes x rounded to bfloat16
                          (round to nearest even)
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    K: int
    N: int
    bits: int
    group: int
    prefill: bool = False
    seed: int = 0
    note: str = field(default="", compare=False)


# The shapes: a single decode matvec, a 2B-class MLP's up and down
# projections, an 8-bit small-batch sweep, a 27B-class FFN in binary Q1, and
# the prefill contraction at the MLP shape plus a tied output head.
WORKLOADS = {w.name: w for w in [
    Workload("decode_int4_k1024_n1024", 1, 1024, 1024, 4, 64,
             note="single decode matvec"),
    Workload("decode_int4_up_k2048_n6144", 1, 2048, 6144, 4, 64,
             note="2B-class MLP up-projection"),
    Workload("decode_int4_down_k6144_n2048", 1, 6144, 2048, 4, 64,
             note="2B-class MLP down-projection"),
    *[Workload(f"decode_int8_k4096_n4096_m{m}", m, 4096, 4096, 8, 64,
               note="small-batch 8-bit decode") for m in (1, 2, 4, 8)],
    Workload("decode_q1_k5120_n17408", 1, 5120, 17408, 1, 128,
             note="27B-class FFN, binary Q1"),
    Workload("prefill_int4_m1024_k2048_n6144", 1024, 2048, 6144, 4, 64, prefill=True,
             note="prefill at the MLP up-projection shape"),
    Workload("prefill_int4_m256_k2048_n151936", 256, 2048, 151936, 4, 64, prefill=True,
             note="prefill through a tied output head"),
    Workload("prefill_int8_m1024_k2048_n6144", 1024, 2048, 6144, 8, 64, prefill=True,
             note="8-bit prefill at the MLP up-projection shape"),
    Workload("prefill_q1_m1024_k5120_n17408", 1024, 5120, 17408, 1, 128, prefill=True,
             note="binary Q1 prefill at the 27B-class FFN shape"),
]}

SCALE_RANGE = {4: (0.001, 0.02), 8: (1e-4, 5e-3), 1: (0.005, 0.05)}
BIAS_NOISE_STD = 1e-3


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); uint16 bit patterns.

    A storage cast of the inputs, not a step of the product.  NaN stays NaN.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = ((u[nan] >> np.uint64(16)) | np.uint64(0x40)).astype(np.uint16)
    return r


def make(M: int, N: int, K: int, bits: int, group: int, seed: int = 0,
         prefill: bool = False, codes: str = "random") -> dict:
    """Draw one set of inputs.

    Returns a dict with
      codes  uint8  [N, K]   (int8 bit patterns for bits=8, 0/1 for bits=1)
      scales uint16 [N, K//group]  binary16 bit patterns
      biases uint16 [N, K//group] or None
      x      float32 [M, K]
      x_bf16 uint16 [M, K]  (bfloat16 bit patterns; only when prefill=True)
    ``codes`` may be "random" (the distributions above), "zeros" or "ones"
    (every code 0 / every code the format's all-ones value: 15, -1 or 1).
    """
    if bits not in (1, 4, 8):
        raise ValueError("bits must be 1, 4 or 8")
    if group <= 0 or K % group:
        raise ValueError("group must divide K")
    rng = np.random.default_rng(seed)
    G = K // group
    if codes == "random":
        if bits == 4:
            c = rng.integers(0, 16, size=(N, K), dtype=np.uint8)
        elif bits == 8:
            c = rng.integers(-127, 128, size=(N, K), dtype=np.int16).astype(np.int8).view(np.uint8)
        else:
            c = rng.integers(0, 2, size=(N, K), dtype=np.uint8)
    elif codes == "zeros":
        c = np.zeros((N, K), dtype=np.uint8)
    elif codes == "ones":
        c = np.full((N, K), {4: 15, 8: 0xFF, 1: 1}[bits], dtype=np.uint8)
    else:
        raise ValueError(codes)
    lo, hi = SCALE_RANGE[bits]
    s16 = rng.uniform(lo, hi, size=(N, G)).astype(np.float16)
    biases = None
    if bits == 4:
        noise = rng.normal(0.0, BIAS_NOISE_STD, size=(N, G))
        biases = (-8.0 * s16.astype(np.float64) + noise).astype(np.float16).view(np.uint16)
    x = rng.standard_normal(size=(M, K)).astype(np.float32)
    out = {"codes": c, "scales": s16.view(np.uint16), "biases": biases, "x": x}
    if prefill:
        out["x_bf16"] = f32_to_bf16_bits(x)
    return out


def make_workload(name: str, seed: int | None = None) -> dict:
    w = WORKLOADS[name]
    return make(w.M, w.N, w.K, w.bits, w.group, w.seed if seed is None else seed, w.prefill)
