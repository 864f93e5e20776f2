"""CPU oracle for the weight-only quantized matrix product (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product (``quantized_weight_gb300``) never
does, and this package never imports the product: the two share no code.

The arithmetic lives in ``qmm_oracle.c`` (plain C, double precision); this
module only compiles it with gcc and marshals numpy arrays through ctypes.
"""
from .oracle import (  # noqa: F401
    build,
    lib_path,
    half_to_double,
    bf16_to_double,
    pack,
    unpack,
    dequant,
    qmm_f32x,
    qmm_bf16x,
    qmm_sampled,
    quantize_affine4,
    float_to_half,
    quantize_affine4_f32,
)
