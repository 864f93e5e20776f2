"""The shared input module's storage casts, pinned to an independent
implementation: the bfloat16 rounding of the prefill activations against
PyTorch's CPU float32 -> bfloat16 conversion (round to nearest, ties to even)."""
import numpy as np
import torch

from quantized_weight_gb300 import inputs


def torch_bf16_bits(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def check(x):
    ours, ref = inputs.f32_to_bf16_bits(x), torch_bf16_bits(x)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    # NaN stays NaN (exponent all ones, nonzero mantissa); payloads may differ
    for r in (ours[nan], ref[nan]):
        assert np.all((r & 0x7F80) == 0x7F80) and np.all((r & 0x7F) != 0)


def test_random_normals_and_wide_magnitudes():
    rng = np.random.default_rng(3)
    check(rng.standard_normal(100000).astype(np.float32))
    check((rng.standard_normal(20000) * 10.0 ** rng.uniform(-44, 38, 20000)).astype(np.float32))


def test_ties_go_to_even_and_neighbours_round_to_nearest():
    rng = np.random.default_rng(4)
    hi = rng.integers(0, 0x7F7F, 4000, dtype=np.uint32) << 16
    sign = rng.integers(0, 2, 4000, dtype=np.uint32) << 31
    for low in (0x8000, 0x7FFF, 0x8001, 0x0001, 0xFFFF):
        check(((hi | sign) | np.uint32(low)).view(np.float32))


def test_special_values():
    bits = np.array([0x00000000, 0x80000000, 0x00000001, 0x807FFFFF, 0x00008000, 0x00018000,
                     0x7F7FFFFF, 0xFF7FFFFF, 0x7F7F7FFF, 0x7F7F8000, 0x7F800000, 0xFF800000,
                     0x7FC00000, 0xFFC00000, 0x7F800001, 0x7FBFFFFF], dtype=np.uint32)
    check(bits.view(np.float32))
    ours = inputs.f32_to_bf16_bits(bits.view(np.float32))
    assert ours[6] == 0x7F80 and ours[7] == 0xFF80         # overflow of the largest float rounds to infinity
    assert ours[1] == 0x8000                                # -0 keeps its sign
