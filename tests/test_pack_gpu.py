"""GPU pack / unpack / dequant against the oracle: bit-exact."""
import numpy as np
import pytest

from quantized_weight_gb300 import inputs
from helpers import to_device

pytestmark = pytest.mark.gpu

SHAPES = [(1, 128), (7, 256), (33, 1024), (129, 4096)]


@pytest.fixture(scope="module")
def qmm():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_weight_gb300 import build, qmm as q
    build.build()
    return q


@pytest.mark.parametrize("bits", [1, 4, 8])
@pytest.mark.parametrize("N,K", SHAPES)
def test_pack_matches_oracle_and_roundtrips(qmm, oracle_mod, bits, N, K):
    d = inputs.make(1, N, K, bits, 32, seed=N + K + bits)
    t = to_device(d, bits)
    packed = qmm.pack(t["codes"], bits)
    ref = oracle_mod.pack(d["codes"], bits)
    assert np.array_equal(packed.cpu().numpy().view(np.uint32), ref)
    back = qmm.unpack(packed, N, K, bits)
    assert np.array_equal(back.cpu().numpy(), d["codes"])


def test_pack_ignores_bits_above_the_width(qmm):
    import torch
    c = torch.full((2, 64), 0xF7, dtype=torch.uint8, device="cuda")
    assert (qmm.pack(c, 4).cpu().numpy().view(np.uint32) == 0x77777777).all()
    assert (qmm.pack(c, 1).cpu().numpy().view(np.uint32) == 0xFFFFFFFF).all()


@pytest.mark.parametrize("bits,group", [(4, 32), (4, 64), (4, 128), (8, 64), (8, 128), (1, 32), (1, 128)])
def test_dequant_bit_exact(qmm, oracle_mod, bits, group):
    N, K = 37, 512
    d = inputs.make(1, N, K, bits, group, seed=bits * 1000 + group)
    t = to_device(d, bits)
    p = qmm.pack(t["codes"], bits)
    w = qmm.dequant(p, t["scales"], t["biases"], N, K, bits, group).cpu().numpy()
    ref = oracle_mod.dequant(oracle_mod.pack(d["codes"], bits), d["scales"], d["biases"], N, K, bits, group)
    # the exact weight rounded once to float32 is what the kernel must produce
    assert np.array_equal(w.view(np.uint32), ref.astype(np.float32).view(np.uint32))


def test_dequant_signed_zero_and_subnormal_coefficients(qmm, oracle_mod):
    """Fixtures after the exact-decoder lesson on the "Pushing the limits of
    legacy hardware" page: tiny negative coefficients, signed zeros and
    binary16 subnormals must survive dequantization bit for bit."""
    import torch
    N, K, g = 8, 64, 32
    codes = np.zeros((N, K), dtype=np.uint8)
    codes[:, 1::2] = np.arange(1, 16)[np.arange(K // 2) % 15][None, :]
    sc = np.full((N, K // g), 0x3C00, dtype=np.uint16)          # 1.0
    bi = np.zeros((N, K // g), dtype=np.uint16)
    sc[0, :] = 0x0001                 # smallest positive subnormal scale
    sc[1, :] = 0x83FF                 # largest negative subnormal scale
    bi[2, :] = 0x8000                 # -0.0 bias: code 0 with s=1 gives +0 + -0 = +0
    sc[3, :] = 0x8000                 # -0.0 scale, -0.0 bias: -0*q + -0 = -0
    bi[3, :] = 0x8000
    bi[4, :] = 0x8001                 # tiny negative subnormal bias
    sc[5, :] = 0x7BFF                 # largest finite scale
    bi[5, :] = 0xFBFF
    d = {"codes": codes, "scales": sc, "biases": bi, "x": np.zeros((1, K), np.float32)}
    t = to_device(d, 4)
    p = qmm.pack(t["codes"], 4)
    w = qmm.dequant(p, t["scales"], t["biases"], N, K, 4, g).cpu().numpy()
    ref = oracle_mod.dequant(oracle_mod.pack(codes, 4), sc, bi, N, K, 4, g).astype(np.float32)
    assert np.array_equal(w.view(np.uint32), ref.view(np.uint32))
    assert np.signbit(w[3, 0]) and not np.signbit(w[2, 0])
    assert np.signbit(w[4, 0]) and w[4, 0] != 0.0
