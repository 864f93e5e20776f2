"""GPU INT4 quantizer and row gather-dequant against the oracle: bit-exact.

The quantizer's integer codes are decided in float32 on both sides (the
oracle states the same steps in C float), so codes, scales and biases must
match bit for bit; the gather computes each element exactly as the
dequantizer does."""
import numpy as np
import pytest

from quantized_weight_gb300 import inputs
from helpers import to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qmm():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_weight_gb300 import build, qmm as q
    build.build()
    return q


def _quantize_both(qmm, oracle_mod, w, group):
    import torch
    p, s, b = qmm.quantize(torch.from_numpy(w).cuda(), group)
    N, K = w.shape
    codes = qmm.unpack(p, N, K, 4).cpu().numpy()
    rc, rs, rb = oracle_mod.quantize_affine4_f32(w, group)
    return codes, s.cpu().numpy().view(np.uint16), b.cpu().numpy().view(np.uint16), rc, rs, rb


@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("N,K", [(1, 128), (37, 256), (300, 2048), (1001, 1152)])
def test_quantize_bit_exact(qmm, oracle_mod, N, K, group):
    if K % group:
        pytest.skip("K not a multiple of the group")
    rng = np.random.default_rng(N * 7 + K + group)
    w = (rng.standard_normal((N, K)) * rng.uniform(0.01, 2.0, (N, 1)) + rng.normal(0, 0.1, (N, 1)))
    w = w.astype(np.float32)
    c, s, b, rc, rs, rb = _quantize_both(qmm, oracle_mod, w, group)
    assert np.array_equal(s, rs) and np.array_equal(b, rb)
    assert np.array_equal(c, rc)


def test_quantize_edge_groups(qmm, oracle_mod):
    rng = np.random.default_rng(11)
    w = rng.standard_normal((12, 128)).astype(np.float32)
    w[0, :64] = 0.5                                    # constant group
    w[1, :64] = -0.0
    w[1, 3] = 0.0                                      # -0 and +0 in one group
    w[2, 7] = np.nan                                   # NaN weight
    w[3, :64] = np.nan                                 # all-NaN group
    w[4, :64] = np.float32(1e-7) * np.arange(64)       # subnormal binary16 range
    w[5, :64] = 70000.0 + np.arange(64)                # bias overflows binary16
    w[6, :64] = 3.0e4 * np.sign(np.arange(64) - 31.5)  # large range, scale near the binary16 top
    w[7, 10] = np.inf                                  # infinite weight: scale becomes inf
    j = np.arange(64) % 16
    j[1] = 15
    w[8, :64] = np.float32(-1.0) + j.astype(np.float32) * np.float32(0.0625)   # exact grid
    c, s, b, rc, rs, rb = _quantize_both(qmm, oracle_mod, w, 64)
    assert np.array_equal(s, rs) and np.array_equal(b, rb)
    assert np.array_equal(c, rc)
    assert np.array_equal(c[8, :64], j)
    assert rb[3, 0] == 0x7E00 and (c[3, :64] == 0).all()


def test_quantize_quotients_next_to_half_integers(qmm, oracle_mod):
    """Weights placed a few float32 steps from b + (k + 1/2) * s, with scales
    that are not powers of two: the quotient (w - b) / s then sits next to a
    rounding boundary, where only the correctly rounded division decides q."""
    rng = np.random.default_rng(23)
    rows = []
    while len(rows) < 96:
        b16 = np.float16(rng.uniform(-1.0, 0.0))
        s16 = np.float16(rng.uniform(0.003, 0.05))
        b, sc = np.float32(b16), np.float32(s16)
        mx = np.float32(np.float64(b) + 15.0 * np.float64(sc))
        if np.float16(np.float32(np.float32(mx - b) / np.float32(15.0))) != s16:
            continue                                   # the group's own range must give back this scale
        row = np.empty(64, np.float32)
        row[0], row[1] = b, mx
        for i in range(2, 64):
            k = i % 15
            if i % 4 == 0:                              # just outside +-1e-5 of the half-integer
                off = (2e-5 if i % 8 == 0 else -2e-5) * max(1.0, k + 0.5)
                row[i] = np.float32(np.float64(b) + (k + 0.5 + off) * np.float64(sc))
                continue
            t = np.float32(np.float64(b) + (k + 0.5) * np.float64(sc))
            for _ in range(int(rng.integers(0, 4))):    # up to three steps up or down
                t = np.nextafter(t, np.float32(np.inf) if i % 2 else np.float32(-np.inf), dtype=np.float32)
            row[i] = t
        rows.append(row)
    w = np.stack(rows)
    c, s, b, rc, rs, rb = _quantize_both(qmm, oracle_mod, w, 64)
    assert np.array_equal(s, rs) and np.array_equal(b, rb)
    assert np.array_equal(c, rc)


def test_quantize_then_products_roundtrip(qmm, oracle_mod):
    """Quantized weights feed the products unchanged: the GPU product of the
    GPU-quantized matrix equals the oracle product of the oracle-quantized one."""
    import torch
    rng = np.random.default_rng(5)
    w = rng.standard_normal((640, 1024)).astype(np.float32) * np.float32(0.05)
    p, s, b = qmm.quantize(torch.from_numpy(w).cuda(), 64)
    x = rng.standard_normal((1, 1024)).astype(np.float32)
    y = qmm.gemv(torch.from_numpy(x).cuda(), p, s, b, 640, 4, 64).cpu().numpy()
    rc, rs, rb = oracle_mod.quantize_affine4_f32(w, 64)
    ref = oracle_mod.qmm_f32x(x, oracle_mod.pack(rc, 4), rs, rb, 640, 1024, 4, 64)
    assert np.linalg.norm(y - ref) / np.linalg.norm(ref) <= 1e-5


@pytest.mark.parametrize("bits,group", [(4, 64), (4, 128), (8, 64), (1, 128), (4, 32)])
def test_gather_dequant_bit_exact(qmm, oracle_mod, bits, group):
    import torch
    N, K, T = 1000, 512, 77
    d = inputs.make(1, N, K, bits, group, seed=bits + group)
    t = to_device(d, bits)
    p = qmm.pack(t["codes"], bits)
    rng = np.random.default_rng(bits * group)
    ids = rng.integers(0, N, T).astype(np.int32)
    ids[:5] = [0, N - 1, 3, 3, 0]                       # ends of the table and repeats
    out = qmm.gather_dequant(torch.from_numpy(ids).cuda(), p, t["scales"], t["biases"], N, K, bits,
                             group).cpu().numpy()
    ref = oracle_mod.dequant(oracle_mod.pack(d["codes"], bits), d["scales"], d["biases"], N, K, bits, group)
    assert np.array_equal(out.view(np.uint32), ref[ids].astype(np.float32).view(np.uint32))


def test_gather_dequant_bad_ids_and_signed_zero(qmm, oracle_mod):
    import torch
    N, K, g = 4, 64, 32
    codes = np.zeros((N, K), dtype=np.uint8)
    codes[:, 1::2] = 5
    sc = np.full((N, K // g), 0x3C00, dtype=np.uint16)
    bi = np.zeros((N, K // g), dtype=np.uint16)
    bi[1, :] = 0x8000                                   # -0.0 bias: code 0 gives +0
    sc[2, :] = 0x8000
    bi[2, :] = 0x8000                                   # -0 * 0 + -0 = -0
    bi[3, :] = 0x8001                                   # tiny negative subnormal bias
    d = {"codes": codes, "scales": sc, "biases": bi, "x": np.zeros((1, K), np.float32)}
    t = to_device(d, 4)
    p = qmm.pack(t["codes"], 4)
    ids = np.array([1, 2, -1, 3, 4, 1 << 30, 0, 2], dtype=np.int32)
    out = qmm.gather_dequant(torch.from_numpy(ids).cuda(), p, t["scales"], t["biases"], N, K, 4, g)
    out = out.cpu().numpy()
    ref = oracle_mod.dequant(oracle_mod.pack(codes, 4), sc, bi, N, K, 4, g).astype(np.float32)
    ok = (ids >= 0) & (ids < N)
    assert np.array_equal(out[ok].view(np.uint32), ref[ids[ok]].view(np.uint32))
    assert np.isnan(out[~ok]).all()
    assert not np.signbit(out[0, 0]) and np.signbit(out[1, 0]) and np.signbit(out[3, 0]) and out[3, 0] != 0


def test_gather_dequant_empty_is_a_noop(qmm):
    import torch
    p = torch.zeros((3, 8), dtype=torch.int32, device="cuda")
    s = torch.zeros((3, 1), dtype=torch.float16, device="cuda")
    out = qmm.gather_dequant(torch.empty(0, dtype=torch.int32, device="cuda"), p, s, s, 3, 64, 4, 64)
    assert out.shape == (0, 64)
