"""GPU decode product against the FP64 oracle: max per-row relative L2 <= 1e-5."""
import numpy as np
import pytest

from quantized_weight_gb300 import inputs
from helpers import rel_l2_rows, to_device

pytestmark = pytest.mark.gpu
TOL = 1e-5


@pytest.fixture(scope="module")
def qmm():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_weight_gb300 import build, qmm as q
    build.build()
    return q


def fp32_bound(d, bits, group):
    """Forward error bound of the kernel's float32 evaluation, per output:
    (K + 16) * 2^-24 * sum_k (|s q_k| + |b|) |x_k|  -- every float32 operation
    on the way rounds once, and the group bias is factored out of the sum, so
    the bound is taken over |s q| and |b| separately.  Independent of the oracle."""
    s = d["scales"].view(np.float16).astype(np.float64).repeat(group, axis=1)
    c = d["codes"]
    if bits == 4:
        q = c.astype(np.float64)
        mag = np.abs(s) * q + np.abs(d["biases"].view(np.float16).astype(np.float64)).repeat(group, axis=1)
    elif bits == 8:
        mag = np.abs(s) * np.abs(c.view(np.int8).astype(np.float64))
    else:
        mag = np.abs(s)
    K = c.shape[1]
    return (K + 16) * 2.0 ** -24 * (np.abs(d["x"].astype(np.float64)) @ mag.T)


def run_case(qmm, oracle_mod, M, N, K, bits, group, seed):
    d = inputs.make(M, N, K, bits, group, seed=seed)
    t = to_device(d, bits)
    p = qmm.pack(t["codes"], bits)
    y = qmm.gemv(t["x"], p, t["scales"], t["biases"], N, bits, group).cpu().numpy()
    ref = oracle_mod.qmm_f32x(d["x"], oracle_mod.pack(d["codes"], bits), d["scales"], d["biases"],
                             N, K, bits, group)
    return y, ref, t, p, d


# small shapes spanning several K-tiles, ragged K tails and ragged row blocks
# (K a whole number of 1024-weight segments, 512 for INT8, takes the streaming
# kernel at M = 1; the other K values take the register-fed kernel)
SMALL = [
    (4, 64, [128, 1088, 3072]), (4, 32, [96, 2080]), (4, 128, [1152, 2048]),
    (8, 64, [128, 1088, 2048]), (8, 32, [544, 1024]), (8, 128, [2176]),
    (1, 128, [128, 2176, 5120]), (1, 64, [1152, 2048]), (1, 32, [384]),
]


@pytest.mark.parametrize("bits,group,Ks", SMALL)
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8])
def test_small_shapes(qmm, oracle_mod, bits, group, Ks, M):
    for K in Ks:
        for N in (1, 37, 1001):
            y, ref, _, _, d = run_case(qmm, oracle_mod, M, N, K, bits, group, seed=M * 7 + N + K)
            # every element within the float32 forward-error bound
            assert np.all(np.abs(y - ref) <= fp32_bound(d, bits, group)), (M, N, K, bits, group)
            # the 1e-5 per-row relative L2 on rows long enough for a norm; a
            # one-element row is a single, possibly cancelling, sum
            if N >= 32:
                assert rel_l2_rows(y, ref) <= TOL, (M, N, K, bits, group)


DECODE = ["decode_int4_k1024_n1024", "decode_int4_up_k2048_n6144", "decode_int4_down_k6144_n2048",
          "decode_int8_k4096_n4096_m1", "decode_int8_k4096_n4096_m2", "decode_int8_k4096_n4096_m4",
          "decode_int8_k4096_n4096_m8", "decode_q1_k5120_n17408"]


@pytest.mark.parametrize("name", DECODE)
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_full_size_workloads(qmm, oracle_mod, name, seed):
    w = inputs.WORKLOADS[name]
    y, ref, t, p, d = run_case(qmm, oracle_mod, w.M, w.N, w.K, w.bits, w.group, seed)
    assert rel_l2_rows(y, ref) <= TOL, name
    assert np.all(np.abs(y - ref) <= fp32_bound(d, w.bits, w.group)), name
    # fixed reduction order: the same call gives the same bits
    y2 = qmm.gemv(t["x"], p, t["scales"], t["biases"], w.N, w.bits, w.group).cpu().numpy()
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))


def test_nan_and_inf_in_x_propagate(qmm):
    import torch
    M, N, K = 3, 64, 256
    for bits, group in [(4, 64), (8, 64), (1, 128)]:
        d = inputs.make(M, N, K, bits, group, seed=5)
        d["x"][1, 17] = np.nan
        d["x"][2, 3] = np.inf
        t = to_device(d, bits)
        p = qmm.pack(t["codes"], bits)
        y = qmm.gemv(t["x"], p, t["scales"], t["biases"], N, bits, group).cpu().numpy()
        assert np.isfinite(y[0]).all()
        assert np.isnan(y[1]).all()
        assert (~np.isfinite(y[2])).all()


def test_empty_and_degenerate(qmm):
    import torch
    dev = "cuda"
    # K == 0: empty sums, y = 0
    y = torch.full((2, 5), 7.0, device=dev)
    s = torch.empty((5, 0), dtype=torch.float16, device=dev)
    qmm.gemv(torch.empty((2, 0), device=dev), torch.empty((5, 0), dtype=torch.int32, device=dev), s, s,
             5, 4, 64, out=y)
    assert (y.cpu() == 0).all()
    # N == 0 and M == 0 are no-ops
    qmm.gemv(torch.zeros((1, 64), device=dev), torch.empty((0, 8), dtype=torch.int32, device=dev),
             torch.empty((0, 1), dtype=torch.float16, device=dev), torch.empty((0, 1), dtype=torch.float16, device=dev),
             0, 4, 64)
    keep = torch.full((0, 3), 1.0, device=dev)
    qmm.gemv(torch.zeros((0, 64), device=dev), torch.zeros((3, 8), dtype=torch.int32, device=dev),
             torch.zeros((3, 1), dtype=torch.float16, device=dev), torch.zeros((3, 1), dtype=torch.float16, device=dev),
             3, 4, 64, out=keep)


def test_rejected_call_leaves_y_untouched(qmm):
    import torch
    y = torch.full((1, 64), 3.0, device="cuda")
    with pytest.raises(qmm.QmmError):
        # K=96 is not a multiple of the group: rejected before any launch
        qmm.gemv(torch.zeros((1, 96), device="cuda"), torch.zeros((64, 12), dtype=torch.int32, device="cuda"),
                 torch.zeros((64, 1), dtype=torch.float16, device="cuda"),
                 torch.zeros((64, 1), dtype=torch.float16, device="cuda"), 64, 4, 64, out=y)
    assert (y.cpu() == 3.0).all()


def test_chained_products_see_the_previous_output(qmm):
    """Back-to-back decode products overlap through programmatic dependent
    launch; the second must still read the first one's finished output."""
    import torch
    K1, N1, N2 = 2048, 6144, 2048
    a = inputs.make(1, N1, K1, 4, 64, seed=21)
    b = inputs.make(1, N2, N1, 4, 64, seed=22)
    ta, tb = to_device(a, 4), to_device(b, 4)
    pa, pb = qmm.pack(ta["codes"], 4), qmm.pack(tb["codes"], 4)
    torch.cuda.synchronize()
    for _ in range(3):
        y1 = qmm.gemv(ta["x"], pa, ta["scales"], ta["biases"], N1, 4, 64)
        y2 = qmm.gemv(y1, pb, tb["scales"], tb["biases"], N2, 4, 64)
        torch.cuda.synchronize()
        y1s = y1.clone()
        torch.cuda.synchronize()
        y2s = qmm.gemv(y1s, pb, tb["scales"], tb["biases"], N2, 4, 64)
        torch.cuda.synchronize()
        assert torch.equal(y2, y2s)


# small-batch decode at MLP-projection shapes: several 32-row blocks per SM,
# one or two token passes, ragged row blocks
BATCH = [(2, 6144, 2048, 4, 64), (4, 6144, 2048, 4, 64), (8, 2048, 6144, 4, 64), (3, 8192, 4096, 8, 64),
         (8, 8192, 1024, 8, 32), (5, 4100, 2048, 8, 128), (7, 1000, 4096, 4, 128),
         # INT8, 5..8 tokens in one pass: the benchmark shape, fewer rows than SMs, a ragged slab
         (8, 4096, 4096, 8, 64), (6, 150, 512, 8, 64), (7, 2333, 3072, 8, 64),
         # INT8 at the benchmark's two tokens, ragged slabs of 10-16 rows
         (2, 4096, 4096, 8, 64), (4, 3000, 2048, 8, 64), (3, 4864, 1024, 8, 32), (6, 2500, 512, 8, 128),
         # INT8 slabs too long for the streamed kernel's token passes (wide layout): the fallbacks
         (6, 40000, 1024, 8, 64), (2, 40000, 1024, 8, 64)]


# two to eight tokens with K split over a cluster of ks CTAs (ks = K / 1024
# rounded up to a whole split: 2, 3, 4, 5, 6, 8), each CTA a K slice of the
# cluster's rows: many ring laps (40000 rows), clusters left with no rows
# (N = 5), binary codes at the 27B FFN shape, and INT4 shapes whose resident
# slab does not fit (the split is their fallback)
SPLIT = [(8, 5, 4096, 8, 64), (5, 4000, 8192, 8, 64), (6, 3001, 2048, 8, 128), (7, 2333, 3072, 8, 64),
         (2, 17408, 5120, 1, 128), (3, 4000, 5120, 1, 128), (8, 17408, 5120, 1, 128), (4, 7000, 4096, 1, 128),
         (2, 3000, 2048, 1, 64), (8, 2048, 6144, 4, 64), (7, 1000, 6144, 4, 64),
         (4, 2048, 6144, 4, 64), (3, 1000, 4096, 4, 32), (3, 777, 4096, 8, 64), (4, 2000, 2048, 8, 128)]


@pytest.mark.parametrize("M,N,K,bits,group", SPLIT)
def test_k_split_over_a_cluster(qmm, oracle_mod, M, N, K, bits, group):
    y, ref, t, p, d = run_case(qmm, oracle_mod, M, N, K, bits, group, seed=M * N + K)
    assert np.all(np.abs(y - ref) <= fp32_bound(d, bits, group)), (M, N, K, bits, group)
    if N >= 32:
        assert rel_l2_rows(y, ref) <= TOL
    y2 = qmm.gemv(t["x"], p, t["scales"], t["biases"], N, bits, group).cpu().numpy()
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))     # fixed order across the cluster


# The ring layouts on cold weights (every product reads fresh tensors, larger
# than L2 together): copies into a ring slot may land out of order, which once
# let a consumer take a slot's previous lap for its own.  Every output is
# checked against the float32 bound.
RING_COLD = [(1, 151936, 2048, 4, 64), (8, 4096, 4096, 8, 64), (2, 17408, 5120, 1, 128)]


@pytest.mark.parametrize("M,N,K,bits,group", RING_COLD)
def test_ring_layouts_on_cold_weights(qmm, oracle_mod, M, N, K, bits, group):
    for seed in range(3):
        y, ref, t, p, d = run_case(qmm, oracle_mod, M, N, K, bits, group, seed=100 + seed)
        assert np.all(np.abs(y - ref) <= fp32_bound(d, bits, group)), (M, N, K, bits, group, seed)


# M = 1 slabs whose coefficients travel with each code stage (more than 16 KB
# of coefficients per CTA), a ragged last stage included
STAGED = [(40000, 1024, 4, 64), (40013, 1024, 4, 32), (41000, 4096, 8, 64)]


@pytest.mark.parametrize("N,K,bits,group", STAGED)
def test_large_slabs_with_staged_coefficients(qmm, oracle_mod, N, K, bits, group):
    y, ref, t, p, d = run_case(qmm, oracle_mod, 1, N, K, bits, group, seed=N + K)
    assert np.all(np.abs(y - ref) <= fp32_bound(d, bits, group)), (N, K, bits, group)
    assert rel_l2_rows(y, ref) <= TOL


@pytest.mark.parametrize("M,N,K,bits,group", BATCH)
def test_small_batch_projection_shapes(qmm, oracle_mod, M, N, K, bits, group):
    y, ref, t, p, d = run_case(qmm, oracle_mod, M, N, K, bits, group, seed=M + N + K)
    assert np.all(np.abs(y - ref) <= fp32_bound(d, bits, group)), (M, N, K, bits, group)
    assert rel_l2_rows(y, ref) <= TOL
    y2 = qmm.gemv(t["x"], p, t["scales"], t["biases"], N, bits, group).cpu().numpy()
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))
