"""GPU prefill product (tcgen05) against the FP64 oracle on the same bf16 x:
max per-row relative L2 <= 5e-3."""
import numpy as np
import pytest

from quantized_weight_gb300 import inputs
from helpers import rel_l2_rows, to_device

pytestmark = pytest.mark.gpu
TOL = 5e-3


@pytest.fixture(scope="module")
def qmm():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_weight_gb300 import build, qmm as q
    build.build()
    return q


SHAPES = [  # M, N, K, group: single and several tiles, ragged M and N, every BN variant
    (1, 128, 64, 64), (7, 200, 128, 64), (64, 256, 2048, 64), (100, 300, 1024, 128),
    (129, 1000, 512, 64), (256, 384, 2048, 64), (300, 130, 256, 64), (513, 1024, 2048, 64),
    (1024, 640, 1024, 128),
    # more tiles than SMs (ragged M and N, both group sizes); the first and the last two take token
    # tiles wider than 256 (two MMAs per k-slice into one accumulator), the last with a ragged
    # second half
    (700, 7000, 1024, 64), (513, 5000, 512, 128), (1000, 6144, 128, 64), (300, 19456, 128, 64),
    # group 32: two groups per 64-k step (each dequantizing thread's 32 k in one group), with a
    # group count that is a multiple of 8 (vector coefficient loads) and one that is not
    (129, 1000, 512, 32), (7, 200, 320, 32), (513, 2000, 1024, 32),
]


@pytest.mark.parametrize("M,N,K,group", SHAPES)
def test_small_shapes(qmm, oracle_mod, M, N, K, group):
    d = inputs.make(M, N, K, 4, group, seed=M + N + K, prefill=True)
    t = to_device(d, 4, with_bf16=True)
    p = qmm.pack(t["codes"], 4)
    y = qmm.gemm(t["x_bf16"], p, t["scales"], t["biases"], N, 4, group)
    qmm.check()
    y = y.cpu().numpy()
    ref = oracle_mod.qmm_bf16x(d["x_bf16"], oracle_mod.pack(d["codes"], 4), d["scales"], d["biases"],
                              N, K, 4, group)
    err = rel_l2_rows(y, ref)
    assert err <= TOL, (M, N, K, group, err)


FORMATS = [  # M, N, K, bits, group: INT8 and Q1 codes through the same tensor-core pipeline
    (1, 128, 128, 8, 64), (100, 300, 1024, 8, 128), (513, 1024, 2048, 8, 64), (700, 7000, 1024, 8, 64),
    (1, 128, 128, 1, 128), (129, 1000, 512, 1, 64), (300, 130, 256, 1, 128), (1024, 2048, 5120, 1, 128),
    (1000, 6144, 256, 1, 128),   # Q1 where INT4 and INT8 would take token tiles wider than 256
    (100, 300, 1024, 8, 32), (300, 1000, 320, 8, 32), (129, 1000, 512, 1, 32),   # group 32
]


@pytest.mark.parametrize("M,N,K,bits,group", FORMATS)
def test_int8_and_q1_prefill(qmm, oracle_mod, M, N, K, bits, group):
    d = inputs.make(M, N, K, bits, group, seed=M + N + K + bits, prefill=True)
    t = to_device(d, bits, with_bf16=True)
    p = qmm.pack(t["codes"], bits)
    y = qmm.gemm(t["x_bf16"], p, t["scales"], t["biases"], N, bits, group)
    qmm.check()
    y = y.cpu().numpy()
    ref = oracle_mod.qmm_bf16x(d["x_bf16"], oracle_mod.pack(d["codes"], bits), d["scales"], d["biases"],
                              N, K, bits, group)
    assert rel_l2_rows(y, ref) <= TOL, (M, N, K, bits, group)
    y2 = qmm.gemm(t["x_bf16"], p, t["scales"], t["biases"], N, bits, group).cpu().numpy()
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))


@pytest.mark.parametrize("name", ["prefill_int4_m1024_k2048_n6144", "prefill_int4_m256_k2048_n151936",
                                  "prefill_int8_m1024_k2048_n6144", "prefill_q1_m1024_k5120_n17408"])
def test_full_size_sampled(qmm, oracle_mod, name):
    w = inputs.WORKLOADS[name]
    d = inputs.make_workload(name)
    t = to_device(d, w.bits, with_bf16=True)
    p = qmm.pack(t["codes"], w.bits)
    y = qmm.gemm(t["x_bf16"], p, t["scales"], t["biases"], w.N, w.bits, w.group)
    qmm.check()
    rng = np.random.default_rng(123)
    rows = rng.choice(w.M, size=min(48, w.M), replace=False)
    cols = np.concatenate([rng.choice(w.N, size=60, replace=False), [0, w.N - 1]])
    ms, ns = np.repeat(rows, cols.size), np.tile(cols, rows.size)
    ref = oracle_mod.qmm_sampled(d["x_bf16"], oracle_mod.pack(d["codes"], w.bits), d["scales"], d["biases"],
                                 ms, ns, w.N, w.K, w.bits, w.group).reshape(rows.size, cols.size)
    got = y[torch_index(rows), :][:, torch_index(cols)].cpu().numpy()
    # relative L2 over the sampled entries of each row estimates the row's relative L2
    assert rel_l2_rows(got, ref) <= TOL
    y2 = qmm.gemm(t["x_bf16"], p, t["scales"], t["biases"], w.N, w.bits, w.group)
    import torch
    assert torch.equal(y, y2)                    # same bits on every run


def prefill_bound(d, bits, group, chunk=8192):
    """Element-wise error bound of the prefill product against the exact one
    on the same bf16 x: each weight is computed in float32 and rounded to
    bfloat16 (relative error <= 2^-9 + 2^-24, taken as 2^-8), the products of
    two bf16 values are exact in float32, and the float32 accumulation over K
    adds at most (K + 16) * 2^-23 (twice the sequential-sum bound, for the
    tensor core's accumulation order), all relative to sum_k |w_k| |x_k| with
    |w| <= |s| q + |b|.  Independent of the oracle; rows of W in chunks."""
    # a bf16 bit pattern is the upper half of the float32 with the same value
    ax = np.abs((d["x_bf16"].astype(np.uint32) << 16).view(np.float32).astype(np.float64))
    N, K = d["codes"].shape
    out = np.empty((ax.shape[0], N))
    for n0 in range(0, N, chunk):
        sl = slice(n0, min(N, n0 + chunk))
        sc = np.abs(d["scales"][sl].view(np.float16).astype(np.float64)).repeat(group, axis=1)
        c = d["codes"][sl]
        if bits == 4:
            mag = sc * c + np.abs(d["biases"][sl].view(np.float16).astype(np.float64)).repeat(group, axis=1)
        elif bits == 8:
            mag = sc * np.abs(c.view(np.int8).astype(np.float64))
        else:
            mag = sc
        out[:, sl] = ax @ mag.T
    return (2.0 ** -8 + (K + 16) * 2.0 ** -23) * out


# Every output of the full-size prefill shapes (the MLP up-projection at 1024
# tokens in INT4 and INT8, and 256 tokens through the tied 151936-row head)
# against the oracle's FP64 product on all host cores.
@pytest.mark.parametrize("name", ["prefill_int4_m1024_k2048_n6144", "prefill_int8_m1024_k2048_n6144",
                                  "prefill_int4_m256_k2048_n151936"])
def test_full_size_every_output(qmm, oracle_mod, name):
    w = inputs.WORKLOADS[name]
    d = inputs.make_workload(name)
    t = to_device(d, w.bits, with_bf16=True)
    p = qmm.pack(t["codes"], w.bits)
    y = qmm.gemm(t["x_bf16"], p, t["scales"], t["biases"], w.N, w.bits, w.group)
    qmm.check()
    y = y.cpu().numpy().astype(np.float64)
    ref = oracle_mod.qmm_bf16x(d["x_bf16"], oracle_mod.pack(d["codes"], w.bits), d["scales"], d["biases"],
                               w.N, w.K, w.bits, w.group)
    assert rel_l2_rows(y, ref) <= TOL
    assert np.all(np.abs(y - ref) <= prefill_bound(d, w.bits, w.group))


def torch_index(a):
    import torch
    return torch.as_tensor(np.asarray(a), device="cuda", dtype=torch.long)


def test_nan_in_x_propagates_to_its_row_only(qmm):
    M, N, K = 5, 256, 256
    d = inputs.make(M, N, K, 4, 64, seed=9, prefill=True)
    d["x_bf16"][2, 100] = 0x7FC0                   # bf16 NaN
    t = to_device(d, 4, with_bf16=True)
    p = qmm.pack(t["codes"], 4)
    y = qmm.gemm(t["x_bf16"], p, t["scales"], t["biases"], N, 4, 64).cpu().numpy()
    assert np.isnan(y[2]).all()
    assert np.isfinite(np.delete(y, 2, axis=0)).all()


def test_check_reports_ok_after_normal_runs(qmm):
    qmm.check()
