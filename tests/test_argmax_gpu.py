"""Greedy argmax head on the GPU.

Several indices can be "correct" when logits are within rounding of each
other, so the test checks what is unique and that the rest is valid:
  * the index is the argmax (NaN first, ties to the lower index) of the same
    library's logits, and val is that logit bit for bit;
  * against the FP64 oracle, the chosen logit is within the float32 error
    bound of the true maximum."""
import numpy as np
import pytest

from quantized_weight_gb300 import inputs
from helpers import to_device
from test_gemv_gpu import fp32_bound

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qmm():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_weight_gb300 import build, qmm as q
    build.build()
    return q


def np_argmax(y):
    """Reference order on float32 logits: NaN first, larger value, lower index."""
    nan = np.isnan(y)
    if nan.any():
        return int(np.argmax(nan))
    return int(np.argmax(y))                     # numpy returns the first of equal maxima


def run(qmm, d, bits, group, ws=None):
    import torch
    t = to_device(d, bits)
    p = qmm.pack(t["codes"], bits)
    M = d["x"].shape[0]
    N = d["codes"].shape[0]
    if ws is None:
        ws = qmm.argmax_workspace(M, N)
    idx, val = qmm.gemv_argmax(t["x"], p, t["scales"], t["biases"], N, bits, group, ws)
    y = qmm.gemv(t["x"], p, t["scales"], t["biases"], N, bits, group)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), val.cpu().numpy(), y.cpu().numpy(), ws


def valid_against_oracle(oracle_mod, d, bits, group, idx):
    N, K = d["codes"].shape
    ref = oracle_mod.qmm_f32x(d["x"], oracle_mod.pack(d["codes"], bits), d["scales"], d["biases"], N, K, bits, group)
    bound = fp32_bound(d, bits, group)
    for m in range(ref.shape[0]):
        i = idx[m]
        assert ref[m, i] + bound[m, i] >= np.max(ref[m] - bound[m]), (m, i)


@pytest.mark.parametrize("seed", [0, 1])
def test_tied_head_shape(qmm, oracle_mod, seed):
    w = inputs.WORKLOADS["prefill_int4_m256_k2048_n151936"]
    d = inputs.make(1, w.N, w.K, 4, 64, seed=seed)
    idx, val, y, _ = run(qmm, d, 4, 64)
    assert idx[0] == np_argmax(y[0])
    assert val.view(np.uint32)[0] == y[0, idx[0]].view(np.uint32)
    valid_against_oracle(oracle_mod, d, 4, 64, idx)


@pytest.mark.parametrize("bits,group", [(4, 64), (8, 64), (4, 128), (8, 32)])
@pytest.mark.parametrize("N", [1, 37, 1001, 20000])
def test_fused_small_shapes(qmm, oracle_mod, bits, group, N):
    d = inputs.make(1, N, 1024, bits, group, seed=N + bits + group)
    idx, val, y, _ = run(qmm, d, bits, group)
    assert idx[0] == np_argmax(y[0]) and val[0] == y[0, idx[0]]
    valid_against_oracle(oracle_mod, d, bits, group, idx)


@pytest.mark.parametrize("M", [1, 2, 5, 8])
def test_q1_and_batches(qmm, oracle_mod, M):
    d = inputs.make(M, 3000, 1024, 1, 128, seed=M)
    idx, val, y, _ = run(qmm, d, 1, 128)
    valid_against_oracle(oracle_mod, d, 1, 128, idx)
    d = inputs.make(M, 5000, 2048, 4, 64, seed=M + 10)
    idx, val, y, _ = run(qmm, d, 4, 64)
    for m in range(M):
        assert idx[m] == np_argmax(y[m]) and val[m] == y[m, idx[m]]
    valid_against_oracle(oracle_mod, d, 4, 64, idx)


def test_ties_go_to_the_lower_index_across_ctas(qmm):
    N, K = 40000, 1024
    base = inputs.make(1, N, K, 4, 64, seed=9)
    _, _, y, _ = run(qmm, base, 4, 64)
    top = np_argmax(y[0])
    for a, b in [(7, N - 3), (N - 3, 7), (20011, 20012)]:
        d = {k: (None if v is None else v.copy()) for k, v in base.items()}
        for key in ("codes", "scales", "biases"):
            d[key][a] = d[key][top]
            d[key][b] = d[key][top]
        idx, val, y2, _ = run(qmm, d, 4, 64)
        assert y2[0, a] == y2[0, b] and idx[0] == np_argmax(y2[0]) == min(a, b, top)


def test_nan_logits_rank_first(qmm):
    N, K = 3000, 512
    d = inputs.make(1, N, K, 4, 64, seed=4)
    d["scales"][1234, 3] = 0x7E00                  # one NaN scale: one NaN logit
    d["scales"][2345, 0] = 0x7E00
    idx, val, y, _ = run(qmm, d, 4, 64)
    assert idx[0] == 1234 and np.isnan(val[0])
    d["x"][0, 5] = np.nan                          # every logit NaN: the first row wins
    idx, val, y, _ = run(qmm, d, 4, 64)
    assert idx[0] == 0 and np.isnan(val[0])


def test_workspace_is_left_ready(qmm):
    import torch
    d = inputs.make(1, 7000, 2048, 4, 64, seed=2)
    ws = None
    first = None
    for _ in range(4):
        idx, val, y, ws = run(qmm, d, 4, 64, ws)
        first = idx[0] if first is None else first
        assert idx[0] == first
    assert int(ws[:4].view(torch.int32)[0].item()) == 0     # the CTA counter is back to zero
