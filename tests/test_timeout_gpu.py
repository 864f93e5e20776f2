"""A bounded device wait that runs out, on the GPU, without faulting or
hanging it: the library's test hook makes the next tensor-core decode launch
wait on a barrier that nothing completes, with a limit of a fraction of a
millisecond.  The launch must write no output, wait for its own copies in
flight, and report QMM_ERR_DEVICE_TIMEOUT through qmm_check exactly once;
the next call must run normally and match the oracle.  Both ways the decode
kernel holds the weights are covered: a resident slab per CTA (the MLP
shape) and a ring of stages with a producer warp (the tied-head shape), and
the greedy head's work area stays usable after an aborted call."""
import numpy as np
import pytest

from quantized_weight_gb300 import inputs
from helpers import to_device
from test_gemv_gpu import fp32_bound

pytestmark = pytest.mark.gpu

TIMEOUT = -6
SENTINEL = 0x7FC0BEEF            # a NaN bit pattern no product produces


@pytest.fixture(scope="module")
def qmm():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_weight_gb300 import build, qmm as q
    build.build()
    q.check()                     # start from a clean status
    return q


def expect_timeout(qmm):
    with pytest.raises(qmm.QmmError) as e:
        qmm.check()
    assert e.value.status == TIMEOUT
    qmm.check()                   # the record was cleared: the next check is clean


@pytest.mark.parametrize("N,K", [(6144, 2048), (151936, 2048)])
def test_decode_wait_runs_out_then_the_next_call_is_normal(qmm, oracle_mod, N, K):
    import torch
    d = inputs.make(1, N, K, 4, 64, seed=N + K)
    t = to_device(d, 4)
    p = qmm.pack(t["codes"], 4)
    y = torch.full((1, N), 0, dtype=torch.int32, device="cuda").fill_(SENTINEL).view(torch.float32)
    torch.cuda.synchronize()
    qmm.test_timeout_next_decode(200_000)
    qmm.gemv(t["x"], p, t["scales"], t["biases"], N, 4, 64, out=y)
    expect_timeout(qmm)
    assert bool((y.view(torch.int32) == SENTINEL).all())          # nothing was written
    y2 = qmm.gemv(t["x"], p, t["scales"], t["biases"], N, 4, 64, out=y)
    qmm.check()
    got = y2.cpu().numpy().astype(np.float64)
    ref = oracle_mod.qmm_f32x(d["x"], oracle_mod.pack(d["codes"], 4), d["scales"], d["biases"], N, K, 4, 64)
    assert np.all(np.abs(got - ref) <= fp32_bound(d, 4, 64))


def test_argmax_head_wait_runs_out_and_its_workspace_stays_usable(qmm, oracle_mod):
    N, K = 151936, 2048
    d = inputs.make(1, N, K, 4, 64, seed=3)
    t = to_device(d, 4)
    p = qmm.pack(t["codes"], 4)
    ws = qmm.argmax_workspace(1, N)
    qmm.test_timeout_next_decode(200_000)
    i0, v0 = qmm.gemv_argmax(t["x"], p, t["scales"], t["biases"], N, 4, 64, ws)
    expect_timeout(qmm)
    assert int(i0.item()) == 2147483647 and float(v0.item()) == float("-inf")     # no valid winner
    i1, v1 = qmm.gemv_argmax(t["x"], p, t["scales"], t["biases"], N, 4, 64, ws)
    qmm.check()
    y = qmm.gemv(t["x"], p, t["scales"], t["biases"], N, 4, 64).cpu().numpy()[0]
    assert int(i1.item()) == int(np.argmax(y)) and float(v1.item()) == float(y[int(i1.item())])


def test_the_hook_is_one_shot_and_rejects_out_of_range_limits(qmm):
    with pytest.raises(qmm.QmmError):
        qmm.test_timeout_next_decode(10)
    with pytest.raises(qmm.QmmError):
        qmm.test_timeout_next_decode(10 ** 9)
    d = inputs.make(1, 4096, 2048, 4, 64, seed=1)   # an INT4 shape of the tensor-core kernel
    t = to_device(d, 4)
    p = qmm.pack(t["codes"], 4)
    qmm.test_timeout_next_decode(200_000)
    qmm.gemv(t["x"], p, t["scales"], t["biases"], 4096, 4, 64)
    expect_timeout(qmm)
    for _ in range(3):
        qmm.gemv(t["x"], p, t["scales"], t["biases"], 4096, 4, 64)
    qmm.check()                   # the hook was taken by the first launch only
