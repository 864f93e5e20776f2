"""The allocation-free greedy head (qmm_gemv_argmax_noalloc) against the
entry point with a caller workspace (qmm_gemv_argmax).

Named to be collected last: it must pass both alone and after every other
test, since the static work area it uses is shared by all its calls."""
import numpy as np
import pytest

from quantized_weight_gb300 import inputs
from helpers import to_device

UNSUP, SHAPE, ARG, ALIGN = -4, -2, -1, -3
FAKE, MIS = 0x10000, 0x10004


def test_noalloc_validation_on_the_host():
    from quantized_weight_gb300 import build, qmm
    build.build()
    L = qmm.lib()

    def call(x=FAKE, c=FAKE, s=FAKE, b=FAKE, i=FAKE, N=64, K=128, bits=4, g=64):
        return L.qmm_gemv_argmax_noalloc(x, c, s, b, i, None, N, K, bits, g, None)

    assert call(bits=2) == UNSUP
    assert call(g=16) == UNSUP
    assert call(N=0) == SHAPE
    assert call(K=96) == SHAPE
    assert call(i=None) == ARG
    assert call(b=None) == ARG
    assert call(bits=8, b=FAKE) == ARG
    assert call(x=MIS) == ALIGN


@pytest.mark.gpu
def test_noalloc_matches_the_workspace_entry_on_consecutive_calls():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_weight_gb300 import build, qmm
    build.build()
    results = []
    for seed, (N, K, bits, group) in enumerate([(151936, 2048, 4, 64), (151936, 2048, 4, 64),
                                                 (20000, 4096, 8, 64), (7001, 1024, 4, 128)]):
        d = inputs.make(1, N, K, bits, group, seed=seed)
        t = to_device(d, bits)
        p = qmm.pack(t["codes"], bits)
        ws = qmm.argmax_workspace(1, N)
        for _ in range(2):                              # two consecutive calls each
            i0, v0 = qmm.gemv_argmax(t["x"], p, t["scales"], t["biases"], N, bits, group, ws)
            i1, v1 = qmm.gemv_argmax_noalloc(t["x"], p, t["scales"], t["biases"], N, bits, group)
            torch.cuda.synchronize()
            assert int(i1.item()) == int(i0.item())
            assert np.array_equal(v1.cpu().numpy().view(np.uint32), v0.cpu().numpy().view(np.uint32))
            results.append(int(i1.item()))
    assert results[0] == results[1] and results[2] == results[3]      # same inputs, same winner
    # a shape the fused kernel does not take is refused, not computed another way
    d = inputs.make(1, 64, 32 * 17, 4, 32, seed=1)    # K not a whole number of 1024-weight warp segments
    t = to_device(d, 4)
    p = qmm.pack(t["codes"], 4)
    with pytest.raises(qmm.QmmError):
        qmm.gemv_argmax_noalloc(t["x"], p, t["scales"], t["biases"], 64, 4, 32)
