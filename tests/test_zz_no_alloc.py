"""The allocation-free greedy head (qmm_gemv_argmax_noalloc) against the
entry point with a caller workspace (qmm_gemv_argmax).

Named to be collected last: it must pass both alone and after every other
test, since the static work area it uses is shared by all its calls."""
import numpy as np
import pytest

from quantized_weight_gb300 import inputs
from helpers import to_device

UNSUP, SHAPE, ARG, ALIGN = -4, -2, -1, -3
FAKE, MIS, ODD = 0x10000, 0x10004, 0x10002


def test_noalloc_validation_on_the_host():
    from quantized_weight_gb300 import build, qmm
    build.build()
    L = qmm.lib()

    def call(x=FAKE, c=FAKE, s=FAKE, b=FAKE, i=FAKE, v=None, N=64, K=128, bits=4, g=64):
        return L.qmm_gemv_argmax_noalloc(x, c, s, b, i, v, N, K, bits, g, None)

    assert call(bits=2) == UNSUP
    assert call(g=16) == UNSUP
    assert call(N=0) == SHAPE
    assert call(K=96) == SHAPE
    assert call(i=None) == ARG
    assert call(b=None) == ARG
    assert call(bits=8, b=FAKE) == ARG
    assert call(x=MIS) == ALIGN
    assert call(i=ODD) == ALIGN                 # idx and val need 4-byte alignment only
    assert call(v=ODD) == ALIGN
    assert call(x=MIS, i=MIS) == ALIGN


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
    # calls queued back to back on one stream, no host sync between them: each
    # call's CTAs may start before the previous call has finished, and each must
    # still see the counter its predecessor reset; results go straight into
    # tokens[t], a 4-byte-aligned slot of one int32 array
    N, K, bits, group = 151936, 2048, 4, 64
    d = inputs.make(1, N, K, bits, group, seed=11)
    t = to_device(d, bits)
    p = qmm.pack(t["codes"], bits)
    ws = qmm.argmax_workspace(1, N)
    xs = [torch.from_numpy(inputs.make(1, 8, K, bits, group, seed=20 + j)["x"]).cuda() for j in range(4)]
    want = []
    for xj in xs:
        i0, v0 = qmm.gemv_argmax(xj, p, t["scales"], t["biases"], N, bits, group, ws)
        want.append((int(i0.item()), v0.cpu().numpy().view(np.uint32)[0]))
    tokens = torch.full((5,), -1, dtype=torch.int32, device="cuda")
    vals = torch.zeros((5,), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    for j, xj in enumerate(xs):
        qmm.gemv_argmax_noalloc(xj, p, t["scales"], t["biases"], N, bits, group,
                                idx=tokens[j + 1:j + 2], val=vals[j + 1:j + 2])
    torch.cuda.synchronize()
    got = tokens.cpu().numpy()
    gv = vals.cpu().numpy().view(np.uint32)
    assert got[0] == -1
    for j in range(4):
        assert got[j + 1] == want[j][0] and gv[j + 1] == want[j][1]
    # a shape the fused kernel does not take is refused, not computed another way
    d = inputs.make(1, 64, 32 * 17, 4, 32, seed=1)    # K not a whole number of 1024-weight warp segments
    t = to_device(d, 4)
    p = qmm.pack(t["codes"], 4)
    with pytest.raises(qmm.QmmError):
        qmm.gemv_argmax_noalloc(t["x"], p, t["scales"], t["biases"], 64, 4, 32)
