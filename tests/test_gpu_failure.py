"""Failure detection on the GPU without a fault: every wait inside the
weight-streaming kernels is bounded.  The test hook qmm_inject_stall makes
the first CTA's weight producer of the next launch stop after one stage (a
barrier that nothing completes), so a consumer's wait expires after about a
second; the kernel records the timeout, drains what it issued and returns.
The host then reads QMM_ETIMEOUT from qmm_device_status(), and the next call
on the same context is correct."""
import numpy as np
import pytest

import oracle as O
import synth

pytestmark = pytest.mark.gpu


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


# block-per-lane decode (M = 1), tensor-core decode (M = 4), tcgen05 prefill
# (Q4_K raw-weight ring; Q6_K dequantisers copying their own rows)
# (every warp of the first CTA streams at least two stages at these sizes)
CASES = [(synth.Q4_K, 8192, 4096, 1), (synth.Q6_K, 16384, 2048, 2), (synth.Q4_K, 2048, 5120, 4),
         (synth.Q6_K, 1024, 5120, 8), (synth.Q4_K, 512, 4096, 64), (synth.Q6_K, 300, 5120, 64),
         (synth.Q8_0, 512, 4096, 300)]


@pytest.mark.parametrize("qtype,N,K,M", CASES)
def test_expired_wait_is_reported_and_the_next_call_is_right(cuda_lib, qtype, N, K, M):
    q = cuda_lib
    W = synth.weights(qtype, N, K, seed=N + M)
    x = synth.activations(M, K, seed=K + M)
    Wd, xd = _dev(W), _dev(x)
    assert q.qmm_device_status() == 0
    q.inject_stall(1)
    q.qmm(qtype, Wd, N, K, xd)                      # returns at once; the kernel gives up
    assert q.qmm_device_status() == q.QMM_ETIMEOUT
    assert q.qmm_device_status() == 0               # the flag is cleared by the read
    y = q.qmm(qtype, Wd, N, K, xd).cpu().numpy().astype(np.float64)
    assert q.qmm_device_status() == 0
    yo, A = O.qmm(qtype, W, N, K, x)
    assert np.all(np.abs(y - yo) <= 2e-3 * A + 1e-5)


# the group launches: block-per-lane at M = 1, the tensor-core one at M = 6
@pytest.mark.parametrize("M", [1, 6])
def test_expired_wait_in_a_group_launch(cuda_lib, M):
    q = cuda_lib
    K = 5120
    items = [(synth.Q4_K, 8192), (synth.Q6_K, 1024)]
    Ws = [synth.weights(t, N, K, seed=10 + i) for i, (t, N) in enumerate(items)]
    x = synth.activations(M, K, seed=11)
    xd = _dev(x)
    q.inject_stall(1)
    q.qmm_group([(t, _dev(W), N) for (t, N), W in zip(items, Ws)], K, xd)
    assert q.qmm_device_status() == q.QMM_ETIMEOUT
    ys = q.qmm_group([(t, _dev(W), N) for (t, N), W in zip(items, Ws)], K, xd)
    assert q.qmm_device_status() == 0
    for (t, N), W, y in zip(items, Ws, ys):
        yo, A = O.qmm(t, W, N, K, x)
        assert np.all(np.abs(y.cpu().numpy().astype(np.float64) - yo) <= 2e-3 * A + 1e-5)
    assert q.inject_stall(0) == 0                   # nothing left pending
