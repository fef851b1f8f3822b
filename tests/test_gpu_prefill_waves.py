"""GPU parity of the tcgen05 prefill when its tiles leave the last wave of
CTAs partly empty: the whole waves run unsplit in one launch and the
remaining tiles, split along K in clusters, in a second launch that may start
while the first still runs.  Sampled rows (every row of the first and last
weight-row tiles, plus random ones) against the CPU oracle within
|y_gpu - y_oracle| <= 2e-3 * sum_k |w_k xhat_k| + 1e-5, the launch count
(quantiser + two), and bitwise determinism over repeated calls."""
import numpy as np
import pytest

import oracle as O
import synth

pytestmark = pytest.mark.gpu

REL, ABS = 2e-3, 1e-5


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _rows(N, seed):
    rng = np.random.default_rng(seed)
    r = set(range(0, min(N, 128))) | set(range(max(0, N - 256), N))
    r |= set(rng.choice(N, size=min(N, 256), replace=False).tolist())
    return np.array(sorted(r))


# (type, N, K, M): 128-row weight tiles x 256-token tiles; tiles beyond a
# multiple of the CTAs resident at once (one per SM) form the split part
CASES = [(synth.Q4_K, 20000, 1024, 300), (synth.Q6_K, 20000, 2048, 300), (synth.Q4_K, 14336, 4096, 512),
         # 153 tiles: one past a full wave, the last tile split the most ways
         (synth.Q4_K, 19584, 1024, 200), (synth.Q6_K, 19584, 2048, 100)]


@pytest.mark.parametrize("qtype,N,K,M", CASES)
def test_prefill_two_part_schedule(cuda_lib, qtype, N, K, M):
    import torch
    q = cuda_lib
    W = synth.weights(qtype, N, K, seed=N + K)
    x = synth.activations(M, K, seed=M + K, outlier_frac=0.01)
    Wd, xd = _dev(W), _dev(x)
    before = q.qmm_launch_count()
    y = q.qmm(qtype, Wd, N, K, xd)
    launches = q.qmm_launch_count() - before
    torch.cuda.synchronize()
    assert q.qmm_device_status() == 0
    tiles = -(-N // 128) * -(-M // 256)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if tiles > sms and tiles % sms:
        assert launches in (2, 3)   # the quantiser, then one or two GEMM launches
    rows = _rows(N, seed=N)
    rb = synth.row_bytes(qtype, K)
    yo, A = O.qmm(qtype, W.reshape(N, rb)[rows], len(rows), K, x)
    yg = y.cpu().numpy()[:, rows].astype(np.float64)
    err = np.abs(yg - yo)
    assert np.all(err <= REL * A + ABS), float(err.max())
    for _ in range(2):
        assert torch.equal(y, q.qmm(qtype, Wd, N, K, xd))
