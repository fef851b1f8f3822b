"""qmm_noalloc: the product for callers that cannot let a library allocate
device memory -- serving loops that keep every byte of device memory in
their own fixed pool, and loops that must not stall on cudaFree, which waits
for the whole device.  Its output must satisfy the library's accuracy bound
against the CPU oracle, and agree with qmm()'s output within the same
tolerance, on two calls in a row, and the calls must not take device
memory.  Collected last on purpose, so that a run that stops at the first
failure has run every other test before it."""
import numpy as np
import pytest

import oracle as O
import synth

pytestmark = pytest.mark.gpu

REL, ABS = 2e-3, 1e-5


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def test_noalloc_matches_oracle_and_qmm_on_two_calls(cuda_lib):
    import torch
    q = cuda_lib
    cases = [(synth.Q4_K, 300, 2048, 16), (synth.Q6_K, 129, 1024, 64), (synth.Q8_0, 77, 544, 3)]
    data = []
    for qtype, N, K, M in cases:
        W = synth.weights(qtype, N, K, seed=N + K)
        x = synth.activations(M, K, seed=M + K, outlier_frac=0.01)
        yo, A = O.qmm(qtype, W, N, K, x)
        data.append((qtype, N, K, M, _dev(W), _dev(x), yo, A))
    # warm up: loads the module (and its static scratch) and looks its address up
    qtype, N, K, M, Wd, xd, _, _ = data[0]
    q.qmm_noalloc(qtype, Wd, N, K, xd, torch.empty((M, N), device="cuda"))
    torch.cuda.synchronize()
    for qtype, N, K, M, Wd, xd, yo, A in data:   # calls in a row, different shapes
        y_na = torch.full((M, N), float("nan"), device="cuda")
        before = q.qmm_launch_count()
        q.qmm_noalloc(qtype, Wd, N, K, xd, y_na)
        assert q.qmm_launch_count() - before == 2   # the quantiser, then the GEMM
        y_ref = q.qmm(qtype, Wd, N, K, xd)
        torch.cuda.synchronize()
        y_na = y_na.cpu().numpy().astype(np.float64)
        bound = REL * A + ABS
        err = np.abs(y_na - yo)
        assert np.all(err <= bound), (qtype, N, K, M, float(err.max()))
        err = np.abs(y_na - y_ref.cpu().numpy())
        assert np.all(err <= bound), (qtype, N, K, M, float(err.max()))
    # qmm() may have grown its own workspace above; a no-alloc call never does
    y = torch.empty((16, 300), device="cuda")
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        q.qmm_noalloc(data[0][0], data[0][4], 300, 2048, data[0][5], y)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] >= free_before
    assert q.qmm_device_status() == 0
    yo, A = data[0][6], data[0][7]
    assert np.all(np.abs(y.cpu().numpy().astype(np.float64) - yo) <= REL * A + ABS)


def test_noalloc_rejects_oversized_calls(cuda_lib):
    import torch
    q = cuda_lib
    K, M, N = 14336, 1024, 8        # M*K = 14.7 million > the 16 MiB scratch
    W = torch.zeros(N * (K // 256) * 144, dtype=torch.uint8, device="cuda")
    x = torch.zeros((M, K), device="cuda")
    y = torch.zeros((M, N), device="cuda")
    with pytest.raises(q.QmmError) as ei:
        q.qmm_noalloc(q.Q4_K, W, N, K, x, y)
    assert ei.value.status == q.QMM_EINVAL_SHAPE
    assert "scratch" in str(ei.value)
    with pytest.raises(ValueError):     # a y too short for M x N is refused by the binding
        q.qmm_noalloc(q.Q4_K, W, N, K, x[:2], torch.zeros(3, device="cuda"))
