"""GPU parity of the row-per-lane decode kernel (Q4_K, Q5_K, Q6_K, Q3_K and
Q2_K up to M = 8) against the CPU oracle, within the library's
bound |y_gpu - y_oracle| <= 2e-3 * sum_k |w_k xhat_k| + 1e-5.

The shapes cover what the kernel's plan and indexing branch on: a CTA's row
groups of 32 (N below, at and above multiples of 32 and of the CTA count,
N smaller than the grid), both stage widths (8 or 10 super-blocks per
row, chosen by K) with full and ragged last chunks, K large enough that
the ring shrinks to two stages, Q6_K rows that start inside a 16-byte
chunk, and matrices whose last bytes do not end on a 16-byte boundary
(loaded without reading past the end)."""
import numpy as np
import pytest

import oracle as O
import synth

pytestmark = pytest.mark.gpu

REL, ABS = 2e-3, 1e-5


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _check(y, yo, A, what):
    err = np.abs(y.astype(np.float64) - yo)
    bad = err > REL * A + ABS
    assert not bad.any(), f"{what}: {bad.sum()} outside the bound, worst {err.max():.3e}"


@pytest.fixture
def rows_path(cuda_lib):
    prev = cuda_lib.set_decode_path(cuda_lib.DECODE_ROWS)
    yield
    cuda_lib.set_decode_path(prev)


CASES = [
    # (qtype, N, K, M)
    (synth.Q4_K, 1, 256, 1), (synth.Q4_K, 5, 1024, 2), (synth.Q4_K, 31, 512, 2), (synth.Q4_K, 33, 2048, 1),
    (synth.Q4_K, 153, 2560, 1), (synth.Q4_K, 300, 4608, 2), (synth.Q4_K, 4865, 5120, 1),
    (synth.Q4_K, 200, 17408, 2), (synth.Q4_K, 9000, 2048, 2),
    (synth.Q6_K, 1, 256, 1), (synth.Q6_K, 3, 512, 2), (synth.Q6_K, 77, 2048, 1), (synth.Q6_K, 33, 2560, 2),
    (synth.Q6_K, 301, 4608, 2), (synth.Q6_K, 4097, 5120, 1), (synth.Q6_K, 150, 17408, 1),
    (synth.Q3_K, 1, 256, 1), (synth.Q3_K, 77, 2048, 2), (synth.Q3_K, 301, 4608, 1), (synth.Q3_K, 4097, 5120, 2),
    (synth.Q3_K, 150, 17408, 1), (synth.Q2_K, 3, 512, 2), (synth.Q2_K, 33, 2560, 1), (synth.Q2_K, 300, 4608, 2),
    (synth.Q2_K, 4865, 5120, 1), (synth.Q2_K, 200, 17408, 2),
    (synth.Q6_K, 120, 17408, 2),
    (synth.Q5_K, 1, 256, 1), (synth.Q5_K, 77, 2048, 2), (synth.Q5_K, 300, 5120, 1), (synth.Q5_K, 4097, 5120, 2),
    (synth.Q5_K, 150, 17408, 1),
]


# every K-quant with 3 <= M <= 8: four or eight accumulators per lane (the
# rows of the activations past M are computed on and never written)
CASES_WIDE = [
    (synth.Q4_K, 1, 256, 3), (synth.Q4_K, 33, 2048, 4), (synth.Q4_K, 300, 4608, 5), (synth.Q4_K, 4865, 5120, 8),
    (synth.Q4_K, 200, 10240, 6), (synth.Q4_K, 77, 1024, 7), (synth.Q4_K, 5, 5120, 4),
    (synth.Q5_K, 33, 2048, 3), (synth.Q5_K, 300, 5120, 8), (synth.Q5_K, 150, 17408, 4),
    (synth.Q3_K, 1, 256, 5), (synth.Q3_K, 301, 4608, 4), (synth.Q3_K, 200, 5120, 8),
    (synth.Q2_K, 77, 1024, 7), (synth.Q2_K, 4865, 5120, 4), (synth.Q2_K, 120, 17408, 3),
    (synth.Q6_K, 77, 2048, 3), (synth.Q6_K, 301, 4608, 8), (synth.Q6_K, 4097, 5120, 5), (synth.Q6_K, 150, 10240, 4),
]


@pytest.mark.parametrize("qtype,N,K,M", CASES + CASES_WIDE)
def test_rows_decode_matches_oracle(cuda_lib, rows_path, qtype, N, K, M):
    q = cuda_lib
    W = synth.weights(qtype, N, K, seed=3 * N + K + M)
    x = synth.activations(M, K, seed=N + 7 * K + M, outlier_frac=0.01)
    before = q.qmm_launch_count()
    y = q.qmm(qtype, _dev(W), N, K, _dev(x)).cpu().numpy()
    assert q.qmm_launch_count() - before == 1      # x quantised inside the one launch
    assert q.qmm_device_status() == 0
    yo, A = O.qmm(qtype, W, N, K, x)
    _check(y, yo, A, f"type {qtype} N={N} K={K} M={M}")


def test_rows_decode_is_deterministic_and_overwrites_y(cuda_lib, rows_path):
    import torch
    q = cuda_lib
    for qtype, N, K, M in [(synth.Q4_K, 1000, 5120, 1), (synth.Q6_K, 700, 17408, 2)]:
        W = _dev(synth.weights(qtype, N, K, seed=41))
        x = _dev(synth.activations(M, K, seed=42))
        y1 = torch.full((M, N), float("nan"), device="cuda")
        q.qmm(qtype, W, N, K, x, y=y1)
        for _ in range(3):
            assert torch.equal(y1, q.qmm(qtype, W, N, K, x))


@pytest.mark.parametrize("M", [1, 2])
def test_rows_group_one_launch_mixed_types(cuda_lib, rows_path, M):
    q = cuda_lib
    K = 5120
    items = [(synth.Q4_K, 5120), (synth.Q4_K, 0), (synth.Q4_K, 1024), (synth.Q6_K, 1024), (synth.Q6_K, 77)]
    Ws = [synth.weights(t, N, K, seed=60 + i) for i, (t, N) in enumerate(items)]
    x = synth.activations(M, K, seed=61 + M, outlier_frac=0.01)
    before = q.qmm_launch_count()
    ys = q.qmm_group([(t, _dev(W), N) for (t, N), W in zip(items, Ws)], K, _dev(x))
    assert q.qmm_launch_count() - before == 1
    assert q.qmm_device_status() == 0
    for (t, N), W, y in zip(items, Ws, ys):
        if N == 0:
            continue
        yo, A = O.qmm(t, W, N, K, x)
        _check(y.cpu().numpy(), yo, A, f"group entry type {t} N={N} M={M}")


def test_rows_and_block_paths_agree_within_the_bound(cuda_lib):
    q = cuda_lib
    qtype, N, K, M = synth.Q4_K, 2048, 5120, 1
    W = synth.weights(qtype, N, K, seed=71)
    x = synth.activations(M, K, seed=72, outlier_frac=0.01)
    Wd, xd = _dev(W), _dev(x)
    prev = q.set_decode_path(q.DECODE_BLOCK)
    try:
        y_block = q.qmm(qtype, Wd, N, K, xd).cpu().numpy()
    finally:
        q.set_decode_path(prev)
    y_rows = q.qmm(qtype, Wd, N, K, xd).cpu().numpy()
    yo, A = O.qmm(qtype, W, N, K, x)
    _check(y_rows, yo, A, "rows")
    _check(y_block, yo, A, "block")
    # both take exact int32 block dots: only the fp32 order of the scaled
    # sums differs
    assert np.all(np.abs(y_rows.astype(np.float64) - y_block) <= REL * A + ABS)


@pytest.mark.parametrize("M", [4, 8])
def test_rows_group_one_launch_wide(cuda_lib, rows_path, M):
    q = cuda_lib
    K = 5120
    items = [(synth.Q4_K, 5120), (synth.Q4_K, 1024), (synth.Q4_K, 0), (synth.Q4_K, 77)]
    Ws = [synth.weights(t, N, K, seed=80 + i) for i, (t, N) in enumerate(items)]
    x = synth.activations(M, K, seed=81 + M, outlier_frac=0.01)
    before = q.qmm_launch_count()
    ys = q.qmm_group([(t, _dev(W), N) for (t, N), W in zip(items, Ws)], K, _dev(x))
    assert q.qmm_launch_count() - before == 1
    assert q.qmm_device_status() == 0
    for (t, N), W, y in zip(items, Ws, ys):
        if N == 0:
            continue
        yo, A = O.qmm(t, W, N, K, x)
        _check(y.cpu().numpy(), yo, A, f"group entry N={N} M={M}")


# A group of several matrices from M = 3 on (q/k/v with a Q6_K v, as in a
# Q4_K_M model) under the default kernel choice: x is quantised once and the
# matrices share one tensor-core launch.
@pytest.mark.parametrize("M", [3, 4, 8])
def test_group_default_choice_q_k_v(cuda_lib, M):
    q = cuda_lib
    K = 5120
    items = [(synth.Q4_K, 5120), (synth.Q4_K, 1024), (synth.Q6_K, 1024), (synth.Q6_K, 0), (synth.Q6_K, 33)]
    Ws = [synth.weights(t, N, K, seed=90 + i) for i, (t, N) in enumerate(items)]
    x = synth.activations(M, K, seed=91 + M, outlier_frac=0.01)
    before = q.qmm_launch_count()
    ys = q.qmm_group([(t, _dev(W), N) for (t, N), W in zip(items, Ws)], K, _dev(x))
    launches = q.qmm_launch_count() - before
    assert q.qmm_device_status() == 0
    assert launches == 2
    for (t, N), W, y in zip(items, Ws, ys):
        if N == 0:
            continue
        yo, A = O.qmm(t, W, N, K, x)
        _check(y.cpu().numpy(), yo, A, f"group entry type {t} N={N} M={M}")


@pytest.mark.parametrize("M", [4, 8])
def test_rows_group_one_launch_wide_with_q6k(cuda_lib, rows_path, M):
    q = cuda_lib
    K = 2560
    items = [(synth.Q6_K, 2049), (synth.Q4_K, 300), (synth.Q6_K, 77)]
    Ws = [synth.weights(t, N, K, seed=95 + i) for i, (t, N) in enumerate(items)]
    x = synth.activations(M, K, seed=96 + M, outlier_frac=0.01)
    before = q.qmm_launch_count()
    ys = q.qmm_group([(t, _dev(W), N) for (t, N), W in zip(items, Ws)], K, _dev(x))
    assert q.qmm_launch_count() - before == 1
    assert q.qmm_device_status() == 0
    for (t, N), W, y in zip(items, Ws, ys):
        yo, A = O.qmm(t, W, N, K, x)
        _check(y.cpu().numpy(), yo, A, f"group entry type {t} N={N} M={M}")


# Q5_K, Q3_K and Q2_K at M = 8 with K = 17408: neither decode kernel holds the
# activations in shared memory, so the product runs on the tcgen05 prefill
# kernel (the quantiser, then the GEMM) instead of the round-based decode
@pytest.mark.parametrize("qtype,N,M", [(synth.Q5_K, 300, 8), (synth.Q3_K, 200, 8), (synth.Q2_K, 150, 7)])
def test_decode_too_large_for_the_decode_kernels(cuda_lib, qtype, N, M):
    q = cuda_lib
    K = 17408
    W = synth.weights(qtype, N, K, seed=N + M)
    x = synth.activations(M, K, seed=N + 2 * M, outlier_frac=0.01)
    before = q.qmm_launch_count()
    y = q.qmm(qtype, _dev(W), N, K, _dev(x)).cpu().numpy()
    assert q.qmm_device_status() == 0
    assert q.qmm_launch_count() - before == 2
    yo, A = O.qmm(qtype, W, N, K, x)
    _check(y, yo, A, f"type {qtype} N={N} K={K} M={M}")
