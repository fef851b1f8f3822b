"""The products for the other GGUF K-quants (Q5_K, Q3_K, Q2_K) through the C
ABI against the pinned oracle: decode (block-per-lane dp4a kernel, every
M <= 8), prefill (int8 mma.sync kernel, exact block dots), groups and the
gate+up product, element-wise within |dy| <= 2e-3 * sum|w xhat| + 1e-5;
and unit-scale blocks whose product is an exact integer, which pins every
bit-field index of the unpackers."""
import numpy as np
import pytest

import oracle as O
import synth

pytestmark = pytest.mark.gpu

KQ = [synth.Q5_K, synth.Q3_K, synth.Q2_K]


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _assert_bound(y, yo, A, what):
    err = np.abs(y.astype(np.float64) - yo)
    bad = err > 2e-3 * A + 1e-5
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside; worst {err[bad].max():.3e}"


SHAPES = [(37, 256, 1), (300, 1280, 1), (129, 2048, 2), (64, 5120, 3), (77, 768, 4), (50, 2304, 8),
          (8, 17408, 1), (70, 512, 9), (130, 768, 64), (200, 4096, 130), (33, 256, 300)]


@pytest.mark.parametrize("qtype", KQ)
@pytest.mark.parametrize("N,K,M", SHAPES)
def test_qmm_other_k_quants(cuda_lib, qtype, N, K, M):
    W = synth.weights(qtype, N, K, seed=N + K + M + qtype)
    x = synth.activations(M, K, seed=N * K + M, outlier_frac=0.01)
    y = cuda_lib.qmm(qtype, _dev(W), N, K, _dev(x)).cpu().numpy()
    assert cuda_lib.qmm_device_status() == 0
    yo, A = O.qmm(qtype, W, N, K, x)
    _assert_bound(y, yo, A, f"type {qtype} N={N} K={K} M={M}")


@pytest.mark.parametrize("qtype", KQ)
def test_qmm_other_k_quants_full_size_decode(cuda_lib, qtype):
    """A Qwen3-14B-shaped 5120 -> 17408 matrix of each type at M = 1 and 4,
    on sampled rows."""
    N, K = 17408, 5120
    W = synth.weights(qtype, N, K, seed=3000 + qtype)
    rows = np.unique(np.concatenate([np.arange(64), np.arange(N - 64, N),
                                     np.random.default_rng(qtype).choice(N, 256, replace=False)]))
    Wr = W.reshape(N, synth.row_bytes(qtype, K))[rows].reshape(-1)
    Wd = _dev(W)
    for M in (1, 4):
        x = synth.activations(M, K, seed=M)
        y = cuda_lib.qmm(qtype, Wd, N, K, _dev(x)).cpu().numpy()
        assert cuda_lib.qmm_device_status() == 0
        yo, A = O.qmm(qtype, Wr, len(rows), K, x)
        _assert_bound(y[:, rows], yo, A, f"type {qtype} full size M={M}")


def _int_activations(rng, M, K):
    xi = rng.integers(-127, 128, (M, K)).astype(np.float64)
    xi[:, 3::32] = 127.0      # amax 127 in every block: scale exactly 1
    return xi


@pytest.mark.parametrize("M", [1, 3, 8, 24])
def test_unit_scale_products_are_exact(cuda_lib, M):
    """d = 1, scales giving a unit multiplier and no min: w = q exactly, so y
    is an exact integer product (partial sums below 2^24) on every path."""
    rng = np.random.default_rng(M)
    N, K = 70, 1024
    nb = K // 256
    xi = _int_activations(rng, M, K)
    # Q5_K: sc = 1, m = 0, q in 0..31
    q5 = rng.integers(0, 32, (N, nb, 256)).astype(np.uint8)
    W5 = np.concatenate([O.pack_q5_k(0x3C00, 0, np.ones(8, np.uint8), np.zeros(8, np.uint8), q5[n, b])
                         for n in range(N) for b in range(nb)])
    # Q3_K: sc - 32 = 1, q in -4..3
    q3 = rng.integers(-4, 4, (N, nb, 256)).astype(np.int8)
    W3 = np.concatenate([O.pack_q3_k(0x3C00, np.ones(16, np.int8), q3[n, b])
                         for n in range(N) for b in range(nb)])
    # Q2_K: sc = 1, m = 0, q in 0..3
    q2 = rng.integers(0, 4, (N, nb, 256)).astype(np.uint8)
    W2 = np.concatenate([O.pack_q2_k(0x3C00, 0, np.ones(16, np.uint8), np.zeros(16, np.uint8), q2[n, b])
                         for n in range(N) for b in range(nb)])
    for qtype, W, qv in ((synth.Q5_K, W5, q5), (synth.Q3_K, W3, q3), (synth.Q2_K, W2, q2)):
        y = cuda_lib.qmm(qtype, _dev(W), N, K, _dev(xi.astype(np.float32))).cpu().numpy()
        want = xi @ qv.reshape(N, K).astype(np.float64).T
        assert np.array_equal(y.astype(np.float64), want), qtype


def test_group_and_gate_up_with_other_k_quants(cuda_lib):
    """qmm_group over mixed K-quants (run entry by entry) and qmm_gate_up with a
    Q5_K pair (one launch at M = 1) and a Q3_K / Q2_K pair."""
    q = cuda_lib
    K = 2048
    items = [(synth.Q5_K, 300), (synth.Q3_K, 129), (synth.Q2_K, 77), (synth.Q4_K, 64)]
    Ws = [synth.weights(t, N, K, seed=40 + i) for i, (t, N) in enumerate(items)]
    for M in (1, 5, 33):
        x = synth.activations(M, K, seed=M + 7)
        ys = q.qmm_group([(t, _dev(W), N) for (t, N), W in zip(items, Ws)], K, _dev(x))
        for (t, N), W, y in zip(items, Ws, ys):
            yo, A = O.qmm(t, W, N, K, x)
            _assert_bound(y.cpu().numpy(), yo, A, f"group type {t} M={M}")
    N = 300
    for tg, tu, M, launches in ((synth.Q5_K, synth.Q5_K, 1, 1), (synth.Q3_K, synth.Q2_K, 2, None),
                                (synth.Q2_K, synth.Q2_K, 6, None)):
        Wg = synth.weights(tg, N, K, seed=50 + M)
        Wu = synth.weights(tu, N, K, seed=60 + M)
        x = synth.activations(M, K, seed=70 + M)
        before = q.qmm_launch_count()
        h = q.qmm_gate_up(tg, _dev(Wg), tu, _dev(Wu), N, K, _dev(x)).cpu().numpy().astype(np.float64)
        if launches is not None:
            assert q.qmm_launch_count() - before == launches
        ho, B = O.gate_up_silu(tg, Wg, tu, Wu, N, K, x)
        assert np.all(np.abs(h - ho) <= B), (tg, tu, M)


@pytest.mark.parametrize("qtype", KQ)
@pytest.mark.parametrize("N,K,M", [(300, 1024, 64), (200, 2048, 300), (77, 256, 9), (1000, 4096, 130),
                                   (129, 5120, 512), (301, 768, 70), (3, 4352, 33)])
def test_prefill_on_tcgen05_and_int8(cuda_lib, qtype, N, K, M):
    """Prefill of the other K-quants on the tcgen05 kernel (Q5_K: the TMA raw
    ring with the fifth-bit plane in the head box; Q3_K, Q2_K: rows staged by
    the dequantiser warps, ragged matrix ends) and, forced, on the int8
    mma.sync kernel; both against the oracle."""
    q = cuda_lib
    W = synth.weights(qtype, N, K, seed=N + K + 5 + qtype)
    x = synth.activations(M, K, seed=N + M, outlier_frac=0.01)
    yo, A = O.qmm(qtype, W, N, K, x)
    for path in (q.PREFILL_AUTO, q.PREFILL_INT8):
        q.set_prefill_path(path)
        try:
            y = q.qmm(qtype, _dev(W), N, K, _dev(x)).cpu().numpy()
        finally:
            q.set_prefill_path(q.PREFILL_AUTO)
        assert q.qmm_device_status() == 0
        _assert_bound(y, yo, A, f"type {qtype} prefill path {path} N={N} K={K} M={M}")


@pytest.mark.parametrize("qtype", KQ)
def test_prefill_any_magnitude_and_scales(cuda_lib, qtype):
    """The tcgen05 prefill of the other K-quants with x at 1e-30 / 1e30 and
    with super-block scales spread over the whole fp16 range (the per-row
    power of two)."""
    q = cuda_lib
    N, K, M = 200, 2048, 96
    rng = np.random.default_rng(1 + qtype)
    nblk = N * (K // 256)
    for scale, spread in ((1e-30, False), (1e30, False), (1.0, True)):
        W = synth.weights(qtype, N, K, seed=9 + qtype)
        if spread:
            W = synth.with_scale_fields(qtype, W, synth.loguniform_f16_bits(rng, nblk, 2.0 ** -24, 6.0e4),
                                        synth.loguniform_f16_bits(rng, nblk, 2.0 ** -24, 6.0e4))
        x = (synth.activations(M, K, seed=3).astype(np.float64) * scale).astype(np.float32)
        y = q.qmm(qtype, _dev(W), N, K, _dev(x)).cpu().numpy().astype(np.float64)
        yo, A = O.qmm(qtype, W, N, K, x)
        assert np.all(np.abs(y - yo) <= 2e-3 * A + 1e-5 * min(1.0, scale)), (qtype, scale, spread)
