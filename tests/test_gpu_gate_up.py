"""The gated MLP product h = silu(W_gate x) * (W_up x) through the C ABI
against the oracle's gate_up_silu, element-wise within its bound B (the
products' bound e = 2e-3 * A + 1e-5 carried through the SiLU's slope):
the Qwen3-14B gate/up pair at M = 1, 2, 4, 8 (one launch at M <= 2, three
on the tensor-core decode), ragged and mixed-type shapes, and prefill."""
import numpy as np
import pytest

import oracle as O
import synth

pytestmark = pytest.mark.gpu


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _check(q, tg, Wg, tu, Wu, N, K, x, rows=None, launches=None, what=""):
    before = q.qmm_launch_count()
    h = q.qmm_gate_up(tg, _dev(Wg), tu, _dev(Wu), N, K, _dev(x)).cpu().numpy().astype(np.float64)
    assert q.qmm_device_status() == 0
    if launches is not None:
        assert q.qmm_launch_count() - before == launches, what
    if rows is not None:
        rbg, rbu = synth.row_bytes(tg, K), synth.row_bytes(tu, K)
        Wg = Wg.reshape(N, rbg)[rows].reshape(-1)
        Wu = Wu.reshape(N, rbu)[rows].reshape(-1)
        h = h[:, rows]
        N = len(rows)
    ho, B = O.gate_up_silu(tg, Wg, tu, Wu, N, K, x)
    err = np.abs(h - ho)
    bad = err > B
    assert not bad.any(), f"{what}: {bad.sum()} outside; worst {err[bad].max():.3e} vs {B[bad].min():.3e}"


@pytest.mark.parametrize("M,launches", [(1, 1), (2, 1), (4, 3), (8, 3)])
def test_gate_up_qwen3_14b(cuda_lib, M, launches):
    K, N = 5120, 17408
    Wg = synth.config_weights(3, 4)
    Wu = synth.config_weights(3, 5)
    x = synth.config_activations(3, M, K)
    rows = np.unique(np.concatenate([np.arange(64), np.arange(N - 64, N),
                                     np.random.default_rng(M).choice(N, 256, replace=False)]))
    _check(cuda_lib, synth.Q4_K, Wg, synth.Q4_K, Wu, N, K, x, rows=rows, launches=launches,
           what=f"qwen3 gate/up M={M}")


SHAPES = [(synth.Q4_K, synth.Q4_K, 37, 256, 1), (synth.Q4_K, synth.Q4_K, 301, 2048, 2),
          (synth.Q6_K, synth.Q6_K, 129, 1280, 1), (synth.Q8_0, synth.Q8_0, 100, 1056, 2),
          (synth.Q4_K, synth.Q6_K, 77, 2048, 1), (synth.Q4_K, synth.Q6_K, 77, 2048, 5),
          (synth.Q4_K, synth.Q4_K, 300, 5120, 3), (synth.Q6_K, synth.Q6_K, 40, 2048, 7),
          (synth.Q4_K, synth.Q4_K, 200, 2048, 64), (synth.Q8_0, synth.Q4_K, 130, 768, 300)]


@pytest.mark.parametrize("tg,tu,N,K,M", SHAPES)
def test_gate_up_shapes(cuda_lib, tg, tu, N, K, M):
    Wg = synth.weights(tg, N, K, seed=N + K + M)
    Wu = synth.weights(tu, N, K, seed=N + K + M + 1)
    x = synth.activations(M, K, seed=N * M + K, outlier_frac=0.01)
    _check(cuda_lib, tg, Wg, tu, Wu, N, K, x, what=f"types {tg}/{tu} N={N} K={K} M={M}")


def test_gate_up_large_magnitudes(cuda_lib):
    """x around 1e4 on the tensor-core path: |g| is large, silu(g) is g or 0."""
    N, K, M = 300, 2048, 4
    Wg = synth.weights(synth.Q4_K, N, K, seed=3)
    Wu = synth.weights(synth.Q4_K, N, K, seed=4)
    x = synth.activations(M, K, seed=5) * np.float32(1e4)
    _check(cuda_lib, synth.Q4_K, Wg, synth.Q4_K, Wu, N, K, x, what="x*1e4")
