"""GPU parity at every magnitude: the fp16 tensor-core paths (tcgen05
prefill, mma.sync decode) scale activation rows and weight rows by powers of
two into fp16's normal range and undo them in fp32, so the accuracy bound
|y_gpu - y_oracle| <= 2e-3 * sum_k |w_k xhat_k| + 1e-5 holds for x from 1e-30
to 1e30 and for every fp16 weight scale, from the largest (65504) down to
subnormals.  Tiny magnitudes would pass the absolute 1e-5 term trivially, so
these tests also require the relative part alone: |dy| <= 2e-3 * A + 1e-5 * s
with s the magnitude of the case."""
import numpy as np
import pytest

import oracle as O
import synth

pytestmark = pytest.mark.gpu

REL, ABS = 2e-3, 1e-5


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _check(q, qtype, W, N, K, x, scale, what):
    y = q.qmm(qtype, _dev(W), N, K, _dev(x)).cpu().numpy().astype(np.float64)
    assert q.qmm_device_status() == 0
    yo, A = O.qmm(qtype, W, N, K, x)
    assert np.all(np.isfinite(y)), what
    err = np.abs(y - yo)
    bound = REL * A + ABS * min(1.0, scale)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside; worst err {err[bad].max():.3e} "
                           f"vs bound {bound[bad].min():.3e}")


SCALES = [1e-30, 1e-6, 1.0, 1e4, 1e30]
# (type, N, K, M): prefill on tcgen05 (BT = 64 and 256 token tiles, split K
# for the small one), tensor-core decode (M = 3..8) and the dp4a decode
PREFILL = [(synth.Q4_K, 300, 1024, 64), (synth.Q4_K, 200, 2048, 300), (synth.Q6_K, 130, 1536, 64),
           (synth.Q6_K, 257, 1024, 300), (synth.Q8_0, 140, 1024, 64), (synth.Q8_0, 300, 768, 300)]
# (Q6_K with K <= 2048 at M <= 4 runs on the block-per-lane kernel, K = 2560
# at M = 4 on the tensor-core one)
DECODE = [(synth.Q4_K, 300, 5120, 3), (synth.Q4_K, 77, 2048, 8), (synth.Q6_K, 301, 2048, 4),
          (synth.Q6_K, 301, 2560, 4), (synth.Q6_K, 129, 5120, 8), (synth.Q4_K, 300, 2048, 1),
          (synth.Q6_K, 100, 1024, 2)]


@pytest.mark.parametrize("scale", SCALES)
@pytest.mark.parametrize("qtype,N,K,M", PREFILL + DECODE)
def test_any_magnitude_of_x(cuda_lib, qtype, N, K, M, scale):
    W = synth.weights(qtype, N, K, seed=N + K + M)
    x = (synth.activations(M, K, seed=N * 3 + M, outlier_frac=0.01).astype(np.float64) * scale).astype(np.float32)
    _check(cuda_lib, qtype, W, N, K, x, scale, f"type {qtype} N={N} K={K} M={M} scale={scale}")


@pytest.mark.parametrize("qtype,N,K,M", PREFILL + DECODE)
def test_rows_spanning_many_binades(cuda_lib, qtype, N, K, M):
    """Blocks of 32 alternate between magnitudes 1e4 and 1e-4 inside each
    row (26 binades apart), and one row is all zeros."""
    x = synth.activations(M, K, seed=K + M)
    x.reshape(M, K // 32, 32)[:, 1::2, :] *= np.float32(1e-4)
    x.reshape(M, K // 32, 32)[:, 0::2, :] *= np.float32(1e4)
    x[M // 2, :] = 0.0
    W = synth.weights(qtype, N, K, seed=N + 2 * K)
    _check(cuda_lib, qtype, W, N, K, x, 1.0, f"type {qtype} N={N} K={K} M={M}")


# fp16 scale fields: the largest finite value, the smallest normal, subnormals,
# and a log-uniform spread over the whole fp16 range inside every row (the
# tcgen05 kernel's per-row scale then grows while a row streams)
D_CASES = {
    "max": lambda rng, n: np.full(n, 0x7BFF, np.uint16),
    "min_normal": lambda rng, n: np.full(n, 0x0400, np.uint16),
    "subnormal": lambda rng, n: rng.integers(1, 0x400, size=n).astype(np.uint16),
    "spread": lambda rng, n: synth.loguniform_f16_bits(rng, n, 2.0 ** -24, 6.0e4),
}


@pytest.mark.parametrize("case", list(D_CASES))
@pytest.mark.parametrize("qtype,N,K,M", PREFILL + DECODE)
def test_any_fp16_weight_scale(cuda_lib, qtype, N, K, M, case):
    rng = np.random.default_rng(N + K + M + len(case))
    nblk = N * (K // synth.BLOCK_WEIGHTS[qtype])
    W = synth.weights(qtype, N, K, seed=N * 7 + K)
    W = synth.with_scale_fields(qtype, W, D_CASES[case](rng, nblk), D_CASES[case](rng, nblk))
    x = synth.activations(M, K, seed=N + M, outlier_frac=0.01)
    _check(cuda_lib, qtype, W, N, K, x, 1.0, f"type {qtype} N={N} K={K} M={M} d={case}")


def test_growing_weight_scale_inside_each_row(cuda_lib):
    """Q4_K, Q6_K and Q8_0 prefill whose super-block scales grow by 2^6 every
    super-block along each row: the tcgen05 kernel must lower each row's
    power of two (and rescale the accumulator) several times per tile."""
    for qtype in (synth.Q4_K, synth.Q6_K, synth.Q8_0):
        N, K, M = 256, 2048, 96
        per_row = K // synth.BLOCK_WEIGHTS[qtype]
        sb = np.arange(per_row) // (per_row // 8)             # super-block index 0..7 along the row
        vals = (2.0 ** (-20 + 5 * sb)).astype(np.float32)      # 2^-20 .. 2^15
        bits = np.tile(vals.astype(np.float16).view(np.uint16), N)
        W = synth.with_scale_fields(qtype, synth.weights(qtype, N, K, seed=5), bits, bits)
        x = synth.activations(M, K, seed=6)
        _check(cuda_lib, qtype, W, N, K, x, 1.0, f"growing scales type {qtype}")


@pytest.mark.parametrize("scale", [1e-30, 1e30])
@pytest.mark.parametrize("qtype,N,K,M", [(synth.Q4_K, 130, 768, 64), (synth.Q6_K, 70, 1024, 100),
                                         (synth.Q8_0, 77, 544, 33)])
def test_any_magnitude_int8_prefill(cuda_lib, qtype, N, K, M, scale):
    """The int8 mma.sync prefill (exact block dots, fp32 scales) at both ends."""
    cuda_lib.set_prefill_path(cuda_lib.PREFILL_INT8)
    try:
        W = synth.weights(qtype, N, K, seed=N + K)
        x = (synth.activations(M, K, seed=M).astype(np.float64) * scale).astype(np.float32)
        _check(cuda_lib, qtype, W, N, K, x, scale, f"int8 prefill type {qtype} scale={scale}")
    finally:
        cuda_lib.set_prefill_path(cuda_lib.PREFILL_AUTO)


@pytest.mark.parametrize("qtype,N,K,M", [(synth.Q4_K, 200, 2048, 300), (synth.Q6_K, 129, 5120, 8),
                                         (synth.Q8_0, 140, 1024, 64), (synth.Q4_K, 77, 2048, 4)])
def test_x_only_4_byte_aligned(cuda_lib, qtype, N, K, M):
    """x one float past a 16-byte boundary (the ABI asks for 4-byte alignment):
    the fp16 quantiser then reads it with 4-byte loads."""
    import torch
    W = synth.weights(qtype, N, K, seed=N + K + 1)
    x = synth.activations(M, K, seed=M + 1)
    buf = torch.zeros(M * K + 4, dtype=torch.float32, device="cuda")
    xd = buf[1:1 + M * K].view(M, K)
    xd.copy_(torch.from_numpy(x))
    assert xd.data_ptr() % 16 == 4
    y = cuda_lib.qmm(qtype, _dev(W), N, K, xd).cpu().numpy().astype(np.float64)
    yo, A = O.qmm(qtype, W, N, K, x)
    assert np.all(np.abs(y - yo) <= REL * A + ABS)
