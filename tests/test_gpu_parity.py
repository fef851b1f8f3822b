"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bars: dequantisation and the activation quantiser bit-for-bit; qmm outputs
within |y_gpu - y_oracle| <= 2e-3 * sum_k |w_k xhat_k| + 1e-5 element-wise
(the library's stated accuracy), at small shapes spanning several tiles and
ragged tails, and at the full workload sizes on sampled output rows."""
import numpy as np
import pytest

import oracle as O
import synth

pytestmark = pytest.mark.gpu

REL, ABS = 2e-3, 1e-5


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _assert_within_bound(y_gpu, y_or, A, what=""):
    err = np.abs(y_gpu.astype(np.float64) - y_or)
    bound = REL * A + ABS
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside the bound; worst "
                           f"err {err[bad].max():.3e} vs bound {bound[bad].min():.3e}")


def _run_qmm(q, qtype, W, N, K, x):
    y = q.qmm(qtype, _dev(W), N, K, _dev(x))
    assert q.qmm_device_status() == 0
    return y.cpu().numpy()


# ------------------------------------------------------------------ dequant

@pytest.mark.parametrize("qtype", [synth.Q8_0, synth.Q4_K, synth.Q6_K])
@pytest.mark.parametrize("nblocks", [1, 3, 8, 37, 1000])
def test_dequant_bitwise(cuda_lib, qtype, nblocks):
    W = synth.weights(qtype, nblocks, synth.BLOCK_WEIGHTS[qtype], seed=nblocks + 10 * qtype)
    n = nblocks * synth.BLOCK_WEIGHTS[qtype]
    got = cuda_lib.qmm_dequant(qtype, _dev(W), n).cpu().numpy()
    want = O.dequant(qtype, W, n)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("qtype", [synth.Q5_K, synth.Q3_K, synth.Q2_K])
@pytest.mark.parametrize("nblocks", [1, 3, 37, 1000])
def test_dequant_bitwise_other_k_quants(cuda_lib, qtype, nblocks):
    """Q5_K, Q3_K, Q2_K dequantised on the GPU bit for bit as the oracle."""
    W = synth.weights(qtype, nblocks, 256, seed=nblocks + 10 * qtype)
    n = nblocks * 256
    got = cuda_lib.qmm_dequant(qtype, _dev(W), n).cpu().numpy()
    want = O.dequant(qtype, W, n)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("cfg,idx", [(0, 0), (1, 0), (2, 0), (3, 2), (3, 6), (4, 0)])
def test_dequant_bitwise_workload_weights(cuda_lib, cfg, idx):
    name, qtype, K, N = synth.CONFIGS[cfg]["mats"][idx]
    W = synth.config_weights(cfg, idx)
    n = N * K
    got = cuda_lib.qmm_dequant(qtype, _dev(W), n).cpu().numpy()
    want = O.dequant(qtype, W, n)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), name


def test_dequant_extreme_fields(cuda_lib):
    """Extreme scale/min values and fp16 subnormals, packed by the oracle."""
    blocks = []
    for v in (0, 1, 31, 32, 63):
        sc = np.full(8, v, np.uint8)
        m = np.full(8, 63 - v, np.uint8)
        qv = (np.arange(256) % 16).astype(np.uint8)
        for db in (0x0001, 0x03FF, 0x3C00, 0x7BFF, 0x8000):
            blocks.append(O.pack_q4_k(db, 0x0400 | v, sc, m, qv))
    W = np.concatenate(blocks)
    n = len(blocks) * 256
    got = cuda_lib.qmm_dequant(synth.Q4_K, _dev(W), n).cpu().numpy()
    want = O.dequant(synth.Q4_K, W, n)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    blocks = [O.pack_q6_k(db, np.array([-128, 127, 0, -1] * 4, np.int8),
                          (np.arange(256) % 64).astype(np.uint8))
              for db in (0x0001, 0x3C00, 0x7BFF, 0xFBFF)]
    W = np.concatenate(blocks)
    got = cuda_lib.qmm_dequant(synth.Q6_K, _dev(W), 1024).cpu().numpy()
    want = O.dequant(synth.Q6_K, W, 1024)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


# ----------------------------------------------------------------- quantiser

@pytest.mark.parametrize("M,K", [(1, 32), (1, 2048), (3, 5120), (8, 17408), (64, 4096)])
def test_quantizer_bitwise(cuda_lib, M, K):
    x = synth.activations(M, K, seed=M * 7 + K, outlier_frac=0.01)
    x[0, :32] = 0.0                                  # all-zero block
    if K >= 64:
        x[-1, 32:64] = np.float32(127.0) * np.arange(-16, 16) / 16   # exact halves
    q, d, s = cuda_lib.qmm_quantize_act(_dev(x))
    qo, do, so = O.quantize_act(x)
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(d.cpu().numpy().view(np.uint32), do.view(np.uint32))
    assert np.array_equal(s.cpu().numpy(), so)


# ----------------------------------------------------------- qmm, small shapes

SMALL = [
    # (qtype, N, K, M)
    (synth.Q4_K, 37, 256, 1), (synth.Q4_K, 300, 1280, 1), (synth.Q4_K, 129, 2048, 2),
    (synth.Q4_K, 64, 5120, 3), (synth.Q4_K, 77, 768, 4), (synth.Q4_K, 50, 2304, 8),
    (synth.Q6_K, 37, 256, 1), (synth.Q6_K, 301, 1280, 1), (synth.Q6_K, 65, 5120, 2),
    (synth.Q6_K, 33, 768, 5), (synth.Q6_K, 40, 2048, 8), (synth.Q6_K, 8, 17408, 1),
    (synth.Q8_0, 33, 32, 1), (synth.Q8_0, 256, 512, 1), (synth.Q8_0, 100, 1056, 2),
    (synth.Q8_0, 17, 4096, 7), (synth.Q8_0, 1, 96, 8),
]


@pytest.mark.parametrize("qtype,N,K,M", SMALL)
def test_qmm_decode_small(cuda_lib, qtype, N, K, M):
    W = synth.weights(qtype, N, K, seed=N + K + M)
    x = synth.activations(M, K, seed=N * K + M, outlier_frac=0.01)
    y = _run_qmm(cuda_lib, qtype, W, N, K, x)
    yo, A = O.qmm(qtype, W, N, K, x)
    _assert_within_bound(y, yo, A, f"type {qtype} N={N} K={K} M={M}")


# Q4_K decode on the tensor-core kernel (the default path from M = 4 on,
# forced here for every M): groups of sixteen rows split between warps and
# CTAs (N=16 over two CTAs holding 8 rows each), ragged N and a K whose
# super-blocks do not fill the last stage chunk, every M from 2 to 8.
MMA_DECODE = [(16, 8192, 2), (16, 8192, 3), (1000, 4352, 5), (77, 256, 8), (2048, 2048, 4),
              (300, 5120, 6), (9, 1024, 7), (4096, 4096, 8), (5120, 17408, 4),
              # x of all of K does not fit: K taken in phases
              (300, 17408, 8), (40, 17408, 6)]

# Q6_K: rows that are not 16-byte multiples (N*K ragged at the end of the
# matrix: the last bytes are loaded after the wait), odd and even
# super-blocks of a chunk, K in phases (K = 17408 at M = 8), ragged N.
MMA_DECODE_Q6K = [(301, 1536, 2), (1024, 5120, 4), (300, 17408, 8), (77, 2048, 3), (16, 4608, 5),
                  (5120, 17408, 2), (129, 5120, 7)]


@pytest.fixture
def decode_path(cuda_lib):
    def set_path(p):
        cuda_lib.set_decode_path(p)
    yield set_path
    cuda_lib.set_decode_path(cuda_lib.DECODE_AUTO)


@pytest.mark.parametrize("N,K,M", MMA_DECODE)
def test_qmm_decode_tensor_core(cuda_lib, decode_path, N, K, M):
    decode_path(cuda_lib.DECODE_TENSOR)
    W = synth.weights(synth.Q4_K, N, K, seed=N + K + 3 * M)
    x = synth.activations(M, K, seed=N * K + 5 * M, outlier_frac=0.01)
    before = cuda_lib.qmm_launch_count()
    y = _run_qmm(cuda_lib, synth.Q4_K, W, N, K, x)
    assert cuda_lib.qmm_launch_count() - before == 2  # the quantiser, then the tensor-core kernel
    yo, A = O.qmm(synth.Q4_K, W, N, K, x)
    _assert_within_bound(y, yo, A, f"tensor-core decode N={N} K={K} M={M}")


@pytest.mark.parametrize("N,K,M", MMA_DECODE_Q6K)
def test_qmm_decode_tensor_core_q6k(cuda_lib, decode_path, N, K, M):
    decode_path(cuda_lib.DECODE_TENSOR)
    W = synth.weights(synth.Q6_K, N, K, seed=N + K + 7 * M)
    x = synth.activations(M, K, seed=N * K + 11 * M, outlier_frac=0.01)
    before = cuda_lib.qmm_launch_count()
    y = _run_qmm(cuda_lib, synth.Q6_K, W, N, K, x)
    assert cuda_lib.qmm_launch_count() - before == 2  # the quantiser, then the tensor-core kernel
    yo, A = O.qmm(synth.Q6_K, W, N, K, x)
    _assert_within_bound(y, yo, A, f"tensor-core decode Q6_K N={N} K={K} M={M}")


@pytest.mark.parametrize("M", [2, 4, 8])
def test_qmm_decode_block_path_on_request(cuda_lib, decode_path, M):
    decode_path(cuda_lib.DECODE_BLOCK)
    N, K = 300, 5120
    W = synth.weights(synth.Q4_K, N, K, seed=31 + M)
    x = synth.activations(M, K, seed=32 + M, outlier_frac=0.01)
    before = cuda_lib.qmm_launch_count()
    y = _run_qmm(cuda_lib, synth.Q4_K, W, N, K, x)
    assert cuda_lib.qmm_launch_count() - before == 1
    yo, A = O.qmm(synth.Q4_K, W, N, K, x)
    _assert_within_bound(y, yo, A, f"block-per-lane decode N={N} K={K} M={M}")


@pytest.mark.parametrize("M", [3, 4])
def test_small_k_q6k_decode_on_block_per_lane(cuda_lib, M):
    """Q6_K with K <= 2048 at M = 3, 4 takes the block-per-lane kernel (one
    launch, x quantised inside it) by default, and matches the oracle."""
    N, K = 3000, 2048
    W = synth.weights(synth.Q6_K, N, K, seed=M + 11)
    x = synth.activations(M, K, seed=M + 12)
    before = cuda_lib.qmm_launch_count()
    y = _run_qmm(cuda_lib, synth.Q6_K, W, N, K, x)
    assert cuda_lib.qmm_launch_count() - before == 1
    yo, A = O.qmm(synth.Q6_K, W, N, K, x)
    _assert_within_bound(y, yo, A, f"Q6_K K={K} M={M}")


@pytest.mark.parametrize("qtype,K", [(synth.Q4_K, 5120), (synth.Q6_K, 17408)])
def test_qmm_decode_tensor_core_is_deterministic(cuda_lib, decode_path, qtype, K):
    import torch
    decode_path(cuda_lib.DECODE_TENSOR)
    N, M = 300, 8
    W = _dev(synth.weights(qtype, N, K, seed=21))
    x = _dev(synth.activations(M, K, seed=22))
    y1 = cuda_lib.qmm(qtype, W, N, K, x)
    for _ in range(3):
        assert torch.equal(y1, cuda_lib.qmm(qtype, W, N, K, x))


GEMM_SMALL = [
    (synth.Q4_K, 70, 512, 9), (synth.Q4_K, 130, 768, 64), (synth.Q4_K, 64, 256, 100),
    (synth.Q6_K, 70, 512, 9), (synth.Q6_K, 129, 1024, 65), (synth.Q8_0, 70, 544, 33),
    (synth.Q8_0, 64, 256, 64), (synth.Q4_K, 200, 4096, 130),
]


@pytest.mark.parametrize("qtype,N,K,M", GEMM_SMALL)
def test_qmm_prefill_small(cuda_lib, qtype, N, K, M):
    W = synth.weights(qtype, N, K, seed=N + K + M + 1)
    x = synth.activations(M, K, seed=N * K + M + 1, outlier_frac=0.01)
    y = _run_qmm(cuda_lib, qtype, W, N, K, x)
    yo, A = O.qmm(qtype, W, N, K, x)
    _assert_within_bound(y, yo, A, f"type {qtype} N={N} K={K} M={M}")


# Q6_K and Q8_0 prefill on tcgen05 (the dequantisers copy their rows' raw
# bytes): ragged N with the matrix ending off a 4-byte boundary, an odd
# number of super-blocks per row (rows alternately 4- and 2-byte aligned),
# split K (two CTAs per tile), M in each token-tile size.
PREFILL_TC_OTHER = [(synth.Q6_K, 301, 768, 70), (synth.Q6_K, 1000, 2048, 64), (synth.Q6_K, 130, 5120, 300),
                    (synth.Q6_K, 77, 256, 9), (synth.Q8_0, 301, 768, 70), (synth.Q8_0, 1000, 2048, 64),
                    (synth.Q8_0, 257, 4352, 200), (synth.Q8_0, 33, 256, 129)]


@pytest.mark.parametrize("qtype,N,K,M", PREFILL_TC_OTHER)
def test_qmm_prefill_tcgen05_q6k_q8_0(cuda_lib, qtype, N, K, M):
    W = synth.weights(qtype, N, K, seed=N + K + M + 17)
    x = synth.activations(M, K, seed=N * K + M + 17, outlier_frac=0.01)
    y = _run_qmm(cuda_lib, qtype, W, N, K, x)
    yo, A = O.qmm(qtype, W, N, K, x)
    _assert_within_bound(y, yo, A, f"tcgen05 prefill type {qtype} N={N} K={K} M={M}")


# Q4_K prefill shapes on the tcgen05 GEMM with ragged M and N; the two with
# few tiles (256 x 70 and 384 x 40) split K in two, so each output is the
# sum of two partial products added onto a zeroed y.
STREAM_K = [(1000, 2048, 300), (256, 8192, 70), (384, 3072, 40)]


@pytest.mark.parametrize("N,K,M", STREAM_K)
def test_qmm_prefill_split_tiles(cuda_lib, N, K, M):
    qtype = synth.Q4_K
    W = synth.weights(qtype, N, K, seed=N + K + M + 7)
    x = synth.activations(M, K, seed=N * K + M + 7, outlier_frac=0.01)
    y = _run_qmm(cuda_lib, qtype, W, N, K, x)
    yo, A = O.qmm(qtype, W, N, K, x)
    _assert_within_bound(y, yo, A, f"split tiles N={N} K={K} M={M}")


@pytest.fixture
def prefill_path(cuda_lib):
    def set_path(p):
        cuda_lib.set_prefill_path(p)
    yield set_path
    cuda_lib.set_prefill_path(cuda_lib.PREFILL_AUTO)


# The int8 mma.sync prefill (exact int32 block dots) forced for every shape,
# including K multiples of 256 that would otherwise take tcgen05: tiles of 64
# rows with ragged M and N, all three types.
PREFILL_INT8 = GEMM_SMALL + PREFILL_TC_OTHER + [(synth.Q4_K, 1000, 2048, 300), (synth.Q6_K, 200, 5120, 130)]


@pytest.mark.parametrize("qtype,N,K,M", PREFILL_INT8)
def test_qmm_prefill_int8_path(cuda_lib, prefill_path, qtype, N, K, M):
    prefill_path(cuda_lib.PREFILL_INT8)
    W = synth.weights(qtype, N, K, seed=N + K + M + 23)
    x = synth.activations(M, K, seed=N * K + M + 23, outlier_frac=0.01)
    before = cuda_lib.qmm_launch_count()
    y = _run_qmm(cuda_lib, qtype, W, N, K, x)
    assert cuda_lib.qmm_launch_count() - before == 2  # the quantiser, then the mma.sync GEMM
    yo, A = O.qmm(qtype, W, N, K, x)
    _assert_within_bound(y, yo, A, f"int8 prefill type {qtype} N={N} K={K} M={M}")


def test_qmm_prefill_int8_path_workload_full_size(cuda_lib, prefill_path):
    """The Mistral-7B MLP up projection at M=512 on the mma.sync kernel, on
    sampled rows against the oracle."""
    prefill_path(cuda_lib.PREFILL_INT8)
    name, qtype, K, N = synth.CONFIGS[4]["mats"][0]
    W = synth.config_weights(4, 0)
    x = synth.config_activations(4, 512, K)
    y = cuda_lib.qmm(qtype, _dev(W), N, K, _dev(x)).cpu().numpy()
    assert cuda_lib.qmm_device_status() == 0
    rows = _sample_rows(N, k=96, seed=5)
    rb = synth.row_bytes(qtype, K)
    yo, A = O.qmm(qtype, W.reshape(N, rb)[rows], len(rows), K, x)
    _assert_within_bound(y[:, rows], yo, A, f"int8 prefill {name}")


def test_qmm_prefill_is_deterministic(cuda_lib):
    import torch
    N, K, M = STREAM_K[1]
    W = _dev(synth.weights(synth.Q4_K, N, K, seed=11))
    x = _dev(synth.activations(M, K, seed=12))
    y1 = torch.full((M, N), float("nan"), device="cuda")
    cuda_lib.qmm(synth.Q4_K, W, N, K, x, y=y1)
    for _ in range(3):
        y2 = cuda_lib.qmm(synth.Q4_K, W, N, K, x)
        assert torch.equal(y1, y2)
    assert cuda_lib.qmm_device_status() == 0


def test_qmm_prefill_in_cuda_graph_replays(cuda_lib):
    """The split-tile hand-off flags are set and cleared inside each launch,
    so replays of a captured call give the eager result every time."""
    import torch
    N, K, M = STREAM_K[1]
    W = _dev(synth.weights(synth.Q4_K, N, K, seed=13))
    x = _dev(synth.activations(M, K, seed=14))
    ref = cuda_lib.qmm(synth.Q4_K, W, N, K, x)
    st = torch.cuda.Stream()
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    with torch.cuda.stream(st):
        cuda_lib.qmm(synth.Q4_K, W, N, K, x, y=y, stream=st)  # workspace of this stream
    st.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        cuda_lib.qmm(synth.Q4_K, W, N, K, x, y=y, stream=st)
    for _ in range(3):
        y.fill_(float("nan"))
        with torch.cuda.stream(st):
            g.replay()
        st.synchronize()
        assert torch.equal(y, ref)
    assert cuda_lib.qmm_device_status() == 0


# qmm_group: several matrices reading one x, one decode launch (M <= 2), or the
# quantiser and one tensor-core launch (3 <= M <= 8)
QWEN_QKV = [(q, N) for (nm, q, K, N) in synth.QWEN3_14B_LAYER if nm in ("q", "k", "v")]
QWEN_GATE_UP = [(q, N) for (nm, q, K, N) in synth.QWEN3_14B_LAYER if nm in ("gate", "up")]
MIXED = [(synth.Q4_K, 5), (synth.Q6_K, 0), (synth.Q6_K, 3000), (synth.Q8_0, 1), (synth.Q4_K, 700)]


@pytest.mark.parametrize("group,K,M", [(QWEN_QKV, 5120, 1), (QWEN_QKV, 5120, 4), (QWEN_GATE_UP, 5120, 1),
                                       (QWEN_GATE_UP, 5120, 8), (MIXED, 1024, 2), (MIXED, 1024, 16)])
def test_qmm_group_matches_oracle(cuda_lib, group, K, M):
    Ws = [synth.weights(q, N, K, seed=100 + i) for i, (q, N) in enumerate(group)]
    x = synth.activations(M, K, seed=200 + M)
    before = cuda_lib.qmm_launch_count()
    ys = cuda_lib.qmm_group([(q, _dev(W), N) for (q, N), W in zip(group, Ws)], K, _dev(x))
    assert cuda_lib.qmm_device_status() == 0
    if M == 1:
        assert cuda_lib.qmm_launch_count() - before == 1  # the whole group, one launch
    if group is not MIXED and M >= 3:
        # the tensor-core path: x quantised once, one decode launch for the group
        assert cuda_lib.qmm_launch_count() - before == 2
    for (q, N), W, y in zip(group, Ws, ys):
        if N == 0:
            continue
        yo, A = O.qmm(q, W, N, K, x)
        _assert_within_bound(y.cpu().numpy(), yo, A, f"group entry type {q} N={N} K={K} M={M}")


def test_qmm_is_deterministic_and_overwrites_y(cuda_lib):
    import torch
    qtype, N, K = synth.Q6_K, 300, 5120
    W = _dev(synth.weights(qtype, N, K, seed=3))
    x = _dev(synth.activations(2, K, seed=4))
    y1 = torch.full((2, N), float("nan"), device="cuda")
    cuda_lib.qmm(qtype, W, N, K, x, y=y1)
    y2 = cuda_lib.qmm(qtype, W, N, K, x)
    assert torch.equal(y1, y2)


def test_qmm_zero_k_and_empty(cuda_lib):
    import torch
    y = torch.full((3, 5), 7.0, device="cuda")
    x = torch.zeros((3, 0), device="cuda")
    W = torch.zeros(16, dtype=torch.uint8, device="cuda")
    cuda_lib.qmm(synth.Q4_K, W, 5, 0, x, y=y)
    assert torch.all(y.cpu() == 0)


def test_qmm_on_side_stream(cuda_lib):
    import torch
    qtype, N, K = synth.Q4_K, 256, 2048
    W = synth.weights(qtype, N, K, seed=5)
    x = synth.activations(1, K, seed=6)
    s = torch.cuda.Stream()
    Wd, xd = _dev(W), _dev(x)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        y = cuda_lib.qmm(qtype, Wd, N, K, xd, stream=s)
    s.synchronize()
    yo, A = O.qmm(qtype, W, N, K, x)
    _assert_within_bound(y.cpu().numpy(), yo, A)


# ------------------------------------------- the workloads at full size

def _sample_rows(N, k=384, seed=0):
    rng = np.random.default_rng(seed)
    rows = set(range(min(N, 64))) | set(range(max(0, N - 64), N))
    rows |= set(rng.choice(N, size=min(N, k), replace=False).tolist())
    return np.array(sorted(rows))


@pytest.mark.parametrize("cfg", [0, 1, 2, 3])
def test_qmm_workloads_full_size(cuda_lib, cfg):
    c = synth.CONFIGS[cfg]
    for idx, (name, qtype, K, N) in enumerate(c["mats"]):
        W = synth.config_weights(cfg, idx)
        Wdev = _dev(W)
        rb = synth.row_bytes(qtype, K)
        for M in c["M"]:
            x = synth.config_activations(cfg, M, K)
            y = cuda_lib.qmm(qtype, Wdev, N, K, _dev(x)).cpu().numpy()
            assert cuda_lib.qmm_device_status() == 0
            rows = _sample_rows(N, seed=idx + M) if N * K > 4_000_000 else np.arange(N)
            Wr = W.reshape(N, rb)[rows]
            yo, A = O.qmm(qtype, Wr, len(rows), K, x)
            _assert_within_bound(y[:, rows], yo, A, f"cfg {cfg} {name} M={M}")


def test_qmm_prefill_workload_full_size(cuda_lib):
    c = synth.CONFIGS[4]
    for idx, (name, qtype, K, N) in enumerate(c["mats"]):
        W = synth.config_weights(4, idx)
        x = synth.config_activations(4, 512, K)
        y = cuda_lib.qmm(qtype, _dev(W), N, K, _dev(x)).cpu().numpy()
        assert cuda_lib.qmm_device_status() == 0
        rows = _sample_rows(N, k=96, seed=idx)
        rb = synth.row_bytes(qtype, K)
        yo, A = O.qmm(qtype, W.reshape(N, rb)[rows], len(rows), K, x)
        _assert_within_bound(y[:, rows], yo, A, f"prefill {name}")


# the prefill shapes the bench times beyond the Mistral-7B MLP, with the
# bench's inputs: the Q6_K v and down of the Qwen3-14B layer (raw stages by
# TMA, K split in clusters), Q8_0 and the other K-quants in the Mistral up
# shape (raw stages by TMA), all at M = 512
PREFILL_BENCH = [("qwen3_14b_v", 3, 2), ("qwen3_14b_down", 3, 6), ("q8_0_mistral_up", synth.Q8_0, 4100),
                 ("q5_k_mistral_up", synth.Q5_K, 6000 + synth.Q5_K), ("q3_k_mistral_up", synth.Q3_K, 6000 + synth.Q3_K),
                 ("q2_k_mistral_up", synth.Q2_K, 6000 + synth.Q2_K)]


@pytest.mark.parametrize("name,a,b", PREFILL_BENCH)
def test_qmm_prefill_bench_shapes_full_size(cuda_lib, name, a, b):
    """Sampled rows (the first and last 64 and 96 random ones) of the
    prefill products the bench times, against the oracle within the bound."""
    if name.startswith("qwen3"):
        qtype, K, N = synth.CONFIGS[a]["mats"][b][1:]
        W = synth.config_weights(a, b)
    else:
        qtype, K, N = a, 4096, 14336
        W = synth.weights(qtype, N, K, seed=b)
    x = synth.config_activations(4, 512, K)
    y = cuda_lib.qmm(qtype, _dev(W), N, K, _dev(x)).cpu().numpy()
    assert cuda_lib.qmm_device_status() == 0
    rows = _sample_rows(N, k=96, seed=N)
    rb = synth.row_bytes(qtype, K)
    yo, A = O.qmm(qtype, W.reshape(N, rb)[rows], len(rows), K, x)
    _assert_within_bound(y[:, rows], yo, A, f"prefill {name}")


# ------------------------------------------- exact integer special cases

def _int_activations(rng, M, K):
    """Integer activations with max |x| = 127 in every block of 32, so the
    quantiser maps them to themselves with scale 1."""
    xi = rng.integers(-127, 128, (M, K)).astype(np.float64)
    xi[:, 3::32] = 127.0
    return xi


@pytest.mark.parametrize("N,K,M", [(257, 1024, 1), (129, 2048, 2), (64, 512, 5), (33, 4096, 8),
                                   (70, 1024, 24)])
def test_qmm_q8_0_unit_scale_is_exact(cuda_lib, N, K, M):
    """d = 1 Q8_0 weights and integer activations: every path must return the
    exact integer product (all partial sums stay below 2^24)."""
    rng = np.random.default_rng(N + K + M)
    qw = rng.integers(-127, 128, (N, K)).astype(np.int8)
    W = np.concatenate([O.pack_q8_0(0x3C00, qw[n, 32 * b:32 * b + 32])
                        for n in range(N) for b in range(K // 32)])
    xi = _int_activations(rng, M, K)
    y = _run_qmm(cuda_lib, synth.Q8_0, W, N, K, xi.astype(np.float32))
    assert np.array_equal(y.astype(np.float64), xi @ qw.astype(np.float64).T)


@pytest.mark.parametrize("N,K,M", [(300, 2048, 1), (129, 5120, 1), (64, 1024, 3), (40, 2048, 8),
                                   (70, 768, 16)])
def test_qmm_q4_k_unit_scale_is_exact(cuda_lib, N, K, M):
    """Q4_K with d = 1, dmin = 0, every scale 1: w = q, so y is an exact
    integer product; checks the unpacking and every index exactly."""
    rng = np.random.default_rng(3 * N + K + M)
    q = rng.integers(0, 16, (N, K // 256, 256)).astype(np.uint8)
    W = np.concatenate([O.pack_q4_k(0x3C00, 0x0000, np.ones(8, np.uint8), np.zeros(8, np.uint8), q[n, b])
                        for n in range(N) for b in range(K // 256)])
    xi = _int_activations(rng, M, K)
    y = _run_qmm(cuda_lib, synth.Q4_K, W, N, K, xi.astype(np.float32))
    assert np.array_equal(y.astype(np.float64), xi @ q.reshape(N, K).astype(np.float64).T)


@pytest.mark.parametrize("N,K,M", [(300, 2048, 1), (65, 5120, 1), (40, 1280, 4), (70, 1024, 16)])
def test_qmm_q6_k_unit_scale_is_exact(cuda_lib, N, K, M):
    """Q6_K with d = 1 and every scale 1: w = q - 32, exact integer product."""
    rng = np.random.default_rng(5 * N + K + M)
    q = rng.integers(0, 64, (N, K // 256, 256)).astype(np.uint8)
    W = np.concatenate([O.pack_q6_k(0x3C00, np.ones(16, np.int8), q[n, b])
                        for n in range(N) for b in range(K // 256)])
    xi = _int_activations(rng, M, K)
    y = _run_qmm(cuda_lib, synth.Q6_K, W, N, K, xi.astype(np.float32))
    assert np.array_equal(y.astype(np.float64),
                          xi @ (q.reshape(N, K).astype(np.float64) - 32).T)


# ------------------------------------------- qmm_t: the value side of attention

def _run_qmm_t(q, W, H, N, K, x, stream=None):
    y = q.qmm_t(synth.Q8_0, _dev(W), H, N, K, _dev(x), stream=stream)
    assert q.qmm_device_status() == 0
    return y.cpu().numpy()


QMM_T_CASES = [(1, 1, 32, 1), (1, 16, 128, 5), (2, 300, 128, 5), (3, 1000, 64, 8), (1, 777, 256, 16),
               (2, 129, 96, 17), (4, 2049, 160, 3), (1, 5000, 224, 1), (5, 64, 32, 2), (6, 12345, 128, 4),
               (2, 4000, 192, 6),
               # 137 chunks of one matrix: the last CTA adds them over several passes
               (1, 70000, 64, 3)]


@pytest.mark.parametrize("H,N,K,M", QMM_T_CASES)
def test_qmm_t_matches_oracle(cuda_lib, H, N, K, M):
    """Probability rows and signed rows, against the f64 oracle, element-wise
    within the stated bound (M > 16 takes two launches; ragged stages)."""
    W = synth.kv_cache(H, N, K, seed=H * 1000 + N)
    for x in (synth.attention_probs(H, M, N, seed=N + M),
              np.random.default_rng(N).standard_normal((H, M, N)).astype(np.float32)):
        got = _run_qmm_t(cuda_lib, W, H, N, K, x)
        want, A = O.qmm_t(O.Q8_0, W, H, N, K, x)
        _assert_within_bound(got, want, A, f"qmm_t H={H} N={N} K={K} M={M}")


@pytest.mark.parametrize("scale", [1e-30, 1e-6, 1.0, 1e4, 1e30])
def test_qmm_t_any_magnitude_of_x(cuda_lib, scale):
    """The per-chunk power-of-two scaling keeps tiny and huge x inside fp16's
    normal range: the bound holds from 1e-30 to 1e30."""
    H, N, K, M = 2, 700, 128, 5
    W = synth.kv_cache(H, N, K, seed=77)
    x = (np.random.default_rng(8).standard_normal((H, M, N)) * scale).astype(np.float32)
    got = _run_qmm_t(cuda_lib, W, H, N, K, x)
    want, A = O.qmm_t(O.Q8_0, W, H, N, K, x)
    _assert_within_bound(got, want, A, f"scale {scale}")


def test_qmm_t_deterministic_overwrites_and_empty(cuda_lib):
    import torch
    H, N, K, M = 3, 3000, 128, 5
    W = _dev(synth.kv_cache(H, N, K, seed=4))
    x = _dev(synth.attention_probs(H, M, N, seed=4))
    y1 = cuda_lib.qmm_t(synth.Q8_0, W, H, N, K, x)
    y2 = torch.full_like(y1, float("nan"))
    cuda_lib.qmm_t(synth.Q8_0, W, H, N, K, x, y=y2)
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))
    # N = 0: y = 0
    y0 = torch.full((H, M, K), 7.0, device="cuda")
    cuda_lib.qmm_t(synth.Q8_0, W, H, 0, K, torch.zeros((H, M, 0), device="cuda"), y=y0)
    assert torch.count_nonzero(y0).item() == 0
    assert cuda_lib.qmm_device_status() == 0


def test_qmm_t_alternating_shapes_and_streams(cuda_lib):
    """The per-matrix counters return to zero after every call: calls of
    different H, on the default and on a side stream, all stay right."""
    import torch
    side = torch.cuda.Stream()
    for i, (H, N, K, M) in enumerate([(8, 4096, 128, 5), (2, 100, 64, 1), (16, 333, 128, 8), (8, 4096, 128, 5)]):
        W = synth.kv_cache(H, N, K, seed=40 + i)
        x = synth.attention_probs(H, M, N, seed=41 + i)
        st = side if i % 2 else None
        if st is not None:
            with torch.cuda.stream(st):
                Wd, xd = _dev(W), _dev(x)
                y = cuda_lib.qmm_t(synth.Q8_0, Wd, H, N, K, xd, stream=st)
            st.synchronize()
            got = y.cpu().numpy()
        else:
            got = _run_qmm_t(cuda_lib, W, H, N, K, x)
        want, A = O.qmm_t(O.Q8_0, W, H, N, K, x)
        _assert_within_bound(got, want, A, f"call {i}")


def test_qmm_t_kv_cache_full_size(cuda_lib):
    """The Qwen3-14B-shaped value cache (8 heads x 32768 positions x 128) at
    the size the bench times: every output against the oracle."""
    c = synth.KV_CACHE
    H, N, K, M = c["H"], c["N"], c["K"], c["M"]
    W = synth.kv_cache(H, N, K, seed=9)
    x = synth.attention_probs(H, M, N, seed=9)
    got = _run_qmm_t(cuda_lib, W, H, N, K, x)
    want, A = O.qmm_t(O.Q8_0, W, H, N, K, x)
    _assert_within_bound(got, want, A, "kv cache full size")


@pytest.mark.parametrize("N,K,M", [(4096, 128, 5), (777, 64, 1), (32768, 128, 8), (1500, 256, 4)])
def test_attention_scores_on_q8_0_key_cache(cuda_lib, N, K, M):
    """The score side over a q8_0 key cache is qmm itself: N cached positions of
    head_dim K, M query heads (the queries quantised as any activation)."""
    W = synth.kv_cache(1, N, K, seed=N + K)
    x = synth.activations(M, K, seed=M + K)
    got = _run_qmm(cuda_lib, synth.Q8_0, W, N, K, x)
    want, A = O.qmm(synth.Q8_0, W, N, K, x)
    _assert_within_bound(got, want, A, f"scores N={N} K={K} M={M}")


# Large Q8_0 matrices at 3 <= M <= 8 run on the tcgen05 prefill kernel (the
# quantiser, then the GEMM); smaller ones stay on the block-per-lane decode.
# Sampled rows against the oracle.
@pytest.mark.parametrize("N,K,M,launches", [(4096, 4096, 5, 2), (4096, 4096, 8, 2), (12288, 4096, 3, 2),
                                            (4096, 4096, 4, 1), (2048, 4096, 8, 1)])
def test_q8_0_decode_route(cuda_lib, N, K, M, launches):
    q = cuda_lib
    W = synth.weights(synth.Q8_0, N, K, seed=N + M)
    x = synth.activations(M, K, seed=K + M, outlier_frac=0.01)
    before = q.qmm_launch_count()
    y = q.qmm(synth.Q8_0, _dev(W), N, K, _dev(x)).cpu().numpy()
    assert q.qmm_launch_count() - before == launches
    assert q.qmm_device_status() == 0
    rng = np.random.default_rng(N + K + M)
    rows = np.unique(np.concatenate([np.arange(130), np.arange(N - 130, N), rng.choice(N, 200, replace=False)]))
    rb = synth.row_bytes(synth.Q8_0, K)
    yo, A = O.qmm(synth.Q8_0, W.reshape(N, rb)[rows], len(rows), K, x)
    _assert_within_bound(y[:, rows], yo, A, f"Q8_0 N={N} K={K} M={M}")
