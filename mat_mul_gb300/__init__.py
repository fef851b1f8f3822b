"""Python binding of libqmm (include/qmm.h): argument marshalling only.

Every step of the computation runs in the CUDA kernels of libqmm.so; torch is
used for device memory and streams.  There is no CPU fallback: when the
library is missing or no GPU is present the calls raise.

    import mat_mul_gb300 as q
    y = q.qmm(q.Q4_K, W_blocks, N, K, x)          # x: cuda f32 [M, K] -> [M, N]
    ys = q.qmm_group([(q.Q4_K, Wg, N), (q.Q4_K, Wu, N)], K, x)   # one launch, shared x
    h = q.qmm_gate_up(q.Q4_K, Wg, q.Q4_K, Wu, N, K, x)           # silu(Wg x) * (Wu x)
    o = q.qmm_t(q.Q8_0, V_cache, H, T, D, p)      # p: [H, M, T] -> [H, M, D]
    w = q.qmm_dequant(q.Q6_K, blocks, n_elems)    # cuda f32 [n_elems]
"""
from __future__ import annotations

import ctypes
import os

Q8_0, Q4_K, Q6_K, Q5_K, Q3_K, Q2_K = 0, 1, 2, 3, 4, 5  # Q5_K, Q3_K, Q2_K: qmm_dequant only so far
BLOCK_BYTES = {Q8_0: 34, Q4_K: 144, Q6_K: 210, Q5_K: 176, Q3_K: 110, Q2_K: 84}
BLOCK_WEIGHTS = {Q8_0: 32, Q4_K: 256, Q6_K: 256, Q5_K: 256, Q3_K: 256, Q2_K: 256}

QMM_OK = 0
QMM_EINVAL_TYPE = -1
QMM_EINVAL_SHAPE = -2
QMM_EINVAL_PTR = -3
QMM_ENOMEM = -4
QMM_ECUDA = -5
QMM_ETIMEOUT = -6

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libqmm.so")

_lib = None


class QmmError(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        super().__init__(f"{_strerror(status)}: {detail}")


def build(force: bool = False) -> str:
    from . import buildlib
    return buildlib.build(force=force)


def load():
    """Load libqmm.so, (re)building it first when it is absent or older than
    its sources."""
    global _lib
    if _lib is not None:
        return _lib
    build()
    L = ctypes.CDLL(LIB_PATH)
    P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    L.qmm_dequant.argtypes = [I, P, I64, P]
    L.qmm.argtypes = [I, P, I64, I64, P, I64, P, P]
    L.qmm_noalloc.argtypes = [I, P, I64, I64, P, I64, P, P]
    L.qmm_quantize_act.argtypes = [P, I64, I64, P, P, P, P]
    L.qmm_group.argtypes = [I, P, P, P, I64, P, I64, P, P]
    L.qmm_t.argtypes = [I, P, I64, I64, I64, P, I64, P, P]
    L.qmm_gate_up.argtypes = [I, P, I, P, I64, I64, P, I64, P, P]
    L.qmm_strerror.argtypes = [I]
    L.qmm_strerror.restype = ctypes.c_char_p
    L.qmm_last_error.restype = ctypes.c_char_p
    L.qmm_device_status.argtypes = [P]
    L.qmm_launch_count.restype = I64
    L.qmm_set_decode_path.argtypes = [I]
    L.qmm_set_decode_path.restype = I
    L.qmm_set_prefill_path.argtypes = [I]
    L.qmm_set_prefill_path.restype = I
    L.qmm_inject_stall.argtypes = [I]
    L.qmm_inject_stall.restype = I
    for f in ("qmm_dequant", "qmm", "qmm_noalloc", "qmm_quantize_act", "qmm_device_status",
              "qmm_release", "qmm_group", "qmm_t", "qmm_gate_up"):
        getattr(L, f).restype = I
    _lib = L
    return L


def _strerror(status: int) -> str:
    return load().qmm_strerror(int(status)).decode()


def _check(rc: int):
    if rc != QMM_OK:
        raise QmmError(rc, load().qmm_last_error().decode())


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _require_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("libqmm takes device tensors; got a tensor on " + str(t.device))


def qmm_dequant(qtype: int, blocks, n_elems: int, out=None):
    """Unpack n_elems weights of type qtype from a uint8 device tensor."""
    import torch
    _require_cuda(blocks, out)
    if out is None:
        out = torch.empty(n_elems, dtype=torch.float32, device=blocks.device)
    _check(load().qmm_dequant(int(qtype), _ptr(blocks), int(n_elems), _ptr(out)))
    return out


def qmm(qtype: int, W, N: int, K: int, x, y=None, stream=None):
    """y[M,N] = W . x^T for a uint8 device tensor W of packed blocks and a
    device f32 tensor x of shape [M, K] (or [K])."""
    import torch
    _require_cuda(W, x, y)
    if x.dtype != torch.float32 or not x.is_contiguous():
        raise ValueError("x must be a contiguous float32 tensor")
    M = 1 if x.dim() == 1 else x.shape[0]
    if x.shape[-1] != K:
        raise ValueError(f"x has {x.shape[-1]} columns, K = {K}")
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    elif y.dtype != torch.float32 or not y.is_contiguous() or y.device != x.device or y.numel() < M * N:
        raise ValueError(f"y must be a contiguous float32 tensor on {x.device} with at least M*N = {M * N} elements")
    _check(load().qmm(int(qtype), _ptr(W), int(N), int(K), _ptr(x), int(M), _ptr(y),
                      _stream_handle(stream)))
    return y


def qmm_t(qtype: int, W, H: int, N: int, K: int, x, y=None, stream=None):
    """y[h, m, k] = sum_n x[h, m, n] * w[h, n, k] for H matrices of N rows of
    K weights (uint8 device tensor W of packed Q8_0 blocks) and a device f32
    tensor x of shape [H, M, N]; returns y of shape [H, M, K]."""
    import torch
    _require_cuda(W, x, y)
    if x.dtype != torch.float32 or not x.is_contiguous():
        raise ValueError("x must be a contiguous float32 tensor")
    if x.dim() != 3 or x.shape[0] != H or x.shape[2] != N:
        raise ValueError(f"x has shape {tuple(x.shape)}, expected [H={H}, M, N={N}]")
    M = x.shape[1]
    if y is None:
        y = torch.empty((H, M, K), dtype=torch.float32, device=x.device)
    _check(load().qmm_t(int(qtype), _ptr(W), int(H), int(N), int(K), _ptr(x), int(M), _ptr(y),
                        _stream_handle(stream)))
    return y


def qmm_group(items, K: int, x, stream=None):
    """Several products that read the same x [M, K] (or [K]): items is a list
    of (qtype, W, N) or (qtype, W, N, y); returns the list of y tensors
    [M, N_i].  With M <= 8 the group is one decode launch."""
    import torch
    if x.dtype != torch.float32 or not x.is_contiguous():
        raise ValueError("x must be a contiguous float32 tensor")
    M = 1 if x.dim() == 1 else x.shape[0]
    if x.shape[-1] != K:
        raise ValueError(f"x has {x.shape[-1]} columns, K = {K}")
    n = len(items)
    ys = []
    for it in items:
        y = it[3] if len(it) > 3 and it[3] is not None else torch.empty(
            (M, int(it[2])), dtype=torch.float32, device=x.device)
        _require_cuda(it[1], x, y)
        ys.append(y)
    types = (ctypes.c_int * max(n, 1))(*[int(it[0]) for it in items])
    Ws = (ctypes.c_void_p * max(n, 1))(*[_ptr(it[1]) for it in items])
    Ns = (ctypes.c_int64 * max(n, 1))(*[int(it[2]) for it in items])
    Ys = (ctypes.c_void_p * max(n, 1))(*[_ptr(y) for y in ys])
    _check(load().qmm_group(int(n), types, Ws, Ns, int(K), _ptr(x), int(M), Ys, _stream_handle(stream)))
    return ys


def qmm_gate_up(type_gate: int, W_gate, type_up: int, W_up, N: int, K: int, x, h=None, stream=None):
    """h[M,N] = silu(W_gate . x^T) * (W_up . x^T) for device x [M, K] (or
    [K]); one launch for M <= 2 when both matrices have one type."""
    import torch
    _require_cuda(W_gate, W_up, x, h)
    if x.dtype != torch.float32 or not x.is_contiguous():
        raise ValueError("x must be a contiguous float32 tensor")
    M = 1 if x.dim() == 1 else x.shape[0]
    if x.shape[-1] != K:
        raise ValueError(f"x has {x.shape[-1]} columns, K = {K}")
    if h is None:
        h = torch.empty((M, N), dtype=torch.float32, device=x.device)
    elif h.dtype != torch.float32 or not h.is_contiguous() or h.device != x.device or h.numel() < M * N:
        raise ValueError(f"h must be a contiguous float32 tensor on {x.device} with at least M*N = {M * N} elements")
    _check(load().qmm_gate_up(int(type_gate), _ptr(W_gate), int(type_up), _ptr(W_up), int(N), int(K), _ptr(x),
                              int(M), _ptr(h), _stream_handle(stream)))
    return h


def qmm_noalloc(qtype: int, W, N: int, K: int, x, y, stream=None):
    """Same product as qmm() without any device allocation by the library,
    for callers that keep all device memory in their own fixed pool or must
    not stall on cudaFree.  y [M, N] float32 must be given.  Uses a 16 MiB
    scratch inside the library image; calls that overlap on the GPU race on
    it."""
    import torch
    _require_cuda(W, x, y)
    if x.dtype != torch.float32 or not x.is_contiguous():
        raise ValueError("x must be a contiguous float32 tensor")
    M = 1 if x.dim() == 1 else x.shape[0]
    if x.shape[-1] != K:
        raise ValueError(f"x has {x.shape[-1]} columns, K = {K}")
    if y.dtype != torch.float32 or not y.is_contiguous() or y.device != x.device or y.numel() < M * N:
        raise ValueError(f"y must be a contiguous float32 tensor on {x.device} with at least M*N = {M * N} elements")
    _check(load().qmm_noalloc(int(qtype), _ptr(W), int(N), int(K), _ptr(x), int(M), _ptr(y),
                              _stream_handle(stream)))
    return y


def qmm_quantize_act(x, stream=None):
    """Return (q int8 [M,K], d f32 [M,K/32], s int32 [M,K/32]) for device x."""
    import torch
    _require_cuda(x)
    x2 = x if x.dim() == 2 else x.reshape(1, -1)
    M, K = x2.shape
    q = torch.empty((M, K), dtype=torch.int8, device=x.device)
    d = torch.empty((M, K // 32), dtype=torch.float32, device=x.device)
    s = torch.empty((M, K // 32), dtype=torch.int32, device=x.device)
    _check(load().qmm_quantize_act(_ptr(x2), int(M), int(K), _ptr(q), _ptr(d), _ptr(s),
                                   _stream_handle(stream)))
    return q, d, s


def qmm_device_status(stream=None) -> int:
    return int(load().qmm_device_status(_stream_handle(stream)))


def qmm_release() -> None:
    _check(load().qmm_release())


def qmm_launch_count() -> int:
    return int(load().qmm_launch_count())


# Decode kernel choice (qmm_set_decode_path in the C header).
DECODE_AUTO, DECODE_BLOCK, DECODE_TENSOR, DECODE_ROWS = 0, 1, 2, 3


def set_decode_path(path: int) -> int:
    """Select the decode kernel for every later call; returns the previous path."""
    rc = int(load().qmm_set_decode_path(int(path)))
    if rc < 0:
        raise QmmError(rc, load().qmm_last_error().decode())
    return rc


# Prefill kernel choice (qmm_set_prefill_path in the C header).
PREFILL_AUTO, PREFILL_INT8 = 0, 1


def set_prefill_path(path: int) -> int:
    """Select the prefill kernel for every later call; returns the previous path."""
    rc = int(load().qmm_set_prefill_path(int(path)))
    if rc < 0:
        raise QmmError(rc, load().qmm_last_error().decode())
    return rc


def inject_stall(launches: int) -> int:
    """Failure-detection test hook: the next `launches` weight-streaming
    launches stop their first CTA's copies after one stage, so a bounded wait
    expires and qmm_device_status() reports QMM_ETIMEOUT.  Returns the
    previous pending count."""
    rc = int(load().qmm_inject_stall(int(launches)))
    if rc < 0:
        raise QmmError(rc, load().qmm_last_error().decode())
    return rc
