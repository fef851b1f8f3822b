"""ctypes wrapper around the CPU oracle (qmm_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by tests/, the smoke check and the
CPU-baseline leg of bench.py, never by the product package.  It shares no
code with the CUDA library.

Types follow the library numbering: 0 = Q8_0, 1 = Q4_K, 2 = Q6_K; 3 = Q5_K,
4 = Q3_K, 5 = Q2_K (the other K-quants, checked here ahead of their kernels).
"""
import ctypes
import os

import numpy as np

from . import build as _build

Q8_0, Q4_K, Q6_K, Q5_K, Q3_K, Q2_K = 0, 1, 2, 3, 4, 5
BLOCK_BYTES = {Q8_0: 34, Q4_K: 144, Q6_K: 210, Q5_K: 176, Q3_K: 110, Q2_K: 84}
BLOCK_WEIGHTS = {Q8_0: 32, Q4_K: 256, Q6_K: 256, Q5_K: 256, Q3_K: 256, Q2_K: 256}

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i64 = ctypes.c_int64
        L.oracle_half_to_float.restype = ctypes.c_float
        L.oracle_half_to_float.argtypes = [ctypes.c_uint16]
        L.oracle_unpack_q8_0.argtypes = [P, P, P]
        L.oracle_pack_q8_0.argtypes = [ctypes.c_uint16, P, P]
        L.oracle_unpack_q4_k.argtypes = [P, P, P, P, P, P]
        L.oracle_pack_q4_k.argtypes = [ctypes.c_uint16, ctypes.c_uint16, P, P, P, P]
        L.oracle_unpack_q5_k.argtypes = [P, P, P, P, P, P]
        L.oracle_pack_q5_k.argtypes = [ctypes.c_uint16, ctypes.c_uint16, P, P, P, P]
        L.oracle_unpack_q3_k.argtypes = [P, P, P, P]
        L.oracle_pack_q3_k.argtypes = [ctypes.c_uint16, P, P, P]
        L.oracle_unpack_q2_k.argtypes = [P, P, P, P, P, P]
        L.oracle_pack_q2_k.argtypes = [ctypes.c_uint16, ctypes.c_uint16, P, P, P, P]
        L.oracle_unpack_q6_k.argtypes = [P, P, P, P]
        L.oracle_pack_q6_k.argtypes = [ctypes.c_uint16, P, P, P]
        L.oracle_dequant.argtypes = [ctypes.c_int, P, i64, P]
        L.oracle_quantize_act.argtypes = [P, i64, i64, P, P, P]
        L.oracle_qmm.argtypes = [ctypes.c_int, P, i64, i64, P, i64, P, P, ctypes.c_int]
        L.oracle_max_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return int(lib().oracle_max_threads())


def half_to_float(bits: int) -> float:
    return float(lib().oracle_half_to_float(int(bits) & 0xFFFF))


# --- single-block pack / unpack --------------------------------------------

def unpack_q8_0(blk):
    blk = np.ascontiguousarray(blk, dtype=np.uint8)
    d = np.zeros(1, np.uint16)
    q = np.zeros(32, np.int8)
    lib().oracle_unpack_q8_0(_p(blk), _p(d), _p(q))
    return int(d[0]), q


def pack_q8_0(d_bits, q):
    q = np.ascontiguousarray(q, dtype=np.int8)
    out = np.zeros(34, np.uint8)
    lib().oracle_pack_q8_0(int(d_bits), _p(q), _p(out))
    return out


def unpack_q4_k(blk):
    blk = np.ascontiguousarray(blk, dtype=np.uint8)
    d = np.zeros(1, np.uint16)
    dm = np.zeros(1, np.uint16)
    sc = np.zeros(8, np.uint8)
    m = np.zeros(8, np.uint8)
    q = np.zeros(256, np.uint8)
    lib().oracle_unpack_q4_k(_p(blk), _p(d), _p(dm), _p(sc), _p(m), _p(q))
    return int(d[0]), int(dm[0]), sc, m, q


def pack_q4_k(d_bits, dmin_bits, sc, m, q):
    sc = np.ascontiguousarray(sc, dtype=np.uint8)
    m = np.ascontiguousarray(m, dtype=np.uint8)
    q = np.ascontiguousarray(q, dtype=np.uint8)
    out = np.zeros(144, np.uint8)
    lib().oracle_pack_q4_k(int(d_bits), int(dmin_bits), _p(sc), _p(m), _p(q), _p(out))
    return out


def unpack_q5_k(blk):
    blk = np.ascontiguousarray(blk, dtype=np.uint8)
    d = np.zeros(1, np.uint16)
    dm = np.zeros(1, np.uint16)
    sc = np.zeros(8, np.uint8)
    m = np.zeros(8, np.uint8)
    q = np.zeros(256, np.uint8)
    lib().oracle_unpack_q5_k(_p(blk), _p(d), _p(dm), _p(sc), _p(m), _p(q))
    return int(d[0]), int(dm[0]), sc, m, q


def pack_q5_k(d_bits, dmin_bits, sc, m, q):
    sc = np.ascontiguousarray(sc, dtype=np.uint8)
    m = np.ascontiguousarray(m, dtype=np.uint8)
    q = np.ascontiguousarray(q, dtype=np.uint8)
    out = np.zeros(176, np.uint8)
    lib().oracle_pack_q5_k(int(d_bits), int(dmin_bits), _p(sc), _p(m), _p(q), _p(out))
    return out


def unpack_q3_k(blk):
    """(d bits, signed scales sc - 32 [16], q in -4..3 [256])"""
    blk = np.ascontiguousarray(blk, dtype=np.uint8)
    d = np.zeros(1, np.uint16)
    sc = np.zeros(16, np.int8)
    q = np.zeros(256, np.int8)
    lib().oracle_unpack_q3_k(_p(blk), _p(d), _p(sc), _p(q))
    return int(d[0]), sc, q


def pack_q3_k(d_bits, sc, q):
    sc = np.ascontiguousarray(sc, dtype=np.int8)
    q = np.ascontiguousarray(q, dtype=np.int8)
    out = np.zeros(110, np.uint8)
    lib().oracle_pack_q3_k(int(d_bits), _p(sc), _p(q), _p(out))
    return out


def unpack_q2_k(blk):
    blk = np.ascontiguousarray(blk, dtype=np.uint8)
    d = np.zeros(1, np.uint16)
    dm = np.zeros(1, np.uint16)
    sc = np.zeros(16, np.uint8)
    m = np.zeros(16, np.uint8)
    q = np.zeros(256, np.uint8)
    lib().oracle_unpack_q2_k(_p(blk), _p(d), _p(dm), _p(sc), _p(m), _p(q))
    return int(d[0]), int(dm[0]), sc, m, q


def pack_q2_k(d_bits, dmin_bits, sc, m, q):
    sc = np.ascontiguousarray(sc, dtype=np.uint8)
    m = np.ascontiguousarray(m, dtype=np.uint8)
    q = np.ascontiguousarray(q, dtype=np.uint8)
    out = np.zeros(84, np.uint8)
    lib().oracle_pack_q2_k(int(d_bits), int(dmin_bits), _p(sc), _p(m), _p(q), _p(out))
    return out


def unpack_q6_k(blk):
    blk = np.ascontiguousarray(blk, dtype=np.uint8)
    d = np.zeros(1, np.uint16)
    sc = np.zeros(16, np.int8)
    q = np.zeros(256, np.uint8)
    lib().oracle_unpack_q6_k(_p(blk), _p(d), _p(sc), _p(q))
    return int(d[0]), sc, q


def pack_q6_k(d_bits, sc, q):
    sc = np.ascontiguousarray(sc, dtype=np.int8)
    q = np.ascontiguousarray(q, dtype=np.uint8)
    out = np.zeros(210, np.uint8)
    lib().oracle_pack_q6_k(int(d_bits), _p(sc), _p(q), _p(out))
    return out


# --- whole-tensor operations -----------------------------------------------

def dequant(qtype: int, blocks, n_elems: int) -> np.ndarray:
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(-1)
    out = np.empty(n_elems, np.float32)
    rc = lib().oracle_dequant(int(qtype), _p(blocks), int(n_elems), _p(out))
    if rc:
        raise ValueError(f"oracle_dequant failed: {rc}")
    return out


def quantize_act(x):
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim == 1:
        x = x[None]
    M, K = x.shape
    q = np.empty((M, K), np.int8)
    d = np.empty((M, K // 32), np.float32)
    s = np.empty((M, K // 32), np.int32)
    rc = lib().oracle_quantize_act(_p(x), M, K, _p(q), _p(d), _p(s))
    if rc:
        raise ValueError(f"oracle_quantize_act failed: {rc}")
    return q, d, s


def qmm(qtype: int, W, N: int, K: int, x, nthreads: int = 0):
    """Return (y, A): y[M,N] in f64 and the bound scale A = sum_k |w x^|."""
    W = np.ascontiguousarray(W, dtype=np.uint8).reshape(-1)
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim == 1:
        x = x[None]
    M = x.shape[0]
    assert x.shape[1] == K
    need = N * (K // BLOCK_WEIGHTS[qtype]) * BLOCK_BYTES[qtype]
    assert W.size >= need, (W.size, need)
    y = np.empty((M, N), np.float64)
    A = np.empty((M, N), np.float64)
    nt = nthreads if nthreads > 0 else max(1, os.cpu_count() or 1)
    rc = lib().oracle_qmm(int(qtype), _p(W), int(N), int(K), _p(x), int(M), _p(y), _p(A), int(nt))
    if rc:
        raise ValueError(f"oracle_qmm failed: {rc}")
    return y, A


def qmm_t(qtype: int, W, H: int, N: int, K: int, x):
    """Product with the transposed matrices: y[h, m, k] = sum_n x[h, m, n] *
    w[h, n, k] for H matrices of N rows of K weights, w the dequantised
    weights (exact fp32 values of d*q), x used as given (not quantised).

    Follows the value side of attention over a KV cache kept in q8_0 (infr
    landing page, "why > Paged experts, spillable KV": the KV cache can be
    stored as q8_0): each cached position is one row of head_dim weights and
    the output is the probability-weighted sum of the rows.  The definition
    written out: the dequantised rows times x in f64 (numpy's matmul as the
    only library step).  Returns (y, A) in f64, A = sum_n |x w| (the scale of
    the tolerance bound)."""
    W = np.ascontiguousarray(W, dtype=np.uint8).reshape(-1)
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.ndim == 3 and x.shape[0] == H and x.shape[2] == N, x.shape
    M = x.shape[1]
    nblk = N * (K // BLOCK_WEIGHTS[qtype])
    per = nblk * BLOCK_BYTES[qtype]
    assert W.size >= H * per, (W.size, H * per)
    y = np.zeros((H, M, K), np.float64)
    A = np.zeros((H, M, K), np.float64)
    for h in range(H):
        w = dequant(qtype, W[h * per:(h + 1) * per], N * K).reshape(N, K).astype(np.float64)
        xh = x[h].astype(np.float64)
        y[h] = xh @ w
        A[h] = np.abs(xh) @ np.abs(w)
    return y, A


def silu(v):
    """v * sigmoid(v) = v / (1 + exp(-v)), in f64 (overflow-safe for v << 0)."""
    v = np.asarray(v, dtype=np.float64)
    out = np.empty_like(v)
    pos = v >= 0
    out[pos] = v[pos] / (1.0 + np.exp(-v[pos]))
    e = np.exp(v[~pos])
    out[~pos] = v[~pos] * e / (1.0 + e)
    return out


def gate_up_silu(type_gate: int, W_gate, type_up: int, W_up, N: int, K: int, x):
    """The MLP's gated product of one decode step: h = silu(W_gate . x) * (W_up . x),
    the two products as qmm (quantised x) and the activation in f64.

    The pages' infr engine runs gate and up as one dispatch (infr landing page,
    "why > Per-op device profiling": the expert_gateup role); the activation
    between them is the SiLU of the Qwen3 / Llama MLPs those engines serve.
    Returns (h, B): B bounds |h_gpu - h| from the products' bound
    e = 2e-3 * A + 1e-5 through the slopes: |silu'| <= 1.1 everywhere, so
    B = 1.1 * |u| * e_g + |silu(g)| * e_u + e_g * e_u."""
    g, Ag = qmm(type_gate, W_gate, N, K, x)
    u, Au = qmm(type_up, W_up, N, K, x)
    eg, eu = 2e-3 * Ag + 1e-5, 2e-3 * Au + 1e-5
    sg = silu(g)
    h = sg * u
    B = 1.1 * np.abs(u) * eg + np.abs(sg) * eu + 1.1 * eg * eu
    return h, B

