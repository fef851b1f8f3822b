"""Seeded synthetic inputs shared by the tests, the oracle checks and the bench.

This module draws random fields and writes them into their byte positions
inside each block; it holds none of the method's arithmetic (no dequantisation,
no activation quantisation, no dot products), so the CUDA library and the
oracle can both be fed from it without sharing any of the computation.

Field positions per block (the block layouts of the GGUF formats):
  Q8_0 (34 B) : [0,2) fp16 d | [2,34) int8 q[32]
  Q4_K (144 B): [0,2) fp16 d | [2,4) fp16 dmin | [4,16) 12 scale/min bytes
                | [16,144) 128 quant bytes (two 4-bit quants per byte)
  Q6_K (210 B): [0,128) ql (two 4-bit low parts per byte) | [128,192) qh
                (four 2-bit high parts per byte) | [192,208) int8 scales[16]
                | [208,210) fp16 d
  Q5_K (176 B): [0,2) fp16 d | [2,4) fp16 dmin | [4,16) 12 scale/min bytes
                | [16,48) fifth bits | [48,176) 128 nibble bytes
  Q3_K (110 B): [0,32) high bits | [32,96) 2-bit parts | [96,108) 12 bytes
                of sixteen 6-bit scales | [108,110) fp16 d
  Q2_K (84 B) : [0,16) 4-bit scale and min per 16 weights | [16,80) 2-bit
                quants | [80,82) fp16 d | [82,84) fp16 dmin

Drawing uniform random bytes for the packed fields gives uniform fields for
any bijective bit packing: the 12 Q4_K scale bytes carry exactly sixteen 6-bit
values (96 bits), each Q4_K quant byte two 4-bit values, and the Q6_K ql/qh
bytes together exactly 256 6-bit values.  So "6-bit scales/mins uniform
0..63", "quants uniform 0..15" and "6-bit quants uniform 0..63" hold without
this module knowing the bit order.

The model shapes (Llama-3.2-1B, Qwen3-14B, Mistral-7B projections) are the
workloads the GGUF engines on the blazr and infr pages serve; the weights are
synthetic stand-ins for the real GGUF files, which are not used.
"""
from __future__ import annotations

import numpy as np

Q8_0, Q4_K, Q6_K, Q5_K, Q3_K, Q2_K = 0, 1, 2, 3, 4, 5
TYPE_NAMES = {Q8_0: "Q8_0", Q4_K: "Q4_K", Q6_K: "Q6_K", Q5_K: "Q5_K", Q3_K: "Q3_K", Q2_K: "Q2_K"}
BLOCK_BYTES = {Q8_0: 34, Q4_K: 144, Q6_K: 210, Q5_K: 176, Q3_K: 110, Q2_K: 84}
BLOCK_WEIGHTS = {Q8_0: 32, Q4_K: 256, Q6_K: 256, Q5_K: 256, Q3_K: 256, Q2_K: 256}


def row_bytes(qtype: int, K: int) -> int:
    return (K // BLOCK_WEIGHTS[qtype]) * BLOCK_BYTES[qtype]


def matrix_bytes(qtype: int, N: int, K: int) -> int:
    return N * row_bytes(qtype, K)


def _f16_bits(v: np.ndarray) -> np.ndarray:
    return np.asarray(v, dtype=np.float32).astype(np.float16).view(np.uint16)


def _halfnormal_f16(rng, n, sigma):
    return _f16_bits(np.abs(rng.normal(0.0, sigma, size=n)))


def q8_0_blocks(rng, nblocks: int) -> np.ndarray:
    """d fp16 log-uniform in [1e-3, 1e-2]; q int8 uniform in [-127, 127]."""
    out = np.empty((nblocks, 34), np.uint8)
    d = np.exp(rng.uniform(np.log(1e-3), np.log(1e-2), size=nblocks))
    out[:, 0:2] = _f16_bits(d).view(np.uint8).reshape(nblocks, 2)
    out[:, 2:34] = rng.integers(-127, 128, size=(nblocks, 32), dtype=np.int8).view(np.uint8)
    return out.reshape(-1)


def q4_k_blocks(rng, nblocks: int, sigma: float = 1e-3) -> np.ndarray:
    """d, dmin fp16 = |N(0, sigma)|; scales/mins and quants uniform."""
    out = np.empty((nblocks, 144), np.uint8)
    out[:, 0:2] = _halfnormal_f16(rng, nblocks, sigma).view(np.uint8).reshape(nblocks, 2)
    out[:, 2:4] = _halfnormal_f16(rng, nblocks, sigma).view(np.uint8).reshape(nblocks, 2)
    out[:, 4:144] = rng.integers(0, 256, size=(nblocks, 140), dtype=np.uint8)
    return out.reshape(-1)


def q6_k_blocks(rng, nblocks: int, sigma: float = 5e-4) -> np.ndarray:
    """6-bit quants uniform; int8 scales uniform in [-32, 31]; d = |N(0, sigma)|."""
    out = np.empty((nblocks, 210), np.uint8)
    out[:, 0:192] = rng.integers(0, 256, size=(nblocks, 192), dtype=np.uint8)
    out[:, 192:208] = rng.integers(-32, 32, size=(nblocks, 16), dtype=np.int8).view(np.uint8)
    out[:, 208:210] = _halfnormal_f16(rng, nblocks, sigma).view(np.uint8).reshape(nblocks, 2)
    return out.reshape(-1)


def q5_k_blocks(rng, nblocks: int, sigma: float = 1e-3) -> np.ndarray:
    """d, dmin fp16 = |N(0, sigma)|; scales/mins, fifth bits and nibbles uniform."""
    out = np.empty((nblocks, 176), np.uint8)
    out[:, 0:2] = _halfnormal_f16(rng, nblocks, sigma).view(np.uint8).reshape(nblocks, 2)
    out[:, 2:4] = _halfnormal_f16(rng, nblocks, sigma).view(np.uint8).reshape(nblocks, 2)
    out[:, 4:176] = rng.integers(0, 256, size=(nblocks, 172), dtype=np.uint8)
    return out.reshape(-1)


def q3_k_blocks(rng, nblocks: int, sigma: float = 1e-3) -> np.ndarray:
    """High bits, 2-bit parts and 6-bit scales uniform; d = |N(0, sigma)|."""
    out = np.empty((nblocks, 110), np.uint8)
    out[:, 0:108] = rng.integers(0, 256, size=(nblocks, 108), dtype=np.uint8)
    out[:, 108:110] = _halfnormal_f16(rng, nblocks, sigma).view(np.uint8).reshape(nblocks, 2)
    return out.reshape(-1)


def q2_k_blocks(rng, nblocks: int, sigma: float = 1e-3) -> np.ndarray:
    """4-bit scales/mins and 2-bit quants uniform; d, dmin = |N(0, sigma)|."""
    out = np.empty((nblocks, 84), np.uint8)
    out[:, 0:80] = rng.integers(0, 256, size=(nblocks, 80), dtype=np.uint8)
    out[:, 80:82] = _halfnormal_f16(rng, nblocks, sigma).view(np.uint8).reshape(nblocks, 2)
    out[:, 82:84] = _halfnormal_f16(rng, nblocks, sigma).view(np.uint8).reshape(nblocks, 2)
    return out.reshape(-1)


def weights(qtype: int, N: int, K: int, seed: int) -> np.ndarray:
    """Packed weight rows for an N x K matrix (row-major by output row)."""
    rng = np.random.default_rng(seed)
    nblk = N * (K // BLOCK_WEIGHTS[qtype])
    if qtype == Q8_0:
        return q8_0_blocks(rng, nblk)
    if qtype == Q4_K:
        return q4_k_blocks(rng, nblk)
    if qtype == Q6_K:
        return q6_k_blocks(rng, nblk)
    if qtype == Q5_K:
        return q5_k_blocks(rng, nblk)
    if qtype == Q3_K:
        return q3_k_blocks(rng, nblk)
    if qtype == Q2_K:
        return q2_k_blocks(rng, nblk)
    raise ValueError(qtype)


# Byte offsets of the fp16 scale fields inside each block: d, and dmin where
# the format has one (Q5_K's fields sit where Q4_K's do).
D_FIELD = {Q8_0: 0, Q4_K: 0, Q6_K: 208, Q5_K: 0, Q3_K: 108, Q2_K: 80}
DMIN_FIELD = {Q4_K: 2, Q5_K: 2, Q2_K: 82}


def with_scale_fields(qtype: int, W: np.ndarray, d_bits, dmin_bits=None) -> np.ndarray:
    """A copy of the packed blocks W with every block's fp16 d (and dmin, for
    the formats that have one) replaced by the given bit patterns: a scalar
    or one value per block."""
    bb = BLOCK_BYTES[qtype]
    out = np.array(W, dtype=np.uint8).reshape(-1, bb).copy()
    n = out.shape[0]
    pos = D_FIELD[qtype]
    out[:, pos:pos + 2] = np.broadcast_to(np.asarray(d_bits, np.uint16), (n,)).astype("<u2").view(
        np.uint8).reshape(n, 2)
    if dmin_bits is not None and qtype in DMIN_FIELD:
        pos = DMIN_FIELD[qtype]
        out[:, pos:pos + 2] = np.broadcast_to(np.asarray(dmin_bits, np.uint16), (n,)).astype("<u2").view(
            np.uint8).reshape(n, 2)
    return out.reshape(-1)


def loguniform_f16_bits(rng, n: int, lo: float, hi: float) -> np.ndarray:
    """n fp16 bit patterns of values log-uniform in [lo, hi] (rounded to fp16)."""
    return _f16_bits(np.exp(rng.uniform(np.log(lo), np.log(hi), size=n)))


def activations(M: int, K: int, seed: int, outlier_frac: float = 0.0,
                outlier_scale: float = 20.0) -> np.ndarray:
    """x f32 ~ N(0, 1); with outlier_frac > 0, a Bernoulli mask scales entries."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K)).astype(np.float32)
    if outlier_frac > 0:
        mask = rng.random((M, K)) < outlier_frac
        x[mask] *= np.float32(outlier_scale)
    return x


# --- the five workloads -----------------------------------------------------
# Each matrix: (name, qtype, K, N).  Seeds: weights 1000*cfg + index,
# activations 1000*cfg + 500 (+ M for the multi-slot decode cases).

LLAMA_1B = [("q", Q4_K, 2048, 2048), ("kv", Q4_K, 2048, 512),
            ("gate_up", Q4_K, 2048, 8192), ("down", Q4_K, 8192, 2048)]
QWEN3_14B_LAYER = [("q", Q4_K, 5120, 5120), ("k", Q4_K, 5120, 1024),
                   ("v", Q6_K, 5120, 1024), ("o", Q4_K, 5120, 5120),
                   ("gate", Q4_K, 5120, 17408), ("up", Q4_K, 5120, 17408),
                   ("down", Q6_K, 17408, 5120)]
LM_HEAD = [("lm_head", Q6_K, 2048, 128256)]
MISTRAL_MLP = [("up", Q4_K, 4096, 14336), ("down", Q4_K, 14336, 4096)]
Q8_SMALL = [("small", Q8_0, 512, 256)]

CONFIGS = {
    0: dict(name="Q8_0 GEMV K=512 N=256", mats=Q8_SMALL, M=[1], outliers=0.0),
    1: dict(name="Q4_K decode GEMV, Llama-3.2-1B projections", mats=LLAMA_1B, M=[1], outliers=0.0),
    2: dict(name="Q6_K lm_head GEMV K=2048 N=128256", mats=LM_HEAD, M=[1], outliers=0.0),
    3: dict(name="Q4_K_M Qwen3-14B layer decode", mats=QWEN3_14B_LAYER, M=[1, 2, 4, 8], outliers=0.0),
    4: dict(name="Q4_K prefill GEMM M=512, Mistral-7B MLP", mats=MISTRAL_MLP, M=[512], outliers=0.01),
}


def config_weights(cfg: int, index: int) -> np.ndarray:
    _, qtype, K, N = CONFIGS[cfg]["mats"][index]
    if cfg == 0:
        return weights(qtype, N, K, seed=0)
    return weights(qtype, N, K, seed=1000 * cfg + index)


def config_activations(cfg: int, M: int, K: int) -> np.ndarray:
    c = CONFIGS[cfg]
    if cfg == 0:
        return activations(M, K, seed=0)
    return activations(M, K, seed=1000 * cfg + 500 + M + K, outlier_frac=c["outliers"])


# --- the value side of attention over a q8_0 KV cache -------------------------
# Qwen3-14B-shaped attention: 8 KV heads of head_dim 128 shared by 40 query
# heads (5 per KV head), 32768 cached positions; the cache rows are Q8_0
# blocks with the Q8_0 value distribution above.

KV_CACHE = dict(name="Qwen3-14B-shaped q8_0 value cache", H=8, N=32768, K=128, M=5)


def kv_cache(H: int, N: int, K: int, seed: int) -> np.ndarray:
    """H matrices of N cached rows of K Q8_0 weights, matrix after matrix."""
    return weights(Q8_0, H * N, K, seed)


def attention_probs(H: int, M: int, N: int, seed: int, temperature: float = 3.0) -> np.ndarray:
    """Probability rows x[h, m, :] (non-negative, each summing to 1): the
    normalised exponentials of N(0, temperature^2) logits, so that a few
    positions carry most of the weight, as after a softmax over scores."""
    rng = np.random.default_rng(seed)
    z = rng.standard_normal((H, M, N)) * temperature
    z -= z.max(axis=2, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=2, keepdims=True)
    return p.astype(np.float32)
