"""Pins for the CPU oracle: checks against facts fixed outside the oracle
(IEEE binary16 via numpy, hand-worked blocks, closed forms, brute-force f64
dense products built from the fields), so a dropped term, a wrong sign or
index, or a transposed operand in the oracle fails one of them."""
import os

import numpy as np
import pytest

import oracle as O
import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _read_fixture(name):
    rows = {}
    ws = []
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "w":
                ws.append((int(vals[0]), vals[1], vals[2] if len(vals) > 2 else None))
            else:
                rows[key] = vals
    return rows, ws


# ---------------------------------------------------------------- binary16

def test_half_to_float_exhaustive():
    lib = O.lib()
    bits = np.arange(65536, dtype=np.uint32)
    want = bits.astype(np.uint16).view(np.float16).astype(np.float32)
    got = np.array([lib.oracle_half_to_float(int(b)) for b in bits], np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


# ---------------------------------------------------------- golden blocks

def test_golden_q4_k_block():
    rows, ws = _read_fixture("q4_k_block.txt")
    blk = np.frombuffer(bytes.fromhex(rows["header"][0] + rows["qs"][0]), np.uint8)
    assert blk.size == 144
    d, dm, sc, m, q = O.unpack_q4_k(blk)
    assert d == 0x3C00 and dm == 0x3800
    assert list(sc) == [int(v) for v in rows["sc"]]
    assert list(m) == [int(v) for v in rows["m"]]
    w = O.dequant(O.Q4_K, blk, 256)
    for p, qv, wv in ws:
        assert q[p] == int(qv), p
        assert w[p] == np.float32(float(wv)), (p, w[p], wv)


def test_golden_q6_k_block():
    rows, ws = _read_fixture("q6_k_block.txt")
    ql = bytes.fromhex(rows["ql"][0])
    qh = bytes([0xE4] * 64)
    blk = np.frombuffer(ql + qh + bytes.fromhex(rows["scales"][0]) + bytes.fromhex(rows["d"][0]), np.uint8)
    assert blk.size == 210
    d, sc, q = O.unpack_q6_k(blk)
    assert d == 0x3400
    assert list(sc) == list(range(-8, 8))
    w = O.dequant(O.Q6_K, blk, 256)
    for p, qv, wv in ws:
        assert q[p] == int(qv), p
        want = np.float32(float(wv))
        assert w[p] == want and np.signbit(w[p]) == np.signbit(want), (p, w[p], wv)


def test_golden_q8_0_block():
    rows, ws = _read_fixture("q8_0_block.txt")
    qv = np.array([int(v) for v in rows["q"]], np.int8)
    blk = np.frombuffer(bytes.fromhex(rows["d"][0]) + qv.tobytes(), np.uint8)
    d, q = O.unpack_q8_0(blk)
    assert d == 0x2E66 and np.array_equal(q, qv)
    w = O.dequant(O.Q8_0, blk, 32)
    for p, wv, _ in ws:
        assert w[p] == np.float32(float(wv)), (p, w[p], wv)


# ------------------------------------------------------------- round trips

def test_roundtrip_q8_0():
    rng = np.random.default_rng(1)
    for _ in range(50):
        db = int(rng.integers(0, 65536))
        q = rng.integers(-128, 128, 32).astype(np.int8)
        d2, q2 = O.unpack_q8_0(O.pack_q8_0(db, q))
        assert d2 == db and np.array_equal(q2, q)


def test_roundtrip_q4_k_all_scale_values():
    rng = np.random.default_rng(2)
    # every value 0..63 in every scale and min slot
    for v in range(64):
        sc = np.full(8, v, np.uint8)
        m = np.full(8, 63 - v, np.uint8)
        q = rng.integers(0, 16, 256).astype(np.uint8)
        d, dm, sc2, m2, q2 = O.unpack_q4_k(O.pack_q4_k(0x1234, 0xABCD, sc, m, q))
        assert (d, dm) == (0x1234, 0xABCD)
        assert np.array_equal(sc2, sc) and np.array_equal(m2, m) and np.array_equal(q2, q)
    for _ in range(100):
        sc = rng.integers(0, 64, 8).astype(np.uint8)
        m = rng.integers(0, 64, 8).astype(np.uint8)
        q = rng.integers(0, 16, 256).astype(np.uint8)
        _, _, sc2, m2, q2 = O.unpack_q4_k(O.pack_q4_k(0, 0, sc, m, q))
        assert np.array_equal(sc2, sc) and np.array_equal(m2, m) and np.array_equal(q2, q)


def test_roundtrip_q6_k():
    rng = np.random.default_rng(3)
    for _ in range(100):
        sc = rng.integers(-128, 128, 16).astype(np.int8)
        q = rng.integers(0, 64, 256).astype(np.uint8)
        db = int(rng.integers(0, 65536))
        d2, sc2, q2 = O.unpack_q6_k(O.pack_q6_k(db, sc, q))
        assert d2 == db and np.array_equal(sc2, sc) and np.array_equal(q2, q)
    for v in (0, 31, 32, 63):
        q = np.full(256, v, np.uint8)
        _, _, q2 = O.unpack_q6_k(O.pack_q6_k(0, np.zeros(16, np.int8), q))
        assert np.array_equal(q2, q)


def test_synth_bytes_unpack_to_uniform_fields():
    """The generator's uniform bytes give fields over their whole ranges."""
    blk = synth.weights(synth.Q4_K, 64, 256, seed=5).reshape(-1, 144)
    scs, ms, qs = [], [], []
    for b in blk:
        _, _, sc, m, q = O.unpack_q4_k(b)
        scs += list(sc); ms += list(m); qs += list(q)
    assert min(scs) == 0 and max(scs) == 63 and min(ms) == 0 and max(ms) == 63
    assert set(qs) == set(range(16))
    blk = synth.weights(synth.Q6_K, 64, 256, seed=6).reshape(-1, 210)
    allq, allsc = [], []
    for b in blk:
        _, sc, q = O.unpack_q6_k(b)
        allq += list(q); allsc += list(sc)
    assert set(allq) == set(range(64))
    assert min(allsc) == -32 and max(allsc) == 31


# -------------------------------------------------------- hand-worked cases

def test_q4_k_zero_quants_give_minus_dmin_m():
    sc = np.arange(8, dtype=np.uint8) * 7
    m = np.array([0, 1, 2, 3, 60, 61, 62, 63], np.uint8)
    blk = O.pack_q4_k(0x3C00, 0x2E66, sc, m, np.zeros(256, np.uint8))
    w = O.dequant(O.Q4_K, blk, 256)
    dmin = np.float32(np.uint16(0x2E66).view(np.float16))
    for j in range(8):
        want = np.float32(0.0) * np.float32(0) - dmin * np.float32(m[j])
        assert np.all(w[32 * j:32 * j + 32] == want)


def test_q4_k_unit_scale_is_identity():
    rng = np.random.default_rng(4)
    q = rng.integers(0, 16, 256).astype(np.uint8)
    blk = O.pack_q4_k(0x3C00, 0x0000, np.ones(8, np.uint8), np.zeros(8, np.uint8), q)
    assert np.array_equal(O.dequant(O.Q4_K, blk, 256), q.astype(np.float32))


def test_q6_k_q32_is_zero():
    sc = np.arange(-8, 8, dtype=np.int8)
    blk = O.pack_q6_k(0x3C00, sc, np.full(256, 32, np.uint8))
    assert np.all(O.dequant(O.Q6_K, blk, 256) == 0)
    x = synth.activations(2, 256, seed=9)
    y, A = O.qmm(O.Q6_K, blk, 1, 256, x)
    assert np.all(y == 0) and np.all(A == 0)


def test_q8_0_unit_scale_gives_exact_integer_dot():
    rng = np.random.default_rng(7)
    N, K, M = 5, 512, 3
    qw = rng.integers(-127, 128, (N, K)).astype(np.int8)
    W = np.concatenate([O.pack_q8_0(0x3C00, qw[n, 32 * b:32 * b + 32])
                        for n in range(N) for b in range(K // 32)])
    xi = rng.integers(-127, 128, (M, K)).astype(np.int64)
    xi[:, ::32] = 127  # amax = 127 in every block, so d = 1 and q = x exactly
    y, _ = O.qmm(O.Q8_0, W, N, K, xi.astype(np.float32))
    assert np.array_equal(y, (xi @ qw.astype(np.int64).T).astype(np.float64))


def test_subnormal_and_signed_zero_scales():
    q = np.arange(-16, 16, dtype=np.int8)
    w = O.dequant(O.Q8_0, O.pack_q8_0(0x0001, q), 32)   # 2^-24
    assert np.array_equal(w, q.astype(np.float32) * np.float32(2.0 ** -24))
    w = O.dequant(O.Q8_0, O.pack_q8_0(0x8000, q), 32)   # -0
    assert np.all(w == 0) and np.array_equal(np.signbit(w), q >= 0)   # -0 * 0 = -0


# ------------------------------------------------------------- quantiser

def test_quantizer_closed_forms():
    amax = np.float32(3.0)
    k = np.arange(-15, 17, dtype=np.int32)
    k[0] = 127
    d = np.float32(amax / np.float32(127.0))
    x = (k.astype(np.float32) * d).astype(np.float32)
    x[0] = amax
    q, dd, s = O.quantize_act(x)
    assert dd[0, 0] == d
    # x = k*d rounds back to k (the relative error of k*d*(1/d) is far below 0.5/k)
    assert np.array_equal(q[0].astype(np.int32), k)
    assert s[0, 0] == k.sum()


def test_quantizer_ties_round_away_from_zero():
    x = np.zeros(32, np.float32)
    x[0] = 127.0   # d = 1, inv = 1
    x[1:6] = [2.5, -2.5, 0.5, -0.5, 126.5]
    q, d, s = O.quantize_act(x)
    assert d[0, 0] == 1.0
    assert list(q[0, :6]) == [127, 3, -3, 1, -1, 127]
    assert s[0, 0] == 127 + 3 - 3 + 1 - 1 + 127


def test_quantizer_zero_block_and_bounds():
    x = synth.activations(4, 256, seed=11, outlier_frac=0.05)
    x[1, 32:64] = 0
    q, d, s = O.quantize_act(x)
    assert d[1, 1] == 0 and np.all(q[1, 32:64] == 0) and s[1, 1] == 0
    assert np.all(np.abs(q.astype(np.int32)) <= 127)
    blocks = np.abs(x).reshape(4, 8, 32)
    am = blocks.argmax(axis=2)
    qb = q.reshape(4, 8, 32)
    for r in range(4):
        for b in range(8):
            if d[r, b] != 0:
                assert abs(int(qb[r, b, am[r, b]])) == 127
    assert np.array_equal(s, q.reshape(4, 8, 32).astype(np.int32).sum(axis=2))


# ------------------------------------------- qmm against brute-force dense

def _q4_k_fields(rng, N, K):
    nb = K // 256
    f = dict(d=rng.integers(0x1000, 0x3C00, (N, nb)).astype(np.uint16),
             dm=rng.integers(0x1000, 0x3C00, (N, nb)).astype(np.uint16),
             sc=rng.integers(0, 64, (N, nb, 8)).astype(np.uint8),
             m=rng.integers(0, 64, (N, nb, 8)).astype(np.uint8),
             q=rng.integers(0, 16, (N, nb, 256)).astype(np.uint8))
    W = np.concatenate([O.pack_q4_k(f["d"][n, b], f["dm"][n, b], f["sc"][n, b], f["m"][n, b], f["q"][n, b])
                        for n in range(N) for b in range(nb)])
    d = f["d"].view(np.float16).astype(np.float64)
    dm = f["dm"].view(np.float16).astype(np.float64)
    Wd = (d[:, :, None] * np.repeat(f["sc"], 32, axis=2) * f["q"]
          - dm[:, :, None] * np.repeat(f["m"], 32, axis=2)).reshape(N, K)
    return W, Wd


def _q6_k_fields(rng, N, K):
    nb = K // 256
    dbits = rng.integers(0x1000, 0x3C00, (N, nb)).astype(np.uint16)
    sc = rng.integers(-128, 128, (N, nb, 16)).astype(np.int8)
    q = rng.integers(0, 64, (N, nb, 256)).astype(np.uint8)
    W = np.concatenate([O.pack_q6_k(dbits[n, b], sc[n, b], q[n, b]) for n in range(N) for b in range(nb)])
    d = dbits.view(np.float16).astype(np.float64)
    Wd = (d[:, :, None] * np.repeat(sc.astype(np.float64), 16, axis=2)
          * (q.astype(np.float64) - 32)).reshape(N, K)
    return W, Wd


def _q8_0_fields(rng, N, K):
    nb = K // 32
    dbits = rng.integers(0x1000, 0x3C00, (N, nb)).astype(np.uint16)
    q = rng.integers(-127, 128, (N, nb, 32)).astype(np.int8)
    W = np.concatenate([O.pack_q8_0(dbits[n, b], q[n, b]) for n in range(N) for b in range(nb)])
    Wd = (dbits.view(np.float16).astype(np.float64)[:, :, None] * q).reshape(N, K)
    return W, Wd


@pytest.mark.parametrize("qtype,make", [(O.Q4_K, _q4_k_fields), (O.Q6_K, _q6_k_fields),
                                        (O.Q8_0, _q8_0_fields)])
@pytest.mark.parametrize("K", [256, 512])
def test_qmm_matches_dense_f64(qtype, make, K):
    rng = np.random.default_rng(100 + qtype + K)
    N, M = 7, 3
    W, Wd = make(rng, N, K)
    # integer activations with amax 127 per block quantise exactly (d = 1)
    xi = rng.integers(-127, 128, (M, K)).astype(np.float64)
    xi[:, 5::32] = -127
    # a power-of-two scale per row keeps the quantisation exact: x = 2^e * int
    scale = np.array([1.0, 0.25, 8.0])[:, None]
    x = (xi * scale).astype(np.float32)
    y, A = O.qmm(qtype, W, N, K, x)
    yd = (xi * scale) @ Wd.T
    Ad = np.abs(xi * scale) @ np.abs(Wd).T
    np.testing.assert_allclose(y, yd, rtol=1e-12, atol=1e-12 * np.abs(yd).max())
    # A uses the fp32-rounded weights: agreement to fp32 rounding of w
    np.testing.assert_allclose(A, Ad, rtol=1e-6)
    assert np.all(np.abs(y) <= A * (1 + 1e-9))


def test_qmm_linear_in_weight_scale():
    rng = np.random.default_rng(12)
    N, K = 4, 256
    q = rng.integers(-127, 128, (N, K // 32, 32)).astype(np.int8)
    W1 = np.concatenate([O.pack_q8_0(0x2C00, q[n, b]) for n in range(N) for b in range(K // 32)])
    W2 = np.concatenate([O.pack_q8_0(0x3000, q[n, b]) for n in range(N) for b in range(K // 32)])
    x = synth.activations(2, K, seed=13)
    y1, _ = O.qmm(O.Q8_0, W1, N, K, x)
    y2, _ = O.qmm(O.Q8_0, W2, N, K, x)
    np.testing.assert_array_equal(2 * y1, y2)   # 0x3000 = 2 * 0x2C00 exactly


def test_q4_k_unit_scale_is_textbook_int_matmul():
    rng = np.random.default_rng(14)
    N, K, M = 3, 512, 2
    q = rng.integers(0, 16, (N, K // 256, 256)).astype(np.uint8)
    W = np.concatenate([O.pack_q4_k(0x3C00, 0x3C00, np.ones(8, np.uint8), np.zeros(8, np.uint8), q[n, b])
                        for n in range(N) for b in range(K // 256)])
    x = synth.activations(M, K, seed=15)
    xq, xd, _ = O.quantize_act(x)
    y, _ = O.qmm(O.Q4_K, W, N, K, x)
    qk = q.reshape(N, K).astype(np.int64)
    want = np.zeros((M, N))
    for b in range(K // 32):
        I = xq[:, 32 * b:32 * b + 32].astype(np.int64) @ qk[:, 32 * b:32 * b + 32].T
        want += xd[:, b:b + 1].astype(np.float64) * I
    np.testing.assert_allclose(y, want, rtol=1e-13)


def test_planted_mistake_is_caught():
    """A plausible oracle mistake (swapping the two Q4_K nibble halves) breaks
    the golden-block pin: the pins are sensitive to layout errors."""
    rows, ws = _read_fixture("q4_k_block.txt")
    blk = np.frombuffer(bytes.fromhex(rows["header"][0] + rows["qs"][0]), np.uint8).copy()
    qs = blk[16:]
    blk[16:] = ((qs & 15) << 4) | (qs >> 4)   # the mistake, applied to the input
    _, _, _, _, q = O.unpack_q4_k(blk)
    assert any(q[p] != int(qv) for p, qv, _ in ws)


# ------------------------------------------- qmm_t (the value side of attention)

def _q8_0_rows_from_bytes(blob, N, K):
    """Q8_0 rows decoded straight from the bytes, independently of the oracle's
    C code: fp16 d by numpy's binary16, int8 q by two's complement."""
    nb = K // 32
    w = np.zeros((N, K))
    for n in range(N):
        for b in range(nb):
            off = (n * nb + b) * 34
            d = float(np.frombuffer(bytes(blob[off:off + 2]), np.float16)[0])
            for i in range(32):
                q = int(blob[off + 2 + i])
                w[n, 32 * b + i] = d * (q - 256 if q >= 128 else q)
    return w


def test_qmm_t_matches_brute_force_sums():
    """y[h,m,k] = sum_n x[h,m,n] w[h,n,k] by explicit Python loops over the
    byte-decoded rows, on a case small enough to sum term by term."""
    H, N, K, M = 2, 5, 64, 3
    rng = np.random.default_rng(11)
    W = synth.weights(synth.Q8_0, H * N, K, seed=12)
    x = rng.standard_normal((H, M, N)).astype(np.float32)
    y, A = O.qmm_t(O.Q8_0, W, H, N, K, x)
    per = N * (K // 32) * 34
    for h in range(H):
        w = _q8_0_rows_from_bytes(W[h * per:(h + 1) * per], N, K)
        for m in range(M):
            for k in range(K):
                terms = [float(x[h, m, n]) * w[n, k] for n in range(N)]
                s, a = sum(terms), sum(abs(t) for t in terms)
                assert abs(y[h, m, k] - s) <= 1e-12 * max(1.0, a)
                assert abs(A[h, m, k] - a) <= 1e-12 * max(1.0, a)


def test_qmm_t_golden_block_row():
    """One cached position holding the hand-packed golden block: x = 2 gives
    twice the block's hand-worked weights (exact)."""
    rows, ws = _read_fixture("q8_0_block.txt")
    d = bytes.fromhex(rows["d"][0])
    q = bytes((int(v) & 255) for v in rows["q"])
    blk = np.frombuffer(d + q, np.uint8).copy()
    y, _ = O.qmm_t(O.Q8_0, blk, 1, 1, 32, np.full((1, 1, 1), 2.0, np.float32))
    for p, wv, _ in ws:
        assert y[0, 0, p] == 2.0 * float(wv)


def test_qmm_t_unit_rows_pick_rows_and_heads_are_independent():
    """x = e_n picks dequantised row n of its own matrix; permuting the
    matrices together with their x permutes y (no mixing across h)."""
    H, N, K = 3, 7, 96
    W = synth.weights(synth.Q8_0, H * N, K, seed=21)
    per = N * (K // 32) * 34
    x = np.zeros((H, N, N), np.float32)
    for h in range(H):
        x[h] = np.eye(N, dtype=np.float32)
    y, _ = O.qmm_t(O.Q8_0, W, H, N, K, x)
    for h in range(H):
        w = _q8_0_rows_from_bytes(W[h * per:(h + 1) * per], N, K)
        assert np.array_equal(y[h], w)
    perm = [2, 0, 1]
    Wp = np.concatenate([W[p * per:(p + 1) * per] for p in perm])
    rng = np.random.default_rng(5)
    xr = rng.standard_normal((H, 2, N)).astype(np.float32)
    y1, _ = O.qmm_t(O.Q8_0, W, H, N, K, xr)
    y2, _ = O.qmm_t(O.Q8_0, Wp, H, N, K, xr[perm])
    assert np.array_equal(y2, y1[perm])


def test_qmm_t_planted_transpose_is_caught():
    """A transposed operand (w^T in place of w, same shape when N == K) fails
    the brute-force pin: the pin tells the two orientations apart."""
    N = K = 32
    W = synth.weights(synth.Q8_0, N, K, seed=31)
    x = np.random.default_rng(3).standard_normal((1, 1, N)).astype(np.float32)
    w = _q8_0_rows_from_bytes(W, N, K)
    y, _ = O.qmm_t(O.Q8_0, W, 1, N, K, x)
    right = x[0].astype(np.float64) @ w
    wrong = x[0].astype(np.float64) @ w.T   # the mistake
    assert np.allclose(y[0], right, rtol=1e-12, atol=1e-12)
    assert not np.allclose(wrong, right, rtol=1e-6, atol=1e-6)


# ----------------------------------------------- Q5_K (the next K-quant)

def _pack_q5_k_from_layout(d_bits, dmin_bits, sc, m, q):
    """Q5_K bytes written straight from the layout in the golden file's
    header (independent of the oracle's packer)."""
    blk = np.zeros(176, np.uint8)
    blk[0:2] = np.array([d_bits], np.uint16).view(np.uint8)
    blk[2:4] = np.array([dmin_bits], np.uint16).view(np.uint8)
    S = blk[4:16]
    for j in range(4):
        S[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        S[j + 4] = (m[j] & 63) | ((m[j + 4] >> 4) << 6)
        S[j + 8] = (sc[j + 4] & 15) | ((m[j + 4] & 15) << 4)
    for p in range(256):
        j, l = p // 32, p % 32
        blk[16 + l] |= ((int(q[p]) >> 4) & 1) << j
        c, s = p // 64, (p // 32) % 2
        blk[48 + 32 * c + l] |= (int(q[p]) & 15) << (4 * s)
    return blk


def test_golden_q5_k_block():
    rows, ws = _read_fixture("q5_k_block.txt")
    d, dm = int(rows["d"][0], 16), int(rows["dmin"][0], 16)
    sc = np.array([int(v) for v in rows["sc"]], np.uint8)
    m = np.array([int(v) for v in rows["m"]], np.uint8)
    q = np.array([(5 * p + 3 + 7 * (p // 32)) % 32 for p in range(256)], np.uint8)
    blk = _pack_q5_k_from_layout(d, dm, sc, m, q)
    d2, dm2, sc2, m2, q2 = O.unpack_q5_k(blk)
    assert (d2, dm2) == (d, dm)
    assert np.array_equal(sc2, sc) and np.array_equal(m2, m) and np.array_equal(q2, q)
    w = O.dequant(O.Q5_K, blk, 256)
    for p, qv, wv in ws:
        assert q[p] == int(qv)
        assert w[p] == np.float32(float(wv)), (p, w[p], wv)
    # the oracle's packer writes the same bytes
    assert np.array_equal(O.pack_q5_k(d, dm, sc, m, q), blk)


def test_q5_k_without_fifth_bits_is_q4_k():
    """With qh all zero a Q5_K block is the Q4_K block of the same d, dmin,
    scales and nibbles (the pinned Q4_K oracle decides every weight)."""
    W4 = synth.weights(synth.Q4_K, 6, 512, seed=77)
    blocks4 = W4.reshape(-1, 144)
    blocks5 = np.concatenate([np.concatenate([b[:16], np.zeros(32, np.uint8), b[16:]]) for b in blocks4])
    n = blocks4.shape[0] * 256
    assert np.array_equal(O.dequant(O.Q5_K, blocks5, n).view(np.uint32),
                          O.dequant(O.Q4_K, W4, n).view(np.uint32))


def test_q5_k_fifth_bit_index_closed_form():
    """qh[l] = 1 << (l mod 8) sets the fifth bit of weight 32j + l exactly when
    l mod 8 == j: those weights gain 16*d*sc[j] over the Q4_K weight (d = 1,
    dmin = 0: every weight is a small integer, exact), the others are unchanged."""
    W4 = synth.weights(synth.Q4_K, 1, 256, seed=5).reshape(144).copy()
    W4[0:2] = np.array([0x3C00], np.uint16).view(np.uint8)   # d = 1
    W4[2:4] = 0                                               # dmin = 0
    qh = np.array([1 << (l % 8) for l in range(32)], np.uint8)
    blk5 = np.concatenate([W4[:16], qh, W4[16:]])
    w4 = O.dequant(O.Q4_K, W4, 256).astype(np.float64)
    w5 = O.dequant(O.Q5_K, blk5, 256).astype(np.float64)
    _, _, sc, _, _ = O.unpack_q4_k(W4)
    for p in range(256):
        j, l = p // 32, p % 32
        extra = 16.0 * sc[j] if l % 8 == j else 0.0
        assert w5[p] == w4[p] + extra, (p, w5[p], w4[p], extra)


def _q5_k_fields(rng, N, K):
    nb = K // 256
    f = dict(d=rng.integers(0x1000, 0x3C00, (N, nb)).astype(np.uint16),
             dm=rng.integers(0x1000, 0x3C00, (N, nb)).astype(np.uint16),
             sc=rng.integers(0, 64, (N, nb, 8)).astype(np.uint8),
             m=rng.integers(0, 64, (N, nb, 8)).astype(np.uint8),
             q=rng.integers(0, 32, (N, nb, 256)).astype(np.uint8))
    W = np.concatenate([_pack_q5_k_from_layout(f["d"][n, b], f["dm"][n, b], f["sc"][n, b], f["m"][n, b],
                                               f["q"][n, b]) for n in range(N) for b in range(nb)])
    d = f["d"].view(np.float16).astype(np.float64)
    dm = f["dm"].view(np.float16).astype(np.float64)
    Wd = (d[:, :, None] * np.repeat(f["sc"], 32, axis=2) * f["q"]
          - dm[:, :, None] * np.repeat(f["m"], 32, axis=2)).reshape(N, K)
    return W, Wd


@pytest.mark.parametrize("K", [256, 512])
def test_qmm_q5_k_matches_dense_f64(K):
    rng = np.random.default_rng(300 + K)
    N, M = 5, 3
    W, Wd = _q5_k_fields(rng, N, K)
    xi = rng.integers(-127, 128, (M, K)).astype(np.float64)
    xi[:, 7::32] = 127
    scale = np.array([1.0, 0.5, 4.0])[:, None]
    x = (xi * scale).astype(np.float32)
    y, A = O.qmm(O.Q5_K, W, N, K, x)
    yd = (xi * scale) @ Wd.T
    np.testing.assert_allclose(y, yd, rtol=1e-12, atol=1e-12 * np.abs(yd).max())
    assert np.all(np.abs(y) <= A * (1 + 1e-9))


def test_q5_k_planted_bit_index_mistake_is_caught():
    """Reading the fifth bit of sub-block j from bit j + 1 (a plausible slip)
    breaks the golden pin: applied to the input, the listed weights change."""
    rows, ws = _read_fixture("q5_k_block.txt")
    sc = np.array([int(v) for v in rows["sc"]], np.uint8)
    m = np.array([int(v) for v in rows["m"]], np.uint8)
    q = np.array([(5 * p + 3 + 7 * (p // 32)) % 32 for p in range(256)], np.uint8)
    blk = _pack_q5_k_from_layout(int(rows["d"][0], 16), int(rows["dmin"][0], 16), sc, m, q)
    blk[16:48] = (blk[16:48].astype(np.uint16) << 1).astype(np.uint8)   # the mistake
    w = O.dequant(O.Q5_K, blk, 256)
    assert any(w[p] != np.float32(float(wv)) for p, _, wv in ws)


# ---------------------------------------- Q3_K and Q2_K (16-weight sub-blocks)

def _w_rows(name):
    """The 'w' lines of a fixture with every column: position first, the
    expected weight last."""
    out = []
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            parts = line.split()
            if parts and parts[0] == "w":
                out.append((int(parts[1]), parts[2:-1], parts[-1]))
    return out


def _sub16(p):
    h, r = divmod(p, 128)
    j, l = divmod(r, 32)
    return 8 * h + 2 * j + (l >= 16)


def _pack_q2_k_from_layout(d_bits, dmin_bits, sc, m, q):
    blk = np.zeros(84, np.uint8)
    for i in range(16):
        blk[i] = (int(sc[i]) & 15) | ((int(m[i]) & 15) << 4)
    for p in range(256):
        h, r = divmod(p, 128)
        j, l = divmod(r, 32)
        blk[16 + 32 * h + l] |= (int(q[p]) & 3) << (2 * j)
    blk[80:82] = np.array([d_bits], np.uint16).view(np.uint8)
    blk[82:84] = np.array([dmin_bits], np.uint16).view(np.uint8)
    return blk


def _pack_q3_k_from_layout(d_bits, sc_signed, q):
    blk = np.zeros(110, np.uint8)
    S = blk[96:108]
    for i in range(16):
        v = (int(sc_signed[i]) + 32) & 63
        k, G = i % 4, i // 4
        lo, hi = v & 15, v >> 4
        if G == 0:
            S[k] |= lo
        elif G == 1:
            S[4 + k] |= lo
        elif G == 2:
            S[k] |= lo << 4
        else:
            S[4 + k] |= lo << 4
        S[8 + k] |= hi << (2 * G)
    for p in range(256):
        h, r = divmod(p, 128)
        j, l = divmod(r, 32)
        v = int(q[p])
        bit = 1 if v >= 0 else 0
        low = v if bit else v + 4
        blk[32 + 32 * h + l] |= low << (2 * j)
        blk[l] |= bit << (4 * h + j)
    blk[108:110] = np.array([d_bits], np.uint16).view(np.uint8)
    return blk


def test_golden_q2_k_block():
    rows, _ = _read_fixture("q2_k_block.txt")
    ws = [(p, cols[0], wv) for p, cols, wv in _w_rows("q2_k_block.txt")]
    d, dm = int(rows["d"][0], 16), int(rows["dmin"][0], 16)
    sc = np.array([(3 * i + 1) % 16 for i in range(16)], np.uint8)
    m = np.array([(5 * i + 2) % 16 for i in range(16)], np.uint8)
    q = np.array([(3 * p + 1 + 2 * (p // 128)) % 4 for p in range(256)], np.uint8)
    blk = _pack_q2_k_from_layout(d, dm, sc, m, q)
    d2, dm2, sc2, m2, q2 = O.unpack_q2_k(blk)
    assert (d2, dm2) == (d, dm) and np.array_equal(sc2, sc) and np.array_equal(m2, m) and np.array_equal(q2, q)
    w = O.dequant(O.Q2_K, blk, 256)
    for p, qv, wv in ws:
        assert q[p] == int(qv)
        assert w[p] == np.float32(float(wv)), (p, w[p], wv)
    assert np.array_equal(O.pack_q2_k(d, dm, sc, m, q), blk)


def test_golden_q3_k_block():
    rows, _ = _read_fixture("q3_k_block.txt")
    ws = [(p, cols[0], wv) for p, cols, wv in _w_rows("q3_k_block.txt")]
    d = int(rows["d"][0], 16)
    sc = np.array([(7 * i + 3) % 64 - 32 for i in range(16)], np.int8)
    q = np.array([(5 * p + 2 + 3 * (p // 128)) % 8 - 4 for p in range(256)], np.int8)
    blk = _pack_q3_k_from_layout(d, sc, q)
    d2, sc2, q2 = O.unpack_q3_k(blk)
    assert d2 == d and np.array_equal(sc2, sc) and np.array_equal(q2, q)
    w = O.dequant(O.Q3_K, blk, 256)
    for p, qv, wv in ws:
        assert q[p] == int(qv)
        assert w[p] == np.float32(float(wv)), (p, w[p], wv)
    assert np.array_equal(O.pack_q3_k(d, sc, q), blk)


def test_q3_k_high_bit_closed_forms():
    """All high bits set: q is the 2-bit low part (0..3); all clear: low - 4.
    With d = 1 and every scale 33 (sc - 32 = 1) the weights are those integers."""
    S = np.zeros(12, np.uint8)
    for i in range(16):       # every 6-bit scale = 33 = 0b100001
        k, G = i % 4, i // 4
        if G == 0:
            S[k] |= 1
        elif G == 1:
            S[4 + k] |= 1
        elif G == 2:
            S[k] |= 1 << 4
        else:
            S[4 + k] |= 1 << 4
        S[8 + k] |= 2 << (2 * G)
    rng = np.random.default_rng(17)
    qs = rng.integers(0, 256, 64).astype(np.uint8)
    low = np.array([(int(qs[32 * (p // 128) + p % 32]) >> (2 * ((p % 128) // 32))) & 3 for p in range(256)])
    for hm, want in ((0xFF, low), (0x00, low - 4)):
        blk = np.concatenate([np.full(32, hm, np.uint8), qs, S, np.array([0x3C00], np.uint16).view(np.uint8)])
        w = O.dequant(O.Q3_K, blk, 256)
        assert np.array_equal(w, want.astype(np.float32))


def test_q2_k_unit_scales_give_the_quants():
    """dmin = 0 and every scale 1: the weights are d times the 2-bit quants."""
    rng = np.random.default_rng(19)
    qs = rng.integers(0, 256, 64).astype(np.uint8)
    blk = np.concatenate([np.full(16, 0x01, np.uint8), qs, np.array([0x3C00, 0x0000], np.uint16).view(np.uint8)])
    want = np.array([(int(qs[32 * (p // 128) + p % 32]) >> (2 * ((p % 128) // 32))) & 3 for p in range(256)])
    assert np.array_equal(O.dequant(O.Q2_K, blk, 256), want.astype(np.float32))


def test_q3_k_planted_high_bit_mistake_is_caught():
    """Reading the high bit from bit j instead of 4h + j (a plausible slip)
    breaks the golden pin: applied to the input, the listed weights change."""
    rows, _ = _read_fixture("q3_k_block.txt")
    sc = np.array([(7 * i + 3) % 64 - 32 for i in range(16)], np.int8)
    q = np.array([(5 * p + 2 + 3 * (p // 128)) % 8 - 4 for p in range(256)], np.int8)
    blk = _pack_q3_k_from_layout(int(rows["d"][0], 16), sc, q)
    hm = blk[:32].copy()
    blk[:32] = (hm & 0x0F) | ((hm & 0x0F) << 4)   # the mistake: second half reads the first half's bits
    w = O.dequant(O.Q3_K, blk, 256)
    assert any(w[p] != np.float32(float(wv)) for p, _, wv in _w_rows("q3_k_block.txt"))


def _q2_k_fields(rng, N, K):
    nb = K // 256
    d = rng.integers(0x1000, 0x3C00, (N, nb)).astype(np.uint16)
    dm = rng.integers(0x1000, 0x3C00, (N, nb)).astype(np.uint16)
    sc = rng.integers(0, 16, (N, nb, 16)).astype(np.uint8)
    m = rng.integers(0, 16, (N, nb, 16)).astype(np.uint8)
    q = rng.integers(0, 4, (N, nb, 256)).astype(np.uint8)
    W = np.concatenate([_pack_q2_k_from_layout(d[n, b], dm[n, b], sc[n, b], m[n, b], q[n, b])
                        for n in range(N) for b in range(nb)])
    sub = np.array([_sub16(p) for p in range(256)])
    df, dmf = d.view(np.float16).astype(np.float64), dm.view(np.float16).astype(np.float64)
    Wd = (df[:, :, None] * sc[:, :, sub] * q - dmf[:, :, None] * m[:, :, sub]).reshape(N, K)
    return W, Wd


def _q3_k_fields(rng, N, K):
    nb = K // 256
    d = rng.integers(0x1000, 0x3C00, (N, nb)).astype(np.uint16)
    sc = rng.integers(-32, 32, (N, nb, 16)).astype(np.int8)
    q = rng.integers(-4, 4, (N, nb, 256)).astype(np.int8)
    W = np.concatenate([_pack_q3_k_from_layout(d[n, b], sc[n, b], q[n, b]) for n in range(N) for b in range(nb)])
    sub = np.array([_sub16(p) for p in range(256)])
    df = d.view(np.float16).astype(np.float64)
    Wd = (df[:, :, None] * sc[:, :, sub].astype(np.float64) * q).reshape(N, K)
    return W, Wd


@pytest.mark.parametrize("qtype,make", [(O.Q2_K, _q2_k_fields), (O.Q3_K, _q3_k_fields)])
@pytest.mark.parametrize("K", [256, 512])
def test_qmm_q2_k_q3_k_match_dense_f64(qtype, make, K):
    rng = np.random.default_rng(400 + 10 * qtype + K)
    N, M = 5, 3
    W, Wd = make(rng, N, K)
    xi = rng.integers(-127, 128, (M, K)).astype(np.float64)
    xi[:, 3::32] = -127
    scale = np.array([1.0, 0.125, 2.0])[:, None]
    x = (xi * scale).astype(np.float32)
    y, A = O.qmm(qtype, W, N, K, x)
    yd = (xi * scale) @ Wd.T
    np.testing.assert_allclose(y, yd, rtol=1e-12, atol=1e-12 * np.abs(yd).max())
    assert np.all(np.abs(y) <= A * (1 + 1e-9))


# ---------------------------------------------- the gate/up SiLU epilogue

def test_silu_closed_forms():
    """silu(0) = 0, silu(v) - silu(-v) = v (odd part is v/2), silu(v) -> v for
    large v and -> 0 for very negative v; the slope stays below 1.1."""
    v = np.array([0.0, 1.0, -1.0, 2.5, -40.0, 40.0, -1000.0])
    s = O.silu(v)
    assert s[0] == 0.0
    np.testing.assert_allclose(O.silu(v) - O.silu(-v), v, rtol=1e-15, atol=1e-300)
    assert abs(s[5] - 40.0) < 1e-15 * 40 + 40 * np.exp(-40) * 1.01
    assert s[6] == 0.0 or abs(s[6]) < 1e-300
    np.testing.assert_allclose(O.silu(np.array([1.0]))[0], 1.0 / (1.0 + np.exp(-1.0)), rtol=1e-15)
    grid = np.linspace(-20, 20, 400001)
    slope = np.diff(O.silu(grid)) / np.diff(grid)
    assert slope.max() < 1.1 and slope.min() > -0.1


def test_gate_up_silu_composes_the_pinned_products():
    """h is silu of the gate product times the up product, both as the pinned
    qmm oracle computes them; the bound is positive and covers a perturbation
    of either product by its own bound."""
    N, K, M = 9, 512, 3
    Wg = synth.weights(synth.Q4_K, N, K, seed=61)
    Wu = synth.weights(synth.Q6_K, N, K, seed=62)
    x = synth.activations(M, K, seed=63)
    h, B = O.gate_up_silu(O.Q4_K, Wg, O.Q6_K, Wu, N, K, x)
    g, Ag = O.qmm(O.Q4_K, Wg, N, K, x)
    u, Au = O.qmm(O.Q6_K, Wu, N, K, x)
    assert np.array_equal(h, O.silu(g) * u)
    assert np.all(B > 0)
    eg, eu = 2e-3 * Ag + 1e-5, 2e-3 * Au + 1e-5
    for sg_, su_ in ((1, 1), (1, -1), (-1, 1), (-1, -1)):
        hp = O.silu(g + sg_ * eg) * (u + su_ * eu)
        assert np.all(np.abs(hp - h) <= B * (1 + 1e-9))


def test_synth_new_generators():
    """The other K-quants' blocks have their sizes and unpack to in-range
    fields; the attention probabilities are non-negative rows summing to 1."""
    for qt, bb in ((synth.Q5_K, 176), (synth.Q3_K, 110), (synth.Q2_K, 84)):
        W = synth.weights(qt, 3, 512, seed=7)
        assert W.size == 3 * 2 * bb and synth.BLOCK_BYTES[qt] == bb
    _, _, _, _, q5 = O.unpack_q5_k(synth.weights(synth.Q5_K, 1, 256, seed=1))
    assert q5.max() <= 31 and q5.max() >= 16          # the fifth bits are drawn
    _, sc3, q3 = O.unpack_q3_k(synth.weights(synth.Q3_K, 1, 256, seed=1))
    assert q3.min() >= -4 and q3.max() <= 3 and sc3.min() >= -32 and sc3.max() <= 31
    p = synth.attention_probs(2, 3, 1000, seed=4)
    assert p.shape == (2, 3, 1000) and p.min() >= 0
    np.testing.assert_allclose(p.sum(axis=2), 1.0, rtol=1e-5)
    assert synth.kv_cache(2, 10, 128, seed=1).size == 2 * 10 * 4 * 34
