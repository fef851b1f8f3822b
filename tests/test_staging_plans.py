"""CPU models of the address arithmetic of two staging paths, checked before
any GPU run (no GPU needed):

* the value-cache product (qmm_t.cu): the chunks of all CTAs and the row
  ranges of their warps cover every matrix exactly once; every bulk
  copy starts 16-byte aligned, has a 16-byte multiple size, stays inside the
  cache and its shared-memory slot; the bytes a lane reads (quant words,
  scales) lie inside what its stage copied; the warps' pair sums fit in the
  rings after the stream; shared memory stays within the per-block limit;
* the tcgen05 prefill's staging of the super-step types (gemm_tc.cu): by
  TMA for Q8_0, and for Q6_K, Q3_K and Q2_K when two rows are a 16-byte
  multiple and N is even (the boxes' coordinates meet the 16-byte rule, each
  row's super-block lies in its box row, the TMEM lane -> weight row map is a
  permutation whose warps read one box each); otherwise each dequantiser warp's
  16-byte chunk loads stay inside the matrix unless the kernel's "careful"
  test selects the word-by-word path, which it does exactly when a chunk
  would cross the matrix end; the read-back words of a super-block lie inside
  its staged bytes; the shared-memory plans fit.

The constants mirror the kernels (16 warps for K <= 160 else 8, ~192 KB of
rings, stages of 64 / 32 / 16 rows; 14 / 17 chunks per super-step, 60 /
68-word rows)."""
import pytest

SMEM_MAX = 232448
SMS = 152

# --------------------------------------------------------------- qmm_t


def vt_warps(nb):
    return 16 if nb <= 5 else 8


def vt_cfg(nb):
    K, RB = 32 * nb, 34 * nb
    WARPS = vt_warps(nb)
    SR = 64 if nb == 1 else 32 if nb <= 4 else 16
    SLOT = (SR * RB + 32 + 15) & ~15
    D = min(8, (192 * 1024) // (WARPS * SLOT))
    FR = 16 * K
    SMEM = WARPS * D * SLOT + 8 * WARPS * D + 16
    return dict(K=K, RB=RB, SR=SR, SLOT=SLOT, D=D, FR=FR, SMEM=SMEM, WARPS=WARPS)


def vt_chunk_rows(H, N, K, num_sms=SMS):
    w = vt_warps(K // 32)
    per = max(1, num_sms // H)
    R = -(-N // per)
    R = -(-R // w) * w
    return max(R, w)


@pytest.mark.parametrize("nb", range(1, 9))
def test_qmm_t_shared_memory_plan(nb):
    C = vt_cfg(nb)
    assert C["D"] >= 2
    assert C["SMEM"] <= SMEM_MAX
    assert C["SLOT"] % 16 == 0 and C["SR"] % 16 == 0 and C["SR"] >= 16
    # a stage's copy is at least 2 KB (smaller copies are copy-rate bound)
    assert C["SR"] * C["RB"] >= 2048
    # after the stream the rings hold the pair sums [warp % (W/2)][16 K]
    assert (C["WARPS"] // 2) * C["FR"] * 4 <= C["WARPS"] * C["D"] * C["SLOT"]
    # a lane's 16 NB accumulators and the rest fit 65536 / (32 W) registers
    assert 16 * nb <= 65536 // (32 * C["WARPS"]) - 48


@pytest.mark.parametrize("H,N,K", [(1, 1, 32), (1, 15, 64), (2, 300, 128), (8, 4096, 128), (8, 32768, 128),
                                   (3, 1000, 96), (1, 777, 256), (5, 64, 32), (6, 12345, 128), (4, 2049, 160),
                                   (1, 5000, 224), (16, 333, 128), (8, 131072, 128), (1, 129, 256)])
def test_qmm_t_chunks_and_copies(H, N, K):
    nb = K // 32
    C = vt_cfg(nb)
    RB, SR, SLOT = C["RB"], C["SR"], C["SLOT"]
    R = vt_chunk_rows(H, N, K)
    assert R % C["WARPS"] == 0
    nchunk = -(-N // R)
    assert H * nchunk <= max(SMS, H)  # one wave of CTAs (one per SM)
    assert nchunk < 2 ** 31 and H <= 65535
    base = 1 << 20  # W is 16-byte aligned
    w_end = base + H * N * RB
    CPG = 4 * nb
    contig = nb in (1, 2, 4, 8)
    for h in range(H):
        seen = []
        mat0 = base + h * N * RB
        for c in range(nchunk):
            n_lo, n_hi = c * R, min(N, c * R + R)
            W = C["WARPS"]
            rw = R // W
            for w in range(W):
                w_lo = min(n_hi, n_lo + w * rw)
                w_hi = min(n_hi, w_lo + rw)
                if w_lo < w_hi:
                    seen.append((w_lo, w_hi))
                # the L2 warm-up before the dependency wait: at most 16 KB of
                # the warp's own rows, 16-byte aligned, inside the cache
                p16 = (mat0 + w_lo * RB) & ~15
                q16 = min((mat0 + w_hi * RB) & ~15, p16 + 16384)
                if q16 > p16:
                    assert p16 >= base and q16 <= w_end and (q16 - p16) % 16 == 0
                    assert q16 <= ((mat0 + w_hi * RB) + 15) & ~15
                nst = -(-(w_hi - w_lo) // SR)
                for t in range(nst):
                    r0, r1 = w_lo + t * SR, min(w_hi, w_lo + t * SR + SR)
                    a, b = mat0 + r0 * RB, mat0 + r1 * RB
                    a16, b16 = a & ~15, (b + 15) & ~15
                    if b16 > w_end:
                        b16 = b & ~15  # the final bytes by plain loads
                    assert a16 >= base and b16 <= w_end and a16 % 16 == 0 and (b16 - a16) % 16 == 0
                    assert b - a16 <= SLOT  # copied bytes plus plain tail fit the slot
                    # reads of the stage's rows: offset from the slot start
                    off0 = a - a16
                    for r in range(r1 - r0):
                        row = off0 + r * RB
                        if contig:
                            bb = (CPG * 7) // 32  # the lane group with the largest offset
                            q = row + 34 * bb + 2 + (CPG * 7) % 32
                            last = (q & ~3) + 4 * (CPG // 4) + 4  # aligned words read
                        else:
                            q = row + 34 * (nb - 1) + 2 + 4 * 7
                            last = (q & ~3) + 8
                        assert last <= SLOT
                        assert row + RB <= b - a16  # the row itself was copied
        seen.sort()
        pos = 0
        for lo, hi in seen:
            assert lo == pos
            pos = hi
        assert pos == N


def test_qmm_t_counters_and_parts():
    for H, N, K in [(8, 32768, 128), (1, 1, 32), (65535, 16, 32)]:
        R = vt_chunk_rows(H, N, K)
        nchunk = -(-N // R)
        part = H * nchunk * 16 * K * 4
        assert part > 0 and nchunk >= 1


# --------------------------------------------- tcgen05 prefill staging

QMM_Q8_0, QMM_Q4_K, QMM_Q6_K, QMM_Q3_K, QMM_Q2_K = 0, 1, 2, 4, 5
SSB = {QMM_Q6_K: 210, QMM_Q8_0: 272, QMM_Q3_K: 110, QMM_Q2_K: 84}
CHUNKS = {QMM_Q6_K: 14, QMM_Q8_0: 17, QMM_Q3_K: 8, QMM_Q2_K: 6}
PITCH_W = {QMM_Q6_K: 60, QMM_Q8_0: 68, QMM_Q3_K: 36, QMM_Q2_K: 28}
BLOCK_BYTES_TC = {QMM_Q6_K: 210, QMM_Q3_K: 110, QMM_Q2_K: 84}


def tc_smem(BT, T):
    XBOX = BT * 128
    X_BYTES = 2 * XBOX
    RAW_Q = 32 * PITCH_W[T] * 4
    X_FIT = (232448 - 1536 - 4 * RAW_Q) // X_BYTES
    X = min(8, X_FIT)
    OFF_R = X * X_BYTES
    OFF_BAR = OFF_R + 4 * RAW_Q
    return dict(X=X, SMEM=OFF_BAR + 512 + 1024, RAW_Q=RAW_Q)


@pytest.mark.parametrize("T", [QMM_Q6_K, QMM_Q3_K, QMM_Q2_K])
@pytest.mark.parametrize("BT", [64, 128, 256])
def test_tc_own_shared_memory_plan(T, BT):
    P = tc_smem(BT, T)
    assert P["X"] >= 2
    assert P["SMEM"] <= SMEM_MAX
    assert 16 * (P["X"] + 4) + 8 + 64 <= 480  # barrier area
    # the quarter's buffer: 32 rows of CH chunks at a pitch of PW words
    assert CHUNKS[T] * 16 <= PITCH_W[T] * 4
    # odd number of 16-byte chunks per row: conflict-free chunk reads
    assert (PITCH_W[T] * 4 // 16) % 2 == 1


def tc_uses_tma(T, N, K):
    """The dispatch of gemm_tc.cu: raw stages by TMA for Q8_0, and for Q6_K,
    Q3_K and Q2_K when two rows are a 16-byte multiple and N is even."""
    return T == QMM_Q8_0 or ((2 * (K // 256) * BLOCK_BYTES_TC[T]) % 16 == 0 and N % 2 == 0)


@pytest.mark.parametrize("T,N,K", [(QMM_Q6_K, 301, 768), (QMM_Q6_K, 1001, 2048), (QMM_Q6_K, 130, 5376),
                                   (QMM_Q6_K, 77, 256), (QMM_Q6_K, 5121, 17408), (QMM_Q6_K, 3, 4352),
                                   (QMM_Q3_K, 301, 768), (QMM_Q3_K, 77, 256), (QMM_Q3_K, 131, 5120),
                                   (QMM_Q3_K, 3, 4352), (QMM_Q3_K, 130, 1536), (QMM_Q2_K, 301, 768),
                                   (QMM_Q2_K, 77, 256), (QMM_Q2_K, 1000, 768), (QMM_Q2_K, 3, 4352)])
def test_tc_own_chunk_loads(T, N, K):
    """Every 16-byte chunk load of the staging (two warps per quarter, half the
    chunks each) stays inside [W, w_end) unless the careful path is taken, and
    the careful path is taken exactly for the matrix's final super-block
    reaching past the end."""
    assert not tc_uses_tma(T, N, K)
    ssb, CH = SSB[T], CHUNKS[T]
    RB = (K // 32) * 34 if T == QMM_Q8_0 else (K // 256) * BLOCK_BYTES_TC[T]
    odd = T in (QMM_Q6_K, QMM_Q3_K, QMM_Q2_K)  # super-steps not 16-byte multiples
    W = 1 << 24
    w_end = W + N * RB
    nss = K // 256
    HALF = 32 * CH // 2
    NT = -(-HALF // 32)
    careful_seen = 0
    for n0 in range(0, -(-N // 128) * 128, 128):
        for quarter in range(4):
            nrows = min(32, N - (n0 + 32 * quarter))
            rows0 = W + (n0 + 32 * quarter) * RB
            for js in range(nss):
                seg0 = rows0 + js * ssb
                careful = odd and nrows > 0 and \
                    ((seg0 + (nrows - 1) * RB) & ~15) + 16 * CH > w_end
                need = False
                for cp in range(2):
                    for lane in range(32):
                        for t in range(NT):
                            i = lane + 32 * t
                            if i >= HALF:
                                continue
                            g = HALF * cp + i
                            r, c = g // CH, g % CH
                            if r >= nrows:
                                continue
                            a = ((seg0 + r * RB) & ~15) + 16 * c
                            assert a >= W and a % 16 == 0
                            if a + 16 > w_end:
                                need = True
                                assert careful, (n0, quarter, js, r, c)
                            # the super-block's bytes lie inside the row's 14 / 17 chunks
                            seg = seg0 + r * RB
                            assert seg + ssb <= ((seg0 + r * RB) & ~15) + 16 * CH
                            if T == QMM_Q6_K:
                                dl = seg & 15
                                assert dl % 2 == 0
                                # read-back: ql 5 chunks from 4h, qh 3 from 8 + 2h, scale words
                                for h in range(2):
                                    assert 4 * h + 5 <= CH and 8 + 2 * h + 3 <= CH
                                    # the scale word: two aligned words from (dl + 192 + 8h + 4cp) & ~3
                                    assert ((dl + 192 + 8 * h + 4) & ~3) + 8 <= 16 * CH
                                    assert dl + 208 + 2 <= 16 * CH  # d
                                    # realign reads the aligned words (dl >> 2) .. (dl >> 2) + NOUT of
                                    # the loaded chunks: the last byte it touches must lie in them
                                    assert (dl & ~3) + 4 * 16 + 3 < 16 * 5   # ql: 16 words from 5 chunks
                                    assert (dl & ~3) + 4 * 8 + 3 < 16 * 3    # qh: 8 words from 3 chunks
                            elif T == QMM_Q3_K:
                                dl = seg & 15
                                assert dl % 2 == 0
                                for h in range(2):
                                    # mask words from chunks 0..2, 2-bit words from 2 + 2h .. 4 + 2h
                                    assert 4 + 2 * h < CH and (dl & ~3) + 4 * 8 + 3 < 16 * 3
                                # scale words at dl + 96 .. dl + 104 and d at dl + 108, two
                                # aligned words each
                                assert ((dl + 108) & ~3) + 8 <= 16 * CH and ((dl + 104) & ~3) + 8 <= 16 * CH
                            elif T == QMM_Q2_K:
                                dl = seg & 15
                                assert dl % 4 == 0
                                for h in range(2):
                                    assert 3 + 2 * h < CH  # 2-bit words from chunks 1 + 2h .. 3 + 2h
                                    assert dl + 8 * h + 4 + 4 <= 16 * CH  # the scale word
                                assert dl + 80 + 4 <= 16 * CH  # d | dmin
                            else:
                                assert seg % 16 == 0
                if careful:
                    careful_seen += 1
                    assert need or odd
    if odd and (N * RB) % 16:
        assert careful_seen >= 1


# Q6_K / Q8_0 raw stages by TMA: Q6_K two boxes of 64 double rows x 240
# bytes (even rows, odd rows), Q8_0 one box of 128 rows x 272 bytes
TM_ROW = {QMM_Q6_K: 240, QMM_Q3_K: 144, QMM_Q2_K: 112, QMM_Q8_0: 272}
TM_TX = {QMM_Q6_K: 2 * 64 * 240, QMM_Q3_K: 2 * 64 * 144, QMM_Q2_K: 2 * 64 * 112, QMM_Q8_0: 128 * 272}


def tc_tm_smem(BT, T):
    X_BYTES = 2 * BT * 128
    R_BYTES = -(-TM_TX[T] // 1024) * 1024
    X = min(8, (232448 - 1536 - 2 * R_BYTES) // X_BYTES)
    OFF_R = X * X_BYTES
    R = min(8, (232448 - 1536 - OFF_R) // R_BYTES)
    return dict(X=X, R=R, R_BYTES=R_BYTES, OFF_R=OFF_R, SMEM=OFF_R + R * R_BYTES + 512 + 1024)


@pytest.mark.parametrize("T", [QMM_Q6_K, QMM_Q3_K, QMM_Q2_K, QMM_Q8_0])
@pytest.mark.parametrize("BT", [64, 128, 256])
def test_tc_tma_raw_shared_memory_plan(T, BT):
    P = tc_tm_smem(BT, T)
    assert P["X"] >= 2 and P["R"] >= 2
    assert P["SMEM"] <= SMEM_MAX
    assert 16 * (P["X"] + P["R"] + 4) + 8 + 64 <= 480  # barrier area
    assert TM_TX[T] <= P["R_BYTES"]
    # box destinations 128-byte aligned: stages at 1024-byte multiples, the
    # odd-row box 64 rows x ROW bytes after the even one
    assert P["OFF_R"] % 1024 == 0 and P["R_BYTES"] % 1024 == 0 and (64 * TM_ROW[T]) % 128 == 0
    # box rows an odd number of 16-byte chunks apart: conflict-free chunk reads
    assert (TM_ROW[T] // 16) % 2 == 1


@pytest.mark.parametrize("T,N,K", [(QMM_Q6_K, 1000, 2048), (QMM_Q6_K, 130, 5120), (QMM_Q6_K, 5120, 17408),
                                   (QMM_Q6_K, 2, 1024), (QMM_Q6_K, 300, 3072), (QMM_Q3_K, 300, 1024),
                                   (QMM_Q3_K, 14336, 4096), (QMM_Q3_K, 130, 5120), (QMM_Q2_K, 70, 512),
                                   (QMM_Q2_K, 14336, 4096), (QMM_Q2_K, 2, 1536), (QMM_Q8_0, 301, 768),
                                   (QMM_Q8_0, 257, 4352), (QMM_Q8_0, 33, 256), (QMM_Q8_0, 14336, 4096)])
def test_tc_tma_raw_boxes(T, N, K):
    """The tensor map's stride is a 16-byte multiple; every box starts on a
    16-byte boundary (x in bytes); each row's super-step lies inside its box
    row at the offset dl the dequantiser reads from, and its read-back
    (chunks, scale word, d) stays inside the box row; TMEM lanes map onto the
    tile's 128 rows one to one, and a warp's 32 lanes read consecutive rows
    of one box."""
    assert tc_uses_tma(T, N, K)
    W = 1 << 24
    if T != QMM_Q8_0:
        ssb = SSB[T]
        RB = (K // 256) * ssb
        assert (2 * RB) % 16 == 0  # the double rows' stride
        for n0 in range(0, -(-N // 128) * 128, 128):
            assert n0 % 2 == 0
            rows = set()
            for n in range(128):
                wr = 2 * (n & 63) + (n >> 6)
                rows.add(wr)
                box, brow = n >> 6, n & 63
                assert (n0 // 2 + brow) * 2 + box == n0 + wr  # the box row holds weight row n0 + wr
                for gs in range(K // 256):
                    start = box * RB + ssb * gs  # the super-block inside its double row
                    x = start & ~15              # the box's first byte
                    assert x % 16 == 0
                    dl = (W + (n0 + wr) * RB + ssb * gs) & 15  # as the dequantiser computes it
                    assert dl == start - x and dl % 2 == 0
                    assert dl + ssb <= TM_ROW[T]
                    ROW = TM_ROW[T]
                    for h in range(2):
                        if T == QMM_Q6_K:
                            # ql 5 chunks from 4h, qh 3 from 8 + 2h, the scale word, d
                            assert 16 * (4 * h + 5) <= ROW and 16 * (8 + 2 * h + 3) <= ROW
                            assert ((dl + 192 + 8 * h + 4) & ~3) + 8 <= ROW
                        elif T == QMM_Q3_K:
                            # mask chunks 0..2, 2-bit chunks 2 + 2h .. 4 + 2h
                            assert 16 * 3 <= ROW and 16 * (4 + 2 * h + 1) <= ROW
                        else:
                            # 2-bit chunks 1 + 2h .. 3 + 2h, the scale word (4-byte aligned)
                            assert dl % 4 == 0 and 16 * (3 + 2 * h + 1) <= ROW
                            assert dl + 8 * h + 4 + 4 <= ROW
                    if T == QMM_Q6_K:
                        assert dl + 208 + 2 <= ROW
                    elif T == QMM_Q3_K:
                        assert ((dl + 108) & ~3) + 8 <= ROW and ((dl + 104) & ~3) + 8 <= ROW
                    else:
                        assert dl + 80 + 4 <= ROW
            assert rows == set(range(128))
        # warp (quarter q) lanes: rows 32(q % 2) .. of box q // 2, consecutive
        for q in range(4):
            ns = [32 * q + lane for lane in range(32)]
            assert len({n >> 6 for n in ns}) == 1
            brows = [n & 63 for n in ns]
            assert brows == list(range(brows[0], brows[0] + 32))
            for i in range(0, 32, 8):  # 8 lanes per 16-byte wavefront: distinct bank groups
                assert len({(b * TM_ROW[T] // 16) % 8 for b in brows[i:i + 8]}) == 8
    else:
        RB = (K // 32) * 34
        assert RB % 16 == 0
        for gs in range(K // 256):
            assert (136 * gs * 2) % 16 == 0 and 136 * gs * 2 + 272 <= RB
        for i in range(0, 128, 8):
            assert len({(r * TM_ROW[T] // 16) % 8 for r in range(i, i + 8)}) == 8


# ------------------------------------------- tcgen05 prefill TMA coordinates

@pytest.mark.parametrize("K", [256, 512, 4096, 14336, 17408])
@pytest.mark.parametrize("BT", [64, 128, 256])
def test_tc_tma_x_coordinates_are_16_byte_multiples(K, BT):
    """Every tiled TMA copy of the prefill starts at an inner coordinate whose
    byte offset is a multiple of 16 (the rule the hardware does not check):
    the Q4_K head box (16 bytes) at 144*sb, its quant box at 144*sb + 16 +
    64*half; the Q5_K head box (48 bytes: head and fifth bits) at 176*sb, its
    quant box at 176*sb + 48 + 64*half; and the fp16 token boxes at 128*gk
    and 128*gk + 64 elements.  Box widths are 16-byte multiples too."""
    for row, head in ((144, 16), (176, 48)):
        assert head % 16 == 0
        for gk in range(K // 128):
            sb, half = gk >> 1, gk & 1
            for x_bytes in (row * sb, row * sb + head + 64 * half):
                assert x_bytes % 16 == 0
            # the quant box lies inside the super-block
            assert row * sb + head + 64 * half + 64 <= row * (sb + 1)
        # tensor map strides: the rows are 16-byte multiples
        assert ((K // 256) * row) % 16 == 0
    for gk in range(K // 128):
        for box in (0, 1):
            assert ((gk * 128 + 64 * box) * 2) % 16 == 0
    assert (K * 2) % 16 == 0


# ------------------------------------------- qmm_t: replay of the lanes' arithmetic

import numpy as np  # noqa: E402

import oracle as O  # noqa: E402
import synth  # noqa: E402


def _byte_perm(x, y, s):
    """PTX prmt (default mode): byte i of the result is byte (s >> 4i) & 7 of
    the 8 bytes y:x (x the low word)."""
    src = [(x >> (8 * k)) & 255 for k in range(4)] + [(y >> (8 * k)) & 255 for k in range(4)]
    return sum(src[(s >> (4 * i)) & 7] << (8 * i) for i in range(4))


def _h2(v):
    """the fp16 rounding of v (round to nearest even)"""
    return float(np.float16(v))


def _b_pair(wa, wb, j, da, db):
    u = _byte_perm(wa, wb, j | (j << 4) | ((4 + j) << 8) | ((4 + j) << 12))
    v = (u & 0x00FF00FF) ^ 0x64806480
    lo = float(np.array([v & 0xFFFF], np.uint16).view(np.float16)[0])
    hi = float(np.array([v >> 16], np.uint16).view(np.float16)[0])
    # (value - 1152) is exact; then one fp16 product with d
    return _h2((lo - 1152.0) * da), _h2((hi - 1152.0) * db)


def _qmm_t_replay(W, N, K, x):
    """One matrix, all rows in 16-position groups, the lanes of one warp as the
    kernel assigns them; A = x * up rounded to fp16, B pairs as above, the MMA
    summed in f64 from the fragments; returns y[m][k] (m < 16) scaled back."""
    nb = K // 32
    RB = 34 * nb
    CPG = 4 * nb
    contig = nb in (1, 2, 4, 8)
    M = x.shape[0]
    mx = np.abs(x).max()
    ew = max(12, int(np.float32(mx).view(np.uint32) >> 23)) if mx > 0 else 12
    up = 2.0 ** (139 - ew)
    y = np.zeros((16, K))

    def word(row, off):  # 32-bit little-endian word at a 2-byte-aligned byte offset of a row
        b = W[row * RB + off: row * RB + off + 4]
        return int(b[0]) | (int(b[1]) << 8) | (int(b[2]) << 16) | (int(b[3]) << 24)

    def dval(row, blk):
        return float(np.frombuffer(bytes(W[row * RB + 34 * blk: row * RB + 34 * blk + 2]), np.float16)[0])

    for n0 in range(0, N, 16):
        for lane in range(32):
            g, t = lane >> 2, lane & 3
            rows = [n0 + 2 * t, n0 + 2 * t + 1, n0 + 2 * t + 8, n0 + 2 * t + 9]
            valid = [r < N for r in rows]
            # A fragment: rows g, g + 8 of x times up, fp16
            A = {}
            for mm in (g, g + 8):
                for kk, r in zip((2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9), rows):
                    A[(mm, kk)] = _h2(x[mm, r] * up) if (mm < M and r < N) else 0.0
            mmas = []  # (column index of B's n = g, the four B values by k)
            if contig:
                bb = (CPG * g) // 32
                qoff = 34 * bb + 2 + (CPG * g) % 32
                for jj in range(CPG):
                    ws = [word(r, qoff + 4 * (jj >> 2)) if v else 0 for r, v in zip(rows, valid)]
                    ds = [dval(r, bb) if v else 0.0 for r, v in zip(rows, valid)]
                    b01 = _b_pair(ws[0], ws[1], jj & 3, ds[0], ds[1])
                    b89 = _b_pair(ws[2], ws[3], jj & 3, ds[2], ds[3])
                    mmas.append((CPG * g + jj, jj, b01 + b89))
            else:
                for b in range(nb):
                    for j in range(4):
                        ws = [word(r, 34 * b + 2 + 4 * g) if v else 0 for r, v in zip(rows, valid)]
                        ds = [dval(r, b) if v else 0.0 for r, v in zip(rows, valid)]
                        b01 = _b_pair(ws[0], ws[1], j, ds[0], ds[1])
                        b89 = _b_pair(ws[2], ws[3], j, ds[2], ds[3])
                        mmas.append((32 * b + 4 * g + j, 4 * b + j, b01 + b89))
            # this lane's B values at (k, column) for each MMA; the D element
            # (m, column) sums over k the A of lanes (m, k) -- gather per column
            for col, _, bvals in mmas:
                for kk, bv in zip((2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9), bvals):
                    for mm in range(16):
                        a = A.get((mm, kk))
                        if a is None:  # A[m][k] of another lane group: recompute
                            r = n0 + kk
                            a = _h2(x[mm, r] * up) if (mm < M and r < N) else 0.0
                        y[mm, col] += a * bv
    return y[:M] / up


@pytest.mark.parametrize("N,K,M", [(40, 128, 5), (33, 96, 3), (16, 32, 8), (21, 256, 2)])
def test_qmm_t_lane_replay_matches_oracle(N, K, M):
    """The replayed lanes (byte permutes, exact fp16 integers, fp16 roundings of
    x*up and d*q, both column mappings) give the oracle's product within the
    stated bound, and every output column is produced exactly once."""
    W = synth.kv_cache(1, N, K, seed=N + K)
    x = synth.attention_probs(1, M, N, seed=M)[0]
    y = _qmm_t_replay(W, N, K, x)
    want, A = O.qmm_t(O.Q8_0, W, 1, N, K, x[None])
    assert np.all(np.abs(y - want[0]) <= 2e-3 * A[0] + 1e-5)


@pytest.mark.parametrize("nb", range(1, 9))
def test_qmm_t_output_columns_match_the_mma_columns(nb):
    """The reduction writes lane (g, tq)'s accumulator of MMA jj = 4b + j to
    the columns that MMA's output columns 2tq and 2tq + 1 stand for, and the
    lanes of a warp write every column of every row exactly once."""
    CPG = 4 * nb
    contig = nb in (1, 2, 4, 8)

    def col_of(nprime, b, j):  # the head-dim column of MMA (b, j)'s column index nprime
        return CPG * nprime + 4 * b + j if contig else 32 * b + 4 * nprime + j

    seen = {}
    for lane in range(32):
        g, tq = lane >> 2, lane & 3
        for b in range(nb):
            for j in range(4):
                k0 = CPG * 2 * tq + 4 * b + j if contig else 32 * b + 8 * tq + j
                k1 = k0 + CPG if contig else k0 + 4
                assert k0 == col_of(2 * tq, b, j) and k1 == col_of(2 * tq + 1, b, j)
                for m in (g, g + 8):
                    for k in (k0, k1):
                        seen[(m, k)] = seen.get((m, k), 0) + 1
    assert len(seen) == 16 * 32 * nb and all(v == 1 for v in seen.values())


# ------------------------- tcgen05 prefill: replay of the Q6_K / Q8_0 dequantisers

def _realign(words, o, nout):
    """out[j] = the 32-bit word at byte 4j + o of `words` (o even, < 16), by
    the kernel's two selects and a funnel shift."""
    t = [words[j + 1] if (o & 4) else words[j] for j in range(nout + 3)]
    u = [t[j + 2] if (o & 8) else t[j] for j in range(nout + 1)]
    sh = (o & 2) * 8
    return [((u[j] >> sh) | (u[j + 1] << (32 - sh))) & 0xFFFFFFFF if sh else u[j] for j in range(nout)]


def _words(buf, byte0, n):
    return [int.from_bytes(bytes(buf[byte0 + 4 * i: byte0 + 4 * i + 4]), "little") for i in range(n)]


def _half_bits(v):
    return float(np.array([v & 0xFFFF], np.uint16).view(np.float16)[0])


@pytest.mark.parametrize("dl", [0, 2, 4, 6, 8, 10, 12, 14])
def test_tc_q6k_dequantiser_replay(dl):
    """A Q6_K super-block staged at byte dl of its 14 chunks: the realigned ql
    and qh words, the 4+2-bit assembly, the 0x6400 exponent trick and the
    scale words give, for every one of the 256 weights of both K steps, q - 32
    exactly as the oracle unpacks it, times the fp16 rounding of d*sc."""
    blk = synth.weights(synth.Q6_K, 1, 256, seed=dl + 1)
    buf = np.zeros(224, np.uint8)
    buf[dl:dl + 210] = blk
    d_or, sc_or, q_or = O.unpack_q6_k(blk)
    d = _half_bits(d_or)
    for h in range(2):
        wl = _words(buf, 64 * h, 20)
        wh = _words(buf, 128 + 32 * h, 12)
        ql = _realign(wl, dl, 16)
        qh = _realign(wh, dl, 8)
        for cp in range(2):
            off = dl + 192 + 8 * h + 4 * cp
            scw = int.from_bytes(bytes(buf[off: off + 4]), "little")
            for qq in range(2):
                qi = 2 * cp + qq
                for half_l in range(2):  # s_lo for lw < 4, s_hi for lw >= 4
                    sbyte = (scw >> (16 * qq + 8 * half_l)) & 255
                    s = _half_bits(int(np.float16(np.float32(d) * np.float32(sbyte - 256 if sbyte > 127 else sbyte)).view(np.uint16)))
                    for lw in range(4 * half_l, 4 * half_l + 4):
                        w = ql[8 * qq + lw]
                        lo = (w & 0x0F0F0F0F) if cp == 0 else ((w >> 4) & 0x0F0F0F0F)
                        q6 = lo | (((qh[lw] >> (4 * cp + 2 * qq)) & 0x03030303) << 4)
                        for e in range(4):
                            l = 4 * lw + e
                            p = 128 * h + 32 * qi + l
                            qv = (q6 >> (8 * e)) & 255
                            # 0x6400 | q is 1024 + q; minus 1056 is q - 32, exact
                            assert qv - 32 == int(q_or[p]) - 32, (h, cp, qq, lw, e)
                            assert s == _half_bits(int(np.float16(np.float32(d) * np.float32(sc_or[p // 16])).view(np.uint16)))


@pytest.mark.parametrize("E", range(4))
def test_tc_q8_0_dequantiser_replay(E):
    """The Q8_0 dequantiser of half h = E // 2, cp = E % 2 reads blocks 4h + 2cp
    and 4h + 2cp + 1 from the 5 chunks at chunk 4E: every d and quant it
    extracts is the oracle's."""
    W = synth.weights(synth.Q8_0, 1, 256, seed=40 + E)  # eight blocks = one super-step
    words = _words(W, 64 * E, 20)

    def word_at(o):
        i = (o >> 2) + E
        return ((words[i] >> 16) | (words[i + 1] << 16)) & 0xFFFFFFFF if (o + 4 * E) & 2 else words[i]

    for bb in range(2):
        blk = 2 * E + bb  # 4h + 2cp + bb
        d_or, q_or = O.unpack_q8_0(W[34 * blk: 34 * blk + 34])
        ob = 34 * bb
        assert word_at(ob) & 0xFFFF == d_or
        for lw in range(8):
            q = word_at(ob + 2 + 4 * lw)
            for e in range(4):
                b = (q >> (8 * e)) & 255
                assert (b - 256 if b > 127 else b) == int(q_or[4 * lw + e])


@pytest.mark.parametrize("dl", [0, 2, 4, 6, 8, 10, 12, 14])
def test_tc_q3k_dequantiser_replay(dl):
    """A Q3_K super-block staged at byte dl of its 8 chunks: the scale word of
    the warp's four groups, the realigned mask and 2-bit words and the
    0x6400 exponent trick give, for every weight of both K steps and both
    warps of a lane quarter, the oracle's q (-4..3) and signed scale."""
    blk = synth.weights(synth.Q3_K, 1, 256, seed=dl + 3)
    buf = np.zeros(144, np.uint8)
    buf[dl:dl + 110] = blk
    d_or, sc_or, q_or = O.unpack_q3_k(blk)

    def word(o):
        return int.from_bytes(bytes(buf[o:o + 4]), "little")
    assert word(dl + 108) & 0xFFFF == d_or
    for h in range(2):
        for cp in range(2):
            G = 2 * h + cp
            sw, s8 = word(dl + 96 + 4 * (G & 1)), word(dl + 104)
            sc4 = (((sw >> 4) if G & 2 else sw) & 0x0F0F0F0F) | (((s8 >> (2 * G)) & 0x03030303) << 4)
            for k in range(4):
                assert ((sc4 >> (8 * k)) & 255) - 32 == int(sc_or[8 * h + 4 * cp + k])
            hm = _realign(_words(buf, 0, 12), dl, 8)
            qs = _realign(_words(buf, 16 * (2 + 2 * h), 12), dl, 8)
            for jj in range(2):
                j = 2 * cp + jj
                for e in range(8):
                    q3 = ((qs[e] >> (2 * j)) & 0x03030303) | (((hm[e] >> (4 * h + j)) & 0x01010101) << 2)
                    for b in range(4):
                        l = 4 * e + b
                        p = 128 * h + 32 * j + l
                        assert ((q3 >> (8 * b)) & 255) - 4 == int(q_or[p]), (h, cp, jj, e, b)
                        # the scale the kernel applies is group 8h + 4cp + 2jj + (e >= 4)
                        assert 8 * h + 4 * cp + 2 * jj + (e >> 2) == p // 16


@pytest.mark.parametrize("dl", [0, 4, 8, 12])
def test_tc_q2k_dequantiser_replay(dl):
    """A Q2_K super-block staged at byte dl (a multiple of 4) of its 6 chunks:
    d, dmin, the scale/min word of the warp's four groups and the realigned
    2-bit words give every weight's q, scale and min as the oracle unpacks."""
    blk = synth.weights(synth.Q2_K, 1, 256, seed=dl + 5)
    buf = np.zeros(112, np.uint8)
    buf[dl:dl + 84] = blk
    d_or, dmin_or, sc_or, m_or, q_or = O.unpack_q2_k(blk)

    def word(o):
        assert o % 4 == 0
        return int.from_bytes(bytes(buf[o:o + 4]), "little")
    dd = word(dl + 80)
    assert dd & 0xFFFF == d_or and dd >> 16 == dmin_or
    for h in range(2):
        for cp in range(2):
            sw = word(dl + 8 * h + 4 * cp)
            for k in range(4):
                g = 8 * h + 4 * cp + k
                assert (sw >> (8 * k)) & 15 == int(sc_or[g]) and (sw >> (8 * k + 4)) & 15 == int(m_or[g])
            qs = _realign(_words(buf, 16 * (1 + 2 * h), 12), dl, 8)
            for jj in range(2):
                j = 2 * cp + jj
                for e in range(8):
                    q2 = (qs[e] >> (2 * j)) & 0x03030303
                    for b in range(4):
                        p = 128 * h + 32 * j + 4 * e + b
                        assert (q2 >> (8 * b)) & 255 == int(q_or[p])
                        assert 8 * h + 4 * cp + 2 * jj + (e >> 2) == p // 16
