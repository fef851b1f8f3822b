"""CPU model of the decode kernel's address arithmetic (gemv.cu), checked
before any GPU run: every bulk copy starts 16-byte aligned, has a size that
is a multiple of 16, stays inside the weight buffer and its shared-memory
slot; every block a lane reads lies inside the bytes its stage copied; the
stages of all CTAs cover the matrix exactly once; the activation copies are
16-byte multiples.  The constants mirror gemv.cu (16 compute warps, ~20 KB
stages, 2..8 stage ring, 64-byte slot slack, 512-byte header)."""
import numpy as np
import pytest

import synth

NW, SLOT_SLACK, HEAD = 16, 64, 512
UPB = {synth.Q8_0: 1, synth.Q4_K: 8, synth.Q6_K: 4}
SMEM_MAX = 232448        # GB300 opt-in shared memory per block
SMS = 152
OVERREAD = {synth.Q8_0: 38, synth.Q4_K: 144, synth.Q6_K: 214}  # last byte read + 1, per block


def align(v, a):
    return (v + a - 1) // a * a


def plan(qtype, M, K):
    BB = synth.BLOCK_BYTES[qtype]
    rb = (32 // UPB[qtype]) * BB
    MT = 1 if M <= 1 else 2 if M <= 2 else 4 if M <= 4 else 8
    xd_ld = align(K // 32, 4)
    xs_ld = align(K // 16, 4)
    xq_b, xd_b, xs_b = align(MT * K, 16), align(MT * xd_ld * 4, 16), align(MT * xs_ld * 4, 16)
    nr = max(NW, NW * ((20480 + NW * rb // 2) // (NW * rb)))
    while nr >= NW // 2:
        slot = align(nr * rb + SLOT_SLACK, 128)
        for ns in range(8, 1, -1):
            off = HEAD
            off = align(off + ns * nr * MT * 4, 128)
            off = align(off + xq_b, 128)
            off = align(off + xd_b, 128)
            off = align(off + xs_b, 128)
            if off + ns * slot <= SMEM_MAX:
                return dict(NR=nr, NS=ns, slot=slot, xd_ld=xd_ld, xs_ld=xs_ld, smem=off + ns * slot)
        nr = nr - NW if nr > NW else nr - NW // 2
    return None


def check(qtype, N, K, M=1):
    BB, QK = synth.BLOCK_BYTES[qtype], synth.BLOCK_WEIGHTS[qtype]
    nb = K // QK
    RB = nb * BB
    UPR = nb * UPB[qtype]
    RPR = (UPR + 31) // 32
    total = N * RB
    P = plan(qtype, M, K)
    assert P is not None
    assert P["NR"] % NW == 0 or P["NR"] == NW // 2
    # activation copies
    for nbytes in (M * K, M * P["xd_ld"] * 4, M * P["xs_ld"] * 4):
        assert nbytes % 16 == 0

    def rbeg(R):
        row, rr = divmod(R, RPR)
        return row * RB + (32 * rr // UPB[qtype]) * BB

    def rend(R):
        row, rr = divmod(R, RPR)
        return row * RB + (min(32 * (rr + 1), UPR) // UPB[qtype]) * BB

    grid = min(SMS, N)
    covered = []
    for c in range(grid):
        r0, r1 = N * c // grid, N * (c + 1) // grid
        cta_byte = r0 * RB
        Wc = cta_byte & ~15
        cta_off = cta_byte & 15
        avail = total - Wc
        nrounds = (r1 - r0) * RPR
        nstages = -(-nrounds // P["NR"])
        for s in range(nstages):
            R0, R1 = s * P["NR"], min((s + 1) * P["NR"], nrounds)
            a, b = cta_off + rbeg(R0), cta_off + rend(R1 - 1)
            a16 = a & ~15
            b16 = (b + 15) & ~15
            tail = 0
            if b16 > avail:
                b16 = b & ~15
                tail = b - b16
            nbytes = b16 - a16
            assert (Wc + a16) % 16 == 0 and nbytes % 16 == 0 and nbytes >= 0
            assert Wc + b16 <= total and Wc + b16 + tail <= total
            assert b - a16 <= P["slot"]
            covered.append((Wc + a, Wc + b))
            # every lane's block inside the stage's bytes, over-read inside the slot
            for R in range(R0, R1):
                row, rr = divmod(R, RPR)
                nu = min(32, UPR - 32 * rr)
                for lane in range(nu):
                    kb = (32 * rr + lane) // UPB[qtype]
                    blk = cta_off + row * RB + kb * BB - a16      # offset in the slot
                    assert blk >= a - a16 and blk + BB <= b - a16
                    assert blk + OVERREAD[qtype] <= P["slot"]
                    assert blk % 2 == 0
                    if qtype == synth.Q4_K:
                        assert blk % 16 == 0
    covered.sort()
    assert covered[0][0] == 0 and covered[-1][1] == total
    for (x0, x1), (y0, y1) in zip(covered, covered[1:]):
        assert x1 == y0


SHAPES = [(q, N, K) for (_, q, K, N) in
          synth.LLAMA_1B + synth.QWEN3_14B_LAYER + synth.LM_HEAD + synth.Q8_SMALL]
SHAPES += [(synth.Q4_K, 37, 256), (synth.Q4_K, 300, 1280), (synth.Q6_K, 37, 256),
           (synth.Q6_K, 301, 1280), (synth.Q6_K, 65, 5120), (synth.Q6_K, 8, 17408),
           (synth.Q8_0, 33, 32), (synth.Q8_0, 100, 1056), (synth.Q8_0, 17, 4096),
           (synth.Q8_0, 1, 96), (synth.Q6_K, 1000, 768), (synth.Q6_K, 153, 256 * 7)]


@pytest.mark.parametrize("qtype,N,K", SHAPES)
def test_gemv_address_arithmetic(qtype, N, K):
    check(qtype, N, K)


@pytest.mark.parametrize("M", [2, 3, 4, 8])
def test_gemv_plan_fits_multi_slot(M):
    for (_, q, K, N) in synth.QWEN3_14B_LAYER:
        assert plan(q, M, K) is not None
        check(q, min(N, 400), K, M)


# ---- the block-per-lane decode kernel (gemv_sb.cu) --------------------------
SB_NWARP, SB_SU, SB_HEAD, SB_MAXNSW, SB_XPITCH = 12, 32, 2048, 6, 272


def plan_sb(qtype, M, K):
    MT = 1 if M <= 1 else 2 if M <= 2 else 4 if M <= 4 else 8
    BB = synth.BLOCK_BYTES[qtype]
    q_ld = -(-K // 256) * SB_XPITCH
    meta_ld = align((K // 32) * 4, 16) if qtype == synth.Q8_0 else (K // 256) * (80 if qtype == synth.Q4_K else 112)
    off = SB_HEAD
    off = align(off + MT * q_ld, 128)
    off = align(off + MT * meta_ld, 128)
    slot = align(SB_SU * BB + 32, 128)
    nsw = min(SB_MAXNSW, (SMEM_MAX - off) // (SB_NWARP * slot))
    if nsw < 2:
        return None
    return dict(NSW=nsw, slot=slot, ring=off, q_ld=q_ld, meta_ld=meta_ld)


def check_sb(qtype, N, K, M=1, grid=None):
    BB, QK = synth.BLOCK_BYTES[qtype], synth.BLOCK_WEIGHTS[qtype]
    nb = K // QK
    RB = nb * BB
    total = N * RB
    P = plan_sb(qtype, M, K)
    assert P is not None
    assert SB_NWARP * SB_MAXNSW * 8 + 2 * SB_NWARP * 4 + 2 * SB_NWARP * 8 * 4 <= SB_HEAD
    assert P["q_ld"] % 16 == 0 and P["meta_ld"] % 16 == 0
    grid = min(SMS, N) if grid is None else grid
    covered = []
    read_end = {synth.Q8_0: 38, synth.Q4_K: 144, synth.Q6_K: 212}[qtype]
    q, r = divmod(N, grid)
    for c in range(grid):
        r0 = q * c + min(c, r)
        r1 = r0 + q + (1 if c < r else 0)
        cta_byte = r0 * RB
        Wc, cta_off = cta_byte & ~15, cta_byte & 15
        avail = total - Wc
        U = (r1 - r0) * nb
        for w in range(SB_NWARP):
            uw0, uw1 = U * w // SB_NWARP, U * (w + 1) // SB_NWARP
            for t in range(-(-(uw1 - uw0) // SB_SU)):
                u0, u1 = uw0 + SB_SU * t, min(uw0 + SB_SU * (t + 1), uw1)
                a, b = cta_off + u0 * BB, cta_off + u1 * BB
                a16, b16 = a & ~15, (b + 15) & ~15
                tail = 0
                if b16 > avail:
                    b16 = b & ~15
                    tail = b - b16
                assert (Wc + a16) % 16 == 0 and (b16 - a16) % 16 == 0 and b16 >= a16
                assert Wc + b16 + tail <= total
                assert b - a16 <= P["slot"]
                covered.append((Wc + a, Wc + b))
                for u in range(u0, u1):
                    blk = cta_off + u * BB - a16
                    assert 0 <= blk and blk + read_end <= P["slot"] and blk % 2 == 0
                    if qtype == synth.Q4_K:
                        assert blk % 16 == 0
    covered.sort()
    assert covered[0][0] == 0 and covered[-1][1] == total
    for (x0, x1), (y0, y1) in zip(covered, covered[1:]):
        assert x1 == y0


@pytest.mark.parametrize("qtype,N,K", SHAPES)
def test_gemv_sb_address_arithmetic(qtype, N, K):
    if plan_sb(qtype, 1, K) is None:
        pytest.skip("does not fit")
    check_sb(qtype, N, K)


def test_gemv_sb_fits_the_workloads():
    for (_, q, K, N) in synth.LLAMA_1B + synth.QWEN3_14B_LAYER + synth.LM_HEAD:
        assert plan_sb(q, 1, K) is not None, (q, K)


# ---- row of a block by multiply-high (gemv_sb.cu, launch_gemv_sb) ----------
def nb_magic(rows_q, nb):
    """Mirror of the host rule: the multiplier, or 0 when the CTA's block
    indices are too large for the multiply-high identity."""
    u_max = (rows_q + 1) * nb
    return (1 << 32) // nb + 1 if u_max * nb < (1 << 32) else 0


def umulhi(a, b):
    return (a * b) >> 32


@pytest.mark.parametrize("nb", [1, 2, 3, 7, 8, 16, 20, 32, 68, 160, 544, 4096, 65535])
def test_row_by_multiply_high_exact(nb):
    rows_q = min(4096, ((1 << 32) - 1) // (nb * nb) - 1)
    magic = nb_magic(rows_q, nb)
    assert magic
    U = (rows_q + 1) * nb
    import numpy as np
    u = np.arange(U, dtype=np.uint64)
    got = (u * np.uint64(magic)) >> np.uint64(32)
    assert np.array_equal(got, u // np.uint64(nb))


def test_row_by_multiply_high_workloads():
    for (_, q, K, N) in synth.LLAMA_1B + synth.QWEN3_14B_LAYER + synth.LM_HEAD + synth.Q8_SMALL:
        nb = K // synth.BLOCK_WEIGHTS[q]
        rows_q = N // min(SMS, N)
        magic = nb_magic(rows_q, nb)
        assert magic, (K, N)
        for u in range((rows_q + 1) * nb):
            assert umulhi(u, magic) == u // nb


def test_row_by_multiply_high_refuses_large_products():
    # Q8_0 with K = 4M (nb = 131072) and thousands of rows per CTA: divide instead
    assert nb_magic(10000, 131072) == 0


# ---- one launch for several matrices that share x (qmm_group) -------------
def group_ctas(bytes_, rows, need, num_sms):
    """Mirror of group_ctas in gemv_sb.cu: CTAs in proportion to the bytes
    (largest remainders, at most one extra each), at least one per matrix and
    at least `need`, at most one per row."""
    total = sum(bytes_)
    g, frac = [], []
    for b, r, nd in zip(bytes_, rows, need):
        want = num_sms * b / total if total else 1.0
        gi = int(want)
        frac.append(want - gi)
        gi = min(max(gi, 1, nd), r)
        g.append(gi)
    used = sum(g)
    while used < num_sms:
        best = None
        for i in range(len(g)):
            if frac[i] >= 0 and g[i] < rows[i] and (best is None or frac[i] > frac[best]):
                best = i
        if best is None:
            break
        g[best] += 1
        frac[best] = -1.0
        used += 1
    return g


GROUPS = [
    [(q, K, N) for (nm, q, K, N) in synth.QWEN3_14B_LAYER if nm in ("q", "k", "v")],
    [(q, K, N) for (nm, q, K, N) in synth.QWEN3_14B_LAYER if nm in ("gate", "up")],
    [(q, K, N) for (nm, q, K, N) in synth.LLAMA_1B if nm in ("q", "kv")],
    [(synth.Q4_K, 1024, 5), (synth.Q6_K, 1024, 3000), (synth.Q8_0, 1024, 1)],
]


@pytest.mark.parametrize("group", GROUPS)
def test_group_split_covers_every_matrix(group):
    rbs = [(K // synth.BLOCK_WEIGHTS[q]) * synth.BLOCK_BYTES[q] for (q, K, N) in group]
    bytes_ = [N * rb for (q, K, N), rb in zip(group, rbs)]
    rows = [N for (q, K, N) in group]
    need = [-(-N // ((1 << 30) // rb)) for (q, K, N), rb in zip(group, rbs)]
    g = group_ctas(bytes_, rows, need, SMS)
    assert all(1 <= gi <= N for gi, (q, K, N) in zip(g, group))
    assert sum(g) <= SMS + len(group)
    for (q, K, N), gi in zip(group, g):
        check_sb(q, N, K, grid=gi)


# ---- the tensor-core decode kernel for 2 <= M <= 8 (gemv_mma.cu) ----------
MM_W, MM_GR, MM_MAXNS = 8, 16, 4
MM_HEAD = 1152 + 2 * MM_W * 128 * 4  # barriers, groups | zeros | edge sums


def plan_mm(M, K, units_at=None):
    x_ld = align(2 * K + K // 8, 128) + 16
    o_x = align(MM_HEAD, 128)
    ring = align(o_x + M * x_ld, 128)
    best = None
    for ch in (5, 3, 1):
        slot = MM_GR * 144 * ch
        ns = (SMEM_MAX - ring) // (MM_W * slot)
        if ns < 2:
            continue
        best = (ch, ns, slot)
        u = units_at(ch) if units_at else 0
        if u <= 0 or u >= 3 * MM_W:
            break
    if best is None:
        return None
    ch, ns, slot = best
    ns = min(MM_MAXNS, ns)
    return dict(NS=ns, CH=ch, pitch=144 * ch, slot=slot, ring=ring, x_ld=x_ld, off_x=o_x,
                smem=ring + MM_W * ns * slot)


def mm_launch(N, K, M):
    halves = -(-N // 8)
    grid = max(1, min(SMS, halves))
    nb = K // 256
    max_groups = (halves // grid + 2) // 2
    P = plan_mm(M, K, lambda ch: max_groups * (-(-nb // ch)))
    return P, halves, grid


def check_mm(N, K, M):
    P, halves, grid = mm_launch(N, K, M)
    assert P is not None and P["smem"] <= SMEM_MAX
    CH, pitch = P["CH"], P["pitch"]
    # activation rows: bulk copies of 2K + K/8 bytes to 16-byte aligned rows
    # whose 8 ldmatrix rows (tokens) fall in distinct 16-byte bank groups
    row_bytes = 2 * K + K // 8
    assert P["x_ld"] % 128 == 16 and P["off_x"] % 128 == 0 and P["off_x"] >= MM_HEAD
    assert P["ring"] >= P["off_x"] + M * P["x_ld"] and row_bytes % 16 == 0 and M * row_bytes < 2 ** 20
    assert row_bytes <= P["x_ld"]
    # tensor copies: 128-byte aligned destinations, box inner extent of 18*CH
    # 8-byte elements (<= 256, a multiple of 16 bytes), inner coordinate
    # 18*sb0 elements = 144*sb0 bytes (a multiple of 16)
    assert CH % 2 == 1 and 18 * CH <= 256 and (144 * CH) % 16 == 0
    assert P["ring"] % 128 == 0 and P["slot"] % 128 == 0 and (8 * pitch) % 128 == 0
    # an ldmatrix reads 16 bytes of 8 consecutive rows: 8 distinct bank groups
    assert len({(r * pitch // 16) % 8 for r in range(8)}) == 8
    nb = K // 256
    q, r = divmod(halves, grid)
    nq = -(-nb // CH)
    covered = set()
    for c in range(grid):
        h0 = q * c + min(c, r)
        nh = q + (1 if c < r else 0)
        r0, r1 = 8 * h0, min(N, 8 * (h0 + nh))
        assert r1 > r0
        ng = (nh + 1) // 2
        U = ng * nq
        for w in range(MM_W):
            uw0, uw1 = U * w // MM_W, U * (w + 1) // MM_W
            groups_of_warp = sorted({u // nq for u in range(uw0, uw1)})
            for u in range(uw0, uw1):
                gi, qi = divmod(u, nq)
                sb0 = qi * CH
                nsb = min(CH, nb - sb0)
                row0 = r0 + MM_GR * gi
                boxes = 2 if r1 - row0 > 8 else 1
                assert (18 * sb0 * 8) % 16 == 0 and row0 + 8 * boxes <= 8 * halves
                # the boxes load rows [row0, row0 + 8*boxes): every one this CTA owns,
                # none of another CTA's (rows past N arrive as zeros)
                assert row0 + 8 * boxes >= min(r1, row0 + 16) and (boxes == 1 or row0 + 16 <= r1 or r1 == N)
                for rr in range(min(8 * boxes, N - row0)):
                    for s in range(nsb):
                        key = (row0 + rr, sb0 + s)
                        assert key not in covered
                        covered.add(key)
                # every read of the stage stays inside the slot: headers and the
                # ldmatrix rows (row 15, segment 7 of the last super-block)
                assert 15 * pitch + 144 * (nsb - 1) + 16 + 16 * 7 + 16 <= P["slot"]
                # activation reads: x of sub-block 7, matrix 3; sums hi | lo
                last = sb0 + nsb - 1
                assert last * 512 + 64 * 7 + 16 * 3 + 16 <= 2 * K
                assert 2 * K + 32 * last + 16 + 16 <= row_bytes
            # only the first and the last group of a warp's range can be partial
            for gi in groups_of_warp[1:-1]:
                assert all(uw0 <= gi * nq + qi < uw1 for qi in range(nq))
    assert len(covered) == N * nb


MM_SHAPES = [(5120, 5120), (1024, 5120), (17408, 5120), (5120, 17408), (2048, 2048), (512, 2048),
             (8192, 2048), (2048, 8192), (1000, 4352), (77, 256), (16, 17408), (9, 1024), (14336, 4096)]


@pytest.mark.parametrize("N,K", MM_SHAPES)
@pytest.mark.parametrize("M", [2, 4, 8])
def test_gemv_mma_address_arithmetic(N, K, M):
    if plan_mm(M, K) is None:
        pytest.skip("does not fit (the block-per-lane kernel runs it)")
    check_mm(N, K, M)


def test_gemv_mma_fits_the_q4k_workloads():
    fits = {}
    for (_, q, K, N) in synth.LLAMA_1B + synth.QWEN3_14B_LAYER:
        if q == synth.Q4_K:
            for M in (2, 4, 8):
                fits[(K, M)] = plan_mm(M, K) is not None
    # fp16 activations of M tokens take 2*M*K bytes of shared memory: all the
    # Q4_K shapes fit but M = 8 at K = 17408 (none of which is Q4_K here)
    assert all(fits.values()), fits
    assert plan_mm(8, 17408) is None and plan_mm(4, 17408) is not None


def quantiser_mma_position(l):
    """Where the activation quantiser (quantize.cu, xh_mma) stores element l of a block of 32."""
    return ((l >> 4) * 2 + (l & 1)) * 8 + ((l >> 2) & 3) * 2 + ((l >> 1) & 1)


def test_quantiser_mma_order_is_a_permutation():
    assert sorted(quantiser_mma_position(l) for l in range(32)) == list(range(32))


# ---- the same kernel's fragment arithmetic, replayed on the CPU -------------
def _f16(v):
    return np.float16(np.float64(v))


def _h(bits):
    """fp16 value of the low 16 bits."""
    return float(np.array([bits & 0xFFFF], np.uint16).view(np.float16)[0])


def _h2(word):
    return _h(word), _h(word >> 16)


def _bits(v):
    return int(np.array([v], np.float16).view(np.uint16)[0])


def _word(lo, hi):
    return _bits(lo) | (_bits(hi) << 16)


def _u32(b, off):
    return int.from_bytes(bytes(b[off:off + 4]), "little")


def _ldmatrix(rows16):
    """ldmatrix m8n8 .b16 of one matrix: rows16[r] = 16 bytes of row r;
    lane (g, t) receives 32-bit word t of row g."""
    return [_u32(rows16[lane >> 2], 4 * (lane & 3)) for lane in range(32)]


def _mma(a, b):
    """m16n8k16 f16 MMA from per-lane registers a[lane] = (a0..a3), b[lane] =
    (b0, b1): returns C[16][8] (exact products and sums)."""
    A = np.zeros((16, 16))
    B = np.zeros((16, 8))
    for lane in range(32):
        g, t = lane >> 2, lane & 3
        a0, a1, a2, a3 = a[lane]
        A[g, 2 * t:2 * t + 2] = _h2(a0)
        A[g + 8, 2 * t:2 * t + 2] = _h2(a1)
        A[g, 2 * t + 8:2 * t + 10] = _h2(a2)
        A[g + 8, 2 * t + 8:2 * t + 10] = _h2(a3)
        b0, b1 = b[lane]
        B[2 * t:2 * t + 2, g] = _h2(b0)
        B[2 * t + 8:2 * t + 10, g] = _h2(b1)
    return A @ B


def _lane_scales(hdr, t):
    """(s0, s1, m01) as q4k_lane_scales: fp32 scales, fp16 pair of -dmin*m."""
    hx, hy, hz, hw = (_u32(hdr, 4 * i) for i in range(4))
    d, dmin = np.float32(_h(hx)), np.float32(_h(hx >> 16))
    if t < 2:
        scw, mnw = hy & 0x3F3F3F3F, hz & 0x3F3F3F3F
    else:
        scw = (hw & 0x0F0F0F0F) | ((hy >> 2) & 0x30303030)
        mnw = ((hw >> 4) & 0x0F0F0F0F) | ((hz >> 2) & 0x30303030)
    sh = 16 * (t & 1)
    s0 = np.float32(np.float32(d * np.float32((scw >> sh) & 0xFF)) * np.float32(2.0 ** 24))
    s1 = np.float32(np.float32(d * np.float32((scw >> (sh + 8)) & 0xFF)) * np.float32(2.0 ** 20))
    m0 = _f16(-np.float32(dmin * np.float32((mnw >> sh) & 0xFF)))
    m1 = _f16(-np.float32(dmin * np.float32((mnw >> (sh + 8)) & 0xFF)))
    return s0, s1, _word(m0, m1)


def _token_row(xh):
    """One token's shared-memory row for one super-block: 256 fp16 in the
    quantiser's order, then the 8 block sums hi and the 8 lo, as bytes."""
    st = np.zeros(256, np.float16)
    hi = np.zeros(8, np.float16)
    lo = np.zeros(8, np.float16)
    for b in range(8):
        for l in range(32):
            st[32 * b + quantiser_mma_position(l)] = xh[32 * b + l]
        xs = np.float32(0)
        for v in xh[32 * b:32 * b + 32]:
            xs = np.float32(xs + np.float32(v))  # any order: the values are exact in fp32 here
        hi[b] = _f16(xs)
        lo[b] = _f16(np.float32(xs - np.float32(hi[b])))
    return np.concatenate([st.view(np.uint8), hi.view(np.uint8), lo.view(np.uint8)])


def mma_replay(rows, xh, M):
    """y[16 rows][8 tokens] of one super-block column: rows = 16 Q4_K blocks
    (144 bytes), xh = fp16 activations [M][256].  Registers are built exactly
    as gemv_mma.cu builds them (ldmatrix words, nibble masks, shuffled
    scales, the min-term MMA)."""
    zero = np.zeros(544, np.uint8)
    tok = [_token_row(xh[m]) for m in range(M)] + [zero] * (8 - M)
    c = np.zeros((16, 8))
    # lane scales: (s0, s1, m01) for rows g and g+8
    ls = [(_lane_scales(rows[lane >> 2][:16], lane & 3), _lane_scales(rows[(lane >> 2) + 8][:16], lane & 3))
          for lane in range(32)]
    # min term: hi | lo planes
    xhi = _ldmatrix([tok[r][512:528] for r in range(8)])
    xlo = _ldmatrix([tok[r][528:544] for r in range(8)])
    a = [(ls[l][0][2], ls[l][1][2], ls[l][0][2], ls[l][1][2]) for l in range(32)]
    c += _mma(a, [(xhi[l], xlo[l]) for l in range(32)])
    for cc in range(4):
        seg = lambda rr, e: [rows[r + rr][16 + 16 * (2 * cc + e): 32 + 16 * (2 * cc + e)] for r in range(8)]
        wa0, wb0, wa1, wb1 = _ldmatrix(seg(0, 0)), _ldmatrix(seg(8, 0)), _ldmatrix(seg(0, 1)), _ldmatrix(seg(8, 1))
        for h in range(2):
            mk = 0x00F000F0 if h else 0x000F000F
            j = 2 * cc + h
            xw = [_ldmatrix([tok[r][64 * j + 16 * q: 64 * j + 16 * q + 16] for r in range(8)]) for q in range(4)]
            d = _mma([(wa0[l] & mk, wb0[l] & mk, (wa0[l] >> 8) & mk, (wb0[l] >> 8) & mk) for l in range(32)],
                     [(xw[0][l], xw[1][l]) for l in range(32)])
            d += _mma([(wa1[l] & mk, wb1[l] & mk, (wa1[l] >> 8) & mk, (wb1[l] >> 8) & mk) for l in range(32)],
                      [(xw[2][l], xw[3][l]) for l in range(32)])
            for lane in range(32):
                g, t = lane >> 2, lane & 3
                src = (lane & ~3) | cc  # the shuffle source in the quad
                sa = float(ls[src][0][h])
                sb = float(ls[src][1][h])
                c[g, 2 * t:2 * t + 2] += sa * d[g, 2 * t:2 * t + 2]
                c[g + 8, 2 * t:2 * t + 2] += sb * d[g + 8, 2 * t:2 * t + 2]
    return c


@pytest.mark.parametrize("M", [2, 5, 8])
def test_gemv_mma_fragments_reproduce_the_product(M):
    import oracle as O
    rows = synth.weights(synth.Q4_K, 16, 256, seed=40 + M).reshape(16, 144)
    x = synth.activations(M, 256, seed=50 + M, outlier_frac=0.05)
    q, d, _ = O.quantize_act(x)
    xh = np.array([[_f16(np.float32(d[m, k // 32]) * np.float32(q[m, k])) for k in range(256)]
                   for m in range(M)], np.float16)
    C = mma_replay(rows, xh, M)
    w = O.dequant(synth.Q4_K, rows.reshape(-1), 16 * 256).reshape(16, 256).astype(np.float64)
    exact = w @ xh.astype(np.float64).T          # [16][M]
    scale = np.abs(w) @ np.abs(xh.astype(np.float64)).T
    err = np.abs(C[:, :M] - exact)
    # fp16 of dmin*m (relative 2^-11) is the only rounding left in the weights
    assert (err <= 2e-3 * scale + 1e-7).all(), float((err / (scale + 1e-30)).max())
    assert np.all(C[:, M:] == 0.0)
