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
MM_GR, MM_MAXNS, MM_MAXP = 16, 6, 8


def mm_cw(K):
    """Consumer warps = super-blocks per stage: 8 or 10, fewer empty slots, 10 on a tie."""
    nb = K // 256
    return min((8, 10), key=lambda cw: (-(-nb // cw) * cw, -cw))


def mm_head(cw):
    return 1152 + 2 * cw * 128 * 4  # barriers, flag | zeros | partial sums of two groups


def mm_pitch(qtype, cw):
    return cw * 144 + 16 if qtype == synth.Q4_K else (((cw * 210 + 41) // 16) | 1) * 16


def mm_max_groups(N):
    halves = -(-N // 8)
    grid = max(1, min(SMS, halves))
    return (halves // grid + 2) // 2, halves, grid


def plan_mm(qtype, M, K, max_groups=0):
    nb = K // 256
    if qtype == synth.Q6_K and nb % 2:
        return None
    cw = mm_cw(K)
    pitch = mm_pitch(qtype, cw)
    xs_token = 32 if qtype == synth.Q4_K else 0
    stage = MM_GR * pitch
    for P in range(1, MM_MAXP + 1):
        nbp = nb
        if P > 1:
            nbp = -(-(-(-nb // P)) // cw) * cw
            if nbp * (P - 1) >= nb:
                continue
        x_ld = align(nbp * (512 + xs_token), 128) + 16
        o_x = mm_head(cw)
        o_xs = align(o_x + M * x_ld, 128)
        o_table = o_xs + (nbp * 512 if qtype == synth.Q6_K else 0)
        o_ring = align(o_table + (max_groups * 512 if P > 1 else 0), 128)
        ns = (SMEM_MAX - o_ring) // stage
        if ns < 2:
            continue
        ns = min(MM_MAXNS, ns)
        return dict(NS=ns, P=P, nbp=nbp, CW=cw, x_ld=x_ld, pitch=pitch, stage=stage, off_x=o_x, off_xs=o_xs,
                    off_table=o_table, ring=o_ring, smem=o_ring + ns * stage)
    return None


def check_mm(qtype, N, K, M):
    mg, halves, grid = mm_max_groups(N)
    P = plan_mm(qtype, M, K, mg)
    assert P is not None and P["smem"] <= SMEM_MAX
    pitch, nbp, nph, stage, CW = P["pitch"], P["nbp"], P["P"], P["stage"], P["CW"]
    nb = K // 256
    RB = nb * synth.BLOCK_BYTES[qtype]
    w_end = N * RB            # the matrix at address 0 (16-byte aligned)
    assert P["x_ld"] % 128 == 16 and P["off_x"] % 128 == 0 and P["off_x"] >= mm_head(CW)
    assert P["ring"] % 128 == 0 and stage % 128 == 0
    # an ldmatrix reads 16 bytes of 8 consecutive rows: 8 distinct bank groups
    assert len({(r * pitch // 16) % 8 for r in range(8)}) == 8
    assert (pitch // 16) % 2 == 1 and pitch % 16 == 0
    if qtype == synth.Q4_K:
        assert (pitch // 8) <= 256 and (8 * pitch) % 128 == 0
    else:
        assert nb % 2 == 0 and CW % 2 == 0 and pitch >= 210 * CW + 26
    if nph > 1:
        assert nbp % CW == 0 and nbp * (nph - 1) < nb
    row_bytes = 2 * K + K // 8   # quantiser output per token; then [K/16][8] fp32 sums
    for p in range(nph):
        sb, nsb = p * nbp, min(nbp, nb - p * nbp)
        assert nsb > 0
        xb = 512 * nsb
        assert xb % 16 == 0 and 512 * sb + xb <= 2 * K and xb <= P["x_ld"]
        if qtype == synth.Q4_K:
            assert 2 * K + 32 * sb + 32 * nsb <= row_bytes and 512 * nbp + 32 * nsb + 16 <= P["x_ld"]
            tx = M * xb + M * 32 * nsb
        else:
            assert (M * row_bytes) % 16 == 0 and 512 * sb + 512 * nsb <= 2 * K
            assert P["off_xs"] % 128 == 0 and P["off_xs"] + 512 * nsb <= P["off_table"]
            tx = M * xb + 512 * nsb
        assert tx < 2 ** 20
    q, r = divmod(halves, grid)
    covered = set()
    for c in range(grid):
        h0 = q * c + min(c, r)
        nh = q + (1 if c < r else 0)
        r0, r1 = 8 * h0, min(N, 8 * (h0 + nh))
        ng = (nh + 1) // 2
        assert ng <= mg
        for p in range(nph):
            sbp, nsbp = p * nbp, min(nbp, nb - p * nbp)
            nq = -(-nsbp // CW)
            for gi in range(ng):
                row0 = r0 + MM_GR * gi
                rows = min(MM_GR, r1 - row0)
                assert 1 <= rows <= MM_GR
                for kc in range(nq):
                    sb0 = sbp + kc * CW
                    nsb = min(CW, sbp + nsbp - sb0)
                    assert nsb >= 1
                    if qtype == synth.Q4_K:
                        boxes = 2 if r1 - row0 > 8 else 1
                        assert (sb0 * 144) % 16 == 0 and boxes * 8 * pitch < 2 ** 20
                        # the boxes load rows [row0, row0 + 8*boxes): every one this CTA
                        # owns, none of another CTA's (rows past N arrive as zeros)
                        assert row0 + 8 * boxes >= row0 + rows and (boxes == 1 or row0 + 16 <= r1 or r1 == N)
                        assert 15 * pitch + 144 * (CW - 1) + 16 + 16 * 7 + 16 <= stage
                    else:
                        total = 0
                        for rr in range(rows):
                            start = (row0 + rr) * RB + 210 * sb0
                            src = start & ~15
                            end = min((start + 210 * nsb + 15) & ~15, w_end & ~15)
                            nbytes = end - src
                            total += nbytes
                            assert nbytes > 0 and nbytes % 16 == 0 and src % 16 == 0
                            assert src >= 0 and end <= w_end
                            assert rr * pitch + nbytes <= stage
                            oa = start & 15
                            assert oa % 4 == 0        # even super-blocks 4-byte aligned
                            data_end = oa + 210 * nsb
                            tail = (src + data_end) - end   # bytes loaded after the wait
                            if tail > 0:
                                assert row0 + rr == N - 1 and sb0 + nsb == nb and tail == (w_end & 15)
                                assert r1 == N and row0 + MM_GR >= N
                                assert tail % 4 == 0 and rr * pitch + nbytes + tail <= stage
                            assert rr * pitch + data_end <= stage
                        assert total < 2 ** 20
                    for idx in range(nsb):
                        for rr in range(rows):
                            key = (row0 + rr, sb0 + idx)
                            assert key not in covered
                            covered.add(key)
    assert len(covered) == N * nb


MM_SHAPES = [(5120, 5120), (1024, 5120), (17408, 5120), (5120, 17408), (2048, 2048), (512, 2048),
             (8192, 2048), (2048, 8192), (1000, 4352), (77, 256), (16, 17408), (9, 1024), (14336, 4096),
             (128256, 2048), (301, 1536)]


@pytest.mark.parametrize("qtype", [synth.Q4_K, synth.Q6_K])
@pytest.mark.parametrize("N,K", MM_SHAPES)
@pytest.mark.parametrize("M", [2, 4, 8])
def test_gemv_mma_address_arithmetic(qtype, N, K, M):
    if plan_mm(qtype, M, K, mm_max_groups(N)[0]) is None:
        pytest.skip("does not fit (the block-per-lane kernel runs it)")
    check_mm(qtype, N, K, M)


def test_gemv_mma_fits_the_workloads():
    for (_, q, K, N) in synth.LLAMA_1B + synth.QWEN3_14B_LAYER + synth.LM_HEAD:
        for M in (2, 4, 8):
            P = plan_mm(q, M, K, mm_max_groups(N)[0])
            assert P is not None, (q, K, N, M)
    # x of 8 tokens at K = 17408 needs phases
    assert plan_mm(synth.Q6_K, 8, 17408, mm_max_groups(5120)[0])["P"] > 1
    assert plan_mm(synth.Q4_K, 2, 5120, mm_max_groups(5120)[0])["P"] == 1


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
    """(s0, s1, m01) as q4k_lane_scales for sub-blocks t and t+4: fp32 scales
    d*sc*fs (fs = 2^24, 2^20 for odd t), fp16 pair of -dmin*m (dmin kept
    unscaled here: the power of two 2^g cancels against um)."""
    hx, hy, hz, hw = (_u32(hdr, 4 * i) for i in range(4))
    d, dmin = np.float32(_h(hx)), np.float32(_h(hx >> 16))
    sc_lo, mn_lo = hy & 0x3F3F3F3F, hz & 0x3F3F3F3F
    sc_hi = (hw & 0x0F0F0F0F) | ((hy >> 2) & 0x30303030)
    mn_hi = ((hw >> 4) & 0x0F0F0F0F) | ((hz >> 2) & 0x30303030)
    fs = np.float32(2.0 ** 20 if t & 1 else 2.0 ** 24)
    byte = lambda w: np.float32((w >> (8 * t)) & 0xFF)
    s0 = np.float32(np.float32(d * fs) * byte(sc_lo))
    s1 = np.float32(np.float32(d * fs) * byte(sc_hi))
    m0 = _f16(-np.float32(dmin * byte(mn_lo)))
    m1 = _f16(-np.float32(dmin * byte(mn_hi)))
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
        slot = 2 * (b & 3) + (b >> 2)   # the quantiser's order of the block sums
        hi[slot] = _f16(xs)
        lo[slot] = _f16(np.float32(xs - np.float32(hi[slot])))
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
            j = 2 * cc + h              # the sub-block
            for lane in range(32):
                g, t = lane >> 2, lane & 3
                src = (lane & ~3) | (j & 3)  # the shuffle source in the quad: its first or second value
                sa = float(ls[src][0][j >> 2])
                sb = float(ls[src][1][j >> 2])
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


def _lane_q6k_scales(blk, t):
    """Sa[0..3] as q6k_superblock: d * 2^24/f * sc[4t + i] in fp32 (exact)."""
    fs = np.float32(2.0 ** 20 if t & 1 else 2.0 ** 24)
    d = np.float32(np.float32(_h(_u32(blk, 208) & 0xFFFF)) * fs)
    return [np.float32(d * np.float32(np.int8(blk[192 + 4 * t + i]))) for i in range(4)]


def _q6k_scale_pair(blk, off):
    """q6k_scale_pair: the int8 scales at off, off+1 as fp16 subnormals sc * 2^-24."""
    v = (int(blk[off]) | (int(blk[off + 1]) << 8)) ^ 0x8080
    u = (v & 0xFF) | ((v >> 8) << 16)
    k = 128 * 2.0 ** -24
    return _word(_f16(_h(u) - k), _f16(_h(u >> 16) - k))


def q6k_group_tiles(xh, M):
    """The quantiser's group-sum tiles of one super-block: X_G * 2^-4 as fp16
    hi and lo planes, [plane][G][token] (zeros for tokens >= M)."""
    t = np.zeros((2, 16, 8), np.float16)
    for m in range(M):
        for G in range(16):
            acc = np.float32(0)
            for v in xh[m, 16 * G:16 * G + 16]:
                acc = np.float32(acc + np.float32(v))
            v = np.float32(acc * np.float32(0.0625))
            t[0, G, m] = _f16(v)
            t[1, G, m] = _f16(np.float32(v - np.float32(t[0, G, m])))
    return t


def q6k_mma_replay(rows, xh, M):
    """y[16 rows][8 tokens] of one Q6_K super-block column, with the registers
    built as q6k_superblock builds them: six-bit fields assembled by
    mask/multiply/add into fp16 subnormals, one MMA per group of 16 scaled by
    the shuffled group scale, and the offset -32 d sum_G sc_G X_G as two MMAs
    over the group-sum tiles (ldmatrix rows = tokens)."""
    zero = np.zeros(512, np.uint8)
    tok = [_token_row(xh[m])[:512] for m in range(M)] + [zero] * (8 - M)
    tiles = q6k_group_tiles(xh, M)
    # ldmatrix x4 over [plane][half][token][8]: matrix q = (plane, half)
    xg = [_ldmatrix([np.ascontiguousarray(tiles[q_ >> 1, 8 * (q_ & 1):8 * (q_ & 1) + 8, r]).view(np.uint8)
                     for r in range(8)]) for q_ in range(4)]
    c = np.zeros((16, 8))
    a = []
    for lane in range(32):
        g, t = lane >> 2, lane & 3
        a.append((_q6k_scale_pair(rows[g], 192 + 2 * t), _q6k_scale_pair(rows[g + 8], 192 + 2 * t),
                  _q6k_scale_pair(rows[g], 200 + 2 * t), _q6k_scale_pair(rows[g + 8], 200 + 2 * t)))
    r = _mma(a, [(xg[0][l], xg[1][l]) for l in range(32)]) + _mma(a, [(xg[2][l], xg[3][l]) for l in range(32)])
    for row in range(16):
        k = np.float32(np.float32(_h(_u32(rows[row], 208) & 0xFFFF)) * np.float32(-(2.0 ** 33)))
        c[row, :] += float(k) * r[row, :]
    S = [(_lane_q6k_scales(rows[lane >> 2], lane & 3), _lane_q6k_scales(rows[(lane >> 2) + 8], lane & 3))
         for lane in range(32)]
    for n in range(2):
        for qi in range(4):
            xw = [_ldmatrix([tok[r][64 * (4 * n + qi) + 16 * q_: 64 * (4 * n + qi) + 16 * q_ + 16]
                             for r in range(8)]) for q_ in range(4)]
            mlo = 0x00F000F0 if qi >= 2 else 0x000F000F
            mhi = 0x00030003 << (2 * qi)
            mul = 4 if qi & 1 else 16
            for lh in range(2):
                G = 8 * n + 2 * qi + lh
                a = []
                for lane in range(32):
                    g, t = lane >> 2, lane & 3
                    regs = []
                    for r in (g, g + 8):
                        ql = _u32(rows[r], 64 * n + 32 * (qi & 1) + 16 * lh + 4 * t)
                        qh = _u32(rows[r], 128 + 32 * n + 16 * lh + 4 * t)
                        regs.append(((((qh & mhi) * mul) + (ql & mlo)) & 0xFFFFFFFF,
                                     ((((qh >> 8) & mhi) * mul) + ((ql >> 8) & mlo)) & 0xFFFFFFFF))
                    a.append((regs[0][0], regs[1][0], regs[0][1], regs[1][1]))
                b = [((xw[2][l], xw[3][l]) if lh else (xw[0][l], xw[1][l])) for l in range(32)]
                d = _mma(a, b)
                for lane in range(32):
                    g, t = lane >> 2, lane & 3
                    src = (lane & ~3) | (G >> 2)
                    c[g, 2 * t:2 * t + 2] += float(S[src][0][G & 3]) * d[g, 2 * t:2 * t + 2]
                    c[g + 8, 2 * t:2 * t + 2] += float(S[src][1][G & 3]) * d[g + 8, 2 * t:2 * t + 2]
    return c


@pytest.mark.parametrize("M", [2, 5, 8])
def test_gemv_mma_q6k_fragments_reproduce_the_product(M):
    import oracle as O
    rows = synth.weights(synth.Q6_K, 16, 256, seed=60 + M).reshape(16, 210)
    x = synth.activations(M, 256, seed=70 + M, outlier_frac=0.05)
    q, d, _ = O.quantize_act(x)
    xh = np.array([[_f16(np.float32(d[m, k // 32]) * np.float32(q[m, k])) for k in range(256)]
                   for m in range(M)], np.float16)
    C = q6k_mma_replay(rows, xh, M)
    w = O.dequant(synth.Q6_K, rows.reshape(-1), 16 * 256).reshape(16, 256).astype(np.float64)
    exact = w @ xh.astype(np.float64).T
    scale = np.abs(w) @ np.abs(xh.astype(np.float64)).T
    err = np.abs(C[:, :M] - exact)
    # no rounding left in the weights: only fp32 sums differ
    assert (err <= 1e-5 * scale + 1e-9).all(), float((err / (scale + 1e-30)).max())
    assert np.all(np.abs(C[:, M:]) == 0.0)
