"""CPU model of the decode kernel's address arithmetic (gemv.cu), checked
before any GPU run: every bulk copy starts 16-byte aligned, has a size that
is a multiple of 16, stays inside the weight buffer and its shared-memory
slot; every block a lane reads lies inside the bytes its stage copied; the
stages of all CTAs cover the matrix exactly once; the activation copies are
16-byte multiples.  The constants mirror gemv.cu (16 compute warps, ~20 KB
stages, 2..8 stage ring, 64-byte slot slack, 512-byte header)."""
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
