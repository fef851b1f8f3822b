"""CPU model of the row-per-lane decode kernel's plan and address arithmetic
(gemv_rows.cuh), checked before any GPU run (no GPU needed):

* the shape choice (CW consumer warps, H column parts) and the shared-memory
  plan: at least two ring stages, a row pitch that is an odd number of 16-byte
  chunks and holds the largest row copy, everything within the per-block
  limit, and the shapes the GPU tests rely on fitting or not;
* the producer's copies: for every CTA, row group, chunk and row, the bulk
  copy starts on a 16-byte boundary, has a 16-byte multiple size, never reads
  past the matrix, stays inside its row's pitch, and together with the plain
  tail loads (only at the matrix end) covers the row's span of super-blocks;
* the consumers' reads: each lane's super-block (and, for the 2-byte aligned
  Q6_K rows, the up to 2 bytes its 32-bit word loads reach past it) lies
  inside what its row's copy wrote.

The constants and formulas mirror the kernel's host code (choose_shape,
plan_rows, fill_rows) and device code (the producer and consumer loops)."""
import pytest

SMEM_MAX = 232448
SMS = 152
XPITCH = 272
HEAD = 256
MAX_NS = 8
Q4_K, Q5_K, Q6_K, Q3_K, Q2_K = 1, 3, 2, 4, 5
BB = {Q4_K: 144, Q5_K: 176, Q6_K: 210, Q3_K: 110, Q2_K: 84}
REC = {Q4_K: 80, Q5_K: 80, Q6_K: 112, Q3_K: 112, Q2_K: 112}


def choose_shape(nb, bb):
    best = (8, 1, -1.0)
    for cw in (10, 8):
        for h in (1, 2):
            ch = cw * h
            fill = nb / (-(-nb // ch) * ch)
            span = min(ch, nb) * bb
            sc = fill * min(1.0, span / 2048.0)
            if sc > best[2] + 1e-9:
                best = (cw, h, sc)
    return best


def align(v, a):
    return -(-v // a) * a


def plan_rows(qtype, M, K, CW, H, max_smem=SMEM_MAX):
    MT = 1 if M <= 1 else 2 if M <= 2 else 4 if M <= 4 else 8
    bb = BB[qtype]
    GR = 32 // H
    nb = K // 256
    q_ld, meta_ld = nb * XPITCH, nb * REC[qtype]
    CH = CW * H
    chunks = CH * bb // 16 if bb % 16 == 0 else (CH * bb + 30) // 16
    pitch = 16 * (chunks | 1)
    stage = GR * pitch
    o_meta = align(HEAD + MT * q_ld, 128)
    o_red = align(o_meta + MT * meta_ld, 128)
    for ns in range(MAX_NS, 1, -1):
        o_ring = align(o_red + (ns + 1) * CW * MT * GR * 4, 128)
        need = o_ring + ns * stage
        if need <= max_smem:
            return dict(NS=ns, pitch=pitch, stage=stage, nq=-(-nb // CH), smem=need, GR=GR, CH=CH, CW=CW, H=H,
                        o_ring=o_ring, MT=MT)
    return None


def fits(qtype, M, K):
    if qtype not in BB or M < 1 or M > 8 or K < 256 or K % 256:
        return None
    cw, h, _ = choose_shape(K // 256, BB[qtype])
    return plan_rows(qtype, M, K, cw, h)


@pytest.mark.parametrize("qtype", [Q4_K, Q5_K, Q6_K, Q3_K, Q2_K])
@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_shared_memory_plan(qtype, M):
    for K in range(256, 65536 + 1, 256):
        p = fits(qtype, M, K)
        if p is None:
            continue
        assert p["NS"] >= 2 and p["smem"] <= SMEM_MAX
        assert p["pitch"] % 16 == 0 and (p["pitch"] // 16) % 2 == 1
        # the largest copy of a row: CH super-blocks from up to 15 bytes into a chunk
        longest = p["CH"] * BB[qtype] + (15 if BB[qtype] % 16 else 0)
        assert align(longest, 16) <= p["pitch"]
        assert p["o_ring"] % 128 == 0 and p["stage"] % 16 == 0


def test_the_shapes_the_gpu_tests_expect():
    # one launch on the row-per-lane kernel (tests/test_gpu_rows.py) ...
    for qtype, K, M in [(Q4_K, 5120, 8), (Q4_K, 10240, 6), (Q4_K, 2048, 4), (Q6_K, 17408, 2), (Q5_K, 17408, 1),
                        (Q4_K, 17408, 2), (Q6_K, 17408, 1), (Q6_K, 4608, 8), (Q6_K, 10240, 4), (Q6_K, 5120, 5),
                        (Q6_K, 2560, 8)]:
        assert fits(qtype, M, K) is not None, (qtype, K, M)
    # ... and one it does not take (the tensor-core path then runs)
    assert fits(Q4_K, 6, 14336) is None
    # the shapes of the decode workload
    assert choose_shape(20, 144)[:2] == (10, 2)    # Qwen3-14B K=5120, Q4_K: 2.9 KB row copies
    assert choose_shape(8, 144)[:2] == (8, 1)      # Llama-3.2-1B K=2048, Q4_K
    assert choose_shape(68, 210)[:2] == (10, 1)    # Qwen3-14B down K=17408, Q6_K


def cta_rows(N, g, cta):
    q, r = divmod(N, g)
    r0 = q * cta + min(cta, r)
    return r0, q + (1 if cta < r else 0)


def grid_of(N, K, qtype):
    RB = (K // 256) * BB[qtype]
    g = max(SMS, -(-(N * RB) // (1 << 30)))
    return min(g, N)


@pytest.mark.parametrize("qtype,N,K,M", [
    (Q4_K, 1, 256, 1), (Q4_K, 5, 1024, 2), (Q4_K, 153, 2560, 1), (Q4_K, 300, 4608, 2), (Q4_K, 4865, 5120, 1),
    (Q4_K, 200, 17408, 2), (Q4_K, 17408, 5120, 1), (Q4_K, 77, 1024, 7),
    (Q6_K, 1, 256, 1), (Q6_K, 3, 512, 2), (Q6_K, 77, 2048, 1), (Q6_K, 301, 4608, 2), (Q6_K, 150, 17408, 1),
    (Q6_K, 5120, 17408, 1), (Q6_K, 4097, 5120, 1), (Q6_K, 77, 2048, 3), (Q6_K, 301, 4608, 8),
    (Q6_K, 150, 10240, 4), (Q6_K, 4097, 5120, 5),
    (Q5_K, 1, 256, 1), (Q5_K, 77, 2048, 2), (Q5_K, 4097, 5120, 2), (Q5_K, 150, 17408, 1),
    (Q3_K, 1, 256, 1), (Q3_K, 77, 2048, 2), (Q3_K, 301, 4608, 1), (Q3_K, 4097, 5120, 2), (Q3_K, 150, 17408, 1),
    (Q2_K, 3, 512, 2), (Q2_K, 33, 2560, 1), (Q2_K, 300, 4608, 2), (Q2_K, 4865, 5120, 1), (Q2_K, 200, 17408, 2),
])
def test_copies_cover_each_row_span_and_reads_stay_inside(qtype, N, K, M):
    p = fits(qtype, M, K)
    assert p is not None
    bb, nb = BB[qtype], K // 256
    RB = nb * bb
    W = 1 << 20                        # a 16-byte aligned base address
    w_end = W + N * RB
    GR, CH, pitch = p["GR"], p["CH"], p["pitch"]
    g = grid_of(N, K, qtype)
    seen_rows = 0
    for cta in range(g):
        r0, rows = cta_rows(N, g, cta)
        seen_rows += rows
        ng = -(-rows // GR)
        for gi in range(ng):
            for kc in range(p["nq"]):
                sb0 = kc * CH
                nsb = min(CH, nb - sb0)
                for lane in range(GR):
                    if GR * gi + lane >= rows:
                        continue
                    row = r0 + GR * gi + lane
                    start = W + row * RB + bb * sb0
                    end = start + bb * nsb
                    src = start & ~15
                    e16 = (end + 15) & ~15
                    plain = 0
                    if e16 > w_end:
                        e16 = max(end & ~15, src)
                        plain = end - e16
                    nbytes = e16 - src
                    # the bulk copy: aligned, a 16-byte multiple, inside the matrix and the pitch
                    assert src % 16 == 0 and nbytes % 16 == 0 and src >= W and e16 <= w_end
                    assert end - src <= pitch and nbytes <= pitch
                    # the bulk bytes (rounded out to 16) and the plain tail bytes
                    # (only at the matrix end, where they end exactly at the span's
                    # end) cover [start, end)
                    assert src <= start
                    assert (plain == 0 and e16 >= end) or (plain > 0 and e16 + plain == end and end == w_end)
                    # the consumers: lane (row, part) of warp w reads super-block js of the stage
                    off = (W + row * RB + bb * sb0) & 15
                    for js in range(nsb):
                        first = off + js * bb
                        last = first + bb + (2 if bb % 4 else 0)   # 2-byte aligned rows: word loads reach 2 bytes past
                        assert first >= 0 and first + bb <= max(nbytes, end - src)
                        assert last <= pitch
    assert seen_rows == N
