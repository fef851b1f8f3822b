// gemm_tc.cu -- prefill product y[M,N] = W[N,K] . x[M,K]^T for Q4_K, Q6_K
// and Q8_0 weights on the fifth-generation tensor cores (tcgen05, operands
// and accumulators in tensor memory).
//
// sm_103a has no integer tcgen05 mode, so the contraction runs in kind::f16
// with the roles chosen so that the dequantised weights never pass through
// shared memory:
//   A (128 x 128 per K step) = the weights (Q4_K d*sc*q - dmin*m, Q6_K
//       d*sc*(q-32), Q8_0 d*q) rounded to fp16, written straight into TMEM
//       by eight dequantiser warps (tcgen05.st) from the raw block bytes in
//       shared memory;
//   B (BT x 128) = the dequantised activations d_x*q_x rounded to fp16 (from the
//       quantiser), loaded by TMA with the 128-byte swizzle; BT = 64/128/256
//       tokens, so the weight tile is reused across up to 256 tokens;
//   D (128 x BT) = fp32 in TMEM: row = weight row n, column = token m.
// Each product term carries two fp16 roundings (relative 2^-11 each) and
// the sum is accumulated in fp32, well inside |dy| <= 2e-3*sum|w*x| + 1e-5.
//
// fp16 holds 2^-24 .. 65504, so both operands are scaled by powers of two
// into its normal range and the scales are undone exactly in fp32 in the
// epilogue: each token row arrives from the quantiser times 2^e_m (its
// largest |d*q| in [2^14, 2^15)), and each weight row n is dequantised times
// 2^f_n, f_n chosen from the super-block scales as they stream (the first
// puts the row's largest possible |w| 2^8 below fp16's top; when a later
// super-block would overflow, f_n drops and the row's accumulator in TMEM
// is multiplied by the exact factor once the MMAs of the earlier K steps
// have completed).
//
// Every CTA loads its own token tile: the activations are re-read from L2
// by each weight tile, which the L2 serves far below its bandwidth at these
// arithmetic intensities.
//
// Warp roles (11 warps), per 128-wide K step (half a super-block):
//   0 = token producer: the step's two 64-wide token boxes (ring released
//       by this CTA's MMA commits);
//   10 = raw weight producer: Q4_K / Q5_K the super-block head and the 64
//       quant bytes of each of the 128 weight rows per K step; Q8_0 (rows
//       are 16-byte multiples) and Q6_K (when two rows are: K a multiple of
//       1024, N even) the whole super-step of the 128 rows (ring released
//       by the dequantisers, so dequantisation runs ahead of the MMA); the
//       other Q6_K shapes, Q3_K and Q2_K have rows that are no 16-byte
//       multiples, so there the dequantisers load their rows' bytes
//       themselves;
//   1 = MMA issuer (and TMEM owner);
//   2..9 = dequantisers, two per TMEM lane quarter (warp w serves lanes
//       32*(w%4).. and the K step's weights 64*((w-2)/4)..), then epilogue
//       (TMEM -> y, half of the token columns each).
// When the tiles alone would leave SMs idle, K is split (grid z): the
// splits of a tile form a cluster, each keeps its partial tile in its own
// shared memory, and each sums a share of the tile over the cluster's CTAs
// in K order (distributed shared memory; deterministic, no atomics on y).
// All waits are bounded; on a timeout the CTA stops issuing, drains what it
// issued, frees TMEM and returns with the status word set.
#include <cuda.h>

#include <type_traits>

#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qk {

namespace {

__host__ __device__ constexpr int qk_weights(int t) { return t == QMM_Q8_0 ? 32 : 256; }
__host__ __device__ constexpr int qk_block_bytes(int t) {
    return t == QMM_Q8_0 ? 34 : t == QMM_Q6_K ? 210 : t == QMM_Q5_K ? 176 : t == QMM_Q3_K ? 110 : t == QMM_Q2_K ? 84 : 144;
}

constexpr int BW = 128, BK = 128;  // weight rows per tile, K per step (half a super-block)
constexpr int A_STAGES = 4;        // dequantised weight stages in TMEM (64 columns each)
constexpr int A_COLS = BK / 2;     // two fp16 weights per 32-bit TMEM column
// warps 2..9: dequantisers, two per TMEM lane quarter (warp w serves lanes
// 32*(w%4).. and weights 64*((w-2)/4).. of every K step)
constexpr int W_XLOAD = 0, W_MMA = 1, W_RLOAD = 10;
constexpr int NTHREADS = 11 * 32;
// Q4_K and Q5_K raw-weight stages (TMA): per weight row the super-block's
// head -- d, dmin and the 12 scale bytes (Q4_K: 16 bytes), plus the 32
// bytes of fifth bits (Q5_K: 48 bytes) -- and this K step's 64 quant bytes
// (64-byte swizzle)
template <int T>
struct RawTma {
    static constexpr int ROW = T == QMM_Q5_K ? 176 : 144;  // bytes per super-block
    static constexpr int HB = T == QMM_Q5_K ? 48 : 16;     // head bytes per row
    static constexpr int QOFF = HB;                        // first quant byte of a super-block
    static constexpr int H_BYTES = BW * HB;
    static constexpr int Q_BYTES = BW * 64;
    static constexpr int R_BYTES = H_BYTES + Q_BYTES;
};

// Q6_K (the shapes the TMA stages below do not take), Q3_K, Q2_K: rows are
// not 16-byte multiples, so no tensor map describes them; each dequantiser
// warp reads the raw bytes of its 32 rows itself with 16-byte loads into
// registers, one super-step (two K steps, 256 weights: one super-block)
// ahead, and stores them into two buffers of 32 rows x PITCH_W words, read
// back as whole 16-byte chunks (an odd number of chunks per row:
// conflict-free): the chunks from the 16-byte boundary at or below the
// super-block's start (rows are only 2-byte aligned).  (The Q8_0 entry sizes
// this path's registers when it is compiled for the TMA-staged Q8_0, where
// it never runs.)
template <int T>
struct RawStep {
    static constexpr int BYTES = 0, CHUNKS = 0, PITCH_W = 0;
};
template <>
struct RawStep<QMM_Q6_K> {
    static constexpr int BYTES = 210, CHUNKS = 14, PITCH_W = 60;
};
template <>
struct RawStep<QMM_Q8_0> {
    static constexpr int BYTES = 272, CHUNKS = 17, PITCH_W = 68;
};
// Q3_K: 110-byte super-blocks (2-byte aligned), 8 chunks from the boundary
// at or below the start; Q2_K: 84 bytes (4-byte aligned), 6 chunks
template <>
struct RawStep<QMM_Q3_K> {
    static constexpr int BYTES = 110, CHUNKS = 8, PITCH_W = 36;
};
template <>
struct RawStep<QMM_Q2_K> {
    static constexpr int BYTES = 84, CHUNKS = 6, PITCH_W = 28;
};

// Raw stages by TMA (TM): one super-step of the tile's 128 rows per stage.
//   Q6_K, Q3_K, Q2_K, when two rows are a 16-byte multiple (K a multiple of
//     1024; for Q2_K of 512) and N is even: the matrix seen as N/2 double
//     rows of 2*RB bytes; two boxes of 64 double rows x ROW bytes from the
//     16-byte boundary at or below the super-block's start in the even rows
//     (box 0) and in the odd rows (box 1), ROW an odd number of 16-byte
//     chunks that holds the super-block at any even offset and every chunk
//     and word the dequantiser reads (240 / 144 / 112 bytes).  TMEM lane n
//     holds weight row 2*(n % 64) + n / 64, so that each dequantiser warp
//     reads consecutive rows of one box (conflict-free).
//   Q8_0 (rows are 16-byte multiples when K is a multiple of 256): one box of
//     128 rows x 272 bytes (136 two-byte elements), 17 chunks apart.
template <int T>
struct RawTile {
    static constexpr int ROW = 0, BOX = 0, TX = 0, R_BYTES = 1024;
};
template <>
struct RawTile<QMM_Q6_K> {
    static constexpr int ROW = 240, BOX = 64 * ROW, TX = 2 * BOX, R_BYTES = (TX + 1023) / 1024 * 1024;
};
template <>
struct RawTile<QMM_Q3_K> {
    static constexpr int ROW = 144, BOX = 64 * ROW, TX = 2 * BOX, R_BYTES = (TX + 1023) / 1024 * 1024;
};
template <>
struct RawTile<QMM_Q2_K> {
    static constexpr int ROW = 112, BOX = 64 * ROW, TX = 2 * BOX, R_BYTES = (TX + 1023) / 1024 * 1024;
};
template <>
struct RawTile<QMM_Q8_0> {
    static constexpr int ROW = 272, BOX = 128 * ROW, TX = BOX, R_BYTES = (TX + 1023) / 1024 * 1024;
};

template <int BT, int T, bool TM = false>
struct TcCfg {
    // raw bytes by super-steps (two K steps): every type but Q4_K and Q5_K
    static constexpr bool SUPER = T != QMM_Q4_K && T != QMM_Q5_K;
    static_assert(!TM || SUPER, "raw stages by TMA: the super-step types");
    static constexpr bool OWN = SUPER && !TM;  // the dequantisers copy their own raw bytes
    static constexpr bool TMA_RAW = TM;
    static constexpr bool PERM = TM && T != QMM_Q8_0;  // double rows: TMEM lane n holds weight row 2*(n%64) + n/64
    static constexpr int R_BYTES = TM ? RawTile<T>::R_BYTES : RawTma<T>::R_BYTES;
    static constexpr int XBOX = BT * 128;   // one 64-wide K box of tokens (128-byte swizzle rows)
    static constexpr int X_BYTES = 2 * XBOX;
    static constexpr int RAW_Q = 32 * RawStep<T>::PITCH_W * 4;  // one super-step of a lane quarter's rows (OWN)
    static constexpr int X_FIT = (232448 - 1536 - 4 * RAW_Q) / X_BYTES;
    // (Q5_K's larger raw stages leave room for two 256-token stages)
    static constexpr int X_FIT_TM = (232448 - 1536 - 2 * R_BYTES) / X_BYTES;  // two raw stages at least
    static constexpr int X_STAGES = OWN  ? (X_FIT > 8 ? 8 : X_FIT)
                                    : TM ? (X_FIT_TM > 8 ? 8 : X_FIT_TM)
                                         : (BT == 256 ? (T == QMM_Q5_K ? 2 : 3) : BT == 128 ? 5 : 8);
    static constexpr int OFF_R = X_STAGES * X_BYTES;
    static constexpr int R_STAGES_FIT = OWN ? 0 : (232448 - 1536 - OFF_R) / R_BYTES;
    static constexpr int R_STAGES = R_STAGES_FIT > 8 ? 8 : R_STAGES_FIT;
    static constexpr int OFF_BAR = OFF_R + (OWN ? 4 * RAW_Q : R_STAGES * R_BYTES);
    static constexpr int SMEM_BYTES = OFF_BAR + 512 + 1024;  // barriers + base alignment slack
    static constexpr int A_COL0 = BT;                         // TMEM columns of the A stages
    static constexpr int TMEM_COLS = BT + A_COLS * A_STAGES <= 256 ? 256 : 512;
    // D fp32, A and B fp16, both K-major, M = 128 weight rows, N = BT tokens
    static constexpr uint32_t IDESC = (1u << 4) | ((BT >> 3) << 17) | ((BW >> 4) << 24);
    static_assert(X_BYTES % 1024 == 0 && R_BYTES % 1024 == 0, "stage alignment");
    static_assert(OWN || R_STAGES >= (TM ? 2 : 3), "raw ring depth");
    static_assert(SMEM_BYTES <= 232448, "shared memory");
    static_assert(16 * (X_STAGES + R_STAGES + A_STAGES) + 8 + 64 <= 480, "barrier area");
    static_assert(BT + A_COLS * A_STAGES <= TMEM_COLS, "tensor memory");
};

struct TcParams {
    const uint8_t *W;  // the blocks (read by the dequantisers for Q6_K, Q8_0)
    const float *xinv; // [M] 2^-e_m: undoes the quantiser's power of two of token row m
    int64_t RB;        // bytes per weight row
    uint64_t w_end;    // first byte past the matrix
    int M, N;
    int ksteps;   // 128-wide K steps of the whole product
    int splits;   // K ranges per tile (grid z); split z takes its share of whole super-steps
    int tile0;    // this launch's first tile (tiles numbered token-tile-major: t = mt * nt + n-tile)
    int nt;       // weight-row tiles
    float *y;
    int *status;
    int stop_step;  // the first CTA's token producer issues no step from this one on (failure test hook)
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// Shared-memory matrix descriptor for a K-major operand in the 128-byte
// swizzle layout: rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    uint64_t d = static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>(16 >> 4) << 16;    // leading byte offset (unused here)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;  // stride byte offset: next 8-row group
    d |= static_cast<uint64_t>(1) << 46;          // descriptor version
    d |= static_cast<uint64_t>(2) << 61;          // 128-byte swizzle
    return d;
}

// D[tmem] (+)= A[tmem] . B[smem]^T
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                       uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The four fp32 at the (16-byte aligned) address of `p` in this CTA's
// shared memory, read from the shared memory of the cluster's CTA `rank`.
__device__ __forceinline__ float4 ld_cluster_f32x4(const float *p, uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(a)
                 : "memory");
    return v;
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 16 consecutive fp32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    // The load writes r asynchronously: the wait is given r as operands so
    // that no use of r can be scheduled before it.
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                   "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 consecutive 32-bit columns (64 fp16 weights) into this warp's 32 TMEM
// lanes; complete after tmem_wait_st().
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 16 consecutive 32-bit columns into this warp's 32 TMEM lanes; complete
// after tmem_wait_st().
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// Weight-row scale: largest exponent E + f_n of a super-block scale that the
// type's largest |w| keeps below fp16's top (Q4_K |w| < 2^10 * max(|d|,
// |dmin|), Q6_K < 2^12 |d|, Q8_0 < 2^8 |d|, each bounded by 2^15), and the
// headroom left when f_n is (re)chosen.
// The first K step sets f_n from the larger of the row's own scale and 2^-6
// of the largest scale among the warp's 32 rows (but at most 2^6 above the
// row's own), so that a row whose first super-block happens to be small
// does not start far below its later ones, while the row's largest
// super-block always keeps its weights at or above 2^(TMAX-14)*|q| (fp16
// normals).
template <int T>
struct RowScale {
    // (Q3_K |w| < 2^7 |d|, Q2_K < 2^6 max(|d|, |dmin|))
    static constexpr int TMAX =
        T == QMM_Q4_K ? 4 : T == QMM_Q5_K ? 3 : T == QMM_Q6_K ? 2 : T == QMM_Q2_K ? 8 : 7;
    static constexpr int HEAD = 8;
    static constexpr int NEIGHBOUR = 6;
    static constexpr int UNSET = 1 << 20;  // no non-zero scale seen yet (the accumulator row is zero)
};

__device__ __forceinline__ uint32_t abs_bits(float v) { return __float_as_uint(v) & 0x7fffffffu; }

// Weight bytes read from global memory into registers (read once per CTA:
// not kept in L1).
__device__ __forceinline__ uint32_t ldg_b32(uint64_t a) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.b32 %0, [%1];" : "=r"(v) : "l"(a));
    return v;
}
__device__ __forceinline__ uint32_t ldg_u16(uint64_t a) {
    unsigned short v;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(a));
    return v;
}
__device__ __forceinline__ uint4 ldg_b128(uint64_t a) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(a));
    return v;
}

// The 32-bit word at byte offset `off` (2-byte aligned) of a row buffer that
// is 4-byte aligned: two aligned words shifted together.
__device__ __forceinline__ uint32_t row_word(const uint8_t *row, int off) {
    const uint32_t *a = reinterpret_cast<const uint32_t *>(row + (off & ~3));
    return __funnelshift_r(a[0], a[1], (off & 2) * 8);
}

// out[j] = the 32-bit word at byte 4j + o (o even, o < 16) of the words w,
// for registers w: the word offset o >> 2 is chosen by two selects per word
// (no indexing of w by a variable), then the half-word offset by a shift.
template <int NIN, int NOUT>
__device__ __forceinline__ void realign(const uint32_t (&w)[NIN], int o, uint32_t (&out)[NOUT]) {
    static_assert(NIN >= NOUT + 4, "realign reads NOUT + 4 words");
    uint32_t t[NOUT + 3], u[NOUT + 1];
#pragma unroll
    for (int j = 0; j < NOUT + 3; ++j) t[j] = (o & 4) ? w[j + 1] : w[j];
#pragma unroll
    for (int j = 0; j < NOUT + 1; ++j) u[j] = (o & 8) ? t[j + 2] : t[j];
#pragma unroll
    for (int j = 0; j < NOUT; ++j) out[j] = __funnelshift_r(u[j], u[j + 1], (o & 2) * 8);
}

// out[j] = the 32-bit word at byte o + 4j (o even) past the 4-byte aligned
// p, from 4-byte loads at p + (o & ~3) shifted by (o & 2) * 8: for a warp
// whose lanes share o (the double-row TMA stages), cheaper than loading
// whole chunks and choosing words per lane.
template <int NOUT>
__device__ __forceinline__ void words_at(const uint8_t *p, int o, uint32_t (&out)[NOUT]) {
    const uint32_t *a = reinterpret_cast<const uint32_t *>(p + (o & ~3));
    const uint32_t sh = static_cast<uint32_t>(o & 2) * 8u;
    uint32_t prev = a[0];
#pragma unroll
    for (int j = 0; j < NOUT; ++j) {
        const uint32_t next = a[j + 1];
        out[j] = __funnelshift_r(prev, next, sh);
        prev = next;
    }
}

// Four fp16 weights from the four bytes of a quant word (low nibbles, or
// high ones when hi; plus, for Q5_K, the fifth bits at bit 4 of each byte):
// w = q*a + nb with q recovered exactly from the fp16 bit pattern
// 0x6400 | q = 1024 + q.  Weights (b0,b1) -> out0, (b2,b3) -> out1.
__device__ __forceinline__ void dequant4(uint32_t w, bool hi, uint32_t fifth, __half2 a, __half2 nb,
                                         uint32_t &out0, uint32_t &out1) {
    const __half2 k1024 = __half2half2(__ushort_as_half(0x6400));
    const uint32_t m = ((hi ? (w >> 4) : w) & 0x0F0F0F0Fu) | fifth;
    uint32_t t0 = __byte_perm(m, 0x64646464u, 0x4140u);
    uint32_t t1 = __byte_perm(m, 0x64646464u, 0x4342u);
    const __half2 w0 = __hfma2(__hsub2(*reinterpret_cast<const __half2 *>(&t0), k1024), a, nb);
    const __half2 w1 = __hfma2(__hsub2(*reinterpret_cast<const __half2 *>(&t1), k1024), a, nb);
    out0 = *reinterpret_cast<const uint32_t *>(&w0);
    out1 = *reinterpret_cast<const uint32_t *>(&w1);
}

template <int T, int BT, bool TM>
__global__ void __launch_bounds__(NTHREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmH,
                   const __grid_constant__ CUtensorMap tmQ, const TcParams P) {
    using C = TcCfg<BT, T, TM>;
    extern __shared__ uint8_t smem_raw[];
    // stages need 1024-byte alignment for the 128-byte swizzle; the base is
    // advanced by an offset from the array itself (not through an integer
    // round trip), so that the compiler keeps every pointer derived from it
    // in the shared state space and reads through them are shared loads
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = P.tile0 + static_cast<int>(blockIdx.x);
    const int n0 = (tile % P.nt) * BW, m0 = (tile / P.nt) * BT;
    // this split's K steps [k_step0, k_step0 + nsteps): an even share of the
    // product's super-steps (Q6_K, Q8_0 load whole super-steps) or K steps
    constexpr int KU = C::SUPER ? 2 : 1;
    const int ku = P.ksteps / KU;
    const int k_step0 = KU * static_cast<int>(static_cast<int64_t>(blockIdx.z) * ku / P.splits);
    const int nsteps = KU * static_cast<int>(static_cast<int64_t>(blockIdx.z + 1) * ku / P.splits) - k_step0;

    const uint32_t sX = smem_u32(smem), sR = smem_u32(smem + C::OFF_R);
    const uint32_t bar = smem_u32(smem + C::OFF_BAR);
    const uint32_t bar_x_full = bar, bar_x_empty = bar_x_full + 8 * C::X_STAGES;
    const uint32_t bar_r_full = bar_x_empty + 8 * C::X_STAGES, bar_r_empty = bar_r_full + 8 * C::R_STAGES;
    const uint32_t bar_a_full = bar_r_empty + 8 * C::R_STAGES, bar_a_empty = bar_a_full + 8 * A_STAGES;
    const uint32_t bar_acc = bar_a_empty + 8 * A_STAGES;
    // Q6_K / Q8_0: per lane quarter, its raw super-step buffer is full / has been read
    const uint32_t bar_p_full = bar_acc + 8, bar_p_empty = bar_p_full + 32;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_BAR + 480);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_BAR + 488);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::X_STAGES; ++s) {
            mbar_init(bar_x_full + 8 * s, 1);
            mbar_init(bar_x_empty + 8 * s, 1);  // this CTA's MMA commit
        }
        for (int s = 0; s < C::R_STAGES; ++s) {
            mbar_init(bar_r_full + 8 * s, 1);
            mbar_init(bar_r_empty + 8 * s, 8);  // the eight dequantiser warps
        }
        for (int s = 0; s < A_STAGES; ++s) {
            mbar_init(bar_a_full + 8 * s, 8);
            mbar_init(bar_a_empty + 8 * s, 1);
        }
        mbar_init(bar_acc, 1);
        for (int qd = 0; qd < 4; ++qd) {
            mbar_init(bar_p_full + 8 * qd, 64);  // every lane of the quarter's two warps
            mbar_init(bar_p_empty + 8 * qd, 64);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == W_MMA) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(C::TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // barriers initialised and the TMEM address published before any role starts
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // a launch of the remaining tiles that follows this one on the stream
    // (the split second part of a two-part schedule) may start as SMs free
    pdl_trigger();

    if (warp == W_XLOAD) {
        // ------------------------------------------ token tile producer
        if (lane == 0) {
            // steps from `stop` on are never issued (only with the test hook:
            // the MMA issuer's bounded wait on step `stop` then expires)
            const int stop = P.tile0 == 0 && (blockIdx.x | blockIdx.z) == 0 ? P.stop_step : NO_STOP;
            int issued = 0;
            for (int kk = 0; kk < nsteps && kk < stop; ++kk) {
                const int s = kk % C::X_STAGES;
                if (kk >= C::X_STAGES &&
                    (*abort_flag || !mbar_wait(bar_x_empty + 8 * s, ((kk / C::X_STAGES) - 1) & 1, P.status))) {
                    *abort_flag = 1;
                    break;
                }
                const int gk = k_step0 + kk;  // global 128-wide K step
                const uint32_t st = sX + s * C::X_BYTES;
                mbar_arrive_expect_tx(bar_x_full + 8 * s, C::X_BYTES);
                tma_load_2d(st, &tmX, gk * BK, m0, bar_x_full + 8 * s);
                tma_load_2d(st + C::XBOX, &tmX, gk * BK + 64, m0, bar_x_full + 8 * s);
                ++issued;
            }
            // drain: every copy into this CTA has landed and the last MMA
            // commits have arrived before the CTA may exit
            for (int kk = issued > C::X_STAGES ? issued - C::X_STAGES : 0; kk < issued; ++kk) {
                mbar_wait(bar_x_full + 8 * (kk % C::X_STAGES), (kk / C::X_STAGES) & 1, P.status);
                if (!*abort_flag) mbar_wait(bar_x_empty + 8 * (kk % C::X_STAGES), (kk / C::X_STAGES) & 1, P.status);
            }
        }
    } else if (warp == W_RLOAD) {
        // ------------------------------ raw weight producer (Q4_K, Q5_K; TM)
        if constexpr (C::TMA_RAW) {
            if (lane == 0) {
                const int nss = nsteps / 2, js0 = k_step0 / 2;  // this CTA's super-steps
                int issued = 0;
                for (int js = 0; js < nss; ++js) {
                    const int r = js % C::R_STAGES;
                    if (js >= C::R_STAGES &&
                        (*abort_flag || !mbar_wait(bar_r_empty + 8 * r, ((js / C::R_STAGES) - 1) & 1, P.status))) {
                        *abort_flag = 1;
                        break;
                    }
                    const int gs = js0 + js;  // global super-step
                    const uint32_t st = sR + r * C::R_BYTES;
                    mbar_arrive_expect_tx(bar_r_full + 8 * r, RawTile<T>::TX);
                    if constexpr (C::PERM) {
                        // boxes from the 16-byte boundary at or below the super-block
                        // in the even (0) and the odd (1) rows of the double rows
                        const int rb = static_cast<int>(P.RB), ssb = RawStep<T>::BYTES;
                        tma_load_2d(st, &tmH, (ssb * gs) & ~15, n0 / 2, bar_r_full + 8 * r);
                        tma_load_2d(st + RawTile<T>::BOX, &tmH, (rb + ssb * gs) & ~15, n0 / 2, bar_r_full + 8 * r);
                    } else {
                        tma_load_2d(st, &tmH, 136 * gs, n0, bar_r_full + 8 * r);
                    }
                    ++issued;
                }
                for (int js = issued > C::R_STAGES ? issued - C::R_STAGES : 0; js < issued; ++js)
                    mbar_wait(bar_r_full + 8 * (js % C::R_STAGES), (js / C::R_STAGES) & 1, P.status);
            }
        } else if constexpr (!C::OWN) {
            if (lane == 0) {
                int issued = 0;
                for (int kk = 0; kk < nsteps; ++kk) {
                    const int r = kk % C::R_STAGES;
                    if (kk >= C::R_STAGES &&
                        (*abort_flag || !mbar_wait(bar_r_empty + 8 * r, ((kk / C::R_STAGES) - 1) & 1, P.status))) {
                        *abort_flag = 1;
                        break;
                    }
                    const int gk = k_step0 + kk;  // half gk&1 of super-block gk>>1
                    using RT = RawTma<T>;
                    const uint32_t st = sR + r * RT::R_BYTES;
                    mbar_arrive_expect_tx(bar_r_full + 8 * r, RT::R_BYTES);
                    tma_load_2d(st, &tmH, (gk >> 1) * RT::ROW, n0, bar_r_full + 8 * r);
                    tma_load_2d(st + RT::H_BYTES, &tmQ, (gk >> 1) * RT::ROW + RT::QOFF + 64 * (gk & 1), n0,
                                bar_r_full + 8 * r);
                    ++issued;
                }
                for (int kk = issued > C::R_STAGES ? issued - C::R_STAGES : 0; kk < issued; ++kk)
                    mbar_wait(bar_r_full + 8 * (kk % C::R_STAGES), (kk / C::R_STAGES) & 1, P.status);
            }
        }
    } else if (warp == W_MMA) {
        // -------------------------------------------------- MMA issuer
        if (lane == 0) {
            for (int kk = 0; kk < nsteps; ++kk) {
                const int s = kk % C::X_STAGES, sa = kk % A_STAGES;
                if (*abort_flag || !mbar_wait(bar_x_full + 8 * s, (kk / C::X_STAGES) & 1, P.status) ||
                    !mbar_wait(bar_a_full + 8 * sa, (kk / A_STAGES) & 1, P.status)) {
                    *abort_flag = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t sx = sX + s * C::X_BYTES;
                const uint32_t ta = tmem + C::A_COL0 + A_COLS * sa;
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)
                    mma_ts(tmem, ta + 8 * k, desc_sw128(sx + (k >> 2) * C::XBOX + 32 * (k & 3)), C::IDESC,
                           (kk | k) ? 1u : 0u);
                mma_commit(bar_x_empty + 8 * s);
                mma_commit(bar_a_empty + 8 * sa);
            }
            // the accumulator is final once every MMA issued above completes
            mma_commit(bar_acc);
        }
    } else {
        // ------------------------------------- dequantiser, then epilogue
        // The eight warps take every K step in order, so each parity wait on
        // a ring stage is at most one phase ahead of the stage.  Warp w fills
        // the TMEM lanes of quarter w % 4 (weight rows 32*(w%4)..) with weights
        // 64*cp .. 64*cp+63 of the K step, cp = (w - 2) / 4.
        const int quarter = warp & 3, cp = (warp - 2) >> 2;
        const int n = 32 * quarter + lane;  // TMEM lane
        const int wr = C::PERM ? 2 * (n & 63) + (n >> 6) : n;  // the weight row (within the tile) it holds
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * quarter) << 16);
        const uint32_t a_col = C::A_COL0 + 32 * cp;  // + A_COLS * stage
        // this row's power of two f_n; both warps of the quarter see the same
        // scales in the same order, so they hold the same f_n throughout
        using RS = RowScale<T>;
        int f = RS::UNSET;
        // K step kk's largest super-block scale (bits of |v|, 0 if all are
        // zero): f_n is set or lowered; on a drop, warp cp == 0 rescales the
        // quarter's accumulator rows after the MMAs of step kk - 1 complete
        // (the MMA of step kk waits for this warp's arrival).  False when a
        // wait gave up.
        auto scale_step = [&](uint32_t ab, int kk) -> bool {
            bool grow = false;
            float fac = 1.0f;
            if (kk == 0) {
                const int E = ab != 0 ? min(exponent_of(ab), 15) : -1000;
                const int Ew = __reduce_max_sync(0xffffffffu, E);
                if (ab != 0) f = RS::TMAX - RS::HEAD - min(max(E, Ew - RS::NEIGHBOUR), E + RS::NEIGHBOUR);
                return true;
            }
            if (ab != 0) {
                const int E = min(exponent_of(ab), 15);
                if (f == RS::UNSET) {
                    f = RS::TMAX - RS::HEAD - E;
                } else if (E + f > RS::TMAX) {
                    const int fn = RS::TMAX - RS::HEAD - E;
                    fac = pow2f(fn - f);
                    f = fn;
                    grow = true;
                }
            }
            if (cp != 0 || kk == 0 || !__any_sync(0xffffffffu, grow)) return true;
            const int kp = kk - 1;
            if (!__all_sync(0xffffffffu, mbar_wait(bar_a_empty + 8 * (kp % A_STAGES), (kp / A_STAGES) & 1, P.status)))
                return false;
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < BT; c += 16) {
                float v[16];
                tmem_ld16(lane_base + static_cast<uint32_t>(c), v);
                uint32_t r[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(v[i] * fac);
                tmem_st16(lane_base + static_cast<uint32_t>(c), r);
            }
            tmem_wait_st();
            return true;
        };
        auto wfac = [&]() { return f == RS::UNSET ? 1.0f : pow2f(f); };
        if constexpr (!C::SUPER) {
            for (int kk = 0; kk < nsteps; ++kk) {
                const int r = kk % C::R_STAGES, sa = kk % A_STAGES;
                bool ok = !*abort_flag;
                if (ok) ok = mbar_wait(bar_r_full + 8 * r, (kk / C::R_STAGES) & 1, P.status);
                if (ok && kk >= A_STAGES) ok = mbar_wait(bar_a_empty + 8 * sa, ((kk / A_STAGES) - 1) & 1, P.status);
                if (__any_sync(0xffffffffu, !ok)) {
                    *abort_flag = 1;
                    break;
                }
                tc_fence_after();
                using RT = RawTma<T>;
                const int h = (k_step0 + kk) & 1;  // which half of the super-block
                const uint8_t *st = smem + C::OFF_R + r * RT::R_BYTES;
                const uint4 hdr = *reinterpret_cast<const uint4 *>(st + RT::HB * n);
                // six-bit scales and mins of sub-blocks 4h..4h+3 (byte i: sub-block
                // 4h+i), GGUF packing
                uint32_t scw, mw;
                if (h == 0) {
                    scw = hdr.y & 0x3F3F3F3Fu;
                    mw = hdr.z & 0x3F3F3F3Fu;
                } else {
                    scw = (hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u);
                    mw = ((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u);
                }
                const float d0 = half_bits_to_float(hdr.x), dm0 = half_bits_to_float(hdr.x >> 16);
                if (!scale_step(max(abs_bits(d0), abs_bits(dm0)), kk)) {
                    *abort_flag = 1;
                    break;
                }
                const float d = d0 * wfac(), dmin = dm0 * wfac();
                // the quant row: 64 bytes whose 16-byte chunk f sits at f ^ ((n >> 1) & 3)
                // (TMA 64-byte swizzle), so a quarter warp's loads hit distinct banks
                const uint8_t *qrow = st + RT::H_BYTES + 64 * n;
                const int sw = (n >> 1) & 3;
                // chunk cp of 64 weights: quant bytes 32cp..32cp+31, low nibbles
                // -> sub-block 4h+2cp, high nibbles -> sub-block 4h+2cp+1
                const uint4 qa = *reinterpret_cast<const uint4 *>(qrow + 16 * ((2 * cp) ^ sw));
                const uint4 qb = *reinterpret_cast<const uint4 *>(qrow + 16 * ((2 * cp + 1) ^ sw));
                const int sh = 16 * cp;
                const __half2 ha0 = __float2half2_rn(d * static_cast<float>((scw >> sh) & 0xFF));
                const __half2 ha1 = __float2half2_rn(d * static_cast<float>((scw >> (sh + 8)) & 0xFF));
                const __half2 hb0 = __float2half2_rn(-(dmin * static_cast<float>((mw >> sh) & 0xFF)));
                const __half2 hb1 = __float2half2_rn(-(dmin * static_cast<float>((mw >> (sh + 8)) & 0xFF)));
                // weight l < 32 of the chunk is the low nibble of quant byte l,
                // weight 32 + l its high nibble; TMEM column i holds weights 2i, 2i+1
                const uint32_t qw[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
                // Q5_K: the fifth bit of weight l of sub-block j is bit j of byte l
                // of the fifth-bit plane (bytes 16..47 of the head), moved to bit 4
                uint32_t qh[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
                if constexpr (T == QMM_Q5_K) {
                    const uint4 h0 = *reinterpret_cast<const uint4 *>(st + RT::HB * n + 16);
                    const uint4 h1 = *reinterpret_cast<const uint4 *>(st + RT::HB * n + 32);
                    qh[0] = h0.x, qh[1] = h0.y, qh[2] = h0.z, qh[3] = h0.w;
                    qh[4] = h1.x, qh[5] = h1.y, qh[6] = h1.z, qh[7] = h1.w;
                }
                const int jlo = 4 * h + 2 * cp;  // the chunk's two sub-blocks: jlo (low nibbles), jlo + 1
                uint32_t rr[32];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t f_lo = ((qh[i] >> jlo) & 0x01010101u) << 4;
                    const uint32_t f_hi = ((qh[i] >> (jlo + 1)) & 0x01010101u) << 4;
                    dequant4(qw[i], false, f_lo, ha0, hb0, rr[2 * i], rr[2 * i + 1]);
                    dequant4(qw[i], true, f_hi, ha1, hb1, rr[16 + 2 * i], rr[16 + 2 * i + 1]);
                }
                tmem_st32(lane_base + a_col + A_COLS * sa, rr);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar_a_full + 8 * sa);
                    mbar_arrive(bar_r_empty + 8 * r);
                }
            }
        } else {
            // Q6_K, Q8_0, Q3_K, Q2_K: one super-step at a time.  TM: from the
            // raw stages the producer fills (r_full / r_empty, the eight warps
            // arriving).  Otherwise the quarter's 32 rows are in one buffer
            // that its two warps fill (half the chunks each) and read; p_full /
            // p_empty hand it over (each completes once per super-step, 64
            // lanes arriving)
            constexpr int SSB = RawStep<T>::BYTES, PW = RawStep<T>::PITCH_W;
            uint8_t *raw = smem + C::OFF_R + quarter * C::RAW_Q;
            const uint32_t p_full = bar_p_full + 8 * quarter, p_empty = bar_p_empty + 8 * quarter;
            const int nss = nsteps / 2;  // super-steps of this CTA (its K range starts on one)
            const int js0 = k_step0 / 2;
            const int nrows = min(32, P.N - (n0 + 32 * quarter));  // rows of the matrix (may be <= 0)
            const uint64_t rows0 = reinterpret_cast<uint64_t>(P.W) + static_cast<uint64_t>(n0 + 32 * quarter) * P.RB;
            // this warp's half of the 32 x CH chunks (row-major): chunk
            // HALF*cp + lane + 32t, t < NT, while lane + 32t < HALF
            constexpr int CH = RawStep<T>::CHUNKS, HALF = 32 * CH / 2, NT = (HALF + 31) / 32;
            uint32_t stg[4 * NT];
            auto load = [&](int js) {
                const uint64_t seg0 = rows0 + static_cast<uint64_t>(js0 + js) * SSB;
                // Q6_K, Q3_K, Q2_K: the chunks of the matrix's final super-block
                // may reach past its end; there each word is loaded only as far
                // as it lies inside (a 2-byte load for a word that straddles it)
                const bool careful = (T == QMM_Q6_K || T == QMM_Q3_K || T == QMM_Q2_K) && nrows > 0 &&
                                     ((seg0 + static_cast<uint64_t>(nrows - 1) * P.RB) & ~uint64_t(15)) + 16 * CH > P.w_end;
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const int i = lane + 32 * t, g = HALF * cp + i, r = g / CH, c = g - CH * r;
                    uint4 v = make_uint4(0u, 0u, 0u, 0u);
                    if ((HALF % 32 == 0 || i < HALF) && r < nrows) {
                        const uint64_t a = ((seg0 + static_cast<uint64_t>(r) * P.RB) & ~uint64_t(15)) + 16 * c;
                        if (!careful || a + 16 <= P.w_end) {
                            v = ldg_b128(a);
                        } else {
                            uint32_t e[4];
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const uint64_t aq = a + 4 * q;
                                e[q] = aq + 4 <= P.w_end ? ldg_b32(aq) : aq + 2 <= P.w_end ? ldg_u16(aq) : 0u;
                            }
                            v = make_uint4(e[0], e[1], e[2], e[3]);
                        }
                    }
                    stg[4 * t] = v.x;
                    stg[4 * t + 1] = v.y;
                    stg[4 * t + 2] = v.z;
                    stg[4 * t + 3] = v.w;
                }
            };
            // into the buffer (the quarter's reads of the previous super-step are done)
            auto store = [&]() {
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const int i = lane + 32 * t, g = HALF * cp + i, r = g / CH, c = g - CH * r;
                    if (HALF % 32 == 0 || i < HALF)
                        *reinterpret_cast<uint4 *>(raw + r * (PW * 4) + 16 * c) =
                            make_uint4(stg[4 * t], stg[4 * t + 1], stg[4 * t + 2], stg[4 * t + 3]);
                }
            };
            if constexpr (C::OWN) {
                load(0);
                store();
                mbar_arrive(p_full);
                if (nss > 1) load(1);
            }
            // this lane's row of the super-step's raw bytes: from the 16-byte
            // boundary at or below the super-block (Q6_K, Q3_K, Q2_K) or the
            // super-step's first block (Q8_0)
            const uint8_t *row = raw + lane * PW * 4;
            auto tm_row = [&](int js) {
                const uint8_t *st = smem + C::OFF_R + (js % max(1, C::R_STAGES)) * C::R_BYTES;
                return C::PERM ? st + (n >> 6) * RawTile<T>::BOX + (n & 63) * RawTile<T>::ROW
                               : st + n * RawTile<T>::ROW;
            };
            for (int kk = 0; kk < nsteps; ++kk) {
                const int js = kk >> 1, h = kk & 1, sa = kk % A_STAGES;
                bool ok = !*abort_flag;
                if (ok && kk >= A_STAGES) ok = mbar_wait(bar_a_empty + 8 * sa, ((kk / A_STAGES) - 1) & 1, P.status);
                if (ok && h == 0) {
                    if constexpr (C::TMA_RAW)
                        ok = mbar_wait(bar_r_full + 8 * (js % C::R_STAGES), (js / C::R_STAGES) & 1, P.status);
                    else
                        ok = mbar_wait(p_full, js & 1, P.status);
                }
                if (__any_sync(0xffffffffu, !ok)) {
                    *abort_flag = 1;
                    break;
                }
                tc_fence_after();
                if constexpr (C::TMA_RAW) row = tm_row(js);
                uint32_t rr[32];
                if constexpr (T == QMM_Q6_K) {
                    // the super-block starts at this (even) byte of its first chunk
                    const int dl = static_cast<int>((reinterpret_cast<uint64_t>(P.W) +
                                                     static_cast<uint64_t>(n0 + wr) * P.RB +
                                                     static_cast<uint64_t>(js0 + js) * SSB) & 15);
                    // half h of the super-block: ql bytes 64h.., qh 128+32h.., scales
                    // 192+8h.., d at 208; weight 32qi + l: low bits from ql byte
                    // 32(qi&1) + l (nibble qi>>1), high bits (qh byte l >> 2qi) & 3,
                    // scale 8h + 2qi + (l >= 16); w = d*sc * (q - 32).  This warp:
                    // qi = 2cp, 2cp+1.
                    const float d0 = __half2float(*reinterpret_cast<const __half *>(row + dl + 208));
                    if (!scale_step(abs_bits(d0), kk)) {
                        *abort_flag = 1;
                        break;
                    }
                    const float d = d0 * wfac();
                    const uint32_t scw = row_word(row, dl + 192 + 8 * h + 4 * cp);
                    // ql bytes 64h .. 64h+63 lie in chunks 4h .. 4h+4, qh bytes
                    // 128+32h .. 128+32h+31 in chunks 8+2h .. 10+2h
                    uint32_t qh[8], ql[16];
                    if constexpr (C::PERM) {
                        words_at(row + 64 * h, dl, ql);
                        words_at(row + 128 + 32 * h, dl, qh);
                    } else {
                        uint32_t wl[20], wh[12];
#pragma unroll
                        for (int c = 0; c < 5; ++c) {
                            const uint4 v = *reinterpret_cast<const uint4 *>(row + 16 * (4 * h + c));
                            wl[4 * c] = v.x;
                            wl[4 * c + 1] = v.y;
                            wl[4 * c + 2] = v.z;
                            wl[4 * c + 3] = v.w;
                        }
#pragma unroll
                        for (int c = 0; c < 3; ++c) {
                            const uint4 v = *reinterpret_cast<const uint4 *>(row + 16 * (8 + 2 * h + c));
                            wh[4 * c] = v.x;
                            wh[4 * c + 1] = v.y;
                            wh[4 * c + 2] = v.z;
                            wh[4 * c + 3] = v.w;
                        }
                        realign(wl, dl, ql);
                        realign(wh, dl, qh);
                    }
                    const __half2 k1056 = __half2half2(__ushort_as_half(0x6420));  // 1056 = 1024 + 32
#pragma unroll
                    for (int qq = 0; qq < 2; ++qq) {
                        const int sb = 16 * qq;  // byte of scale 8h + 2qi in scw
                        const __half2 s_lo = __float2half2_rn(d * static_cast<float>(static_cast<int8_t>(scw >> sb)));
                        const __half2 s_hi =
                            __float2half2_rn(d * static_cast<float>(static_cast<int8_t>(scw >> (sb + 8))));
                        const int hsh = 4 * cp + 2 * qq;  // 2qi: the qh bit pair
#pragma unroll
                        for (int lw = 0; lw < 8; ++lw) {
                            const uint32_t lo = cp == 0 ? (ql[8 * qq + lw] & 0x0F0F0F0Fu)
                                                        : ((ql[8 * qq + lw] >> 4) & 0x0F0F0F0Fu);
                            const uint32_t q6 = lo | (((qh[lw] >> hsh) & 0x03030303u) << 4);
                            const uint32_t p0 = __byte_perm(q6, 0x64646464u, 0x4140u);
                            const uint32_t p1 = __byte_perm(q6, 0x64646464u, 0x4342u);
                            const __half2 s = lw < 4 ? s_lo : s_hi;
                            const __half2 w0 = __hmul2(__hsub2(*reinterpret_cast<const __half2 *>(&p0), k1056), s);
                            const __half2 w1 = __hmul2(__hsub2(*reinterpret_cast<const __half2 *>(&p1), k1056), s);
                            rr[16 * qq + 2 * lw] = *reinterpret_cast<const uint32_t *>(&w0);
                            rr[16 * qq + 2 * lw + 1] = *reinterpret_cast<const uint32_t *>(&w1);
                        }
                    }
                } else if constexpr (T == QMM_Q3_K) {
                    // the super-block starts at this (even) byte of its first chunk
                    const int dl = static_cast<int>((reinterpret_cast<uint64_t>(P.W) +
                                                     static_cast<uint64_t>(n0 + wr) * P.RB +
                                                     static_cast<uint64_t>(js0 + js) * SSB) & 15);
                    // weight 128h + 32j + l, j = 2cp + jj: low bits (byte 32 + 32h + l
                    // >> 2j) & 3, high bit (mask byte l >> 4h + j) & 1, q + 4 = low |
                    // high << 2; its group 8h + 2j + (l >= 16) = 4G + k with G = 2h + cp,
                    // k = 2jj + (l >= 16), so one word of scale bytes serves the warp:
                    // the low (G < 2) or high nibble of byte (G & 1) * 4 + k and the
                    // pair (byte 8 + k >> 2G) & 3; w = d*(sc - 32) * q
                    const float d0 = half_bits_to_float(row_word(row, dl + 108));
                    if (!scale_step(abs_bits(d0), kk)) {
                        *abort_flag = 1;
                        break;
                    }
                    const float d = d0 * wfac();
                    const int G = 2 * h + cp;
                    const uint32_t sw = row_word(row, dl + 96 + 4 * (G & 1)), s8 = row_word(row, dl + 104);
                    const uint32_t sc4 = (((G & 2) ? (sw >> 4) : sw) & 0x0F0F0F0Fu) | (((s8 >> (2 * G)) & 0x03030303u) << 4);
                    __half2 sk[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        sk[k] = __float2half2_rn(d * static_cast<float>(static_cast<int>((sc4 >> (8 * k)) & 0xFFu) - 32));
                    // mask bytes 0..31 lie in chunks 0..2, the 2-bit bytes 32 + 32h ..
                    // in chunks 2 + 2h .. 4 + 2h
                    uint32_t hm[8], qs[8];
                    if constexpr (C::PERM) {
                        words_at(row, dl, hm);
                        words_at(row + 32 + 32 * h, dl, qs);
                    } else {
                        uint32_t wm[12], wq[12];
#pragma unroll
                        for (int c = 0; c < 3; ++c) {
                            const uint4 vm = *reinterpret_cast<const uint4 *>(row + 16 * c);
                            const uint4 vq = *reinterpret_cast<const uint4 *>(row + 16 * (2 + 2 * h + c));
                            wm[4 * c] = vm.x, wm[4 * c + 1] = vm.y, wm[4 * c + 2] = vm.z, wm[4 * c + 3] = vm.w;
                            wq[4 * c] = vq.x, wq[4 * c + 1] = vq.y, wq[4 * c + 2] = vq.z, wq[4 * c + 3] = vq.w;
                        }
                        realign(wm, dl, hm);
                        realign(wq, dl, qs);
                    }
                    const __half2 k1028 = __half2half2(__ushort_as_half(0x6404));  // 1028 = 1024 + 4
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj) {
                        const int j = 2 * cp + jj;
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const uint32_t q3 =
                                ((qs[e] >> (2 * j)) & 0x03030303u) | (((hm[e] >> (4 * h + j)) & 0x01010101u) << 2);
                            const uint32_t p0 = __byte_perm(q3, 0x64646464u, 0x4140u);
                            const uint32_t p1 = __byte_perm(q3, 0x64646464u, 0x4342u);
                            const __half2 sc = sk[2 * jj + (e >> 2)];
                            const __half2 w0 = __hmul2(__hsub2(*reinterpret_cast<const __half2 *>(&p0), k1028), sc);
                            const __half2 w1 = __hmul2(__hsub2(*reinterpret_cast<const __half2 *>(&p1), k1028), sc);
                            rr[16 * jj + 2 * e] = *reinterpret_cast<const uint32_t *>(&w0);
                            rr[16 * jj + 2 * e + 1] = *reinterpret_cast<const uint32_t *>(&w1);
                        }
                    }
                } else if constexpr (T == QMM_Q2_K) {
                    // the super-block starts at this (4-byte multiple) byte of its first chunk
                    const int dl = static_cast<int>((reinterpret_cast<uint64_t>(P.W) +
                                                     static_cast<uint64_t>(n0 + wr) * P.RB +
                                                     static_cast<uint64_t>(js0 + js) * SSB) & 15);
                    // weight 128h + 32j + l, j = 2cp + jj: q = (byte 16 + 32h + l >> 2j)
                    // & 3; its group 8h + 4cp + k, k = 2jj + (l >= 16), with scale and
                    // min the low and high nibble of scale byte 8h + 4cp + k;
                    // w = (d*sc)*q - dmin*m
                    // (dl is a multiple of 4: the words are read directly)
                    const uint32_t dd = *reinterpret_cast<const uint32_t *>(row + dl + 80);  // d | dmin << 16
                    const float d0 = half_bits_to_float(dd), dm0 = half_bits_to_float(dd >> 16);
                    if (!scale_step(max(abs_bits(d0), abs_bits(dm0)), kk)) {
                        *abort_flag = 1;
                        break;
                    }
                    const float d = d0 * wfac(), dmin = dm0 * wfac();
                    const uint32_t sw = *reinterpret_cast<const uint32_t *>(row + dl + 8 * h + 4 * cp);
                    __half2 ak[4], bk[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        ak[k] = __float2half2_rn(d * static_cast<float>((sw >> (8 * k)) & 15u));
                        bk[k] = __float2half2_rn(-(dmin * static_cast<float>((sw >> (8 * k + 4)) & 15u)));
                    }
                    // the 2-bit bytes 16 + 32h .. lie in chunks 1 + 2h .. 3 + 2h
                    uint32_t qs[8];
                    if constexpr (C::PERM) {
                        words_at(row + 16 + 32 * h, dl, qs);
                    } else {
                        uint32_t wq[12];
#pragma unroll
                        for (int c = 0; c < 3; ++c) {
                            const uint4 vq = *reinterpret_cast<const uint4 *>(row + 16 * (1 + 2 * h + c));
                            wq[4 * c] = vq.x, wq[4 * c + 1] = vq.y, wq[4 * c + 2] = vq.z, wq[4 * c + 3] = vq.w;
                        }
                        realign(wq, dl, qs);
                    }
                    const __half2 k1024 = __half2half2(__ushort_as_half(0x6400));
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj) {
                        const int j = 2 * cp + jj;
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const uint32_t q2 = (qs[e] >> (2 * j)) & 0x03030303u;
                            const uint32_t p0 = __byte_perm(q2, 0x64646464u, 0x4140u);
                            const uint32_t p1 = __byte_perm(q2, 0x64646464u, 0x4342u);
                            const int k = 2 * jj + (e >> 2);
                            const __half2 w0 = __hfma2(__hsub2(*reinterpret_cast<const __half2 *>(&p0), k1024), ak[k], bk[k]);
                            const __half2 w1 = __hfma2(__hsub2(*reinterpret_cast<const __half2 *>(&p1), k1024), ak[k], bk[k]);
                            rr[16 * jj + 2 * e] = *reinterpret_cast<const uint32_t *>(&w0);
                            rr[16 * jj + 2 * e + 1] = *reinterpret_cast<const uint32_t *>(&w1);
                        }
                    }
                } else {
                    // the K step's four blocks 4h..4h+3 (both warps): their largest d
                    uint32_t ab = 0;
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        ab = max(ab, abs_bits(half_bits_to_float(
                                         *reinterpret_cast<const unsigned short *>(row + 34 * (4 * h + i)))));
                    if (!scale_step(ab, kk)) {
                        *abort_flag = 1;
                        break;
                    }
                    const float wf = wfac();
                    // blocks 4h+2cp, 4h+2cp+1 of the eight: d (fp16), then 32 int8;
                    // w = d * q.  They are the 68 bytes from byte 4E of chunk 4E,
                    // E = 2h + cp (a constant below, so that every word index is one).
                    auto dequant_pair = [&](auto ec) {
                        constexpr int E = decltype(ec)::value;
                        uint32_t w[20];
#pragma unroll
                        for (int c = 0; c < 5; ++c) {
                            const uint4 v = *reinterpret_cast<const uint4 *>(row + 16 * (4 * E + c));
                            w[4 * c] = v.x;
                            w[4 * c + 1] = v.y;
                            w[4 * c + 2] = v.z;
                            w[4 * c + 3] = v.w;
                        }
                        // the 32-bit word at (even) byte offset o of the 68
                        auto word_at = [&](int o) {
                            return ((o + 4 * E) & 2) ? __funnelshift_r(w[(o >> 2) + E], w[(o >> 2) + E + 1], 16)
                                                     : w[(o >> 2) + E];
                        };
                        const __half2 k1152 = __half2half2(__ushort_as_half(0x6480));  // 1152 = 1024 + 128
#pragma unroll
                        for (int bb = 0; bb < 2; ++bb) {
                            const int ob = 34 * bb;
                            const __half2 s = __float2half2_rn(half_bits_to_float(word_at(ob)) * wf);
#pragma unroll
                            for (int lw = 0; lw < 8; ++lw) {
                                const uint32_t q = word_at(ob + 2 + 4 * lw);
                                // bytes (q0 ^ 0x80, 0x64, q1 ^ 0x80, 0x64): 1024 + 128 + q
                                const uint32_t p0 = __byte_perm(q, 0x64646464u, 0x4140u) ^ 0x00800080u;
                                const uint32_t p1 = __byte_perm(q, 0x64646464u, 0x4342u) ^ 0x00800080u;
                                const __half2 w0 = __hmul2(__hsub2(*reinterpret_cast<const __half2 *>(&p0), k1152), s);
                                const __half2 w1 = __hmul2(__hsub2(*reinterpret_cast<const __half2 *>(&p1), k1152), s);
                                rr[16 * bb + 2 * lw] = *reinterpret_cast<const uint32_t *>(&w0);
                                rr[16 * bb + 2 * lw + 1] = *reinterpret_cast<const uint32_t *>(&w1);
                            }
                        }
                    };
                    switch (2 * h + cp) {
                        case 0: dequant_pair(std::integral_constant<int, 0>{}); break;
                        case 1: dequant_pair(std::integral_constant<int, 1>{}); break;
                        case 2: dequant_pair(std::integral_constant<int, 2>{}); break;
                        default: dequant_pair(std::integral_constant<int, 3>{}); break;
                    }
                }
                tmem_st32(lane_base + a_col + A_COLS * sa, rr);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_a_full + 8 * sa);
                if constexpr (C::TMA_RAW) {
                    // super-step js is read: its raw stage may be refilled
                    if (h == 1 && lane == 0) mbar_arrive(bar_r_empty + 8 * (js % C::R_STAGES));
                } else if (h == 1) {
                    // super-step js is read; once the other warp has read it too,
                    // the next one goes into the buffer and the one after that
                    // into the registers
                    mbar_arrive(p_empty);
                    if (js + 1 < nss) {
                        if (__any_sync(0xffffffffu, !mbar_wait(p_empty, js & 1, P.status))) {
                            *abort_flag = 1;
                            break;
                        }
                        store();
                        mbar_arrive(p_full);
                        if (js + 2 < nss) load(js + 2);
                    }
                }
            }
        }
        // epilogue: TMEM lanes of this quarter, token columns of this warp's
        // half, into y (one split) or into this CTA's partial tile in shared
        // memory (split K: the rings are idle once the accumulator is final)
        const bool ok = mbar_wait(bar_acc, 0, P.status);
        const int ncol = n0 + wr;
        if (__all_sync(0xffffffffu, ok) && !*abort_flag) {
            tc_fence_after();
            const float rowf = f == RS::UNSET ? 1.0f : pow2f(-f);
            float *red = reinterpret_cast<float *>(smem);  // [BT][BW] fp32, token-major
#pragma unroll 1
            for (int cc = cp * (BT / 2); cc < (cp + 1) * (BT / 2); cc += 16) {
                float v[16];
                tmem_ld16(lane_base + static_cast<uint32_t>(cc), v);
                const float *xf = P.xinv + m0 + cc;
                const int mrem = P.M - (m0 + cc);
                if (P.splits > 1) {
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        red[(cc + i) * BW + wr] = i < mrem ? v[i] * rowf * __ldg(xf + i) : 0.0f;
                } else if (ncol < P.N) {
                    float *yc = P.y + static_cast<int64_t>(m0 + cc) * P.N + ncol;
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (i < mrem) yc[static_cast<int64_t>(i) * P.N] = v[i] * rowf * __ldg(xf + i);
                }
            }
        }
    }
    if (P.splits > 1) {
        // Split K: the tile's splits are the CTAs of one cluster (along z).
        // Once every one holds its partial tile in shared memory, CTA r sums
        // token columns [r*BT/s, (r+1)*BT/s) of the tile over the cluster's
        // CTAs in rank (= K) order -- a fixed order, so the result is
        // deterministic -- and writes them to y.  Every thread takes part in
        // both cluster barriers, also after a failed wait.
        cluster_sync_all();
        const int s_ = P.splits, r = static_cast<int>(blockIdx.z);
        const int c0 = r * BT / s_, c1 = (r + 1) * BT / s_;
        const float *red = reinterpret_cast<const float *>(smem);
        // four consecutive weight rows per thread and item; every split's
        // load of an item is issued before the sum
        constexpr int MAXS = 8;
        for (int idx = threadIdx.x; idx < (c1 - c0) * (BW / 4); idx += NTHREADS) {
            const int c = c0 + idx / (BW / 4), nn = 4 * (idx % (BW / 4));
            float4 v[MAXS];
#pragma unroll
            for (int q = 0; q < MAXS; ++q)
                if (q < s_) v[q] = ld_cluster_f32x4(red + c * BW + nn, static_cast<uint32_t>(q));
            float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
            for (int q = 0; q < MAXS; ++q)
                if (q < s_) {
                    acc.x += v[q].x;
                    acc.y += v[q].y;
                    acc.z += v[q].z;
                    acc.w += v[q].w;
                }
            if (m0 + c < P.M) {
                float *yr = P.y + static_cast<int64_t>(m0 + c) * P.N + n0 + nn;
                const float a4[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (n0 + nn + i < P.N) yr[i] = a4[i];
            }
        }
        // no CTA leaves while another may still read its shared memory
        cluster_sync_all();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == W_MMA) {
        // every MMA must have completed before TMEM is released
        mbar_wait(bar_acc, 0, P.status);
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS)
                     : "memory");
    }
    // The second part of a two-part schedule reads nothing the first part
    // writes (disjoint tiles of y, the same inputs, complete before the first
    // part started); it ends only after the first part has, so that what
    // follows on the stream sees both.  (No-op when launched without the
    // programmatic dependency.)
    pdl_wait();
}

bool tc_supported(int type, int64_t N, int64_t K, int64_t M) {
    return (type == QMM_Q4_K || type == QMM_Q5_K || type == QMM_Q6_K || type == QMM_Q3_K || type == QMM_Q2_K ||
            type == QMM_Q8_0) && K % 256 == 0 &&
           K >= 256 && N >= 1 && M >= 1 && N <= (int64_t(1) << 30) &&
           M <= (int64_t(1) << 30) && K <= (int64_t(1) << 24) && tensor_map_encoder() != nullptr;
}

// K splits per tile (cluster size along z, at most 8), only while the tiles
// alone leave SMs idle: the count that minimises the estimated time, waves
// of clusters x (K steps per split + a fixed cost of about 6 K steps per
// CTA, + 1 for the cluster's sum), with the clusters that fit at once taken
// from the occupancy calculator (a cluster's CTAs must share one GPC).
// Cached per kernel and cluster size.
// Clusters of s CTAs of the kernel resident at once (cached; -1: unknown,
// do not split this way).
template <int T, int BT, bool TM>
int clusters_resident(int s, int num_sms) {
    using C = TcCfg<BT, T, TM>;
    static int fit[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0};  // 0: not asked yet
    if (fit[s] == 0) {
        int n = 0;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1, 1, s);
        cfg.blockDim = dim3(NTHREADS);
        cfg.dynamicSmemBytes = C::SMEM_BYTES;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = s;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<T, BT, TM>, &cfg) != cudaSuccess || n < 1) {
            (void)cudaGetLastError();
            n = s == 1 ? num_sms : -1;
        }
        fit[s] = n;
    }
    return fit[s];
}

template <int T, int BT, bool TM>
int choose_splits(int64_t tiles, int ksteps, int num_sms) {
    using C = TcCfg<BT, T, TM>;
    const int kunits = C::SUPER ? ksteps / 2 : ksteps;
    int best = 1;
    double best_cost = 0.0;
    int fit[9];
    for (int s = 1; s <= 8 && s <= kunits; ++s) {
        fit[s] = clusters_resident<T, BT, TM>(s, num_sms);
        if (fit[s] < 1) continue;
        // splitting pays only while the tiles leave SMs idle in one wave
        if (s > 1 && tiles >= fit[1]) break;
        const int64_t waves = (tiles + fit[s] - 1) / fit[s];
        const double cost =
            static_cast<double>(waves) * (static_cast<double>(ksteps) / s + 6.0 + (s > 1 ? 1.0 : 0.0));
        if (s == 1 || cost < best_cost) {
            best = s;
            best_cost = cost;
        }
    }
    return best;
}

template <int T, int BT, bool TM>
cudaError_t launch_bt(EncodeTiled enc, const void *W, int64_t N, int64_t K, const void *xh, const float *xinv,
                      int64_t M, float *y, cudaStream_t st, int num_sms, int *status) {
    using C = TcCfg<BT, T, TM>;
    CUtensorMap tx = {}, th = {}, tq = {};
    // tokens: fp16 [M][K], boxes of 64 K x BT rows, 128-byte swizzle
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
        const cuuint32_t box[2] = {64, BT};
        const cuuint32_t es[2] = {1, 1};
        if (enc(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(xh), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // raw weights as bytes [N][row bytes]: 16-byte boxes (super-block header)
    // and 64-byte boxes (one K step's quants, 64-byte swizzle), 128 rows each
    const int64_t rb = (K / 256) * RawTma<T>::ROW;
    for (int which = 0; which < 2 && !C::SUPER; ++which) {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(rb), static_cast<cuuint64_t>(N)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(rb)};
        const cuuint32_t box[2] = {which ? 64u : static_cast<cuuint32_t>(RawTma<T>::HB), static_cast<cuuint32_t>(BW)};
        const cuuint32_t es[2] = {1, 1};
        if (enc(which ? &tq : &th, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(W), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, which ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    if constexpr (TM) {
        // Q6_K, Q3_K, Q2_K: N/2 double rows of 2*RB bytes, boxes of ROW bytes x
        // 64 double rows; Q8_0: N rows of RB bytes as two-byte elements, boxes
        // of 136 elements (272 bytes) x 128 rows.  Out-of-range parts arrive
        // as zeros.
        const int64_t RB = (K / qk_weights(T)) * qk_block_bytes(T);
        const bool dr = C::PERM;
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(dr ? 2 * RB : RB / 2),
                                    static_cast<cuuint64_t>(dr ? N / 2 : N)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(dr ? 2 * RB : RB)};
        const cuuint32_t box[2] = {dr ? static_cast<cuuint32_t>(RawTile<T>::ROW) : 136u, dr ? 64u : 128u};
        const cuuint32_t es[2] = {1, 1};
        if (enc(&th, dr ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(W),
                dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const int nt = static_cast<int>((N + BW - 1) / BW), mt = static_cast<int>((M + BT - 1) / BT);
    const int ksteps = static_cast<int>(K / BK);
    cudaError_t e = set_smem_attrs(gemm_tc_kernel<T, BT, TM>, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int64_t tiles = static_cast<int64_t>(nt) * mt;
    TcParams P;
    P.W = static_cast<const uint8_t *>(W);
    P.xinv = xinv;
    P.RB = (K / qk_weights(T)) * qk_block_bytes(T);
    P.w_end = reinterpret_cast<uint64_t>(W) + static_cast<uint64_t>(N) * P.RB;
    P.M = static_cast<int>(M);
    P.N = static_cast<int>(N);
    P.y = y;
    P.ksteps = ksteps;
    P.nt = nt;
    P.status = status;
    P.stop_step = inject_stop_stage();
    // tiles [tile0, tile0 + count) in clusters of `splits` along K; with
    // `after` the launch may start while the one before it on the stream
    // still runs (programmatic dependent launch)
    auto launch = [&](int64_t tile0, int64_t count, int splits, bool after) {
        P.tile0 = static_cast<int>(tile0);
        P.splits = splits;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(count), 1, splits);
        cfg.blockDim = dim3(NTHREADS);
        cfg.dynamicSmemBytes = C::SMEM_BYTES;
        cfg.stream = st;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = splits;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = after ? 2 : 1;
        return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<T, BT, TM>, tx, th, tq, P);
    };
    // Two parts when the tiles leave the last wave partly empty: the whole
    // waves unsplit, then the remaining tiles split along K (clusters) so
    // that they fill the SMs the first part frees.
    const int fit1 = clusters_resident<T, BT, TM>(1, num_sms);
    if (fit1 > 0 && tiles > fit1 && tiles % fit1 != 0) {
        const int64_t full = tiles / fit1 * fit1, rest = tiles - full;
        const int s_rest = choose_splits<T, BT, TM>(rest, ksteps, num_sms);
        if (s_rest > 1) {
            cudaError_t e2 = launch(0, full, 1, false);
            if (e2 != cudaSuccess) return e2;
            P.stop_step = NO_STOP;
            e2 = launch(full, rest, s_rest, true);
            if (e2 == cudaSuccess) count_launches(1);
            return e2;
        }
    }
    return launch(0, tiles, choose_splits<T, BT, TM>(tiles, ksteps, num_sms), false);
}

}  // namespace

EncodeTiled tensor_map_encoder() {
    static EncodeTiled fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeTiled>(nullptr);
        return reinterpret_cast<EncodeTiled>(p);
    }();
    return fn;
}

bool gemm_tc_supported(int type, int64_t N, int64_t K, int64_t M) { return tc_supported(type, N, K, M); }

cudaError_t launch_gemm_tc(int type, const void *W, int64_t N, int64_t K, const void *xh, const float *xinv,
                           int64_t M, float *y, cudaStream_t st, int num_sms, int *status) {
    if (!gemm_tc_supported(type, N, K, M)) return cudaErrorNotSupported;
    EncodeTiled enc = tensor_map_encoder();
    auto run = [&](auto t, auto tm) {
        constexpr int T = decltype(t)::value;
        constexpr bool TM = decltype(tm)::value;
        if (M <= 64) return launch_bt<T, 64, TM>(enc, W, N, K, xh, xinv, M, y, st, num_sms, status);
        if (M <= 128) return launch_bt<T, 128, TM>(enc, W, N, K, xh, xinv, M, y, st, num_sms, status);
        return launch_bt<T, 256, TM>(enc, W, N, K, xh, xinv, M, y, st, num_sms, status);
    };
    const std::false_type own;
    const std::true_type tma;
    // Q6_K, Q3_K, Q2_K raw stages by TMA when two rows are a 16-byte multiple
    // and N is even; Q8_0 rows are 16-byte multiples
    const bool pairs = (2 * (K / 256) * qk_block_bytes(type)) % 16 == 0 && N % 2 == 0;
    if (type == QMM_Q6_K)
        return pairs ? run(std::integral_constant<int, QMM_Q6_K>{}, tma) : run(std::integral_constant<int, QMM_Q6_K>{}, own);
    if (type == QMM_Q3_K)
        return pairs ? run(std::integral_constant<int, QMM_Q3_K>{}, tma) : run(std::integral_constant<int, QMM_Q3_K>{}, own);
    if (type == QMM_Q2_K)
        return pairs ? run(std::integral_constant<int, QMM_Q2_K>{}, tma) : run(std::integral_constant<int, QMM_Q2_K>{}, own);
    if (type == QMM_Q5_K) return run(std::integral_constant<int, QMM_Q5_K>{}, own);
    if (type == QMM_Q8_0) return run(std::integral_constant<int, QMM_Q8_0>{}, tma);
    return run(std::integral_constant<int, QMM_Q4_K>{}, own);
}

}  // namespace qk
