// qmm_t.cu -- the product with the transposed block matrices,
//   y[h][m][k] = sum_n x[h][m][n] * w[h][n][k],   h < H, m < M, k < K,
// for H matrices of N rows of K Q8_0 weights: the value side of attention
// over a KV cache stored as q8_0 (infr landing page, "why > Paged experts,
// spillable KV": the KV cache can be kept in q8_0), one row of head_dim
// weights per cached position, x the attention probabilities of the M query
// heads that share the cache head.
//
// Memory-bound: every weight byte is read once.  Each CTA owns a contiguous
// range of one matrix's rows (a chunk), split evenly between its warps
// (sixteen for K <= 160, eight beyond, where a lane's accumulators need more
// than the 128 registers of a 512-thread block); each warp streams its rows
// through a private ring of shared-memory stages of about 4 KB with bulk
// async copies (its lane 0 refills a stage as soon as the warp has read it),
// so 16 (8) copy streams per SM keep the bytes in flight.  The contraction is
// issue-bound: four warps per scheduler hide its latencies better than two.  A warp
// contracts 16 rows at a time on the tensor cores (mma.sync m16n8k16, fp16
// operands, fp32 accumulation):
//   A (16 x 16) = x[m][n] * 2^e for the 16 positions n (rows m >= M zero),
//       2^e a power of two per warp that puts the largest |x| the warp has
//       met into [2^12, 2^13) (fp16's normal range): when a group of 16
//       positions raises that maximum, the accumulators are rescaled by the
//       exact power of two, and the scale is undone at the end;
//   B (16 x 8)  = d*q of the 16 positions for eight of the K columns: the
//       int8 q of two rows are paired by one byte permute, made exact fp16
//       integers by the 0x6400 exponent trick, and scaled by their rows' d
//       (one fp16 rounding of the exact d*q).
// Columns (g the MMA's column index, 0..7): for K = 32, 64, 128 or 256 the
// MMA j covers columns CPG*g + j with CPG = K/8, so each lane reads CPG
// contiguous quant bytes of one block per row (one d per row) and ends up
// holding 2*CPG consecutive columns; for the other K the MMA j (0..3) of
// block b covers columns 32b + 4g + j, a 4-byte group per row and block.
// Reduction, in a fixed order so that the result is bitwise reproducible:
// the warps' sums, scaled back, meet in shared memory (with W warps, warp
// w + W/2 added to warp w, then the W/2 pair sums in warp order), each CTA
// writes its chunk sum to the workspace, and the CTA that finishes a matrix
// last (a counter per matrix, reset by that CTA) adds the chunk sums in chunk
// order and writes y.
//
// Bounded waits only: a wait that expires raises the status word; the warp
// still drains its copies and the CTA completes the reduction protocol.
#include <type_traits>

#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qk {

namespace {

constexpr int VT_MG = 16;                              // rows of x per launch
constexpr int VT_RING = 192 * 1024;                    // shared-memory ring bytes of all warps (about)

// warps per CTA: sixteen while a lane's NB x 16 accumulators leave room in
// the 128 registers that 512 threads may use; eight beyond
constexpr int vt_warps(int nb) { return nb <= 5 ? 16 : 8; }

template <int NB>
struct VtCfg {
    static constexpr int WARPS = vt_warps(NB), HALF = WARPS / 2, THREADS = 32 * WARPS;
    static constexpr int K = 32 * NB, RB = 34 * NB;
    // rows per stage, a multiple of 16: copies of 2 to 4.4 KB (much smaller
    // ones are limited by the copy engine's rate, not by HBM), at least two
    // stages per warp in flight
    static constexpr int SR = NB == 1 ? 64 : NB <= 4 ? 32 : 16;
    // a stage, + room for the 16-byte rounding of both ends
    static constexpr int SLOT = (SR * RB + 32 + 15) & ~15;
    static constexpr int D_FIT = VT_RING / (WARPS * SLOT);
    static constexpr int D = D_FIT > 8 ? 8 : D_FIT;           // ring depth per warp
    static constexpr int FR = 16 * K;                         // floats of one warp's sums
    static constexpr int SMEM = WARPS * D * SLOT + 8 * WARPS * D + 16;
    // after the stream the rings hold the pair sums, [HALF][FR] floats
    static_assert(HALF * FR * 4 <= WARPS * D * SLOT, "warp sums fit in the rings");
    static_assert(D >= 2, "at least two stages per warp");
};

// 2^(e - 127) as a float for a biased exponent 1 <= e <= 254, else 0
__device__ __forceinline__ float pow2_biased(int e) {
    return e >= 1 && e <= 254 ? __uint_as_float(static_cast<uint32_t>(e) << 23) : 0.0f;
}

struct VtParams {
    const uint8_t *W;   // H*N rows of RB bytes
    uint64_t w_end;     // first byte past the matrices
    int64_t N;          // rows per matrix
    int64_t R;          // rows per chunk (a multiple of the warps per CTA)
    int nchunk;         // chunks per matrix
    const float *x;     // [H][M][N]
    int64_t M;
    int m0, mg;         // this launch's rows of x: m0 .. m0 + mg - 1 (mg <= 16)
    float *y;           // [H][M][K]
    float *part;        // [H][nchunk][16][K] chunk sums
    unsigned *count;    // [H] finished chunks, zero between calls
    int *status;
};

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// The B pair (d_a*q_a[j], d_b*q_b[j]) from byte j of the quant words of two
// rows: bytes (q_a ^ 0x80, 0x64, q_b ^ 0x80, 0x64) are the fp16 values
// 1152 + q, so subtracting 1152 gives q exactly; then one multiply by (d_a, d_b).
__device__ __forceinline__ uint32_t b_pair(uint32_t wa, uint32_t wb, int j, __half2 dd) {
    const uint32_t u = __byte_perm(wa, wb, j | (j << 4) | ((4 + j) << 8) | ((4 + j) << 12));
    const uint32_t v = (u & 0x00FF00FFu) ^ 0x64806480u;
    const __half2 k1152 = __half2half2(__ushort_as_half(0x6480));
    const __half2 r = __hmul2(__hsub2(*reinterpret_cast<const __half2 *>(&v), k1152), dd);
    return *reinterpret_cast<const uint32_t *>(&r);
}

// Rows are read from the rings through plain pointers into the dynamic
// shared memory (the compiler then folds the constant offsets into the loads
// and schedules them freely after the stage's barrier wait, whose asm clobbers
// memory).

// The fp16 d of block b of a row (2-byte aligned), as raw bits; zero for a
// row past the matrix.
__device__ __forceinline__ uint32_t row_d(const uint8_t *row, int b, bool valid) {
    return valid ? *reinterpret_cast<const uint16_t *>(row + 34 * b) : 0u;
}

// NW consecutive 32-bit words starting sh / 8 bytes past the 4-byte-aligned
// q; zeros for a row past the matrix.
template <int NW>
__device__ __forceinline__ void row_words(const uint8_t *q, uint32_t sh, bool valid, uint32_t (&w)[NW]) {
    const uint32_t *p = reinterpret_cast<const uint32_t *>(q);
    uint32_t prev = valid ? p[0] : 0u;
#pragma unroll
    for (int i = 0; i < NW; ++i) {
        const uint32_t next = valid ? p[i + 1] : 0u;
        w[i] = __funnelshift_r(prev, next, sh);
        prev = next;
    }
}

// Quant bytes 4g .. 4g+3 of block b of a row (2-byte aligned; base is the
// 16-byte-aligned start of the shared memory).
__device__ __forceinline__ uint32_t row_q4(const uint8_t *base, const uint8_t *row, int b, int g, bool valid) {
    if (!valid) return 0u;
    const uint32_t a = static_cast<uint32_t>(row - base) + 34u * b + 2u + 4u * g;
    const uint32_t *p = reinterpret_cast<const uint32_t *>(base + (a & ~3u));
    return __funnelshift_r(p[0], p[1], (a & 3u) * 8u);
}

// This lane's accumulators times `down`, stored (ADD false) or added to what
// is there (ADD true: own + stored) in the fragment order [b][j][lane][e < EH]
// at sw: one EH-float vector per MMA, so a warp's access covers 32 x EH
// consecutive words (no bank conflicts).
template <int NB, int EH, bool ADD>
__device__ __forceinline__ void put_sums(float *sw, int lane, const float (&acc)[NB][4][4], float down) {
    using V = typename std::conditional<EH == 4, float4, float2>::type;
    V *vp = reinterpret_cast<V *>(sw) + lane;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        V old[4];
        if (ADD) {
#pragma unroll
            for (int j = 0; j < 4; ++j) old[j] = vp[(b * 4 + j) * 32];
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float f[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) f[e] = acc[b][j][e] * down;
            V v;
            if constexpr (EH == 4) {
                v = make_float4(f[0], f[1], f[2], f[3]);
                if (ADD) v = make_float4(f[0] + old[j].x, f[1] + old[j].y, f[2] + old[j].z, f[3] + old[j].w);
            } else {
                v = make_float2(f[0], f[1]);
                if (ADD) v = make_float2(f[0] + old[j].x, f[1] + old[j].y);
            }
            vp[(b * 4 + j) * 32] = v;
        }
    }
}

template <int NB>
__global__ void __launch_bounds__(VtCfg<NB>::THREADS) qmm_t_kernel(const VtParams P) {
    using C = VtCfg<NB>;
    constexpr int K = C::K, RB = C::RB, SR = C::SR, SLOT = C::SLOT, D = C::D, FR = C::FR;
    constexpr int WARPS = C::WARPS, HALF = C::HALF, THREADS = C::THREADS;
    constexpr bool CONTIG = NB == 1 || NB == 2 || NB == 4 || NB == 8;
    constexpr int CPG = 4 * NB, NW = CPG / 4;  // columns per MMA column index, their words
    extern __shared__ __align__(16) uint8_t smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + WARPS * D * SLOT);  // [warp][D]
    int *last = reinterpret_cast<int *>(bars + WARPS * D);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.y, c = blockIdx.x;
    // this warp's rows: the w-th sixteenth of the chunk
    const int64_t n_lo = static_cast<int64_t>(c) * P.R, n_hi = min(P.N, n_lo + P.R);
    const int64_t rw = P.R / WARPS;
    const int64_t w_lo = min(n_hi, n_lo + warp * rw), w_hi = min(n_hi, w_lo + rw);
    const int nst = static_cast<int>((w_hi - w_lo + SR - 1) / SR);
    const uint64_t mat0 = reinterpret_cast<uint64_t>(P.W) + static_cast<uint64_t>(h) * P.N * RB;
    uint8_t *ring = smem + warp * D * SLOT;
    const uint32_t bar0 = smem_u32(bars + warp * D);

    if (lane == 0) {
        for (int s = 0; s < D; ++s) mbar_init(bar0 + 8u * s, 1);
        fence_mbar_init();
        // while the preceding grid finishes: warm L2 with this warp's first
        // 16 KB (L2 is the point of coherence, so this is safe even if that
        // grid writes the cache); nothing else is read, and nothing written,
        // before the wait
        const uint64_t a16 = (mat0 + static_cast<uint64_t>(w_lo) * RB) & ~uint64_t(15);
        const uint64_t b16 = min((mat0 + static_cast<uint64_t>(w_hi) * RB) & ~uint64_t(15), a16 + 16384);
        if (b16 > a16) bulk_prefetch_l2(reinterpret_cast<const void *>(a16), static_cast<uint32_t>(b16 - a16));
    }
    pdl_trigger();
    pdl_wait();
    __syncwarp();
    // issue stage t of this warp into slot t % D (lane 0): its rows rounded out
    // to 16 bytes (the bulk-copy rule); the matrices' last bytes, past the
    // final 16-byte boundary, by plain loads
    const uint64_t pol = policy_evict_first();
    auto issue = [&](int t) {
        const int s = t % D;
        const int64_t r0 = w_lo + static_cast<int64_t>(t) * SR, r1 = min(w_hi, r0 + SR);
        const uint64_t a = mat0 + static_cast<uint64_t>(r0) * RB, b = mat0 + static_cast<uint64_t>(r1) * RB;
        const uint64_t a16 = a & ~uint64_t(15);
        uint64_t b16 = (b + 15) & ~uint64_t(15);
        uint8_t *dst = ring + s * SLOT;
        if (b16 > P.w_end) {
            b16 = b & ~uint64_t(15);
            for (uint64_t i = b16; i < b; ++i) dst[i - a16] = *reinterpret_cast<const uint8_t *>(i);
        }
        const uint32_t bytes = static_cast<uint32_t>(b16 - a16);
        mbar_arrive_expect_tx(bar0 + 8u * s, bytes);
        if (bytes) bulk_g2s(smem_u32(dst), reinterpret_cast<const void *>(a16), bytes, bar0 + 8u * s, pol);
    };
    int issued = 0;
    if (lane == 0)
        for (; issued < min(D, nst); ++issued) issue(issued);

    const int g = lane >> 2, tq = lane & 3;
    // contiguous mapping: this lane's columns CPG*g .. lie in block bb of each row
    const int bb = (CPG * g) / 32;
    const uint32_t qoff = 34u * bb + 2u + static_cast<uint32_t>((CPG * g) % 32);
    const float *xh = P.x + (static_cast<int64_t>(h) * P.M + P.m0) * P.N;  // row m of this launch: xh + m*N
    const int ra = 2 * tq, rb = ra + 1, rc = ra + 8, rd = ra + 9;  // this lane's four rows of a group
    // positions are counted from w_lo from here on (32-bit): the warp's rows are [0, nw)
    const int nw = static_cast<int>(w_hi - w_lo);
    // x of rows g and g + 8 at position ra of the warp's first group; rows
    // g + 8 exist only when this launch has more than 8 rows of x
    const float *xp0 = xh + static_cast<int64_t>(g) * P.N + w_lo + ra;
    const float *xp1 = xp0 + 8 * P.N;
    const bool vm0 = g < P.mg, vm1 = g + 8 < P.mg, two = P.mg > 8;
    // x of this lane's four positions of the group at o (ra, rb, rc, rd), rows
    // g and g + 8 (zero past the warp's rows or past this launch's rows of x)
    auto load_x = [&](int o, float (&v)[2][4]) {
        const float *p0 = xp0 + o, *p1 = xp1 + o;
        if (o + 16 <= nw) {
            v[0][0] = vm0 ? __ldg(p0) : 0.0f;
            v[0][1] = vm0 ? __ldg(p0 + 1) : 0.0f;
            v[0][2] = vm0 ? __ldg(p0 + 8) : 0.0f;
            v[0][3] = vm0 ? __ldg(p0 + 9) : 0.0f;
            if (two) {
                v[1][0] = vm1 ? __ldg(p1) : 0.0f;
                v[1][1] = vm1 ? __ldg(p1 + 1) : 0.0f;
                v[1][2] = vm1 ? __ldg(p1 + 8) : 0.0f;
                v[1][3] = vm1 ? __ldg(p1 + 9) : 0.0f;
            }
        } else {
            const int n = nw - o;  // positions left in the group
            v[0][0] = vm0 && ra < n ? __ldg(p0) : 0.0f;
            v[0][1] = vm0 && rb < n ? __ldg(p0 + 1) : 0.0f;
            v[0][2] = vm0 && rc < n ? __ldg(p0 + 8) : 0.0f;
            v[0][3] = vm0 && rd < n ? __ldg(p0 + 9) : 0.0f;
            if (two) {
                v[1][0] = vm1 && ra < n ? __ldg(p1) : 0.0f;
                v[1][1] = vm1 && rb < n ? __ldg(p1 + 1) : 0.0f;
                v[1][2] = vm1 && rc < n ? __ldg(p1 + 8) : 0.0f;
                v[1][3] = vm1 && rd < n ? __ldg(p1 + 9) : 0.0f;
            }
        }
    };

    float acc[NB][4][4];
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[b][j][e] = 0.0f;
    int ew = 12;           // biased exponent of the warp's running max |x| (at least 12)
    float up = 0x1p127f;   // 2^(139 - ew): that max times up lies in [2^12, 2^13)

    // one group of 16 positions whose rows start at `rows` in shared memory;
    // nv of them are the warp's (16 for every group but perhaps the last)
    auto contract = [&](const float (&xc)[2][4], const uint8_t *rows, int nv) {
        const bool va = ra < nv, vb = rb < nv, vc = rc < nv, vd = rd < nv;
        // A: x * up of positions ra, rb (a0, a1) and rc, rd (a2, a3); rows g, g + 8
        const uint32_t a0 = pack_half2(xc[0][0] * up, xc[0][1] * up), a2 = pack_half2(xc[0][2] * up, xc[0][3] * up);
        const uint32_t a1 = two ? pack_half2(xc[1][0] * up, xc[1][1] * up) : 0u;
        const uint32_t a3 = two ? pack_half2(xc[1][2] * up, xc[1][3] * up) : 0u;
        const uint8_t *row_a = rows + ra * RB, *row_b = rows + rb * RB, *row_c = rows + rc * RB,
                      *row_dd = rows + rd * RB;
        if constexpr (CONTIG) {
            // CPG contiguous quant bytes of block bb per row, one d per row:
            // from the 4-byte word at or below them, shifted by their offset
            // in it (the same for every row when RB is a multiple of 4, since
            // the stage then starts on a 4-byte boundary too)
            uint32_t wa[NW], wb[NW], wc[NW], wd[NW];
            if constexpr (RB % 4 == 0) {
                const uint32_t sh = (qoff & 3u) * 8u, q4 = qoff & ~3u;
                row_words(row_a + q4, sh, va, wa);
                row_words(row_b + q4, sh, vb, wb);
                row_words(row_c + q4, sh, vc, wc);
                row_words(row_dd + q4, sh, vd, wd);
            } else {
                auto at = [&](const uint8_t *row) { return static_cast<uint32_t>(row - smem) + qoff; };
                row_words(smem + (at(row_a) & ~3u), (at(row_a) & 3u) * 8u, va, wa);
                row_words(smem + (at(row_b) & ~3u), (at(row_b) & 3u) * 8u, vb, wb);
                row_words(smem + (at(row_c) & ~3u), (at(row_c) & 3u) * 8u, vc, wc);
                row_words(smem + (at(row_dd) & ~3u), (at(row_dd) & 3u) * 8u, vd, wd);
            }
            const uint32_t dab = row_d(row_a, bb, va) | (row_d(row_b, bb, vb) << 16);
            const uint32_t dcd = row_d(row_c, bb, vc) | (row_d(row_dd, bb, vd) << 16);
            const __half2 d01 = *reinterpret_cast<const __half2 *>(&dab);
            const __half2 d89 = *reinterpret_cast<const __half2 *>(&dcd);
#pragma unroll
            for (int j = 0; j < CPG; ++j)
                mma16816(acc[j >> 2][j & 3], a0, a1, a2, a3, b_pair(wa[j >> 2], wb[j >> 2], j & 3, d01),
                         b_pair(wc[j >> 2], wd[j >> 2], j & 3, d89));
        } else {
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const uint32_t wa = row_q4(smem, row_a, b, g, va), wb = row_q4(smem, row_b, b, g, vb);
                const uint32_t wc = row_q4(smem, row_c, b, g, vc), wd = row_q4(smem, row_dd, b, g, vd);
                const uint32_t dab = row_d(row_a, b, va) | (row_d(row_b, b, vb) << 16);
                const uint32_t dcd = row_d(row_c, b, vc) | (row_d(row_dd, b, vd) << 16);
                const __half2 d01 = *reinterpret_cast<const __half2 *>(&dab);
                const __half2 d89 = *reinterpret_cast<const __half2 *>(&dcd);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    mma16816(acc[b][j], a0, a1, a2, a3, b_pair(wa, wb, j, d01), b_pair(wc, wd, j, d89));
            }
        }
    };

    float xn[2][4] = {};  // x of the next group, in flight while the current one is contracted
    load_x(0, xn);
    bool ok = true;
    for (int t = 0; t < nst && ok; ++t) {
        const int s = t % D;
        // an expired wait leaves this chunk's sum incomplete (the status word
        // reports it); the CTA still takes part in the reduction
        ok = __all_sync(0xffffffffu, mbar_wait(bar0 + 8u * s, (t / D) & 1, P.status));
        if (!ok) break;
        const uint64_t a = mat0 + static_cast<uint64_t>(w_lo + static_cast<int64_t>(t) * SR) * RB;
        const uint8_t *stage = ring + s * SLOT + (a & 15);
#pragma unroll 1
        for (int gi = 0; gi < SR / 16; ++gi) {
            const int o = t * SR + 16 * gi;  // these 16 positions
            if (o >= nw) break;
            float xc[2][4];
#pragma unroll
            for (int hm = 0; hm < 2; ++hm)
#pragma unroll
                for (int e = 0; e < 4; ++e) xc[hm][e] = xn[hm][e];
            if (o + 16 < nw) load_x(o + 16, xn);
            // the running scale: the warp's max |x| so far
            float mloc = 0.0f;
#pragma unroll
            for (int hm = 0; hm < 2; ++hm)
#pragma unroll
                for (int e = 0; e < 4; ++e) mloc = fmaxf(mloc, fabsf(xc[hm][e]));
            const uint32_t mbits = __reduce_max_sync(0xffffffffu, __float_as_uint(mloc));
            const int eg = min(254, static_cast<int>(mbits >> 23));
            if (eg > ew) {
                const float f = pow2_biased(127 + ew - eg);  // exact: a power of two, or 0 far below
#pragma unroll
                for (int b = 0; b < NB; ++b)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[b][j][e] *= f;
                ew = eg;
                up = pow2_biased(266 - ew);
            }
            const uint8_t *rows = stage + 16 * gi * RB;
            if (o + 16 <= nw) contract(xc, rows, 16);  // a full group: no per-row checks
            else contract(xc, rows, nw - o);
        }
        __syncwarp();
        if (lane == 0 && issued < nst) {
            // the slot just read is refilled: order the reads before the async write
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(issued);
            ++issued;
        }
    }
    // no copy into this warp's ring may be in flight when its slots are reused
    if (lane == 0)
        for (int t = issued > D ? issued - D : 0; t < issued; ++t) mbar_wait(bar0 + 8u * (t % D), (t / D) & 1, P.status);
    // back to the true scale: 1 / up = 2^(ew - 139) (exact)
    const float down = ew > 12 ? pow2_biased(ew - 12) : 0x1p-127f;
    // every warp's ring is drained: the rings now hold the pair sums in the
    // MMA fragments' own order, [warp % HALF][b][j][lane][e < EH]: the upper
    // half of the warps store theirs, then the lower half add their own.
    // Elements e = 2, 3 (rows g + 8) are kept only when this launch has more
    // than 8 rows of x.
    __syncthreads();
    float *sums = reinterpret_cast<float *>(smem);
    const int EH = P.mg > 8 ? 4 : 2;
    if (warp >= HALF) {
        if (EH == 4) put_sums<NB, 4, false>(sums + (warp - HALF) * FR, lane, acc, down);
        else put_sums<NB, 2, false>(sums + (warp - HALF) * FR, lane, acc, down);
    }
    __syncthreads();
    if (warp < HALF) {
        if (EH == 4) put_sums<NB, 4, true>(sums + warp * FR, lane, acc, down);
        else put_sums<NB, 2, true>(sums + warp * FR, lane, acc, down);
    }
    __syncthreads();
    // the chunk sum into the workspace, in the same fragment order (coalesced)
    const int nf = FR / 4 * EH;
    float *part_hc = P.part + (static_cast<int64_t>(h) * P.nchunk + c) * FR;
    for (int i = threadIdx.x; i < nf; i += THREADS) {
        float v[HALF];
#pragma unroll
        for (int w = 0; w < HALF; ++w) v[w] = sums[w * FR + i];
        float sum = v[0];
#pragma unroll
        for (int w = 1; w < HALF; ++w) sum += v[w];  // in warp order
        part_hc[i] = sum;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned done = atomicAdd(P.count + h, 1u);
        *last = done == static_cast<unsigned>(P.nchunk - 1);
    }
    __syncthreads();
    if (!*last) return;
    // the last CTA of matrix h: chunk sums in chunk order, two fragment words
    // per thread and 24 chunks in flight at a time; fragment word i is element
    // e = i % EH of lane (g, tq) = (((i / EH) % 32) / 4, (i / EH) % 4) in MMA
    // (b, j) = (i / (128 EH), (i / (32 EH)) % 4): row g + 8 (e / 2) and, for odd e, the
    // second of the lane's two columns (with the contiguous mapping MMA 4b + j
    // gives the lane columns CPG*2tq + 4b + j and CPG*(2tq+1) + 4b + j, else
    // 32b + 8tq + j and 32b + 8tq + j + 4)
    __threadfence();
    const float *part_h = P.part + static_cast<int64_t>(h) * P.nchunk * FR;
    float *yh = P.y + (static_cast<int64_t>(h) * P.M + P.m0) * K;
    auto put = [&](int i, float v) {
        const int e = i % EH, ln = (i / EH) & 31, bj = i / (32 * EH), j = bj & 3, b = bj >> 2;
        const int m = (ln >> 2) + 8 * (e >> 1), t = ln & 3;
        const int k0 = CONTIG ? CPG * 2 * t + 4 * b + j : 32 * b + 8 * t + j;
        if (m < P.mg) yh[m * K + ((e & 1) ? k0 + (CONTIG ? CPG : 4) : k0)] = v;
    };
    for (int i0 = threadIdx.x; i0 < nf; i0 += 2 * THREADS) {
        const int i1 = i0 + THREADS;
        const bool two = i1 < nf;
        float s0 = 0.0f, s1 = 0.0f;
        for (int c0 = 0; c0 < P.nchunk; c0 += 24) {
            float v0[24], v1[24];
#pragma unroll
            for (int u = 0; u < 24; ++u) {
                const bool ok = c0 + u < P.nchunk;
                const float *pc = part_h + static_cast<int64_t>(c0 + u) * FR;
                v0[u] = ok ? __ldcg(pc + i0) : 0.0f;
                v1[u] = ok && two ? __ldcg(pc + i1) : 0.0f;
            }
#pragma unroll
            for (int u = 0; u < 24; ++u)
                if (c0 + u < P.nchunk) {
                    s0 += v0[u];
                    s1 += v1[u];
                }
        }
        put(i0, s0);
        if (two) put(i1, s1);
    }
    if (threadIdx.x == 0) P.count[h] = 0u;  // ready for the next call on this stream
}

// Programmatic dependent launch: the CTAs start (and warm L2 with their rows)
// as SMs free up at the end of the preceding grid, then wait for it.
template <int NB>
cudaError_t launch_nb(const VtParams &P, int64_t H, cudaStream_t st) {
    const int smem = VtCfg<NB>::SMEM;
    cudaError_t e = set_smem_attrs(qmm_t_kernel<NB>, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(P.nchunk, static_cast<unsigned>(H));
    cfg.blockDim = dim3(VtCfg<NB>::THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, qmm_t_kernel<NB>, P);
}

}  // namespace

int64_t qmm_t_chunk_rows(int64_t H, int64_t N, int64_t K, int num_sms) {
    // one CTA per SM over all matrices (the rings fill most of an SM's shared
    // memory, so one CTA is resident per SM), each chunk split evenly between
    // the warps (a warp's last 16-row group may be partly empty)
    const int64_t want = static_cast<int64_t>(num_sms);
    const int64_t w = vt_warps(static_cast<int>(K / 32));
    int64_t per = want / H;  // chunks per matrix: all CTAs in one wave
    if (per < 1) per = 1;
    int64_t R = (N + per - 1) / per;
    R = (R + w - 1) / w * w;
    return R < w ? w : R;
}

size_t qmm_t_part_bytes(int64_t H, int64_t N, int64_t K, int num_sms) {
    const int64_t R = qmm_t_chunk_rows(H, N, K, num_sms);
    const int64_t nchunk = (N + R - 1) / R;
    return static_cast<size_t>(H * nchunk * 16 * K) * sizeof(float);
}

cudaError_t launch_qmm_t(const void *W, int64_t H, int64_t N, int64_t K, const float *x, int64_t M, float *y,
                         float *part, unsigned *count, cudaStream_t st, int num_sms, int *status) {
    VtParams P;
    P.W = static_cast<const uint8_t *>(W);
    P.N = N;
    P.w_end = reinterpret_cast<uint64_t>(W) + static_cast<uint64_t>(H * N) * (K / 32) * 34;
    P.R = qmm_t_chunk_rows(H, N, K, num_sms);
    P.nchunk = static_cast<int>((N + P.R - 1) / P.R);
    P.x = x;
    P.M = M;
    P.y = y;
    P.part = part;
    P.count = count;
    P.status = status;
    const int nb = static_cast<int>(K / 32);
    for (int64_t m0 = 0; m0 < M; m0 += VT_MG) {
        P.m0 = static_cast<int>(m0);
        P.mg = static_cast<int>(min(static_cast<int64_t>(VT_MG), M - m0));
        cudaError_t e;
        switch (nb) {
        case 1: e = launch_nb<1>(P, H, st); break;
        case 2: e = launch_nb<2>(P, H, st); break;
        case 3: e = launch_nb<3>(P, H, st); break;
        case 4: e = launch_nb<4>(P, H, st); break;
        case 5: e = launch_nb<5>(P, H, st); break;
        case 6: e = launch_nb<6>(P, H, st); break;
        case 7: e = launch_nb<7>(P, H, st); break;
        default: e = launch_nb<8>(P, H, st); break;
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace qk
