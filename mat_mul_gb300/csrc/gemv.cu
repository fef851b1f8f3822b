// gemv.cu -- the memory-bound decode product y[M,N] = W[N,K] . x[M,K]^T for
// M <= 8 (the GEMV bucket of infr's per-op profile; M > 1 is its concurrent
// generation slots, "--parallel N").
//
// Design (sm_103a):
//   * One CTA per SM, each owning a contiguous range of whole output rows, so
//     every y element is produced by exactly one CTA with a fixed summation
//     order (deterministic, no atomics, no zero-fill).
//   * One producer thread streams the CTA's weight bytes through a ring of
//     shared-memory stages with 1-D bulk async copies (cp.async.bulk) that
//     complete on mbarriers; tens of KB per SM are in flight, independent of
//     how the consumers map lanes to data.  Row starts of Q6_K/Q8_0 matrices
//     are not 16-byte aligned, so a stage is copied from its start rounded
//     down to 16 bytes and the consumers index from the remainder.
//   * The quantised activations (produced by the quantiser kernel launched
//     just before, with programmatic dependent launch so that this kernel's
//     weight stream starts while the quantiser runs) are bulk-copied into
//     shared memory once per CTA.
//   * Eight consumer warps.  The weight stream is cut into "rounds" of 32
//     units, a unit being one lane's share of a block (Q4_K: one 32-weight
//     sub-block; Q6_K: 64 weights = 16 positions x 4 groups; Q8_0: one block).
//     A round never crosses a row, so a warp reduces a round with shuffles and
//     one lane parks the total in shared memory; after each stage warp 0 adds
//     the round totals of every row in order and stores the finished rows.
//   * Dot products are exact int32 dp4a over a block; the fp32 scale and min
//     terms are applied per block, as in the oracle's arithmetic.
#include "qmm_device.cuh"

namespace qk {

namespace {

constexpr int NW = 8;             // consumer warps
constexpr int NTHREADS = (NW + 1) * 32;
constexpr int SLOT_SLACK = 64;    // alignment head + over-read of the word helpers

template <int T> struct Units;
template <> struct Units<QMM_Q8_0> { static constexpr int UPB = 1; };
template <> struct Units<QMM_Q4_K> { static constexpr int UPB = 8; };
template <> struct Units<QMM_Q6_K> { static constexpr int UPB = 4; };

struct GemvParams {
    const uint8_t *W;
    int64_t total_bytes;  // N * row_bytes
    int64_t N;
    int K, M;
    int RB;    // bytes per row
    int UPR;   // units per row
    int RPR;   // rounds per row
    int NR;    // rounds per stage
    int NS;    // stages in the ring
    int slot_bytes;
    const int8_t *xq;  // [M][K]
    const float *xd;   // [M][xd_ld]
    const int32_t *xs; // [M][xd_ld]
    int xd_ld;
    float *y;  // [M][N]
    // shared-memory layout (byte offsets from the dynamic base)
    int off_rt, off_xq, off_xd, off_xs, off_ring;
    int pdl;
    int *status;  // device status word (bounded-wait timeouts)
};

// Byte range [round_begin, round_end) of local round R of a CTA whose first
// row is r0.
template <int T>
__device__ __forceinline__ int64_t round_begin(const GemvParams &P, int64_t r0, int64_t R) {
    constexpr int UPB = Units<T>::UPB, BB = Fmt<T>::BB;
    const int64_t row = R / P.RPR;
    const int rr = static_cast<int>(R - row * P.RPR);
    return (r0 + row) * P.RB + static_cast<int64_t>(32 * rr / UPB) * BB;
}

template <int T>
__device__ __forceinline__ int64_t round_end(const GemvParams &P, int64_t r0, int64_t R) {
    constexpr int UPB = Units<T>::UPB, BB = Fmt<T>::BB;
    const int64_t row = R / P.RPR;
    const int rr = static_cast<int>(R - row * P.RPR);
    const int ue = min(32 * (rr + 1), P.UPR);
    return (r0 + row) * P.RB + static_cast<int64_t>(ue / UPB) * BB;
}

// --------------------------------------------------------------------------
// Per-unit dot products.  `blk` is the shared address of the unit's block,
// `kb` the block index within its row; acc[m] gains the unit's fp32 share.
// --------------------------------------------------------------------------

template <int MT>
__device__ __forceinline__ void unit_q4k(uint32_t blk, int kb, int j, const GemvParams &P,
                                         uint32_t sxq, uint32_t sxd, uint32_t sxs, float (&acc)[MT]) {
    // Sub-block j (32 weights): nibbles of qs[32c .. 32c+31], c = j/2, low
    // nibble for even j, high for odd j.
    const uint4 hdr = lds128(blk);
    const int c = j >> 1;
    uint4 qa = lds128(blk + 16 + 32 * c);
    uint4 qb = lds128(blk + 32 + 32 * c);
    const uint32_t sh = (j & 1) * 4;
    uint32_t w[8] = {(qa.x >> sh) & 0x0F0F0F0Fu, (qa.y >> sh) & 0x0F0F0F0Fu,
                     (qa.z >> sh) & 0x0F0F0F0Fu, (qa.w >> sh) & 0x0F0F0F0Fu,
                     (qb.x >> sh) & 0x0F0F0F0Fu, (qb.y >> sh) & 0x0F0F0F0Fu,
                     (qb.z >> sh) & 0x0F0F0F0Fu, (qb.w >> sh) & 0x0F0F0F0Fu};
    // six-bit scale and min of sub-block j
    uint32_t scw, mw;
    if (j < 4) {
        scw = hdr.y & 0x3F3F3F3Fu;
        mw = hdr.z & 0x3F3F3F3Fu;
    } else {
        scw = (hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u);
        mw = ((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u);
    }
    const int bsh = (j & 3) * 8;
    const int sc = (scw >> bsh) & 0xFF, mn = (mw >> bsh) & 0xFF;
    const float d = half_bits_to_float(hdr.x), dmin = half_bits_to_float(hdr.x >> 16);
    // The two 16-byte activation pieces are read in an order rotated by
    // (j >> 2) so the eight lanes of a quarter warp hit distinct banks.
    const int rot = (j >> 2) & 1;
    uint32_t wf[4], ws[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        wf[i] = rot ? w[4 + i] : w[i];
        ws[i] = rot ? w[i] : w[4 + i];
    }
    const int b32 = kb * 8 + j;
    const uint32_t xoff = static_cast<uint32_t>(kb * 256 + 32 * j);
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        const uint32_t xr = sxq + static_cast<uint32_t>(m * P.K) + xoff;
        const uint4 xf = lds128(xr + 16 * rot);
        const uint4 xs2 = lds128(xr + 16 * (1 - rot));
        int I = __dp4a(static_cast<int>(wf[0]), static_cast<int>(xf.x), 0);
        I = __dp4a(static_cast<int>(wf[1]), static_cast<int>(xf.y), I);
        I = __dp4a(static_cast<int>(wf[2]), static_cast<int>(xf.z), I);
        I = __dp4a(static_cast<int>(wf[3]), static_cast<int>(xf.w), I);
        I = __dp4a(static_cast<int>(ws[0]), static_cast<int>(xs2.x), I);
        I = __dp4a(static_cast<int>(ws[1]), static_cast<int>(xs2.y), I);
        I = __dp4a(static_cast<int>(ws[2]), static_cast<int>(xs2.z), I);
        I = __dp4a(static_cast<int>(ws[3]), static_cast<int>(xs2.w), I);
        const uint32_t di = static_cast<uint32_t>((m * P.xd_ld + b32) * 4);
        const float dx = ldsf(sxd + di);
        const int sx = static_cast<int>(lds32(sxs + di));
        acc[m] += dx * (d * static_cast<float>(sc * I) - dmin * static_cast<float>(mn * sx));
    }
}

template <int MT>
__device__ __forceinline__ void unit_q6k(uint32_t blk, int kb, int u, int lane,
                                         const GemvParams &P, uint32_t sxq, uint32_t sxd,
                                         float (&acc)[MT]) {
    // Unit u = 2h + t: half h, positions l = 16t .. 16t+15 of each of the four
    // 32-weight groups g of the half; group g uses scale 8h + 2g + t and the
    // activations at 128h + 32g + 16t.
    const int h = u >> 1, t = u & 1;
    uint32_t qla[4], qlb[4], qhw[4], scw[2];
    lds_words_u16aligned<4>(blk + 64 * h + 16 * t, qla);
    lds_words_u16aligned<4>(blk + 64 * h + 32 + 16 * t, qlb);
    lds_words_u16aligned<4>(blk + 128 + 32 * h + 16 * t, qhw);
    lds_words_u16aligned<2>(blk + 192 + 8 * h + t, scw);  // bytes s, s+2, s+4, s+6 used
    const float d = half_bits_to_float(lds16(blk + 208));
    // Groups are visited in an order rotated by (block parity, h) so the
    // activation reads of a quarter warp fall in distinct banks.
    const int rot = ((lane >> 2) & 1) * 2 + h;
    int sc[4];
    uint32_t q[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int g = (i + rot) & 3;
        const uint32_t sel = (g < 2) ? scw[0] : scw[1];
        sc[i] = static_cast<int>(static_cast<int8_t>((sel >> ((g & 1) * 16)) & 0xFF));
        const uint32_t lsh = (g >= 2) ? 4u : 0u;
        const uint32_t hsh = 2u * static_cast<uint32_t>(g);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint32_t lo = (((g & 1) ? qlb[e] : qla[e]) >> lsh) & 0x0F0F0F0Fu;
            const uint32_t hi = ((qhw[e] >> hsh) << 4) & 0x30303030u;
            // (lo|hi) in 0..63 per byte; +96 then flipping bit 7 yields q-32 as int8
            q[i][e] = ((lo | hi) + 0x60606060u) ^ 0x80808080u;
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        float part = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int g = (i + rot) & 3;
            const uint4 xv = lds128(sxq + static_cast<uint32_t>(m * P.K + kb * 256 + 128 * h + 32 * g + 16 * t));
            int I = __dp4a(static_cast<int>(q[i][0]), static_cast<int>(xv.x), 0);
            I = __dp4a(static_cast<int>(q[i][1]), static_cast<int>(xv.y), I);
            I = __dp4a(static_cast<int>(q[i][2]), static_cast<int>(xv.z), I);
            I = __dp4a(static_cast<int>(q[i][3]), static_cast<int>(xv.w), I);
            const float dx = ldsf(sxd + static_cast<uint32_t>((m * P.xd_ld + kb * 8 + 4 * h + g) * 4));
            part += dx * static_cast<float>(sc[i] * I);
        }
        acc[m] += d * part;
    }
}

template <int MT>
__device__ __forceinline__ void unit_q80(uint32_t blk, int kb, int lane, const GemvParams &P,
                                         uint32_t sxq, uint32_t sxd, float (&acc)[MT]) {
    uint32_t qw[8];
    lds_words_u16aligned<8>(blk + 2, qw);
    const float d = half_bits_to_float(lds16(blk));
    const int rot = (lane >> 2) & 1;
    uint32_t wf[4], ws[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        wf[i] = rot ? qw[4 + i] : qw[i];
        ws[i] = rot ? qw[i] : qw[4 + i];
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        const uint32_t xr = sxq + static_cast<uint32_t>(m * P.K + kb * 32);
        const uint4 xf = lds128(xr + 16 * rot);
        const uint4 xs2 = lds128(xr + 16 * (1 - rot));
        int I = __dp4a(static_cast<int>(wf[0]), static_cast<int>(xf.x), 0);
        I = __dp4a(static_cast<int>(wf[1]), static_cast<int>(xf.y), I);
        I = __dp4a(static_cast<int>(wf[2]), static_cast<int>(xf.z), I);
        I = __dp4a(static_cast<int>(wf[3]), static_cast<int>(xf.w), I);
        I = __dp4a(static_cast<int>(ws[0]), static_cast<int>(xs2.x), I);
        I = __dp4a(static_cast<int>(ws[1]), static_cast<int>(xs2.y), I);
        I = __dp4a(static_cast<int>(ws[2]), static_cast<int>(xs2.z), I);
        I = __dp4a(static_cast<int>(ws[3]), static_cast<int>(xs2.w), I);
        const float dx = ldsf(sxd + static_cast<uint32_t>((m * P.xd_ld + kb) * 4));
        acc[m] += dx * (d * static_cast<float>(I));
    }
}

// --------------------------------------------------------------------------
// The kernel.
// --------------------------------------------------------------------------
template <int T, int MT>
__global__ void __launch_bounds__(NTHREADS, 1) gemv_kernel(const __grid_constant__ GemvParams P) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int UPB = Units<T>::UPB, BB = Fmt<T>::BB;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // rows of this CTA
    const int64_t r0 = (P.N * blockIdx.x) / gridDim.x;
    const int64_t r1 = (P.N * (blockIdx.x + 1)) / gridDim.x;
    const int64_t nrounds = (r1 - r0) * P.RPR;
    const int64_t nstages = (nrounds + P.NR - 1) / P.NR;

    // barriers: full[NS], empty[NS], xbar; then carry[MT] and the abort flag
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    const uint32_t bar_full = smem_u32(bars);
    const uint32_t bar_empty = bar_full + 8u * P.NS;
    const uint32_t bar_x = bar_empty + 8u * P.NS;
    float *carry = reinterpret_cast<float *>(smem + 8 * (2 * P.NS + 1));  // < 256 bytes in all
    float *rt = reinterpret_cast<float *>(smem + P.off_rt);
    const uint32_t sxq = smem_u32(smem + P.off_xq);
    const uint32_t sxd = smem_u32(smem + P.off_xd);
    const uint32_t sxs = smem_u32(smem + P.off_xs);
    const uint32_t sring = smem_u32(smem + P.off_ring);

    if (threadIdx.x == 0) {
        for (int i = 0; i < P.NS; ++i) {
            mbar_init(bar_full + 8u * i, 1);
            mbar_init(bar_empty + 8u * i, 1);
        }
        mbar_init(bar_x, 1);
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == NW) {
        // ------------------------------------------------------- producer
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_x = policy_evict_last();
            bool x_issued = false;
            int64_t issued = 0;
            for (int64_t s = 0; s < nstages; ++s) {
                const int slot = static_cast<int>(s % P.NS);
                if (s >= P.NS) {
                    const uint32_t par = static_cast<uint32_t>(((s / P.NS) - 1) & 1);
                    if (!mbar_wait(bar_empty + 8u * slot, par, P.status)) break;
                }
                const int64_t R0 = s * P.NR;
                const int64_t R1 = min(R0 + P.NR, nrounds);
                const int64_t a = round_begin<T>(P, r0, R0);
                const int64_t b = round_end<T>(P, r0, R1 - 1);
                const int64_t a16 = a & ~int64_t(15);
                int64_t b16 = (b + 15) & ~int64_t(15);
                const uint32_t dst = sring + static_cast<uint32_t>(slot) * P.slot_bytes;
                if (b16 > P.total_bytes) {
                    // the last bytes of the matrix: plain loads for the tail
                    b16 = b & ~int64_t(15);
                    for (int64_t i = b16; i < b; ++i) {
                        const uint8_t v = P.W[i];
                        asm volatile("st.shared.u8 [%0], %1;" ::"r"(dst + static_cast<uint32_t>(i - a16)),
                                     "h"(static_cast<unsigned short>(v)));
                    }
                }
                const uint32_t nbytes = static_cast<uint32_t>(b16 - a16);
                mbar_arrive_expect_tx(bar_full + 8u * slot, nbytes);
                if (nbytes) bulk_g2s(dst, P.W + a16, nbytes, bar_full + 8u * slot, pol_w);
                ++issued;
                if (!x_issued && (s + 1 == P.NS || s + 1 == nstages)) {
                    if (P.pdl) pdl_wait();
                    const uint32_t nq = static_cast<uint32_t>(P.M * P.K);
                    const uint32_t nd = static_cast<uint32_t>(P.M * P.xd_ld * 4);
                    mbar_arrive_expect_tx(bar_x, nq + 2 * nd);
                    bulk_g2s(sxq, P.xq, nq, bar_x, pol_x);
                    bulk_g2s(sxd, P.xd, nd, bar_x, pol_x);
                    bulk_g2s(sxs, P.xs, nd, bar_x, pol_x);
                    x_issued = true;
                }
            }
            if (!x_issued) {
                // no weight stage at all (empty row range): still arm the
                // activation barrier so nobody waits on it
                mbar_arrive(bar_x);
            }
            // drain: every copy issued must have landed before the CTA exits
            for (int64_t s = (issued > P.NS ? issued - P.NS : 0); s < issued; ++s) {
                const int slot = static_cast<int>(s % P.NS);
                mbar_wait(bar_full + 8u * slot, static_cast<uint32_t>((s / P.NS) & 1), P.status);
            }
            if (x_issued) mbar_wait(bar_x, 0, P.status);
        }
        return;
    }

    // ----------------------------------------------------------- consumers
    bool failed = false;
    if (nstages > 0) failed = !mbar_wait(bar_x, 0, P.status);
    for (int64_t s = 0; s < nstages; ++s) {
        const int slot = static_cast<int>(s % P.NS);
        const int64_t R0 = s * P.NR;
        const int64_t R1 = min(R0 + P.NR, nrounds);
        if (!failed) failed = !mbar_wait(bar_full + 8u * slot, static_cast<uint32_t>((s / P.NS) & 1), P.status);
        float *rts = rt + static_cast<int64_t>(slot) * P.NR * MT;
        if (!failed) {
            const int64_t a16 = round_begin<T>(P, r0, R0) & ~int64_t(15);
            const uint32_t base = sring + static_cast<uint32_t>(slot) * P.slot_bytes;
            for (int j = warp; j < static_cast<int>(R1 - R0); j += NW) {
                const int64_t R = R0 + j;
                const int64_t row = R / P.RPR;
                const int rr = static_cast<int>(R - row * P.RPR);
                const int nu = min(32, P.UPR - 32 * rr);
                float acc[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m) acc[m] = 0.0f;
                if (lane < nu) {
                    const int ur = 32 * rr + lane;
                    const int kb = ur / UPB, su = ur - kb * UPB;
                    const uint32_t blk = base + static_cast<uint32_t>(
                        (r0 + row) * P.RB + static_cast<int64_t>(kb) * BB - a16);
                    if constexpr (T == QMM_Q4_K) unit_q4k<MT>(blk, kb, su, P, sxq, sxd, sxs, acc);
                    else if constexpr (T == QMM_Q6_K) unit_q6k<MT>(blk, kb, su, lane, P, sxq, sxd, acc);
                    else unit_q80<MT>(blk, kb, lane, P, sxq, sxd, acc);
                }
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    float v = acc[m];
                    v += __shfl_xor_sync(0xffffffffu, v, 16);
                    v += __shfl_xor_sync(0xffffffffu, v, 8);
                    v += __shfl_xor_sync(0xffffffffu, v, 4);
                    v += __shfl_xor_sync(0xffffffffu, v, 2);
                    v += __shfl_xor_sync(0xffffffffu, v, 1);
                    if (lane == m) rts[j * MT + m] = v;
                }
            }
        }
        // every consumer takes the same decision: stop if any of them failed
        if (named_barrier_or(1, NW * 32, failed)) break;
        if (warp == 0) {
            // finish the rows of this stage in round order
            const int64_t row_first = R0 / P.RPR, row_last = (R1 - 1) / P.RPR;
            float cin[MT];
#pragma unroll
            for (int m = 0; m < MT; ++m) cin[m] = carry[m];
            __syncwarp();
            for (int64_t k = row_first + lane; k <= row_last; k += 32) {
                const int64_t jb = max(R0, k * P.RPR) - R0;
                const int64_t je = min(R1, (k + 1) * P.RPR) - R0;
                float tot[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m) tot[m] = (k * P.RPR < R0) ? cin[m] : 0.0f;
                for (int64_t j = jb; j < je; ++j) {
#pragma unroll
                    for (int m = 0; m < MT; ++m) tot[m] += rts[j * MT + m];
                }
                if ((k + 1) * P.RPR <= R1) {
#pragma unroll
                    for (int m = 0; m < MT; ++m)
                        if (m < P.M) P.y[static_cast<int64_t>(m) * P.N + r0 + k] = tot[m];
                } else {
#pragma unroll
                    for (int m = 0; m < MT; ++m) carry[m] = tot[m];
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8u * slot);
        }
    }
}

template <int T, int MT>
cudaError_t launch_t(const GemvParams &P, int grid, int smem, cudaStream_t st) {
    auto kfn = gemv_kernel<T, MT>;
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = P.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kfn, P);
}

template <int T>
cudaError_t launch_m(const GemvParams &P, int MT, int grid, int smem, cudaStream_t st) {
    switch (MT) {
    case 1: return launch_t<T, 1>(P, grid, smem, st);
    case 2: return launch_t<T, 2>(P, grid, smem, st);
    case 4: return launch_t<T, 4>(P, grid, smem, st);
    default: return launch_t<T, 8>(P, grid, smem, st);
    }
}

}  // namespace

// Plan the shared-memory layout for a shape: stage size (rounds per stage, a
// multiple of the consumer-warp count, ~20 KB), ring depth (2..8 stages) and
// the offsets of every region.  Returns false when the activations of M rows
// do not leave room for a two-stage ring.
static bool plan_gemv(int type, int M, int K, int xd_ld, int max_smem, GemvParams &P, int &smem) {
    const int BB = block_bytes(type);
    const int UPB = type == QMM_Q8_0 ? 1 : type == QMM_Q4_K ? 8 : 4;
    const int round_bytes = (32 / UPB) * BB;
    const int MT = M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8;
    auto align = [](int64_t v, int64_t a) { return (v + a - 1) / a * a; };
    const int64_t xq_bytes = align(static_cast<int64_t>(MT) * K, 16);
    const int64_t xd_bytes = align(static_cast<int64_t>(MT) * xd_ld * 4, 16);
    int nr = NW * ((20480 + NW * round_bytes / 2) / (NW * round_bytes));
    if (nr < NW) nr = NW;
    for (; nr >= NW; nr -= NW) {
        const int64_t slot = align(static_cast<int64_t>(nr) * round_bytes + SLOT_SLACK, 128);
        for (int ns = 8; ns >= 2; --ns) {
            int64_t off = 256;  // mbarriers (2 * 8 + 1) and the carry
            const int64_t o_rt = off;
            off = align(off + static_cast<int64_t>(ns) * nr * MT * 4, 128);
            const int64_t o_xq = off;
            off = align(off + xq_bytes, 128);
            const int64_t o_xd = off;
            off = align(off + xd_bytes, 128);
            const int64_t o_xs = off;
            off = align(off + xd_bytes, 128);
            const int64_t o_ring = off;
            off += ns * slot;
            if (off <= max_smem) {
                P.NR = nr;
                P.NS = ns;
                P.slot_bytes = static_cast<int>(slot);
                P.off_rt = static_cast<int>(o_rt);
                P.off_xq = static_cast<int>(o_xq);
                P.off_xd = static_cast<int>(o_xd);
                P.off_xs = static_cast<int>(o_xs);
                P.off_ring = static_cast<int>(o_ring);
                smem = static_cast<int>(off);
                return true;
            }
        }
    }
    return false;
}

// True when the decode kernel can hold M rows of K activations.
bool gemv_fits(int type, int M, int64_t K, int xd_ld, int max_smem) {
    if (K > (1 << 24)) return false;
    GemvParams P = {};
    int smem = 0;
    return plan_gemv(type, M, static_cast<int>(K), xd_ld, max_smem, P, smem);
}

// Host entry.  xq/xd/xs: quantised activations ([M][K] int8, [M][xd_ld] fp32
// scales and int32 sums), 16-byte aligned, xd_ld a multiple of 4.
cudaError_t launch_gemv(int type, const void *W, int64_t N, int64_t K, const int8_t *xq,
                        const float *xd, const int32_t *xs, int xd_ld, int M, float *y,
                        cudaStream_t st, bool pdl, int num_sms, int max_smem, int *status) {
    const int BB = block_bytes(type), QK = block_weights(type);
    const int UPB = type == QMM_Q8_0 ? 1 : type == QMM_Q4_K ? 8 : 4;
    const int nb = static_cast<int>(K / QK);
    GemvParams P = {};
    int smem = 0;
    if (!plan_gemv(type, M, static_cast<int>(K), xd_ld, max_smem, P, smem))
        return cudaErrorInvalidValue;
    const int MT = M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8;
    P.W = static_cast<const uint8_t *>(W);
    P.N = N;
    P.K = static_cast<int>(K);
    P.M = M;
    P.RB = nb * BB;
    P.total_bytes = N * static_cast<int64_t>(P.RB);
    P.UPR = nb * UPB;
    P.RPR = (P.UPR + 31) / 32;
    P.xq = xq;
    P.xd = xd;
    P.xs = xs;
    P.xd_ld = xd_ld;
    P.y = y;
    P.pdl = pdl ? 1 : 0;
    P.status = status;
    int grid = num_sms;
    if (N < grid) grid = static_cast<int>(N);
    if (grid < 1) grid = 1;
    switch (type) {
    case QMM_Q8_0: return launch_m<QMM_Q8_0>(P, MT, grid, smem, st);
    case QMM_Q4_K: return launch_m<QMM_Q4_K>(P, MT, grid, smem, st);
    default: return launch_m<QMM_Q6_K>(P, MT, grid, smem, st);
    }
}

}  // namespace qk
