// gemv.cu -- the memory-bound decode product y[M,N] = W[N,K] . x[M,K]^T for
// M <= 8 (the GEMV bucket of infr's per-op profile; M > 1 is its concurrent
// generation slots, "--parallel N").
//
// Design (sm_103a):
//   * One CTA per SM, each owning a contiguous range of whole output rows, so
//     every y element is produced by exactly one CTA with a fixed summation
//     order (deterministic, no atomics, no zero-fill).
//   * A producer thread streams the CTA's weight bytes through a ring of
//     shared-memory stages with 1-D bulk async copies (cp.async.bulk) that
//     complete on mbarriers, so tens of KB per SM are in flight whatever the
//     consumers do.  Q6_K/Q8_0 rows are not 16-byte aligned: a stage is
//     copied from its start rounded down to 16 bytes and consumers index from
//     the remainder.
//   * The quantised activations (from the quantiser kernel launched just
//     before, with programmatic dependent launch so the weight stream starts
//     while the quantiser still runs) are bulk-copied into shared memory once.
//   * Sixteen compute warps.  The weight stream is cut into rounds of 32
//     units, a unit being one lane's share of a block (Q4_K: one 32-weight
//     sub-block; Q6_K: 64 weights = 16 positions x 4 groups; Q8_0: one
//     block).  A round never crosses a row; warp w takes rounds w, w+16, ...
//     with 32-bit incremental index arithmetic, reduces each round with
//     shuffles and parks the total in shared memory.
//   * A finalizer warp adds the round totals of each row in round order once
//     a stage is complete (an mbarrier counts the compute warps), stores the
//     finished rows and hands the stage back to the producer.  No CTA-wide
//     barrier: every wait is a bounded mbarrier wait.
//   * Dot products are exact int32 dp4a over a 16- or 32-element group; the
//     fp32 scale and min terms are applied per group as in the oracle.
#include "qmm_device.cuh"

namespace qk {

namespace {

constexpr int NW = 16;  // compute warps: 1..NW; warp 0 finalizes; warp NW+1 produces
constexpr int PROD_WARP = NW + 1;
constexpr int NTHREADS = (NW + 2) * 32;
constexpr int SLOT_SLACK = 64;  // alignment head + over-read of the word helpers
constexpr int HEAD_BYTES = 512; // mbarriers, stage bases, carry, abort flag

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
    int NR;    // rounds per stage (a multiple of NW, or NW/2)
    int NS;    // stages in the ring
    int slot_bytes;
    const int8_t *xq;    // [M][K]
    const float *xd;     // [M][xd_ld]   scale per 32-block
    const int32_t *xs;   // [M][xs_ld]   sum per 16-element half block
    int xd_ld, xs_ld;
    float *y;  // [M][N]
    // shared-memory layout (byte offsets from the dynamic base)
    int off_rt, off_xq, off_xd, off_xs, off_ring;
    int pdl;
    int *status;  // device status word (bounded-wait timeouts)
};

// Byte offset, relative to the CTA's first row, of the start / end of local
// round R.
template <int T>
__device__ __forceinline__ int round_begin(const GemvParams &P, int R) {
    constexpr int UPB = Units<T>::UPB, BB = Fmt<T>::BB;
    const int row = R / P.RPR, rr = R - row * P.RPR;
    return row * P.RB + (32 * rr / UPB) * BB;
}

template <int T>
__device__ __forceinline__ int round_end(const GemvParams &P, int R) {
    constexpr int UPB = Units<T>::UPB, BB = Fmt<T>::BB;
    const int row = R / P.RPR, rr = R - row * P.RPR;
    const int ue = min(32 * (rr + 1), P.UPR);
    return row * P.RB + (ue / UPB) * BB;
}

// n consecutive 32-bit words at byte offset `off` of shared memory `sm`
// (any alignment): aligned words are loaded and funnel-shifted into place.
template <int N>
__device__ __forceinline__ void ld_words(const uint8_t *sm, int off, uint32_t (&w)[N]) {
    const uint32_t *a = reinterpret_cast<const uint32_t *>(sm + (off & ~3));
    const uint32_t sh = static_cast<uint32_t>(off & 3) * 8u;
    uint32_t prev = a[0];
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const uint32_t next = a[i + 1];
        w[i] = __funnelshift_r(prev, next, sh);
        prev = next;
    }
}

__device__ __forceinline__ uint4 ld16(const uint8_t *sm, int off) {
    return *reinterpret_cast<const uint4 *>(sm + off);
}

__device__ __forceinline__ int dot16(const uint32_t (&w)[4], const uint4 x, int acc) {
    acc = __dp4a(static_cast<int>(w[0]), static_cast<int>(x.x), acc);
    acc = __dp4a(static_cast<int>(w[1]), static_cast<int>(x.y), acc);
    acc = __dp4a(static_cast<int>(w[2]), static_cast<int>(x.z), acc);
    return __dp4a(static_cast<int>(w[3]), static_cast<int>(x.w), acc);
}

// Shared-memory views of the activations.
struct XView {
    const uint8_t *sm;
    int xq, xd, xs;  // byte offsets
    int K, xd_ld, xs_ld;
};

// --------------------------------------------------------------------------
// Per-unit dot products.  `blk` is the byte offset of the unit's block in
// shared memory, `kb` its block index within the row; acc[m] gains the unit's
// fp32 share.
// --------------------------------------------------------------------------

// Q4_K, sub-block j (32 weights): nibbles of qs[32c .. 32c+31], c = j/2, low
// nibble for even j and high for odd j;  y += dx*(d*(sc*I) - dmin*(m*s)).
template <int MT>
__device__ __forceinline__ void unit_q4k(const XView &X, int blk, int kb, int j, float (&acc)[MT]) {
    const uint8_t *sm = X.sm;
    const uint4 hdr = ld16(sm, blk);
    const int c = j >> 1;
    const uint4 qa = ld16(sm, blk + 16 + 32 * c);
    const uint4 qb = ld16(sm, blk + 32 + 32 * c);
    const uint32_t sh = (j & 1) * 4;
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
    const uint4 f = rot ? qb : qa, s = rot ? qa : qb;
    uint32_t wf[4] = {(f.x >> sh) & 0x0F0F0F0Fu, (f.y >> sh) & 0x0F0F0F0Fu,
                      (f.z >> sh) & 0x0F0F0F0Fu, (f.w >> sh) & 0x0F0F0F0Fu};
    uint32_t ws[4] = {(s.x >> sh) & 0x0F0F0F0Fu, (s.y >> sh) & 0x0F0F0F0Fu,
                      (s.z >> sh) & 0x0F0F0F0Fu, (s.w >> sh) & 0x0F0F0F0Fu};
    const int b32 = kb * 8 + j;
    const int xo = kb * 256 + 32 * j;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        const int xr = X.xq + m * X.K + xo;
        int I = dot16(wf, ld16(sm, xr + 16 * rot), 0);
        I = dot16(ws, ld16(sm, xr + 16 * (1 - rot)), I);
        const float dx = *reinterpret_cast<const float *>(sm + X.xd + 4 * (m * X.xd_ld + b32));
        const int2 s2 = *reinterpret_cast<const int2 *>(sm + X.xs + 4 * (m * X.xs_ld + 2 * b32));
        acc[m] += dx * (d * static_cast<float>(sc * I) - dmin * static_cast<float>(mn * (s2.x + s2.y)));
    }
}

// Q6_K, unit u = 2h + t: half h, positions l = 16t .. 16t+15 of each of the
// four 32-weight groups g of the half.  Group g uses scale 8h + 2g + t and
// the activations at 128h + 32g + 16t.  The 6-bit q (0..63) is used as is
// and 32*sum(x) subtracted:  sum (q-32)*x = sum q*x - 32*sum x.
template <int MT>
__device__ __forceinline__ void unit_q6k(const XView &X, int blk, int kb, int u, int lane,
                                         float (&acc)[MT]) {
    const uint8_t *sm = X.sm;
    const int h = u >> 1, t = u & 1;
    uint32_t qla[4], qlb[4], qhw[4], scw[2];
    ld_words<4>(sm, blk + 64 * h + 16 * t, qla);
    ld_words<4>(sm, blk + 64 * h + 32 + 16 * t, qlb);
    ld_words<4>(sm, blk + 128 + 32 * h + 16 * t, qhw);
    ld_words<2>(sm, blk + 192 + 8 * h + t, scw);  // scale of group g at byte 2g
    const float d = half_bits_to_float(*reinterpret_cast<const uint16_t *>(sm + blk + 208));
    // Groups are visited in an order rotated by (block parity, h) so the
    // activation reads of a quarter warp fall in distinct banks.
    const int rot = ((lane >> 2) & 1) * 2 + h;
    int sc[4];
    uint32_t q[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int g = (i + rot) & 3;
        const uint32_t sel = (g & 2) ? scw[1] : scw[0];
        sc[i] = static_cast<int>(static_cast<int8_t>((sel >> ((g & 1) * 16)) & 0xFF));
        const uint32_t lsh = (g & 2) ? 4u : 0u;
        const uint32_t hsh = 2u * static_cast<uint32_t>(g);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint32_t lo = (((g & 1) ? qlb[e] : qla[e]) >> lsh) & 0x0F0F0F0Fu;
            const uint32_t hi = ((qhw[e] >> hsh) << 4) & 0x30303030u;
            q[i][e] = lo | hi;
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        float part = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int g = (i + rot) & 3;
            const uint4 xv = ld16(sm, X.xq + m * X.K + kb * 256 + 128 * h + 32 * g + 16 * t);
            const int sx = *reinterpret_cast<const int *>(
                sm + X.xs + 4 * (m * X.xs_ld + kb * 16 + 8 * h + 2 * g + t));
            const int I = dot16(q[i], xv, -32 * sx);
            const float dx = *reinterpret_cast<const float *>(
                sm + X.xd + 4 * (m * X.xd_ld + kb * 8 + 4 * h + g));
            part += dx * static_cast<float>(sc[i] * I);
        }
        acc[m] += d * part;
    }
}

// Q8_0: one block of 32 weights; y += dx * (d * I).
template <int MT>
__device__ __forceinline__ void unit_q80(const XView &X, int blk, int kb, int lane, float (&acc)[MT]) {
    const uint8_t *sm = X.sm;
    uint32_t qw[8];
    ld_words<8>(sm, blk + 2, qw);
    const float d = half_bits_to_float(*reinterpret_cast<const uint16_t *>(sm + blk));
    const int rot = (lane >> 2) & 1;
    uint32_t wf[4], ws[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        wf[i] = rot ? qw[4 + i] : qw[i];
        ws[i] = rot ? qw[i] : qw[4 + i];
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        const int xr = X.xq + m * X.K + kb * 32;
        int I = dot16(wf, ld16(sm, xr + 16 * rot), 0);
        I = dot16(ws, ld16(sm, xr + 16 * (1 - rot)), I);
        const float dx = *reinterpret_cast<const float *>(sm + X.xd + 4 * (m * X.xd_ld + kb));
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
    // rows [r0, r1) of this CTA
    const int64_t r0 = (P.N * blockIdx.x) / gridDim.x;
    const int64_t r1 = (P.N * (blockIdx.x + 1)) / gridDim.x;
    const int nrows = static_cast<int>(r1 - r0);
    const int nrounds = nrows * P.RPR;
    const int nstages = (nrounds + P.NR - 1) / P.NR;

    // header: full[NS], empty[NS], done[NS], xbar | stage base[NS] | carry[8] | abort
    const uint32_t bar_full = smem_u32(smem);
    const uint32_t bar_empty = bar_full + 8u * P.NS;
    const uint32_t bar_done = bar_empty + 8u * P.NS;
    const uint32_t bar_x = bar_done + 8u * P.NS;
    int *stage_base = reinterpret_cast<int *>(smem + 8 * (3 * P.NS + 1));
    float *carry = reinterpret_cast<float *>(stage_base + P.NS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(carry + 8);
    float *rt = reinterpret_cast<float *>(smem + P.off_rt);

    if (threadIdx.x == 0) {
        for (int i = 0; i < P.NS; ++i) {
            mbar_init(bar_full + 8u * i, 1);
            mbar_init(bar_empty + 8u * i, 1);
            mbar_init(bar_done + 8u * i, NW);
        }
        mbar_init(bar_x, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == PROD_WARP) {
        // ------------------------------------------------------- producer
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_x = policy_evict_last();
            // offsets are relative to Wc, the CTA's first byte rounded down to
            // 16 bytes, so a multiple of 16 in them is 16-byte aligned in memory
            const int64_t cta_byte = r0 * P.RB;
            const uint8_t *Wc = P.W + (cta_byte & ~int64_t(15));
            const int cta_off = static_cast<int>(cta_byte & 15);
            const int64_t avail = P.total_bytes - (cta_byte & ~int64_t(15));  // bytes from Wc to the end
            const uint32_t ring = smem_u32(smem + P.off_ring);
            bool x_issued = false;
            int issued = 0;
            for (int s = 0; s < nstages; ++s) {
                const int slot = s % P.NS;
                if (s >= P.NS) {
                    const uint32_t par = static_cast<uint32_t>(((s / P.NS) - 1) & 1);
                    if (*abort_flag || !mbar_wait(bar_empty + 8u * slot, par, P.status)) {
                        *abort_flag = 1;
                        break;
                    }
                }
                const int R0 = s * P.NR;
                const int R1 = min(R0 + P.NR, nrounds);
                const int a = cta_off + round_begin<T>(P, R0);
                const int b = cta_off + round_end<T>(P, R1 - 1);
                const int a16 = a & ~15;
                int b16 = (b + 15) & ~15;
                const uint32_t dst = ring + static_cast<uint32_t>(slot) * P.slot_bytes;
                if (b16 > avail) {
                    // the last bytes of the matrix: plain loads for the tail
                    b16 = b & ~15;
                    for (int i = b16; i < b; ++i)
                        smem[P.off_ring + slot * P.slot_bytes + (i - a16)] = Wc[i];
                }
                stage_base[slot] = a16;
                const uint32_t nbytes = static_cast<uint32_t>(b16 - a16);
                mbar_arrive_expect_tx(bar_full + 8u * slot, nbytes);
                if (nbytes) bulk_g2s(dst, Wc + a16, nbytes, bar_full + 8u * slot, pol_w);
                ++issued;
                if (!x_issued && (s + 1 == P.NS || s + 1 == nstages)) {
                    if (P.pdl) pdl_wait();
                    const uint32_t nq = static_cast<uint32_t>(P.M * P.K);
                    const uint32_t nd = static_cast<uint32_t>(P.M * P.xd_ld * 4);
                    const uint32_t ns = static_cast<uint32_t>(P.M * P.xs_ld * 4);
                    mbar_arrive_expect_tx(bar_x, nq + nd + ns);
                    bulk_g2s(smem_u32(smem + P.off_xq), P.xq, nq, bar_x, pol_x);
                    bulk_g2s(smem_u32(smem + P.off_xd), P.xd, nd, bar_x, pol_x);
                    bulk_g2s(smem_u32(smem + P.off_xs), P.xs, ns, bar_x, pol_x);
                    x_issued = true;
                }
            }
            // drain: every copy issued must have landed before the CTA exits
            for (int s = (issued > P.NS ? issued - P.NS : 0); s < issued; ++s)
                mbar_wait(bar_full + 8u * (s % P.NS), static_cast<uint32_t>((s / P.NS) & 1), P.status);
            if (x_issued) mbar_wait(bar_x, 0, P.status);
        }
        return;
    }

    if (warp == 0) {
        // ------------------------------------------------------ finalizer
        for (int s = 0; s < nstages; ++s) {
            const int slot = s % P.NS;
            if (*abort_flag || !mbar_wait(bar_done + 8u * slot, static_cast<uint32_t>((s / P.NS) & 1), P.status)) {
                *abort_flag = 1;
                break;
            }
            const float *rts = rt + slot * P.NR * MT;
            const int R0 = s * P.NR;
            const int R1 = min(R0 + P.NR, nrounds);
            const int row_first = R0 / P.RPR, row_last = (R1 - 1) / P.RPR;
            float cin[MT];
#pragma unroll
            for (int m = 0; m < MT; ++m) cin[m] = carry[m];
            __syncwarp();
            for (int k = row_first + lane; k <= row_last; k += 32) {
                const int jb = max(R0, k * P.RPR) - R0;
                const int je = min(R1, (k + 1) * P.RPR) - R0;
                float tot[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m) tot[m] = (k * P.RPR < R0) ? cin[m] : 0.0f;
                for (int j = jb; j < je; ++j) {
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
        return;
    }

    // ------------------------------------------------------------- compute
    const int wi = warp - 1;
    XView X;
    X.sm = smem;
    X.xq = P.off_xq;
    X.xd = P.off_xd;
    X.xs = P.off_xs;
    X.K = P.K;
    X.xd_ld = P.xd_ld;
    X.xs_ld = P.xs_ld;
    if (nstages > 0 && !mbar_wait(bar_x, 0, P.status)) *abort_flag = 1;
    const int cta_off = static_cast<int>((r0 * P.RB) & 15);
    // in stage s this warp takes the stage's rounds wi, wi + NW, ...
    const int step_q = NW / P.RPR, step_r = NW - step_q * P.RPR;
    const int per_stage = (P.NR + NW - 1) / NW;
    for (int s = 0; s < nstages; ++s) {
        int R = s * P.NR + wi;
        int row = R / P.RPR, rr = R - row * P.RPR;
        const int Rend = min((s + 1) * P.NR, nrounds);
        if (*abort_flag) break;
        const int slot = s % P.NS;
        if (!mbar_wait(bar_full + 8u * slot, static_cast<uint32_t>((s / P.NS) & 1), P.status)) {
            *abort_flag = 1;
            break;
        }
        // shared-memory byte offset of the CTA's first weight byte for this stage
        const int base = P.off_ring + slot * P.slot_bytes - stage_base[slot] + cta_off;
        float *rts = rt + slot * P.NR * MT;
        for (int t = 0; t < per_stage; ++t) {
            if (R < Rend) {
                const int nu = min(32, P.UPR - 32 * rr);
                float acc[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m) acc[m] = 0.0f;
                if (lane < nu) {
                    const int ur = 32 * rr + lane;
                    const int kb = ur / UPB, su = ur - kb * UPB;
                    const int blk = base + row * P.RB + kb * BB;
                    if constexpr (T == QMM_Q4_K) unit_q4k<MT>(X, blk, kb, su, acc);
                    else if constexpr (T == QMM_Q6_K) unit_q6k<MT>(X, blk, kb, su, lane, acc);
                    else unit_q80<MT>(X, blk, kb, lane, acc);
                }
                const int j = wi + t * NW;
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
            R += NW;
            row += step_q;
            rr += step_r;
            if (rr >= P.RPR) {
                rr -= P.RPR;
                ++row;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_done + 8u * slot);
    }
}

template <int T, int MT>
cudaError_t launch_t(const GemvParams &P, int grid, int smem, cudaStream_t st) {
    auto kfn = gemv_kernel<T, MT>;
    cudaError_t e = set_smem_attrs(kfn, smem);
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

int mt_of(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8; }

// Plan the shared-memory layout for a shape: stage size (rounds per stage, a
// multiple of the compute-warp count, ~20 KB), ring depth (2..8 stages) and
// the offsets of every region.  Returns false when the activations of M rows
// do not leave room for a two-stage ring.
bool plan_gemv(int type, int M, int K, int xd_ld, int xs_ld, int max_smem, GemvParams &P, int &smem) {
    const int BB = block_bytes(type);
    const int UPB = type == QMM_Q8_0 ? 1 : type == QMM_Q4_K ? 8 : 4;
    const int round_bytes = (32 / UPB) * BB;
    const int MT = mt_of(M);
    auto align = [](int64_t v, int64_t a) { return (v + a - 1) / a * a; };
    const int64_t xq_bytes = align(static_cast<int64_t>(MT) * K, 16);
    const int64_t xd_bytes = align(static_cast<int64_t>(MT) * xd_ld * 4, 16);
    const int64_t xs_bytes = align(static_cast<int64_t>(MT) * xs_ld * 4, 16);
    // NR: a multiple of NW near 20 KB; a single half-size step (NW/2 rounds,
    // half the compute warps idle) when the activations leave no more room
    int nr = NW * ((20480 + NW * round_bytes / 2) / (NW * round_bytes));
    if (nr < NW) nr = NW;
    for (; nr >= NW / 2; nr = (nr > NW) ? nr - NW : nr - NW / 2) {
        const int64_t slot = align(static_cast<int64_t>(nr) * round_bytes + SLOT_SLACK, 128);
        for (int ns = 8; ns >= 2; --ns) {
            int64_t off = HEAD_BYTES;
            const int64_t o_rt = off;
            off = align(off + static_cast<int64_t>(ns) * nr * MT * 4, 128);
            const int64_t o_xq = off;
            off = align(off + xq_bytes, 128);
            const int64_t o_xd = off;
            off = align(off + xd_bytes, 128);
            const int64_t o_xs = off;
            off = align(off + xs_bytes, 128);
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

}  // namespace

// True when the decode kernel can hold M rows of K activations.
bool gemv_fits(int type, int M, int64_t K, int xd_ld, int xs_ld, int max_smem) {
    if (M < 1 || M > 8 || K > (1 << 22)) return false;
    if (type != QMM_Q8_0 && type != QMM_Q4_K && type != QMM_Q6_K) return false;  // its three unit kinds
    GemvParams P = {};
    int smem = 0;
    return plan_gemv(type, M, static_cast<int>(K), xd_ld, xs_ld, max_smem, P, smem);
}

// Host entry.  xq/xd/xs: quantised activations ([M][K] int8, [M][xd_ld] fp32
// scale per 32-block, [M][xs_ld] int32 sum per 16-element half block), all
// 16-byte aligned, xd_ld and xs_ld multiples of 4.
cudaError_t launch_gemv(int type, const void *W, int64_t N, int64_t K, const int8_t *xq,
                        const float *xd, const int32_t *xs, int xd_ld, int xs_ld, int M, float *y,
                        cudaStream_t st, bool pdl, int num_sms, int max_smem, int *status) {
    const int BB = block_bytes(type), QK = block_weights(type);
    const int UPB = type == QMM_Q8_0 ? 1 : type == QMM_Q4_K ? 8 : 4;
    const int nb = static_cast<int>(K / QK);
    GemvParams P = {};
    int smem = 0;
    if (!plan_gemv(type, M, static_cast<int>(K), xd_ld, xs_ld, max_smem, P, smem))
        return cudaErrorInvalidValue;
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
    P.xs_ld = xs_ld;
    P.y = y;
    P.pdl = pdl ? 1 : 0;
    P.status = status;
    // one CTA per SM, more when a CTA's byte range would not fit 31 bits
    int64_t grid = num_sms;
    const int64_t max_rows = ((int64_t(1) << 30) / P.RB);
    if ((N + grid - 1) / grid > max_rows) grid = (N + max_rows - 1) / max_rows;
    if (N < grid) grid = N;
    if (grid < 1) grid = 1;
    if (grid > 0x7fffffff) return cudaErrorInvalidValue;
    const int g = static_cast<int>(grid);
    switch (type) {
    case QMM_Q8_0: return launch_m<QMM_Q8_0>(P, mt_of(M), g, smem, st);
    case QMM_Q4_K: return launch_m<QMM_Q4_K>(P, mt_of(M), g, smem, st);
    default: return launch_m<QMM_Q6_K>(P, mt_of(M), g, smem, st);
    }
}

}  // namespace qk
