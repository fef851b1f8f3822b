// gemv_mma.cu -- decode product y[M,N] = W[N,K] . x[M,K]^T for 2 <= M <= 8
// activation rows and Q4_K weights, on the tensor cores (mma.sync with fp16
// operands and fp32 accumulation).
//
// The block-per-lane decode kernel (gemv_sb.cu) gives every lane its own
// weight block and its own slice of x, so each extra activation row adds a
// full pass of dp4a work and of activation reads from shared memory; from
// M = 2 on it is bound by those reads, not by the weight stream.  Here
// sixteen weight rows are one operand of mma.m16n8k16, and the product is
// taken per Q4_K sub-block j (32 weights with one six-bit scale sc_j and
// min m_j):
//   y[t][r] = sum_j d*sc_j * sum_{k in j} q_k x_k  -  sum_j dmin*m_j * X_j,
// X_j = sum_{k in j} x_k, x = d_x*q_x the quantised activations in fp16.
//   * The quant sums: two MMAs per sub-block, A = the sixteen rows' nibbles
//     q as fp16 subnormals q * 2^-24 (exact; one LOP3 per pair of weights,
//     no offset to remove), B = x (tokens in columns, columns M..7 zero).
//     Their fp32 result is scaled by d*sc_j * 2^24 (exact in fp32) into the
//     row's accumulators.  High nibbles are read in place as 16q * 2^-24, so
//     their scale carries 2^20.
//   * The min term: one MMA per super-block, A = -dmin*m_j in fp16 (rows x
//     sub-blocks), B = X_j in two fp16 parts hi + lo (sub-blocks x tokens),
//     so X_j enters with about 22 bits.
// Rounding: x to fp16 (as the prefill kernel) and dmin*m_j to fp16; the
// scale d*sc_j is exact and every sum is fp32.  The int8 form of the
// instruction runs at about 158 TOPS on this part, a quarter of the f16
// rate, too slow for the weight stream once the dots are scaled.
//
// k order inside one MMA.  The sum over the 16 k slots does not depend on
// which k each slot holds, as long as A and B agree.  Lane (g, t) supplies
// slots 2t, 2t+1, 2t+8, 2t+9.  For the MMA of half e of sub-block
// j = 2c + h they hold weights l = 16e + 4t + (0, 2 | 1, 3) of the
// sub-block: the nibbles h of the four bytes at 32c + 16e + 4t, in the order
// (byte 0, byte 2 | byte 1, byte 3) that one LOP3 per fp16 pair produces
// (bytes 1 and 3 after one shift).  ldmatrix delivers exactly that word to
// lane (g, t) from 8 rows of 16 bytes; the quantiser stores x so that
// ldmatrix delivers the matching B registers (see quantize.cu, xh_mma).
//
// Streaming.  Rows are taken in groups of 16.  CTA c (one per SM) owns a
// range of 8-row halves, balanced to within one half, i.e. whole groups plus
// at most one half group; its (group, chunk of CH super-blocks) units are
// split evenly between eight warps.  Each warp streams its units through a
// private ring: a stage is one chunk of the group's rows, brought in by one
// or two 2-D tensor copies of 8 rows x CH super-blocks (rows past N and
// bytes past the row end arrive as zeros).  The rows land densely, 144*CH
// bytes apart; CH is odd (5, 3 or 1), so the eight rows of an ldmatrix are
// eight distinct 16-byte bank groups.  A group whose units are split between
// warps leaves partial sums in shared memory that are added in warp order at
// the end; every y element is written once (deterministic).
//
// Activations.  The activation quantiser runs just before this kernel and
// writes x (fp16, fragment order) and the block sums (hi, lo) per token row;
// this kernel copies all of it into shared memory with one bulk copy per
// token row.  It is launched with programmatic dependent launch and the
// quantiser triggers it only after its own wait for the kernels before it,
// so the first weight stages are issued before this kernel waits (every
// kernel that could write the weights has completed by then) and the
// activations are read after.  All waits are bounded.
#include "qmm_device.cuh"
#include "qmm_internal.h"

#include <cuda_fp16.h>

namespace qk {

namespace {

constexpr int FW = 8;  // warps
constexpr int FTHREADS = FW * 32;
constexpr int GR = 16;            // weight rows per group (the MMA's m)
constexpr int MAX_NS = 4;         // stages per warp ring
constexpr int EDGE_FLOATS = 128;  // a partial group: 16 rows x 8 tokens
// shared-memory head: stage barriers | activation barrier | edge groups |
// zeros (the B rows of tokens M..7) | edge sums.  The activation rows start
// on a 128-byte boundary and are 16 bytes past a 128-byte multiple apart, so
// token m's 16-byte ldmatrix rows sit in bank group m (+ a common offset);
// the zero rows sit in bank group 7, which no token uses while M < 8.
constexpr int OFF_XBAR = 8 * FW * MAX_NS;
constexpr int OFF_EDGE_GROUP = OFF_XBAR + 16;
constexpr int OFF_ZERO = 624;
constexpr int ZERO_BYTES = 512;
constexpr int OFF_EDGE_SUM = 1152;
constexpr int HEAD = OFF_EDGE_SUM + 2 * FW * EDGE_FLOATS * 4;
static_assert(OFF_EDGE_GROUP + 2 * FW * 4 <= OFF_ZERO && OFF_ZERO + ZERO_BYTES <= OFF_EDGE_SUM, "head layout");
static_assert(OFF_ZERO % 128 == 112 && HEAD % 128 == 0, "zero rows in bank group 7");
constexpr int SB_WORDS = 144 / 8;  // a super-block in the tensor map's 8-byte elements

struct MmParams {
    int64_t N;
    int K, M;
    int nb;            // super-blocks per row
    int64_t halves_q;  // 8-row halves per CTA: halves / gridDim.x
    int halves_r;      // halves % gridDim.x: the first halves_r CTAs take one more
    const uint8_t *xh; // quantiser output [M][2K + K/8 bytes]: x fp16 | block sums
    int x_ld;          // bytes per token row in shared memory (= 16 mod 128)
    float *y;
    int NS, slot_bytes;
    int CH;            // super-blocks per row per stage (5, 3 or 1)
    int row_pitch;     // stage bytes per row, 144 * CH
    int off_x, off_ring;
    int *status;
};

// 2-D tensor copy global -> shared completing on `bar`, with an L2 policy.
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint32_t bar,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t &r0, uint32_t &r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

// c = A.B + c (fp32 accumulate)
__device__ __forceinline__ void mma_acc(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// c = A.B (fresh accumulator)
__device__ __forceinline__ void mma_new(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    const float z = 0.0f;
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(z));
}

// Scales of this lane's sub-blocks 2t (low nibbles) and 2t+1 (high nibbles)
// from a Q4_K header (d, dmin, GGUF six-bit packing): s0, s1 = d*sc * 2^24
// and d*sc * 2^20 in fp32 (exact), m01 = (-dmin*m_2t, -dmin*m_2t+1) in fp16.
__device__ __forceinline__ void q4k_lane_scales(uint4 h, int t, float &s0, float &s1, uint32_t &m01) {
    const float d = half_bits_to_float(h.x), dmin = half_bits_to_float(h.x >> 16);
    uint32_t scw, mnw;  // bytes: scales (mins) of sub-blocks 0..3 or 4..7
    if (t < 2) {
        scw = h.y & 0x3F3F3F3Fu;
        mnw = h.z & 0x3F3F3F3Fu;
    } else {
        scw = (h.w & 0x0F0F0F0Fu) | ((h.y >> 2) & 0x30303030u);
        mnw = ((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u);
    }
    const int sh = 16 * (t & 1);
    s0 = d * static_cast<float>((scw >> sh) & 0xFF) * 16777216.0f;
    s1 = d * static_cast<float>((scw >> (sh + 8)) & 0xFF) * 1048576.0f;
    const __half2 m = __floats2half2_rn(-(dmin * static_cast<float>((mnw >> sh) & 0xFF)),
                                        -(dmin * static_cast<float>((mnw >> (sh + 8)) & 0xFF)));
    m01 = *reinterpret_cast<const uint32_t *>(&m);
}

__global__ void __launch_bounds__(FTHREADS, 1)
    gemv_mma_q4k_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ MmParams P) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;

    // this CTA's rows [r0, r1): whole 8-row halves; groups of 16 from r0
    const int cta = blockIdx.x;
    const int64_t h0 = P.halves_q * cta + min(cta, P.halves_r);
    const int nh = static_cast<int>(P.halves_q + (cta < P.halves_r ? 1 : 0));
    const int64_t r0 = 8 * h0;
    const int64_t r1 = min(P.N, 8 * (h0 + nh));
    const int ng = (nh + 1) / 2;
    const int nq = (P.nb + P.CH - 1) / P.CH;
    const int U = ng * nq;
    const int uw0 = static_cast<int>((static_cast<int64_t>(U) * warp) / FW);
    const int uw1 = static_cast<int>((static_cast<int64_t>(U) * (warp + 1)) / FW);
    const int nst = uw1 - uw0;

    const uint32_t my_bar = smem_u32(smem) + 8u * warp * MAX_NS;
    const uint32_t xbar = smem_u32(smem + OFF_XBAR);
    int *edge_group = reinterpret_cast<int *>(smem + OFF_EDGE_GROUP);
    float *edge_sum = reinterpret_cast<float *>(smem + OFF_EDGE_SUM);
    if (lane == 0) {
        for (int i = 0; i < P.NS; ++i) mbar_init(my_bar + 8u * i, 1);
        if (warp == 0) mbar_init(xbar, 1);
        fence_mbar_init();
    }
    if (lane < 2) edge_group[2 * warp + lane] = -1;
    if (threadIdx.x < ZERO_BYTES / 16)
        reinterpret_cast<uint4 *>(smem + OFF_ZERO)[threadIdx.x] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();

    const int ring = P.off_ring + warp * P.NS * P.slot_bytes;
    const uint64_t pol_w = policy_evict_first();
    // unit u (group, chunk) into `slot`: rows 0..7 of the group, and 8..15
    // when the CTA owns them (a CTA's rows end on a half or at N)
    auto issue = [&](int u, int slot) {
        if (lane != 0) return;
        const int gi = u / nq, qi = u - gi * nq;
        const int64_t row0 = r0 + GR * gi;
        const int boxes = r1 - row0 > 8 ? 2 : 1;
        const uint32_t bar = my_bar + 8u * slot;
        const uint32_t dst = smem_u32(smem + ring + slot * P.slot_bytes);
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(boxes * 8 * P.row_pitch));
        for (int bx = 0; bx < boxes; ++bx)
            tma_load_2d_hint(dst + bx * 8 * P.row_pitch, &tmW, qi * P.CH * SB_WORDS, static_cast<int>(row0 + 8 * bx),
                             bar, pol_w);
    };

    // the first stage of every warp before the wait for the quantiser (see
    // the header); the others after the activation copy, which would wait
    // behind them in the copy engine otherwise
    pdl_trigger();
    int issued = 0;
    if (nst > 0) issue(uw0, 0), issued = 1;
    pdl_wait();
    if (threadIdx.x == 0) {
        const uint32_t row_bytes = static_cast<uint32_t>(2 * P.K + P.K / 8);
        mbar_arrive_expect_tx(xbar, row_bytes * P.M);
        for (int m = 0; m < P.M; ++m)
            bulk_g2s(smem_u32(smem + P.off_x + m * P.x_ld), P.xh + static_cast<int64_t>(m) * row_bytes, row_bytes,
                     xbar, pol_w);
    }
    __syncthreads();  // the activation copy goes first
    for (; issued < min(P.NS, nst); ++issued) issue(uw0 + issued, issued);
    bool failed = !__all_sync(0xffffffffu, mbar_wait(xbar, 0, P.status));

    // ldmatrix row addresses of this lane (it names row lane & 7 of matrix lane >> 3)
    const int lr = lane & 7, lm = lane >> 3;
    // weights: matrices (rows 0-7 | 8-15) x (16-byte segment 2c | 2c + 1)
    const uint32_t a_off = static_cast<uint32_t>((lr + 8 * (lm & 1)) * P.row_pitch + 16 + 16 * (lm >> 1));
    // activations of token lr: matrices (half e, B register) of one
    // sub-block, and the block sums (hi | lo); tokens >= M read zeros
    const bool tok_ok = lr < P.M;
    const uint32_t x_row = smem_u32(smem + P.off_x + lr * P.x_ld);
    const uint32_t zero = smem_u32(smem + OFF_ZERO);
    const uint32_t x_base = (tok_ok ? x_row : zero) + 16 * lm;
    const uint32_t xs_base = (tok_ok ? x_row + 2 * P.K : zero) + 16 * (lm & 1);
    const uint32_t x_step = tok_ok ? 512u : 0u, xs_step = tok_ok ? 32u : 0u;  // per super-block
    const int quad = lane & ~3;

    // rows g, g+8 of the current group x tokens 2t, 2t+1; even and odd
    // sub-blocks accumulate separately (two independent chains), c = c + c2
    float c[4] = {0.0f, 0.0f, 0.0f, 0.0f}, c2[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    int cur = -1;       // group of c (CTA-local), -1 none
    int cur_first = 0;  // c holds the group from its first chunk
    int consumed = 0, slot = 0, islot = min(P.NS, nst) % P.NS;
    uint32_t phase = 0;

    // c of group `gi` complete for this warp: y if it covered the group's
    // whole K, else an edge record (first or last group of this warp's range)
    auto flush = [&](int gi, bool whole) {
#pragma unroll
        for (int i = 0; i < 4; ++i) c[i] += c2[i];
        if (whole) {
            const int64_t row = r0 + GR * gi + g;
            const int tk = 2 * t;
            if (row < r1) {
                if (tk < P.M) P.y[static_cast<int64_t>(tk) * P.N + row] = c[0];
                if (tk + 1 < P.M) P.y[static_cast<int64_t>(tk + 1) * P.N + row] = c[1];
            }
            if (row + 8 < r1) {
                if (tk < P.M) P.y[static_cast<int64_t>(tk) * P.N + row + 8] = c[2];
                if (tk + 1 < P.M) P.y[static_cast<int64_t>(tk + 1) * P.N + row + 8] = c[3];
            }
        } else {
            const int e = 2 * warp + (gi == (uw0 / nq) ? 0 : 1);
            if (lane == 0) edge_group[e] = gi;
            *reinterpret_cast<float4 *>(edge_sum + e * EDGE_FLOATS + 4 * lane) = make_float4(c[0], c[1], c[2], c[3]);
        }
    };

    for (int k = 0; k < nst && !failed; ++k) {
        // every lane waits; the warp goes on only if all of them saw the stage
        if (!__all_sync(0xffffffffu, mbar_wait(my_bar + 8u * slot, phase, P.status))) {
            failed = true;
            break;
        }
        consumed = k + 1;
        const int u = uw0 + k, gi = u / nq, qi = u - gi * nq;
        if (gi != cur) {  // a new group (the last one was flushed at its last unit)
            cur = gi;
            cur_first = qi == 0;
            c[0] = c[1] = c[2] = c[3] = 0.0f;
            c2[0] = c2[1] = c2[2] = c2[3] = 0.0f;
        }
        const int sb0 = qi * P.CH, nsb = min(P.CH, P.nb - sb0);
        const uint8_t *st = smem + ring + slot * P.slot_bytes;
        const uint32_t a_stage = smem_u32(st) + a_off;
#pragma unroll 1
        for (int s = 0; s < nsb; ++s) {
            const int kb = sb0 + s;
            // scales of sub-blocks 2t, 2t+1 for rows g and g+8
            float sa0, sa1, sb0f, sb1f;
            uint32_t ma, mb;
            q4k_lane_scales(*reinterpret_cast<const uint4 *>(st + g * P.row_pitch + 144 * s), t, sa0, sa1, ma);
            q4k_lane_scales(*reinterpret_cast<const uint4 *>(st + (g + 8) * P.row_pitch + 144 * s), t, sb0f, sb1f,
                            mb);
            // the min term: k slots 2t, 2t+1 = sub-blocks 2t, 2t+1 (sums hi),
            // slots 2t+8, 2t+9 = the same sub-blocks (sums lo)
            {
                uint32_t xhi, xlo;
                ldsm_x2(xs_base + kb * xs_step, xhi, xlo);
                mma_acc(c2, ma, mb, ma, mb, xhi, xlo);
            }
            const uint32_t a_sb = a_stage + 144 * s;
            const uint32_t x_sb = x_base + kb * x_step;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {  // quant bytes 32cc..32cc+31: sub-blocks 2cc, 2cc+1
                uint32_t wa0, wb0, wa1, wb1;  // rows g | g+8, halves e = 0 | 1
                ldsm_x4(a_sb + 32 * cc, wa0, wb0, wa1, wb1);
                const uint32_t wa0s = wa0 >> 8, wb0s = wb0 >> 8, wa1s = wa1 >> 8, wb1s = wb1 >> 8;
                // scales of sub-blocks 2cc, 2cc+1 from the quad's lane cc
                const float s_a0 = __shfl_sync(0xffffffffu, sa0, quad | cc);
                const float s_a1 = __shfl_sync(0xffffffffu, sa1, quad | cc);
                const float s_b0 = __shfl_sync(0xffffffffu, sb0f, quad | cc);
                const float s_b1 = __shfl_sync(0xffffffffu, sb1f, quad | cc);
#pragma unroll
                for (int h = 0; h < 2; ++h) {  // sub-block 2cc + h: low or high nibbles
                    const uint32_t mk = h ? 0x00F000F0u : 0x000F000Fu;
                    uint32_t x0, x1, x2, x3;
                    ldsm_x4(x_sb + 64 * (2 * cc + h), x0, x1, x2, x3);
                    float d[4];
                    mma_new(d, wa0 & mk, wb0 & mk, wa0s & mk, wb0s & mk, x0, x1);
                    mma_acc(d, wa1 & mk, wb1 & mk, wa1s & mk, wb1s & mk, x2, x3);
                    float(&acc)[4] = h ? c2 : c;
                    const float sa = h ? s_a1 : s_a0, sb = h ? s_b1 : s_b0;
                    acc[0] = fmaf(sa, d[0], acc[0]);
                    acc[1] = fmaf(sa, d[1], acc[1]);
                    acc[2] = fmaf(sb, d[2], acc[2]);
                    acc[3] = fmaf(sb, d[3], acc[3]);
                }
            }
        }
        __syncwarp();
        if (issued < nst) {
            // the slot just read is refilled: order the reads before the async write
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(uw0 + issued, islot);
            ++issued;
            if (++islot == P.NS) islot = 0;
        }
        if (++slot == P.NS) slot = 0, phase ^= 1u;
        // the group ends here for this warp: flush
        if (k == nst - 1 || (uw0 + k + 1) / nq != gi) flush(gi, cur_first && qi == nq - 1);
    }
    // no bulk copy may still be in flight when the CTA exits
    if (lane == 0)
        for (int k = consumed; k < issued; ++k)
            mbar_wait(my_bar + 8u * (k % P.NS), static_cast<uint32_t>((k / P.NS) & 1), P.status);
    if (threadIdx.x == 0) mbar_wait(xbar, 0, P.status);
    __syncthreads();
    if (failed) return;
    // groups cut by warp boundaries: records e = 2w + {0, 1} in warp order;
    // the first record of a group adds the others in record order
    for (int e = warp; e < 2 * FW; e += FW) {
        const int gi = edge_group[e];
        if (gi < 0) continue;
        bool first = true;
        for (int f = 0; f < e; ++f) first = first && edge_group[f] != gi;
        if (!first) continue;
        float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int f = e; f < 2 * FW; ++f)
            if (edge_group[f] == gi) {
                const float4 v = *reinterpret_cast<const float4 *>(edge_sum + f * EDGE_FLOATS + 4 * lane);
                s[0] += v.x;
                s[1] += v.y;
                s[2] += v.z;
                s[3] += v.w;
            }
        c[0] = s[0];
        c[1] = s[1];
        c[2] = s[2];
        c[3] = s[3];
        c2[0] = c2[1] = c2[2] = c2[3] = 0.0f;
        flush(gi, true);
    }
}

// Shared-memory plan: head | activation rows [M][x_ld] | FW rings of NS
// slots, each GR rows of CH super-blocks.  CH is the widest of 5, 3, 1 that
// leaves two stages per warp and, when there is a choice, at least three
// units per warp (units_at(ch) = a CTA's units for that chunk width; <= 0
// when unknown).
template <typename F>
bool plan_mm(int M, int64_t K, int max_smem, F units_at, MmParams &P, int &smem) {
    const int64_t x_ld = ((2 * K + K / 8 + 127) / 128) * 128 + 16;
    const int64_t o_x = (HEAD + 127) / 128 * 128;
    const int64_t o_ring = (o_x + M * x_ld + 127) / 128 * 128;
    int best = 0;
    int64_t best_ns = 0;
    for (int ch = 5; ch >= 1; ch -= 2) {
        const int64_t slot = static_cast<int64_t>(GR) * 144 * ch;
        const int64_t ns = (max_smem - o_ring) / (FW * slot);
        if (ns < 2) continue;
        best = ch;
        best_ns = ns;
        const int64_t units = units_at(ch);
        if (units <= 0 || units >= 3 * FW) break;
    }
    if (best == 0) return false;
    const int64_t ns = best_ns > MAX_NS ? MAX_NS : best_ns;
    P.NS = static_cast<int>(ns);
    P.CH = best;
    P.row_pitch = 144 * best;
    P.slot_bytes = GR * P.row_pitch;
    P.x_ld = static_cast<int>(x_ld);
    P.off_x = static_cast<int>(o_x);
    P.off_ring = static_cast<int>(o_ring);
    smem = static_cast<int>(o_ring + FW * ns * P.slot_bytes);
    return true;
}

}  // namespace

bool gemv_mma_fits(int type, int M, int64_t K, int max_smem) {
    if (type != QMM_Q4_K || M < 2 || M > 8 || K < 256 || K % 256 || K > (1 << 20)) return false;
    if (tensor_map_encoder() == nullptr) return false;
    MmParams P = {};
    int smem = 0;
    return plan_mm(M, K, max_smem, [](int) { return int64_t(0); }, P, smem);
}

cudaError_t launch_gemv_mma(int type, const void *W, int64_t N, int64_t K, const void *xh, int M, float *y,
                            cudaStream_t st, int num_sms, int max_smem, int *status) {
    if (!gemv_mma_fits(type, M, K, max_smem) || N > (int64_t(1) << 30)) return cudaErrorNotSupported;
    const int64_t halves = (N + 7) / 8;
    int64_t grid = num_sms;
    if (grid > halves) grid = halves;
    if (grid < 1) grid = 1;
    const int nb = static_cast<int>(K / 256);
    // a CTA's units for chunk width ch: its groups x chunks per row
    const int64_t max_groups = (halves / grid + 2) / 2;
    auto units_at = [&](int ch) { return max_groups * ((nb + ch - 1) / ch); };
    MmParams P = {};
    int smem = 0;
    plan_mm(M, K, max_smem, units_at, P, smem);
    if (units_at(P.CH) > (int64_t(1) << 30)) return cudaErrorInvalidValue;
    // the weights as 8-byte elements [N][18 * nb]: boxes of CH super-blocks x 8 rows
    CUtensorMap tmW;
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(nb) * SB_WORDS, static_cast<cuuint64_t>(N)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(nb) * 144};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(P.CH * SB_WORDS), 8u};
        const cuuint32_t es[2] = {1, 1};
        if (tensor_map_encoder()(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void *>(W), dims, strides, box,
                                 es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    P.N = N;
    P.K = static_cast<int>(K);
    P.M = M;
    P.nb = nb;
    P.halves_q = halves / grid;
    P.halves_r = static_cast<int>(halves % grid);
    P.xh = static_cast<const uint8_t *>(xh);
    P.y = y;
    P.status = status;
    cudaError_t e = cudaFuncSetAttribute(gemv_mma_q4k_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(FTHREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_mma_q4k_kernel, tmW, P);
}

}  // namespace qk
