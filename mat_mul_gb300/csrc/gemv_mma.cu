// gemv_mma.cu -- decode product y[M,N] = W[N,K] . x[M,K]^T for 2 <= M <= 8
// activation rows and Q4_K or Q6_K weights, on the tensor cores (mma.sync
// with fp16 operands and fp32 accumulation).
//
// The block-per-lane decode kernel (gemv_sb.cu) gives every lane its own
// weight block and its own slice of x, so each extra activation row adds a
// full pass of dp4a work and of activation reads from shared memory; from
// M = 2 on it is bound by those reads, not by the weight stream.  Here
// sixteen weight rows are the A operand of mma.m16n8k16 and the tokens the B
// operand (columns M..7 zero), and no weight is dequantised: the quants go
// into the MMA exactly, as fp16 subnormals v * 2^-24, and each MMA covers one
// scale group, so its fp32 result is scaled once by the group's exact fp32
// scale.  x = d_x*q_x are the quantised activations rounded to fp16.
//   Q4_K (sub-blocks j of 32, scale sc_j, min m_j):
//     y = sum_j d*sc_j * sum_{k in j} q_k x_k  -  sum_j dmin*m_j * X_j
//     two MMAs per sub-block (A = nibbles, one LOP3 per pair; high nibbles
//     read in place as 16q, the 16 folded into the scale); the min term is
//     one MMA per super-block, A = -dmin*m_j (fp16), B = X_j = sum_{k in j}
//     x_k as fp16 hi + lo (about 22 bits).
//   Q6_K (groups G of 16, int8 scale sc_G, q = 6 bits, offset 32):
//     y = sum_G d*sc_G * sum_{k in G} q_k x_k  -  32 d * sum_G sc_G X_G
//     one MMA per group; A = the six-bit values assembled from the 4-bit and
//     2-bit fields in place (two LOP3 and one IMAD per pair; groups 8..15 of
//     a half read the high nibbles as 16x); the offset term is two MMAs per
//     super-block with the 16 groups as the k slots: A = sc_G (fp16
//     subnormals, exact), B = X_G = the sum of the group's fp16 x as fp16 hi
//     + lo (about 22 bits).
// Rounding: x to fp16 (as the tcgen05 prefill kernel), for Q4_K dmin*m_j to
// fp16, and the Q4_K block sums and Q6_K group sums to 22 bits; every scale
// is exact and every other sum fp32.  Both fp16 operands are
// scaled by powers of two into fp16's normal range first: x per token row
// by the quantiser (its fp32 results are multiplied by the row's xinv at the
// store), -dmin*m_j per row and super-block by 2^g with dmin*2^g in
// [2^8, 2^9) (and X_j arrives times 2^-5), the min-term MMA's result then
// multiplied by 2^(5-g) in fp32, so any fp16 dmin and any finite x stay
// inside the accuracy bound.  The int8 form of the
// instruction runs at about 158 TOPS on this part, a quarter of the f16
// rate, too slow for the weight stream once the dots are scaled.
//
// k order inside one MMA.  The sum over the 16 k slots does not depend on
// which k each slot holds, as long as A and B agree.  Lane (g, t) supplies
// slots 2t, 2t+1, 2t+8, 2t+9; for the 16 weights l0..l0+15 of an MMA they
// hold l0 + 4t + (0, 2 | 1, 3): the four bytes of one 32-bit quant word in
// the order (byte 0, byte 2 | byte 1, byte 3) that one LOP3 per fp16 pair
// produces (bytes 1 and 3 after one shift).  ldmatrix delivers exactly that
// word of 8 rows of 16 bytes to lane (g, t); the quantiser stores x so that
// ldmatrix delivers the matching B registers (see quantize.cu, xh_mma).
//
// Streaming.  Rows are taken in groups of 16.  CTA c (one per SM) owns a
// range of 8-row halves, balanced to within one half, i.e. whole groups plus
// at most one half group.  A producer warp fills a ring of stages shared by
// CW consumer warps (8 or 10, whichever tiles a row's super-blocks with
// fewer empty slots); a stage is one group's 16 rows x CW super-blocks, and
// consumer warp w computes super-block (w + chunk) mod CW of it, so the
// copies are 1.2-1.5 KB (Q4_K) or 1.7-2.1 KB (Q6_K) per row and the warps
// share every stage evenly (the copy engine's cost per row segment is what
// limits short ones).
//   Q4_K: a stage is two 2-D tensor copies of 8 rows x (CW super-blocks and
//     16 bytes), rows past N and bytes past the row end arriving as zeros, so
//     rows land 16 bytes past a 128-byte multiple apart and the eight rows of
//     an ldmatrix are eight distinct 16-byte bank groups.
//   Q6_K: rows are 210-byte multiples, not 16-byte ones, so each row span is
//     one bulk copy rounded out to 16 bytes (the matrix's last bytes
//     excepted: they are loaded after the wait instead of reading past the
//     end), read from its offset inside the copy, in a pitch of an odd number
//     of 16-byte chunks.  With an even number of super-blocks per row a
//     stage's even super-blocks are 4-byte aligned and its odd ones 2-byte
//     aligned (their words are loaded in two aligned halves and shifted
//     together); the rotation gives every warp both kinds in turn.
// At a group's last stage the consumers' partial sums are added in warp
// order; every y element is written once (deterministic).
// When the activations of all of K do not fit in shared memory beside the
// ring, K is taken in P phases: the activations of one K window at a time,
// the CTA's stages of that window, then the next; a group's phase results
// are added in phase order in a shared table.
//
// Activations.  The activation quantiser runs just before this kernel and
// writes x (fp16, fragment order), the Q4_K block sums (hi, lo) per token
// row and the Q6_K group sums ([K/16][8 tokens], zeros for tokens >= M); this
// kernel copies each K window into shared memory with bulk copies.  It is
// launched with programmatic dependent launch and the quantiser triggers it
// only after its own wait for the kernels before it, so the first weight
// stages are issued before this kernel waits (every kernel that could write
// the weights has completed by then) and the activations are read after.
//
// Groups.  Matrices that read the same quantised x (q/k/v, gate/up) can
// share one launch: its CTAs are split between them by weight bytes, and
// each CTA runs its own matrix (type, tensor map, shared-memory plan).
//
// All waits are bounded.
#include "qmm_device.cuh"
#include "qmm_internal.h"

#include <cuda_fp16.h>

#include <type_traits>

namespace qk {

namespace {

constexpr int GR = 16;                 // weight rows per group (the MMA's m)
constexpr int MAX_NS = 6;              // stages in the ring
constexpr int MAX_PHASES = 8;
constexpr int EDGE_FLOATS = 128;       // a group's result: 16 rows x 8 tokens
// stage bytes per row: Q4_K boxes of 8 super-blocks and 16 bytes (so rows
// sit 16 bytes past a 128-byte multiple apart), Q6_K spans of 8 super-blocks
// rounded out to 16 bytes in a pitch of an odd number of 16-byte chunks

// shared-memory head: full barriers | empty barriers | activation barrier |
// failure flag | zeros (the B rows of tokens M..7) | partial sums of the
// consumer warps, two groups.  The activation rows start on a 128-byte
// boundary and are 16 bytes past a 128-byte multiple apart, so token m's
// 16-byte ldmatrix rows sit in bank group m (+ a common offset); the zero
// rows sit in bank group 7, which no token uses while M < 8.
constexpr int OFF_FULL = 0;
constexpr int OFF_EMPTY = 64;
constexpr int OFF_XBAR = 128;
constexpr int OFF_FAIL = 144;
constexpr int OFF_ZERO = 624;
constexpr int ZERO_BYTES = 512;
constexpr int OFF_PART = 1152;
static_assert(8 * MAX_NS <= 64 && OFF_ZERO + ZERO_BYTES <= OFF_PART, "head layout");
static_assert(OFF_ZERO % 128 == 112 && OFF_PART % 128 == 0, "zero rows in bank group 7");

// The kernel for CW consumer warps (warp CW is the producer): a stage is one
// group's 16 rows x CW super-blocks, one per consumer warp.  Stage bytes per
// row: Q4_K boxes of CW super-blocks and 16 bytes, Q6_K spans of CW
// super-blocks rounded out to 16 bytes; both an odd number of 16-byte
// chunks, so the 8 rows of an ldmatrix sit in 8 distinct bank groups.
template <int CW>
struct Shape {
    static constexpr int NTHREADS = (CW + 1) * 32;
    static constexpr int CHS = CW;
    static constexpr int Q4K_PITCH = CW * 144 + 16;
    static constexpr int Q6K_PITCH = ((CW * 210 + 41) / 16 | 1) * 16;
    static constexpr int HEAD = OFF_PART + 2 * CW * EDGE_FLOATS * 4;  // partial sums of two groups
    static_assert((Q4K_PITCH / 16) % 2 == 1 && (Q6K_PITCH / 16) % 2 == 1, "row pitches");
    static_assert(HEAD % 128 == 0 && Q4K_PITCH / 8 <= 256, "head and box");
};
constexpr int CW_CHOICES[2] = {8, 10};
constexpr int SB_WORDS = 144 / 8;  // a Q4_K super-block in the tensor map's 8-byte elements

// f(integral_constant<int, I>) for I = B .. E-1: the loop index is a
// compile-time constant in the body (register arrays, masks, shuffle sources)
template <int B, int E, class F>
__device__ __forceinline__ void static_for(F &&f) {
    if constexpr (B < E) {
        f(std::integral_constant<int, B>{});
        static_for<B + 1, E>(f);
    }
}

template <int T>
struct Mm;
template <>
struct Mm<QMM_Q4_K> {
    static constexpr int BB = 144;
    static constexpr int XS_TOKEN = 32;  // per super-block per token: block sums hi | lo
};
template <>
struct Mm<QMM_Q6_K> {
    static constexpr int BB = 210;
    static constexpr int XS_TOKEN = 0;   // the group sums are one array for all tokens
};

struct MmParams {
    const uint8_t *W;   // the blocks (Q6_K: per-row bulk copies)
    uint64_t w_end;     // first byte past the matrix
    int64_t N;
    int K, M;
    int nb;             // super-blocks per row
    int64_t RB;         // bytes per row
    int64_t halves_q;   // 8-row halves per CTA: halves / gridDim.x
    int halves_r;       // halves % gridDim.x: the first halves_r CTAs take one more
    const uint8_t *xh;  // quantiser output [M][2K + K/8 bytes]: x fp16 | Q4_K block sums
    const uint8_t *xs16;  // Q6_K group sums: per super-block [hi | lo][2][8 tokens][8] fp16 (x 2^-4)
    const float *xinv;    // [M] 2^-e_m: undoes the quantiser's power of two of token row m
    const float *gate;    // null, or g [M][N] from the preceding launch: y = silu(g) * (this product)
    int nphase;         // K phases
    int nbp;            // super-blocks per phase (a multiple of 8 when nphase > 1)
    int x_ld;           // bytes per token row of the activation window (= 16 mod 128)
    float *y;
    int NS;             // stages in the ring
    int stage_bytes;
    int row_pitch;      // stage bytes per row
    int off_x, off_xs, off_table, off_ring;
    int *status;
    int stop_stage;  // the first CTA's producer issues no stage from this one on (failure test hook)
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

// A 32-bit word of shared memory at a 4-byte (ODD false) or 2-byte (ODD
// true: two aligned loads shifted together) aligned address.
template <bool ODD>
__device__ __forceinline__ uint32_t word_at(const uint8_t *p) {
    if (!ODD) return *reinterpret_cast<const uint32_t *>(p);
    const uint32_t *a = reinterpret_cast<const uint32_t *>(p - 2);
    return __funnelshift_r(a[0], a[1], 16);
}

// Scales of this lane's sub-blocks t and t+4 from a Q4_K header (d, dmin,
// GGUF six-bit packing: sub-blocks 0-3 in the low six bits of bytes 0-7, 4-7
// in the nibbles of bytes 8-11 with the top bits of bytes 0-7): s0, s1 =
// d*sc_t * fs and d*sc_(t+4) * fs in fp32 (exact), fs = 2^24, or 2^20 for
// odd t (odd sub-blocks are read from the high nibbles in place as 16q);
// m01 = (-dmin*m_t, -dmin*m_(t+4)) * 2^g in fp16 with |dmin|*2^g in
// [2^8, 2^9) (g = 0 when dmin is 0), um = 2^(5-g): the factor that takes the
// min-term MMA (whose B operand carries 2^-5) back to the scale of the
// other terms.  sel picks byte t of a word under the bits 0x4B000000, which
// make it the fp32 2^23 + b; one FMA then gives b * scale exactly.
__device__ __forceinline__ void q4k_lane_scales(uint4 h, uint32_t sel, float fs, float &s0, float &s1,
                                                uint32_t &m01, float &um) {
    const float d = half_bits_to_float(h.x);
    const float dmin0 = half_bits_to_float(h.x >> 16);
    const uint32_t mb = __float_as_uint(dmin0) & 0x7fffffffu;
    const int g = mb ? 8 - exponent_of(mb) : 0;
    const float dmin = dmin0 * pow2f(g);
    um = pow2f(5 - g);
    // the six-bit scales and mins of sub-blocks 0-3 and 4-7, a byte each
    const uint32_t sc_lo = h.y & 0x3F3F3F3Fu, mn_lo = h.z & 0x3F3F3F3Fu;
    const uint32_t sc_hi = (h.w & 0x0F0F0F0Fu) | ((h.y >> 2) & 0x30303030u);
    const uint32_t mn_hi = ((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u);
    const float ds = d * fs;
    const float kd = -8388608.0f * ds;
    s0 = fmaf(__uint_as_float(__byte_perm(sc_lo, 0x4B000000u, sel)), ds, kd);
    s1 = fmaf(__uint_as_float(__byte_perm(sc_hi, 0x4B000000u, sel)), ds, kd);
    const float km = 8388608.0f * dmin;
    const float m0 = fmaf(__uint_as_float(__byte_perm(mn_lo, 0x4B000000u, sel)), -dmin, km);
    const float m1 = fmaf(__uint_as_float(__byte_perm(mn_hi, 0x4B000000u, sel)), -dmin, km);
    const __half2 m = __floats2half2_rn(m0, m1);
    m01 = *reinterpret_cast<const uint32_t *>(&m);
}

// One Q4_K super-block of the 16 rows: ra_sb = this lane's ldmatrix address
// of the weight words, hdr_a / hdr_b = the headers of rows g and g+8,
// x_sb = the lane's ldmatrix address of the activations, xs_sb = of the
// block sums.
__device__ __forceinline__ void q4k_superblock(uint32_t a_sb, const uint8_t *hdr_a, const uint8_t *hdr_b,
                                               uint32_t x_sb, uint32_t xs_sb, uint32_t sel, float fs, int quad,
                                               float (&c)[4], float (&c2)[4]) {
    float sa0, sa1, sb0, sb1, ua, ub;
    uint32_t ma, mb;
    q4k_lane_scales(*reinterpret_cast<const uint4 *>(hdr_a), sel, fs, sa0, sa1, ma, ua);
    q4k_lane_scales(*reinterpret_cast<const uint4 *>(hdr_b), sel, fs, sb0, sb1, mb, ub);
    // the min term: k slots 2t, 2t+1 = sub-blocks t, t+4 (sums hi; the
    // quantiser stores sub-block j's sums at slot 2(j mod 4) + j/4), slots
    // 2t+8, 2t+9 = the same sub-blocks (sums lo); rows g | g+8 scaled back
    // by their own factors
    {
        uint32_t xhi, xlo;
        ldsm_x2(xs_sb, xhi, xlo);
        float dm[4];
        mma_new(dm, ma, mb, ma, mb, xhi, xlo);
        c2[0] = fmaf(ua, dm[0], c2[0]);
        c2[1] = fmaf(ua, dm[1], c2[1]);
        c2[2] = fmaf(ub, dm[2], c2[2]);
        c2[3] = fmaf(ub, dm[3], c2[3]);
    }
    static_for<0, 4>([&](auto cc_) {  // quant bytes 32cc..32cc+31: sub-blocks 2cc, 2cc+1
        constexpr int cc = decltype(cc_)::value;
        uint32_t wa0, wb0, wa1, wb1;  // rows g | g+8, halves e = 0 | 1
        ldsm_x4(a_sb + 32 * cc, wa0, wb0, wa1, wb1);
        const uint32_t wa0s = wa0 >> 8, wb0s = wb0 >> 8, wa1s = wa1 >> 8, wb1s = wb1 >> 8;
        // scales of sub-blocks 2cc, 2cc+1: the first (cc < 2) or second value
        // of the quad's lanes 2cc mod 4 and 2cc+1 mod 4
        constexpr int l0 = (2 * cc) & 3, l1 = (2 * cc + 1) & 3;
        const float s_a0 = __shfl_sync(0xffffffffu, cc < 2 ? sa0 : sa1, quad | l0);
        const float s_a1 = __shfl_sync(0xffffffffu, cc < 2 ? sa0 : sa1, quad | l1);
        const float s_b0 = __shfl_sync(0xffffffffu, cc < 2 ? sb0 : sb1, quad | l0);
        const float s_b1 = __shfl_sync(0xffffffffu, cc < 2 ? sb0 : sb1, quad | l1);
        static_for<0, 2>([&](auto h_) {  // sub-block 2cc + h: low or high nibbles
            constexpr int h = decltype(h_)::value;
            constexpr uint32_t mk = h ? 0x00F000F0u : 0x000F000Fu;
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
        });
    });
}

// The int8 scales of groups G, G+1 at p (2-byte aligned) as the fp16
// subnormal pair (sc_G, sc_G+1) * 2^-24, exact: the bytes with their sign
// bits flipped are sc + 128 in the low byte of each half, and 128 * 2^-24
// is taken off.
__device__ __forceinline__ uint32_t q6k_scale_pair(const uint8_t *p) {
    const uint32_t v = *reinterpret_cast<const uint16_t *>(p) ^ 0x8080u;
    const uint32_t u = __byte_perm(v, 0u, 0x4140);
    const __half2 k128 = __half2half2(__ushort_as_half(0x0080));
    const __half2 r = __hsub2(*reinterpret_cast<const __half2 *>(&u), k128);
    return *reinterpret_cast<const uint32_t *>(&r);
}

// One Q6_K super-block of the 16 rows: ra / rb = its bytes for rows g and
// g+8 (2-byte aligned when ODD), x_sb = the lane's ldmatrix address of the
// activations, xg_sb = the lane's ldmatrix address of the group-sum tiles.
template <bool ODD>
__device__ __forceinline__ void q6k_superblock(const uint8_t *ra, const uint8_t *rb, uint32_t x_sb,
                                               uint32_t xg_sb, int t, int quad, float (&c)[4], float (&c2)[4]) {
    // scales of groups 4t..4t+3 for rows g and g+8: d*sc * 2^24 / f, f = 16
    // for the groups read from high nibbles (groups 4..7 and 12..15: t odd)
    const float fs = (t & 1) ? 1048576.0f : 16777216.0f;
    const float da = __half2float(*reinterpret_cast<const __half *>(ra + 208)) * fs;
    const float db = __half2float(*reinterpret_cast<const __half *>(rb + 208)) * fs;
    const uint32_t sca = word_at<ODD>(ra + 192 + 4 * t), scb = word_at<ODD>(rb + 192 + 4 * t);
    float Sa[4], Sb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        Sa[i] = da * static_cast<float>(static_cast<int8_t>(sca >> (8 * i)));
        Sb[i] = db * static_cast<float>(static_cast<int8_t>(scb >> (8 * i)));
    }
    // the offset: -32 d sum_G sc_G X_G, one MMA per plane of the group sums
    // (k slots = groups: A = sc * 2^-24, B = X * 2^-4 as hi and lo), so the
    // result times -32 d 2^28
    {
        uint32_t xhi0, xhi1, xlo0, xlo1;
        ldsm_x4(xg_sb, xhi0, xhi1, xlo0, xlo1);
        const uint32_t a0 = q6k_scale_pair(ra + 192 + 2 * t), a1 = q6k_scale_pair(rb + 192 + 2 * t);
        const uint32_t a2 = q6k_scale_pair(ra + 200 + 2 * t), a3 = q6k_scale_pair(rb + 200 + 2 * t);
        float r[4];
        mma_new(r, a0, a1, a2, a3, xhi0, xhi1);
        mma_acc(r, a0, a1, a2, a3, xlo0, xlo1);
        const float ka = __half2float(*reinterpret_cast<const __half *>(ra + 208)) * -8589934592.0f;
        const float kb = __half2float(*reinterpret_cast<const __half *>(rb + 208)) * -8589934592.0f;
        c[0] = fmaf(ka, r[0], c[0]);
        c[1] = fmaf(ka, r[1], c[1]);
        c[2] = fmaf(kb, r[2], c[2]);
        c[3] = fmaf(kb, r[3], c[3]);
    }
    static_for<0, 2>([&](auto n_) {  // weights 128n .. 128n+127
        constexpr int n = decltype(n_)::value;
        // quant words of this lane for l = 16lh + 4t .. +3: low fields (q1,
        // q3: ql bytes 64n + l), (q2, q4: 64n + 32 + l), high fields 128 + 32n + l
        uint32_t la[2][2], lb[2][2], ha[2], hb[2];
        static_for<0, 2>([&](auto lh_) {
            constexpr int lh = decltype(lh_)::value;
            la[lh][0] = word_at<ODD>(ra + 64 * n + 16 * lh + 4 * t);
            la[lh][1] = word_at<ODD>(ra + 64 * n + 32 + 16 * lh + 4 * t);
            lb[lh][0] = word_at<ODD>(rb + 64 * n + 16 * lh + 4 * t);
            lb[lh][1] = word_at<ODD>(rb + 64 * n + 32 + 16 * lh + 4 * t);
            ha[lh] = word_at<ODD>(ra + 128 + 32 * n + 16 * lh + 4 * t);
            hb[lh] = word_at<ODD>(rb + 128 + 32 * n + 16 * lh + 4 * t);
        });
        static_for<0, 4>([&](auto qi_) {  // weights 128n + 32qi + l
            constexpr int qi = decltype(qi_)::value;
            uint32_t x0, x1, x2, x3;  // the 32-block 4n + qi: halves lh = 0 | 1
            ldsm_x4(x_sb + 64 * (4 * n + qi), x0, x1, x2, x3);
            constexpr uint32_t mlo = qi >= 2 ? 0x00F000F0u : 0x000F000Fu;
            constexpr uint32_t mhi = 0x00030003u << (2 * qi);
            constexpr uint32_t mul = (qi & 1) ? 4u : 16u;
            static_for<0, 2>([&](auto lh_) {
                constexpr int lh = decltype(lh_)::value;
                constexpr int G = 8 * n + 2 * qi + lh;
                const uint32_t qla = la[lh][qi & 1], qlb = lb[lh][qi & 1];
                const uint32_t a0 = (ha[lh] & mhi) * mul + (qla & mlo);
                const uint32_t a1 = (hb[lh] & mhi) * mul + (qlb & mlo);
                const uint32_t a2 = ((ha[lh] >> 8) & mhi) * mul + ((qla >> 8) & mlo);
                const uint32_t a3 = ((hb[lh] >> 8) & mhi) * mul + ((qlb >> 8) & mlo);
                float d[4];
                mma_new(d, a0, a1, a2, a3, lh ? x2 : x0, lh ? x3 : x1);
                const float sa = __shfl_sync(0xffffffffu, Sa[G & 3], quad | (G >> 2));
                const float sb = __shfl_sync(0xffffffffu, Sb[G & 3], quad | (G >> 2));
                float(&acc)[4] = lh ? c2 : c;
                acc[0] = fmaf(sa, d[0], acc[0]);
                acc[1] = fmaf(sa, d[1], acc[1]);
                acc[2] = fmaf(sb, d[2], acc[2]);
                acc[3] = fmaf(sb, d[3], acc[3]);
            });
        });
    });
}

// Stage s of the CTA (phase p, group gi, chunk kc), in the order the
// producer fills the ring and the consumers use it.
struct StageCursor {
    int p, gi, kc;
    int sb, nsb;  // the phase's first super-block and its count
    int nq;       // chunks per row in the phase
};

template <int CHS>
__device__ __forceinline__ void cursor_phase(const MmParams &P, StageCursor &c, int p) {
    c.p = p;
    c.gi = 0;
    c.kc = 0;
    c.sb = p * P.nbp;
    c.nsb = min(P.nbp, P.nb - c.sb);
    c.nq = (c.nsb + CHS - 1) / CHS;
}

template <int CHS>
__device__ __forceinline__ void cursor_next(const MmParams &P, StageCursor &c, int ng) {
    if (++c.kc == c.nq) {
        c.kc = 0;
        if (++c.gi == ng) cursor_phase<CHS>(P, c, c.p + 1);
    }
}

// The work of CTA `cta` of one matrix (tmW: its Q4_K tensor map).
template <int T, int CW>
__device__ __forceinline__ void mma_body(const CUtensorMap *tmW, const MmParams &P, const int cta) {
    constexpr int NTHREADS = Shape<CW>::NTHREADS, CHS = Shape<CW>::CHS;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // this CTA's rows [r0, r1): whole 8-row halves; groups of 16 from r0
    const int64_t h0 = P.halves_q * cta + min(cta, P.halves_r);
    const int nh = static_cast<int>(P.halves_q + (cta < P.halves_r ? 1 : 0));
    const int64_t r0 = 8 * h0;
    const int64_t r1 = min(P.N, 8 * (h0 + nh));
    const int ng = (nh + 1) / 2;
    int total = 0;  // stages of the CTA
    for (int p = 0; p < P.nphase; ++p) {
        const int nsb = min(P.nbp, P.nb - p * P.nbp);
        total += ng * ((nsb + CHS - 1) / CHS);
    }

    const uint32_t full0 = smem_u32(smem + OFF_FULL), empty0 = smem_u32(smem + OFF_EMPTY);
    const uint32_t xbar = smem_u32(smem + OFF_XBAR);
    volatile int *fail_flag = reinterpret_cast<volatile int *>(smem + OFF_FAIL);
    float *part = reinterpret_cast<float *>(smem + OFF_PART);
    float *table = reinterpret_cast<float *>(smem + P.off_table);
    if (threadIdx.x == 0) {
        for (int i = 0; i < P.NS; ++i) {
            mbar_init(full0 + 8u * i, 1);
            mbar_init(empty0 + 8u * i, CW);
        }
        mbar_init(xbar, 1);
        fence_mbar_init();
        *fail_flag = 0;
    }
    if (threadIdx.x < ZERO_BYTES / 16)
        reinterpret_cast<uint4 *>(smem + OFF_ZERO)[threadIdx.x] = make_uint4(0u, 0u, 0u, 0u);
    if (P.nphase > 1)
        for (int i = threadIdx.x; i < ng * EDGE_FLOATS; i += NTHREADS) table[i] = 0.0f;
    __syncthreads();
    pdl_trigger();
    const uint64_t pol = policy_evict_first();

    // the activation window of phase p (one thread): x rows, then the sums
    auto load_x = [&](int p) {
        const int K = P.K;
        const int sb = p * P.nbp, nsb = min(P.nbp, P.nb - sb);
        const uint32_t xb = static_cast<uint32_t>(512 * nsb);
        const uint32_t xsb = static_cast<uint32_t>((T == QMM_Q4_K ? 32 : 512) * nsb);
        mbar_arrive_expect_tx(xbar, P.M * xb + (T == QMM_Q4_K ? P.M : 1) * xsb);
        const uint8_t *src_row = P.xh;
        for (int m = 0; m < P.M; ++m, src_row += 2 * K + K / 8) {
            const uint32_t dst = smem_u32(smem + P.off_x + m * P.x_ld);
            bulk_g2s(dst, src_row + static_cast<int64_t>(512) * sb, xb, xbar, pol);
            if (T == QMM_Q4_K)
                bulk_g2s(dst + 512 * P.nbp, src_row + 2 * K + static_cast<int64_t>(32) * sb, xsb, xbar, pol);
        }
        if (T == QMM_Q6_K) bulk_g2s(smem_u32(smem + P.off_xs), P.xs16 + static_cast<int64_t>(512) * sb, xsb, xbar, pol);
    };

    if (warp == CW) {
        // ---- producer: fills the ring in stage order --------------------
        StageCursor c;
        cursor_phase<CHS>(P, c, 0);
        // stages from `stop` on are never issued (only with the test hook:
        // the consumers' bounded wait on stage `stop` then expires)
        const int stop = cta == 0 ? P.stop_stage : NO_STOP;
        int issued = 0;
        for (int s = 0; s < total; ++s, cursor_next<CHS>(P, c, ng)) {
            const int slot = s % P.NS;
            if (s >= P.NS) {
                // the consumers' release of this slot's previous stage
                bool ok = true;
                if (lane == 0) ok = mbar_wait(empty0 + 8u * slot, static_cast<uint32_t>((s / P.NS - 1) & 1), P.status);
                if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
                    if (lane == 0) *fail_flag = 1;
                    break;
                }
            }
            if (s >= stop) break;
            issued = s + 1;
            const int sb0 = c.sb + c.kc * CHS, nsb = min(CHS, c.sb + c.nsb - sb0);
            const int64_t row0 = r0 + GR * c.gi;
            const uint32_t bar = full0 + 8u * slot;
            const uint32_t dst = smem_u32(smem + P.off_ring) + slot * P.stage_bytes;
            if constexpr (T == QMM_Q4_K) {
                // rows 0..7 of the group, and 8..15 when the CTA owns them (a
                // CTA's rows end on a half or at N); a box is 8 super-blocks
                // and 16 bytes (rows 16 bytes past a 128-byte multiple apart)
                if (lane == 0) {
                    const int boxes = r1 - row0 > 8 ? 2 : 1;
                    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(boxes * 8 * P.row_pitch));
                    for (int bx = 0; bx < boxes; ++bx)
                        tma_load_2d_hint(dst + bx * 8 * P.row_pitch, tmW, sb0 * SB_WORDS,
                                         static_cast<int>(row0 + 8 * bx), bar, pol);
                }
            } else {
                // lane r copies row r's span rounded out to 16 bytes (never past
                // the end of the matrix)
                const int64_t left = r1 - row0;
                const int rows = left < GR ? static_cast<int>(left) : GR;
                uint64_t src = 0;
                uint32_t bytes = 0;
                if (lane < rows) {
                    const uint64_t start = reinterpret_cast<uint64_t>(P.W) + static_cast<uint64_t>(row0 + lane) * P.RB +
                                           static_cast<uint64_t>(210) * sb0;
                    src = start & ~uint64_t(15);
                    uint64_t end = (start + static_cast<uint64_t>(210) * nsb + 15) & ~uint64_t(15);
                    if (end > P.w_end) end = P.w_end & ~uint64_t(15);
                    bytes = static_cast<uint32_t>(end - src);
                }
                const uint32_t all = __reduce_add_sync(0xffffffffu, bytes);
                if (lane == 0) mbar_arrive_expect_tx(bar, all);
                if (bytes > 0)
                    bulk_g2s(dst + lane * P.row_pitch, reinterpret_cast<const void *>(src), bytes, bar, pol);
            }
            if (s == 0) {
                // the first stage before the wait for the quantiser (see the
                // header); the activations next, the other stages after them
                pdl_wait();
                if (lane == 0) load_x(0);
            }
        }
        if (total == 0) {
            pdl_wait();
            if (lane == 0) load_x(0);
        }
        // no copy may still be in flight when the CTA exits (stages that were
        // never issued are not waited for)
        if (lane == 0)
            for (int s = max(0, issued - P.NS); s < issued; ++s)
                mbar_wait(full0 + 8u * (s % P.NS), static_cast<uint32_t>((s / P.NS) & 1), P.status);
        return;
    }

    // ---- consumers: warp w takes super-block (w + kc) mod 8 of each stage ---
    pdl_wait();  // y is written after the kernels before the quantiser completed
    const int g = lane >> 2, t = lane & 3;
    const int quad = lane & ~3;
    // ldmatrix row addresses of this lane (it names row lane & 7 of matrix lane >> 3)
    const int lr = lane & 7, lm = lane >> 3;
    // Q4_K weights: matrices (rows 0-7 | 8-15) x (16-byte segment 2c | 2c + 1)
    const uint32_t a_off = static_cast<uint32_t>((lr + 8 * (lm & 1)) * P.row_pitch + 16 + 16 * (lm >> 1));
    // activations of token lr: matrices (half e, B register) of one 32-block;
    // Q4_K block sums (hi | lo); tokens >= M read zeros
    const bool tok_ok = lr < P.M;
    const uint32_t x_row = smem_u32(smem + P.off_x + lr * P.x_ld);
    const uint32_t zero = smem_u32(smem + OFF_ZERO);
    const uint32_t x_base = (tok_ok ? x_row : zero) + 16 * lm;
    const uint32_t xs_base = (tok_ok ? x_row + 512 * P.nbp : zero) + 16 * (lm & 1);
    const uint32_t x_step = tok_ok ? 512u : 0u, xs_step = tok_ok ? 32u : 0u;  // per super-block
    // Q4_K scale decode of this lane (sub-blocks t and t+4): the byte selector
    // and the fp32 factor of its nibble half
    const uint32_t q4k_sel = 0x7650u + static_cast<uint32_t>(t);
    const float q4k_fs = (t & 1) ? 1048576.0f : 16777216.0f;
    // Q6_K group-sum tiles: lane l reads row l & 7 of matrix l >> 3 (16 bytes each)
    const uint32_t xg_base = smem_u32(smem + P.off_xs) + 16 * lane;
    const int tid = threadIdx.x;  // 0 .. 255

    // an element of a group's 16 x 8 result in fragment order -> y
    auto store_y = [&](int gi, int e, float v) {
        const int ln = e >> 2, i = e & 3;
        const int64_t row = r0 + GR * gi + (ln >> 2) + 8 * (i >> 1);
        const int tk = 2 * (ln & 3) + (i & 1);
        if (row < r1 && tk < P.M) {
            float val = v * __ldg(P.xinv + tk);
            if (P.gate) {
                // gate.x, written by the launch before this one (complete:
                // the consumers passed griddepcontrol.wait)
                const float g = P.gate[static_cast<int64_t>(tk) * P.N + row];
                val = g / (1.0f + expf(-g)) * val;
            }
            P.y[static_cast<int64_t>(tk) * P.N + row] = val;
        }
    };

    bool failed = false;
    int s = 0;
    for (int p = 0; p < P.nphase; ++p) {
        StageCursor c;
        cursor_phase<CHS>(P, c, p);
        if (p > 0) {
            // every consumer is done with the previous window
            named_barrier(1, CW * 32);
            if (tid == 0 && *fail_flag == 0) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                load_x(p);
            }
        }
        if (!failed && !__all_sync(0xffffffffu, mbar_wait(xbar, static_cast<uint32_t>(p & 1), P.status)))
            failed = true;
        for (int gi = 0; gi < ng; ++gi) {
            float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f}, acc2[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            for (int kc = 0; kc < c.nq; ++kc, ++s) {
                const int slot = s % P.NS;
                if (!failed && !__all_sync(0xffffffffu, mbar_wait(full0 + 8u * slot,
                                                                    static_cast<uint32_t>((s / P.NS) & 1), P.status)))
                    failed = true;
                const int sb0 = c.sb + kc * CHS, nsb = min(CHS, c.sb + c.nsb - sb0);
                const int idx = (warp + kc) % CHS;
                const uint8_t *st = smem + P.off_ring + slot * P.stage_bytes;
                if (!failed && idx < nsb) {
                    const int kw = sb0 + idx - c.sb;  // super-block inside the window
                    if constexpr (T == QMM_Q4_K) {
                        q4k_superblock(smem_u32(st) + a_off + 144 * idx, st + g * P.row_pitch + 144 * idx,
                                       st + (g + 8) * P.row_pitch + 144 * idx, x_base + kw * x_step,
                                       xs_base + kw * xs_step, q4k_sel, q4k_fs, quad, acc, acc2);
                    } else {
                        const int64_t row0 = r0 + GR * gi;
                        const uint64_t base = reinterpret_cast<uint64_t>(P.W) + static_cast<uint64_t>(210) * sb0;
                        const int oa = static_cast<int>((base + static_cast<uint64_t>(row0 + g) * P.RB) & 15);
                        const int ob = static_cast<int>((base + static_cast<uint64_t>(row0 + g + 8) * P.RB) & 15);
                        // the matrix's last bytes, not copied: loaded here by the
                        // warp that reads them (the last row's last super-block)
                        if (sb0 + idx == P.nb - 1 && r1 == P.N && row0 + GR >= P.N && (P.w_end & 15) != 0) {
                            const int rl = static_cast<int>(P.N - 1 - row0);
                            const uint64_t start = base + static_cast<uint64_t>(P.N - 1) * P.RB;
                            const uint64_t copied = (P.w_end & ~uint64_t(15)) - (start & ~uint64_t(15));
                            const int tail = static_cast<int>(P.w_end & 15);
                            if (lane < tail / 4) {
                                const uint32_t v = __ldg(reinterpret_cast<const unsigned int *>(
                                    (P.w_end & ~uint64_t(15)) + 4 * lane));
                                *reinterpret_cast<uint32_t *>(const_cast<uint8_t *>(st) + rl * P.row_pitch + copied +
                                                              4 * lane) = v;
                            }
                            __syncwarp();
                        }
                        const uint8_t *ra = st + g * P.row_pitch + oa + 210 * idx;
                        const uint8_t *rb = st + (g + 8) * P.row_pitch + ob + 210 * idx;
                        if (idx & 1)
                            q6k_superblock<true>(ra, rb, x_base + kw * x_step, xg_base + 512 * kw, t, quad, acc, acc2);
                        else
                            q6k_superblock<false>(ra, rb, x_base + kw * x_step, xg_base + 512 * kw, t, quad, acc, acc2);
                    }
                }
                // this warp is done with the stage
                __syncwarp();
                if (lane == 0) mbar_arrive(empty0 + 8u * slot);
            }
            // the group's phase result: the warps' partial sums added in warp order
            float *pb = part + (gi & 1) * (CW * EDGE_FLOATS);
            *reinterpret_cast<float4 *>(pb + warp * EDGE_FLOATS + 4 * lane) =
                make_float4(acc[0] + acc2[0], acc[1] + acc2[1], acc[2] + acc2[2], acc[3] + acc2[3]);
            if (failed && lane == 0) *fail_flag = 1;
            named_barrier(2, CW * 32);
            if (tid < EDGE_FLOATS && *fail_flag == 0) {
                float v = 0.0f;
#pragma unroll
                for (int w = 0; w < CW; ++w) v += pb[w * EDGE_FLOATS + tid];
                if (P.nphase == 1) store_y(gi, tid, v);
                else table[gi * EDGE_FLOATS + tid] += v;
            }
        }
    }
    if (tid == 0 && P.nphase > 0) mbar_wait(xbar, static_cast<uint32_t>((P.nphase - 1) & 1), P.status);
    if (P.nphase == 1) return;
    named_barrier(1, CW * 32);
    if (*fail_flag != 0) return;
    for (int e = tid; e < ng * EDGE_FLOATS; e += CW * 32) store_y(e / EDGE_FLOATS, e % EDGE_FLOATS, table[e]);
}

template <int T, int CW>
__global__ void __launch_bounds__(Shape<CW>::NTHREADS, 1)
    gemv_mma_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ MmParams P) {
    mma_body<T, CW>(&tmW, P, static_cast<int>(blockIdx.x));
}

// Several matrices that share K and the quantised x in one launch: CTAs
// [cta_begin[i], cta_begin[i+1]) work on matrix i, each with its own
// shared-memory plan (the launch has the largest).
struct MmGroup {
    CUtensorMap tm[QMM_GROUP_MAX];  // the Q4_K entries' tensor maps
    MmParams p[QMM_GROUP_MAX];
    int type[QMM_GROUP_MAX];
    int cta_begin[QMM_GROUP_MAX + 1];
    int n;
};

// Q6K: the launch holds a Q6_K matrix (else Q4_K only)
template <int CW, bool Q6K>
__global__ void __launch_bounds__(Shape<CW>::NTHREADS, 1) gemv_mma_group_kernel(const __grid_constant__ MmGroup G) {
    int i = 0;
    while (i + 1 < G.n && static_cast<int>(blockIdx.x) >= G.cta_begin[i + 1]) ++i;
    const int cta = static_cast<int>(blockIdx.x) - G.cta_begin[i];
    if (!Q6K || G.type[i] == QMM_Q4_K) mma_body<QMM_Q4_K, CW>(&G.tm[i], G.p[i], cta);
    else mma_body<QMM_Q6_K, CW>(&G.tm[i], G.p[i], cta);
}

// Shared-memory plan: head | activation window [M][x_ld] | Q6_K group sums
// window | phase table | ring of NS stages of GR rows x CW super-blocks.  The
// fewest phases that fit with at least two stages.
struct Plan {
    int NS, nphase, nbp, x_ld, row_pitch, stage_bytes, off_x, off_xs, off_table, off_ring, smem;
};

template <int T, int CW>
bool plan_mm(int M, int64_t K, int64_t max_groups, int max_smem, Plan &pl) {
    using S = Shape<CW>;
    constexpr int CHS = S::CHS, HEAD = S::HEAD;
    const int nb = static_cast<int>(K / 256);
    const int pitch = T == QMM_Q4_K ? S::Q4K_PITCH : S::Q6K_PITCH;
    const int64_t stage = static_cast<int64_t>(GR) * pitch;
    for (int P = 1; P <= MAX_PHASES; ++P) {
        int nbp = nb;
        if (P > 1) {
            nbp = (nb + P - 1) / P;
            nbp = (nbp + CHS - 1) / CHS * CHS;
            if (static_cast<int64_t>(nbp) * (P - 1) >= nb) continue;  // an empty last phase
        }
        const int64_t x_ld = (static_cast<int64_t>(nbp) * (512 + Mm<T>::XS_TOKEN) + 127) / 128 * 128 + 16;
        const int64_t o_x = HEAD;
        const int64_t o_xs = (o_x + M * x_ld + 127) / 128 * 128;
        const int64_t o_table = o_xs + (T == QMM_Q6_K ? static_cast<int64_t>(nbp) * 512 : 0);
        const int64_t o_ring = (o_table + (P > 1 ? max_groups * EDGE_FLOATS * 4 : 0) + 127) / 128 * 128;
        int64_t ns = (max_smem - o_ring) / stage;
        if (ns < 2) continue;
        if (ns > MAX_NS) ns = MAX_NS;
        pl = {static_cast<int>(ns), P, nbp, static_cast<int>(x_ld), pitch, static_cast<int>(stage),
              static_cast<int>(o_x), static_cast<int>(o_xs), static_cast<int>(o_table), static_cast<int>(o_ring),
              static_cast<int>(o_ring + ns * stage)};
        return true;
    }
    return false;
}

int64_t max_groups_of(int64_t N, int num_sms, int64_t *grid_out) {
    const int64_t halves = (N + 7) / 8;
    int64_t grid = num_sms;
    if (grid > halves) grid = halves;
    if (grid < 1) grid = 1;
    if (grid_out) *grid_out = grid;
    return (halves / grid + 2) / 2;
}

bool type_ok(int type, int M, int64_t K, int64_t N) {
    if (M < 2 || M > 8 || K < 256 || K % 256 || K > (1 << 20) || N < 1 || N > (int64_t(1) << 30)) return false;
    if (type == QMM_Q4_K) return tensor_map_encoder() != nullptr;
    if (type == QMM_Q6_K) return (K / 256) % 2 == 0;
    return false;
}

// Consumer warps (= super-blocks per stage): the count of CW_CHOICES that
// leaves the fewest empty slots in a row's stages, the larger on a tie.
int consumer_warps(int64_t K) {
    const int64_t nb = K / 256;
    int best = CW_CHOICES[0];
    int64_t best_slots = -1;
    for (int cw : CW_CHOICES) {
        const int64_t slots = (nb + cw - 1) / cw * cw;
        if (best_slots < 0 || slots <= best_slots) {
            best = cw;
            best_slots = slots;
        }
    }
    return best;
}

bool plan_for(int type, int cw, int M, int64_t K, int64_t mg, int max_smem, Plan &pl) {
    if (type == QMM_Q4_K)
        return cw == 10 ? plan_mm<QMM_Q4_K, 10>(M, K, mg, max_smem, pl) : plan_mm<QMM_Q4_K, 8>(M, K, mg, max_smem, pl);
    return cw == 10 ? plan_mm<QMM_Q6_K, 10>(M, K, mg, max_smem, pl) : plan_mm<QMM_Q6_K, 8>(M, K, mg, max_smem, pl);
}

// The launch arguments of one matrix split over `grid` CTAs (one per 8-row
// half at most) with the plan pl; tm receives the Q4_K tensor map.
cudaError_t fill_mm(MmParams &P, CUtensorMap &tm, int type, const void *W, int64_t N, int64_t K, const void *xh,
                    int M, float *y, int *status, const float *gate, int64_t grid, const Plan &pl) {
    const int nb = static_cast<int>(K / 256);
    const int bb = type == QMM_Q4_K ? Mm<QMM_Q4_K>::BB : Mm<QMM_Q6_K>::BB;
    P = {};
    P.W = static_cast<const uint8_t *>(W);
    P.RB = static_cast<int64_t>(nb) * bb;
    P.w_end = reinterpret_cast<uint64_t>(W) + static_cast<uint64_t>(N) * P.RB;
    P.N = N;
    P.K = static_cast<int>(K);
    P.M = M;
    P.nb = nb;
    const int64_t halves = (N + 7) / 8;
    P.halves_q = halves / grid;
    P.halves_r = static_cast<int>(halves % grid);
    P.xh = static_cast<const uint8_t *>(xh);
    P.xs16 = P.xh + static_cast<int64_t>(M) * (2 * K + K / 8);
    P.xinv = reinterpret_cast<const float *>(P.xs16 + 2 * K);
    P.gate = gate;
    P.nphase = pl.nphase;
    P.nbp = pl.nbp;
    P.x_ld = pl.x_ld;
    P.y = y;
    P.NS = pl.NS;
    P.stage_bytes = pl.stage_bytes;
    P.row_pitch = pl.row_pitch;
    P.off_x = pl.off_x;
    P.off_xs = pl.off_xs;
    P.off_table = pl.off_table;
    P.off_ring = pl.off_ring;
    P.status = status;
    P.stop_stage = NO_STOP;
    tm = {};
    if (type == QMM_Q4_K) {
        // the weights as 8-byte elements [N][18 * nb]: boxes of CW super-blocks
        // and 2 elements (the next header, or zeros past the row end) x 8 rows
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(nb) * SB_WORDS, static_cast<cuuint64_t>(N)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(nb) * 144};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(pl.row_pitch / 8), 8u};
        const cuuint32_t es[2] = {1, 1};
        if (tensor_map_encoder()(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void *>(W), dims, strides, box,
                                 es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    return cudaSuccess;
}

template <class Kern, class... Args>
cudaError_t launch_mm(Kern kern, int64_t grid, int cw, int smem, cudaStream_t st, const Args &...args) {
    cudaError_t e = set_smem_attrs(kern, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3((cw + 1) * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace

bool gemv_mma_fits(int type, int M, int64_t N, int64_t K, int max_smem, int num_sms) {
    if (!type_ok(type, M, K, N)) return false;
    const int64_t mg = max_groups_of(N, num_sms, nullptr);
    Plan pl;
    return plan_for(type, consumer_warps(K), M, K, mg, max_smem, pl);
}

cudaError_t launch_gemv_mma(int type, const void *W, int64_t N, int64_t K, const void *xh, int M, float *y,
                            cudaStream_t st, int num_sms, int max_smem, int *status, const float *gate) {
    if (!type_ok(type, M, K, N)) return cudaErrorNotSupported;
    int64_t grid = 0;
    const int64_t mg = max_groups_of(N, num_sms, &grid);
    const int cw = consumer_warps(K);
    Plan pl;
    if (!plan_for(type, cw, M, K, mg, max_smem, pl)) return cudaErrorNotSupported;
    // a CTA's stages count in int
    if (mg * ((K / 256 + cw - 1) / cw + pl.nphase) > (int64_t(1) << 30)) return cudaErrorInvalidValue;
    MmParams P;
    CUtensorMap tmW;
    cudaError_t e = fill_mm(P, tmW, type, W, N, K, xh, M, y, status, gate, grid, pl);
    if (e != cudaSuccess) return e;
    P.stop_stage = inject_stop_stage();
    auto kern = type == QMM_Q4_K ? (cw == 10 ? gemv_mma_kernel<QMM_Q4_K, 10> : gemv_mma_kernel<QMM_Q4_K, 8>)
                                 : (cw == 10 ? gemv_mma_kernel<QMM_Q6_K, 10> : gemv_mma_kernel<QMM_Q6_K, 8>);
    return launch_mm(kern, grid, cw, pl.smem, st, tmW, P);
}

cudaError_t launch_gemv_mma_group(int n, const int *types, const void *const *Ws, const int64_t *Ns, int64_t K,
                                  const void *xh, int M, float *const *ys, cudaStream_t st, int num_sms,
                                  int max_smem, int *status) {
    if (n < 1 || n > QMM_GROUP_MAX) return cudaErrorInvalidValue;
    const int cw = consumer_warps(K);
    int idx[QMM_GROUP_MAX], m = 0;
    int64_t bytes[QMM_GROUP_MAX], halves[QMM_GROUP_MAX], need[QMM_GROUP_MAX];
    bool q6k = false;
    for (int i = 0; i < n; ++i) {
        if (Ns[i] <= 0) continue;  // an empty matrix gets no CTA
        if (!type_ok(types[i], M, K, Ns[i])) return cudaErrorNotSupported;
        q6k = q6k || types[i] == QMM_Q6_K;
        bytes[m] = Ns[i] * (K / 256) * (types[i] == QMM_Q4_K ? Mm<QMM_Q4_K>::BB : Mm<QMM_Q6_K>::BB);
        halves[m] = (Ns[i] + 7) / 8;
        need[m] = 1;
        idx[m++] = i;
    }
    if (m == 0) return cudaSuccess;
    int g[QMM_GROUP_MAX];
    group_ctas(m, bytes, halves, need, num_sms, g);
    MmGroup G = {};
    G.n = m;
    int64_t grid = 0;
    int smem = 0;
    for (int j = 0; j < m; ++j) {
        const int i = idx[j];
        const int64_t mg = (halves[j] / g[j] + 2) / 2;
        Plan pl;
        if (!plan_for(types[i], cw, M, K, mg, max_smem, pl)) return cudaErrorNotSupported;
        if (mg * ((K / 256 + cw - 1) / cw + pl.nphase) > (int64_t(1) << 30)) return cudaErrorInvalidValue;
        cudaError_t e = fill_mm(G.p[j], G.tm[j], types[i], Ws[i], Ns[i], K, xh, M, ys[i], status, nullptr, g[j], pl);
        if (e != cudaSuccess) return e;
        G.type[j] = types[i];
        G.cta_begin[j] = static_cast<int>(grid);
        grid += g[j];
        if (pl.smem > smem) smem = pl.smem;
    }
    G.cta_begin[m] = static_cast<int>(grid);
    G.p[0].stop_stage = inject_stop_stage();
    if (q6k)
        return cw == 10 ? launch_mm(gemv_mma_group_kernel<10, true>, grid, cw, smem, st, G)
                        : launch_mm(gemv_mma_group_kernel<8, true>, grid, cw, smem, st, G);
    return cw == 10 ? launch_mm(gemv_mma_group_kernel<10, false>, grid, cw, smem, st, G)
                    : launch_mm(gemv_mma_group_kernel<8, false>, grid, cw, smem, st, G);
}

}  // namespace qk
