// gemv_sb.cuh -- the block-per-lane decode kernel (see gemv_sb.cu for the
// design): its device code and launch templates, shared by the translation
// units that instantiate it for different block types (gemv_sb.cu: Q8_0,
// Q4_K, Q6_K; gemv_sb_kq.cu: Q5_K, Q3_K, Q2_K), so they compile in parallel.
#pragma once

#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qk {
namespace sbk {


constexpr int NWARP = 12;
constexpr int NTHREADS = NWARP * 32;
constexpr int SU = 32;           // blocks per stage (one per lane)
constexpr int HEAD_BYTES = 2048; // mbarriers and warp-edge records
constexpr int MAX_NSW = 6;
constexpr int XPITCH = 272;      // shared-memory bytes per super-block of activations

struct SbParams {
    int type;             // qmm_type of W
    const uint8_t *W;
    int64_t total_bytes;  // N * RB
    int64_t N;
    int K, M;
    int nb;  // blocks per row
    int RB;  // bytes per row
    int NSW, slot_bytes;
    uint32_t nb_magic;  // floor(2^32 / nb) + 1 when u / nb == umulhi(u, nb_magic) for every
                        // block index u of a CTA (u * nb < 2^32), else 0 (divide)
    int64_t rows_q;  // N / (CTAs of this matrix)
    int rows_r;      // N % (CTAs of this matrix): the first rows_r CTAs take one row more
    const float *x;  // [M][K] activations, fp32
    int x_vec;       // x is 16-byte aligned: load four at a time
    int q_ld;        // bytes per activation row of q (super-blocks at XPITCH bytes)
    int meta_ld;     // bytes per activation row of scale records (Q8_0: of d)
    float *y;
    int off_edge, off_xq, off_meta, off_ring;
    int *status;
    int stop_stage;  // the first CTA's warps issue no stage from this one on (failure test hook)
    // gate+up launch: W is the gate matrix, W2 the up matrix (same type and
    // shape), y receives h = silu(gate.x) * (up.x); off_tab is the
    // shared-memory table of the CTA's row results [2][rows][MT]
    const uint8_t *W2;
    int off_tab;
};

__device__ __forceinline__ uint4 ld16(const uint8_t *sm, int off) {
    return *reinterpret_cast<const uint4 *>(sm + off);
}

// n consecutive 32-bit words at byte offset `off` of shared memory (any
// alignment): aligned words loaded and funnel-shifted into place.
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

__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {
    return __dp4a(static_cast<int>(a), static_cast<int>(b), c);
}

// a as four unsigned bytes, b as four signed bytes
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Shared-memory activations.  q: int8, super-block kb of row m at
// m*q_ld + kb*XPITCH: the 16 spare bytes per super-block put the same chunk
// of consecutive super-blocks (read by consecutive lanes) in distinct banks,
// and every chunk is an immediate offset from the super-block's start.  Per super-block kb of row m, a record at meta + m*meta_ld +
// kb*REC holds the eight block scales d (bytes 0..31) and, for Q4_K, the
// eight products d*sum (32..63) or, for Q6_K, the sixteen half-block sums
// (32..95); REC = 80 (Q4_K) or 112 (Q6_K) bytes, odd multiples of 16 so that
// lanes reading consecutive super-blocks hit distinct banks.  Q8_0 keeps a
// plain array of block scales.
template <int T> struct Rec { static constexpr int B = 0; };
template <> struct Rec<QMM_Q4_K> { static constexpr int B = 80; };
template <> struct Rec<QMM_Q6_K> { static constexpr int B = 112; };
// Q5_K takes Q4_K's records (scale and d*sum per 32), Q3_K and Q2_K Q6_K's
// (scale and the two 16-element sums per 32)
template <> struct Rec<QMM_Q5_K> { static constexpr int B = 80; };
template <> struct Rec<QMM_Q3_K> { static constexpr int B = 112; };
template <> struct Rec<QMM_Q2_K> { static constexpr int B = 112; };
template <int T> constexpr bool kRecDs = T == QMM_Q4_K || T == QMM_Q5_K;
template <int T> constexpr bool kRecHalves = T == QMM_Q6_K || T == QMM_Q3_K || T == QMM_Q2_K;

struct XS {
    const uint8_t *sm;
    int xq, meta;
    int q_ld, meta_ld;
};

// Shared-memory byte offset of 16-byte chunk c of super-block kb, row m.
__device__ __forceinline__ int xchunk(const XS &X, int m, int kb, int c) {
    return X.xq + m * X.q_ld + kb * XPITCH + 16 * c;
}

// ---- Q4_K: w = d*sc*q - dmin*m over eight 32-weight sub-blocks ----------
//   y += d * sum_j dx_j*sc_j*I_j  -  dmin * sum_j m_j*(dx_j*s_j)
// I_j for odd j uses the high nibbles in place (x16), folded into d/16.
template <int MT>
__device__ __forceinline__ void sb_q4k(const XS &X, int blk, int kb, float (&v)[MT]) {
    const uint8_t *sm = X.sm;
    const uint4 hdr = ld16(sm, blk);
    const float d = half_bits_to_float(hdr.x), dmin = half_bits_to_float(hdr.x >> 16);
    const uint32_t sc_lo = hdr.y & 0x3F3F3F3Fu, mn_lo = hdr.z & 0x3F3F3F3Fu;
    const uint32_t sc_hi = (hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u);
    const uint32_t mn_hi = ((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u);
    int sc[8];
    float mf[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t sw = j < 4 ? sc_lo : sc_hi, mw = j < 4 ? mn_lo : mn_hi;
        sc[j] = static_cast<int>((sw >> (8 * (j & 3))) & 0xFF);
        mf[j] = static_cast<float>((mw >> (8 * (j & 3))) & 0xFF);
    }
    uint4 q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = ld16(sm, blk + 16 + 16 * i);
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        const float4 *rec = reinterpret_cast<const float4 *>(sm + X.meta + m * X.meta_ld + kb * Rec<QMM_Q4_K>::B);
        const float4 dx0 = rec[0], dx1 = rec[1], ds0 = rec[2], ds1 = rec[3];
        const float dxs[8] = {dx0.x, dx0.y, dx0.z, dx0.w, dx1.x, dx1.y, dx1.z, dx1.w};
        float acc_min = mf[0] * ds0.x;
        acc_min += mf[1] * ds0.y;
        acc_min += mf[2] * ds0.z;
        acc_min += mf[3] * ds0.w;
        acc_min += mf[4] * ds1.x;
        acc_min += mf[5] * ds1.y;
        acc_min += mf[6] * ds1.z;
        acc_min += mf[7] * ds1.w;
        float acc_lo = 0.0f, acc_hi = 0.0f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint4 qa = q[2 * c], qb = q[2 * c + 1];
            const uint4 x0 = ld16(sm, xchunk(X, m, kb, 4 * c));
            const uint4 x1 = ld16(sm, xchunk(X, m, kb, 4 * c + 1));
            const uint4 x2 = ld16(sm, xchunk(X, m, kb, 4 * c + 2));
            const uint4 x3 = ld16(sm, xchunk(X, m, kb, 4 * c + 3));
            constexpr uint32_t LO = 0x0F0F0F0Fu, HI = 0xF0F0F0F0u;
            int I0 = dp4a_ss(qa.x & LO, x0.x, 0);
            I0 = dp4a_ss(qa.y & LO, x0.y, I0);
            I0 = dp4a_ss(qa.z & LO, x0.z, I0);
            I0 = dp4a_ss(qa.w & LO, x0.w, I0);
            I0 = dp4a_ss(qb.x & LO, x1.x, I0);
            I0 = dp4a_ss(qb.y & LO, x1.y, I0);
            I0 = dp4a_ss(qb.z & LO, x1.z, I0);
            I0 = dp4a_ss(qb.w & LO, x1.w, I0);
            int I1 = dp4a_us(qa.x & HI, x2.x, 0);
            I1 = dp4a_us(qa.y & HI, x2.y, I1);
            I1 = dp4a_us(qa.z & HI, x2.z, I1);
            I1 = dp4a_us(qa.w & HI, x2.w, I1);
            I1 = dp4a_us(qb.x & HI, x3.x, I1);
            I1 = dp4a_us(qb.y & HI, x3.y, I1);
            I1 = dp4a_us(qb.z & HI, x3.z, I1);
            I1 = dp4a_us(qb.w & HI, x3.w, I1);
            acc_lo += dxs[2 * c] * static_cast<float>(sc[2 * c] * I0);
            acc_hi += dxs[2 * c + 1] * static_cast<float>(sc[2 * c + 1] * I1);
        }
        v[m] += d * acc_lo + (d * 0.0625f) * acc_hi - dmin * acc_min;
    }
}

// ---- Q6_K: w = d*sc*(q-32), sixteen 16-weight groups ---------------------
//   y += d * sum_g dx_g * sc_g * (sum q*x - 32 * sum x)
template <int MT>
__device__ __forceinline__ void sb_q6k(const XS &X, int blk, int kb, float (&v)[MT]) {
    const uint8_t *sm = X.sm;
    uint32_t scw[4];
    ld_words<4>(sm, blk + 192, scw);
    const float d = half_bits_to_float(*reinterpret_cast<const uint16_t *>(sm + blk + 208));
    float acc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = 0.0f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t ql[16], qh[8];
        ld_words<16>(sm, blk + 64 * h, ql);
        ld_words<8>(sm, blk + 128 + 32 * h, qh);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            uint32_t q[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const uint32_t src = ql[(g & 1) * 8 + e];
                const uint32_t lo = ((g & 2) ? (src >> 4) : src) & 0x0F0F0F0Fu;
                uint32_t hi;
                if (g == 0) hi = (qh[e] << 4) & 0x30303030u;
                else if (g == 1) hi = (qh[e] << 2) & 0x30303030u;
                else if (g == 2) hi = qh[e] & 0x30303030u;
                else hi = (qh[e] >> 2) & 0x30303030u;
                q[e] = lo | hi;
            }
            const int si = 8 * h + 2 * g;  // scales si, si+1
            const int sa = static_cast<int>(static_cast<int8_t>((scw[si >> 2] >> (8 * (si & 3))) & 0xFF));
            const int sb = static_cast<int>(static_cast<int8_t>((scw[si >> 2] >> (8 * ((si + 1) & 3))) & 0xFF));
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const uint4 xa = ld16(sm, xchunk(X, m, kb, 8 * h + 2 * g));
                const uint4 xb = ld16(sm, xchunk(X, m, kb, 8 * h + 2 * g + 1));
                const int rec = X.meta + m * X.meta_ld + kb * Rec<QMM_Q6_K>::B;
                const float dxg = *reinterpret_cast<const float *>(sm + rec + 4 * (4 * h + g));
                const int2 s2 = *reinterpret_cast<const int2 *>(sm + rec + 32 + 8 * (4 * h + g));
                int Ia = dp4a_ss(q[0], xa.x, -32 * s2.x);
                Ia = dp4a_ss(q[1], xa.y, Ia);
                Ia = dp4a_ss(q[2], xa.z, Ia);
                Ia = dp4a_ss(q[3], xa.w, Ia);
                int Ib = dp4a_ss(q[4], xb.x, -32 * s2.y);
                Ib = dp4a_ss(q[5], xb.y, Ib);
                Ib = dp4a_ss(q[6], xb.z, Ib);
                Ib = dp4a_ss(q[7], xb.w, Ib);
                acc[m] += dxg * static_cast<float>(sa * Ia + sb * Ib);
            }
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) v[m] += d * acc[m];
}

// ---- Q5_K: Q4_K with a fifth bit per quant (q in 0..31) -------------------
//   y += d * sum_j dx_j*sc_j*I_j  -  dmin * sum_j m_j*(dx_j*s_j)
// Weight 64c + 32s + l: the low (s = 0) or high (s = 1) nibble of quant
// byte 32c + l, plus bit 2c + s of fifth-bit byte l as bit 4.
template <int MT>
__device__ __forceinline__ void sb_q5k(const XS &X, int blk, int kb, float (&v)[MT]) {
    const uint8_t *sm = X.sm;
    const uint4 hdr = ld16(sm, blk);
    const float d = half_bits_to_float(hdr.x), dmin = half_bits_to_float(hdr.x >> 16);
    const uint32_t sc_lo = hdr.y & 0x3F3F3F3Fu, mn_lo = hdr.z & 0x3F3F3F3Fu;
    const uint32_t sc_hi = (hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u);
    const uint32_t mn_hi = ((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u);
    int sc[8];
    float mf[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t sw = j < 4 ? sc_lo : sc_hi, mw = j < 4 ? mn_lo : mn_hi;
        sc[j] = static_cast<int>((sw >> (8 * (j & 3))) & 0xFF);
        mf[j] = static_cast<float>((mw >> (8 * (j & 3))) & 0xFF);
    }
    const uint4 h0 = ld16(sm, blk + 16), h1 = ld16(sm, blk + 32);
    const uint32_t hw[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
    uint4 q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = ld16(sm, blk + 48 + 16 * i);
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        const float4 *rec = reinterpret_cast<const float4 *>(sm + X.meta + m * X.meta_ld + kb * Rec<QMM_Q5_K>::B);
        const float4 dx0 = rec[0], dx1 = rec[1], ds0 = rec[2], ds1 = rec[3];
        const float dxs[8] = {dx0.x, dx0.y, dx0.z, dx0.w, dx1.x, dx1.y, dx1.z, dx1.w};
        float acc_min = mf[0] * ds0.x;
        acc_min += mf[1] * ds0.y;
        acc_min += mf[2] * ds0.z;
        acc_min += mf[3] * ds0.w;
        acc_min += mf[4] * ds1.x;
        acc_min += mf[5] * ds1.y;
        acc_min += mf[6] * ds1.z;
        acc_min += mf[7] * ds1.w;
        float acc = 0.0f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t qw[8] = {q[2 * c].x, q[2 * c].y, q[2 * c].z, q[2 * c].w,
                                    q[2 * c + 1].x, q[2 * c + 1].y, q[2 * c + 1].z, q[2 * c + 1].w};
            int I0 = 0, I1 = 0;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const uint4 xa = ld16(sm, xchunk(X, m, kb, 4 * c + (e >> 2)));
                const uint4 xb = ld16(sm, xchunk(X, m, kb, 4 * c + 2 + (e >> 2)));
                const uint32_t xl[4] = {xa.x, xa.y, xa.z, xa.w}, xh[4] = {xb.x, xb.y, xb.z, xb.w};
                const uint32_t lo = (qw[e] & 0x0F0F0F0Fu) | (((hw[e] >> (2 * c)) & 0x01010101u) << 4);
                const uint32_t hi = ((qw[e] >> 4) & 0x0F0F0F0Fu) | (((hw[e] >> (2 * c + 1)) & 0x01010101u) << 4);
                I0 = dp4a_ss(lo, xl[e & 3], I0);
                I1 = dp4a_ss(hi, xh[e & 3], I1);
            }
            acc += dxs[2 * c] * static_cast<float>(sc[2 * c] * I0) +
                   dxs[2 * c + 1] * static_cast<float>(sc[2 * c + 1] * I1);
        }
        v[m] += d * acc - dmin * acc_min;
    }
}

// ---- Q3_K: w = d*(sc-32)*q, q in -4..3, sixteen 16-weight groups -----------
//   y += d * sum_g dx_g * sc_g * (sum (q+4)*x - 4 * sum x)
// Weight 128h + 32j + l: low bits (byte 32h + l of the 2-bit plane >> 2j) & 3,
// high bit 4h + j of mask byte l; q + 4 = low | high << 2.  Group 8h + 2j +
// (l >= 16); its 6-bit scale: the low (G = 0, 1) or high (G = 2, 3) nibble of
// scale byte k or 4 + k (G odd) and the pair (byte 8 + k >> 2G) & 3, with
// k = group mod 4, G = group / 4.
template <int MT>
__device__ __forceinline__ void sb_q3k(const XS &X, int blk, int kb, float (&v)[MT]) {
    const uint8_t *sm = X.sm;
    uint32_t S[3], hm[8];
    ld_words<3>(sm, blk + 96, S);
    ld_words<8>(sm, blk, hm);
    const float d = half_bits_to_float(*reinterpret_cast<const uint16_t *>(sm + blk + 108));
    int sc[16];
#pragma unroll
    for (int G = 0; G < 4; ++G) {
        const uint32_t lo = ((G & 2) ? (S[G & 1] >> 4) : S[G & 1]) & 0x0F0F0F0Fu;
        const uint32_t w = lo | (((S[2] >> (2 * G)) & 0x03030303u) << 4);
#pragma unroll
        for (int k = 0; k < 4; ++k) sc[4 * G + k] = static_cast<int>((w >> (8 * k)) & 0xFF) - 32;
    }
    float acc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = 0.0f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t qs[8];
        ld_words<8>(sm, blk + 32 + 32 * h, qs);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t q[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
                q[e] = ((qs[e] >> (2 * j)) & 0x03030303u) | (((hm[e] >> (4 * h + j)) & 0x01010101u) << 2);
            const int sa = sc[8 * h + 2 * j], sb = sc[8 * h + 2 * j + 1];
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const uint4 xa = ld16(sm, xchunk(X, m, kb, 8 * h + 2 * j));
                const uint4 xb = ld16(sm, xchunk(X, m, kb, 8 * h + 2 * j + 1));
                const int rec = X.meta + m * X.meta_ld + kb * Rec<QMM_Q3_K>::B;
                const float dxg = *reinterpret_cast<const float *>(sm + rec + 4 * (4 * h + j));
                const int2 s2 = *reinterpret_cast<const int2 *>(sm + rec + 32 + 8 * (4 * h + j));
                int Ia = dp4a_ss(q[0], xa.x, -4 * s2.x);
                Ia = dp4a_ss(q[1], xa.y, Ia);
                Ia = dp4a_ss(q[2], xa.z, Ia);
                Ia = dp4a_ss(q[3], xa.w, Ia);
                int Ib = dp4a_ss(q[4], xb.x, -4 * s2.y);
                Ib = dp4a_ss(q[5], xb.y, Ib);
                Ib = dp4a_ss(q[6], xb.z, Ib);
                Ib = dp4a_ss(q[7], xb.w, Ib);
                acc[m] += dxg * static_cast<float>(sa * Ia + sb * Ib);
            }
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) v[m] += d * acc[m];
}

// ---- Q2_K: w = d*sc*q - dmin*m, q in 0..3, sixteen 16-weight groups ------
//   y += sum_g dx_g * (d * sc_g * sum q*x  -  dmin * m_g * sum x)
// Weight 128h + 32j + l: (byte 32h + l of the 2-bit plane >> 2j) & 3; group
// 8h + 2j + (l >= 16) with scale / min the low / high nibble of byte group.
template <int MT>
__device__ __forceinline__ void sb_q2k(const XS &X, int blk, int kb, float (&v)[MT]) {
    const uint8_t *sm = X.sm;
    uint32_t scw[4], dd[1];
    ld_words<4>(sm, blk, scw);
    ld_words<1>(sm, blk + 80, dd);
    const float d = half_bits_to_float(dd[0]), dmin = half_bits_to_float(dd[0] >> 16);
    float acc[MT], accm[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = accm[m] = 0.0f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t qs[8];
        ld_words<8>(sm, blk + 16 + 32 * h, qs);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t q[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) q[e] = (qs[e] >> (2 * j)) & 0x03030303u;
            const int ga = 8 * h + 2 * j, gb = ga + 1;
            const uint32_t ba = (scw[ga >> 2] >> (8 * (ga & 3))) & 0xFF, bb = (scw[gb >> 2] >> (8 * (gb & 3))) & 0xFF;
            const int sa = static_cast<int>(ba & 15), sb = static_cast<int>(bb & 15);
            const int ma = static_cast<int>(ba >> 4), mb = static_cast<int>(bb >> 4);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const uint4 xa = ld16(sm, xchunk(X, m, kb, 8 * h + 2 * j));
                const uint4 xb = ld16(sm, xchunk(X, m, kb, 8 * h + 2 * j + 1));
                const int rec = X.meta + m * X.meta_ld + kb * Rec<QMM_Q2_K>::B;
                const float dxg = *reinterpret_cast<const float *>(sm + rec + 4 * (4 * h + j));
                const int2 s2 = *reinterpret_cast<const int2 *>(sm + rec + 32 + 8 * (4 * h + j));
                int Ia = dp4a_ss(q[0], xa.x, 0);
                Ia = dp4a_ss(q[1], xa.y, Ia);
                Ia = dp4a_ss(q[2], xa.z, Ia);
                Ia = dp4a_ss(q[3], xa.w, Ia);
                int Ib = dp4a_ss(q[4], xb.x, 0);
                Ib = dp4a_ss(q[5], xb.y, Ib);
                Ib = dp4a_ss(q[6], xb.z, Ib);
                Ib = dp4a_ss(q[7], xb.w, Ib);
                acc[m] += dxg * static_cast<float>(sa * Ia + sb * Ib);
                accm[m] += dxg * static_cast<float>(ma * s2.x + mb * s2.y);
            }
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) v[m] += d * acc[m] - dmin * accm[m];
}

// ---- Q8_0: w = d*q, one 32-weight block ----------------------------------
template <int MT>
__device__ __forceinline__ void sb_q80(const XS &X, int blk, int kb, float (&v)[MT]) {
    const uint8_t *sm = X.sm;
    uint32_t qw[8];
    ld_words<8>(sm, blk + 2, qw);
    const float d = half_bits_to_float(*reinterpret_cast<const uint16_t *>(sm + blk));
    const int sbk = kb >> 3, j = kb & 7;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        const uint4 x0 = ld16(sm, xchunk(X, m, sbk, 2 * j));
        const uint4 x1 = ld16(sm, xchunk(X, m, sbk, 2 * j + 1));
        int I = dp4a_ss(qw[0], x0.x, 0);
        I = dp4a_ss(qw[1], x0.y, I);
        I = dp4a_ss(qw[2], x0.z, I);
        I = dp4a_ss(qw[3], x0.w, I);
        I = dp4a_ss(qw[4], x1.x, I);
        I = dp4a_ss(qw[5], x1.y, I);
        I = dp4a_ss(qw[6], x1.z, I);
        I = dp4a_ss(qw[7], x1.w, I);
        const float dx = *reinterpret_cast<const float *>(sm + X.meta + m * X.meta_ld + 4 * kb);
        v[m] += dx * (d * static_cast<float>(I));
    }
}

// ---- the activation quantiser, into shared memory --------------------------
// Same arithmetic as the standalone quantiser (and the oracle): per block of
// 32, amax = max|x|, d = amax/127, inv = 1/d (0 if d == 0; the correctly
// rounded reciprocal equals the IEEE quotient 1/d), q = round half away from
// zero of x*inv clamped to +-127.  TPB consecutive threads share a block
// (32/TPB values each, loaded 16 bytes at a time), combining the maximum and
// the sums with shuffles; TPB is chosen so one pass covers all blocks when
// they are few.
// Quantise one value: round half away from zero of v = x*inv.  For finite x,
// |x*inv| <= amax*(1/d) <= 127*(1 + 2^-22) < 127.5, so the +-127 clamp of the
// definition can never change the result and is not applied here.
__device__ __forceinline__ int quant1(float x, float inv) { return static_cast<int>(roundf(__fmul_rn(x, inv))); }

// Pack four int8 values (given as ints) into one little-endian word.
__device__ __forceinline__ uint32_t pack4(int a, int b, int c, int d) {
    const uint32_t lo = __byte_perm(static_cast<uint32_t>(a), static_cast<uint32_t>(b), 0x0040);
    const uint32_t hi = __byte_perm(static_cast<uint32_t>(c), static_cast<uint32_t>(d), 0x0040);
    return __byte_perm(lo, hi, 0x5410);
}

// max |a[i]| over N values as a balanced tree
template <int N>
__device__ __forceinline__ float absmax(const float (&a)[N]) {
    float t[N];
#pragma unroll
    for (int i = 0; i < N; ++i) t[i] = fabsf(a[i]);
#pragma unroll
    for (int w = N / 2; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) t[i] = fmaxf(t[i], t[i + w]);
    return t[0];
}

template <int T, int TPB, int R, int NT, class F>
__device__ __forceinline__ void quantize_tpb(const SbParams &P, uint8_t *smem, F &&after_loads) {
    constexpr int EPT = 32 / TPB;
    const int nb32 = P.K / 32;
    const int items = P.M * nb32 * TPB;
    for (int base = 0; base < items; base += R * NT) {
        // every load of this pass first: R items of EPT values per thread
        float a[R][EPT];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int it = base + r * NT + static_cast<int>(threadIdx.x);
            const bool ok = it < items;
            const int id = ok ? it / TPB : 0;
            const int m = id / nb32, b = id - m * nb32;
            const float *src = P.x + static_cast<int64_t>(m) * P.K + 32 * b + EPT * (it & (TPB - 1));
            if (P.x_vec) {
#pragma unroll
                for (int i = 0; i < EPT / 4; ++i) {
                    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (ok) v = __ldg(reinterpret_cast<const float4 *>(src) + i);
                    a[r][4 * i] = v.x; a[r][4 * i + 1] = v.y; a[r][4 * i + 2] = v.z; a[r][4 * i + 3] = v.w;
                }
            } else {
#pragma unroll
                for (int i = 0; i < EPT; ++i) a[r][i] = ok ? __ldg(src + i) : 0.0f;
            }
        }
        if (base == 0) after_loads();
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int it = base + r * NT + static_cast<int>(threadIdx.x);
            const bool ok = it < items;
            const int id = ok ? it / TPB : 0;
            const int part = it & (TPB - 1);
            const int m = id / nb32, b = id - m * nb32;
            float am = absmax<EPT>(a[r]);
#pragma unroll
            for (int o = 1; o < TPB; o <<= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
            const float db = __fdiv_rn(am, 127.0f);
            const float inv = (db != 0.0f) ? __frcp_rn(db) : 0.0f;
            uint32_t w[EPT / 4];
            int s0 = 0, s1 = 0;  // this thread's values in the first / second half block
#pragma unroll
            for (int i = 0; i < EPT / 4; ++i) {
                int q[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) q[e] = quant1(a[r][4 * i + e], inv);
                const int s4 = q[0] + q[1] + q[2] + q[3];
                if (EPT * part + 4 * i < 16) s0 += s4; else s1 += s4;
                w[i] = pack4(q[0], q[1], q[2], q[3]);
            }
#pragma unroll
            for (int o = 1; o < TPB; o <<= 1) {
                s0 += __shfl_xor_sync(0xffffffffu, s0, o);
                s1 += __shfl_xor_sync(0xffffffffu, s1, o);
            }
            if (!ok) continue;
            // this thread's bytes: elements [EPT*part, EPT*part + EPT) of the block,
            // inside chunks 2*(b & 7) and 2*(b & 7) + 1 of super-block b >> 3
            const int sb = b >> 3;
            uint8_t *row = smem + P.off_xq + m * P.q_ld + sb * XPITCH;
            if constexpr (EPT == 32) {
                const int c0 = 2 * (b & 7), c1 = 2 * (b & 7) + 1;
                *reinterpret_cast<uint4 *>(row + 16 * c0) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4 *>(row + 16 * c1) = make_uint4(w[4], w[5], w[6], w[7]);
            } else if constexpr (EPT == 16) {
                const int c = 2 * (b & 7) + part;
                *reinterpret_cast<uint4 *>(row + 16 * c) = make_uint4(w[0], w[1], w[2], w[3]);
            } else {
                const int c = 2 * (b & 7) + (part >> 1);
                *reinterpret_cast<uint2 *>(row + 16 * c + 8 * (part & 1)) = make_uint2(w[0], w[1]);
            }
            if (part == 0) {
                if (T == QMM_Q8_0) {
                    reinterpret_cast<float *>(smem + P.off_meta + m * P.meta_ld)[b] = db;
                } else {
                    uint8_t *rec = smem + P.off_meta + m * P.meta_ld + sb * Rec<T>::B;
                    reinterpret_cast<float *>(rec)[b & 7] = db;
                    if (kRecDs<T>) reinterpret_cast<float *>(rec + 32)[b & 7] = db * static_cast<float>(s0 + s1);
                    if (kRecHalves<T>) reinterpret_cast<int2 *>(rec + 32)[b & 7] = make_int2(s0, s1);
                }
            }
        }
    }
}

// Run by threads 0 .. NT-1 of the CTA.  after_loads() runs once, after the
// first pass's activation loads are issued and before their values are used.
// The split (threads per block TPB, items per thread R) keeps one pass and
// the fewest values per thread.
template <int T, int NT = NTHREADS, class F>
__device__ __forceinline__ void quantize_to_smem(const SbParams &P, uint8_t *smem, F &&after_loads) {
    const int total = P.M * (P.K / 32);
    if (4 * total <= NT) quantize_tpb<T, 4, 1, NT>(P, smem, after_loads);
    else if (2 * total <= NT) quantize_tpb<T, 2, 1, NT>(P, smem, after_loads);
    else if (total <= NT) quantize_tpb<T, 1, 1, NT>(P, smem, after_loads);
    else if (2 * total <= 2 * NT) quantize_tpb<T, 2, 2, NT>(P, smem, after_loads);
    else if (2 * total <= 3 * NT) quantize_tpb<T, 2, 3, NT>(P, smem, after_loads);
    else quantize_tpb<T, 2, 4, NT>(P, smem, after_loads);
}

// The work of CTA `cta` of one matrix (its share of the rows).  With GATEUP
// the CTA takes the same rows of two matrices, gate (W) and up (W2): warps
// 0..5 stream the gate rows, warps 6..11 the up rows, both from the one
// quantised x; the row results meet in a shared-memory table and the CTA
// writes h = silu(gate) * up.
template <int T, int MT, bool GATEUP = false>
__device__ __forceinline__ void sb_body(const SbParams &P, const int cta) {
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int BB = Fmt<T>::BB;
    constexpr int NW = GATEUP ? NWARP / 2 : NWARP;  // warps per matrix
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wg = GATEUP ? warp / NW : 0;  // the matrix of this warp: 0 = W, 1 = W2
    const int wi = warp - wg * NW;          // the warp's index among its matrix's warps

    const int64_t r0 = P.rows_q * cta + min(cta, P.rows_r);
    const int64_t r1 = r0 + P.rows_q + (cta < P.rows_r ? 1 : 0);
    const int rows = static_cast<int>(r1 - r0);
    const int U = rows * P.nb;  // blocks of this CTA (of each matrix)
    const int uw0 = static_cast<int>((static_cast<int64_t>(U) * wi) / NW);
    const int uw1 = static_cast<int>((static_cast<int64_t>(U) * (wi + 1)) / NW);
    float *tab = reinterpret_cast<float *>(smem + P.off_tab);  // GATEUP: [2][rows][MT]
    const int nst = (uw1 - uw0 + SU - 1) / SU;

    const uint32_t bar0 = smem_u32(smem);
    int *edge_row = reinterpret_cast<int *>(smem + P.off_edge);
    float *edge_val = reinterpret_cast<float *>(edge_row + 2 * NWARP);

    // Each warp's lane 0 sets up its own barriers and starts its stream at
    // once; warp 0 clears the edge records (read only after the CTA barrier
    // that follows the activation quantiser).
    const uint32_t my_bar = bar0 + 8u * warp * MAX_NSW;
    if (lane == 0) {
        for (int i = 0; i < P.NSW; ++i) mbar_init(my_bar + 8u * i, 1);
        fence_mbar_init();
    }
    if (warp == 0 && lane < 2 * NWARP) edge_row[lane] = -1;
    __syncwarp();

    // weights of this CTA, relative to its first byte rounded down to 16
    const int64_t cta_byte = r0 * P.RB;
    const uint8_t *Wc = (wg ? P.W2 : P.W) + (cta_byte & ~int64_t(15));
    const int cta_off = static_cast<int>(cta_byte & 15);
    const int64_t avail = P.total_bytes - (cta_byte & ~int64_t(15));
    const int ring = P.off_ring + warp * P.NSW * P.slot_bytes;

    // stages from `stop` on are never issued (only with the test hook: the
    // consumer's bounded wait on stage `stop` then expires)
    const int stop = cta == 0 ? P.stop_stage : NO_STOP;
    // issue stage t of this warp into `slot` (= t % NSW; lane 0 only)
    auto issue = [&](int t, int slot, uint64_t pol) {
        if (t >= stop) return;
        const int u0 = uw0 + SU * t, u1 = min(u0 + SU, uw1);
        const int a = cta_off + u0 * BB, b = cta_off + u1 * BB;
        const int a16 = a & ~15;
        int b16 = (b + 15) & ~15;
        const int dst = ring + slot * P.slot_bytes;
        if (b16 > avail) {  // the last bytes of the matrix: plain loads for the tail
            b16 = b & ~15;
            for (int i = b16; i < b; ++i) smem[dst + (i - a16)] = Wc[i];
        }
        const uint32_t nbytes = static_cast<uint32_t>(b16 - a16);
        mbar_arrive_expect_tx(my_bar + 8u * slot, nbytes);
        if (nbytes) bulk_g2s(smem_u32(smem + dst), Wc + a16, nbytes, my_bar + 8u * slot, pol);
    };

    // The next kernel on the stream may start launching now.  Until the
    // preceding kernel completes (it may produce x) this CTA only warms L2:
    // each warp's first stages of weights (which no kernel of the library
    // writes) and x (an L2 prefetch cannot leave a stale copy; x itself is
    // read after the wait), so the weight stream of this call overlaps the
    // tail of the last one.  After the wait: this thread's activation loads,
    // and only then the rest of the weight stream into shared memory, so the
    // loads do not return behind tens of KB of bulk copies into this SM.
    pdl_trigger();
    uint64_t pol_w = 0;
    int issued = 0;
    if (lane == 0) {
        pol_w = policy_evict_first();
        // the first stage goes into shared memory at once for Q4_K (measured:
        // 3-6 % off the Q4_K launches) and for rows of at least 4096 weights
        // (their x takes longer to quantise: 1.5 us off the decode step); for
        // short rows of the other types the copies delay x's loads more than
        // they gain (the 2048 x 128256 Q6_K lm_head: 33.0 against 34.2 us)
        if ((T == QMM_Q4_K || P.K >= 4096) && nst > 0) issue(0, 0, pol_w), issued = 1;
        for (int t = issued; t < min(P.NSW, nst); ++t) {
            const int u0 = uw0 + SU * t, u1 = min(u0 + SU, uw1);
            const int a16 = (cta_off + u0 * BB) & ~15;
            int b16 = (cta_off + u1 * BB + 15) & ~15;
            if (b16 > avail) b16 = (cta_off + u1 * BB) & ~15;
            if (b16 > a16) bulk_prefetch_l2(Wc + a16, static_cast<uint32_t>(b16 - a16));
        }
    }
    if (threadIdx.x == 32 && P.x_vec && ((P.M * P.K * 4) & 15) == 0)
        bulk_prefetch_l2(P.x, static_cast<uint32_t>(P.M * P.K * 4));
    pdl_wait();
    quantize_to_smem<T>(P, smem, [&] {
        if (lane == 0)
            for (; issued < min(P.NSW, nst); ++issued) issue(issued, issued, pol_w);
    });
    __syncthreads();

    XS X;
    X.sm = smem;
    X.xq = P.off_xq;
    X.meta = P.off_meta;
    X.q_ld = P.q_ld;
    X.meta_ld = P.meta_ld;

    bool failed = false;
    int carry_row = -1;
    float carry[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) carry[m] = 0.0f;
    int consumed = 0;
    int slot = 0, islot = min(P.NSW, nst) % P.NSW;  // ring slots of stage t and of the next issue
    uint32_t phase = 0;                              // parity of stage t's slot
    for (int t = 0; t < nst && !failed; ++t) {
        if (!mbar_wait(my_bar + 8u * slot, phase, P.status)) {
            failed = true;
            break;
        }
        consumed = t + 1;
        const int u0 = uw0 + SU * t, u1 = min(u0 + SU, uw1), nv = u1 - u0;
        const int a16 = (cta_off + u0 * BB) & ~15;
        // shared-memory offset of CTA-relative block 0 for this stage
        const int base = ring + slot * P.slot_bytes - a16 + cta_off;
        const int u = u0 + lane;
        const bool valid = lane < nv;
        const int row = !valid ? -1
                        : P.nb_magic ? static_cast<int>(__umulhi(static_cast<uint32_t>(u), P.nb_magic))
                                     : u / P.nb;
        float v[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) v[m] = 0.0f;
        if (valid) {
            const int kb = u - row * P.nb;
            const int blk = base + u * BB;
            if constexpr (T == QMM_Q4_K) sb_q4k<MT>(X, blk, kb, v);
            else if constexpr (T == QMM_Q6_K) sb_q6k<MT>(X, blk, kb, v);
            else if constexpr (T == QMM_Q5_K) sb_q5k<MT>(X, blk, kb, v);
            else if constexpr (T == QMM_Q3_K) sb_q3k<MT>(X, blk, kb, v);
            else if constexpr (T == QMM_Q2_K) sb_q2k<MT>(X, blk, kb, v);
            else sb_q80<MT>(X, blk, kb, v);
        }
        __syncwarp();
        if (lane == 0 && issued < nst) {
            // the slot just read is refilled: order the reads before the async write
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(issued, islot, pol_w);
            ++issued;
            if (++islot == P.NSW) islot = 0;
        }
        // segmented suffix sums: lane i gets the sum of its row over lanes i..seg_last
        const int row_start = row * P.nb, row_end = row_start + P.nb;
        const int seg_last = valid ? min(nv, row_end - u0) - 1 : -1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const float o = __shfl_down_sync(0xffffffffu, v[m], off);
                if (lane + off <= seg_last) v[m] += o;
            }
        }
        const bool head = valid && (lane == 0 || u == row_start);
        if (head && lane == 0 && row == carry_row) {
#pragma unroll
            for (int m = 0; m < MT; ++m) v[m] += carry[m];
        }
        // the stage's last row continues into this warp's next stage?
        const int row_last = P.nb_magic ? static_cast<int>(__umulhi(static_cast<uint32_t>(u1 - 1), P.nb_magic))
                                         : (u1 - 1) / P.nb;
        const int head_last = max(0, row_last * P.nb - u0);
        const bool cont = (row_last + 1) * P.nb > u1 && u1 < uw1;
        if (head && !(cont && row == row_last)) {
            if (row_start < uw0 || row_end > uw1) {
                const int e = 2 * warp + (row_start < uw0 ? 0 : 1);
                edge_row[e] = row + (wg << 30);  // (matrix, row): rows < 2^30
#pragma unroll
                for (int m = 0; m < MT; ++m) edge_val[e * 8 + m] = v[m];
            } else if (GATEUP) {
#pragma unroll
                for (int m = 0; m < MT; ++m) tab[(wg * rows + row) * MT + m] = v[m];
            } else {
#pragma unroll
                for (int m = 0; m < MT; ++m)
                    if (m < P.M) P.y[static_cast<int64_t>(m) * P.N + r0 + row] = v[m];
            }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) carry[m] = __shfl_sync(0xffffffffu, v[m], head_last);
        carry_row = cont ? row_last : -1;
        if (++slot == P.NSW) slot = 0, phase ^= 1u;
    }
    // no bulk copy may still be in flight when the CTA exits
    if (lane == 0)
        for (int t = consumed; t < min(issued, stop); ++t)
            mbar_wait(my_bar + 8u * (t % P.NSW), static_cast<uint32_t>((t / P.NSW) & 1), P.status);
    __syncthreads();
    if (warp == 0) {
        // Rows cut by warp boundaries: record e = 2w + {0, 1} holds warp w's
        // partial of its first / last row.  Rows are nondecreasing in e; the
        // first record of each row adds the others in record order.
        const int e = lane;
        const int r = e < 2 * NWARP ? edge_row[e] : -1;
        const unsigned same = __match_any_sync(0xffffffffu, r);
        float mine[MT], acc[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            mine[m] = r >= 0 ? edge_val[e * 8 + m] : 0.0f;
            acc[m] = 0.0f;
        }
#pragma unroll 4
        for (int j = 0; j < 2 * NWARP; ++j) {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const float vj = __shfl_sync(0xffffffffu, mine[m], j);
                if ((same >> j) & 1u) acc[m] += vj;
            }
        }
        if (r >= 0 && (__ffs(same) - 1) == lane) {
            const int rw = r & ((1 << 30) - 1), mw = r >> 30;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (GATEUP) tab[(mw * rows + rw) * MT + m] = acc[m];
                else if (m < P.M) P.y[static_cast<int64_t>(m) * P.N + r0 + rw] = acc[m];
            }
        }
    }
    if constexpr (GATEUP) {
        // h = silu(g) * u for every row of the CTA, silu(g) = g / (1 + e^-g)
        __syncthreads();
        for (int i = threadIdx.x; i < rows * P.M; i += NTHREADS) {
            const int row = i / P.M, m = i - row * P.M;
            const float g = tab[row * MT + m], u = tab[(rows + row) * MT + m];
            P.y[static_cast<int64_t>(m) * P.N + r0 + row] = g / (1.0f + expf(-g)) * u;
        }
    }
}

template <int T, int MT>
__global__ void __launch_bounds__(NTHREADS, 1) gemv_sb_kernel(const __grid_constant__ SbParams P) {
    sb_body<T, MT>(P, static_cast<int>(blockIdx.x));
}

// gate and up (same type and shape) in one launch, writing h = silu(g) * u
template <int T, int MT>
__global__ void __launch_bounds__(NTHREADS, 1) gemv_sb_gateup_kernel(const __grid_constant__ SbParams P) {
    sb_body<T, MT, true>(P, static_cast<int>(blockIdx.x));
}

template <int T, int MT>
cudaError_t launch_t(const SbParams &P, int grid, int smem, cudaStream_t st) {
    auto kfn = gemv_sb_kernel<T, MT>;
    if constexpr (MT <= 2)
        if (P.W2) kfn = gemv_sb_gateup_kernel<T, MT>;
    cudaError_t e = set_smem_attrs(kfn, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kfn, P);
}

template <int T>
cudaError_t launch_m(const SbParams &P, int MT, int grid, int smem, cudaStream_t st) {
    switch (MT) {
    case 1: return launch_t<T, 1>(P, grid, smem, st);
    case 2: return launch_t<T, 2>(P, grid, smem, st);
    case 4: return launch_t<T, 4>(P, grid, smem, st);
    default: return launch_t<T, 8>(P, grid, smem, st);
    }
}


}  // namespace sbk

// The launches of the block-per-lane kernel for Q5_K, Q3_K and Q2_K
// (gemv_sb_kq.cu).
cudaError_t launch_sb_kquant(int type, const sbk::SbParams &P, int MT, int grid, int smem, cudaStream_t st);

}  // namespace qk
