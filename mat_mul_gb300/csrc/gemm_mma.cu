// gemm_mma.cu -- prefill product y[M,N] = W[N,K] . x[M,K]^T for M > 8 on the
// warp-level integer tensor-core path (mma.sync ... s8.s8.s32), exact int32
// per-block dot products and fp32 per-block scaling.
//
// This is the reference-grade tensor-core path: simple, exact per block, and
// used for shapes and types the tcgen05 pipeline does not cover.  The
// activations arrive quantised (int8 q, fp32 scale, int32 sum per 32-block,
// for Q2_K the sums of the 16-element halves) from the quantiser kernel; the
// weights are unpacked to int8 in shared memory by the CTA (Q4_K: q in
// 0..15, Q5_K: 0..31, Q6_K: q-32, Q3_K: -4..3, Q2_K: 0..3, Q8_0: q) together
// with their scales (and mins).
//
// Tile: 64 activation rows x 64 weight rows per CTA, one 256-wide K step per
// iteration (one super-block, eight Q8_0 blocks); four warps of 32x32
// outputs, each issuing m16n8k32 (Q4_K, Q5_K, Q8_0: one 32-block) or two
// m16n8k16 (Q6_K, Q3_K, Q2_K: one 16-weight group each) per 32-wide block.
#include "qmm_device.cuh"

#include <type_traits>

namespace qk {

namespace {

constexpr int BM = 64, BN = 64, BK = 256;
constexpr int LDS_ROW = BK + 16;  // padded row (bytes): conflict-free fragment loads

struct GemmSmem {
    int8_t a[BM][LDS_ROW];
    int8_t b[BN][LDS_ROW];
    float xd[BM][8];
    int32_t xs[BM][8];
    int16_t xs2[BM][16];  // Q2_K: the sums of the two 16-element halves of every block
    float wd[BN];       // d (the K-quants)
    float wdmin[BN];    // dmin (Q4_K, Q5_K, Q2_K)
    float wd8[BN][8];   // per-block d (Q8_0)
    int16_t wsc[BN][16];  // Q4_K, Q5_K: sc[8]; Q6_K, Q3_K (sc - 32), Q2_K: sc[16]
    int16_t wm[BN][16];   // Q4_K, Q5_K: m[8]; Q2_K: m[16]
};

// Sixteen 16-weight groups per 32-block pair of K-steps (two mma k16 per block)
template <int T> constexpr bool kGroups16 = T == QMM_Q6_K || T == QMM_Q3_K || T == QMM_Q2_K;

__device__ __forceinline__ void mma_k32(int (&c)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__device__ __forceinline__ void mma_k16(int (&c)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5}, {%6}, "
        "{%0,%1,%2,%3};"
        : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3])
        : "r"(a0), "r"(a1), "r"(b0));
}

template <int T>
__device__ void load_weights(GemmSmem &S, const uint8_t *__restrict__ W, int64_t N, int64_t K,
                             int64_t n0, int64_t k0) {
    const int tid = threadIdx.x;
    const int r = tid >> 1, part = tid & 1;  // 128 threads: two per weight row
    const int64_t n = n0 + r;
    int8_t *dst = S.b[r];
    if constexpr (T == QMM_Q4_K || T == QMM_Q5_K) {
        constexpr int BB = Fmt<T>::BB, QOFF = T == QMM_Q5_K ? 48 : 16;  // quant bytes
        if (n >= N) {
            for (int i = part * 128; i < part * 128 + 128; ++i) dst[i] = 0;
            if (part == 0) {
                S.wd[r] = 0.f;
                S.wdmin[r] = 0.f;
                for (int j = 0; j < 8; ++j) S.wsc[r][j] = S.wm[r][j] = 0;
            }
            return;
        }
        const uint8_t *B = W + (n * (K / 256) + k0 / 256) * BB;
        if (part == 0) {
            const uint8_t *Sb = B + 4;
            S.wd[r] = half_bits_to_float(B[0] | (B[1] << 8));
            S.wdmin[r] = half_bits_to_float(B[2] | (B[3] << 8));
            for (int j = 0; j < 8; ++j) {
                int sc, m;
                if (j < 4) {
                    sc = Sb[j] & 63;
                    m = Sb[j + 4] & 63;
                } else {
                    sc = (Sb[j + 4] & 15) | ((Sb[j - 4] >> 6) << 4);
                    m = (Sb[j + 4] >> 4) | ((Sb[j] >> 6) << 4);
                }
                S.wsc[r][j] = static_cast<int16_t>(sc);
                S.wm[r][j] = static_cast<int16_t>(m);
            }
        }
        // chunks c = 2*part, 2*part+1: qs[32c+l] -> weights 64c+l (low), 64c+32+l
        // (high); Q5_K: plus bit 2c (low) / 2c+1 (high) of fifth-bit byte l as bit 4
        for (int c = 2 * part; c < 2 * part + 2; ++c) {
            const uint4 *src = reinterpret_cast<const uint4 *>(B + QOFF + 32 * c);
            for (int v = 0; v < 2; ++v) {
                const uint4 w = __ldg(src + v);
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
                uint32_t lo[4], hi[4];
                uint32_t hb[4] = {0u, 0u, 0u, 0u};
                if constexpr (T == QMM_Q5_K) {
                    const uint4 h = __ldg(reinterpret_cast<const uint4 *>(B + 16) + v);
                    hb[0] = h.x, hb[1] = h.y, hb[2] = h.z, hb[3] = h.w;
                }
                for (int e = 0; e < 4; ++e) {
                    lo[e] = (ws[e] & 0x0F0F0F0Fu) | (((hb[e] >> (2 * c)) & 0x01010101u) << 4);
                    hi[e] = ((ws[e] >> 4) & 0x0F0F0F0Fu) | (((hb[e] >> (2 * c + 1)) & 0x01010101u) << 4);
                }
                *reinterpret_cast<uint4 *>(dst + 64 * c + 16 * v) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                *reinterpret_cast<uint4 *>(dst + 64 * c + 32 + 16 * v) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            }
        }
    } else if constexpr (T == QMM_Q6_K) {
        if (n >= N) {
            for (int i = part * 128; i < part * 128 + 128; ++i) dst[i] = 0;
            if (part == 0) {
                S.wd[r] = 0.f;
                for (int j = 0; j < 16; ++j) S.wsc[r][j] = 0;
            }
            return;
        }
        const uint8_t *B = W + (n * (K / 256) + k0 / 256) * 210;
        if (part == 0) {
            S.wd[r] = half_bits_to_float(B[208] | (B[209] << 8));
            for (int j = 0; j < 16; ++j) S.wsc[r][j] = static_cast<int8_t>(B[192 + j]);
        }
        const int h = part;  // half h: weights 128h + 32g + l
        for (int g = 0; g < 4; ++g)
            for (int l = 0; l < 32; ++l) {
                const int lo = (B[64 * h + l + 32 * (g & 1)] >> ((g >= 2) ? 4 : 0)) & 15;
                const int hi = (B[128 + 32 * h + l] >> (2 * g)) & 3;
                dst[128 * h + 32 * g + l] = static_cast<int8_t>((lo | (hi << 4)) - 32);
            }
    } else if constexpr (T == QMM_Q3_K) {
        if (n >= N) {
            for (int i = part * 128; i < part * 128 + 128; ++i) dst[i] = 0;
            if (part == 0) {
                S.wd[r] = 0.f;
                for (int j = 0; j < 16; ++j) S.wsc[r][j] = 0;
            }
            return;
        }
        const uint8_t *B = W + (n * (K / 256) + k0 / 256) * 110;
        if (part == 0) {
            const uint8_t *Sb = B + 96;
            S.wd[r] = half_bits_to_float(B[108] | (B[109] << 8));
            for (int i = 0; i < 16; ++i) {
                const int k = i & 3, G = i >> 2;
                const int lo = (G & 2 ? Sb[(G & 1) * 4 + k] >> 4 : Sb[(G & 1) * 4 + k]) & 15;
                const int hi = (Sb[8 + k] >> (2 * G)) & 3;
                S.wsc[r][i] = static_cast<int16_t>((lo | (hi << 4)) - 32);
            }
        }
        // half h: weights 128h + 32j + l; four weights per 32-bit word: the
        // low bits (byte l of the 2-bit plane >> 2j) & 3 and the high bit
        // (mask byte l >> 4h + j) & 1 make q + 4, one SIMD byte subtract q
        // (the block is 2-byte aligned: its words are read as halves)
        const int h = part;
        uint32_t qs[8], hm[8];
        for (int e = 0; e < 8; ++e) {
            const uint16_t *p2 = reinterpret_cast<const uint16_t *>(B + 32 + 32 * h + 4 * e);
            const uint16_t *m2 = reinterpret_cast<const uint16_t *>(B + 4 * e);
            qs[e] = static_cast<uint32_t>(__ldg(p2)) | (static_cast<uint32_t>(__ldg(p2 + 1)) << 16);
            hm[e] = static_cast<uint32_t>(__ldg(m2)) | (static_cast<uint32_t>(__ldg(m2 + 1)) << 16);
        }
        for (int j = 0; j < 4; ++j) {
            uint32_t w[8];
            for (int e = 0; e < 8; ++e)
                w[e] = __vsub4(((qs[e] >> (2 * j)) & 0x03030303u) | (((hm[e] >> (4 * h + j)) & 0x01010101u) << 2),
                               0x04040404u);
            *reinterpret_cast<uint4 *>(dst + 128 * h + 32 * j) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4 *>(dst + 128 * h + 32 * j + 16) = make_uint4(w[4], w[5], w[6], w[7]);
        }
    } else if constexpr (T == QMM_Q2_K) {
        if (n >= N) {
            for (int i = part * 128; i < part * 128 + 128; ++i) dst[i] = 0;
            if (part == 0) {
                S.wd[r] = S.wdmin[r] = 0.f;
                for (int j = 0; j < 16; ++j) S.wsc[r][j] = S.wm[r][j] = 0;
            }
            return;
        }
        const uint8_t *B = W + (n * (K / 256) + k0 / 256) * 84;
        if (part == 0) {
            S.wd[r] = half_bits_to_float(B[80] | (B[81] << 8));
            S.wdmin[r] = half_bits_to_float(B[82] | (B[83] << 8));
            for (int i = 0; i < 16; ++i) {
                S.wsc[r][i] = static_cast<int16_t>(B[i] & 15);
                S.wm[r][i] = static_cast<int16_t>(B[i] >> 4);
            }
        }
        // half h: four weights per 32-bit word (the block is 4-byte aligned)
        const int h = part;
        uint32_t qs[8];
        for (int e = 0; e < 8; ++e) qs[e] = __ldg(reinterpret_cast<const uint32_t *>(B + 16 + 32 * h + 4 * e));
        for (int j = 0; j < 4; ++j) {
            uint32_t w[8];
            for (int e = 0; e < 8; ++e) w[e] = (qs[e] >> (2 * j)) & 0x03030303u;
            *reinterpret_cast<uint4 *>(dst + 128 * h + 32 * j) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4 *>(dst + 128 * h + 32 * j + 16) = make_uint4(w[4], w[5], w[6], w[7]);
        }
    } else {
        // Q8_0: this thread covers blocks 4*part .. 4*part+3 of the K step
        for (int bb = 4 * part; bb < 4 * part + 4; ++bb) {
            const int64_t kb = k0 / 32 + bb;
            if (n >= N || kb * 32 >= K) {
                for (int i = 0; i < 32; ++i) dst[32 * bb + i] = 0;
                S.wd8[r][bb] = 0.f;
                continue;
            }
            const uint8_t *B = W + (n * (K / 32) + kb) * 34;
            S.wd8[r][bb] = half_bits_to_float(B[0] | (B[1] << 8));
            for (int i = 0; i < 32; ++i) dst[32 * bb + i] = static_cast<int8_t>(B[2 + i]);
        }
    }
}

template <int T>
__global__ void __launch_bounds__(128) gemm_mma_kernel(const uint8_t *__restrict__ W, int64_t N,
                                                       int64_t K, const int8_t *__restrict__ xq,
                                                       const float *__restrict__ xd,
                                                       const int32_t *__restrict__ xs, int xd_ld,
                                                       const int32_t *__restrict__ xs16, int xs16_ld,
                                                       int64_t M, float *__restrict__ y) {
    __shared__ __align__(16) GemmSmem S;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int wm = warp >> 1, wn = warp & 1;
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * BM;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * BN;

    float acc[2][4][4];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[a][b][c] = 0.f;

    for (int64_t k0 = 0; k0 < K; k0 += BK) {
        const int64_t rem32 = (K - k0) / 32;
        const int nsub = rem32 < 8 ? static_cast<int>(rem32) : 8;
        // activations: 64 rows x 256 bytes, 16 B per thread per step
        for (int i = tid; i < BM * (BK / 16); i += 128) {
            const int r = i / (BK / 16), c16 = i % (BK / 16);
            const int64_t m = m0 + r;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (m < M && k0 + 16 * c16 < K) v = __ldg(reinterpret_cast<const uint4 *>(xq + m * K + k0 + 16 * c16));
            *reinterpret_cast<uint4 *>(&S.a[r][16 * c16]) = v;
        }
        for (int i = tid; i < BM * 8; i += 128) {
            const int r = i >> 3, j = i & 7;
            const int64_t m = m0 + r;
            const bool ok = m < M && j < nsub;
            S.xd[r][j] = ok ? xd[m * xd_ld + k0 / 32 + j] : 0.f;
            if constexpr (T == QMM_Q2_K) {
                // |half-block sum| <= 16 * 127: fits int16
                S.xs2[r][2 * j] = static_cast<int16_t>(ok ? xs16[m * xs16_ld + 2 * (k0 / 32 + j)] : 0);
                S.xs2[r][2 * j + 1] = static_cast<int16_t>(ok ? xs16[m * xs16_ld + 2 * (k0 / 32 + j) + 1] : 0);
            } else {
                S.xs[r][j] = ok ? xs[m * xd_ld + k0 / 32 + j] : 0;
            }
        }
        load_weights<T>(S, W, N, K, n0, k0);
        __syncthreads();

        for (int j = 0; j < nsub; ++j) {
            int I[2][4][4];
            int I2[2][4][4];
#pragma unroll
            for (int mi = 0; mi < 2; ++mi) {
                const int ra = 32 * wm + 16 * mi + g;
                uint32_t a[4];
                a[0] = *reinterpret_cast<const uint32_t *>(&S.a[ra][32 * j + 4 * t]);
                a[1] = *reinterpret_cast<const uint32_t *>(&S.a[ra + 8][32 * j + 4 * t]);
                a[2] = *reinterpret_cast<const uint32_t *>(&S.a[ra][32 * j + 16 + 4 * t]);
                a[3] = *reinterpret_cast<const uint32_t *>(&S.a[ra + 8][32 * j + 16 + 4 * t]);
#pragma unroll
                for (int ni = 0; ni < 4; ++ni) {
                    const int cb = 32 * wn + 8 * ni + g;
                    uint32_t b[2];
                    b[0] = *reinterpret_cast<const uint32_t *>(&S.b[cb][32 * j + 4 * t]);
                    b[1] = *reinterpret_cast<const uint32_t *>(&S.b[cb][32 * j + 16 + 4 * t]);
#pragma unroll
                    for (int e = 0; e < 4; ++e) I[mi][ni][e] = I2[mi][ni][e] = 0;
                    if constexpr (kGroups16<T>) {
                        mma_k16(I[mi][ni], a[0], a[1], b[0]);
                        mma_k16(I2[mi][ni], a[2], a[3], b[1]);
                    } else {
                        mma_k32(I[mi][ni], a, b);
                    }
                }
            }
            // per-block scaling
#pragma unroll
            for (int mi = 0; mi < 2; ++mi)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int r = 32 * wm + 16 * mi + g + 8 * hh;
                    const float dx = S.xd[r][j];
                    const int sx = T == QMM_Q2_K ? 0 : S.xs[r][j];
                    const int sa = T == QMM_Q2_K ? S.xs2[r][2 * j] : 0, sb = T == QMM_Q2_K ? S.xs2[r][2 * j + 1] : 0;
#pragma unroll
                    for (int ni = 0; ni < 4; ++ni)
#pragma unroll
                        for (int cc = 0; cc < 2; ++cc) {
                            const int c = 32 * wn + 8 * ni + 2 * t + cc;
                            const int e = 2 * hh + cc;
                            float v;
                            if constexpr (T == QMM_Q4_K || T == QMM_Q5_K) {
                                v = S.wd[c] * static_cast<float>(S.wsc[c][j] * I[mi][ni][e]) -
                                    S.wdmin[c] * static_cast<float>(S.wm[c][j] * sx);
                            } else if constexpr (T == QMM_Q6_K || T == QMM_Q3_K) {
                                const int J = S.wsc[c][2 * j] * I[mi][ni][e] + S.wsc[c][2 * j + 1] * I2[mi][ni][e];
                                v = S.wd[c] * static_cast<float>(J);
                            } else if constexpr (T == QMM_Q2_K) {
                                const int J = S.wsc[c][2 * j] * I[mi][ni][e] + S.wsc[c][2 * j + 1] * I2[mi][ni][e];
                                const int Mn = S.wm[c][2 * j] * sa + S.wm[c][2 * j + 1] * sb;
                                v = S.wd[c] * static_cast<float>(J) - S.wdmin[c] * static_cast<float>(Mn);
                            } else {
                                v = S.wd8[c][j] * static_cast<float>(I[mi][ni][e]);
                            }
                            acc[mi][ni][e] += dx * v;
                        }
                }
        }
        __syncthreads();
    }
    // store
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int64_t m = m0 + 32 * wm + 16 * mi + g + 8 * hh;
            if (m >= M) continue;
#pragma unroll
            for (int ni = 0; ni < 4; ++ni)
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int64_t n = n0 + 32 * wn + 8 * ni + 2 * t + cc;
                    if (n < N) y[m * N + n] = acc[mi][ni][2 * hh + cc];
                }
        }
}

}  // namespace

cudaError_t launch_gemm_mma(int type, const void *W, int64_t N, int64_t K, const int8_t *xq,
                            const float *xd, const int32_t *xs, int xd_ld, int64_t M, float *y,
                            cudaStream_t st, const int32_t *xs16, int xs16_ld) {
    if (type == QMM_Q2_K && !xs16) return cudaErrorInvalidValue;
    const dim3 grid(static_cast<unsigned>((N + BN - 1) / BN), static_cast<unsigned>((M + BM - 1) / BM));
    const auto *w = static_cast<const uint8_t *>(W);
    auto run = [&](auto t) {
        constexpr int T = decltype(t)::value;
        prefer_max_shared(gemm_mma_kernel<T>);
        gemm_mma_kernel<T><<<grid, 128, 0, st>>>(w, N, K, xq, xd, xs, xd_ld, xs16, xs16_ld, M, y);
    };
    switch (type) {
    case QMM_Q8_0: run(std::integral_constant<int, QMM_Q8_0>{}); break;
    case QMM_Q4_K: run(std::integral_constant<int, QMM_Q4_K>{}); break;
    case QMM_Q5_K: run(std::integral_constant<int, QMM_Q5_K>{}); break;
    case QMM_Q3_K: run(std::integral_constant<int, QMM_Q3_K>{}); break;
    case QMM_Q2_K: run(std::integral_constant<int, QMM_Q2_K>{}); break;
    default: run(std::integral_constant<int, QMM_Q6_K>{}); break;
    }
    return cudaGetLastError();
}

}  // namespace qk
