// gemm_tc.cu -- prefill product y[M,N] = W[N,K] . x[M,K]^T for Q4_K weights
// on the fifth-generation tensor cores (tcgen05, operands and accumulators in
// tensor memory).
//
// sm_103a has no integer tcgen05 mode, so the contraction runs in kind::f16
// with the roles chosen so that the dequantised weights never pass through
// shared memory:
//   A (128 x 64 per K step) = weights d*sc*q - dmin*m rounded to fp16, written
//       straight into TMEM by eight dequantiser warps (tcgen05.st) from the
//       raw super-block bytes that TMA brings into shared memory;
//   B (BT x 64) = the dequantised activations d_x*q_x rounded to fp16 (from the
//       quantiser), loaded by TMA with the 128-byte swizzle; BT = 64/128/256
//       tokens, so the weight tile is reused across up to 256 tokens;
//   D (128 x BT) = fp32 in TMEM: row = weight row n, column = token m.
// Each product term carries two fp16 roundings (relative 2^-11 each) and
// the sum is accumulated in fp32, well inside |dy| <= 2e-3*sum|w*x| + 1e-5.
//
// Warp roles: 0 = TMA producer (per 64-wide K step: the token tile, the
// 16-byte super-block header and the 32 quant bytes of each of the 128 weight
// rows), 1 = MMA issuer (and TMEM owner), then G groups of four dequantiser
// warps (warp w serves TMEM lanes 32*(w%4)..; group g takes the K steps
// g, g+G, ..., so G steps are dequantised at once) that finish as the
// epilogue (TMEM -> y).
// All waits are bounded; on a timeout the CTA stops issuing, drains what it
// issued, frees TMEM and returns with the status word set.
#include <cuda.h>
#include <stdlib.h>

#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qk {

namespace {

constexpr int BW = 128, BK = 64;  // weight rows per tile, K per step
constexpr int A_STAGES = 4;       // dequantised weight stages in TMEM (32 columns each)
constexpr int W_LOAD = 0, W_MMA = 1, W_DQ0 = 2;
constexpr int RAW_ROW = 144;        // one Q4_K super-block per weight row
constexpr int H_BYTES = BW * 16;    // d, dmin and the 12 scale bytes of each row
constexpr int Q_BYTES = BW * 32;    // this K step's 32 quant bytes of each row

template <int BT, int G>
struct TcCfg {
    static constexpr int NDQ = 4 * G;  // dequantiser warps: G groups of four lane quarters
    static constexpr int NTHREADS = (W_DQ0 + NDQ) * 32;
    static constexpr int X_BYTES = BT * BK * 2;
    static constexpr int L_BYTES = X_BYTES + H_BYTES + Q_BYTES;  // a multiple of 1024
    static constexpr int L_STAGES = BT == 256 ? 5 : 6;
    static constexpr int OFF_BAR = L_STAGES * L_BYTES;
    static constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;  // barriers + base alignment slack
    static constexpr int A_COL0 = BT;                         // TMEM columns of the A stages
    static constexpr int TMEM_COLS = BT + 32 * A_STAGES <= 256 ? 256 : 512;
    // D fp32, A and B fp16, both K-major, M = 128 weight rows, N = BT tokens
    static constexpr uint32_t IDESC = (1u << 4) | ((BT >> 3) << 17) | ((BW >> 4) << 24);
    static_assert(L_BYTES % 1024 == 0, "stage alignment");
    static_assert((BT / 16) % G == 0, "epilogue split");
    static_assert(SMEM_BYTES <= 232448, "shared memory");
};

struct TcParams {
    int M, N;
    int nsteps;   // 64-wide K steps per split; split z starts at z*nsteps
    float *y;
    int atomic;   // split K: add into y instead of storing
    int *status;
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
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 consecutive 32-bit columns (64 fp16 weights) into this warp's 32 TMEM
// lanes; the stores are complete when the function returns.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Four fp16 weights from the four bytes of a quant word (low nibbles, or
// high ones when hi): w = q*a + nb with q recovered exactly from the fp16
// bit pattern 0x6400 | q = 1024 + q.  Weights (b0,b1) -> out0, (b2,b3) -> out1.
__device__ __forceinline__ void dequant4(uint32_t w, bool hi, __half2 a, __half2 nb, uint32_t &out0,
                                         uint32_t &out1) {
    const __half2 k1024 = __half2half2(__ushort_as_half(0x6400));
    const uint32_t m = (hi ? (w >> 4) : w) & 0x0F0F0F0Fu;
    uint32_t t0 = __byte_perm(m, 0x64646464u, 0x4140u);
    uint32_t t1 = __byte_perm(m, 0x64646464u, 0x4342u);
    const __half2 w0 = __hfma2(__hsub2(*reinterpret_cast<const __half2 *>(&t0), k1024), a, nb);
    const __half2 w1 = __hfma2(__hsub2(*reinterpret_cast<const __half2 *>(&t1), k1024), a, nb);
    out0 = *reinterpret_cast<const uint32_t *>(&w0);
    out1 = *reinterpret_cast<const uint32_t *>(&w1);
}

template <int BT, int G>
__global__ void __launch_bounds__(TcCfg<BT, G>::NTHREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmH,
                   const __grid_constant__ CUtensorMap tmQ, const TcParams P) {
    using C = TcCfg<BT, G>;
    extern __shared__ uint8_t smem_raw[];
    // stages need 1024-byte alignment for the 128-byte swizzle
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BW, m0 = blockIdx.y * BT;
    const int k_step0 = blockIdx.z * P.nsteps;

    const uint32_t sL = smem_u32(smem);
    const uint32_t bar = smem_u32(smem + C::OFF_BAR);
    const uint32_t bar_l_full = bar, bar_l_empty = bar + 8 * C::L_STAGES;
    const uint32_t bar_a_full = bar + 16 * C::L_STAGES, bar_a_empty = bar_a_full + 8 * A_STAGES;
    const uint32_t bar_acc = bar_a_empty + 8 * A_STAGES;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_BAR + 224);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_BAR + 232);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::L_STAGES; ++s) {
            mbar_init(bar_l_full + 8 * s, 1);
            mbar_init(bar_l_empty + 8 * s, 1 + 4);  // the MMA commit + the four warps of the K step's group
        }
        for (int s = 0; s < A_STAGES; ++s) {
            mbar_init(bar_a_full + 8 * s, 4);
            mbar_init(bar_a_empty + 8 * s, 1);
        }
        mbar_init(bar_acc, 1);
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
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == W_LOAD) {
        // ------------------------------------------------------- producer
        if (lane == 0) {
            int issued = 0;
            for (int kk = 0; kk < P.nsteps; ++kk) {
                const int s = kk % C::L_STAGES;
                if (kk >= C::L_STAGES &&
                    (*abort_flag || !mbar_wait(bar_l_empty + 8 * s, ((kk / C::L_STAGES) - 1) & 1, P.status))) {
                    *abort_flag = 1;
                    break;
                }
                const int gk = k_step0 + kk;  // global 64-wide K step
                const uint32_t st = sL + s * C::L_BYTES;
                mbar_arrive_expect_tx(bar_l_full + 8 * s, C::L_BYTES);
                tma_load_2d(st, &tmX, gk * BK, m0, bar_l_full + 8 * s);
                tma_load_2d(st + C::X_BYTES, &tmH, (gk >> 2) * RAW_ROW, n0, bar_l_full + 8 * s);
                tma_load_2d(st + C::X_BYTES + H_BYTES, &tmQ, (gk >> 2) * RAW_ROW + 16 + 32 * (gk & 3), n0,
                            bar_l_full + 8 * s);
                ++issued;
            }
            // drain what is still in flight (only matters after an abort)
            for (int kk = issued > C::L_STAGES ? issued - C::L_STAGES : 0; kk < issued; ++kk)
                mbar_wait(bar_l_full + 8 * (kk % C::L_STAGES), (kk / C::L_STAGES) & 1, P.status);
        }
    } else if (warp == W_MMA) {
        // -------------------------------------------------- MMA issuer
        if (lane == 0) {
            for (int kk = 0; kk < P.nsteps; ++kk) {
                const int s = kk % C::L_STAGES, sa = kk % A_STAGES;
                if (*abort_flag || !mbar_wait(bar_l_full + 8 * s, (kk / C::L_STAGES) & 1, P.status) ||
                    !mbar_wait(bar_a_full + 8 * sa, (kk / A_STAGES) & 1, P.status)) {
                    *abort_flag = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t sx = sL + s * C::L_BYTES;
                const uint32_t ta = tmem + C::A_COL0 + 32 * sa;
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)
                    mma_ts(tmem, ta + 8 * k, desc_sw128(sx + 32 * k), C::IDESC, (kk | k) ? 1u : 0u);
                mma_commit(bar_l_empty + 8 * s);
                mma_commit(bar_a_empty + 8 * sa);
            }
            // the accumulator is final once every MMA issued above completes
            mma_commit(bar_acc);
        }
    } else {
        // ------------------------------------- dequantiser, then epilogue
        // group g = (warp - 2) / 4 dequantises the K steps kk = g, g+G, ...
        const int quarter = warp & 3, g = (warp - W_DQ0) >> 2;
        const int n = 32 * quarter + lane;  // weight row within the tile (= TMEM lane)
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * quarter) << 16);
        for (int kk = g; kk < P.nsteps; kk += G) {
            const int s = kk % C::L_STAGES, sa = kk % A_STAGES, c = (k_step0 + kk) & 3;
            bool ok = !*abort_flag;
            if (ok) ok = mbar_wait(bar_l_full + 8 * s, (kk / C::L_STAGES) & 1, P.status);
            if (ok && kk >= A_STAGES) ok = mbar_wait(bar_a_empty + 8 * sa, ((kk / A_STAGES) - 1) & 1, P.status);
            if (__any_sync(0xffffffffu, !ok)) {
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            const uint8_t *st = smem + s * C::L_BYTES + C::X_BYTES;
            const uint4 hdr = *reinterpret_cast<const uint4 *>(st + 16 * n);
            const uint4 qa = *reinterpret_cast<const uint4 *>(st + H_BYTES + 32 * n);
            const uint4 qb = *reinterpret_cast<const uint4 *>(st + H_BYTES + 32 * n + 16);
            // six-bit scales and mins of sub-blocks 2c (low nibbles) and 2c+1
            // (high nibbles), GGUF packing
            uint32_t scw, mw;
            if (c < 2) {
                scw = hdr.y & 0x3F3F3F3Fu;
                mw = hdr.z & 0x3F3F3F3Fu;
            } else {
                scw = (hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u);
                mw = ((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u);
            }
            const int sh = 16 * (c & 1);
            const float d = half_bits_to_float(hdr.x), dmin = half_bits_to_float(hdr.x >> 16);
            const __half2 ha0 = __float2half2_rn(d * static_cast<float>((scw >> sh) & 0xFF));
            const __half2 ha1 = __float2half2_rn(d * static_cast<float>((scw >> (sh + 8)) & 0xFF));
            const __half2 hb0 = __float2half2_rn(-(dmin * static_cast<float>((mw >> sh) & 0xFF)));
            const __half2 hb1 = __float2half2_rn(-(dmin * static_cast<float>((mw >> (sh + 8)) & 0xFF)));
            // weight l < 32 of the step is the low nibble of quant byte l,
            // weight 32 + l its high nibble; TMEM column i holds weights 2i, 2i+1
            const uint32_t qw[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
            uint32_t r[32];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                dequant4(qw[i], false, ha0, hb0, r[2 * i], r[2 * i + 1]);
                dequant4(qw[i], true, ha1, hb1, r[16 + 2 * i], r[16 + 2 * i + 1]);
            }
            tmem_st32(lane_base + C::A_COL0 + 32 * sa, r);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar_a_full + 8 * sa);
                mbar_arrive(bar_l_empty + 8 * s);
            }
        }
        // epilogue: TMEM lanes of this quarter, token columns [g*BT/G, (g+1)*BT/G)
        const bool ok = mbar_wait(bar_acc, 0, P.status);
        if (__all_sync(0xffffffffu, ok) && !*abort_flag) {
            tc_fence_after();
            const int ncol = n0 + n;
#pragma unroll 1
            for (int cc = g * (BT / G); cc < (g + 1) * (BT / G); cc += 16) {
                float v[16];
                tmem_ld16(lane_base + static_cast<uint32_t>(cc), v);
                if (ncol < P.N) {
                    float *yc = P.y + static_cast<int64_t>(m0 + cc) * P.N + ncol;
                    const int mrem = P.M - (m0 + cc);
                    if (P.atomic) {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (i < mrem) atomicAdd(yc + static_cast<int64_t>(i) * P.N, v[i]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (i < mrem) yc[static_cast<int64_t>(i) * P.N] = v[i];
                    }
                }
            }
        }
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
}

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
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

bool tc_supported(int type, int64_t N, int64_t K, int64_t M) {
    return type == QMM_Q4_K && K % 256 == 0 && K >= 256 && N >= 1 && M >= 1 && N <= (int64_t(1) << 30) &&
           M <= (int64_t(1) << 30) && K <= (int64_t(1) << 24) && encoder() != nullptr;
}

template <int BT, int G>
cudaError_t launch_bt(EncodeTiled enc, const void *W, int64_t N, int64_t K, const void *xh, int64_t M, float *y,
                      cudaStream_t st, int num_sms, int *status) {
    using C = TcCfg<BT, G>;
    CUtensorMap tx, th, tq;
    // tokens: fp16 [M][K], boxes of 64 K x BT rows, 128-byte swizzle
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
        const cuuint32_t box[2] = {BK, BT};
        const cuuint32_t es[2] = {1, 1};
        if (enc(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(xh), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // raw weights as bytes [N][row bytes]: 16-byte boxes (super-block header)
    // and 32-byte boxes (one K step's quants), 128 rows each
    const int64_t rb = (K / 256) * RAW_ROW;
    for (int which = 0; which < 2; ++which) {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(rb), static_cast<cuuint64_t>(N)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(rb)};
        const cuuint32_t box[2] = {which ? 32u : 16u, static_cast<cuuint32_t>(BW)};
        const cuuint32_t es[2] = {1, 1};
        if (enc(which ? &tq : &th, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(W), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const int nt = static_cast<int>((N + BW - 1) / BW), mt = static_cast<int>((M + BT - 1) / BT);
    const int ksteps = static_cast<int>(K / BK);
    // Split K in two when the tiles alone would leave most SMs idle (two
    // contributions per output keep the fp32 result independent of order).
    int splits = 1;
    if (2 * static_cast<int64_t>(nt) * mt <= num_sms && ksteps % 2 == 0) splits = 2;
    TcParams P;
    P.M = static_cast<int>(M);
    P.N = static_cast<int>(N);
    P.y = y;
    P.atomic = splits > 1;
    P.status = status;
    if (splits > 1) {
        cudaError_t e = cudaMemsetAsync(y, 0, static_cast<size_t>(M * N) * sizeof(float), st);
        if (e != cudaSuccess) return e;
    }
    cudaError_t e =
        cudaFuncSetAttribute(gemm_tc_kernel<BT, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    P.nsteps = ksteps / splits;
    gemm_tc_kernel<BT, G><<<dim3(nt, mt, splits), C::NTHREADS, C::SMEM_BYTES, st>>>(tx, th, tq, P);
    return cudaGetLastError();
}

}  // namespace

bool gemm_tc_supported(int type, int64_t N, int64_t K, int64_t M) { return tc_supported(type, N, K, M); }

cudaError_t launch_gemm_tc(int type, const void *W, int64_t N, int64_t K, const void *xh, int64_t M, float *y,
                           cudaStream_t st, int num_sms, int *status) {
    if (!gemm_tc_supported(type, N, K, M)) return cudaErrorNotSupported;
    EncodeTiled enc = encoder();
    static const int groups = [] {
        const char *e = getenv("QMM_TC_GROUPS");
        return e ? atoi(e) : 2;
    }();
#define QK_TC_LAUNCH(G)                                                                  \
    do {                                                                                 \
        if (M <= 64) return launch_bt<64, G>(enc, W, N, K, xh, M, y, st, num_sms, status);   \
        if (M <= 128) return launch_bt<128, G>(enc, W, N, K, xh, M, y, st, num_sms, status); \
        return launch_bt<256, G>(enc, W, N, K, xh, M, y, st, num_sms, status);               \
    } while (0)
    if (groups == 1) QK_TC_LAUNCH(1);
    if (groups == 4) QK_TC_LAUNCH(4);
    QK_TC_LAUNCH(2);
#undef QK_TC_LAUNCH
}

}  // namespace qk
