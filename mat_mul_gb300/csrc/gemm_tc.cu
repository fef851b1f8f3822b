// gemm_tc.cu -- prefill product y[M,N] = W[N,K] . x[M,K]^T for Q4_K weights
// on the fifth-generation tensor cores (tcgen05, accumulators in TMEM).
//
// sm_103a has no integer tcgen05 mode, so the contraction runs in kind::f16:
//   A = the dequantised activations d_x*q_x rounded to fp16 (from the
//       quantiser), loaded by TMA with the 128-byte swizzle;
//   B = the dequantised weights d*sc*q - dmin*m rounded to fp16, produced in
//       shared memory by eight warps from raw super-blocks that TMA brings in;
//   D = fp32 in TMEM, 128 x 256 per CTA.
// Each product term carries two fp16 roundings (relative 2^-11 each) and
// the sum is accumulated in fp32, well inside |dy| <= 2e-3*sum|w*x| + 1e-5.
//
// Warp roles (11 warps): 0 = TMA producer of A, 1 = MMA issuer (and TMEM
// owner), 2 = TMA producer of raw weight super-blocks, 3..10 = dequantiser
// (one weight row each per K step) and then epilogue (TMEM -> y).
// Pipelines: A/B ring of 3 stages of 64 K, raw ring of 2 super-blocks.  All
// waits are bounded; on a timeout the CTA stops issuing, drains what it
// issued, frees TMEM and returns with the status word set.
#include <cuda.h>

#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qk {

namespace {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int STAGES = 3, RAW_STAGES = 2;
constexpr int NDQ = 8;
constexpr int W_A = 0, W_MMA = 1, W_RAW = 2, W_DQ0 = 3;
constexpr int NTHREADS = (W_DQ0 + NDQ) * 32;
constexpr int A_BYTES = BM * BK * 2;   // 16 KB
constexpr int B_BYTES = BN * BK * 2;   // 32 KB
constexpr int RAW_ROW = 144;           // one Q4_K super-block per weight row
constexpr int RAW_BYTES = BN * RAW_ROW;
constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
constexpr int OFF_RAW = OFF_B + STAGES * B_BYTES;
constexpr int OFF_BAR = OFF_RAW + RAW_STAGES * RAW_BYTES;
constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;  // barriers + base alignment slack
constexpr int TMEM_COLS = 256;

struct TcParams {
    int M, N;
    int nsteps;   // 64-wide K steps per split (a multiple of 4); split z starts at z*nsteps
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

// Instruction descriptor: D fp32, A and B fp16, both K-major, M = 128, N = 256.
constexpr uint32_t IDESC = (1u << 4) | (0u << 7) | (0u << 10) | ((BN >> 3) << 17) | ((BM >> 4) << 24);

__device__ __forceinline__ void mma_f16(uint32_t tmem, uint64_t a, uint64_t b, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
        "l"(a), "l"(b), "r"(IDESC), "r"(acc)
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

__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 32 consecutive fp32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
          "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
          "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Eight fp16 weights (one 16-byte chunk) from the nibbles of two quant words:
// hi selects the high nibbles; w = q*a + nb with q recovered exactly from the
// fp16 bit pattern 0x6400 | q = 1024 + q.
__device__ __forceinline__ uint4 dequant8(uint32_t w0, uint32_t w1, bool hi, __half2 a, __half2 nb) {
    const __half2 k1024 = __half2half2(__ushort_as_half(0x6400));
    uint32_t out[4];
    const uint32_t ws[2] = {w0, w1};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            // bytes 2p and 2p+1 of the word into the low byte of each 16-bit half
            uint32_t t = __byte_perm(ws[i], 0u, p ? 0x4342u : 0x4140u);
            if (hi) t >>= 4;
            t = (t & 0x000F000Fu) | 0x64006400u;
            const __half2 q = __hsub2(*reinterpret_cast<const __half2 *>(&t), k1024);
            const __half2 wv = __hfma2(q, a, nb);
            out[2 * i + p] = *reinterpret_cast<const uint32_t *>(&wv);
        }
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
}

__global__ void __launch_bounds__(NTHREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                   const TcParams P) {
    extern __shared__ uint8_t smem_raw[];
    // stages need 1024-byte alignment for the 128-byte swizzle
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BN, m0 = blockIdx.y * BM;
    const int k_step0 = blockIdx.z * P.nsteps;

    const uint32_t sA = smem_u32(smem + OFF_A), sB = smem_u32(smem + OFF_B), sRaw = smem_u32(smem + OFF_RAW);
    const uint32_t bar = smem_u32(smem + OFF_BAR);
    const uint32_t bar_a_full = bar, bar_b_full = bar + 8 * STAGES, bar_ab_empty = bar + 16 * STAGES;
    const uint32_t bar_raw_full = bar + 24 * STAGES, bar_raw_empty = bar_raw_full + 8 * RAW_STAGES;
    const uint32_t bar_acc = bar_raw_empty + 8 * RAW_STAGES;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_BAR + 200);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_BAR + 208);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_a_full + 8 * s, 1);
            mbar_init(bar_b_full + 8 * s, NDQ);
            mbar_init(bar_ab_empty + 8 * s, 1);
        }
        for (int r = 0; r < RAW_STAGES; ++r) {
            mbar_init(bar_raw_full + 8 * r, 1);
            mbar_init(bar_raw_empty + 8 * r, NDQ);
        }
        mbar_init(bar_acc, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == W_MMA) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int nsb = P.nsteps / 4;  // super-blocks of this split

    if (warp == W_A) {
        // ---------------------------------------------------- A producer
        if (lane == 0) {
            int issued = 0;
            for (int kk = 0; kk < P.nsteps; ++kk) {
                const int s = kk % STAGES;
                if (kk >= STAGES &&
                    (*abort_flag || !mbar_wait(bar_ab_empty + 8 * s, ((kk / STAGES) - 1) & 1, P.status))) {
                    *abort_flag = 1;
                    break;
                }
                mbar_arrive_expect_tx(bar_a_full + 8 * s, A_BYTES);
                tma_load_2d(sA + s * A_BYTES, &tmA, (k_step0 + kk) * BK, m0, bar_a_full + 8 * s);
                ++issued;
            }
            // drain what is still in flight (only matters after an abort)
            for (int kk = issued > STAGES ? issued - STAGES : 0; kk < issued; ++kk)
                mbar_wait(bar_a_full + 8 * (kk % STAGES), (kk / STAGES) & 1, P.status);
        }
    } else if (warp == W_RAW) {
        // ------------------------------------------- raw weight producer
        if (lane == 0) {
            int issued = 0;
            for (int sb = 0; sb < nsb; ++sb) {
                const int r = sb % RAW_STAGES;
                if (sb >= RAW_STAGES &&
                    (*abort_flag || !mbar_wait(bar_raw_empty + 8 * r, ((sb / RAW_STAGES) - 1) & 1, P.status))) {
                    *abort_flag = 1;
                    break;
                }
                mbar_arrive_expect_tx(bar_raw_full + 8 * r, RAW_BYTES);
                tma_load_2d(sRaw + r * RAW_BYTES, &tmW, (k_step0 / 4 + sb) * RAW_ROW, n0, bar_raw_full + 8 * r);
                ++issued;
            }
            for (int sb = issued > RAW_STAGES ? issued - RAW_STAGES : 0; sb < issued; ++sb)
                mbar_wait(bar_raw_full + 8 * (sb % RAW_STAGES), (sb / RAW_STAGES) & 1, P.status);
        }
    } else if (warp == W_MMA) {
        // -------------------------------------------------- MMA issuer
        if (lane == 0) {
            for (int kk = 0; kk < P.nsteps; ++kk) {
                const int s = kk % STAGES;
                const uint32_t par = (kk / STAGES) & 1;
                if (*abort_flag || !mbar_wait(bar_a_full + 8 * s, par, P.status) ||
                    !mbar_wait(bar_b_full + 8 * s, par, P.status)) {
                    *abort_flag = 1;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)
                    mma_f16(tmem, desc_sw128(sA + s * A_BYTES + 32 * k), desc_sw128(sB + s * B_BYTES + 32 * k),
                            (kk | k) ? 1u : 0u);
                mma_commit(bar_ab_empty + 8 * s);
            }
            // the accumulator is final once every MMA issued above completes
            mma_commit(bar_acc);
        }
    } else {
        // ------------------------------------- dequantiser, then epilogue
        const int dq = warp - W_DQ0;
        const int n = dq * 32 + lane;  // weight row within the tile
        for (int kk = 0; kk < P.nsteps; ++kk) {
            const int s = kk % STAGES, c = kk & 3, sb = kk >> 2, r = sb % RAW_STAGES;
            bool ok = !*abort_flag;
            if (ok && c == 0) ok = mbar_wait(bar_raw_full + 8 * r, (sb / RAW_STAGES) & 1, P.status);
            if (ok && kk >= STAGES) ok = mbar_wait(bar_ab_empty + 8 * s, ((kk / STAGES) - 1) & 1, P.status);
            if (__any_sync(0xffffffffu, !ok)) {
                *abort_flag = 1;
                break;
            }
            const uint8_t *row = smem + OFF_RAW + r * RAW_BYTES + n * RAW_ROW;
            const uint4 hdr = *reinterpret_cast<const uint4 *>(row);
            const uint4 qa = *reinterpret_cast<const uint4 *>(row + 16 + 32 * c);
            const uint4 qb = *reinterpret_cast<const uint4 *>(row + 32 + 32 * c);
            // six-bit scales and mins of sub-blocks 2c (low nibbles) and 2c+1 (high)
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
            const float a0 = d * static_cast<float>((scw >> sh) & 0xFF);
            const float a1 = d * static_cast<float>((scw >> (sh + 8)) & 0xFF);
            const float b0 = dmin * static_cast<float>((mw >> sh) & 0xFF);
            const float b1 = dmin * static_cast<float>((mw >> (sh + 8)) & 0xFF);
            const __half2 ha0 = __float2half2_rn(a0), ha1 = __float2half2_rn(a1);
            const __half2 hb0 = __float2half2_rn(-b0), hb1 = __float2half2_rn(-b1);
            // chunk i holds weights 8i..8i+7 of this K step: i < 4 low nibbles
            // of qs bytes 8i.., i >= 4 high nibbles of bytes 8(i-4)..
            uint4 ch[8];
            ch[0] = dequant8(qa.x, qa.y, false, ha0, hb0);
            ch[1] = dequant8(qa.z, qa.w, false, ha0, hb0);
            ch[2] = dequant8(qb.x, qb.y, false, ha0, hb0);
            ch[3] = dequant8(qb.z, qb.w, false, ha0, hb0);
            ch[4] = dequant8(qa.x, qa.y, true, ha1, hb1);
            ch[5] = dequant8(qa.z, qa.w, true, ha1, hb1);
            ch[6] = dequant8(qb.x, qb.y, true, ha1, hb1);
            ch[7] = dequant8(qb.z, qb.w, true, ha1, hb1);
            uint8_t *brow = smem + OFF_B + s * B_BYTES + (n >> 3) * 1024 + (n & 7) * 128;
#pragma unroll
            for (int i = 0; i < 8; ++i) *reinterpret_cast<uint4 *>(brow + 16 * (i ^ (n & 7))) = ch[i];
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar_b_full + 8 * s);
                if (c == 3) mbar_arrive(bar_raw_empty + 8 * r);
            }
        }
        // epilogue: this warp reads TMEM lanes 32*(warp%4).., half of the columns
        const bool ok = mbar_wait(bar_acc, 0, P.status);
        if (__all_sync(0xffffffffu, ok) && !*abort_flag) {
            tc_fence_after();
            const int q = warp & 3, half = dq >> 2;
            const int m = m0 + 32 * q + lane;
#pragma unroll 1
            for (int cc = 0; cc < BN / 2; cc += 32) {
                float v[32];
                tmem_ld32(tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(half * (BN / 2) + cc), v);
                const int nc = n0 + half * (BN / 2) + cc;
                if (m < P.M) {
                    float *yr = P.y + static_cast<int64_t>(m) * P.N + nc;
                    if (P.atomic) {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (nc + i < P.N) atomicAdd(yr + i, v[i]);
                    } else if (nc + 32 <= P.N && (P.N & 3) == 0) {
#pragma unroll
                        for (int i = 0; i < 32; i += 4)
                            *reinterpret_cast<float4 *>(yr + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (nc + i < P.N) yr[i] = v[i];
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
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS)
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

}  // namespace

bool gemm_tc_supported(int type, int64_t N, int64_t K, int64_t M) {
    return type == QMM_Q4_K && K % 256 == 0 && K >= 256 && N >= 1 && M >= 1 && N <= (int64_t(1) << 30) &&
           M <= (int64_t(1) << 30) && K <= (int64_t(1) << 24) && encoder() != nullptr;
}

cudaError_t launch_gemm_tc(int type, const void *W, int64_t N, int64_t K, const void *xh, int64_t M, float *y,
                           cudaStream_t st, int num_sms, int *status) {
    if (!gemm_tc_supported(type, N, K, M)) return cudaErrorNotSupported;
    EncodeTiled enc = encoder();
    CUtensorMap ta, tw;
    // A: fp16 [M][K], boxes of 64 K x 128 rows, 128-byte swizzle
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
        const cuuint32_t box[2] = {BK, BM};
        const cuuint32_t es[2] = {1, 1};
        if (enc(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(xh), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // raw weights: bytes [N][row bytes], boxes of one super-block x 256 rows
    {
        const int64_t rb = (K / 256) * RAW_ROW;
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(rb), static_cast<cuuint64_t>(N)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(rb)};
        const cuuint32_t box[2] = {RAW_ROW, BN};
        const cuuint32_t es[2] = {1, 1};
        if (enc(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(W), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const int nt = static_cast<int>((N + BN - 1) / BN), mt = static_cast<int>((M + BM - 1) / BM);
    const int ksteps = static_cast<int>(K / BK);
    // split K in two when the tiles would leave most SMs idle
    int splits = 1;
    if (2 * nt * mt <= num_sms && (ksteps / 4) % 2 == 0) splits = 2;
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
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    P.nsteps = ksteps / splits;
    gemm_tc_kernel<<<dim3(nt, mt, splits), NTHREADS, SMEM_BYTES, st>>>(ta, tw, P);
    return cudaGetLastError();
}

}  // namespace qk
