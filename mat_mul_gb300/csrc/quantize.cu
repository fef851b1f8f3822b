// quantize.cu -- the Q8_1-style activation quantiser: x[M,K] fp32 -> int8
// blocks of 32 with an fp32 scale and the int32 sum of the quantised values.
//
// Per block of 32 (the problem statement of the library; the pages only say
// that the dp4a kernels of blazr and infr take int8 activations):
//   amax = max|x|, d = amax/127, inv = 1/d (0 if d == 0),
//   q = round_half_away_from_zero(x * inv) clamped to [-127, 127], s = sum q.
// Every step is a separately rounded IEEE operation, so the output is
// bit-for-bit the same on every run and equal to a scalar CPU evaluation.
//
// Two kernels:
//   quantize_act_kernel: the int8 outputs (q, d, sums) for the dp4a decode
//     and the int8 mma.sync prefill, one warp per block of 32;
//   quantize_xh_kernel: the fp16 activations d*q of the fp16 tensor-core
//     paths (tcgen05 prefill, mma.sync decode).  fp16 holds 2^-24 .. 65504,
//     so each token row m is scaled by a power of two 2^e_m that puts the
//     row's largest |d*q| in [2^14, 2^15): the fp16 value is d*q*2^e_m with
//     one rounding, whatever the magnitude of x, and the consumers multiply
//     their fp32 results by xinv[m] = 2^-e_m (exact).  S CTAs per row each
//     find the row maximum themselves and quantise a slice of the row's
//     blocks; each thread quantises chunks of 8 elements, four lanes per
//     block.
#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qk {

namespace {

// The block of 32 held by lane i as v: the quantised value, the block scale
// and the block sum (warp-collective; every lane returns the same d, sum).
struct Quant {
    int q;
    float d;
    int sum;
};
__device__ __forceinline__ Quant quantize_block(float v) {
    // max of non-negative floats = max of their bit patterns as unsigned
    const uint32_t abits = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v)));
    const float amax = __uint_as_float(abits);
    const float db = __fdiv_rn(amax, 127.0f);
    const float inv = (db != 0.0f) ? __fdiv_rn(1.0f, db) : 0.0f;
    float r = roundf(__fmul_rn(v, inv));
    r = fminf(fmaxf(r, -127.0f), 127.0f);
    const int qi = static_cast<int>(r);
    const int sum = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<uint32_t>(qi)));
    return {qi, db, sum};
}

}  // namespace

// One warp per block of 32 activations, lane i holding element i: the int8
// outputs (q, d, s32, s16, dsf).
__global__ void __launch_bounds__(256) quantize_act_kernel(const float *__restrict__ x, int64_t M,
                                                           int64_t K, QuantOut o,
                                                           int trigger_dependents) {
    // a no-op unless launched with programmatic dependent launch
    pdl_wait();
    if (trigger_dependents) pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t nb = K / 32;
    const int64_t nblk = M * nb;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t g = warp; g < nblk; g += nwarps) {
        const int64_t m = g / nb, b = g - m * nb;
        const Quant r = quantize_block(__ldg(x + m * K + 32 * b + lane));
        const int qi = r.q;
        const int64_t k = 32 * b + lane;
        int64_t pos = k;
        if (o.swizzle) {
            const int64_t sb = k >> 8;
            const int c = static_cast<int>((k >> 4) & 15) ^ static_cast<int>(sb & 7);
            pos = (sb << 8) + 16 * c + (k & 15);
        }
        if (o.q) o.q[m * o.q_ld + pos] = static_cast<int8_t>(qi);
        int lo = 0;
        if (o.s16)
            lo = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<uint32_t>(lane < 16 ? qi : 0)));
        if (lane == 0) {
            if (o.d) o.d[m * o.d_ld + b] = r.d;
            if (o.s32) o.s32[m * o.d_ld + b] = r.sum;
            if (o.dsf) o.dsf[m * o.d_ld + b] = r.d * static_cast<float>(r.sum);
            if (o.s16) {
                o.s16[m * o.s16_ld + 2 * b] = lo;
                o.s16[m * o.s16_ld + 2 * b + 1] = r.sum - lo;
            }
        }
    }
}

namespace {

constexpr int XH_THREADS = 256;  // threads per CTA

// e_m for a row whose largest |x| has the bits amax_bits: the largest
// |d*q| (= amax up to one rounding) lands in [2^14, 2^15); clamped so that
// 2^e_m and 2^-e_m are normal fp32 values (rows below 2^-111 keep their
// values under 2^14, rows of zeros take e_m = 0).
__device__ __forceinline__ int row_exponent(uint32_t amax_bits) {
    if (amax_bits == 0) return 0;
    const int e = 14 - exponent_of(amax_bits);
    return min(max(e, -125), 125);
}

// Eight consecutive floats: two 16-byte loads when x is 16-byte aligned (the
// row starts are, K being a multiple of 32), else eight 4-byte loads.
__device__ __forceinline__ void load8(const float *p, bool vec, float (&v)[8]) {
    if (vec) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
        v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = b.x, v[5] = b.y, v[6] = b.z, v[7] = b.w;
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = __ldg(p + i);
    }
}

__device__ __forceinline__ uint32_t max_abs_bits8(const float (&v)[8]) {
    uint32_t a = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) a = max(a, __float_as_uint(fabsf(v[i])));
    return a;
}

}  // namespace

// fp16 activations with a per-row power of two.  CTA c of the grid works on
// row c / S and on slice c % S of the row's blocks of 32.  Each CTA first
// finds the largest |x| of the whole row itself (the row is read S times,
// from L2 after the first), then quantises its slice.  A thread takes chunks
// of 8 consecutive elements (chunk k: elements 8k .. 8k+7), so the four
// chunks of a block sit in four neighbouring lanes and one warp quantises
// eight blocks at once.
__global__ void __launch_bounds__(XH_THREADS) quantize_xh_kernel(const float *__restrict__ x, int64_t M,
                                                                int64_t K, QuantOut o, int S,
                                                                int trigger_dependents) {
    pdl_wait();
    if (trigger_dependents) pdl_trigger();
    __shared__ uint32_t s_warp[XH_THREADS / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t m = blockIdx.x / S;
    const int slice = static_cast<int>(blockIdx.x % S);
    const int64_t nb = K / 32, nch = K / 8;
    const int64_t bps = (nb + S - 1) / S;
    const int64_t c0 = 4 * slice * bps, c1 = 4 * min(nb, (slice + 1) * bps);  // the slice's chunks
    const float *xr = x + m * K;
    const bool vec = (reinterpret_cast<uintptr_t>(x) & 15) == 0;

    // pass 1: the row's largest |x|
    uint32_t amax = 0;
#pragma unroll 4
    for (int64_t c = tid; c < nch; c += XH_THREADS) {
        float w[8];
        load8(xr + 8 * c, vec, w);
        amax = max(amax, max_abs_bits8(w));
    }
    amax = __reduce_max_sync(0xffffffffu, amax);
    if (lane == 0) s_warp[warp] = amax;
    __syncthreads();
    amax = 0;
#pragma unroll
    for (int w = 0; w < XH_THREADS / 32; ++w) amax = max(amax, s_warp[w]);
    const int e = row_exponent(amax);
    const float scale = pow2f(e);
    if (slice == 0 && tid == 0 && o.xinv) o.xinv[m] = pow2f(-e);

    __half *row = static_cast<__half *>(o.xh) + m * o.xh_ld;
    const int u = lane & 3;  // which quarter of its block the chunk is
    // pass 2: the slice's chunks, c0 + tid + 256 t; a round exists for the
    // whole warp when its first chunk lies in the slice (warps stay
    // converged for the shuffles), lanes past the slice store nothing
    for (int64_t cw = c0 + (tid & ~31); cw < c1; cw += XH_THREADS) {
        const int64_t c = cw + lane;
        const bool live = c < c1;
        float w[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
        if (live) load8(xr + 8 * c, vec, w);
        uint32_t ab = max_abs_bits8(w);
        ab = max(ab, __shfl_xor_sync(0xffffffffu, ab, 1));
        ab = max(ab, __shfl_xor_sync(0xffffffffu, ab, 2));
        const float db = __fdiv_rn(__uint_as_float(ab), 127.0f);
        const float inv = (db != 0.0f) ? __fdiv_rn(1.0f, db) : 0.0f;
        __half hq[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float r = fminf(fmaxf(roundf(__fmul_rn(w[i], inv)), -127.0f), 127.0f);
            hq[i] = __float2half_rn(__fmul_rn(__fmul_rn(db, r), scale));
        }
        const int64_t b = c >> 2;
        if (!o.xh_mma) {
            if (live) {
                uint4 pk;
                pk.x = static_cast<uint32_t>(__half_as_ushort(hq[0])) | (static_cast<uint32_t>(__half_as_ushort(hq[1])) << 16);
                pk.y = static_cast<uint32_t>(__half_as_ushort(hq[2])) | (static_cast<uint32_t>(__half_as_ushort(hq[3])) << 16);
                pk.z = static_cast<uint32_t>(__half_as_ushort(hq[4])) | (static_cast<uint32_t>(__half_as_ushort(hq[5])) << 16);
                pk.w = static_cast<uint32_t>(__half_as_ushort(hq[6])) | (static_cast<uint32_t>(__half_as_ushort(hq[7])) << 16);
                *reinterpret_cast<uint4 *>(row + 8 * c) = pk;
            }
            continue;
        }
        // fragment order: element l of block b at 32b + ((l>>4)*2 + (l&1))*8
        // + ((l>>2)&3)*2 + ((l>>1)&1); then the block sums of the fp16
        // values times 2^-5 (so that 32 values below 2^15 sum below 2^15),
        // X = hi + lo, in two planes of 8 per super-block after K
        float x8 = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int l = 8 * u + i;
            if (live) row[32 * b + ((l >> 4) * 2 + (l & 1)) * 8 + ((l >> 2) & 3) * 2 + ((l >> 1) & 1)] = hq[i];
            x8 += __half2float(hq[i]);
        }
        // the sums of the two groups of 16 and of the block.  A group sum
        // X_G times 2^-4 (16 values below 2^15 sum below 2^15) as fp16 hi +
        // lo, in the B-operand tiles of the Q6_K kernel: per super-block
        // [hi | lo][groups 0-7 | 8-15][8 tokens][8 groups], zeros for the
        // tokens M..7 (written with token 0)
        const float x16 = x8 + __shfl_xor_sync(0xffffffffu, x8, 1);
        const float xs = x16 + __shfl_xor_sync(0xffffffffu, x16, 2);
        if (live && o.xs16 && (u & 1) == 0) {
            const int64_t gidx = 2 * b + (u >> 1);
            const int G = static_cast<int>(gidx & 15);
            __half *tile = reinterpret_cast<__half *>(o.xs16) + (gidx >> 4) * 256 + (G >> 3) * 64 + (G & 7);
            const float v = x16 * 0.0625f;
            const __half hi = __float2half_rn(v);
            tile[8 * m] = hi;
            tile[128 + 8 * m] = __float2half_rn(v - __half2float(hi));
            if (m == 0)
                for (int64_t mm = M; mm < 8; ++mm) tile[8 * mm] = tile[128 + 8 * mm] = __float2half_rn(0.0f);
        }
        if (live && u == 0) {
            // sub-block j of the super-block at slot 2(j mod 4) + j/4: the
            // tensor-core kernel's lane t holds the mins of sub-blocks t, t+4
            const int j = static_cast<int>(b & 7);
            const int slot = 2 * (j & 3) + (j >> 2);
            const float xs5 = xs * 0.03125f;
            const __half hi = __float2half_rn(xs5);
            const __half lo = __float2half_rn(xs5 - __half2float(hi));
            row[K + (b >> 3) * 16 + slot] = hi;
            row[K + (b >> 3) * 16 + 8 + slot] = lo;
        }
    }
}

// CTAs per row for the fp16 quantiser: one chunk of 8 per thread for the
// few rows of a decode call (parallelism), about eight for a prefill
// (each CTA re-reads the row to find its maximum).
int xh_slices(int64_t M, int64_t K) {
    const int64_t per_cta = static_cast<int64_t>(XH_THREADS) * 8 * (M <= 8 ? 1 : 8);
    int64_t s = (K + per_cta - 1) / per_cta;
    return static_cast<int>(s < 1 ? 1 : s > 64 ? 64 : s);
}

// Host launcher.  int8 outputs: enough warps for every block, capped at a
// few waves.  fp16 outputs: xh_slices(M, K) CTAs per row.
cudaError_t launch_quantize(const float *x, int64_t M, int64_t K, const QuantOut &o, cudaStream_t st,
                            bool trigger_dependents, int num_sms, bool pdl_launch) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    int na = 0;
    if (pdl_launch) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.stream = st;
    if (o.xh) {
        const int S = xh_slices(M, K);
        if (M * S > 0x7fffffffLL) return cudaErrorInvalidValue;
        cfg.gridDim = dim3(static_cast<unsigned>(M * S));
        cfg.blockDim = dim3(XH_THREADS);
        cfg.attrs = na ? attr : nullptr;
        cfg.numAttrs = na;
        const cudaError_t e = prefer_max_shared(quantize_xh_kernel);
        if (e != cudaSuccess) return e;
        return cudaLaunchKernelEx(&cfg, quantize_xh_kernel, x, M, K, o, S, trigger_dependents ? 1 : 0);
    }
    const int64_t nblk = M * (K / 32);
    int64_t grid = (nblk + 7) / 8;
    const int64_t cap = static_cast<int64_t>(num_sms) * 16;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(256);
    cfg.attrs = na ? attr : nullptr;
    cfg.numAttrs = na;
    const cudaError_t e = prefer_max_shared(quantize_act_kernel);
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&cfg, quantize_act_kernel, x, M, K, o, trigger_dependents ? 1 : 0);
}

}  // namespace qk
