// quantize.cu -- the Q8_1-style activation quantiser: x[M,K] fp32 -> int8
// blocks of 32 with an fp32 scale and the int32 sum of the quantised values.
//
// Per block of 32 (the problem statement of the library; the pages only say
// that the dp4a kernels of blazr and infr take int8 activations):
//   amax = max|x|, d = amax/127, inv = 1/d (0 if d == 0),
//   q = round_half_away_from_zero(x * inv) clamped to [-127, 127], s = sum q.
// Every step is a separately rounded IEEE operation, so the output is
// bit-for-bit the same on every run and equal to a scalar CPU evaluation.
#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qk {

// One warp per block of 32 activations, lane i holding element i.
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
        const float v = __ldg(x + m * K + 32 * b + lane);
        // max of non-negative floats = max of their bit patterns as unsigned
        const uint32_t abits = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v)));
        const float amax = __uint_as_float(abits);
        const float db = __fdiv_rn(amax, 127.0f);
        const float inv = (db != 0.0f) ? __fdiv_rn(1.0f, db) : 0.0f;
        float r = roundf(__fmul_rn(v, inv));
        r = fminf(fmaxf(r, -127.0f), 127.0f);
        const int qi = static_cast<int>(r);
        const int sum = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<uint32_t>(qi)));
        const int64_t k = 32 * b + lane;
        int64_t pos = k;
        if (o.swizzle) {
            const int64_t sb = k >> 8;
            const int c = static_cast<int>((k >> 4) & 15) ^ static_cast<int>(sb & 7);
            pos = (sb << 8) + 16 * c + (k & 15);
        }
        if (o.q) o.q[m * o.q_ld + pos] = static_cast<int8_t>(qi);
        if (o.xh) {
            const __half hq = __float2half_rn(__fmul_rn(db, static_cast<float>(qi)));
            __half *row = static_cast<__half *>(o.xh) + m * o.xh_ld;
            if (!o.xh_mma) {
                row[k] = hq;
            } else {
                // fragment order: element l of block b at 32b + ((l>>4)*2 + (l&1))*8
                // + ((l>>2)&3)*2 + ((l>>1)&1); then the block sums of the fp16
                // values, X = hi + lo, in two planes of 8 per super-block after K
                row[32 * b + ((lane >> 4) * 2 + (lane & 1)) * 8 + ((lane >> 2) & 3) * 2 + ((lane >> 1) & 1)] = hq;
                float x16 = __half2float(hq);
#pragma unroll
                for (int o2 = 8; o2 >= 1; o2 >>= 1) x16 += __shfl_xor_sync(0xffffffffu, x16, o2);
                const float xs = x16 + __shfl_xor_sync(0xffffffffu, x16, 16);
                // the sums of the two groups of 16: [K/16][8 tokens], zeros for
                // the tokens M..7 (written with token 0)
                if (o.xs16 && (lane & 15) == 0) {
                    float *gs = o.xs16 + (2 * b + (lane >> 4)) * 8;
                    gs[m] = x16;
                    if (m == 0)
                        for (int64_t mm = M; mm < 8; ++mm) gs[mm] = 0.0f;
                }
                if (lane == 0) {
                    const __half hi = __float2half_rn(xs);
                    const __half lo = __float2half_rn(xs - __half2float(hi));
                    row[K + (b >> 3) * 16 + (b & 7)] = hi;
                    row[K + (b >> 3) * 16 + 8 + (b & 7)] = lo;
                }
            }
        }
        int lo = 0;
        if (o.s16)
            lo = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<uint32_t>(lane < 16 ? qi : 0)));
        if (lane == 0) {
            if (o.d) o.d[m * o.d_ld + b] = db;
            if (o.s32) o.s32[m * o.d_ld + b] = sum;
            if (o.dsf) o.dsf[m * o.d_ld + b] = db * static_cast<float>(sum);
            if (o.s16) {
                o.s16[m * o.s16_ld + 2 * b] = lo;
                o.s16[m * o.s16_ld + 2 * b + 1] = sum - lo;
            }
        }
    }
}

// Host launcher.  Grid: enough warps for every block, capped at a few waves.
cudaError_t launch_quantize(const float *x, int64_t M, int64_t K, const QuantOut &o, cudaStream_t st,
                            bool trigger_dependents, int num_sms, bool pdl_launch) {
    const int64_t nblk = M * (K / 32);
    const int threads = 256;
    int64_t grid = (nblk + 7) / 8;
    const int64_t cap = static_cast<int64_t>(num_sms) * 16;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    if (!pdl_launch) {
        quantize_act_kernel<<<static_cast<unsigned>(grid), threads, 0, st>>>(x, M, K, o,
                                                                            trigger_dependents ? 1 : 0);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(threads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, quantize_act_kernel, x, M, K, o, trigger_dependents ? 1 : 0);
}

}  // namespace qk
