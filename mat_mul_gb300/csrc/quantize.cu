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

namespace qk {

// One warp per block of 32 activations, lane i holding element i.
// q rows have stride q_ld bytes and d rows ds_ld floats.  With sum16 == 0, s
// holds one int32 sum per block (rows of ds_ld); with sum16 != 0 it holds the
// sums of the two 16-element halves of every block (rows of s_ld), the form
// the decode kernels use.
__global__ void __launch_bounds__(256) quantize_act_kernel(const float *__restrict__ x, int64_t M,
                                                           int64_t K, int8_t *__restrict__ q,
                                                           int64_t q_ld, float *__restrict__ d,
                                                           int32_t *__restrict__ s, int64_t ds_ld,
                                                           int64_t s_ld, int sum16,
                                                           int trigger_dependents) {
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
        q[m * q_ld + 32 * b + lane] = static_cast<int8_t>(qi);
        if (sum16) {
            const int lo = static_cast<int>(
                __reduce_add_sync(0xffffffffu, static_cast<uint32_t>(lane < 16 ? qi : 0)));
            if (lane == 0) {
                d[m * ds_ld + b] = db;
                s[m * s_ld + 2 * b] = lo;
                s[m * s_ld + 2 * b + 1] = sum - lo;
            }
        } else if (lane == 0) {
            d[m * ds_ld + b] = db;
            s[m * ds_ld + b] = sum;
        }
    }
}

// Host launcher.  Grid: enough warps for every block, capped at a few waves.
cudaError_t launch_quantize(const float *x, int64_t M, int64_t K, int8_t *q, int64_t q_ld, float *d,
                            int32_t *s, int64_t ds_ld, int64_t s_ld, bool sum16, cudaStream_t st,
                            bool trigger_dependents, int num_sms) {
    const int64_t nblk = M * (K / 32);
    const int threads = 256;
    int64_t grid = (nblk + 7) / 8;
    const int64_t cap = static_cast<int64_t>(num_sms) * 16;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    quantize_act_kernel<<<static_cast<unsigned>(grid), threads, 0, st>>>(
        x, M, K, q, q_ld, d, s, ds_ld, s_ld, sum16 ? 1 : 0, trigger_dependents ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace qk
