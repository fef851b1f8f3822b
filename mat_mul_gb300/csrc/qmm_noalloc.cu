// qmm_noalloc.cu -- qmm_noalloc(): the prefill product (activation quantiser
// + integer tensor-core GEMM) run entirely out of a fixed scratch area that
// is part of the library image, so the call itself never allocates.
//
// Who needs it: callers that cannot let a library allocate device memory --
// serving loops that keep every byte of device memory in their own fixed
// pool (a library cudaMalloc would take memory outside that budget, and may
// fail at the worst moment when the pool has claimed the rest), and
// latency-critical loops that must not stall on cudaFree, which synchronises
// the whole device.  qmm() instead grows a per-stream workspace on demand.
//
// The scratch is a file-scope __device__ array: every GPU that loads the
// library reserves it until the process exits.  Host code must not use the
// array's name as a device address (on the host it names a stand-in, not
// the GPU copy); each device's address is looked up once with
// cudaGetSymbolAddress while that device is current.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/qmm.h"
#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;  // 16 MiB
__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
struct NoallocDevice {
    bool ready = false;
    void *scratch = nullptr;  // device address of g_noalloc_scratch on this device
    int num_sms = 0;
};
std::mutex g_noalloc_mu;
NoallocDevice g_noalloc_dev[kMaxDevices];

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Scratch layout for M rows of K activations: q int8 [M][K] | d fp32
// [M][ld] | s int32 [M][ld], ld = K/32 rounded up to 4, each part on 256 B.
size_t scratch_need(int64_t M, int64_t K, int64_t *ld) {
    *ld = static_cast<int64_t>(round_up(static_cast<size_t>(K / 32), 4));
    return round_up(static_cast<size_t>(M * K), 256) + 2 * round_up(static_cast<size_t>(M * *ld) * 4, 256);
}

int err(int code, const char *fmt, long long a = 0, long long b = 0) {
    char buf[256];
    snprintf(buf, sizeof buf, fmt, a, b);
    return qk::record_error(code, buf);
}

}  // namespace

extern "C" QMM_API int qmm_noalloc(int type, const void *W_blocks, int64_t N, int64_t K, const float *x,
                                   int64_t M, float *y, void *stream) {
    if (type != QMM_Q8_0 && type != QMM_Q4_K && type != QMM_Q6_K)
        return err(QMM_EINVAL_TYPE, "block type %lld: qmm_noalloc takes Q8_0, Q4_K and Q6_K", type);
    const int qkw = qk::block_weights(type);
    if (N < 0 || M < 0 || K < 0 || K % qkw)
        return err(QMM_EINVAL_SHAPE, "N, K, M must be >= 0 and K a multiple of %lld (K=%lld)", qkw, K);
    if (K > (int64_t(1) << 24)) return err(QMM_EINVAL_SHAPE, "K=%lld exceeds 2^24", K);
    // M*K and M*ld*4 below must not wrap: M is bounded by what the scratch
    // could hold at all before anything is multiplied
    if (K > 0 && M > static_cast<int64_t>(kScratchBytes) / K)
        return err(QMM_EINVAL_SHAPE, "M=%lld rows of K=%lld exceed the static scratch", M, K);
    if (N > (int64_t(1) << 31)) return err(QMM_EINVAL_SHAPE, "N=%lld exceeds 2^31", N);
    if (M == 0 || N == 0) return qk::record_error(QMM_OK, "");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (!y || (reinterpret_cast<uintptr_t>(y) & 3)) return err(QMM_EINVAL_PTR, "y must be non-null and 4-byte aligned");
    if (K == 0) {
        cudaError_t e = cudaMemsetAsync(y, 0, static_cast<size_t>(M * N) * sizeof(float), st);
        if (e != cudaSuccess) return err(QMM_ECUDA, "zero fill failed (cuda error %lld)", e);
        return qk::record_error(QMM_OK, "");
    }
    if (!W_blocks || !x) return err(QMM_EINVAL_PTR, "null pointer");
    if (reinterpret_cast<uintptr_t>(W_blocks) & 15) return err(QMM_EINVAL_PTR, "W_blocks must be 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(x) & 3) return err(QMM_EINVAL_PTR, "x must be 4-byte aligned");
    int64_t ld = 0;
    const size_t need = scratch_need(M, K, &ld);
    if (need > kScratchBytes)
        return err(QMM_EINVAL_SHAPE,
                   "M*K too large for the static scratch: needs %lld bytes, the scratch holds %lld",
                   static_cast<long long>(need), static_cast<long long>(kScratchBytes));

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return err(QMM_ECUDA, "cudaGetDevice failed (cuda error %lld)", e);
    if (dev < 0 || dev >= kMaxDevices) return err(QMM_ECUDA, "device index %lld out of range", dev);
    NoallocDevice d;
    {
        std::lock_guard<std::mutex> lk(g_noalloc_mu);
        NoallocDevice &slot = g_noalloc_dev[dev];
        if (!slot.ready) {
            // first call on this device: find the scratch's device address
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess) return err(QMM_ECUDA, "cudaGetSymbolAddress failed (cuda error %lld)", e);
            int sms = 0;
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return err(QMM_ECUDA, "device query failed (cuda error %lld)", e);
            slot.scratch = p;
            slot.num_sms = sms;
            slot.ready = true;
        }
        d = slot;
    }
    char *s = static_cast<char *>(d.scratch);
    const size_t q_bytes = round_up(static_cast<size_t>(M * K), 256);
    const size_t d_bytes = round_up(static_cast<size_t>(M * ld) * 4, 256);
    qk::QuantOut o = {};
    o.q = reinterpret_cast<int8_t *>(s);
    o.q_ld = K;
    o.d = reinterpret_cast<float *>(s + q_bytes);
    o.s32 = reinterpret_cast<int32_t *>(s + q_bytes + d_bytes);
    o.d_ld = ld;
    e = qk::launch_quantize(x, M, K, o, st, false, d.num_sms);
    if (e != cudaSuccess) return err(QMM_ECUDA, "quantize launch failed (cuda error %lld)", e);
    qk::count_launches(1);
    e = qk::launch_gemm_mma(type, W_blocks, N, K, o.q, o.d, o.s32, static_cast<int>(ld), M, y, st);
    if (e != cudaSuccess) return err(QMM_ECUDA, "gemm launch failed (cuda error %lld)", e);
    qk::count_launches(1);
    return qk::record_error(QMM_OK, "");
}
