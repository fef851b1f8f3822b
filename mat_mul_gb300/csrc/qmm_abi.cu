// qmm_abi.cu -- the C ABI of libqmm (include/qmm.h): argument validation,
// dispatch between the decode GEMV (M <= 8) and the prefill GEMM, the
// per-(device, stream) activation workspace, status and error reporting.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "../../include/qmm.h"
#include "qmm_device.cuh"

#include "qmm_internal.h"

namespace {

thread_local char g_err[512] = "";
// QMM_PREFILL_KERNEL=mma keeps the prefill on the mma.sync kernel.
const bool g_force_mma_gemm = [] {
    const char *v = getenv("QMM_PREFILL_KERNEL");
    return v && strcmp(v, "mma") == 0;
}();
// QMM_DECODE_KERNEL=rounds selects the round-based decode kernel wherever the
// block-per-lane one would run; =sb keeps 2 <= M <= 8 on the block-per-lane
// kernel instead of the tensor-core one (for comparisons; read once at load).
const bool g_force_round_gemv = [] {
    const char *v = getenv("QMM_DECODE_KERNEL");
    return v && strcmp(v, "rounds") == 0;
}();
const bool g_no_mma_gemv = [] {
    const char *v = getenv("QMM_DECODE_KERNEL");
    return v && (strcmp(v, "sb") == 0 || strcmp(v, "rounds") == 0);
}();
std::atomic<int64_t> g_launches{0};
std::atomic<int> g_decode_path{QMM_DECODE_AUTO};
std::atomic<int> g_prefill_path{QMM_PREFILL_AUTO};
std::atomic<int> g_inject{0};  // pending qmm_inject_stall launches

int fail(int code, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char *what) {
    return fail(QMM_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

struct DeviceInfo {
    int num_sms = 0;
    int max_smem = 0;
    int *status = nullptr;  // device word raised by bounded waits that expired
};

struct Workspace {
    void *ptr = nullptr;
    size_t bytes = 0;
};

std::mutex g_mu;
std::map<int, DeviceInfo> g_dev;
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;
// qmm_t's per-matrix completion counters, per (device, stream): zero between
// calls (each call's last CTA of a matrix resets its counter)
std::map<std::pair<int, cudaStream_t>, Workspace> g_counters;
// qmm_gate_up's intermediate products g (and u), per (device, stream)
std::map<std::pair<int, cudaStream_t>, Workspace> g_gate;

int device_info(int dev, DeviceInfo &out) {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_dev.find(dev);
    if (it != g_dev.end()) {
        out = it->second;
        return QMM_OK;
    }
    DeviceInfo di;
    cudaError_t e = cudaDeviceGetAttribute(&di.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&di.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return cuda_fail(e, "device query");
    e = cudaMalloc(&di.status, 256);
    if (e != cudaSuccess) return fail(QMM_ENOMEM, "status word: %s", cudaGetErrorString(e));
    e = cudaMemset(di.status, 0, 256);
    if (e != cudaSuccess) return cuda_fail(e, "status word init");
    g_dev[dev] = di;
    out = di;
    return QMM_OK;
}

// Workspace of at least `bytes` for (dev, stream).  Growing synchronises the
// stream before the old buffer is released.
int workspace(int dev, cudaStream_t st, size_t bytes, void **ptr) {
    std::lock_guard<std::mutex> lk(g_mu);
    Workspace &w = g_ws[{dev, st}];
    if (w.bytes >= bytes) {
        *ptr = w.ptr;
        return QMM_OK;
    }
    size_t want = bytes + bytes / 2;
    want = (want + (2u << 20) - 1) & ~size_t((2u << 20) - 1);
    if (w.ptr) {
        cudaError_t e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) return cuda_fail(e, "workspace grow (sync)");
        cudaFree(w.ptr);
        w.ptr = nullptr;
        w.bytes = 0;
    }
    cudaError_t e = cudaMalloc(&w.ptr, want);
    if (e != cudaSuccess) {
        w.ptr = nullptr;
        return fail(QMM_ENOMEM, "workspace of %zu bytes: %s", want, cudaGetErrorString(e));
    }
    w.bytes = want;
    *ptr = w.ptr;
    return QMM_OK;
}

// The gate/up intermediate buffer of at least `bytes` for (dev, stream);
// growing synchronises the stream before the old buffer is released.
int gate_buffer(int dev, cudaStream_t st, size_t bytes, float **ptr) {
    std::lock_guard<std::mutex> lk(g_mu);
    Workspace &w = g_gate[{dev, st}];
    if (w.bytes < bytes) {
        if (w.ptr) {
            cudaError_t e = cudaStreamSynchronize(st);
            if (e != cudaSuccess) return cuda_fail(e, "gate buffer grow (sync)");
            cudaFree(w.ptr);
            w.ptr = nullptr;
            w.bytes = 0;
        }
        const size_t want = (bytes + (2u << 20) - 1) & ~size_t((2u << 20) - 1);
        cudaError_t e = cudaMalloc(&w.ptr, want);
        if (e != cudaSuccess) {
            w.ptr = nullptr;
            return fail(QMM_ENOMEM, "gate buffer of %zu bytes: %s", want, cudaGetErrorString(e));
        }
        w.bytes = want;
    }
    *ptr = static_cast<float *>(w.ptr);
    return QMM_OK;
}

// At least n zeroed counters for (dev, stream).  Growing synchronises the
// stream before the old array is released; the new one is zeroed on it.
int counters(int dev, cudaStream_t st, int64_t n, unsigned **ptr) {
    std::lock_guard<std::mutex> lk(g_mu);
    Workspace &w = g_counters[{dev, st}];
    const size_t bytes = static_cast<size_t>(n) * sizeof(unsigned);
    if (w.bytes >= bytes) {
        *ptr = static_cast<unsigned *>(w.ptr);
        return QMM_OK;
    }
    size_t want = 4096;
    while (want < bytes) want *= 2;
    if (w.ptr) {
        cudaError_t e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) return cuda_fail(e, "counters grow (sync)");
        cudaFree(w.ptr);
        w.ptr = nullptr;
        w.bytes = 0;
    }
    cudaError_t e = cudaMalloc(&w.ptr, want);
    if (e != cudaSuccess) {
        w.ptr = nullptr;
        return fail(QMM_ENOMEM, "counters of %zu bytes: %s", want, cudaGetErrorString(e));
    }
    e = cudaMemsetAsync(w.ptr, 0, want, st);
    if (e != cudaSuccess) return cuda_fail(e, "counters init");
    w.bytes = want;
    *ptr = static_cast<unsigned *>(w.ptr);
    return QMM_OK;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// The products (qmm, qmm_group, qmm_gate_up) take every type of the enum;
// qmm_t takes Q8_0 and qmm_noalloc Q8_0, Q4_K, Q6_K (checked there).
int check_type(int type) {
    if (type < QMM_Q8_0 || type > QMM_Q2_K) return fail(QMM_EINVAL_TYPE, "unknown block type %d", type);
    return QMM_OK;
}

// qmm_dequant takes every type of the enum.
int check_dequant_type(int type) {
    if (type < QMM_Q8_0 || type > QMM_Q2_K) return fail(QMM_EINVAL_TYPE, "unknown block type %d", type);
    return QMM_OK;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace

namespace qk {
// Record the calling thread's last-error text for qmm_last_error(); returns code.
int record_error(int code, const char *msg) { return fail(code, "%s", msg); }
// Add n kernel launches to qmm_launch_count().
void count_launches(int64_t n) { g_launches.fetch_add(n); }
int inject_stop_stage() {
    int v = g_inject.load();
    while (v > 0)
        if (g_inject.compare_exchange_weak(v, v - 1)) return 1;
    return NO_STOP;
}
}  // namespace qk

namespace {
// The quantiser for the tensor-core decode: fp16 d*q*2^e_m in fragment
// order, the block and group sums and the row factors into the workspace
// ([M][2K + K/8 bytes] | [K/16][8] fp32 | [8] fp32), launched so that the
// decode kernels after it (programmatic dependent launch) stream weights
// while it runs.
int quantize_for_tensor_cores(int dev, cudaStream_t st, const float *x, int64_t M, int64_t K, const DeviceInfo &di,
                              void **ws) {
    const size_t xh_bytes = static_cast<size_t>(M * (K + K / 16)) * 2;
    const size_t xs_bytes = static_cast<size_t>(K) * 2;  // [K/16][8] fp32
    if (int rc = workspace(dev, st, align_up(xh_bytes + xs_bytes + 8 * sizeof(float), 256), ws)) return rc;
    qk::QuantOut o = {};
    o.xh = *ws;
    o.xh_ld = K + K / 16;
    o.xh_mma = 1;
    o.xs16 = reinterpret_cast<float *>(static_cast<char *>(*ws) + xh_bytes);
    o.xinv = reinterpret_cast<float *>(static_cast<char *>(*ws) + xh_bytes + xs_bytes);
    cudaError_t e = qk::launch_quantize(x, M, K, o, st, true, di.num_sms, true);
    if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
    g_launches.fetch_add(1);
    return QMM_OK;
}

// The decode product of this type and shape runs on the row-per-lane kernel
// (unless the tensor-core one takes it first).
bool decode_on_rows(int type, int64_t M, int64_t N, int64_t K, const DeviceInfo &di) {
    if (M < 1 || M > 8 || g_no_mma_gemv) return false;
    const int path = g_decode_path.load();
    if (path == QMM_DECODE_BLOCK) return false;
    if (path != QMM_DECODE_ROWS && !qk::gemv_rows_preferred(type, static_cast<int>(M), N, K)) return false;
    return qk::gemv_rows_fits(type, static_cast<int>(M), K, di.max_smem);
}

// Large Q8_0 matrices from M = 3 on: the tcgen05 prefill kernel (the
// quantiser, then one 64-token tile per weight tile) instead of the
// block-per-lane decode, whose per-lane activation reads grow with M
// (QMM_DECODE_AUTO only).  Measured (rotating copies): from 2^24 weights at
// M >= 5 (4096 x 4096 at M = 8: 15.6 against 20.5 us) and from 3 * 2^24 at
// M = 3, 4 (4096 -> 14336: 27.8 against 40.4 us; 5120 x 5120: 20.8 against
// 18.8 us, so smaller ones stay).
bool q8_0_decode_on_prefill(int type, int64_t M, int64_t N, int64_t K) {
    const int64_t min_weights = (M >= 5 ? int64_t(1) : int64_t(3)) << 24;
    return type == QMM_Q8_0 && M >= QMM_TENSOR_MIN_M && M <= 8 && N * K >= min_weights &&
           g_decode_path.load() == QMM_DECODE_AUTO && !g_no_mma_gemv && !g_force_mma_gemm &&
           g_prefill_path.load() == QMM_PREFILL_AUTO && qk::gemm_tc_supported(type, N, K, M);
}

// Under QMM_DECODE_ROWS the row-per-lane kernel goes before the tensor-core one.
bool rows_first() { return g_decode_path.load() == QMM_DECODE_ROWS; }

// The decode product of this type and shape runs on the tensor-core kernel.
bool decode_on_tensor_cores(int type, int64_t M, int64_t N, int64_t K, const DeviceInfo &di) {
    if (M < 2 || M > 8 || g_force_round_gemv) return false;
    const int path = g_decode_path.load();
    if (path == QMM_DECODE_BLOCK) return false;
    if ((path == QMM_DECODE_AUTO || path == QMM_DECODE_ROWS) && (M < QMM_TENSOR_MIN_M || g_no_mma_gemv)) return false;
    // Q6_K rows of at most 8 super-blocks at M <= 4: a tensor-core stage is a
    // whole 16-row group, so the group-end sums come every stage; the
    // block-per-lane kernel was faster there (the 2048 x 128256 lm_head at
    // M = 3 / 4: 58.6 / 60.3 against 71.5 us)
    if ((path == QMM_DECODE_AUTO || path == QMM_DECODE_ROWS) && type == QMM_Q6_K && K <= 8 * 256 && M <= 4)
        return false;
    return qk::gemv_mma_fits(type, static_cast<int>(M), N, K, di.max_smem, di.num_sms);
}

// The entries of a qmm_group call take one launch of the row-per-lane kernel:
// each of them would on its own.  (At M = 3, 4 such a launch of Q4_K / Q6_K
// matrices measured faster per call than the quantiser and the tensor-core
// launch, q+k+v 16.9 -> 13.0 us, but slower inside a layer whose other
// products run on the tensor cores: each switch between the two kinds of
// launch cost 3-10 us, the Qwen3-14B layer at M = 4 106 us against 95 us.)
bool group_on_rows(int n, const int *types, const int64_t *Ns, int64_t K, int64_t M, const DeviceInfo &di) {
    for (int i = 0; i < n; ++i) {
        if (Ns[i] == 0) continue;
        if (!decode_on_rows(types[i], M, Ns[i], K, di) ||
            (!rows_first() && decode_on_tensor_cores(types[i], M, Ns[i], K, di)))
            return false;
    }
    return true;
}
}  // namespace

extern "C" {

const char *qmm_strerror(int status) {
    switch (status) {
    case QMM_OK: return "QMM_OK";
    case QMM_EINVAL_TYPE: return "QMM_EINVAL_TYPE";
    case QMM_EINVAL_SHAPE: return "QMM_EINVAL_SHAPE";
    case QMM_EINVAL_PTR: return "QMM_EINVAL_PTR";
    case QMM_ENOMEM: return "QMM_ENOMEM";
    case QMM_ECUDA: return "QMM_ECUDA";
    case QMM_ETIMEOUT: return "QMM_ETIMEOUT";
    default: return "QMM_UNKNOWN";
    }
}

const char *qmm_last_error(void) { return g_err; }

int64_t qmm_launch_count(void) { return g_launches.load(); }

int qmm_set_decode_path(int path) {
    if (path != QMM_DECODE_AUTO && path != QMM_DECODE_BLOCK && path != QMM_DECODE_TENSOR && path != QMM_DECODE_ROWS)
        return fail(QMM_EINVAL_SHAPE, "unknown decode path %d", path);
    return g_decode_path.exchange(path);
}

int qmm_inject_stall(int launches) {
    if (launches < 0) return fail(QMM_EINVAL_SHAPE, "launches=%d must be >= 0", launches);
    return g_inject.exchange(launches);
}

int qmm_set_prefill_path(int path) {
    if (path != QMM_PREFILL_AUTO && path != QMM_PREFILL_INT8)
        return fail(QMM_EINVAL_SHAPE, "unknown prefill path %d", path);
    return g_prefill_path.exchange(path);
}

int qmm_dequant(int type, const void *blocks, int64_t n_elems, float *out_f32) {
    g_err[0] = 0;
    if (int rc = check_dequant_type(type)) return rc;
    const int qk_ = qk::block_weights(type);
    if (n_elems < 0 || n_elems % qk_)
        return fail(QMM_EINVAL_SHAPE, "n_elems=%lld is not a non-negative multiple of %d",
                    static_cast<long long>(n_elems), qk_);
    if (n_elems == 0) return QMM_OK;
    if (!blocks || !out_f32) return fail(QMM_EINVAL_PTR, "null pointer");
    if (!aligned(blocks, 16) || !aligned(out_f32, 16))
        return fail(QMM_EINVAL_PTR, "blocks and out_f32 must be 16-byte aligned");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    DeviceInfo di;
    if (int rc = device_info(dev, di)) return rc;
    e = qk::launch_dequant(type, blocks, n_elems, out_f32, 0, di.num_sms);
    if (e != cudaSuccess) return cuda_fail(e, "dequant launch");
    g_launches.fetch_add(1);
    return QMM_OK;
}

int qmm_quantize_act(const float *x, int64_t M, int64_t K, int8_t *q, float *d, int32_t *s,
                     void *stream) {
    g_err[0] = 0;
    if (M < 0 || K < 0 || K % 32)
        return fail(QMM_EINVAL_SHAPE, "M=%lld K=%lld: K must be a non-negative multiple of 32",
                    static_cast<long long>(M), static_cast<long long>(K));
    if (M == 0 || K == 0) return QMM_OK;
    if (!x || !q || !d || !s) return fail(QMM_EINVAL_PTR, "null pointer");
    if (!aligned(x, 4) || !aligned(d, 4) || !aligned(s, 4))
        return fail(QMM_EINVAL_PTR, "x, d and s must be 4-byte aligned");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    DeviceInfo di;
    if (int rc = device_info(dev, di)) return rc;
    qk::QuantOut o = {};
    o.q = q;
    o.q_ld = K;
    o.d = d;
    o.s32 = s;
    o.d_ld = K / 32;
    e = qk::launch_quantize(x, M, K, o, static_cast<cudaStream_t>(stream), false, di.num_sms);
    if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
    g_launches.fetch_add(1);
    return QMM_OK;
}

int qmm(int type, const void *W_blocks, int64_t N, int64_t K, const float *x, int64_t M, float *y,
        void *stream) {
    g_err[0] = 0;
    if (int rc = check_type(type)) return rc;
    const int qk_ = qk::block_weights(type);
    if (N < 0 || M < 0 || K < 0 || K % qk_)
        return fail(QMM_EINVAL_SHAPE, "N=%lld K=%lld M=%lld: sizes must be >= 0 and K a multiple of %d",
                    static_cast<long long>(N), static_cast<long long>(K), static_cast<long long>(M), qk_);
    if (K > (int64_t(1) << 24))
        return fail(QMM_EINVAL_SHAPE, "K=%lld exceeds 2^24", static_cast<long long>(K));
    if (M == 0 || N == 0) return QMM_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (!y) return fail(QMM_EINVAL_PTR, "null y");
    if (!aligned(y, 4)) return fail(QMM_EINVAL_PTR, "y must be 4-byte aligned");
    if (K == 0) {
        cudaError_t e = cudaMemsetAsync(y, 0, static_cast<size_t>(M * N) * sizeof(float), st);
        if (e != cudaSuccess) return cuda_fail(e, "zero fill");
        return QMM_OK;
    }
    if (!W_blocks || !x) return fail(QMM_EINVAL_PTR, "null pointer");
    if (!aligned(W_blocks, 16)) return fail(QMM_EINVAL_PTR, "W_blocks must be 16-byte aligned");
    if (!aligned(x, 4)) return fail(QMM_EINVAL_PTR, "x must be 4-byte aligned");

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    DeviceInfo di;
    if (int rc = device_info(dev, di)) return rc;

    // Four paths, chosen by M and by what fits in shared memory:
    //   mma  : decode, Q4_K / Q6_K with QMM_TENSOR_MIN_M <= M <= 8
    //          (qmm_set_decode_path widens or closes it): the quantiser (fp16
    //          d*q and sums into the workspace), then sixteen weight rows per
    //          f16 mma.sync
    //   sb   : decode, one weight block per lane, quantises x itself (one
    //          launch, no workspace); M <= 8 when the activations fit
    //   gemv : decode, 32 units per round, after the quantiser kernel
    //   gemm : prefill after the quantiser: on tcgen05 (fp16 operands, fp32
    //          accumulators) when K is a multiple of 256, else on the int8
    //          mma.sync kernel; also a decode (M <= 8) that none of the
    //          decode kernels above can hold (their activations do not fit),
    //          which the round-based decode would take many times longer for
    if (!(rows_first() && decode_on_rows(type, M, N, K, di)) && decode_on_tensor_cores(type, M, N, K, di)) {
        void *ws = nullptr;
        if (int rc = quantize_for_tensor_cores(dev, st, x, M, K, di, &ws)) return rc;
        e = qk::launch_gemv_mma(type, W_blocks, N, K, ws, static_cast<int>(M), y, st, di.num_sms, di.max_smem,
                                di.status);
        if (e != cudaSuccess) return cuda_fail(e, "tensor-core gemv launch");
        g_launches.fetch_add(1);
        return QMM_OK;
    }
    if (decode_on_rows(type, M, N, K, di)) {
        e = qk::launch_gemv_rows(type, W_blocks, N, K, x, static_cast<int>(M), y, st, di.num_sms, di.max_smem,
                                 di.status);
        if (e != cudaSuccess) return cuda_fail(e, "gemv launch");
        g_launches.fetch_add(1);
        return QMM_OK;
    }
    if (M <= 8 && !g_force_round_gemv && qk::gemv_sb_fits(type, static_cast<int>(M), K, di.max_smem) &&
        !q8_0_decode_on_prefill(type, M, N, K)) {
        e = qk::launch_gemv_sb(type, W_blocks, N, K, x, static_cast<int>(M), y, st, di.num_sms, di.max_smem,
                               di.status);
        if (e != cudaSuccess) return cuda_fail(e, "gemv launch");
        g_launches.fetch_add(1);
        return QMM_OK;
    }
    // Prefill on the tcgen05 kernel: fp16 activations d*q [M][K].  (At M <= 8
    // only when none of the decode kernels fits: e.g. Q5_K / Q3_K / Q2_K at
    // M = 8 and K = 17408, 14x faster than the round-based decode.)
    if ((M > 8 || !g_force_round_gemv) && !g_force_mma_gemm && g_prefill_path.load() == QMM_PREFILL_AUTO &&
        qk::gemm_tc_supported(type, N, K, M)) {
        const size_t xh_bytes = align_up(static_cast<size_t>(M * K) * 2, 256);
        const size_t xinv_bytes = align_up(static_cast<size_t>(M) * 4, 256);
        void *ws = nullptr;
        if (int rc = workspace(dev, st, xh_bytes + xinv_bytes, &ws)) return rc;
        qk::QuantOut o = {};
        o.xh = ws;
        o.xh_ld = K;
        o.xinv = reinterpret_cast<float *>(static_cast<char *>(ws) + xh_bytes);
        e = qk::launch_quantize(x, M, K, o, st, false, di.num_sms);
        if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
        g_launches.fetch_add(1);
        e = qk::launch_gemm_tc(type, W_blocks, N, K, ws, o.xinv, M, y, st, di.num_sms, di.status);
        if (e != cudaSuccess) return cuda_fail(e, "gemm launch");
        g_launches.fetch_add(1);
        return QMM_OK;
    }
    // Workspace (per device and stream): q int8 [M][K] | d fp32 [M][d_ld] |
    // s16 int32 [M][s16_ld] (gemv) or s32 int32 [M][d_ld] (gemm).
    const int64_t d_ld = static_cast<int64_t>(align_up(static_cast<size_t>(K / 32), 4));
    const int64_t s16_ld = static_cast<int64_t>(align_up(static_cast<size_t>(K / 16), 4));
    const bool gemv = M <= 8 && qk::gemv_fits(type, static_cast<int>(M), K, static_cast<int>(d_ld),
                                               static_cast<int>(s16_ld), di.max_smem);
    // the round-based decode and the Q2_K prefill read 16-element sums, the
    // other prefills 32-element ones
    const bool halves = gemv || type == QMM_Q2_K;
    const size_t q_bytes = align_up(static_cast<size_t>(M * K), 256);
    const size_t d_bytes = align_up(static_cast<size_t>(M * d_ld) * 4, 256);
    const size_t a_bytes = align_up(static_cast<size_t>(M * (halves ? s16_ld : d_ld)) * 4, 256);
    void *ws = nullptr;
    if (int rc = workspace(dev, st, q_bytes + d_bytes + a_bytes, &ws)) return rc;
    char *wsb = static_cast<char *>(ws);
    qk::QuantOut o = {};
    o.q = reinterpret_cast<int8_t *>(wsb);
    o.q_ld = K;
    o.d = reinterpret_cast<float *>(wsb + q_bytes);
    o.d_ld = d_ld;
    o.s16_ld = s16_ld;
    if (halves) o.s16 = reinterpret_cast<int32_t *>(wsb + q_bytes + d_bytes);
    else o.s32 = reinterpret_cast<int32_t *>(wsb + q_bytes + d_bytes);
    e = qk::launch_quantize(x, M, K, o, st, gemv, di.num_sms);
    if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
    g_launches.fetch_add(1);
    if (gemv) {
        e = qk::launch_gemv(type, W_blocks, N, K, o.q, o.d, o.s16, static_cast<int>(d_ld),
                            static_cast<int>(s16_ld), static_cast<int>(M), y, st, true, di.num_sms,
                            di.max_smem, di.status);
        if (e != cudaSuccess) return cuda_fail(e, "gemv launch");
    } else {
        e = qk::launch_gemm_mma(type, W_blocks, N, K, o.q, o.d, o.s32, static_cast<int>(d_ld), M, y, st, o.s16,
                                static_cast<int>(s16_ld));
        if (e != cudaSuccess) return cuda_fail(e, "gemm launch");
    }
    g_launches.fetch_add(1);
    return QMM_OK;
}

int qmm_t(int type, const void *W_blocks, int64_t H, int64_t N, int64_t K, const float *x, int64_t M, float *y,
          void *stream) {
    g_err[0] = 0;
    if (int rc = check_type(type)) return rc;
    if (type != QMM_Q8_0) return fail(QMM_EINVAL_TYPE, "qmm_t takes Q8_0 blocks (the KV cache format), not type %d", type);
    if (H < 0 || N < 0 || K < 0 || M < 0 || K % 32 || K > 256)
        return fail(QMM_EINVAL_SHAPE, "H=%lld N=%lld K=%lld M=%lld: sizes must be >= 0 and K a multiple of 32 up to 256",
                    static_cast<long long>(H), static_cast<long long>(N), static_cast<long long>(K),
                    static_cast<long long>(M));
    if (H > 65535 || N > (int64_t(1) << 31) || M > (int64_t(1) << 24))
        return fail(QMM_EINVAL_SHAPE, "H=%lld N=%lld M=%lld: H <= 65535, N <= 2^31, M <= 2^24",
                    static_cast<long long>(H), static_cast<long long>(N), static_cast<long long>(M));
    if (H == 0 || M == 0 || K == 0) return QMM_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (!y) return fail(QMM_EINVAL_PTR, "null y");
    if (!aligned(y, 4)) return fail(QMM_EINVAL_PTR, "y must be 4-byte aligned");
    if (N == 0) {
        cudaError_t e = cudaMemsetAsync(y, 0, static_cast<size_t>(H * M * K) * sizeof(float), st);
        if (e != cudaSuccess) return cuda_fail(e, "zero fill");
        return QMM_OK;
    }
    if (!W_blocks || !x) return fail(QMM_EINVAL_PTR, "null pointer");
    if (!aligned(W_blocks, 16)) return fail(QMM_EINVAL_PTR, "W_blocks must be 16-byte aligned");
    if (!aligned(x, 4)) return fail(QMM_EINVAL_PTR, "x must be 4-byte aligned");

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    DeviceInfo di;
    if (int rc = device_info(dev, di)) return rc;
    void *ws = nullptr;
    if (int rc = workspace(dev, st, qk::qmm_t_part_bytes(H, N, K, di.num_sms), &ws)) return rc;
    unsigned *cnt = nullptr;
    if (int rc = counters(dev, st, H, &cnt)) return rc;
    e = qk::launch_qmm_t(W_blocks, H, N, K, x, M, y, static_cast<float *>(ws), cnt, st, di.num_sms, di.status);
    if (e != cudaSuccess) return cuda_fail(e, "qmm_t launch");
    g_launches.fetch_add((M + 15) / 16);
    return QMM_OK;
}

int qmm_group(int n, const int *types, const void *const *Ws, const int64_t *Ns, int64_t K, const float *x,
              int64_t M, float *const *ys, void *stream) {
    g_err[0] = 0;
    if (n < 1 || n > QMM_GROUP_MAX) return fail(QMM_EINVAL_SHAPE, "n=%d: a group has 1..%d matrices", n, QMM_GROUP_MAX);
    if (!types || !Ws || !Ns || !ys) return fail(QMM_EINVAL_PTR, "null array");
    if (M < 0 || K < 0 || K > (int64_t(1) << 24))
        return fail(QMM_EINVAL_SHAPE, "K=%lld M=%lld", static_cast<long long>(K), static_cast<long long>(M));
    // types and shapes of every entry first, then pointers
    for (int i = 0; i < n; ++i) {
        if (int rc = check_type(types[i])) return rc;
        if (Ns[i] < 0 || K % qk::block_weights(types[i]))
            return fail(QMM_EINVAL_SHAPE, "entry %d: N=%lld K=%lld (K a multiple of %d)", i,
                        static_cast<long long>(Ns[i]), static_cast<long long>(K), qk::block_weights(types[i]));
    }
    bool any = false;
    for (int i = 0; i < n; ++i) {
        if (Ns[i] == 0 || M == 0) continue;
        any = true;
        if (!ys[i] || !aligned(ys[i], 4)) return fail(QMM_EINVAL_PTR, "entry %d: y null or not 4-byte aligned", i);
        if (K > 0 && (!Ws[i] || !aligned(Ws[i], 16)))
            return fail(QMM_EINVAL_PTR, "entry %d: W null or not 16-byte aligned", i);
    }
    if (!any) return QMM_OK;
    if (K > 0 && (!x || !aligned(x, 4))) return fail(QMM_EINVAL_PTR, "x null or not 4-byte aligned");

    if (K > 0 && M <= 8 && !g_force_round_gemv) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
        DeviceInfo di;
        if (int rc = device_info(dev, di)) return rc;
        // one launch when the entries take the row-per-lane kernel
        if (group_on_rows(n, types, Ns, K, M, di)) {
            e = qk::launch_gemv_rows_group(n, types, Ws, Ns, K, x, static_cast<int>(M), ys,
                                           static_cast<cudaStream_t>(stream), di.num_sms, di.max_smem, di.status);
            if (e == cudaSuccess) {
                g_launches.fetch_add(1);
                return QMM_OK;
            }
            if (e != cudaErrorNotSupported) return cuda_fail(e, "group gemv launch");
        }
        // else one launch when every entry takes the block-per-lane kernel (an
        // entry for the tensor-core one makes them separate calls)
        bool fits = true;
        for (int i = 0; i < n; ++i)
            fits = fits && (Ns[i] == 0 || (qk::gemv_sb_fits(types[i], static_cast<int>(M), K, di.max_smem) &&
                                           !decode_on_tensor_cores(types[i], M, Ns[i], K, di)));
        if (fits) {
            e = qk::launch_gemv_sb_group(n, types, Ws, Ns, K, x, static_cast<int>(M), ys,
                                         static_cast<cudaStream_t>(stream), di.num_sms, di.max_smem, di.status);
            if (e == cudaSuccess) {
                g_launches.fetch_add(1);
                return QMM_OK;
            }
            // (the one-launch group takes Q8_0, Q4_K and Q6_K; other types run entry by entry)
            if (e != cudaErrorNotSupported) return cuda_fail(e, "group gemv launch");
        }
        // every entry on the tensor-core kernel: x quantised once, then one
        // decode launch for all the matrices (CTAs split by their bytes), or
        // one per matrix if that does not fit
        bool tensor = true;
        for (int i = 0; i < n; ++i) tensor = tensor && (Ns[i] == 0 || decode_on_tensor_cores(types[i], M, Ns[i], K, di));
        if (tensor) {
            cudaStream_t st = static_cast<cudaStream_t>(stream);
            void *ws = nullptr;
            if (int rc = quantize_for_tensor_cores(dev, st, x, M, K, di, &ws)) return rc;
            e = qk::launch_gemv_mma_group(n, types, Ws, Ns, K, ws, static_cast<int>(M), ys, st, di.num_sms,
                                          di.max_smem, di.status);
            if (e == cudaSuccess) {
                g_launches.fetch_add(1);
                return QMM_OK;
            }
            if (e != cudaErrorNotSupported) return cuda_fail(e, "tensor-core group gemv launch");
            for (int i = 0; i < n; ++i) {
                if (Ns[i] == 0) continue;
                e = qk::launch_gemv_mma(types[i], Ws[i], Ns[i], K, ws, static_cast<int>(M), ys[i], st, di.num_sms,
                                        di.max_smem, di.status);
                if (e != cudaSuccess) return cuda_fail(e, "tensor-core gemv launch");
                g_launches.fetch_add(1);
            }
            return QMM_OK;
        }
    }
    for (int i = 0; i < n; ++i) {
        if (Ns[i] == 0) continue;
        if (int rc = qmm(types[i], Ws[i], Ns[i], K, x, M, ys[i], stream)) return rc;
    }
    return QMM_OK;
}

int qmm_gate_up(int type_gate, const void *W_gate, int type_up, const void *W_up, int64_t N, int64_t K,
                const float *x, int64_t M, float *h, void *stream) {
    g_err[0] = 0;
    if (int rc = check_type(type_gate)) return rc;
    if (int rc = check_type(type_up)) return rc;
    if (N < 0 || M < 0 || K < 0 || K % qk::block_weights(type_gate) || K % qk::block_weights(type_up))
        return fail(QMM_EINVAL_SHAPE, "N=%lld K=%lld M=%lld: sizes must be >= 0 and K a multiple of both block sizes",
                    static_cast<long long>(N), static_cast<long long>(K), static_cast<long long>(M));
    if (K > (int64_t(1) << 24)) return fail(QMM_EINVAL_SHAPE, "K=%lld exceeds 2^24", static_cast<long long>(K));
    if (M == 0 || N == 0) return QMM_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (!h || !aligned(h, 4)) return fail(QMM_EINVAL_PTR, "h null or not 4-byte aligned");
    if (K == 0) {  // g = u = 0, so h = silu(0) * 0 = 0
        cudaError_t e = cudaMemsetAsync(h, 0, static_cast<size_t>(M * N) * sizeof(float), st);
        if (e != cudaSuccess) return cuda_fail(e, "zero fill");
        return QMM_OK;
    }
    if (!W_gate || !W_up || !x) return fail(QMM_EINVAL_PTR, "null pointer");
    if (!aligned(W_gate, 16) || !aligned(W_up, 16)) return fail(QMM_EINVAL_PTR, "W_gate and W_up must be 16-byte aligned");
    if (!aligned(x, 4)) return fail(QMM_EINVAL_PTR, "x must be 4-byte aligned");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    DeviceInfo di;
    if (int rc = device_info(dev, di)) return rc;

    // one launch: both matrices of one type on the block-per-lane kernel
    if (type_gate == type_up && M <= 2 && !g_force_round_gemv && !decode_on_tensor_cores(type_gate, M, N, K, di) &&
        qk::gemv_sb_fits(type_gate, static_cast<int>(M), K, di.max_smem)) {
        e = qk::launch_gemv_sb_gateup(type_gate, W_gate, W_up, N, K, x, static_cast<int>(M), h, st, di.num_sms,
                                      di.max_smem, di.status);
        if (e == cudaSuccess) {
            g_launches.fetch_add(1);
            return QMM_OK;
        }
        if (e != cudaErrorNotSupported) return cuda_fail(e, "gate+up launch");
    }
    float *gbuf = nullptr;
    // tensor-core decode: x quantised once, g into the buffer, then the up
    // launch, which reads g and writes h (three launches)
    if (decode_on_tensor_cores(type_gate, M, N, K, di) && decode_on_tensor_cores(type_up, M, N, K, di)) {
        if (int rc = gate_buffer(dev, st, static_cast<size_t>(M * N) * sizeof(float), &gbuf)) return rc;
        void *ws = nullptr;
        if (int rc = quantize_for_tensor_cores(dev, st, x, M, K, di, &ws)) return rc;
        e = qk::launch_gemv_mma(type_gate, W_gate, N, K, ws, static_cast<int>(M), gbuf, st, di.num_sms, di.max_smem,
                                di.status);
        if (e != cudaSuccess) return cuda_fail(e, "tensor-core gemv launch (gate)");
        g_launches.fetch_add(1);
        e = qk::launch_gemv_mma(type_up, W_up, N, K, ws, static_cast<int>(M), h, st, di.num_sms, di.max_smem,
                                di.status, gbuf);
        if (e != cudaSuccess) return cuda_fail(e, "tensor-core gemv launch (up)");
        g_launches.fetch_add(1);
        return QMM_OK;
    }
    // otherwise the two products as qmm(), then h = silu(g) * u
    if (int rc = gate_buffer(dev, st, static_cast<size_t>(2 * M * N) * sizeof(float), &gbuf)) return rc;
    float *ubuf = gbuf + M * N;
    if (int rc = qmm(type_gate, W_gate, N, K, x, M, gbuf, stream)) return rc;
    if (int rc = qmm(type_up, W_up, N, K, x, M, ubuf, stream)) return rc;
    e = qk::launch_silu_mul(gbuf, ubuf, h, M * N, st, di.num_sms);
    if (e != cudaSuccess) return cuda_fail(e, "silu-mul launch");
    g_launches.fetch_add(1);
    return QMM_OK;
}

int qmm_device_status(void *stream) {
    g_err[0] = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    DeviceInfo di;
    if (int rc = device_info(dev, di)) return rc;
    e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    int word = 0;
    e = cudaMemcpy(&word, di.status, sizeof word, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "status read");
    if (word) {
        e = cudaMemset(di.status, 0, sizeof word);
        if (e != cudaSuccess) return cuda_fail(e, "status clear");
        return fail(QMM_ETIMEOUT, "a bounded device wait expired (status word 0x%x)", word);
    }
    return QMM_OK;
}

int qmm_release(void) {
    g_err[0] = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "device synchronize");
    std::lock_guard<std::mutex> lk(g_mu);
    for (auto *m : {&g_ws, &g_counters, &g_gate}) {
        for (auto it = m->begin(); it != m->end();) {
            if (it->first.first == dev) {
                cudaFree(it->second.ptr);
                it = m->erase(it);
            } else {
                ++it;
            }
        }
    }
    return QMM_OK;
}

}  // extern "C"
