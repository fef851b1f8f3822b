// qmm_device.cuh -- device-side building blocks of libqmm for sm_103a:
// block-format constants, inline-PTX wrappers for mbarriers, bulk async
// copies and programmatic dependent launch, bounded waits, and small
// shared-memory load helpers.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/qmm.h"

namespace qk {

// ---------------------------------------------------------------------------
// Launch attributes (host).  Every kernel of the library asks for the
// largest shared-memory carveout, whatever it uses: an SM changes its
// carveout only when it is idle, so consecutive launches that asked for
// different ones could not overlap on it (programmatic dependent launch).
// ---------------------------------------------------------------------------
template <class F>
inline cudaError_t prefer_max_shared(F kern) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                static_cast<int>(cudaSharedmemCarveoutMaxShared));
}

// The dynamic shared memory a launch of kern needs, and the carveout.
template <class F>
inline cudaError_t set_smem_attrs(F kern, int smem) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    return e != cudaSuccess ? e : prefer_max_shared(kern);
}

// ---------------------------------------------------------------------------
// Block formats (GGUF): bytes per block and weights per block.
// ---------------------------------------------------------------------------
template <int T> struct Fmt;
template <> struct Fmt<QMM_Q8_0> { static constexpr int BB = 34, QK = 32; };
template <> struct Fmt<QMM_Q4_K> { static constexpr int BB = 144, QK = 256; };
template <> struct Fmt<QMM_Q6_K> { static constexpr int BB = 210, QK = 256; };
template <> struct Fmt<QMM_Q5_K> { static constexpr int BB = 176, QK = 256; };
template <> struct Fmt<QMM_Q3_K> { static constexpr int BB = 110, QK = 256; };
template <> struct Fmt<QMM_Q2_K> { static constexpr int BB = 84, QK = 256; };

inline int block_bytes(int t) {
    switch (t) {
    case QMM_Q8_0: return 34;
    case QMM_Q4_K: return 144;
    case QMM_Q6_K: return 210;
    case QMM_Q5_K: return 176;
    case QMM_Q3_K: return 110;
    default: return 84;  // QMM_Q2_K
    }
}
inline int block_weights(int t) { return t == QMM_Q8_0 ? 32 : 256; }

// Status bits a kernel may raise in the per-device status word.
enum : int { STATUS_TIMEOUT = 1 };

// Limit of every bounded wait, in SM clock cycles (2^31: about one second at
// the 2 GHz class clocks of this part, longer at lower clocks).  The cycle
// counter is read instead of %globaltimer because it is a register read,
// cheap enough to sit in the polling loops of the pipelines.
constexpr long long WAIT_LIMIT_CYCLES = 1ll << 31;

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// The same test, letting the thread sleep until the phase completes, for
// at most SUSPEND_NS nanoseconds per call (a waiting warp then takes no
// issue slots from the working ones).
constexpr uint32_t SUSPEND_NS = 10000;
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "n"(SUSPEND_NS)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete, giving up after
// WAIT_LIMIT_CYCLES; on expiry the status word `status` (device memory owned
// by the library) records a timeout and the function returns false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int *status) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait_sleep(bar, parity)) return true;
        if (clock64() - t0 > WAIT_LIMIT_CYCLES) {
            atomicOr(status, STATUS_TIMEOUT);
            return false;
        }
    }
}

// One-dimensional bulk async copy global -> shared, completing on `bar`.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Warm L2 with [src, src + bytes) (16-byte aligned address and size).  L2 is
// the point of coherence, so this is safe even while another grid may still
// write the range.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Programmatic dependent launch: wait for the preceding grid's results /
// allow the next grid to start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void named_barrier(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also returns the OR of `pred` over all participants, so
// every participant takes the same decision after it.
__device__ __forceinline__ bool named_barrier_or(int id, int nthreads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "barrier.cta.red.or.pred po, %2, %3, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// Shared-memory loads by 32-bit shared address.
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t a) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a));
    return v;
}
__device__ __forceinline__ float ldsf(uint32_t a) { return __uint_as_float(lds32(a)); }

// Read n consecutive 32-bit words starting at a 2-byte-aligned shared
// address: aligned words are loaded and shifted into place.
template <int NWORDS>
__device__ __forceinline__ void lds_words_u16aligned(uint32_t a, uint32_t (&w)[NWORDS]) {
    const uint32_t base = a & ~3u;
    const uint32_t sh = (a & 3u) * 8u;
    uint32_t prev = lds32(base);
#pragma unroll
    for (int i = 0; i < NWORDS; ++i) {
        uint32_t next = lds32(base + 4u * (i + 1));
        w[i] = __funnelshift_r(prev, next, sh);
        prev = next;
    }
}

// 2^e as fp32 for -126 <= e <= 127 (exact).
__device__ __forceinline__ float pow2f(int e) { return __uint_as_float(static_cast<uint32_t>(127 + e) << 23); }

// floor(log2 |v|) of a finite non-zero fp32 given by its bits (subnormals
// count as -127: below every normal value).
__device__ __forceinline__ int exponent_of(uint32_t bits) {
    const int be = static_cast<int>((bits >> 23) & 0xFF);
    return be == 0 ? -127 : be - 127;
}

__device__ __forceinline__ float half_bits_to_float(uint32_t bits) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits & 0xffffu)));
}

}  // namespace qk
