// gate_up.cu -- the SiLU-gated product of an MLP's gate and up projections,
// h = silu(g) * u with silu(v) = v / (1 + e^-v), elementwise over the two
// products.  The infr landing page ("why > Per-op device profiling") runs an
// expert's gate and up as one dispatch (expert_gateup); the SiLU between them
// is the activation of the Qwen3 / Llama MLPs the pages' engines serve.
//
// The decode kernels apply it inside their own epilogues (gemv_sb.cu: gate
// and up rows in one CTA; gemv_mma.cu: the up launch reads g); this kernel
// serves the other shapes (prefill, mixed block types) after the two
// products.  Memory-bound: 8 bytes in and 4 out per element.
#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qk {

__global__ void __launch_bounds__(256) silu_mul_kernel(const float *__restrict__ g, const float *__restrict__ u,
                                                       float *__restrict__ h, int64_t n) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        const float gv = g[i];
        h[i] = gv / (1.0f + expf(-gv)) * u[i];
    }
}

cudaError_t launch_silu_mul(const float *g, const float *u, float *h, int64_t n, cudaStream_t st, int num_sms) {
    if (n <= 0) return cudaSuccess;
    int64_t grid = (n + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (grid > cap) grid = cap;
    const cudaError_t e = prefer_max_shared(silu_mul_kernel);
    if (e != cudaSuccess) return e;
    silu_mul_kernel<<<static_cast<unsigned>(grid), 256, 0, st>>>(g, u, h, n);
    return cudaGetLastError();
}

}  // namespace qk
