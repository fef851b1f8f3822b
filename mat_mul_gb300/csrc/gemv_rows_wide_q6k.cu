// gemv_rows_wide_q6k.cu -- the row-per-lane decode kernel (gemv_rows.cuh) for
// 3 <= M <= 8 activation rows with Q6_K weights: single matrices (on request:
// the block-per-lane and tensor-core kernels are faster on large Q6_K
// matrices) and groups that hold a Q6_K matrix (q/k/v with a Q6_K v), MT = 4
// or 8 accumulators per lane; a translation unit of its own so that it
// compiles in parallel with the others.
#include "gemv_rows.cuh"

namespace qk {
namespace rwk {

cudaError_t launch_rows_wide_q6k(const RwParams &R, int MT, int CW, int H, int grid, int smem, cudaStream_t st) {
    if (R.q.type != QMM_Q6_K) return cudaErrorNotSupported;
    return MT == 4 ? launch_single<QMM_Q6_K, 4>(R, CW, H, grid, smem, st)
                   : launch_single<QMM_Q6_K, 8>(R, CW, H, grid, smem, st);
}

cudaError_t launch_rows_wide_group_q6k(const RwGroup &G, int MT, int CW, int H, int grid, int smem, cudaStream_t st) {
    return MT == 4 ? launch_group<4, true>(G, CW, H, grid, smem, st) : launch_group<8, true>(G, CW, H, grid, smem, st);
}

}  // namespace rwk
}  // namespace qk
