// gemv_rows_wide_kq.cu -- the row-per-lane decode kernel (gemv_rows.cuh) for
// 3 <= M <= 8 activation rows, Q3_K and Q2_K (MT = 4 or 8 accumulators per
// lane, as gemv_rows_wide.cu does for Q4_K and Q5_K); a translation unit of
// its own so that it compiles in parallel with the others.
#include "gemv_rows.cuh"

namespace qk {
namespace rwk {

cudaError_t launch_rows_wide_kq(const RwParams &R, int MT, int CW, int H, int grid, int smem, cudaStream_t st) {
    if (R.q.type == QMM_Q3_K)
        return MT == 4 ? launch_single<QMM_Q3_K, 4>(R, CW, H, grid, smem, st)
                       : launch_single<QMM_Q3_K, 8>(R, CW, H, grid, smem, st);
    if (R.q.type == QMM_Q2_K)
        return MT == 4 ? launch_single<QMM_Q2_K, 4>(R, CW, H, grid, smem, st)
                       : launch_single<QMM_Q2_K, 8>(R, CW, H, grid, smem, st);
    return cudaErrorNotSupported;
}

}  // namespace rwk
}  // namespace qk
