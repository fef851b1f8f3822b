// gemv_rows_wide.cu -- the row-per-lane decode kernel (gemv_rows.cuh) for
// 3 <= M <= 8 activation rows, Q4_K and Q5_K (Q3_K and Q2_K in
// gemv_rows_wide_kq.cu, Q6_K in gemv_rows_wide_q6k.cu): the same stages and lanes, MT = 4 or 8 accumulators
// per lane (rows M .. MT-1 of the activations are computed on and never
// written).  Translation units of their own so that they compile in parallel
// with the M <= 2 instantiations.
#include "gemv_rows.cuh"

namespace qk {
namespace rwk {

cudaError_t launch_rows_wide(const RwParams &R, int MT, int CW, int H, int grid, int smem, cudaStream_t st) {
    switch (R.q.type) {
    case QMM_Q4_K:
        return MT == 4 ? launch_single<QMM_Q4_K, 4>(R, CW, H, grid, smem, st)
                       : launch_single<QMM_Q4_K, 8>(R, CW, H, grid, smem, st);
    case QMM_Q5_K:
        return MT == 4 ? launch_single<QMM_Q5_K, 4>(R, CW, H, grid, smem, st)
                       : launch_single<QMM_Q5_K, 8>(R, CW, H, grid, smem, st);
    case QMM_Q3_K:
    case QMM_Q2_K: return launch_rows_wide_kq(R, MT, CW, H, grid, smem, st);
    case QMM_Q6_K: return launch_rows_wide_q6k(R, MT, CW, H, grid, smem, st);
    default: return cudaErrorNotSupported;
    }
}

cudaError_t launch_rows_wide_group(const RwGroup &G, int MT, int CW, int H, int grid, int smem, cudaStream_t st) {
    bool q6k = false;
    for (int i = 0; i < G.n; ++i) {
        if (G.p[i].q.type != QMM_Q4_K && G.p[i].q.type != QMM_Q6_K) return cudaErrorNotSupported;
        q6k = q6k || G.p[i].q.type == QMM_Q6_K;
    }
    if (q6k) return launch_rows_wide_group_q6k(G, MT, CW, H, grid, smem, st);
    return MT == 4 ? launch_group<4, false>(G, CW, H, grid, smem, st)
                   : launch_group<8, false>(G, CW, H, grid, smem, st);
}

}  // namespace rwk
}  // namespace qk
