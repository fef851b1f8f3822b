// gemv_sb_kq.cu -- the block-per-lane decode kernel (gemv_sb.cuh) for the
// other K-quants, Q5_K, Q3_K and Q2_K: their instantiations live in a
// translation unit of their own so that the build compiles them beside
// gemv_sb.cu's.
#include "gemv_sb.cuh"

namespace qk {

cudaError_t launch_sb_kquant(int type, const sbk::SbParams &P, int MT, int grid, int smem, cudaStream_t st) {
    switch (type) {
    case QMM_Q5_K: return sbk::launch_m<QMM_Q5_K>(P, MT, grid, smem, st);
    case QMM_Q3_K: return sbk::launch_m<QMM_Q3_K>(P, MT, grid, smem, st);
    case QMM_Q2_K: return sbk::launch_m<QMM_Q2_K>(P, MT, grid, smem, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qk
