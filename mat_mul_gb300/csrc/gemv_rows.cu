// gemv_rows.cu -- the row-per-lane decode kernel (gemv_rows.cuh has the
// design) for M <= 2 (Q4_K, Q5_K, Q6_K, Q3_K, Q2_K), and the entry points of
// every M (gemv_rows_wide.cu and gemv_rows_wide_kq.cu: 3 <= M <= 8).
#include "gemv_rows.cuh"

namespace qk {

using namespace rwk;

bool gemv_rows_fits(int type, int M, int64_t K, int max_smem) {
    // Q4_K, Q5_K, Q6_K, Q3_K and Q2_K for M <= 8
    if ((type != QMM_Q4_K && type != QMM_Q5_K && type != QMM_Q6_K && type != QMM_Q3_K && type != QMM_Q2_K) ||
        M < 1 || M > 8 ||
        K < 256 || K % 256 != 0 || K > (1 << 22))
        return false;
    const Shape sh = choose_shape(K / 256, block_bytes(type));
    RwParams R = {};
    int smem = 0;
    return plan_rows(type, M, K, max_smem, sh.CW, sh.H, R, smem);
}

bool gemv_rows_preferred(int type, int M, int64_t N, int64_t K) {
    // Q6_K rows are 2-byte aligned and read as 32-bit words: at any 16-byte
    // row pitch, 32 lanes on GR rows meet GR/8-way bank conflicts, which the
    // block-per-lane kernel (lanes on consecutive blocks) does not have
    if (type != QMM_Q4_K && type != QMM_Q5_K && type != QMM_Q3_K && type != QMM_Q2_K) return false;
    // Q4_K from M = 3 on runs on the tensor cores
    if (type == QMM_Q4_K && M > 2) return false;
    // from M = 2 on the block-per-lane kernel's per-lane activation reads
    // multiply; the row-per-lane kernel was as fast or faster on every Q5_K,
    // Q3_K and Q2_K shape measured (5120 -> 17408, 17408 -> 5120, 2048 ->
    // 8192; M = 2, 4, 8)
    if (M >= 2 && type != QMM_Q4_K) return true;
    // Q3_K and Q2_K at M = 1: faster on rows at K = 2048 and 5120, slower at
    // K = 17408 (measured)
    if (type == QMM_Q3_K || type == QMM_Q2_K) return K <= 8192;
    // below full copy efficiency the block-per-lane kernel's long contiguous
    // copies win on large matrices; small ones gain from the shorter setup
    // (Q5_K at 17408 -> 5120, score 0.85, measured faster on rows)
    const Shape sh = choose_shape(K / 256, block_bytes(type));
    const double need = type == QMM_Q5_K ? 0.8 : 0.9;
    return sh.score >= need || N * (K / 256) * block_bytes(type) <= (int64_t(16) << 20);
}

cudaError_t launch_gemv_rows(int type, const void *W, int64_t N, int64_t K, const float *x, int M, float *y,
                             cudaStream_t st, int num_sms, int max_smem, int *status) {
    const Shape sh = choose_shape(K / 256, block_bytes(type));
    RwParams R = {};
    int smem = 0;
    if (!gemv_rows_fits(type, M, K, max_smem) || !plan_rows(type, M, K, max_smem, sh.CW, sh.H, R, smem))
        return cudaErrorNotSupported;
    // one CTA per SM (fewer when there are fewer rows); a CTA's rows stay
    // below 2^31 bytes of weights in every offset the kernel forms in int
    const int64_t RB = (K / 256) * block_bytes(type);
    int64_t grid = num_sms;
    if (grid < (N * RB + (int64_t(1) << 30) - 1) >> 30) grid = (N * RB + (int64_t(1) << 30) - 1) >> 30;
    if (N < grid) grid = N;
    if (grid < 1 || grid > 0x7fffffff) return cudaErrorInvalidValue;
    fill_rows(R, type, W, N, K, x, M, y, status, static_cast<int>(grid));
    R.q.stop_stage = inject_stop_stage();
    const int g = static_cast<int>(grid);
    if (M > 2) return launch_rows_wide(R, M <= 4 ? 4 : 8, sh.CW, sh.H, g, smem, st);
    if (type == QMM_Q4_K)
        return M <= 1 ? launch_single<QMM_Q4_K, 1>(R, sh.CW, sh.H, g, smem, st)
                      : launch_single<QMM_Q4_K, 2>(R, sh.CW, sh.H, g, smem, st);
    if (type == QMM_Q5_K)
        return M <= 1 ? launch_single<QMM_Q5_K, 1>(R, sh.CW, sh.H, g, smem, st)
                      : launch_single<QMM_Q5_K, 2>(R, sh.CW, sh.H, g, smem, st);
    if (type == QMM_Q3_K)
        return M <= 1 ? launch_single<QMM_Q3_K, 1>(R, sh.CW, sh.H, g, smem, st)
                      : launch_single<QMM_Q3_K, 2>(R, sh.CW, sh.H, g, smem, st);
    if (type == QMM_Q2_K)
        return M <= 1 ? launch_single<QMM_Q2_K, 1>(R, sh.CW, sh.H, g, smem, st)
                      : launch_single<QMM_Q2_K, 2>(R, sh.CW, sh.H, g, smem, st);
    return M <= 1 ? launch_single<QMM_Q6_K, 1>(R, sh.CW, sh.H, g, smem, st)
                  : launch_single<QMM_Q6_K, 2>(R, sh.CW, sh.H, g, smem, st);
}

cudaError_t launch_gemv_rows_group(int n, const int *types, const void *const *Ws, const int64_t *Ns, int64_t K,
                                   const float *x, int M, float *const *ys, cudaStream_t st, int num_sms,
                                   int max_smem, int *status) {
    if (n < 1 || n > QMM_GROUP_MAX) return cudaErrorInvalidValue;
    // one shape for the launch: that of the entry with the most bytes
    int64_t most = -1;
    Shape sh = {};
    for (int i = 0; i < n; ++i) {
        if (Ns[i] <= 0) continue;
        // the group launch takes Q4_K and Q6_K
        if ((types[i] != QMM_Q4_K && types[i] != QMM_Q6_K) || !gemv_rows_fits(types[i], M, K, max_smem))
            return cudaErrorNotSupported;
        const int64_t b = Ns[i] * (K / 256) * block_bytes(types[i]);
        if (b > most) most = b, sh = choose_shape(K / 256, block_bytes(types[i]));
    }
    RwGroup G = {};
    int idx[QMM_GROUP_MAX], smem = 0, m = 0;
    int64_t bytes[QMM_GROUP_MAX], rows[QMM_GROUP_MAX], need[QMM_GROUP_MAX];
    for (int i = 0; i < n; ++i) {
        if (Ns[i] <= 0) continue;  // an empty matrix gets no CTA
        int sm = 0;
        if (!plan_rows(types[i], M, K, max_smem, sh.CW, sh.H, G.p[m], sm)) return cudaErrorNotSupported;
        if (sm > smem) smem = sm;
        const int64_t RB = (K / 256) * block_bytes(types[i]);
        bytes[m] = Ns[i] * RB;
        rows[m] = Ns[i];
        need[m] = (Ns[i] * RB + (int64_t(1) << 30) - 1) >> 30;
        idx[m++] = i;
    }
    if (m == 0) return cudaSuccess;
    int g[QMM_GROUP_MAX];
    group_ctas(m, bytes, rows, need, num_sms, g);
    G.n = m;
    int64_t grid = 0;
    for (int j = 0; j < m; ++j) {
        const int i = idx[j];
        G.cta_begin[j] = static_cast<int>(grid);
        fill_rows(G.p[j], types[i], Ws[i], Ns[i], K, x, M, ys[i], status, g[j]);
        grid += g[j];
    }
    if (grid > 0x7fffffff) return cudaErrorInvalidValue;
    G.cta_begin[m] = static_cast<int>(grid);
    G.p[0].q.stop_stage = inject_stop_stage();
    const int gr = static_cast<int>(grid);
    if (M > 2) return launch_rows_wide_group(G, M <= 4 ? 4 : 8, sh.CW, sh.H, gr, smem, st);
    return M <= 1 ? launch_group<1, true>(G, sh.CW, sh.H, gr, smem, st)
                  : launch_group<2, true>(G, sh.CW, sh.H, gr, smem, st);
}

}  // namespace qk
