// gemv_sb.cu -- decode product y[M,N] = W[N,K] . x[M,K]^T for small M with
// one weight block per lane: a whole 256-weight super-block for Q4_K/Q6_K,
// one 32-weight block for Q8_0.
//
// Design (sm_103a):
//   * One CTA per SM owns a contiguous range of whole output rows.  Its
//     blocks, in memory order, are split evenly (to one block) between
//     twelve warps.
//   * Every warp streams its own slice through a private ring of stages of
//     32 blocks with 1-D bulk async copies (cp.async.bulk + mbarrier, issued
//     by lane 0), so each SM keeps ~80-160 KB in flight.  Q6_K/Q8_0 blocks
//     are only 2-byte aligned: a stage is copied from its start rounded down
//     to 16 bytes and indexed from the remainder.
//   * Lane i computes block i of the stage with exact int32 dp4a dot products
//     against the quantised activations in shared memory; the per-block
//     scale handling (six-bit scales and mins, 16-weight groups) is amortised
//     over 256 weights.  The activations are stored at a pitch of 272 bytes
//     per super-block so lanes reading consecutive super-blocks hit distinct
//     banks.
//   * A segmented shuffle scan sums the lanes of each row inside a stage;
//     rows crossing stages carry in registers; rows cut by a warp boundary
//     are parked in shared memory and added in warp order after a final CTA
//     barrier.  Every y element is produced once, in a fixed order.
//   * All waits are bounded mbarrier waits; the quantiser runs just before
//     with programmatic dependent launch, so the weight stream starts first.
#include "gemv_sb.cuh"

namespace qk {

namespace {

using namespace sbk;

// Several matrices that share K and x in one launch: CTAs
// [cta_begin[i], cta_begin[i+1]) work on matrix i, each as in the single
// launch (its own type, shared-memory plan and share of rows).
struct SbGroup {
    int n;
    int cta_begin[QMM_GROUP_MAX + 1];
    SbParams p[QMM_GROUP_MAX];
};

template <int MT>
__global__ void __launch_bounds__(NTHREADS, 1) gemv_sb_group_kernel(const __grid_constant__ SbGroup G) {
    int i = 0;
    while (i + 1 < G.n && static_cast<int>(blockIdx.x) >= G.cta_begin[i + 1]) ++i;
    const SbParams &P = G.p[i];
    const int cta = static_cast<int>(blockIdx.x) - G.cta_begin[i];
    switch (P.type) {
    case QMM_Q4_K: sb_body<QMM_Q4_K, MT>(P, cta); break;
    case QMM_Q6_K: sb_body<QMM_Q6_K, MT>(P, cta); break;
    default: sb_body<QMM_Q8_0, MT>(P, cta); break;  // the group launch takes Q8_0, Q4_K, Q6_K
    }
}

int mt_of(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8; }

int64_t align64(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

// Shared-memory plan: header | activations | NWARP rings of NSW stages.
bool plan_sb(int type, int M, int64_t K, int max_smem, SbParams &P, int &smem) {
    const int MT = mt_of(M);
    const int BB = block_bytes(type);
    const int64_t q_ld = ((K + 255) / 256) * XPITCH;
    const int64_t meta_ld = type == QMM_Q8_0 ? align64((K / 32) * 4, 16)
                                             : (K / 256) * (type == QMM_Q4_K || type == QMM_Q5_K ? 80 : 112);
    int64_t off = HEAD_BYTES;
    const int64_t o_xq = off;
    off = align64(off + MT * q_ld, 128);
    const int64_t o_meta = off;
    off = align64(off + MT * meta_ld, 128);
    const int64_t o_ring = off;
    const int64_t slot = align64(static_cast<int64_t>(SU) * BB + 32, 128);
    int64_t nsw = (max_smem - o_ring) / (NWARP * slot);
    if (nsw > MAX_NSW) nsw = MAX_NSW;
    if (nsw < 2) return false;
    P.NSW = static_cast<int>(nsw);
    P.slot_bytes = static_cast<int>(slot);
    P.off_edge = 8 * NWARP * MAX_NSW;
    P.q_ld = static_cast<int>(q_ld);
    P.meta_ld = static_cast<int>(meta_ld);
    P.off_xq = static_cast<int>(o_xq);
    P.off_meta = static_cast<int>(o_meta);
    P.off_ring = static_cast<int>(o_ring);
    smem = static_cast<int>(o_ring + NWARP * nsw * slot);
    return true;
}

}  // namespace

bool gemv_sb_fits(int type, int M, int64_t K, int max_smem) {
    if (M < 1 || M > 8 || K > (1 << 22)) return false;
    SbParams P = {};
    int smem = 0;
    return plan_sb(type, M, K, max_smem, P, smem);
}

namespace {

// CTAs a matrix needs at least, so that one CTA's bytes fit 30 bits.
int64_t min_ctas(int64_t N, int RB) {
    const int64_t max_rows = (int64_t(1) << 30) / RB;
    return (N + max_rows - 1) / max_rows;
}

// Everything but the shared-memory plan: matrix, activations, and the split
// of the N rows over g CTAs.
void fill(SbParams &P, int type, const void *W, int64_t N, int64_t K, const float *x, int M, float *y,
          int *status, int g) {
    P.type = type;
    P.W = static_cast<const uint8_t *>(W);
    P.N = N;
    P.K = static_cast<int>(K);
    P.M = M;
    P.nb = static_cast<int>(K / block_weights(type));
    P.RB = P.nb * block_bytes(type);
    P.total_bytes = N * static_cast<int64_t>(P.RB);
    P.x = x;
    P.x_vec = (reinterpret_cast<uintptr_t>(x) & 15) == 0 ? 1 : 0;
    P.y = y;
    P.status = status;
    P.stop_stage = NO_STOP;
    P.rows_q = N / g;
    P.rows_r = static_cast<int>(N % g);
    // Row of block u by multiply-high: with M = floor(2^32/nb) + 1 and
    // e = M*nb - 2^32 in (0, nb], u*M/2^32 = u/nb + u*e/(nb*2^32), whose
    // floor is floor(u/nb) whenever u*e < 2^32, which u*nb < 2^32 ensures.
    const uint64_t u_max = static_cast<uint64_t>(P.rows_q + 1) * static_cast<uint64_t>(P.nb);
    P.nb_magic = u_max * static_cast<uint64_t>(P.nb) < (uint64_t(1) << 32)
                     ? static_cast<uint32_t>((uint64_t(1) << 32) / static_cast<uint64_t>(P.nb) + 1)
                     : 0u;
}

template <int MT>
cudaError_t launch_group_mt(const SbGroup &G, int grid, int smem, cudaStream_t st) {
    auto kfn = gemv_sb_group_kernel<MT>;
    cudaError_t e = set_smem_attrs(kfn, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kfn, G);
}

}  // namespace

cudaError_t launch_gemv_sb(int type, const void *W, int64_t N, int64_t K, const float *x, int M,
                           float *y, cudaStream_t st, int num_sms, int max_smem, int *status) {
    SbParams P = {};
    int smem = 0;
    if (!plan_sb(type, M, K, max_smem, P, smem)) return cudaErrorInvalidValue;
    // one CTA per SM; more when a CTA's bytes would not fit 30 bits
    int64_t grid = num_sms;
    const int64_t need = min_ctas(N, static_cast<int>(K / block_weights(type)) * block_bytes(type));
    if (grid < need) grid = need;
    if (N < grid) grid = N;
    if (grid < 1) grid = 1;
    if (grid > 0x7fffffff) return cudaErrorInvalidValue;
    const int g = static_cast<int>(grid);
    fill(P, type, W, N, K, x, M, y, status, g);
    P.stop_stage = inject_stop_stage();
    switch (type) {
    case QMM_Q8_0: return launch_m<QMM_Q8_0>(P, mt_of(M), g, smem, st);
    case QMM_Q4_K: return launch_m<QMM_Q4_K>(P, mt_of(M), g, smem, st);
    case QMM_Q5_K:
    case QMM_Q3_K:
    case QMM_Q2_K: return launch_sb_kquant(type, P, mt_of(M), g, smem, st);
    default: return launch_m<QMM_Q6_K>(P, mt_of(M), g, smem, st);
    }
}

cudaError_t launch_gemv_sb_gateup(int type, const void *Wg, const void *Wu, int64_t N, int64_t K, const float *x,
                                  int M, float *h, cudaStream_t st, int num_sms, int max_smem, int *status) {
    if (M > 2) return cudaErrorNotSupported;  // the table holds MT <= 2 values per row
    int64_t grid = num_sms;
    const int64_t need = min_ctas(N, static_cast<int>(K / block_weights(type)) * block_bytes(type));
    if (grid < need) grid = need;
    if (N < grid) grid = N;
    if (grid < 1) grid = 1;
    if (grid > 0x7fffffff) return cudaErrorInvalidValue;
    const int g = static_cast<int>(grid);
    const int MT = mt_of(M);
    // the row table after the rings: 2 matrices x (rows of the largest CTA) x MT floats
    const int64_t tab_bytes = align64(2 * (N / g + 1) * MT * 4, 128);
    if (tab_bytes > max_smem / 4) return cudaErrorNotSupported;
    SbParams P = {};
    int smem = 0;
    if (!plan_sb(type, M, K, max_smem - static_cast<int>(tab_bytes), P, smem)) return cudaErrorNotSupported;
    fill(P, type, Wg, N, K, x, M, h, status, g);
    P.W2 = static_cast<const uint8_t *>(Wu);
    P.off_tab = smem;
    smem += static_cast<int>(tab_bytes);
    P.stop_stage = inject_stop_stage();
    switch (type) {
    case QMM_Q8_0: return launch_m<QMM_Q8_0>(P, MT, g, smem, st);
    case QMM_Q4_K: return launch_m<QMM_Q4_K>(P, MT, g, smem, st);
    case QMM_Q5_K:
    case QMM_Q3_K:
    case QMM_Q2_K: return launch_sb_kquant(type, P, MT, g, smem, st);
    default: return launch_m<QMM_Q6_K>(P, MT, g, smem, st);
    }
}

void group_ctas(int n, const int64_t *bytes, const int64_t *rows, const int64_t *need, int num_sms, int *g) {
    // CTAs in proportion to the bytes (largest remainders), at least one per
    // matrix (and at least `need`), at most one per row
    int64_t total = 0;
    for (int i = 0; i < n; ++i) total += bytes[i];
    int used = 0;
    double frac[QMM_GROUP_MAX];
    for (int i = 0; i < n; ++i) {
        const double want = total > 0 ? static_cast<double>(num_sms) * static_cast<double>(bytes[i]) /
                                            static_cast<double>(total)
                                      : 1.0;
        int64_t gi = static_cast<int64_t>(want);
        frac[i] = want - static_cast<double>(gi);
        if (gi < 1) gi = 1;
        if (gi < need[i]) gi = need[i];
        if (gi > rows[i]) gi = rows[i];
        g[i] = static_cast<int>(gi);
        used += g[i];
    }
    while (used < num_sms) {
        int best = -1;
        for (int i = 0; i < n; ++i)
            if (frac[i] >= 0.0 && g[i] < rows[i] && (best < 0 || frac[i] > frac[best])) best = i;
        if (best < 0) break;
        ++g[best];
        frac[best] = -1.0;  // at most one extra CTA each
        ++used;
    }
}

cudaError_t launch_gemv_sb_group(int n, const int *types, const void *const *Ws, const int64_t *Ns, int64_t K,
                                 const float *x, int M, float *const *ys, cudaStream_t st, int num_sms,
                                 int max_smem, int *status) {
    if (n < 1 || n > QMM_GROUP_MAX) return cudaErrorInvalidValue;
    for (int i = 0; i < n; ++i)
        if (Ns[i] > 0 && types[i] != QMM_Q8_0 && types[i] != QMM_Q4_K && types[i] != QMM_Q6_K)
            return cudaErrorNotSupported;
    SbGroup G = {};
    int idx[QMM_GROUP_MAX], smem = 0, m = 0;
    int64_t bytes[QMM_GROUP_MAX], rows[QMM_GROUP_MAX], need[QMM_GROUP_MAX];
    for (int i = 0; i < n; ++i) {
        if (Ns[i] <= 0) continue;  // an empty matrix gets no CTA
        int sm = 0;
        if (!plan_sb(types[i], M, K, max_smem, G.p[m], sm)) return cudaErrorNotSupported;
        if (sm > smem) smem = sm;
        const int RB = static_cast<int>(K / block_weights(types[i])) * block_bytes(types[i]);
        bytes[m] = Ns[i] * RB;
        rows[m] = Ns[i];
        need[m] = min_ctas(Ns[i], RB);
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
        fill(G.p[j], types[i], Ws[i], Ns[i], K, x, M, ys[i], status, g[j]);
        grid += g[j];
    }
    if (grid > 0x7fffffff) return cudaErrorInvalidValue;
    G.cta_begin[m] = static_cast<int>(grid);
    G.p[0].stop_stage = inject_stop_stage();
    switch (mt_of(M)) {
    case 1: return launch_group_mt<1>(G, static_cast<int>(grid), smem, st);
    case 2: return launch_group_mt<2>(G, static_cast<int>(grid), smem, st);
    case 4: return launch_group_mt<4>(G, static_cast<int>(grid), smem, st);
    default: return launch_group_mt<8>(G, static_cast<int>(grid), smem, st);
    }
}

}  // namespace qk
