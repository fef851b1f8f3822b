// gemv_rows.cuh -- the row-per-lane decode kernel (device code, shared-memory
// plan and launch templates), instantiated by gemv_rows.cu (M <= 2, Q4_K,
// Q5_K, Q6_K, Q3_K and Q2_K) and gemv_rows_wide.cu / gemv_rows_wide_kq.cu /
// gemv_rows_wide_q6k.cu (3 <= M <= 8, every K-quant): decode product
// y[M,N] = W[N,K] . x[M,K]^T with one weight row per lane.
//
// Design (sm_103a):
//   * One CTA per SM owns a contiguous range of whole rows (balanced to one
//     row), taken in groups of GR = 32 / H: lane i of every consumer warp
//     works on row i mod GR of the group, in part i / GR of its columns.
//   * A producer warp streams the CTA's weights through a ring of stages.  A
//     stage is one group's GR rows x CH = CW*H super-blocks: one bulk copy
//     per row, rounded out to 16 bytes, at a row pitch of an odd number of
//     16-byte chunks, so the lanes reading one 16-byte word each touch
//     distinct bank groups.  A bulk copy costs the SM's copy engine a fixed
//     time (measured: about 23 copies per microsecond per SM, so copies
//     under ~2 KB cap the stream below HBM speed); H = 2 doubles a row's
//     span at the same stage size.  The ring is filled before the wait for
//     the preceding kernel: no kernel of the library writes weights.
//   * Consumer warp w takes super-block w + CW*part of each stage.  The lanes
//     of one part share the super-block index, so every activation and
//     scale-record read is a shared-memory broadcast (one per part); each
//     lane reads only its own row's quants and accumulates in registers over
//     the group's stages, with the exact int32 dp4a block dots of the
//     block-per-lane kernel (gemv_sb.cuh).
//   * At a group's end the parts of a row are added (part order), each warp
//     leaves its GR partial sums in shared memory and counts itself in; the
//     warp that completes the count adds the partials in warp order and
//     writes the group's y.  Every y element is written once, in a fixed
//     order, and no warp waits for another.
//   * The consumers quantise x into shared memory after the wait, while the
//     ring fills.  All waits are bounded.
//
// Compared with the block-per-lane kernel this removes the per-stage
// segmented scan (a lane's row does not change inside a group) and most of
// the shared-memory wavefronts of the activation reads.
#pragma once

#include "gemv_sb.cuh"

#include <algorithm>

namespace qk {
namespace rwk {

using namespace sbk;

constexpr int MAX_NS = 8;   // stages in the ring
constexpr int OFF_FULL = 0, OFF_EMPTY = 64, OFF_CNT = 128, OFF_FAIL = 192;
constexpr int HEAD = 256;
static_assert(OFF_CNT + 4 * (MAX_NS + 1) <= OFF_FAIL, "head layout");

struct RwParams {
    SbParams q;          // matrix, activations, output, row split, quantiser layout
    uint64_t w_end;      // first byte past the matrix
    int nq;              // stages per group: super-blocks per row / (CW*H), rounded up
    int NS;              // stages in the ring
    int nbuf;            // partial-sum buffers (NS + 1)
    int pitch;           // stage bytes per row
    int stage_bytes;     // rows per group * pitch
    int off_red, off_ring;
};

// Several matrices that share K and x in one launch: CTAs
// [cta_begin[i], cta_begin[i+1]) work on matrix i.
struct RwGroup {
    int n;
    int cta_begin[QMM_GROUP_MAX + 1];
    RwParams p[QMM_GROUP_MAX];
};

template <int T, int MT>
__device__ __forceinline__ void superblock(const XS &X, int blk, int kb, float (&v)[MT]) {
    if constexpr (T == QMM_Q4_K) sb_q4k<MT>(X, blk, kb, v);
    else if constexpr (T == QMM_Q5_K) sb_q5k<MT>(X, blk, kb, v);
    else if constexpr (T == QMM_Q3_K) sb_q3k<MT>(X, blk, kb, v);
    else if constexpr (T == QMM_Q2_K) sb_q2k<MT>(X, blk, kb, v);
    else sb_q6k<MT>(X, blk, kb, v);
}

template <int T, int MT, int CW, int H>
__device__ __forceinline__ void rows_body(const RwParams &R, const int cta) {
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int BB = Fmt<T>::BB;
    constexpr int NT = CW * 32;  // consumer threads
    constexpr int GR = 32 / H;   // rows per group
    constexpr int CH = CW * H;   // super-blocks per row per stage
    const SbParams &P = R.q;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int64_t r0 = P.rows_q * cta + min(cta, P.rows_r);
    const int rows = static_cast<int>(P.rows_q + (cta < P.rows_r ? 1 : 0));
    const int ng = (rows + GR - 1) / GR;
    const int total = ng * R.nq;  // stages of the CTA

    const uint32_t full0 = smem_u32(smem + OFF_FULL), empty0 = smem_u32(smem + OFF_EMPTY);
    int *cnt = reinterpret_cast<int *>(smem + OFF_CNT);
    volatile int *fail_flag = reinterpret_cast<volatile int *>(smem + OFF_FAIL);
    if (threadIdx.x == 0) {
        for (int i = 0; i < R.NS; ++i) {
            mbar_init(full0 + 8u * i, 1);
            mbar_init(empty0 + 8u * i, CW);
        }
        fence_mbar_init();
        *fail_flag = 0;
    }
    if (threadIdx.x < R.nbuf) cnt[threadIdx.x] = 0;
    __syncthreads();
    pdl_trigger();

    if (warp == CW) {
        // ---- producer: stage s = (group s / nq, chunk s % nq) ------------
        const uint64_t pol = policy_evict_first();
        // stages from `stop` on are never issued (only with the test hook:
        // the consumers' bounded wait on stage `stop` then expires)
        const int stop = cta == 0 ? P.stop_stage : NO_STOP;
        int issued = 0;
        int gi = 0, kc = 0;
        for (int s = 0; s < total; ++s) {
            const int slot = s % R.NS;
            if (s >= R.NS) {
                // the consumers' release of this slot's previous stage
                bool ok = true;
                if (lane == 0) ok = mbar_wait(empty0 + 8u * slot, static_cast<uint32_t>((s / R.NS - 1) & 1), P.status);
                if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
                    if (lane == 0) *fail_flag = 1;
                    break;
                }
            }
            if (s >= stop) break;
            const int sb0 = kc * CH, nsb = min(CH, P.nb - sb0);
            uint8_t *dst = smem + R.off_ring + slot * R.stage_bytes + lane * R.pitch;
            uint64_t src = 0;
            uint32_t bytes = 0;
            if (lane < GR && GR * gi + lane < rows) {
                const uint64_t start = reinterpret_cast<uint64_t>(P.W) +
                                       static_cast<uint64_t>(r0 + GR * gi + lane) * static_cast<uint64_t>(P.RB) +
                                       static_cast<uint64_t>(BB) * static_cast<uint64_t>(sb0);
                const uint64_t end = start + static_cast<uint64_t>(BB) * static_cast<uint64_t>(nsb);
                src = start & ~uint64_t(15);
                uint64_t e16 = (end + 15) & ~uint64_t(15);
                if (e16 > R.w_end) {
                    // the matrix's last bytes (its end is not on a 16-byte
                    // boundary): plain loads, never reading past the end
                    e16 = end & ~uint64_t(15);
                    if (e16 < src) e16 = src;
                    for (uint64_t a = e16; a < end; ++a)
                        dst[a - src] = *reinterpret_cast<const uint8_t *>(a);
                    // later bulk copies into this slot come after these stores
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                }
                bytes = static_cast<uint32_t>(e16 - src);
            }
            const uint32_t all = __reduce_add_sync(0xffffffffu, bytes);
            __syncwarp();  // the plain tail stores before the arrival that publishes them
            if (lane == 0) mbar_arrive_expect_tx(full0 + 8u * slot, all);
            if (bytes > 0) bulk_g2s(smem_u32(dst), reinterpret_cast<const void *>(src), bytes, full0 + 8u * slot, pol);
            issued = s + 1;
            if (++kc == R.nq) kc = 0, ++gi;
        }
        // no copy may still be in flight when the CTA exits (stages that were
        // never issued are not waited for)
        if (lane == 0)
            for (int s = max(0, issued - R.NS); s < issued; ++s)
                mbar_wait(full0 + 8u * (s % R.NS), static_cast<uint32_t>((s / R.NS) & 1), P.status);
        return;
    }

    // ---- consumers ---------------------------------------------------------
    // warm L2 with x (an L2 prefetch cannot leave a stale copy: L2 is the
    // point of coherence); x itself is read after the wait
    if (threadIdx.x == 0 && P.x_vec && ((P.M * P.K * 4) & 15) == 0)
        bulk_prefetch_l2(P.x, static_cast<uint32_t>(P.M * P.K * 4));
    pdl_wait();  // x is read and y written only after the preceding kernel completed
    quantize_to_smem<T, NT>(P, smem, [] {});
    named_barrier(1, NT);

    XS X;
    X.sm = smem;
    X.xq = P.off_xq;
    X.meta = P.off_meta;
    X.q_ld = P.q_ld;
    X.meta_ld = P.meta_ld;
    float *red = reinterpret_cast<float *>(smem + R.off_red);  // [nbuf][CW][MT][GR]
    const int lr = lane % GR, part = lane / GR;  // this lane's row in the group, its part of the columns

    bool failed = false;
    float v[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) v[m] = 0.0f;
    int gi = 0, kc = 0, slot = 0;
    uint32_t phase = 0;
    for (int s = 0; s < total; ++s) {
        if (!failed && !__all_sync(0xffffffffu, mbar_wait(full0 + 8u * slot, phase, P.status))) failed = true;
        const int rl = GR * gi + lr;                  // this lane's row inside the CTA
        const int js = warp + CW * part;              // its super-block of the stage
        const int kb = kc * CH + js;                  // ... of the row
        if (!failed && kb < P.nb && rl < rows) {
            // the row's span starts (start mod 16) bytes into its copy
            const uint64_t start = static_cast<uint64_t>(r0 + rl) * static_cast<uint64_t>(P.RB) +
                                   static_cast<uint64_t>(BB) * static_cast<uint64_t>(kc * CH);
            const int blk = R.off_ring + slot * R.stage_bytes + lr * R.pitch +
                            static_cast<int>((reinterpret_cast<uint64_t>(P.W) + start) & 15) + js * BB;
            superblock<T, MT>(X, blk, kb, v);
        }
        // this warp is done with the stage
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8u * slot);
        if (++slot == R.NS) slot = 0, phase ^= 1u;
        if (++kc < R.nq) continue;
        // ---- the group's end: the parts of each row added in part order,
        // then the warps' partial sums, added in warp order by the last warp
#pragma unroll
        for (int h = GR; h < 32; h <<= 1)
#pragma unroll
            for (int m = 0; m < MT; ++m) v[m] += __shfl_down_sync(0xffffffffu, v[m], h);
        const int buf = gi % R.nbuf;
        float *pb = red + buf * (CW * MT * GR);
        if (lane < GR)
#pragma unroll
            for (int m = 0; m < MT; ++m) pb[(warp * MT + m) * GR + lane] = v[m];
        __syncwarp();
        int last = 0;
        if (lane == 0) {
            if (failed) *fail_flag = 1;
            __threadfence_block();
            last = atomicAdd(cnt + buf, 1) == CW - 1;
        }
        if (__shfl_sync(0xffffffffu, last, 0)) {
            __threadfence_block();
            if (*fail_flag == 0 && lane < GR && rl < rows) {
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    float acc = 0.0f;
#pragma unroll
                    for (int w = 0; w < CW; ++w) acc += pb[(w * MT + m) * GR + lane];
                    if (m < P.M) P.y[static_cast<int64_t>(m) * P.N + r0 + rl] = acc;
                }
            }
            __syncwarp();
            if (lane == 0) cnt[buf] = 0;
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) v[m] = 0.0f;
        kc = 0;
        ++gi;
    }
}

template <int T, int MT, int CW, int H>
__global__ void __launch_bounds__((CW + 1) * 32, 1) gemv_rows_kernel(const __grid_constant__ RwParams R) {
    rows_body<T, MT, CW, H>(R, static_cast<int>(blockIdx.x));
}

// Q6K: the launch may hold Q6_K matrices (else Q4_K only)
template <int MT, int CW, int H, bool Q6K>
__global__ void __launch_bounds__((CW + 1) * 32, 1) gemv_rows_group_kernel(const __grid_constant__ RwGroup G) {
    int i = 0;
    while (i + 1 < G.n && static_cast<int>(blockIdx.x) >= G.cta_begin[i + 1]) ++i;
    const int cta = static_cast<int>(blockIdx.x) - G.cta_begin[i];
    if (!Q6K || G.p[i].q.type == QMM_Q4_K) rows_body<QMM_Q4_K, MT, CW, H>(G.p[i], cta);
    else rows_body<QMM_Q6_K, MT, CW, H>(G.p[i], cta);
}

inline int64_t align_to(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

// The kernel's shape for a row of nb super-blocks of BB bytes: CW consumer
// warps (8 or 10) and H parts per row (1 or 2), scored by the share of a
// stage's super-block slots that hold work times the copy engine's
// efficiency at the row span's size (full from 2 KB on, in proportion below:
// the measured rate of bulk copies); ties to the larger CW, then to H = 1.
struct Shape {
    int CW, H;
    double score;
};
inline Shape choose_shape(int64_t nb, int BB) {
    Shape best = {8, 1, -1.0};
    const int cws[2] = {10, 8}, hs[2] = {1, 2};
    for (int cw : cws)
        for (int h : hs) {
            const int64_t ch = static_cast<int64_t>(cw) * h;
            const double fill = static_cast<double>(nb) / static_cast<double>((nb + ch - 1) / ch * ch);
            const double span = static_cast<double>(std::min(ch, nb) * BB);
            const double sc = fill * std::min(1.0, span / 2048.0);
            if (sc > best.score + 1e-9) best = {cw, h, sc};
        }
    return best;
}

// Shared-memory plan: head | x quantised [MT][q_ld] | scale records
// [MT][meta_ld] | partial sums [nbuf][CW][MT][GR] | ring of NS stages of GR
// rows x pitch.  The most stages that fit, at least two.
inline bool plan_rows(int type, int M, int64_t K, int max_smem, int CW, int H, RwParams &R, int &smem) {
    const int MT = M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8;
    const int BB = block_bytes(type);
    const int GR = 32 / H;
    const int64_t nb = K / 256;
    const int64_t q_ld = nb * XPITCH;
    const int64_t meta_ld = nb * (type == QMM_Q4_K || type == QMM_Q5_K ? Rec<QMM_Q4_K>::B : Rec<QMM_Q6_K>::B);
    // a row's span: CW*H super-blocks from an offset of up to 15 bytes into
    // its first 16-byte chunk, rounded out; an odd number of chunks
    const int64_t CH = static_cast<int64_t>(CW) * H;
    const int64_t chunks = (BB % 16 == 0) ? CH * BB / 16 : (CH * BB + 30) / 16;
    const int64_t pitch = 16 * (chunks | 1);
    const int64_t stage = GR * pitch;
    const int64_t o_xq = HEAD;
    const int64_t o_meta = align_to(o_xq + MT * q_ld, 128);
    const int64_t o_red = align_to(o_meta + MT * meta_ld, 128);
    for (int ns = MAX_NS; ns >= 2; --ns) {
        const int64_t o_ring = align_to(o_red + static_cast<int64_t>(ns + 1) * CW * MT * GR * 4, 128);
        const int64_t need = o_ring + ns * stage;
        if (need > max_smem) continue;
        R.NS = ns;
        R.nbuf = ns + 1;
        R.pitch = static_cast<int>(pitch);
        R.stage_bytes = static_cast<int>(stage);
        R.nq = static_cast<int>((nb + CH - 1) / CH);
        R.q.q_ld = static_cast<int>(q_ld);
        R.q.meta_ld = static_cast<int>(meta_ld);
        R.q.off_xq = static_cast<int>(o_xq);
        R.q.off_meta = static_cast<int>(o_meta);
        R.off_red = static_cast<int>(o_red);
        R.off_ring = static_cast<int>(o_ring);
        smem = static_cast<int>(need);
        return true;
    }
    return false;
}

// Matrix, activations and the split of the N rows over g CTAs.
inline void fill_rows(RwParams &R, int type, const void *W, int64_t N, int64_t K, const float *x, int M, float *y,
               int *status, int g) {
    SbParams &P = R.q;
    P.type = type;
    P.W = static_cast<const uint8_t *>(W);
    P.N = N;
    P.K = static_cast<int>(K);
    P.M = M;
    P.nb = static_cast<int>(K / 256);
    P.RB = P.nb * block_bytes(type);
    P.total_bytes = N * static_cast<int64_t>(P.RB);
    P.x = x;
    P.x_vec = (reinterpret_cast<uintptr_t>(x) & 15) == 0 ? 1 : 0;
    P.y = y;
    P.status = status;
    P.stop_stage = NO_STOP;
    P.rows_q = N / g;
    P.rows_r = static_cast<int>(N % g);
    R.w_end = reinterpret_cast<uint64_t>(W) + static_cast<uint64_t>(P.total_bytes);
}

template <class Kern, class Arg>
cudaError_t launch_pdl(Kern kfn, const Arg &arg, int grid, int threads, int smem, cudaStream_t st) {
    cudaError_t e = set_smem_attrs(kfn, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kfn, arg);
}

template <int T, int MT>
cudaError_t launch_single(const RwParams &R, int CW, int H, int grid, int smem, cudaStream_t st) {
    if (CW == 8)
        return H == 1 ? launch_pdl(gemv_rows_kernel<T, MT, 8, 1>, R, grid, 9 * 32, smem, st)
                      : launch_pdl(gemv_rows_kernel<T, MT, 8, 2>, R, grid, 9 * 32, smem, st);
    return H == 1 ? launch_pdl(gemv_rows_kernel<T, MT, 10, 1>, R, grid, 11 * 32, smem, st)
                  : launch_pdl(gemv_rows_kernel<T, MT, 10, 2>, R, grid, 11 * 32, smem, st);
}

template <int MT, bool Q6K>
cudaError_t launch_group(const RwGroup &G, int CW, int H, int grid, int smem, cudaStream_t st) {
    if (CW == 8)
        return H == 1 ? launch_pdl(gemv_rows_group_kernel<MT, 8, 1, Q6K>, G, grid, 9 * 32, smem, st)
                      : launch_pdl(gemv_rows_group_kernel<MT, 8, 2, Q6K>, G, grid, 9 * 32, smem, st);
    return H == 1 ? launch_pdl(gemv_rows_group_kernel<MT, 10, 1, Q6K>, G, grid, 11 * 32, smem, st)
                  : launch_pdl(gemv_rows_group_kernel<MT, 10, 2, Q6K>, G, grid, 11 * 32, smem, st);
}

// The launches for 3 <= M <= 8 (gemv_rows_wide.cu, gemv_rows_wide_kq.cu,
// gemv_rows_wide_q6k.cu): MT = 4 or 8.
cudaError_t launch_rows_wide(const RwParams &R, int MT, int CW, int H, int grid, int smem, cudaStream_t st);
cudaError_t launch_rows_wide_kq(const RwParams &R, int MT, int CW, int H, int grid, int smem, cudaStream_t st);
cudaError_t launch_rows_wide_q6k(const RwParams &R, int MT, int CW, int H, int grid, int smem, cudaStream_t st);
cudaError_t launch_rows_wide_group(const RwGroup &G, int MT, int CW, int H, int grid, int smem, cudaStream_t st);
cudaError_t launch_rows_wide_group_q6k(const RwGroup &G, int MT, int CW, int H, int grid, int smem, cudaStream_t st);

}  // namespace rwk
}  // namespace qk
