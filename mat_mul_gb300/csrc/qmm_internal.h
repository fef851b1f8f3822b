// qmm_internal.h -- declarations shared by the translation units of libqmm:
// the quantiser's output description and every kernel launcher.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace qk {

// Output layout of the quantiser.  q rows have stride q_ld bytes; with
// swizzle != 0 the 16-byte chunk c (0..15) of every 256-element super-block
// sb is stored at chunk position c ^ (sb & 7), so lanes that read the same
// chunk of consecutive super-blocks hit distinct shared-memory banks.  Every
// other output is optional (null = not written):
//   d   [M][d_ld]   fp32 scale per block of 32
//   s32 [M][d_ld]   int32 sum per block
//   s16 [M][s16_ld] int32 sums of the two 16-element halves of every block
//   dsf [M][d_ld]   fp32 product d * s32 per block
//   xh  [M][xh_ld]  fp16 of the dequantised activation times a power of
//                   two per row, d * q * 2^e_m (xinv[m] = 2^-e_m): plain
//                   layout, or with xh_mma != 0 the layout of the tensor-core
//                   decode kernel (gemv_mma.cu): element l of block b at half
//                   32b + ((l>>4)*2 + (l&1))*8 + ((l>>2)&3)*2 + ((l>>1)&1),
//                   then after the K halves the block sums of the fp16
//                   values times 2^-5 as hi + lo, per super-block 8 hi then
//                   8 lo, sub-block j at slot 2(j mod 4) + j/4 (xh_ld >=
//                   K + K/16).  When xh is set only the fp16
//                   outputs (xh, xs16, xinv) are written.
struct QuantOut {
    int8_t *q;
    int64_t q_ld;
    int swizzle;
    float *d;
    int32_t *s32;
    int32_t *s16;
    float *dsf;
    int64_t d_ld, s16_ld;
    void *xh;  // __half
    int64_t xh_ld;
    int xh_mma;
    float *xs16;  // with xh_mma: the sums X of the fp16 values per 16 elements times 2^-4 as fp16 hi + lo,
                  // per 256 elements [hi | lo][groups 0-7 | 8-15][8 tokens][8] (512 bytes), tokens >= M zero
    float *xinv;  // with xh: [M] the factor 2^-e_m that undoes row m's power of two
};

// trigger_dependents: let the next kernel (launched with programmatic
// dependent launch) start once every CTA of this one is running; the trigger
// comes after this kernel's own wait for its predecessor, so everything the
// next kernel does before its wait sees all earlier kernels complete.
// pdl_launch: launch this kernel itself with programmatic dependent launch.
cudaError_t launch_quantize(const float *x, int64_t M, int64_t K, const QuantOut &o, cudaStream_t st,
                            bool trigger_dependents, int num_sms, bool pdl_launch = false);

// cuTensorMapEncodeTiled from the driver (null when it cannot be found).
using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiled tensor_map_encoder();

cudaError_t launch_dequant(int type, const void *blocks, int64_t n_elems, float *out,
                           cudaStream_t st, int num_sms);

// Round-based decode kernel (gemv.cu): activations q [M][K] (plain layout),
// d [M][xd_ld], s16 [M][xs_ld].
bool gemv_fits(int type, int M, int64_t K, int xd_ld, int xs_ld, int max_smem);
cudaError_t launch_gemv(int type, const void *W, int64_t N, int64_t K, const int8_t *xq,
                        const float *xd, const int32_t *xs, int xd_ld, int xs_ld, int M, float *y,
                        cudaStream_t st, bool pdl, int num_sms, int max_smem, int *status);

// Block-per-lane decode kernel (gemv_sb.cu): quantises x itself, needs no
// workspace; launched with programmatic dependent launch.
bool gemv_sb_fits(int type, int M, int64_t K, int max_smem);
cudaError_t launch_gemv_sb(int type, const void *W, int64_t N, int64_t K, const float *x, int M,
                           float *y, cudaStream_t st, int num_sms, int max_smem, int *status);
// Several matrices sharing K and x (M <= 8) in one launch of the same kernel;
// CTAs are split between them in proportion to their bytes (group_ctas).
// cudaErrorNotSupported when one of them does not fit the kernel's plan.
cudaError_t launch_gemv_sb_group(int n, const int *types, const void *const *Ws, const int64_t *Ns, int64_t K,
                                 const float *x, int M, float *const *ys, cudaStream_t st, int num_sms,
                                 int max_smem, int *status);
void group_ctas(int n, const int64_t *bytes, const int64_t *rows, const int64_t *need, int num_sms, int *g);

// Row-per-lane decode kernel (gemv_rows.cu): Q4_K, Q5_K, Q6_K, Q3_K and Q2_K
// for M <= 8, K a multiple of 256; quantises x itself (one
// launch, no workspace), launched with programmatic dependent launch.  The
// group launch takes several Q4_K / Q6_K matrices sharing K and x (CTAs
// split as in group_ctas); cudaErrorNotSupported when one of them does not
// fit the kernel's plan or is of another type.
bool gemv_rows_fits(int type, int M, int64_t K, int max_smem);
// Whether the row-per-lane kernel is the faster choice for this matrix (by
// its copy sizes and the matrix size; from M = 2 on always for Q5_K, Q3_K
// and Q2_K, never for Q4_K beyond M = 2); qmm_set_decode_path(
// QMM_DECODE_ROWS) takes it wherever it fits.
bool gemv_rows_preferred(int type, int M, int64_t N, int64_t K);
cudaError_t launch_gemv_rows(int type, const void *W, int64_t N, int64_t K, const float *x, int M, float *y,
                             cudaStream_t st, int num_sms, int max_smem, int *status);
cudaError_t launch_gemv_rows_group(int n, const int *types, const void *const *Ws, const int64_t *Ns, int64_t K,
                                   const float *x, int M, float *const *ys, cudaStream_t st, int num_sms,
                                   int max_smem, int *status);
// The gate and up products of one MLP (same type and shape, M <= 2) in one
// launch of the block-per-lane kernel: h = silu(Wg.x) * (Wu.x).
// cudaErrorNotSupported when the pair does not fit the kernel's plan.
cudaError_t launch_gemv_sb_gateup(int type, const void *Wg, const void *Wu, int64_t N, int64_t K, const float *x,
                                  int M, float *h, cudaStream_t st, int num_sms, int max_smem, int *status);

// h = silu(g) * u elementwise over n values (gate_up.cu).
cudaError_t launch_silu_mul(const float *g, const float *u, float *h, int64_t n, cudaStream_t st, int num_sms);

// Decode for 2 <= M <= 8 on the tensor cores (gemv_mma.cu): Q4_K or Q6_K,
// sixteen weight rows per mma.sync.m16n8k16 (fp16 operands, fp32
// accumulation).  xh: the quantiser's output with xh_mma, [M][2K + K/8
// bytes] (16-byte aligned), then the group sums (xs16: 512 bytes per 256 of
// K, fp16 hi/lo tiles), then
// the row factors xinv [8] fp32; the kernel copies one K window of it at a
// time into shared memory.
// Launched with programmatic dependent launch right after that quantiser
// (launched with trigger_dependents): the kernel streams weights before it
// waits, and reads xh after.
// With gate (g [M][N], written by the launch just before on the stream)
// the kernel writes y = silu(g) * (W.x) instead of W.x.
bool gemv_mma_fits(int type, int M, int64_t N, int64_t K, int max_smem, int num_sms);
cudaError_t launch_gemv_mma(int type, const void *W, int64_t N, int64_t K, const void *xh, int M, float *y,
                            cudaStream_t st, int num_sms, int max_smem, int *status, const float *gate = nullptr);
// Several Q4_K / Q6_K matrices that share K and xh in one launch (CTAs split
// as in group_ctas, at most one per 8-row half); cudaErrorNotSupported when
// one of them does not fit the kernel.
cudaError_t launch_gemv_mma_group(int n, const int *types, const void *const *Ws, const int64_t *Ns, int64_t K,
                                  const void *xh, int M, float *const *ys, cudaStream_t st, int num_sms,
                                  int max_smem, int *status);

// Prefill GEMM on tcgen05 (gemm_tc.cu): Q4_K, Q6_K or Q8_0 weights with K a
// multiple of 256, fp16 activations xh [M][K] (d*q*2^e_m from the
// quantiser) and the row factors xinv [M] = 2^-e_m.  Returns
// cudaErrorNotSupported for shapes it does not take.
bool gemm_tc_supported(int type, int64_t N, int64_t K, int64_t M);
cudaError_t launch_gemm_tc(int type, const void *W, int64_t N, int64_t K, const void *xh, const float *xinv,
                           int64_t M, float *y, cudaStream_t st, int num_sms, int *status);

// Prefill GEMM on mma.sync (gemm_mma.cu), every block type: q [M][K], d
// and s32 [M][xd_ld]; Q2_K also needs the 16-element sums s16 [M][xs16_ld]
// (two per block).
cudaError_t launch_gemm_mma(int type, const void *W, int64_t N, int64_t K, const int8_t *xq,
                            const float *xd, const int32_t *xs, int xd_ld, int64_t M, float *y,
                            cudaStream_t st, const int32_t *xs16 = nullptr, int xs16_ld = 0);

// Product with the transposed Q8_0 matrices (qmm_t.cu): y[h][m][k] =
// sum_n x[h][m][n] * w[h][n][k], K a multiple of 32 up to 256.  part: the
// workspace of qmm_t_part_bytes() bytes; count: H unsigned counters that are
// zero before the call and are left zero by it.  One launch per 16 rows of x.
int64_t qmm_t_chunk_rows(int64_t H, int64_t N, int64_t K, int num_sms);
size_t qmm_t_part_bytes(int64_t H, int64_t N, int64_t K, int num_sms);
cudaError_t launch_qmm_t(const void *W, int64_t H, int64_t N, int64_t K, const float *x, int64_t M, float *y,
                         float *part, unsigned *count, cudaStream_t st, int num_sms, int *status);

// Set the calling thread's qmm_last_error() text; returns code.
int record_error(int code, const char *msg);
// Add n kernel launches to the count qmm_launch_count() reports.
void count_launches(int64_t n);

// Failure-detection test hook (qmm_inject_stall): the stage at which the
// first CTA's producer of the next weight-streaming launch stops issuing
// copies (1 while an injection is pending, consumed by this call), else a
// value no launch reaches.
int inject_stop_stage();
constexpr int NO_STOP = 0x7fffffff;

}  // namespace qk
