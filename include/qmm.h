/*
 * qmm.h -- C ABI of libqmm: the quantized-weight matrix product y = W.x on
 * NVIDIA GB300 (sm_103a), with W stored in GGUF block formats.
 *
 * The operation is the one the LLM engines on the blazr README ("Model
 * Formats > GGUF": dp4a CUDA kernels for Q4_K, Q6_K and Q8_0) and the infr
 * landing page ("models": in-shader dequant with dp4a mmq; default quant
 * Q4_K_M; "Per-op device profiling": GEMV and GEMM buckets) spend their
 * decode time in.  Neither page fixes an interface; the calls below follow
 * the problem statement of this library.
 *
 * Conventions shared by every entry point
 *   - Every buffer pointer is a DEVICE pointer owned by the caller; the
 *     library never frees or retains it beyond the call.
 *   - W is row-major by output row: row n holds the K/QK consecutive blocks
 *     of weights W[n, 0..K), QK = 32 (Q8_0) or 256 (Q4_K, Q6_K).  The base
 *     of a weight or block buffer must be 16-byte aligned (GGUF aligns tensor
 *     data to 32 bytes; torch allocations to 256).
 *   - x is row-major [M, K] fp32, y row-major [M, N] fp32; both 4-byte
 *     aligned.  y is overwritten, never accumulated into.
 *   - Status: 0 on success, a negative QMM_E* code otherwise.  All checks
 *     happen before any launch; on error nothing is launched and
 *     qmm_last_error() holds a one-line reason (thread-local).  Nothing
 *     aborts.  Kernels run asynchronously: device-side faults surface at the
 *     caller's next synchronisation, and a bounded device wait that expired
 *     is reported by qmm_device_status().
 *   - Empty problems (M == 0, N == 0, n_elems == 0) are valid and launch
 *     nothing.  K == 0 with M, N > 0 writes y = 0.
 */
#ifndef QMM_H
#define QMM_H

#include <stdint.h>

#if defined(__GNUC__)
#define QMM_API __attribute__((visibility("default")))
#else
#define QMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Weight block formats (this library's own numbering). */
typedef enum {
    QMM_Q8_0 = 0, /* fp16 d | int8 q[32]                         34 B / 32 w  */
    QMM_Q4_K = 1, /* fp16 d | fp16 dmin | 12 B six-bit sc,m | 128 B nibbles
                     w = d*sc*q - dmin*m                        144 B / 256 w */
    QMM_Q6_K = 2, /* 128 B ql | 64 B qh | int8 sc[16] | fp16 d
                     w = d*sc*(q-32)                            210 B / 256 w */
    /* The other K-quants: qmm_dequant only so far (the products return
       QMM_EINVAL_TYPE for them). */
    QMM_Q5_K = 3, /* fp16 d | fp16 dmin | 12 B six-bit sc,m | 32 B fifth bits
                     | 128 B nibbles; w = d*sc*q - dmin*m, q 0..31  176 B / 256 w */
    QMM_Q3_K = 4, /* 32 B high bits | 64 B 2-bit parts | 12 B sixteen six-bit sc
                     | fp16 d; w = d*(sc-32)*q, q -4..3            110 B / 256 w */
    QMM_Q2_K = 5  /* 16 B 4-bit sc,m | 64 B 2-bit quants | fp16 d | fp16 dmin
                     w = d*sc*q - dmin*m, q 0..3                   84 B / 256 w  */
} qmm_type;

/* Status codes. */
enum {
    QMM_OK = 0,
    QMM_EINVAL_TYPE = -1,  /* unknown qmm_type                                */
    QMM_EINVAL_SHAPE = -2, /* negative size, K or n_elems not a block multiple */
    QMM_EINVAL_PTR = -3,   /* null or misaligned pointer for a non-empty call  */
    QMM_ENOMEM = -4,       /* workspace allocation failed                      */
    QMM_ECUDA = -5,        /* CUDA runtime error (detail in qmm_last_error)    */
    QMM_ETIMEOUT = -6      /* a bounded device wait expired (qmm_device_status)*/
};

/*
 * qmm_dequant -- unpack n_elems weights from `blocks` into out_f32[n_elems].
 *   type     : qmm_type of the blocks.
 *   blocks   : device, n_elems/QK consecutive blocks, 16-byte aligned.
 *   n_elems  : number of weights, a multiple of QK (32 or 256).
 *   out_f32  : device, n_elems floats, 16-byte aligned.
 * Each weight is computed with a fixed fp32 order and no FMA contraction:
 *   Q8_0: d*q;  Q4_K, Q5_K, Q2_K: ((d*sc)*q) - (dmin*m);  Q6_K: (d*sc)*(q-32);
 *   Q3_K: (d*(sc-32))*q,
 * so the result is bit-for-bit reproducible.  Runs asynchronously on the
 * legacy default stream (the call has no stream argument).
 */
QMM_API int qmm_dequant(int type, const void *blocks, int64_t n_elems, float *out_f32);

/*
 * qmm -- y[M,N] = W[N,K] . x[M,K]^T with the activations quantised to int8
 * in blocks of 32 (Q8_1 style: fp32 scale max|x|/127, round half away from
 * zero, block sum), exact int32 per-block dot products, fp32 scaling (the
 * prefill with K a multiple of 256 instead contracts the dequantised weights
 * and activations, each rounded to fp16, with fp32 accumulation on the
 * tcgen05 tensor cores: sm_103a has no integer tcgen05 mode).
 *   type     : qmm_type of W: QMM_Q8_0, QMM_Q4_K or QMM_Q6_K.
 *   W_blocks : device, N*(K/QK) blocks, row-major by output row, 16-B aligned.
 *   N, K     : output rows and reduction length; K a multiple of QK.
 *   x        : device, M*K floats row-major (the activations).
 *   M        : activation rows.  M <= 8 runs the decode GEMV (weights
 *              streamed once through shared memory by bulk async copies;
 *              dp4a dot products, or for Q4_K / Q6_K from M = 3 mma.sync on
 *              sixteen weight rows at a time, fp16 operands and fp32
 *              accumulation); M > 8 runs the prefill GEMM.
 *   y        : device, M*N floats, overwritten.
 *   stream   : cudaStream_t to run on (NULL = legacy default stream).
 * Accuracy: |y - y_exact| <= 2e-3 * sum_k |w_k * xhat_k| + 1e-5, where
 * y_exact is the f64 result of the same quantised arithmetic.
 * Decode launches use programmatic dependent launch: they start streaming W
 * while the preceding kernel of this library on the stream finishes (x is
 * read only after it completes), which is safe because no kernel of this
 * library writes block data.
 * The call uses a library-owned device workspace per (device, stream) for
 * the quantised activations.  It is allocated, or grown, on the first call
 * that needs it, so make one call of the largest M*K on a stream before
 * capturing that stream into a CUDA graph.  Calls on one stream are ordered;
 * calls on different streams use different workspaces.
 */
QMM_API int qmm(int type, const void *W_blocks, int64_t N, int64_t K, const float *x, int64_t M,
        float *y, void *stream);

/*
 * qmm_group -- several products that read the same activations:
 *   y_i[M,N_i] = W_i[N_i,K] . x[M,K]^T for i < n, each as
 *   qmm(types[i], Ws[i], Ns[i], K, x, M, ys[i], stream).
 * (An attention layer's q, k and v projections read one x, as do an MLP's
 * gate and up; the infr page runs gate and up of an expert as one op.)
 *   n          : 1 <= n <= QMM_GROUP_MAX.
 *   types, Ws, Ns, ys : HOST arrays of n entries; the types may differ; every
 *                W 16-byte aligned, K a multiple of every type's QK; an entry
 *                with N = 0 is skipped.
 *   K, x, M, stream : shared by all entries, as in qmm().
 * When every entry takes one of the one-weight-stream decode kernels (the
 * row-per-lane one for Q4_K and Q6_K, the block-per-lane one for Q8_0, Q4_K
 * and Q6_K; M <= 2, see qmm_set_decode_path) the whole group is ONE launch of
 * that kernel: its CTAs are split between the matrices in proportion to
 * their weight bytes and each quantises x itself.
 * When every entry takes the tensor-core decode kernel (Q4_K / Q6_K, up to
 * M = 8) x is quantised once and the matrices share one decode launch (its
 * CTAs split by weight bytes).
 * Otherwise the products run one after another as qmm() calls.  Accuracy as
 * qmm().
 * Every entry is validated before anything is launched; errors as qmm(),
 * QMM_EINVAL_SHAPE for n out of range, QMM_EINVAL_PTR for a null array.
 */
#define QMM_GROUP_MAX 8
QMM_API int qmm_group(int n, const int *types, const void *const *Ws, const int64_t *Ns, int64_t K,
                      const float *x, int64_t M, float *const *ys, void *stream);

/*
 * qmm_quantize_act -- the activation quantiser on its own (test hook and
 * building block): for each row of x[M,K] and each block b of 32,
 *   d[m,b] = max|x|/127, q = round_half_away(x * (1/d)) (0 when d == 0),
 *   s[m,b] = sum of the 32 q as int32.
 *   x : device [M,K] fp32; q : device [M,K] int8; d : device [M,K/32] fp32;
 *   s : device [M,K/32] int32.  K must be a multiple of 32.
 * Bit-for-bit reproducible (IEEE division, separately rounded multiply).
 */
QMM_API int qmm_quantize_act(const float *x, int64_t M, int64_t K, int8_t *q, float *d, int32_t *s,
                     void *stream);

/*
 * qmm_noalloc -- the same product as qmm(), for callers that cannot let the
 * library allocate device memory: serving loops that hold all device memory
 * in their own fixed pool (a cudaMalloc by the library would fall outside
 * that budget, and can fail once the pool has taken the rest), and loops
 * that must not stall on cudaFree, which waits for the whole device.  The
 * pages have no counterpart of this call; it is part of this library's
 * interface only.
 *   Arguments, layouts and accuracy as for qmm().  Every M takes the prefill
 *   path (activation quantiser + integer mma.sync GEMM, exact int32 block
 *   dots), whose quantised activations live in a 16 MiB scratch array
 *   compiled into the library: it needs
 *   align256(M*K) + 2*align256(4*M*ceil4(K/32)) bytes, so about
 *   M*K <= 13.4 million; larger calls (and K > 2^24, N > 2^31) return
 *   QMM_EINVAL_SHAPE and launch nothing.
 *   Nothing is allocated by the call (no cudaMalloc, no cudaFree, no
 *   allocating library routine).  The scratch is reserved on every GPU that
 *   loads the library, until the process exits.  The first call on a device
 *   looks the scratch's device address up with cudaGetSymbolAddress while
 *   that device is current; make that first call before any stream capture.
 *   All calls share the one scratch array, which keeps the last call's
 *   contents; each call overwrites every part it reads.  Calls whose kernels
 *   overlap on the GPU (different streams, no ordering between them) race on
 *   it and must be serialised by the caller.  Two kernel launches per call.
 */
QMM_API int qmm_noalloc(int type, const void *W_blocks, int64_t N, int64_t K, const float *x,
                        int64_t M, float *y, void *stream);

/*
 * qmm_t -- y[h][m][k] = sum_n x[h][m][n] * w[h][n][k]: H independent products
 * with the transposed weight matrices, the value side of attention over a KV
 * cache kept as q8_0 (infr landing page, "why > Paged experts, spillable KV":
 * the KV cache can be stored as q8_0).  Matrix h holds N rows (cached
 * positions) of K weights (head_dim); x[h] holds the M probability rows of
 * the query heads that share it.  The score side, x . w^T over the key cache,
 * is qmm itself (one call per cache head, N = positions, K = head_dim).
 *   type     : QMM_Q8_0 (other types: QMM_EINVAL_TYPE).
 *   W_blocks : device, H*N*(K/32) blocks, matrix-major then row-major, 16-B aligned.
 *   H        : matrices, 0 <= H <= 65535.
 *   N        : rows per matrix (>= 0; N = 0 writes y = 0).
 *   K        : weights per row, a multiple of 32, at most 256.
 *   x        : device, H*M*N floats ([H][M][N]), 4-byte aligned; not quantised.
 *   M        : rows of x per matrix (>= 0).
 *   y        : device, H*M*K floats ([H][M][K]), overwritten.
 *   stream   : cudaStream_t to run on (NULL = legacy default stream).
 * The cache rows are streamed once through shared memory and contracted on
 * the tensor cores: each weight d*q enters as fp16 (one rounding of the exact
 * value) and each x scaled by a power of two as fp16 (one rounding), products
 * summed in fp32 in a fixed order, so the result is bitwise reproducible and
 * |y - y_exact| <= 2e-3 * sum_n |x w| + 1e-5 with y_exact the f64 product of
 * x and qmm_dequant's weights.  Uses the per-(device, stream) workspace of
 * qmm (about H*16*K*4 bytes per SM-sized chunk) and H counters per (device,
 * stream); one kernel launch per 16 rows of x.
 */
QMM_API int qmm_t(int type, const void *W_blocks, int64_t H, int64_t N, int64_t K, const float *x, int64_t M,
                  float *y, void *stream);

/*
 * qmm_gate_up -- the gated MLP product of one step:
 *   h[M,N] = silu(W_gate . x^T) * (W_up . x^T),  silu(v) = v / (1 + e^-v),
 * the two products as qmm() (the same quantised x) and the SiLU between
 * them; the infr landing page runs an expert's gate and up as one dispatch
 * ("why > Per-op device profiling": expert_gateup) and its Qwen3 / Llama
 * MLPs apply the SiLU there.
 *   type_gate, W_gate, type_up, W_up : the two matrices, N x K each, as in
 *              qmm() (the types may differ; K a multiple of both QK).
 *   N, K, x, M, stream : as in qmm().
 *   h        : device, M*N floats, overwritten.
 * Launches: M <= 2 with one type for both on the block-per-lane decode
 * kernel is ONE launch (each CTA streams the same rows of both matrices and
 * writes h); on the tensor-core decode (Q4_K / Q6_K, 3 <= M <= 8) x is
 * quantised once and the up launch applies the SiLU to the gate launch's
 * result (three launches); every other case runs the two products, then an
 * elementwise kernel.  The last two use a per-(device, stream) buffer of the
 * library for g (and u), grown on demand like qmm()'s workspace.
 * Accuracy: with e = 2e-3 * sum_k |w_k xhat_k| + 1e-5 the bound of each
 * product, |h - h_exact| <= 1.1 |u| e_gate + |silu(g)| e_up + 1.1 e_gate e_up
 * (|silu'| < 1.1).  Errors as qmm().
 */
QMM_API int qmm_gate_up(int type_gate, const void *W_gate, int type_up, const void *W_up, int64_t N, int64_t K,
                        const float *x, int64_t M, float *h, void *stream);

/* Name of a status code. */
QMM_API const char *qmm_strerror(int status);

/* Detail of the last error raised on the calling thread ("" if none). */
QMM_API const char *qmm_last_error(void);

/*
 * qmm_device_status -- synchronise `stream` and report whether any kernel of
 * this library on the current device gave up on a bounded wait since the
 * last call (QMM_ETIMEOUT; the flag is then cleared), or QMM_ECUDA if the
 * synchronisation itself failed.
 */
QMM_API int qmm_device_status(void *stream);

/* Free every workspace of the library on the current device (synchronises
 * the device first).  Later calls allocate again. */
QMM_API int qmm_release(void);

/* Number of kernel launches this library issued on the calling process
 * since it was loaded (for launch accounting in benchmarks). */
QMM_API int64_t qmm_launch_count(void);

/*
 * qmm_set_decode_path -- which kernel qmm() and qmm_group() use for the
 * decode product (M <= 8), process-wide, for every later call:
 *   QMM_DECODE_AUTO   : chosen by type and M (default).  Q4_K and Q6_K with
 *                       QMM_TENSOR_MIN_M <= M <= 8 run on the tensor-core
 *                       decode kernel (quantiser + mma.sync, two launches;
 *                       not Q6_K with K <= 2048 at M <= 4),
 *                       Q4_K with M <= 2 and Q5_K, Q3_K and Q2_K with
 *                       M <= 8 on the row-per-lane dp4a kernel (one weight
 *                       row per lane) where its copy sizes suit the shape
 *                       (from M = 2 on always for Q5_K, Q3_K and Q2_K),
 *                       everything else on the block-per-lane dp4a kernel;
 *                       a product that no decode kernel holds (x too large
 *                       for shared memory), and a Q8_0 product with
 *                       QMM_TENSOR_MIN_M <= M <= 8 of at least 2^24 weights
 *                       (3 * 2^24 at M <= 4), on the prefill kernel.
 *   QMM_DECODE_BLOCK  : the block-per-lane kernel wherever it fits.
 *   QMM_DECODE_TENSOR : the tensor-core kernel for every Q4_K / Q6_K product
 *                       with 2 <= M <= 8 that fits it (Q6_K: K a multiple
 *                       of 512); M = 1 as with QMM_DECODE_AUTO.
 *   QMM_DECODE_ROWS   : the row-per-lane kernel for every product it takes
 *                       (Q4_K, Q5_K, Q6_K, Q3_K and Q2_K with M <= 8 when
 *                       the activations fit), else as QMM_DECODE_AUTO.
 * Results of the paths agree within the accuracy bound of qmm(), not bit
 * for bit.  Returns the previous path, or QMM_EINVAL_SHAPE for an unknown
 * value (nothing changes).  Needs no GPU.
 */
#define QMM_DECODE_AUTO 0
#define QMM_DECODE_BLOCK 1
#define QMM_DECODE_TENSOR 2
#define QMM_DECODE_ROWS 3
#define QMM_TENSOR_MIN_M 3
QMM_API int qmm_set_decode_path(int path);

/*
 * qmm_set_prefill_path -- which kernel qmm() and qmm_group() use for the
 * prefill product (M > 8), process-wide, for every later call:
 *   QMM_PREFILL_AUTO : the tcgen05 kernel (fp16 operands, fp32 accumulation
 *                      in tensor memory) when K is a multiple of 256, else
 *                      the int8 mma.sync kernel (default).
 *   QMM_PREFILL_INT8 : the int8 mma.sync kernel for every shape: exact int32
 *                      block dots as in the decode kernels, fp32 scaling.
 * Both stay within the accuracy bound of qmm().  Returns the previous path,
 * or QMM_EINVAL_SHAPE for an unknown value (nothing changes).  Needs no GPU.
 */
#define QMM_PREFILL_AUTO 0
#define QMM_PREFILL_INT8 1
QMM_API int qmm_set_prefill_path(int path);

/*
 * qmm_inject_stall -- test hook for failure detection (no counterpart in
 * the pages).  The next `launches` launches of the weight-streaming product
 * kernels (block-per-lane and tensor-core decode, tcgen05 prefill) are
 * launched with their first CTA's weight producer stopping after its first
 * stage, so a consumer's bounded wait (about 2^31 SM cycles, one second at
 * full clock) expires: the kernel records the timeout in the device status
 * word, stops, waits for the copies it did issue, releases its tensor memory
 * and returns.  That call returns QMM_OK with y incomplete, and the next
 * qmm_device_status() reports QMM_ETIMEOUT; later calls run normally.  No
 * fault, trap or unbounded wait is involved.  launches >= 0 (0 cancels);
 * returns the previous pending count, or QMM_EINVAL_SHAPE.  Needs no GPU.
 */
QMM_API int qmm_inject_stall(int launches);

#ifdef __cplusplus
}
#endif

#endif /* QMM_H */
