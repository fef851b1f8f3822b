/*
 * qmm_oracle.c -- plain, slow, obviously-correct CPU oracle for the
 * quantized-weight matrix product y = W.x over GGUF block formats
 * (Q8_0, Q4_K, Q6_K; Q4_K_M mixes Q4_K and Q6_K).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * execute this file; only tests/, the smoke check and the CPU-baseline leg of
 * the benchmark use it.  It shares no code, header, table or helper with the
 * CUDA library.
 *
 * Source of the method: the blazr README ("Model Formats > GGUF": CUDA dp4a
 * kernels for Q4_K, Q6_K, Q8_0; CPU kernels for all formats) and the infr
 * landing page ("why > Vulkan-first, Metal too": a CPU reference backend that
 * GPU output is checked against; default quant Q4_K_M).  Neither page gives
 * the block layouts, so they are taken from the problem statement of this
 * library:
 *   Q8_0 : fp16 d + 32 int8                        (34 B / 32 weights)
 *   Q4_K : fp16 d, fp16 dmin, 12 B of eight 6-bit scales and eight 6-bit mins,
 *          128 B of 4-bit quants                   (144 B / 256 weights)
 *          w = d*sc*q - dmin*m
 *   Q6_K : 128 B low nibbles, 64 B high 2-bit pairs, 16 int8 scales, fp16 d
 *                                                  (210 B / 256 weights)
 *          w = d*sc*(q-32)
 *   activations: Q8_1-style int8 blocks of 32, fp32 scale = max|x|/127,
 *          round half away from zero, plus the block sum.
 * Readings where the statement is silent (bit order inside the 12 scale bytes,
 * nibble order of the quants, fp32 operation order) follow the GGUF
 * convention and are listed in the design notes.
 *
 * Compile with -ffp-contract=off and without -ffast-math: every fp32 step is
 * a separately rounded IEEE-754 operation.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_Q8_0 = 0, OR_Q4_K = 1, OR_Q6_K = 2, OR_Q5_K = 3, OR_Q3_K = 4, OR_Q2_K = 5 };

/* ----------------------------------------------------------------------- */
/* binary16 -> binary32, from the IEEE-754 bit definition (sign, 5-bit      */
/* exponent with bias 15, 10-bit fraction; subnormals are frac * 2^-24).    */
/* The conversion is exact for every finite input.                          */
/* ----------------------------------------------------------------------- */
float oracle_half_to_float(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    float mag;
    if (e == 0)
        mag = ldexpf((float)f, -24);
    else if (e == 31)
        mag = f ? NAN : INFINITY;
    else
        mag = ldexpf((float)(f + 1024), e - 25);
    return sign ? -mag : mag;
}

static uint16_t rd16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static void wr16(uint8_t *p, uint16_t v) { p[0] = (uint8_t)(v & 0xff); p[1] = (uint8_t)(v >> 8); }

int oracle_block_bytes(int type)
{
    switch (type) {
    case OR_Q8_0: return 34;
    case OR_Q4_K: return 144;
    case OR_Q6_K: return 210;
    case OR_Q5_K: return 176;
    case OR_Q3_K: return 110;
    case OR_Q2_K: return 84;
    default: return -1;
    }
}

int oracle_block_weights(int type)
{
    switch (type) {
    case OR_Q8_0: return 32;
    case OR_Q4_K: return 256;
    case OR_Q6_K: return 256;
    case OR_Q5_K: return 256;
    case OR_Q3_K: return 256;
    case OR_Q2_K: return 256;
    default: return -1;
    }
}

/* ----------------------------------------------------------------------- */
/* Q8_0: bytes [0,2) fp16 d, [2,34) int8 q[32].                             */
/* ----------------------------------------------------------------------- */
void oracle_unpack_q8_0(const uint8_t *blk, uint16_t *d_bits, int8_t q[32])
{
    *d_bits = rd16(blk);
    for (int i = 0; i < 32; ++i)
        q[i] = (int8_t)blk[2 + i];
}

void oracle_pack_q8_0(uint16_t d_bits, const int8_t q[32], uint8_t *blk)
{
    wr16(blk, d_bits);
    for (int i = 0; i < 32; ++i)
        blk[2 + i] = (uint8_t)q[i];
}

/* ----------------------------------------------------------------------- */
/* Q4_K: [0,2) d, [2,4) dmin, [4,16) scale bytes S[12], [16,144) qs[128].   */
/* Eight sub-blocks j of 32 weights; sub-block j has 6-bit scale sc[j] and  */
/* 6-bit min m[j].  Scale bytes (GGUF convention):                          */
/*   j < 4 : sc[j] = S[j] & 63,      m[j] = S[j+4] & 63                     */
/*   j >= 4: sc[j] = (S[j+4] & 15) | (S[j-4] >> 6) << 4                     */
/*           m[j]  = (S[j+4] >> 4) | (S[j]   >> 6) << 4                     */
/* Quants: for chunk c = 0..3 and l = 0..31, byte qs[32c+l] holds weight    */
/* 64c+l (sub-block 2c) in its low nibble and weight 64c+32+l (sub-block    */
/* 2c+1) in its high nibble.                                                */
/* ----------------------------------------------------------------------- */
void oracle_unpack_q4_k(const uint8_t *blk, uint16_t *d_bits, uint16_t *dmin_bits,
                        uint8_t sc[8], uint8_t m[8], uint8_t q[256])
{
    const uint8_t *S = blk + 4;
    const uint8_t *qs = blk + 16;
    *d_bits = rd16(blk);
    *dmin_bits = rd16(blk + 2);
    for (int j = 0; j < 8; ++j) {
        if (j < 4) {
            sc[j] = S[j] & 63;
            m[j] = S[j + 4] & 63;
        } else {
            sc[j] = (uint8_t)((S[j + 4] & 15) | ((S[j - 4] >> 6) << 4));
            m[j] = (uint8_t)((S[j + 4] >> 4) | ((S[j] >> 6) << 4));
        }
    }
    for (int c = 0; c < 4; ++c)
        for (int l = 0; l < 32; ++l) {
            q[64 * c + l] = qs[32 * c + l] & 15;
            q[64 * c + 32 + l] = qs[32 * c + l] >> 4;
        }
}

void oracle_pack_q4_k(uint16_t d_bits, uint16_t dmin_bits, const uint8_t sc[8],
                      const uint8_t m[8], const uint8_t q[256], uint8_t *blk)
{
    uint8_t *S = blk + 4;
    uint8_t *qs = blk + 16;
    wr16(blk, d_bits);
    wr16(blk + 2, dmin_bits);
    for (int j = 0; j < 4; ++j) {
        S[j] = (uint8_t)((sc[j] & 63) | ((sc[j + 4] >> 4) << 6));
        S[j + 4] = (uint8_t)((m[j] & 63) | ((m[j + 4] >> 4) << 6));
        S[j + 8] = (uint8_t)((sc[j + 4] & 15) | ((m[j + 4] & 15) << 4));
    }
    for (int c = 0; c < 4; ++c)
        for (int l = 0; l < 32; ++l)
            qs[32 * c + l] = (uint8_t)((q[64 * c + l] & 15) | ((q[64 * c + 32 + l] & 15) << 4));
}

/* ----------------------------------------------------------------------- */
/* Q6_K: [0,128) ql, [128,192) qh, [192,208) int8 scales[16], [208,210) d.  */
/* Sixteen sub-blocks of 16 weights; weight p uses scale p/16.  Two halves  */
/* h = 0,1 of 128 weights use ql[64h..] and qh[32h..]; inside a half,       */
/* weight 32g+l (g = 0..3, l = 0..31) takes                                 */
/*   low 4 bits  : ql[64h + l + 32(g&1)], low nibble for g<2, high for g>=2 */
/*   high 2 bits : (qh[32h + l] >> 2g) & 3                                  */
/* q = low | high << 4 in 0..63, and the weight is d*sc*(q-32).             */
/* ----------------------------------------------------------------------- */
void oracle_unpack_q6_k(const uint8_t *blk, uint16_t *d_bits, int8_t sc[16], uint8_t q[256])
{
    const uint8_t *ql = blk;
    const uint8_t *qh = blk + 128;
    for (int i = 0; i < 16; ++i)
        sc[i] = (int8_t)blk[192 + i];
    *d_bits = rd16(blk + 208);
    for (int h = 0; h < 2; ++h)
        for (int g = 0; g < 4; ++g)
            for (int l = 0; l < 32; ++l) {
                uint8_t lo = ql[64 * h + l + 32 * (g & 1)];
                lo = (g < 2) ? (uint8_t)(lo & 15) : (uint8_t)(lo >> 4);
                uint8_t hi = (uint8_t)((qh[32 * h + l] >> (2 * g)) & 3);
                q[128 * h + 32 * g + l] = (uint8_t)(lo | (hi << 4));
            }
}

void oracle_pack_q6_k(uint16_t d_bits, const int8_t sc[16], const uint8_t q[256], uint8_t *blk)
{
    uint8_t *ql = blk;
    uint8_t *qh = blk + 128;
    memset(blk, 0, 192);
    for (int h = 0; h < 2; ++h)
        for (int g = 0; g < 4; ++g)
            for (int l = 0; l < 32; ++l) {
                uint8_t v = q[128 * h + 32 * g + l] & 63;
                int li = 64 * h + l + 32 * (g & 1);
                if (g < 2)
                    ql[li] = (uint8_t)(ql[li] | (v & 15));
                else
                    ql[li] = (uint8_t)(ql[li] | ((v & 15) << 4));
                qh[32 * h + l] = (uint8_t)(qh[32 * h + l] | ((v >> 4) << (2 * g)));
            }
    for (int i = 0; i < 16; ++i)
        blk[192 + i] = (uint8_t)sc[i];
    wr16(blk + 208, d_bits);
}

/* ----------------------------------------------------------------------- */
/* Q5_K: [0,2) d, [2,4) dmin, [4,16) scale bytes S[12] (packed as Q4_K's),  */
/* [16,48) qh[32], [48,176) qs[128].  Weight p = 64c + 32s + l (c = 0..3,   */
/* s = 0,1, l = 0..31) is in sub-block j = 2c + s; its low four bits are    */
/* the low (s = 0) or high (s = 1) nibble of qs[32c + l] as in Q4_K, its    */
/* fifth bit is bit j of qh[l]; q = low | fifth << 4 in 0..31 and the       */
/* weight is d*sc[j]*q - dmin*m[j] (GGUF convention, as Q4_K with one more  */
/* bit per quant).                                                          */
/* ----------------------------------------------------------------------- */
void oracle_unpack_q5_k(const uint8_t *blk, uint16_t *d_bits, uint16_t *dmin_bits,
                        uint8_t sc[8], uint8_t m[8], uint8_t q[256])
{
    /* the fields shared with Q4_K: d, dmin, scales; then the two bit planes */
    uint8_t as4[144];
    memcpy(as4, blk, 16);
    memcpy(as4 + 16, blk + 48, 128);
    oracle_unpack_q4_k(as4, d_bits, dmin_bits, sc, m, q);
    const uint8_t *qh = blk + 16;
    for (int p = 0; p < 256; ++p) {
        int j = p / 32, l = p % 32;
        q[p] = (uint8_t)(q[p] | (((qh[l] >> j) & 1) << 4));
    }
}

void oracle_pack_q5_k(uint16_t d_bits, uint16_t dmin_bits, const uint8_t sc[8],
                      const uint8_t m[8], const uint8_t q[256], uint8_t *blk)
{
    uint8_t as4[144], lo[256];
    for (int p = 0; p < 256; ++p)
        lo[p] = (uint8_t)(q[p] & 15);
    oracle_pack_q4_k(d_bits, dmin_bits, sc, m, lo, as4);
    memcpy(blk, as4, 16);
    memcpy(blk + 48, as4 + 16, 128);
    uint8_t *qh = blk + 16;
    memset(qh, 0, 32);
    for (int p = 0; p < 256; ++p) {
        int j = p / 32, l = p % 32;
        qh[l] = (uint8_t)(qh[l] | (((q[p] >> 4) & 1) << j));
    }
}

/* ----------------------------------------------------------------------- */
/* Q3_K: [0,32) hmask, [32,96) qs (2-bit low parts), [96,108) scale bytes   */
/* S[12] (sixteen 6-bit scales), [108,110) d.  Weight p = 128h + 32j + l    */
/* (h = 0,1, j = 0..3, l = 0..31) is in sub-block i = 8h + 2j + (l >= 16)   */
/* of 16 weights; its low two bits are (qs[32h + l] >> 2j) & 3 and its high */
/* bit is bit 4h + j of hmask[l]; q = low - 4 when that bit is clear, else  */
/* low, in -4..3.  Scale i = low nibble | high pair << 4, with k = i mod 4  */
/* and G = i / 4: the low nibble of S[k], S[4+k] for G = 0, 1, the high     */
/* nibble of S[k], S[4+k] for G = 2, 3, and the pair (S[8+k] >> 2G) & 3;    */
/* the weight is d*(sc - 32)*q (GGUF convention).                           */
/* ----------------------------------------------------------------------- */
void oracle_unpack_q3_k(const uint8_t *blk, uint16_t *d_bits, int8_t sc[16], int8_t q[256])
{
    const uint8_t *hm = blk, *qs = blk + 32, *S = blk + 96;
    *d_bits = rd16(blk + 108);
    for (int i = 0; i < 16; ++i) {
        int k = i % 4, G = i / 4;
        int lo = (G == 0) ? (S[k] & 15) : (G == 1) ? (S[4 + k] & 15) : (G == 2) ? (S[k] >> 4) : (S[4 + k] >> 4);
        int hi = (S[8 + k] >> (2 * G)) & 3;
        sc[i] = (int8_t)((lo | (hi << 4)) - 32);
    }
    for (int h = 0; h < 2; ++h)
        for (int j = 0; j < 4; ++j)
            for (int l = 0; l < 32; ++l) {
                int low = (qs[32 * h + l] >> (2 * j)) & 3;
                int bit = (hm[l] >> (4 * h + j)) & 1;
                q[128 * h + 32 * j + l] = (int8_t)(bit ? low : low - 4);
            }
}

/* sc: the signed scales (sc - 32 in -32..31); q in -4..3 */
void oracle_pack_q3_k(uint16_t d_bits, const int8_t sc[16], const int8_t q[256], uint8_t *blk)
{
    uint8_t *hm = blk, *qs = blk + 32, *S = blk + 96;
    memset(blk, 0, 110);
    for (int i = 0; i < 16; ++i) {
        int v = (sc[i] + 32) & 63, k = i % 4, G = i / 4;
        int lo = v & 15, hi = v >> 4;
        if (G == 0) S[k] = (uint8_t)(S[k] | lo);
        else if (G == 1) S[4 + k] = (uint8_t)(S[4 + k] | lo);
        else if (G == 2) S[k] = (uint8_t)(S[k] | (lo << 4));
        else S[4 + k] = (uint8_t)(S[4 + k] | (lo << 4));
        S[8 + k] = (uint8_t)(S[8 + k] | (hi << (2 * G)));
    }
    for (int h = 0; h < 2; ++h)
        for (int j = 0; j < 4; ++j)
            for (int l = 0; l < 32; ++l) {
                int v = q[128 * h + 32 * j + l];  /* -4..3 */
                int bit = v >= 0, low = bit ? v : v + 4;
                qs[32 * h + l] = (uint8_t)(qs[32 * h + l] | (low << (2 * j)));
                hm[l] = (uint8_t)(hm[l] | (bit << (4 * h + j)));
            }
    wr16(blk + 108, d_bits);
}

/* ----------------------------------------------------------------------- */
/* Q2_K: [0,16) scale bytes (sub-block i: scale = low nibble, min = high    */
/* nibble), [16,80) qs (2-bit quants), [80,82) d, [82,84) dmin.  Weight     */
/* p = 128h + 32j + l is in sub-block i = 8h + 2j + (l >= 16); its quant    */
/* is (qs[32h + l] >> 2j) & 3 in 0..3 and the weight d*sc*q - dmin*m (GGUF  */
/* convention).                                                             */
/* ----------------------------------------------------------------------- */
void oracle_unpack_q2_k(const uint8_t *blk, uint16_t *d_bits, uint16_t *dmin_bits, uint8_t sc[16],
                        uint8_t m[16], uint8_t q[256])
{
    const uint8_t *qs = blk + 16;
    for (int i = 0; i < 16; ++i) {
        sc[i] = blk[i] & 15;
        m[i] = blk[i] >> 4;
    }
    *d_bits = rd16(blk + 80);
    *dmin_bits = rd16(blk + 82);
    for (int h = 0; h < 2; ++h)
        for (int j = 0; j < 4; ++j)
            for (int l = 0; l < 32; ++l)
                q[128 * h + 32 * j + l] = (uint8_t)((qs[32 * h + l] >> (2 * j)) & 3);
}

void oracle_pack_q2_k(uint16_t d_bits, uint16_t dmin_bits, const uint8_t sc[16], const uint8_t m[16],
                      const uint8_t q[256], uint8_t *blk)
{
    uint8_t *qs = blk + 16;
    memset(blk, 0, 84);
    for (int i = 0; i < 16; ++i)
        blk[i] = (uint8_t)((sc[i] & 15) | ((m[i] & 15) << 4));
    for (int h = 0; h < 2; ++h)
        for (int j = 0; j < 4; ++j)
            for (int l = 0; l < 32; ++l)
                qs[32 * h + l] = (uint8_t)(qs[32 * h + l] | ((q[128 * h + 32 * j + l] & 3) << (2 * j)));
    wr16(blk + 80, d_bits);
    wr16(blk + 82, dmin_bits);
}

/* ----------------------------------------------------------------------- */
/* Dequantisation of one block into fp32, fixed operation order, no FMA:    */
/*   Q8_0: w = d*q                                                          */
/*   Q4_K, Q5_K: t1 = d*sc, t2 = t1*q, t3 = dmin*m, w = t2 - t3             */
/*   Q6_K: t1 = d*sc, w = t1*(q-32)                                         */
/*   Q3_K: t1 = d*(sc-32), w = t1*q                                         */
/*   Q2_K: t1 = d*sc, t2 = t1*q, t3 = dmin*m, w = t2 - t3 (16-weight sub-blocks) */
/* (the scale products are formed first, reading "d*sc*q - dmin*m" from     */
/* left to right).                                                          */
/* ----------------------------------------------------------------------- */
static void dequant_block(int type, const uint8_t *blk, float *w)
{
    if (type == OR_Q8_0) {
        uint16_t db;
        int8_t q[32];
        oracle_unpack_q8_0(blk, &db, q);
        float d = oracle_half_to_float(db);
        for (int i = 0; i < 32; ++i)
            w[i] = d * (float)q[i];
    } else if (type == OR_Q4_K || type == OR_Q5_K) {
        uint16_t db, dmb;
        uint8_t sc[8], m[8], q[256];
        if (type == OR_Q4_K)
            oracle_unpack_q4_k(blk, &db, &dmb, sc, m, q);
        else
            oracle_unpack_q5_k(blk, &db, &dmb, sc, m, q);
        float d = oracle_half_to_float(db), dmin = oracle_half_to_float(dmb);
        for (int p = 0; p < 256; ++p) {
            int j = p / 32;
            float t1 = d * (float)sc[j];
            float t2 = t1 * (float)q[p];
            float t3 = dmin * (float)m[j];
            w[p] = t2 - t3;
        }
    } else if (type == OR_Q3_K) {
        uint16_t db;
        int8_t sc[16], q[256];
        oracle_unpack_q3_k(blk, &db, sc, q);
        float d = oracle_half_to_float(db);
        for (int p = 0; p < 256; ++p) {
            float t1 = d * (float)sc[p / 16];
            w[p] = t1 * (float)q[p];
        }
    } else if (type == OR_Q2_K) {
        uint16_t db, dmb;
        uint8_t sc[16], m[16], q[256];
        oracle_unpack_q2_k(blk, &db, &dmb, sc, m, q);
        float d = oracle_half_to_float(db), dmin = oracle_half_to_float(dmb);
        for (int p = 0; p < 256; ++p) {
            int i = p / 16;
            float t1 = d * (float)sc[i];
            float t2 = t1 * (float)q[p];
            float t3 = dmin * (float)m[i];
            w[p] = t2 - t3;
        }
    } else {
        uint16_t db;
        int8_t sc[16];
        uint8_t q[256];
        oracle_unpack_q6_k(blk, &db, sc, q);
        float d = oracle_half_to_float(db);
        for (int p = 0; p < 256; ++p) {
            float t1 = d * (float)sc[p / 16];
            w[p] = t1 * (float)((int)q[p] - 32);
        }
    }
}

int oracle_dequant(int type, const uint8_t *blocks, int64_t n_elems, float *out)
{
    int bb = oracle_block_bytes(type), bw = oracle_block_weights(type);
    if (bb < 0) return -1;
    if (n_elems < 0 || n_elems % bw) return -2;
    int64_t nblk = n_elems / bw;
    for (int64_t b = 0; b < nblk; ++b)
        dequant_block(type, blocks + b * bb, out + b * bw);
    return 0;
}

/* ----------------------------------------------------------------------- */
/* Activation quantiser (Q8_1 style).  For each row and each block of 32:   */
/*   amax = max |x_i|,  d = amax / 127,  inv = 1/d (0 when d == 0),         */
/*   q_i = round_half_away_from_zero(x_i * inv) clamped to [-127, 127],     */
/*   s = sum of the q_i as a 32-bit integer.                                */
/* ----------------------------------------------------------------------- */
int oracle_quantize_act(const float *x, int64_t M, int64_t K, int8_t *q, float *d, int32_t *s)
{
    if (M < 0 || K < 0 || K % 32) return -2;
    int64_t nb = K / 32;
    for (int64_t r = 0; r < M; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            const float *xb = x + r * K + b * 32;
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) {
                float a = fabsf(xb[i]);
                if (a > amax) amax = a;
            }
            float db = amax / 127.0f;
            float inv = (db != 0.0f) ? 1.0f / db : 0.0f;
            int32_t sum = 0;
            for (int i = 0; i < 32; ++i) {
                float v = roundf(xb[i] * inv);
                if (v > 127.0f) v = 127.0f;
                if (v < -127.0f) v = -127.0f;
                int8_t qi = (int8_t)v;
                q[r * K + b * 32 + i] = qi;
                sum += qi;
            }
            d[r * nb + b] = db;
            s[r * nb + b] = sum;
        }
    return 0;
}

/* ----------------------------------------------------------------------- */
/* y[m,n] = sum over 32-blocks b of row n, accumulated in f64 in increasing */
/* b, with exact int32 block dots:                                          */
/*   Q8_0: y += dx_b * dw_b * I_b,           I_b = sum q_w q_x              */
/*   Q4_K: y += dx_b * (d*(sc_j*I_b) - dmin*(m_j*s_b)),  j = sub-block of b */
/*   Q6_K: y += dx_b * d * J_b,  J_b = sum over the two 16-sub-blocks a of  */
/*         b of sc_a * sum (q-32) q_x                                       */
/* A[m,n] = sum_k |w_k * xhat_k| in f64, with w the fp32 dequantised weight */
/* and xhat = dx * q_x: the scale of the acceptance bound.                  */
/* ----------------------------------------------------------------------- */
static void qmm_row(int type, const uint8_t *row, int64_t K, const int8_t *xq, const float *xd,
                    const int32_t *xs, int64_t M, int64_t N, int64_t n, double *y, double *A)
{
    int bb = oracle_block_bytes(type), bw = oracle_block_weights(type);
    int64_t nblk = K / bw, nb32 = K / 32;
    float *w = (float *)malloc(sizeof(float) * (size_t)K);
    for (int64_t b = 0; b < nblk; ++b)
        dequant_block(type, row + b * bb, w + b * bw);
    for (int64_t mm = 0; mm < M; ++mm) {
        const int8_t *qx = xq + mm * K;
        const float *dx = xd + mm * nb32;
        const int32_t *sx = xs + mm * nb32;
        double acc = 0.0, a = 0.0;
        for (int64_t blk = 0; blk < nblk; ++blk) {
            const uint8_t *B = row + blk * bb;
            if (type == OR_Q8_0) {
                uint16_t db;
                int8_t q[32];
                oracle_unpack_q8_0(B, &db, q);
                int32_t I = 0;
                for (int i = 0; i < 32; ++i)
                    I += (int32_t)q[i] * (int32_t)qx[blk * 32 + i];
                acc += (double)dx[blk] * (double)oracle_half_to_float(db) * (double)I;
            } else if (type == OR_Q4_K || type == OR_Q5_K) {
                uint16_t db, dmb;
                uint8_t sc[8], m[8], q[256];
                if (type == OR_Q4_K)
                    oracle_unpack_q4_k(B, &db, &dmb, sc, m, q);
                else
                    oracle_unpack_q5_k(B, &db, &dmb, sc, m, q);
                double d = oracle_half_to_float(db), dmin = oracle_half_to_float(dmb);
                for (int j = 0; j < 8; ++j) {
                    int64_t b32 = blk * 8 + j;
                    int32_t I = 0;
                    for (int i = 0; i < 32; ++i)
                        I += (int32_t)q[32 * j + i] * (int32_t)qx[b32 * 32 + i];
                    int32_t scI = (int32_t)sc[j] * I;
                    int32_t ms = (int32_t)m[j] * sx[b32];
                    acc += (double)dx[b32] * (d * (double)scI - dmin * (double)ms);
                }
            } else if (type == OR_Q3_K || type == OR_Q2_K) {
                /* sixteen sub-blocks of 16: exact int32 dots per sub-block */
                int8_t qs3[256], sc3[16];
                uint8_t q2[256], sc2[16], m2[16];
                uint16_t db, dmb = 0;
                if (type == OR_Q3_K)
                    oracle_unpack_q3_k(B, &db, sc3, qs3);
                else
                    oracle_unpack_q2_k(B, &db, &dmb, sc2, m2, q2);
                double d = oracle_half_to_float(db), dmin = oracle_half_to_float(dmb);
                for (int j = 0; j < 8; ++j) {
                    int64_t b32 = blk * 8 + j;
                    int32_t J = 0, Mn = 0;
                    for (int half = 0; half < 2; ++half) {
                        int i16 = 2 * j + half;
                        int32_t I = 0, S = 0;
                        for (int i = 0; i < 16; ++i) {
                            int p = 16 * i16 + i;
                            int32_t qv = (type == OR_Q3_K) ? (int32_t)qs3[p] : (int32_t)q2[p];
                            I += qv * (int32_t)qx[blk * 256 + p];
                            S += (int32_t)qx[blk * 256 + p];
                        }
                        if (type == OR_Q3_K) {
                            J += (int32_t)sc3[i16] * I;
                        } else {
                            J += (int32_t)sc2[i16] * I;
                            Mn += (int32_t)m2[i16] * S;
                        }
                    }
                    acc += (double)dx[b32] * (d * (double)J - dmin * (double)Mn);
                }
            } else {
                uint16_t db;
                int8_t sc[16];
                uint8_t q[256];
                oracle_unpack_q6_k(B, &db, sc, q);
                double d = oracle_half_to_float(db);
                for (int j = 0; j < 8; ++j) {
                    int64_t b32 = blk * 8 + j;
                    int32_t J = 0;
                    for (int half = 0; half < 2; ++half) {
                        int32_t I = 0;
                        for (int i = 0; i < 16; ++i) {
                            int p = 32 * j + 16 * half + i;
                            I += ((int32_t)q[p] - 32) * (int32_t)qx[blk * 256 + p];
                        }
                        J += (int32_t)sc[2 * j + half] * I;
                    }
                    acc += (double)dx[b32] * d * (double)J;
                }
            }
        }
        for (int64_t k = 0; k < K; ++k)
            a += fabs((double)w[k] * ((double)dx[k / 32] * (double)qx[k]));
        y[mm * N + n] = acc;
        if (A) A[mm * N + n] = a;
    }
    free(w);
}

int oracle_qmm(int type, const uint8_t *W, int64_t N, int64_t K, const float *x, int64_t M,
               double *y, double *A, int nthreads)
{
    int bb = oracle_block_bytes(type), bw = oracle_block_weights(type);
    if (bb < 0) return -1;
    if (N < 0 || M < 0 || K <= 0 || K % bw) return -2;
    int64_t nb32 = K / 32;
    int8_t *xq = (int8_t *)malloc((size_t)(M * K) + 1);
    float *xd = (float *)malloc(sizeof(float) * (size_t)(M * nb32) + 4);
    int32_t *xs = (int32_t *)malloc(sizeof(int32_t) * (size_t)(M * nb32) + 4);
    oracle_quantize_act(x, M, K, xq, xd, xs);
    int64_t rb = (K / bw) * bb;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 16) num_threads(nthreads)
#endif
    for (int64_t n = 0; n < N; ++n)
        qmm_row(type, W + n * rb, K, xq, xd, xs, M, N, n, y, A);
    free(xq);
    free(xd);
    free(xs);
    return 0;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
