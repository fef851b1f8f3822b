// dequant.cu -- the super-block unpacker: GGUF blocks -> fp32 weights.
//
// Weights per the block formats of the library's problem statement, with the
// GGUF bit order for the packed fields, and a fixed fp32 operation order with
// no FMA contraction (explicit __fmul_rn / __fsub_rn):
//   Q8_0 : w = d*q
//   Q4_K : w = ((d*sc)*q) - (dmin*m)      (sc, m: six-bit, from 12 bytes)
//   Q6_K : w = (d*sc)*(q-32)              (q: 4 low bits from ql, 2 from qh)
//   Q5_K : as Q4_K, q with a fifth bit    (0..31)
//   Q3_K : w = (d*(sc-32))*q              (q: 2 low bits and a high bit, -4..3)
//   Q2_K : w = ((d*sc)*q) - (dmin*m)      (sc, m: four-bit, per 16 weights)
//
// Work split: a warp produces 128 consecutive weights per step (lane i the
// four weights 4i..4i+3, one 16-byte store), so the fp32 output -- four to
// seven times the bytes read -- is written fully coalesced.
#include "qmm_device.cuh"

#include <type_traits>

namespace qk {

// Q4_K six-bit scale and min of sub-block j from the 12 scale bytes S.
__device__ __forceinline__ void q4k_scale_min(const uint8_t *S, int j, int &sc, int &m) {
    if (j < 4) {
        sc = S[j] & 63;
        m = S[j + 4] & 63;
    } else {
        sc = (S[j + 4] & 15) | ((S[j - 4] >> 6) << 4);
        m = (S[j + 4] >> 4) | ((S[j] >> 6) << 4);
    }
}

template <int T>
__device__ __forceinline__ void dequant4(const uint8_t *__restrict__ blocks, int64_t p, float4 &o);

// Q8_0: weights p..p+3 lie in one block (p is a multiple of 4).
template <>
__device__ __forceinline__ void dequant4<QMM_Q8_0>(const uint8_t *__restrict__ blocks, int64_t p,
                                                   float4 &o) {
    const uint8_t *B = blocks + (p >> 5) * 34;
    const int i = static_cast<int>(p & 31);
    const float d = half_bits_to_float(B[0] | (B[1] << 8));
    const uint8_t *q = B + 2 + i;
    o.x = __fmul_rn(d, static_cast<float>(static_cast<int8_t>(q[0])));
    o.y = __fmul_rn(d, static_cast<float>(static_cast<int8_t>(q[1])));
    o.z = __fmul_rn(d, static_cast<float>(static_cast<int8_t>(q[2])));
    o.w = __fmul_rn(d, static_cast<float>(static_cast<int8_t>(q[3])));
}

// Q4_K: weight position r = p mod 256; chunk c = r/64 holds sub-blocks 2c
// (low nibbles of qs[32c..32c+31]) and 2c+1 (high nibbles).
template <>
__device__ __forceinline__ void dequant4<QMM_Q4_K>(const uint8_t *__restrict__ blocks, int64_t p,
                                                   float4 &o) {
    const uint8_t *B = blocks + (p >> 8) * 144;
    const int r = static_cast<int>(p & 255);
    const int j = r >> 5, c = r >> 6, l = r & 31;
    const uint32_t hdr = *reinterpret_cast<const uint32_t *>(B);
    const float d = half_bits_to_float(hdr), dmin = half_bits_to_float(hdr >> 16);
    int sc, m;
    q4k_scale_min(B + 4, j, sc, m);
    uint32_t qw = *reinterpret_cast<const uint32_t *>(B + 16 + 32 * c + l);
    if (j & 1) qw >>= 4;
    const float t1 = __fmul_rn(d, static_cast<float>(sc));
    const float t3 = __fmul_rn(dmin, static_cast<float>(m));
    o.x = __fsub_rn(__fmul_rn(t1, static_cast<float>(qw & 15)), t3);
    o.y = __fsub_rn(__fmul_rn(t1, static_cast<float>((qw >> 8) & 15)), t3);
    o.z = __fsub_rn(__fmul_rn(t1, static_cast<float>((qw >> 16) & 15)), t3);
    o.w = __fsub_rn(__fmul_rn(t1, static_cast<float>((qw >> 24) & 15)), t3);
}

// Q6_K: weight position r = 128h + 32g + l takes its low four bits from
// ql[64h + l + 32(g&1)] (low nibble for g<2, high for g>=2) and its high two
// bits from (qh[32h + l] >> 2g) & 3; scale index r/16.
template <>
__device__ __forceinline__ void dequant4<QMM_Q6_K>(const uint8_t *__restrict__ blocks, int64_t p,
                                                   float4 &o) {
    const uint8_t *B = blocks + (p >> 8) * 210;
    const int r = static_cast<int>(p & 255);
    const int h = r >> 7, g = (r >> 5) & 3, l = r & 31;
    const float d = half_bits_to_float(B[208] | (B[209] << 8));
    const float t1 = __fmul_rn(d, static_cast<float>(static_cast<int8_t>(B[192 + (r >> 4)])));
    const uint8_t *ql = B + 64 * h + l + 32 * (g & 1);
    const uint8_t *qh = B + 128 + 32 * h + l;
    const int lsh = (g >= 2) ? 4 : 0, hsh = 2 * g;
    float v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int q = ((ql[e] >> lsh) & 15) | (((qh[e] >> hsh) & 3) << 4);
        v[e] = __fmul_rn(t1, static_cast<float>(q - 32));
    }
    o = make_float4(v[0], v[1], v[2], v[3]);
}

// Q5_K: the Q4_K fields (scales at 4, nibbles at 48 + 32c) plus the fifth
// bit of weight r, bit r/32 of qh[r mod 32] (qh at 16).
template <>
__device__ __forceinline__ void dequant4<QMM_Q5_K>(const uint8_t *__restrict__ blocks, int64_t p,
                                                   float4 &o) {
    const uint8_t *B = blocks + (p >> 8) * 176;
    const int r = static_cast<int>(p & 255);
    const int j = r >> 5, c = r >> 6, l = r & 31;
    const uint32_t hdr = *reinterpret_cast<const uint32_t *>(B);
    const float d = half_bits_to_float(hdr), dmin = half_bits_to_float(hdr >> 16);
    int sc, m;
    q4k_scale_min(B + 4, j, sc, m);
    uint32_t qw = *reinterpret_cast<const uint32_t *>(B + 48 + 32 * c + l);
    if (j & 1) qw >>= 4;
    const uint32_t hb = *reinterpret_cast<const uint32_t *>(B + 16 + l) >> j;  // bit j of bytes l..l+3
    const float t1 = __fmul_rn(d, static_cast<float>(sc));
    const float t3 = __fmul_rn(dmin, static_cast<float>(m));
    float v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int q = static_cast<int>(((qw >> (8 * e)) & 15) | (((hb >> (8 * e)) & 1) << 4));
        v[e] = __fsub_rn(__fmul_rn(t1, static_cast<float>(q)), t3);
    }
    o = make_float4(v[0], v[1], v[2], v[3]);
}

// Q3_K (110-byte blocks: only 2-byte aligned, so bytes are read one by one):
// weight r = 128h + 32j + l takes its low two bits from (qs[32h + l] >> 2j)
// and its high bit from bit 4h + j of hmask[l] (q = low - 4 when clear);
// scale i = r/16 is six bits: a nibble of S[k] or S[4+k] (k = i mod 4) and
// the pair (S[8+k] >> 2(i/4)) & 3, offset by 32.
template <>
__device__ __forceinline__ void dequant4<QMM_Q3_K>(const uint8_t *__restrict__ blocks, int64_t p,
                                                   float4 &o) {
    const uint8_t *B = blocks + (p >> 8) * 110;
    const int r = static_cast<int>(p & 255);
    const int h = r >> 7, j = (r >> 5) & 3, l = r & 31, i = r >> 4;
    const uint8_t *S = B + 96;
    const int k = i & 3, G = i >> 2;
    const int lo = (G == 0) ? (S[k] & 15) : (G == 1) ? (S[4 + k] & 15) : (G == 2) ? (S[k] >> 4) : (S[4 + k] >> 4);
    const int sc = (lo | (((S[8 + k] >> (2 * G)) & 3) << 4)) - 32;
    const float d = half_bits_to_float(B[108] | (B[109] << 8));
    const float t1 = __fmul_rn(d, static_cast<float>(sc));
    float v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int low = (B[32 + 32 * h + l + e] >> (2 * j)) & 3;
        const int bit = (B[l + e] >> (4 * h + j)) & 1;
        v[e] = __fmul_rn(t1, static_cast<float>(bit ? low : low - 4));
    }
    o = make_float4(v[0], v[1], v[2], v[3]);
}

// Q2_K: weight r = 128h + 32j + l is (qs[32h + l] >> 2j) & 3 (qs at 16) with
// the four-bit scale and min of sub-block r/16 (byte r/16); d, dmin at 80.
template <>
__device__ __forceinline__ void dequant4<QMM_Q2_K>(const uint8_t *__restrict__ blocks, int64_t p,
                                                   float4 &o) {
    const uint8_t *B = blocks + (p >> 8) * 84;
    const int r = static_cast<int>(p & 255);
    const int h = r >> 7, j = (r >> 5) & 3, l = r & 31;
    const int sm = B[r >> 4];
    const uint32_t hdr = *reinterpret_cast<const uint32_t *>(B + 80);
    const float d = half_bits_to_float(hdr), dmin = half_bits_to_float(hdr >> 16);
    const uint32_t qw = *reinterpret_cast<const uint32_t *>(B + 16 + 32 * h + l) >> (2 * j);
    const float t1 = __fmul_rn(d, static_cast<float>(sm & 15));
    const float t3 = __fmul_rn(dmin, static_cast<float>(sm >> 4));
    float v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
        v[e] = __fsub_rn(__fmul_rn(t1, static_cast<float>((qw >> (8 * e)) & 3)), t3);
    o = make_float4(v[0], v[1], v[2], v[3]);
}

template <int T>
__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t *__restrict__ blocks,
                                                      int64_t n_elems, float *__restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int64_t ngroups = (n_elems + 127) >> 7;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t g = warp; g < ngroups; g += nwarps) {
        const int64_t p = (g << 7) + 4 * lane;
        if (p < n_elems) {
            float4 o;
            dequant4<T>(blocks, p, o);
            __stcs(reinterpret_cast<float4 *>(out + p), o);
        }
    }
}

cudaError_t launch_dequant(int type, const void *blocks, int64_t n_elems, float *out,
                           cudaStream_t st, int num_sms) {
    const int64_t ngroups = (n_elems + 127) / 128;
    int64_t grid = (ngroups + 7) / 8;
    const int64_t cap = static_cast<int64_t>(num_sms) * 32;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    const auto *b = static_cast<const uint8_t *>(blocks);
    const unsigned gx = static_cast<unsigned>(grid);
    auto run = [&](auto t) {
        constexpr int T = decltype(t)::value;
        prefer_max_shared(dequant_kernel<T>);
        dequant_kernel<T><<<gx, 256, 0, st>>>(b, n_elems, out);
    };
    switch (type) {
    case QMM_Q8_0: run(std::integral_constant<int, QMM_Q8_0>{}); break;
    case QMM_Q4_K: run(std::integral_constant<int, QMM_Q4_K>{}); break;
    case QMM_Q5_K: run(std::integral_constant<int, QMM_Q5_K>{}); break;
    case QMM_Q3_K: run(std::integral_constant<int, QMM_Q3_K>{}); break;
    case QMM_Q2_K: run(std::integral_constant<int, QMM_Q2_K>{}); break;
    default: run(std::integral_constant<int, QMM_Q6_K>{}); break;
    }
    return cudaGetLastError();
}

}  // namespace qk
