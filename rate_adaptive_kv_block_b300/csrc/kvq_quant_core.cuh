// The quantizer's arithmetic, shared by kvq_quantize and the fused
// allocate-and-quantize path ("Rate-adaptive KV-cache quantizer", "Key
// formulas": P(q_{i+1} | x) = (x - q_i)/(q_{i+1} - q_i)).
//
// For one block with levels q_0 < ... < q_{k-1} (slots k..15 repeat q_{k-1}):
//   thresholds  T_j = q_j for 1 <= j <= k-2, +inf beyond (binary16 pairs);
//   decision    (-q_i, w_i) with w_i = (q_{i+1} - q_i) 2^-24 (k = 1: w = +inf).
// An entry x gets i = #{j : T_j <= x} and code i + [fl(u w_i) < fl(x - q_i)],
// fp32 round-to-nearest, u = hash >> 8.  hash(seed, n) is word n mod 4 of the
// Philox4x32 block function with 7 rounds (Salmon, Moraes, Dror, Shaw, SC
// 2011) at counter (n >> 2 as two words, 0, 0) and key (seed as two words).
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>
#include <string.h>

namespace kvq {

constexpr int kPhiloxRounds = 7;
constexpr uint32_t kPhiloxM0 = 0xD2511F53u, kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u, kPhiloxW1 = 0xBB67AE85u;

// The round keys of one seed: round r uses (seed_lo + r W0, seed_hi + r W1).
// Passed by value in kernel parameters, so the xors read them from the
// constant bank.
struct PhiloxKey {
    uint32_t k0[kPhiloxRounds], k1[kPhiloxRounds];
};

__host__ __device__ inline PhiloxKey philox_key(uint64_t seed) {
    PhiloxKey K;
    uint32_t a = (uint32_t)seed, b = (uint32_t)(seed >> 32);
    for (int r = 0; r < kPhiloxRounds; ++r) {
        K.k0[r] = a;
        K.k1[r] = b;
        a += kPhiloxW0;
        b += kPhiloxW1;
    }
    return K;
}

// Philox4x32-7 of the counter (c0, c1, 0, 0): round 0 multiplies a zero
// word, so it is one 32 x 32 -> 64-bit product; each later round is two.
__device__ __forceinline__ uint4 philox7(uint32_t c0, uint32_t c1, const PhiloxKey &K) {
    uint64_t p0 = (uint64_t)kPhiloxM0 * c0;
    uint32_t x0 = c1 ^ K.k0[0];
    uint32_t x1 = 0u;
    uint32_t x2 = (uint32_t)(p0 >> 32) ^ K.k1[0];
    uint32_t x3 = (uint32_t)p0;
#pragma unroll
    for (int r = 1; r < kPhiloxRounds; ++r) {
        const uint64_t a = (uint64_t)kPhiloxM0 * x0;
        const uint64_t b = (uint64_t)kPhiloxM1 * x2;
        x0 = (uint32_t)(b >> 32) ^ x1 ^ K.k0[r];
        x1 = (uint32_t)b;
        x2 = (uint32_t)(a >> 32) ^ x3 ^ K.k1[r];
        x3 = (uint32_t)a;
    }
    return make_uint4(x0, x1, x2, x3);
}

// Counter block of global entry n (n a multiple of 4): n >> 2.
__device__ __forceinline__ uint64_t quant_counter(uint64_t index_base, uint64_t flat) {
    return (index_base + flat) >> 2;
}

__device__ __forceinline__ __half2 as_h2(uint32_t u) {
    __half2 h;
    memcpy(&h, &u, 4);
    return h;
}

// Threshold j (0..15) and decision entry j of a block from its 16 codebook
// slots; `k` = number of distinct levels.  NEAREST (the deterministic
// comparator): w_i = q_{i+1} - q_i unscaled.
template <bool NEAREST = false>
__device__ __forceinline__ void quant_table_entry(const float *q, int k, int j, __half2 &thr,
                                                  float2 &qw) {
    const float INF = __int_as_float(0x7f800000);
    const float qj = q[j];
    const float th = (j >= 1 && j <= k - 2) ? qj : INF;
    thr = __floats2half2_rn(th, th);                  // exact: levels are binary16 values
    const float qn = q[j < 15 ? j + 1 : 15];
    float ws = 0.f;
    if (k <= 1) ws = INF;                             // k = 1: never move up
    else if (j <= k - 2)
        ws = NEAREST ? __fsub_rn(qn, qj) : __fmul_rn(__fsub_rn(qn, qj), 5.9604644775390625e-8f);  // 2^-24
    qw = make_float2(-qj, ws);
}

// Codes of 8 consecutive entries (one 16-byte load `raw`) of one block:
// T[1..15] the thresholds as binary16 pairs, qw the decision table, c the
// Philox counter of the first 4 entries (the next 4 use c + 1).  Returns 8
// nibbles, entry e in bits 4e..4e+3.
__device__ __forceinline__ uint32_t quant8(const uint4 raw, const uint32_t (&T)[16],
                                           const float2 *qw, uint64_t c, const PhiloxKey &K) {
    const uint32_t xw0 = raw.x, xw1 = raw.y, xw2 = raw.z, xw3 = raw.w;
    const uint4 ha = philox7((uint32_t)c, (uint32_t)(c >> 32), K);
    const uint64_t c1 = c + 1u;
    const uint4 hb = philox7((uint32_t)c1, (uint32_t)(c1 >> 32), K);
    uint32_t packed = 0;
#pragma unroll
    for (int pr = 0; pr < 4; ++pr) {
        const __half2 X = as_h2(pr == 0 ? xw0 : pr == 1 ? xw1 : pr == 2 ? xw2 : xw3);
        // interval index of both halves: 4-level binary search over T1..T15
        // (sorted, +inf padded); m* are 0xffff-per-half masks
        const uint32_t m1 = __hge2_mask(X, as_h2(T[8]));
        const uint32_t t2 = (T[12] & m1) | (T[4] & ~m1);
        const uint32_t m2 = __hge2_mask(X, as_h2(t2));
        const uint32_t a3 = (T[6] & m2) | (T[2] & ~m2), b3 = (T[14] & m2) | (T[10] & ~m2);
        const uint32_t t3 = (b3 & m1) | (a3 & ~m1);
        const uint32_t m3 = __hge2_mask(X, as_h2(t3));
        const uint32_t a4 = (T[3] & m3) | (T[1] & ~m3), b4 = (T[7] & m3) | (T[5] & ~m3);
        const uint32_t c4 = (T[11] & m3) | (T[9] & ~m3), d4 = (T[15] & m3) | (T[13] & ~m3);
        const uint32_t lo4 = (b4 & m2) | (a4 & ~m2), hi4 = (d4 & m2) | (c4 & ~m2);
        const uint32_t t4 = (hi4 & m1) | (lo4 & ~m1);
        const uint32_t m4 = __hge2_mask(X, as_h2(t4));
        const uint32_t idx = (m1 & 0x00080008u) | (m2 & 0x00040004u) | (m3 & 0x00020002u) |
                             (m4 & 0x00010001u);
        const int i0 = (int)(idx & 15u), i1 = (int)(idx >> 16);
        const float2 e0 = qw[i0], e1 = qw[i1];
        const uint32_t h0 = pr == 0 ? ha.x : pr == 1 ? ha.z : pr == 2 ? hb.x : hb.z;
        const uint32_t h1 = pr == 0 ? ha.y : pr == 1 ? ha.w : pr == 2 ? hb.y : hb.w;
        const float2 xf = __half22float2(X);
        const float2 r = __fadd2_rn(xf, make_float2(e0.x, e1.x));          // x - q_i
        const float2 u = make_float2((float)(h0 >> 8), (float)(h1 >> 8));
        const float2 tw = __fmul2_rn(u, make_float2(e0.y, e1.y));
        const uint32_t c0 = (uint32_t)i0 + (tw.x < r.x ? 1u : 0u);
        const uint32_t cc1 = (uint32_t)i1 + (tw.y < r.y ? 1u : 0u);
        packed |= (c0 | (cc1 << 4)) << (8 * pr);
    }
    return packed;
}

// Codes of 8 consecutive entries rounded to the nearest level (the
// deterministic comparator of "Rate-adaptive KV-cache quantizer",
// "Implementation notes": uniform INT4 at equal bytes): the same interval
// search, then code i + [w_i < 2 (x - q_i)] in fp32 round-to-nearest (a tie
// keeps the lower level).  qw holds (-q_i, w_i).
__device__ __forceinline__ uint32_t quant8_nearest(const uint4 raw, const uint32_t (&T)[16],
                                                   const float2 *qw) {
    const uint32_t xw0 = raw.x, xw1 = raw.y, xw2 = raw.z, xw3 = raw.w;
    uint32_t packed = 0;
#pragma unroll
    for (int pr = 0; pr < 4; ++pr) {
        const __half2 X = as_h2(pr == 0 ? xw0 : pr == 1 ? xw1 : pr == 2 ? xw2 : xw3);
        const uint32_t m1 = __hge2_mask(X, as_h2(T[8]));
        const uint32_t t2 = (T[12] & m1) | (T[4] & ~m1);
        const uint32_t m2 = __hge2_mask(X, as_h2(t2));
        const uint32_t a3 = (T[6] & m2) | (T[2] & ~m2), b3 = (T[14] & m2) | (T[10] & ~m2);
        const uint32_t t3 = (b3 & m1) | (a3 & ~m1);
        const uint32_t m3 = __hge2_mask(X, as_h2(t3));
        const uint32_t a4 = (T[3] & m3) | (T[1] & ~m3), b4 = (T[7] & m3) | (T[5] & ~m3);
        const uint32_t c4 = (T[11] & m3) | (T[9] & ~m3), d4 = (T[15] & m3) | (T[13] & ~m3);
        const uint32_t lo4 = (b4 & m2) | (a4 & ~m2), hi4 = (d4 & m2) | (c4 & ~m2);
        const uint32_t t4 = (hi4 & m1) | (lo4 & ~m1);
        const uint32_t m4 = __hge2_mask(X, as_h2(t4));
        const uint32_t idx = (m1 & 0x00080008u) | (m2 & 0x00040004u) | (m3 & 0x00020002u) |
                             (m4 & 0x00010001u);
        const int i0 = (int)(idx & 15u), i1 = (int)(idx >> 16);
        const float2 e0 = qw[i0], e1 = qw[i1];
        const float2 xf = __half22float2(X);
        const float2 r = __fadd2_rn(xf, make_float2(e0.x, e1.x));          // x - q_i
        const float2 r2 = __fadd2_rn(r, r);                                 // exact
        const uint32_t c0 = (uint32_t)i0 + (e0.y < r2.x ? 1u : 0u);
        const uint32_t c1 = (uint32_t)i1 + (e1.y < r2.y ? 1u : 0u);
        packed |= (c0 | (c1 << 4)) << (8 * pr);
    }
    return packed;
}

}  // namespace kvq
