// The quantizer's arithmetic, shared by kvq_quantize and the fused
// allocate-and-quantize path ("Rate-adaptive KV-cache quantizer", "Key
// formulas": P(q_{i+1} | x) = (x - q_i)/(q_{i+1} - q_i)).
//
// For one block with levels q_0 < ... < q_{k-1} (slots k..15 repeat q_{k-1}):
//   thresholds  T_j = q_j for 1 <= j <= k-2, +inf beyond (binary16 pairs);
//   decision    (-q_i, w_i) with w_i = (q_{i+1} - q_i) 2^-24 (k = 1: w = +inf).
// An entry x gets i = #{j : T_j <= x} (a 4-level binary search over the 15
// sorted thresholds) and code i + [fl(u w_i) < fl(x - q_i)], fp32
// round-to-nearest, u = hash >> 8; hash(seed, n) = SplitMix64 output n>>1,
// high word for even n, low word for odd n.
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>
#include <string.h>

namespace kvq {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ __half2 as_h2(uint32_t u) {
    __half2 h;
    memcpy(&h, &u, 4);
    return h;
}

// SplitMix64 output function (Steele, Lea, Flood 2014), written on the two
// 32-bit halves (hi:lo) of the state so that each step is one funnel shift,
// one xor or one 32-bit multiply-add: returns the output's high and low words.
__device__ __forceinline__ void splitmix_mix(uint32_t lo, uint32_t hi, uint32_t &ohi,
                                             uint32_t &olo) {
    // z ^= z >> 30; z *= 0xBF58476D1CE4E5B9
    lo ^= __funnelshift_r(lo, hi, 30);
    hi ^= hi >> 30;
    const uint32_t nlo0 = lo * 0x1CE4E5B9u;
    const uint32_t nhi0 = __umulhi(lo, 0x1CE4E5B9u) + lo * 0xBF58476Du + hi * 0x1CE4E5B9u;
    // z ^= z >> 27; z *= 0x94D049BB133111EB
    const uint32_t nlo = nlo0 ^ __funnelshift_r(nlo0, nhi0, 27);
    const uint32_t nhi = nhi0 ^ (nhi0 >> 27);
    lo = nlo * 0x133111EBu;
    hi = __umulhi(nlo, 0x133111EBu) + nlo * 0x94D049BBu + nhi * 0x133111EBu;
    // z ^= z >> 31
    olo = lo ^ __funnelshift_r(lo, hi, 31);
    ohi = hi ^ (hi >> 31);
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
// T[1..15] the thresholds as binary16 pairs, qw the decision table, z the
// SplitMix64 state of the first pair.  Returns 8 nibbles, entry e in bits
// 4e..4e+3.
__device__ __forceinline__ uint32_t quant8(const uint4 raw, const uint32_t (&T)[16],
                                           const float2 *qw, uint64_t z) {
    const uint32_t xw0 = raw.x, xw1 = raw.y, xw2 = raw.z, xw3 = raw.w;
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
        uint32_t hhi, hlo;
        splitmix_mix((uint32_t)z, (uint32_t)(z >> 32), hhi, hlo);
        z += kGolden;
        const float2 xf = __half22float2(X);
        const float2 r = __fadd2_rn(xf, make_float2(e0.x, e1.x));          // x - q_i
        const float2 u = make_float2((float)(hhi >> 8), (float)(hlo >> 8));
        const float2 tw = __fmul2_rn(u, make_float2(e0.y, e1.y));
        const uint32_t c0 = (uint32_t)i0 + (tw.x < r.x ? 1u : 0u);
        const uint32_t c1 = (uint32_t)i1 + (tw.y < r.y ? 1u : 0u);
        packed |= (c0 | (c1 << 4)) << (8 * pr);
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

// SplitMix64 state of the pair holding global entry `flat` (even) for `seed`.
__device__ __forceinline__ uint64_t quant_state(uint64_t seed, uint64_t index_base, uint64_t flat) {
    return seed + ((index_base + flat) / 2 + 1) * kGolden;
}

}  // namespace kvq
