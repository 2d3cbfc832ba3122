// kvq_quantize / kvq_dequantize: unbiased stochastic interpolation with
// 4-bit packing, and its decode ("Rate-adaptive KV-cache quantizer", "Key
// formulas": P(q_{i+1} | x) = (x - q_i)/(q_{i+1} - q_i); "Implementation
// notes": store the codebook and the symbol stream; decode before attention).
//
// One CTA per 32-token slab of one stream (32 x D binary16, contiguous), so
// both passes stream HBM with 16-byte loads and stores.  The slab holds D/G
// blocks; their codebooks are staged in shared memory once per slab.  Every
// fp32 operation of the rounding decision is an explicit round-to-nearest
// intrinsic, so no multiply-add contraction can change a code.
#include "kvq_internal.cuh"

namespace kvq {

constexpr int kQThreads = 256;
constexpr int kMaxGroups = 32;

// SplitMix64 output function (Steele, Lea, Flood 2014).
__device__ __forceinline__ uint64_t splitmix_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}
constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

struct QSmem {
    __half2 thr[kMaxGroups][16];   // (q_j, q_j) for 1 <= j <= k-2, +inf beyond
    float2 qw[kMaxGroups][16];     // (q_i, (q_{i+1} - q_i) * 2^-24); k = 1: (q_0, +inf)
    int kmax;
};

// Interval index of two binary16 entries at once: the number of thresholds
// q_1 .. q_{k-2} at or below each entry, counted in a half2 accumulator that
// starts at 1024 (binary16 integers 1024..2047 are exact and their low byte
// is the count).  The comparisons and adds run on the fp16 FMA datapath.
template <int NT>
__device__ __forceinline__ void count_below(const __half2 (&xh)[4], const __half2 *th, int nthr,
                                            uint32_t (&cnt)[4]) {
    const __half2 base = __floats2half2_rn(1024.f, 1024.f);
    __half2 c[4] = {base, base, base, base};
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        if (j < nthr) {
            const __half2 t = th[j];
#pragma unroll
            for (int p = 0; p < 4; ++p) c[p] = __hadd2(c[p], __hge2(xh[p], t));
        }
    }
#pragma unroll
    for (int p = 0; p < 4; ++p) cnt[p] = *reinterpret_cast<const uint32_t *>(&c[p]);
}

// One CTA per 32-token slab; thread t always handles the same 8 features
// (column unit t % (D/8)) on rows t / (D/8), t / (D/8) + 256 / (D/8), ...
// (D / 8 divides 256 for D a power of two <= 2048).
__global__ void __launch_bounds__(kQThreads)
quantize_kernel(const uint16_t *__restrict__ x, kvq_layout L, const float *__restrict__ codebook,
                const uint8_t *__restrict__ kk, uint64_t seed, uint64_t index_base,
                uint8_t *__restrict__ codes, int log2_upr) {
    __shared__ __align__(16) QSmem sm;
    const int D = L.D, G = L.group, nG = D / G;
    const int64_t slab = blockIdx.x;                 // stream * (T/32) + token block
    const int64_t blk0 = slab * nG;
    const int hb = 16 * G;                           // code bytes per block
    if (threadIdx.x == 0) sm.kmax = 0;
    __syncthreads();
    const float INF = __int_as_float(0x7f800000);
    for (int i = threadIdx.x; i < nG * 16; i += kQThreads) {
        const int g = i >> 4, j = i & 15;
        const float *q = codebook + (blk0 + g) * 16;
        const int k = kk[blk0 + g];
        const float qj = q[j];
        const float t = (j >= 1 && j <= k - 2) ? qj : INF;
        sm.thr[g][j] = __floats2half2_rn(t, t);     // exact: levels are binary16 values
        const float qn = q[j < 15 ? j + 1 : 15];
        float ws = 0.f;
        if (k <= 1) ws = INF;                       // k = 1: never move up
        else if (j <= k - 2) ws = __fmul_rn(__fsub_rn(qn, qj), 5.9604644775390625e-8f);  // 2^-24, exact
        sm.qw[g][j] = make_float2(qj, ws);
        if (j == 0) atomicMax(&sm.kmax, k);
    }
    __syncthreads();
    const int upr = 1 << log2_upr;                  // 8-entry units per row
    const int cu = threadIdx.x & (upr - 1);
    const int row0 = threadIdx.x >> log2_upr, rstep = kQThreads >> log2_upr;
    const int f0 = cu * 8;
    const int g = f0 / G;
    const int nthr = sm.kmax - 2;
    __half2 th[14];
#pragma unroll
    for (int j = 0; j < 14; ++j) th[j] = sm.thr[g][j + 1];
    const float2 *qw = sm.qw[g];
    uint8_t *cbase = codes + (blk0 + g) * hb + (f0 % G) / 2;
    const int64_t flat0 = (slab * 32 + row0) * (int64_t)D + f0;
    uint64_t z = seed + ((index_base + (uint64_t)flat0) / 2 + 1) * kGolden;
    const uint64_t zstep = (uint64_t)(rstep * D / 2) * kGolden;
    for (int row = row0; row < 32; row += rstep, z += zstep) {
        const int64_t flat = (slab * 32 + row) * (int64_t)D + f0;
        const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(x + flat));
        __half2 xh[4];
        xh[0] = *reinterpret_cast<const __half2 *>(&raw.x);
        xh[1] = *reinterpret_cast<const __half2 *>(&raw.y);
        xh[2] = *reinterpret_cast<const __half2 *>(&raw.z);
        xh[3] = *reinterpret_cast<const __half2 *>(&raw.w);
        uint32_t cnt[4];
        count_below<14>(xh, th, nthr, cnt);
        uint32_t packed = 0;
        uint64_t zz = z;
#pragma unroll
        for (int pr = 0; pr < 4; ++pr) {
            const uint64_t hz = splitmix_mix(zz);
            zz += kGolden;
            const uint32_t hsh[2] = {(uint32_t)(hz >> 32), (uint32_t)hz};
            const float2 xf = __half22float2(xh[pr]);
            const float xv[2] = {xf.x, xf.y};
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int i = (int)((cnt[pr] >> (16 * q)) & 0xffu);
                const float2 a = qw[i];
                const float r = __fsub_rn(xv[q], a.x);
                const float tw = __fmul_rn((float)(hsh[q] >> 8), a.y);
                const uint32_t code = (uint32_t)i + (tw < r ? 1u : 0u);
                packed |= code << (4 * (2 * pr + q));
            }
        }
        *reinterpret_cast<uint32_t *>(cbase + (int64_t)row * (G / 2)) = packed;
    }
}

__global__ void __launch_bounds__(kQThreads)
dequantize_kernel(const uint8_t *__restrict__ codes, const float *__restrict__ codebook,
                  kvq_layout L, uint16_t *__restrict__ y) {
    __shared__ uint16_t sq[kMaxGroups][16];
    const int D = L.D, G = L.group, nG = D / G;
    const int64_t slab = blockIdx.x;
    const int64_t blk0 = slab * nG;
    const int hb = 16 * G;
    for (int i = threadIdx.x; i < nG * 16; i += kQThreads)
        sq[i >> 4][i & 15] = __half_as_ushort(__float2half_rn(codebook[blk0 * 16 + i]));
    __syncthreads();
    const int units = 4 * D, upr = D / 8;
    for (int u = threadIdx.x; u < units; u += kQThreads) {
        const int row = u / upr, f0 = (u % upr) * 8;
        const int g = f0 / G;
        const int e0 = row * G + (f0 % G);
        const uint32_t c = *reinterpret_cast<const uint32_t *>(codes + (blk0 + g) * hb + e0 / 2);
        uint32_t o[4];
#pragma unroll
        for (int p = 0; p < 4; ++p)
            o[p] = (uint32_t)sq[g][(c >> (8 * p)) & 15u] |
                   ((uint32_t)sq[g][(c >> (8 * p + 4)) & 15u] << 16);
        const int64_t flat = (slab * 32 + row) * (int64_t)D + f0;
        *reinterpret_cast<uint4 *>(y + flat) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

int launch_quantize(const uint16_t *x, const kvq_layout &L, const float *codebook,
                    const uint8_t *k, uint64_t seed, uint64_t index_base, uint8_t *codes,
                    cudaStream_t st) {
    const int64_t slabs = L.S * (L.T / 32);
    if (slabs == 0) return KVQ_OK;
    int log2_upr = 0;
    while ((1 << log2_upr) < L.D / 8) ++log2_upr;
    quantize_kernel<<<(unsigned)slabs, kQThreads, 0, st>>>(x, L, codebook, k, seed, index_base,
                                                          codes, log2_upr);
    return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

int launch_dequantize(const uint8_t *codes, const float *codebook, const kvq_layout &L,
                      uint16_t *y, cudaStream_t st) {
    const int64_t slabs = L.S * (L.T / 32);
    if (slabs == 0) return KVQ_OK;
    dequantize_kernel<<<(unsigned)slabs, kQThreads, 0, st>>>(codes, codebook, L, y);
    return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq
