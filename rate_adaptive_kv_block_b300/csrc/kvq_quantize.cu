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
    float thr[kMaxGroups][16];   // thr[j] = q_j for 1 <= j <= k-2, +inf beyond
    float2 qw[kMaxGroups][16];   // (q_i, (q_{i+1} - q_i) * 2^-24)
    int k[kMaxGroups];
};

__global__ void __launch_bounds__(kQThreads)
quantize_kernel(const uint16_t *__restrict__ x, kvq_layout L, const float *__restrict__ codebook,
                const uint8_t *__restrict__ kk, uint64_t seed, uint64_t index_base,
                uint8_t *__restrict__ codes) {
    __shared__ QSmem sm;
    const int D = L.D, G = L.group, nG = D / G;
    const int64_t slab = blockIdx.x;                 // stream * (T/32) + token block
    const int64_t blk0 = slab * nG;
    const int hb = 16 * G;                           // code bytes per block
    for (int i = threadIdx.x; i < nG * 16; i += kQThreads) {
        const int g = i >> 4, j = i & 15;
        const float *q = codebook + (blk0 + g) * 16;
        const int k = kk[blk0 + g];
        const float qj = q[j];
        sm.thr[g][j] = (j >= 1 && j <= k - 2) ? qj : __int_as_float(0x7f800000);
        const float qn = q[j < 15 ? j + 1 : 15];
        const float w = (j <= k - 2) ? __fsub_rn(qn, qj) : 0.f;
        sm.qw[g][j] = make_float2(qj, __fmul_rn(w, 5.9604644775390625e-8f));   // exact: 2^-24
        if (j == 0) sm.k[g] = k;
    }
    __syncthreads();
    const int units = 4 * D;                         // 8-entry units in the slab
    const int upr = D / 8;
    for (int u = threadIdx.x; u < units; u += kQThreads) {
        const int row = u / upr, f0 = (u % upr) * 8;
        const int g = f0 / G;
        const int e0 = row * G + (f0 % G);
        const int64_t flat = (slab * 32 + row) * (int64_t)D + f0;
        const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(x + flat));
        const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
        const int k = sm.k[g];
        uint64_t z = seed + ((index_base + (uint64_t)flat) / 2 + 1) * kGolden;
        uint32_t packed = 0;
#pragma unroll
        for (int pr = 0; pr < 4; ++pr) {
            const uint64_t hz = splitmix_mix(z);
            z += kGolden;
            const uint32_t hsh[2] = {(uint32_t)(hz >> 32), (uint32_t)hz};
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int el = 2 * pr + q;
                const float xv = __half2float(__ushort_as_half(
                    (unsigned short)((w4[el >> 1] >> ((el & 1) * 16)) & 0xffffu)));
                uint32_t code = 0;
                if (k > 1) {
                    int i = 0;
                    i += (xv >= sm.thr[g][i + 8]) ? 8 : 0;
                    i += (xv >= sm.thr[g][i + 4]) ? 4 : 0;
                    i += (xv >= sm.thr[g][i + 2]) ? 2 : 0;
                    i += (xv >= sm.thr[g][i + 1]) ? 1 : 0;
                    const float2 qw = sm.qw[g][i];
                    const float r = __fsub_rn(xv, qw.x);
                    const float tw = __fmul_rn((float)(hsh[q] >> 8), qw.y);
                    code = (uint32_t)i + (tw < r ? 1u : 0u);
                }
                packed |= code << (4 * el);
            }
        }
        *reinterpret_cast<uint32_t *>(codes + (blk0 + g) * hb + e0 / 2) = packed;
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
    quantize_kernel<<<(unsigned)slabs, kQThreads, 0, st>>>(x, L, codebook, k, seed, index_base,
                                                          codes);
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
