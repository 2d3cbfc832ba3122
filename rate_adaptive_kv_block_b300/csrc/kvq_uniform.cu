// kvq_uniform_codebook: the uniform comparator's codebooks ("Rate-adaptive
// KV-cache quantizer", "Implementation notes": compare uniform INT4 and
// uniform stochastic quantization at equal cache bytes).
//
// Per block, from its minimum m and maximum M (exact binary16 values):
//   delta = fl32(fl32(M - m) / 15)
//   level_j = binary16(fl32(m + fl32(j * delta)))   j = 0 .. 14
//   level_15 = M
// all in fp32 round-to-nearest without contraction, then rounded to binary16
// (the stored levels are binary16 values, as the quantizer's are), kept in
// order with repeats removed (k distinct levels, slots k..15 repeat the top).
// kvq_quantize with these codebooks is uniform stochastic quantization (the
// page's unbiased interpolation on an equally spaced grid);
// kvq_quantize_nearest is uniform INT4 (round to the nearest level).
//
// One warp per block: 16-byte loads of the block's rows, a warp reduction of
// the minimum and maximum (a zero of either sign taken as +0), then lane
// j < 16 forms level j.  Non-finite
// entries set KVQ_ERR_NONFINITE in the status word (the codebook of that
// block is then unspecified).
#include "kvq_internal.cuh"

namespace kvq {

constexpr int kUniThreads = 128;

__global__ void __launch_bounds__(kUniThreads)
uniform_codebook_kernel(const uint16_t *__restrict__ x, kvq_layout L, int64_t nb,
                        float *__restrict__ codebook, uint8_t *__restrict__ kout,
                        int32_t *__restrict__ status) {
    const int lane = threadIdx.x & 31;
    const int64_t b = (int64_t)blockIdx.x * (kUniThreads / 32) + (threadIdx.x >> 5);
    if (b >= nb) return;
    const int G = L.group, D = L.D, nG = D / G;
    const int64_t slab = b / nG;                  // stream * (T / 32) + token block
    const int g = (int)(b % nG);
    const int upr = G / 8;                        // 16-byte units per row
    float mn = __int_as_float(0x7f800000), mx = -mn;
    bool bad = false;
    for (int u = lane; u < 32 * upr; u += 32) {
        const int row = u / upr, cu = u % upr;
        const uint4 w = *reinterpret_cast<const uint4 *>(x + (slab * 32 + row) * (int64_t)D +
                                                         (int64_t)g * G + cu * 8);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int hlf = 0; hlf < 2; ++hlf) {
                const uint16_t hbits = (uint16_t)(ws[i] >> (16 * hlf));
                bad |= (hbits & 0x7c00u) == 0x7c00u;
                const float v = __half2float(__ushort_as_half(hbits));
                mn = fminf(mn, v);
                mx = fmaxf(mx, v);
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicMax(status, (int32_t)KVQ_ERR_NONFINITE);
    mn = __fadd_rn(mn, 0.f);                      // -0 -> +0 (the minimum of -0 and +0 is either)
    mx = __fadd_rn(mx, 0.f);
    // level j on lane j (< 16)
    const float delta = __fdiv_rn(__fsub_rn(mx, mn), 15.f);
    float v = mx;
    if (lane < 15) v = __half2float(__float2half_rn(__fadd_rn(mn, __fmul_rn((float)lane, delta))));
    const float prev = __shfl_up_sync(0xffffffffu, v, 1);
    const bool keep = lane < 16 && (lane == 0 || v != prev);
    const uint32_t km = __ballot_sync(0xffffffffu, keep);
    const int k = __popc(km);
    const int pos = __popc(km & ((1u << lane) - 1u));
    float *cb = codebook + b * 16;
    if (keep) cb[pos] = v;
    if (lane >= k && lane < 16) cb[lane] = mx;    // slots k .. 15 repeat the top level
    if (lane == 0) kout[b] = (uint8_t)k;
}

int launch_uniform_codebook(const uint16_t *x, const kvq_layout &L, float *codebook, uint8_t *k,
                            int32_t *status, cudaStream_t st) {
    const int64_t nb = num_blocks(L);
    if (cudaMemsetAsync(status, 0, sizeof(int32_t), st) != cudaSuccess) return KVQ_ERR_CUDA;
    if (nb == 0) return KVQ_OK;
    const int64_t ctas = (nb + kUniThreads / 32 - 1) / (kUniThreads / 32);
    uniform_codebook_kernel<<<(unsigned)ctas, kUniThreads, 0, st>>>(x, L, nb, codebook, k, status);
    return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq
