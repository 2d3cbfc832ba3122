// kvq_quantize / kvq_dequantize: unbiased stochastic interpolation with
// 4-bit packing, and its decode ("Rate-adaptive KV-cache quantizer", "Key
// formulas": P(q_{i+1} | x) = (x - q_i)/(q_{i+1} - q_i); "Implementation
// notes": store the codebook and the symbol stream; decode before attention).
//
// kvq_quantize is a persistent kernel that streams the tensor through shared
// memory: a tile is 32 tokens x Dc features of one stream (Dc = min(D, 256)),
// copied by the bulk-copy (TMA) engine into a ring of stages, each completing
// on its own mbarrier, several tiles ahead of the warps that consume it; the
// tile's codebooks ride in the same copy.  Per tile, 16 threads per block turn
// the codebook into the interval thresholds and the (-q_i, w_i) table; every
// thread then handles fixed 8-feature columns of the tile.  Per pair of
// entries (binary16x2): the interval index is a 4-level binary search over
// the 15 thresholds (padded with +inf) with packed half2 comparisons and
// bitwise selects, the rounding decision uses packed fp32 add / multiply
// (explicit round-to-nearest, so no multiply-add contraction can change a
// code), and one SplitMix64 output gives both uniforms.
#include "kvq_internal.cuh"
#include "kvq_bulk.cuh"
#include "kvq_quant_core.cuh"

namespace kvq {

constexpr int kQThreads = 128;
constexpr int kQStages = 4;
constexpr int kQMaxCols = 256;               // features per tile (at most)
constexpr int kQMaxGroups = kQMaxCols / 8;   // blocks per tile (at most)
constexpr uint32_t kQWaitLimit = 1u << 22;   // mbarrier polls before giving up


// --------------------------------------------------------------- tiles
struct QGeom {
    int D, G, Dc;          // features, block width, tile width (powers of two)
    int nchunk;            // tiles per 32-token slab
    int ngt;               // blocks per tile
    int upr_log2;          // log2(Dc / 8)
    int chunk_log2;        // log2(nchunk)
    int g_log2;            // log2(G)
    int bps_log2;          // log2(D / G): blocks per slab
    uint32_t x_bytes;      // 64 * Dc
    uint32_t cb_bytes;     // 64 * ngt
    uint32_t stage_bytes;  // x_bytes + cb_bytes, rounded to 128
};

// Issue the copies of tile t into stage buffer `buf`.
__device__ __forceinline__ void issue_tile(const QGeom &g, int64_t t, const uint16_t *x,
                                           const float *codebook, char *buf, uint64_t *bar) {
    const int64_t slab = t >> g.chunk_log2;
    const int chunk = (int)(t & (g.nchunk - 1));
    mbar_expect_tx(bar, g.x_bytes + g.cb_bytes);
    const uint16_t *src = x + slab * 32 * (int64_t)g.D + (int64_t)chunk * g.Dc;
    if (g.Dc == g.D) {
        bulk_g2s(buf, src, g.x_bytes, bar);                 // the slab is contiguous
    } else {
        for (int r = 0; r < 32; ++r)
            bulk_g2s(buf + r * g.Dc * 2, src + (int64_t)r * g.D, (uint32_t)(g.Dc * 2), bar);
    }
    const int64_t blk0 = (slab << g.bps_log2) + (int64_t)chunk * g.ngt;
    bulk_g2s(buf + g.x_bytes, codebook + blk0 * 16, g.cb_bytes, bar);
}

struct QTables {
    __half2 thr[kQMaxGroups][16];   // (q_j, q_j) for 1 <= j <= k-2, +inf beyond; [0] unused
    float2 qw[kQMaxGroups][16];     // (-q_i, (q_{i+1} - q_i) * 2^-24); k = 1: (-q_0, +inf)
};

template <bool NEAREST>
__global__ void __launch_bounds__(kQThreads, 6)
quantize_kernel(const uint16_t *__restrict__ x, const float *__restrict__ codebook, QGeom g,
                int64_t ntiles, uint64_t seed, uint64_t index_base, uint8_t *__restrict__ codes,
                int32_t *__restrict__ status) {
    extern __shared__ __align__(128) char qsm[];
    __shared__ __align__(8) uint64_t bars[kQStages];
    __shared__ __align__(16) QTables tb;
    __shared__ bool failed;
    const int tid = threadIdx.x;
    if (tid == 0) {
        for (int s = 0; s < kQStages; ++s) mbar_init(&bars[s], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        failed = false;
    }
    __syncthreads();
    // prologue: the first kQStages tiles of this CTA in flight
    if (tid == 0) {
        for (int s = 0; s < kQStages; ++s) {
            const int64_t t = (int64_t)blockIdx.x + (int64_t)s * gridDim.x;
            if (t < ntiles) issue_tile(g, t, x, codebook, qsm + s * g.stage_bytes, &bars[s]);
        }
    }
    const int upr = 1 << g.upr_log2;
    const int cu = tid & (upr - 1);
    const int row0 = tid >> g.upr_log2, rstep = kQThreads >> g.upr_log2;
    const int f0 = cu * 8;                       // column inside the tile
    const int gt = f0 >> g.g_log2;               // block inside the tile
    const int hb = 16 * g.G;                     // code bytes per block
    uint32_t n = 0;                              // tiles consumed by this CTA
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++n) {
        const uint32_t s = n % kQStages;
        char *buf = qsm + s * g.stage_bytes;
        if (!mbar_wait(&bars[s], (n / kQStages) & 1u, kQWaitLimit)) {
            if (tid == 0) failed = true;
        }
        __syncthreads();
        if (failed) break;
        // codebook -> thresholds and decision table (16 threads per block)
        const float *cb = reinterpret_cast<const float *>(buf + g.x_bytes);
        for (int i = tid; i < g.ngt * 16; i += kQThreads) {
            const int b = i >> 4, j = i & 15;
            const float *q = cb + b * 16;
            const float top = q[15];
            int k = 1;
#pragma unroll
            for (int m = 0; m < 15; ++m) k += q[m] < top ? 1 : 0;
            quant_table_entry<NEAREST>(q, k, j, tb.thr[b][j], tb.qw[b][j]);
        }
        __syncthreads();
        // this thread's block: 15 thresholds in registers
        uint32_t T[16];
#pragma unroll
        for (int j = 1; j < 16; ++j) {
            const __half2 h = tb.thr[gt][j];
            memcpy(&T[j], &h, 4);
        }
        const float2 *qw = tb.qw[gt];
        const int64_t slab = t >> g.chunk_log2;
        const int chunk = (int)(t & (g.nchunk - 1));
        const int col = chunk * g.Dc + f0;                      // feature of the first entry
        const int64_t blk = (slab << g.bps_log2) + (col >> g.g_log2);
        uint8_t *cbase = codes + blk * hb + ((col & (g.G - 1)) >> 1);
        uint64_t z = quant_state(seed, index_base, (uint64_t)((slab * 32 + row0) * (int64_t)g.D + col));
        const uint64_t zstep = (uint64_t)(rstep * g.D / 2) * kGolden;
        for (int row = row0; row < 32; row += rstep, z += zstep) {
            const uint4 raw = *reinterpret_cast<const uint4 *>(buf + (row * g.Dc + f0) * 2);
            uint32_t cw;
            if constexpr (NEAREST) cw = quant8_nearest(raw, T, qw);
            else cw = quant8(raw, T, qw, z);
            *reinterpret_cast<uint32_t *>(cbase + (int64_t)row * (g.G / 2)) = cw;
        }
        __syncthreads();                         // every thread is done with this stage
        if (tid == 0) {
            const int64_t tn = t + (int64_t)kQStages * gridDim.x;
            if (tn < ntiles) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue_tile(g, tn, x, codebook, buf, &bars[s]);
            }
        }
    }
    if (failed) {
        // a copy never completed: report it, and give the copies this CTA
        // issued a bounded chance to land before the shared memory is released
        if (tid == 0) {
            if (status) atomicExch(status, KVQ_ERR_TIMEOUT);
            for (uint32_t k = 0; k < kQStages; ++k) {
                const uint32_t nk = n + k;
                const int64_t tk = (int64_t)blockIdx.x + (int64_t)nk * gridDim.x;
                if (tk < ntiles) mbar_wait(&bars[nk % kQStages], (nk / kQStages) & 1u, kQWaitLimit);
            }
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kQThreads)
dequantize_kernel(const uint8_t *__restrict__ codes, const float *__restrict__ codebook,
                  kvq_layout L, uint16_t *__restrict__ y) {
    __shared__ uint16_t sq[32][16];
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

static int g_quant_grid[64];

static QGeom geometry(const kvq_layout &L) {
    QGeom g;
    g.D = L.D;
    g.G = L.group;
    g.Dc = L.D < kQMaxCols ? L.D : kQMaxCols;
    g.nchunk = L.D / g.Dc;
    g.ngt = g.Dc / g.G;
    auto lg2 = [](int v) { int l = 0; while ((1 << l) < v) ++l; return l; };
    g.upr_log2 = lg2(g.Dc / 8);
    g.chunk_log2 = lg2(g.nchunk);
    g.g_log2 = lg2(g.G);
    g.bps_log2 = lg2(g.D / g.G);
    g.x_bytes = (uint32_t)(64 * g.Dc);
    g.cb_bytes = (uint32_t)(64 * g.ngt);
    g.stage_bytes = (g.x_bytes + g.cb_bytes + 127u) & ~127u;
    return g;
}

int quantize_init() {
    int dev = 0, sms = 0, occ = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KVQ_ERR_CUDA;
    const int smem = kQStages * ((64 * kQMaxCols + 64 * kQMaxGroups + 127) & ~127);
    if (cudaFuncSetAttribute(quantize_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess ||
        cudaFuncSetAttribute(quantize_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
        return KVQ_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return KVQ_ERR_CUDA;
    // the grid for the llama-shaped tile size (8 KB + codebook per stage)
    const int smem128 = kQStages * ((64 * 128 + 64 + 127) & ~127);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, quantize_kernel<false>, kQThreads, smem128) !=
        cudaSuccess)
        return KVQ_ERR_CUDA;
    g_quant_grid[dev] = (occ < 1 ? 1 : occ) * sms;
    return KVQ_OK;
}

int launch_quantize(const uint16_t *x, const kvq_layout &L, const float *codebook,
                    const uint8_t *k, uint64_t seed, uint64_t index_base, uint8_t *codes,
                    int32_t *status, cudaStream_t st, bool nearest) {
    (void)k;   // the kernel reads k from the codebook (slots k..15 repeat the top level)
    const QGeom g = geometry(L);
    const int64_t ntiles = L.S * (L.T / 32) * g.nchunk;
    if (ntiles == 0) return KVQ_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KVQ_ERR_CUDA;
    int64_t grid = g_quant_grid[dev] > 0 ? g_quant_grid[dev] : 148;
    if (grid > ntiles) grid = ntiles;
    const size_t smem = (size_t)kQStages * g.stage_bytes;
    if (nearest)
        quantize_kernel<true><<<(unsigned)grid, kQThreads, smem, st>>>(x, codebook, g, ntiles, seed,
                                                                       index_base, codes, status);
    else
        quantize_kernel<false><<<(unsigned)grid, kQThreads, smem, st>>>(x, codebook, g, ntiles, seed,
                                                                        index_base, codes, status);
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
