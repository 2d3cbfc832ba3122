// kvq_quantize / kvq_dequantize: unbiased stochastic interpolation with
// 4-bit packing, and its decode ("Rate-adaptive KV-cache quantizer", "Key
// formulas": P(q_{i+1} | x) = (x - q_i)/(q_{i+1} - q_i); "Implementation
// notes": store the codebook and the symbol stream; decode before attention).
//
// Both quantize kernels are persistent and stream the tensor through shared
// memory: the bulk-copy (TMA) engine fills a ring of stages, each completing
// on its own mbarrier, several stages ahead of the warps that consume them;
// a stage's codebooks ride in the same copies.  Per entry the rounding
// decision is fl(u w_i) < fl(x - q_i) with explicit round-to-nearest fp32
// operations (packed pairs; no multiply-add contraction can change a code),
// and one Philox4x32-7 block gives the uniforms of 4 consecutive entries.
//
// The table kernel (blocks of 32 or more features) finds an entry's interval
// with two shared-memory loads and one integer add.  Per block and stage, a
// 256-bin table is indexed by the high byte of the entry's order-preserving
// 16-bit key (the binary16 bits with the sign folded, so that key order is
// value order); each bin holds, in 16 bits, the number of thresholds below
// the bin (ib) and the low key byte t of the threshold inside it (256: none),
// stored as ((ib - bin) << 8) + 256 - t, so that (entry + key) has ib + [low
// key byte >= t] in bits 8..15: the carry of the low byte is the comparison.
// That index addresses the block's (-q_i, w_i) pair.  A block with two
// thresholds in one bin takes the binary search of the search kernel.
//
// The search kernel (narrower blocks, and the nearest-level comparator) finds
// the interval with a 4-level binary search over the 15 thresholds using
// packed half2 comparisons and bitwise selects.
#include "kvq_internal.cuh"
#include "kvq_bulk.cuh"
#include "kvq_quant_core.cuh"

namespace kvq {

constexpr uint32_t kQWaitLimit = 1u << 22;   // mbarrier polls before giving up

// ----------------------------------------------------- shared-memory access
__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ float2 lds_f2(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
    return v;
}
// order-preserving keys of the two binary16 halves of w: a negative half is
// complemented, a non-negative one gets its sign bit set
__device__ __forceinline__ uint32_t key_pair(uint32_t w) {
    uint32_t sgn;
    asm("prmt.b32 %0, %1, 0, 0xBB99;" : "=r"(sgn) : "r"(w));   // sign of each half, replicated
    return w ^ ((sgn & 0x7FFF7FFFu) | 0x80008000u);
}
__device__ __forceinline__ uint32_t key16(float q) {
    const uint32_t h = (uint32_t)__half_as_ushort(__float2half_rn(q));   // exact: q is binary16
    return (h & 0x8000u) ? (h ^ 0xFFFFu) : (h ^ 0x8000u);
}

// ================================================================ table kernel
#ifndef KVQ_QT_THREADS
#define KVQ_QT_THREADS 512
#endif
#ifndef KVQ_QT_STAGES
#define KVQ_QT_STAGES 3
#endif
#ifndef KVQ_QT_STAGEX
#define KVQ_QT_STAGEX 32768
#endif
#ifndef KVQ_QT_MINB
#define KVQ_QT_MINB 1
#endif
constexpr int kTThreads = KVQ_QT_THREADS;
constexpr int kTStages = KVQ_QT_STAGES;
constexpr int kTStageX = KVQ_QT_STAGEX;   // input bytes of a stage (at most)
constexpr int kTMaxBlocks = 16;           // blocks of a stage (at most)
constexpr int kTMinGroup = 32;       // narrower blocks use the search kernel

struct TGeom {
    int D, G, Dc;          // features, block width, tile width
    int nchunk;            // column tiles per 32-token slab (D / Dc)
    int spt;               // slabs per stage (1 when Dc < D)
    int ngt;               // blocks per tile row (Dc / G)
    int upr_log2;          // log2(Dc / 8): 8-entry units per row
    int upt;               // units (rows) per thread
    int g_log2, bps_log2, chunk_log2;
    int64_t nslabs;        // S T / 32
    int64_t nstages;
    uint32_t x_bytes;      // input bytes of a full stage
    uint32_t stage_bytes;  // + codebooks, rounded to 128
};

struct TTables {
    uint16_t bins[2][kTMaxBlocks][256];     // per stage parity and block
    float2 qw[2][kTMaxBlocks][16];          // (-q_i, (q_{i+1} - q_i) 2^-24)
    uint32_t thr[2][kTMaxBlocks][16];       // binary16 pairs for the search path
    int32_t slow[2][kTMaxBlocks][4];        // per quarter of the bins: two thresholds in a bin
};

__device__ __forceinline__ void t_issue(const TGeom &g, int64_t s, const uint16_t *x,
                                        const float *codebook, char *buf, uint64_t *bar) {
    if (g.Dc == g.D) {
        const int64_t slab0 = s * g.spt;
        const int64_t ns = min((int64_t)g.spt, g.nslabs - slab0);
        const uint32_t bx = (uint32_t)(ns * 64 * g.D), bc = (uint32_t)(ns * g.ngt * 64);
        mbar_expect_tx(bar, bx + bc);
        bulk_g2s(buf, x + slab0 * 32 * g.D, bx, bar);
        bulk_g2s(buf + g.x_bytes, codebook + slab0 * g.ngt * 16, bc, bar);
    } else {
        const int64_t slab = s >> g.chunk_log2;
        const int chunk = (int)(s & (g.nchunk - 1));
        mbar_expect_tx(bar, g.x_bytes + (uint32_t)(g.ngt * 64));
        const uint16_t *src = x + slab * 32 * (int64_t)g.D + (int64_t)chunk * g.Dc;
        for (int r = 0; r < 32; ++r)
            bulk_g2s(buf + r * g.Dc * 2, src + (int64_t)r * g.D, (uint32_t)(g.Dc * 2), bar);
        const int64_t blk0 = (slab << g.bps_log2) + (int64_t)chunk * g.ngt;
        bulk_g2s(buf + g.x_bytes, codebook + blk0 * 16, (uint32_t)(g.ngt * 64), bar);
    }
}

// blocks in stage s
__device__ __forceinline__ int t_blocks(const TGeom &g, int64_t s) {
    if (g.Dc < g.D) return g.ngt;
    return (int)min((int64_t)g.spt, g.nslabs - s * g.spt) * g.ngt;
}

// One warp builds quarter `qt` (bins 64 qt .. 64 qt + 63) of block `sl`'s
// table; quarter 0 also writes the decision pairs and the thresholds.  The
// thresholds are lanes 1 .. k-2 (level j in lane j); the bins holding one
// are marked in a 64-bit mask, and a bin's entry needs the thresholds below
// the quarter (a ballot) plus those marked below the bin (a popcount).  A
// mask with fewer bits than thresholds in the quarter means two thresholds
// share a bin: the quarter is flagged, and the block takes the search path.
__device__ __forceinline__ void t_build(TTables &tb, int par, int sl, int qt, const float *cb,
                                        int lane) {
    const float INF = __int_as_float(0x7f800000);
    const float qv = cb[sl * 16 + (lane & 15)];
    const float top = __shfl_sync(0xffffffffu, qv, 15);
    const int k = 1 + __popc(__ballot_sync(0xffffffffu, lane < 15 && qv < top));
    const bool th = lane >= 1 && lane <= k - 2;
    const uint32_t key = key16(qv);
    if (qt == 0 && lane < 16) {
        const float qn = __shfl_sync(0x0000ffffu, qv, min(lane + 1, 15), 16);
        const float thv = th ? qv : INF;
        const __half2 h2 = __floats2half2_rn(thv, thv);
        uint32_t hu;
        memcpy(&hu, &h2, 4);
        tb.thr[par][sl][lane] = hu;
        float ws = 0.f;
        if (k <= 1) ws = INF;
        else if (lane <= k - 2) ws = __fmul_rn(__fsub_rn(qn, qv), 5.9604644775390625e-8f);  // 2^-24
        tb.qw[par][sl][lane] = make_float2(-qv, ws);
    }
    const uint32_t lo = 64u * (uint32_t)qt;
    const uint32_t bin = key >> 8;
    const uint32_t base = __popc(__ballot_sync(0xffffffffu, th && bin < lo));
    const bool local = th && bin >= lo && bin < lo + 64u;
    const uint32_t li = bin - lo;
    const uint32_t mlo = __reduce_or_sync(0xffffffffu, local && li < 32u ? 1u << li : 0u);
    const uint32_t mhi = __reduce_or_sync(0xffffffffu, local && li >= 32u ? 1u << (li - 32u) : 0u);
    const uint64_t M = ((uint64_t)mhi << 32) | mlo;
    const int nloc = __popc(__ballot_sync(0xffffffffu, local));
    uint16_t *row = tb.bins[par][sl];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const uint32_t lb = 2u * (uint32_t)lane + (uint32_t)e;          // bin inside the quarter
        const uint32_t ib = base + (uint32_t)__popcll(M & ((1ull << lb) - 1ull));
        const bool in = (M >> lb) & 1ull;
        const uint32_t tk = __shfl_sync(0xffffffffu, key, (int)min(ib + 1u, 31u));
        const uint32_t t = in ? (tk & 0xFFu) : 256u;
        const uint32_t hb = lo + lb;
        row[hb] = (uint16_t)(((ib - hb) << 8) + 256u - t);
    }
    if (lane == 0) tb.slow[par][sl][qt] = (__popcll(M) != nloc) ? 1 : 0;
}

// Binary16 x (bits in the low or high half of w) minus q_i in one fp32
// round-to-nearest addition (the mixed-precision add converts x exactly).
__device__ __forceinline__ float2 sub_pair(uint32_t w, float nq0, float nq1) {
    float2 r;
    asm("{\n .reg .f16 a, b;\n mov.b32 {a, b}, %2;\n"
        " add.rn.f32.f16 %0, a, %3;\n add.rn.f32.f16 %1, b, %4;\n}"
        : "=f"(r.x), "=f"(r.y)
        : "r"(w), "f"(nq0), "f"(nq1));
    return r;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Codes of 8 consecutive entries through the bin table (binbase: the block's
// bin row, 512-byte aligned; qbase: its decision pairs, 128-byte aligned).
// The interval of the low entry of pair p lands in byte 1 of s0[p], that of
// the high entry in byte 3 of s1[p]; the rounding decision adds 1 to that
// byte, and byte permutes gather the eight code nibbles.
__device__ __forceinline__ uint32_t quant8_table(const uint4 raw, uint32_t binbase, uint32_t qbase,
                                                 uint32_t clo, uint32_t chi, const PhiloxKey &K) {
    const uint4 ha = philox7(clo, chi, K);
    const uint32_t clo1 = clo + 1u;
    const uint4 hb = philox7(clo1, chi + (clo1 == 0u ? 1u : 0u), K);
    uint32_t t0[4], t1[4];
#pragma unroll
    for (int pr = 0; pr < 4; ++pr) {
        const uint32_t w = pr == 0 ? raw.x : pr == 1 ? raw.y : pr == 2 ? raw.z : raw.w;
        const uint32_t key2 = key_pair(w);
        const uint32_t e0 = lds_u16(((key2 >> 7) & 0x1FEu) | binbase);
        const uint32_t e1 = lds_u16(((key2 >> 23) & 0x1FEu) | binbase);
        const uint32_t s0 = e0 + key2;                 // interval in bits 8..11
        const uint32_t s1 = (e1 << 16) + key2;         // interval in bits 24..27
        const float2 d0 = lds_f2(((s0 >> 5) & 0x78u) | qbase);
        const float2 d1 = lds_f2(((s1 >> 21) & 0x78u) | qbase);
        const uint32_t h0 = pr == 0 ? ha.x : pr == 1 ? ha.z : pr == 2 ? hb.x : hb.z;
        const uint32_t h1 = pr == 0 ? ha.y : pr == 1 ? ha.w : pr == 2 ? hb.y : hb.w;
        const float2 r = sub_pair(w, d0.x, d1.x);                          // x - q_i
        const float2 u = make_float2((float)(h0 >> 8), (float)(h1 >> 8));
        const float2 tw = __fmul2_rn(u, make_float2(d0.y, d1.y));
        t0[pr] = s0 + (tw.x < r.x ? 0x100u : 0u);
        t1[pr] = s1 + (tw.y < r.y ? 0x1000000u : 0u);
    }
    const uint32_t a = prmt(prmt(t0[0], t0[1], 0x0051u), prmt(t0[2], t0[3], 0x0051u), 0x5410u);
    const uint32_t b = prmt(prmt(t1[0], t1[1], 0x0073u), prmt(t1[2], t1[3], 0x0073u), 0x5410u);
    return a + (b << 4);
}

__global__ void __launch_bounds__(kTThreads, KVQ_QT_MINB)
quantize_table_kernel(const uint16_t *__restrict__ x, const float *__restrict__ codebook,
                      TGeom g, PhiloxKey K, uint64_t index_base, uint8_t *__restrict__ codes,
                      int32_t *__restrict__ status, uint32_t wait_polls) {
    extern __shared__ __align__(128) char qsm[];
    __shared__ __align__(8) uint64_t bars[kTStages];
    __shared__ __align__(1024) TTables tb;
    __shared__ int failed;
    __shared__ uint32_t issued[kTStages];      // copies issued into each stage buffer
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int kWarps = kTThreads / 32;
    if (tid == 0) {
        for (int s = 0; s < kTStages; ++s) {
            mbar_init(&bars[s], 1);
            issued[s] = 0u;
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        failed = 0;
    }
    __syncthreads();
    const int64_t s0 = blockIdx.x, sstep = gridDim.x;
    if (tid == 0) {
        for (int i = 0; i < kTStages; ++i) {
            const int64_t s = s0 + (int64_t)i * sstep;
            if (s < g.nstages) {
                t_issue(g, s, x, codebook, qsm + i * g.stage_bytes, &bars[i]);
                issued[i] = 1u;
            }
        }
    }
    // this thread's units: column cu, rows rg * upt .. rg * upt + upt - 1 (one slab)
    const int upr = 1 << g.upr_log2;
    const int cu = tid & (upr - 1);
    const int rg = tid >> g.upr_log2;
    const int row0 = rg * g.upt;
    const int sls = row0 >> 5;                           // slab inside the stage
    const int rin = row0 & 31;                           // first row inside the slab
    const int gt = (cu * 8) >> g.g_log2;                 // block inside the tile row
    const int slot = sls * g.ngt + gt;
    const int64_t hbytes = 16 * g.G;                     // code bytes per block
    const uint32_t xoff = (uint32_t)((row0 * g.Dc + cu * 8) << 1);
    const uint32_t xstep = (uint32_t)(g.Dc * 2);
    const uint32_t cstep = (uint32_t)(g.D >> 2);
    const int cbstep = g.G / 2;
    // tables of the first stage
    if (s0 < g.nstages) {
        if (!mbar_wait(&bars[0], 0u, wait_polls)) atomicOr(&failed, 1);
        const float *cb = reinterpret_cast<const float *>(qsm + g.x_bytes);
        const int ntask = 4 * t_blocks(g, s0);
        for (int q = warp; q < ntask; q += kWarps) t_build(tb, 0, q >> 2, q & 3, cb, lane);
    }
    __syncthreads();
    uint32_t n = 0;
    for (int64_t s = s0; s < g.nstages && !failed; s += sstep, ++n) {
        const uint32_t st = n % kTStages, par = n & 1u;
        char *buf = qsm + st * g.stage_bytes;
        // this stage: every thread observes its copy's completion
        if (!mbar_wait(&bars[st], (n / kTStages) & 1u, wait_polls)) atomicOr(&failed, 1);
        int64_t slab_g;
        int col;
        if (g.Dc == g.D) {
            slab_g = s * g.spt + sls;
            col = cu * 8;
        } else {
            slab_g = s >> g.chunk_log2;
            col = (int)(s & (g.nchunk - 1)) * g.Dc + cu * 8;
        }
        if (slab_g < g.nslabs) {
            const int64_t blk = (slab_g << g.bps_log2) + (col >> g.g_log2);
            uint32_t *cp = reinterpret_cast<uint32_t *>(codes + blk * hbytes +
                                                        ((rin * g.G + (col & (g.G - 1))) >> 1));
            const uint64_t c = (index_base + (uint64_t)((slab_g * 32 + rin) * (int64_t)g.D + col)) >> 2;
            uint32_t clo = (uint32_t)c, chi = (uint32_t)(c >> 32);
            const uint32_t xs = smem_addr(buf) + xoff;
            const int4 sl4 = *reinterpret_cast<const int4 *>(tb.slow[par][slot]);
            if ((sl4.x | sl4.y | sl4.z | sl4.w) == 0) {
                const uint32_t binbase = smem_addr(&tb.bins[par][slot][0]);
                const uint32_t qbase = smem_addr(&tb.qw[par][slot][0]);
#pragma unroll 4
                for (int j = 0; j < g.upt; ++j) {
                    uint4 raw;
                    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(raw.x), "=r"(raw.y), "=r"(raw.z), "=r"(raw.w)
                                 : "r"(xs + (uint32_t)j * xstep));
                    cp[j * (cbstep >> 2)] = quant8_table(raw, binbase, qbase, clo, chi, K);
                    const uint32_t nlo = clo + cstep;
                    chi += nlo < clo ? 1u : 0u;
                    clo = nlo;
                }
            } else {
                uint32_t T[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) T[j] = tb.thr[par][slot][j];
                const float2 *qw = tb.qw[par][slot];
                for (int j = 0; j < g.upt; ++j) {
                    const uint4 raw = *reinterpret_cast<const uint4 *>(buf + xoff + j * xstep);
                    cp[j * (cbstep >> 2)] = quant8(raw, T, qw, ((uint64_t)chi << 32) | clo, K);
                    const uint32_t nlo = clo + cstep;
                    chi += nlo < clo ? 1u : 0u;
                    clo = nlo;
                }
            }
        }
        // tables of the next stage (its copies were issued stages ago), split
        // over every warp by quarters of the bins
        const int64_t sn = s + sstep;
        if (sn < g.nstages) {
            const uint32_t nn = n + 1;
            const int ntask = 4 * t_blocks(g, sn);
            if (warp < ntask) {
                if (!mbar_wait(&bars[nn % kTStages], (nn / kTStages) & 1u, wait_polls))
                    atomicOr(&failed, 1);
                const float *cb = reinterpret_cast<const float *>(qsm + (nn % kTStages) * g.stage_bytes +
                                                                  g.x_bytes);
                for (int q = warp; q < ntask; q += kWarps)
                    t_build(tb, (int)(par ^ 1u), q >> 2, q & 3, cb, lane);
            }
        }
        __syncthreads();            // stage buffer and this parity's tables are free
        if (tid == 0 && !failed) {  // after a failed wait nothing more is issued
            const int64_t sf = s + (int64_t)kTStages * sstep;
            if (sf < g.nstages) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                t_issue(g, sf, x, codebook, buf, &bars[st]);
                ++issued[st];
            }
        }
    }
    if (failed) {
        // a wait gave up: report it, and give the last copy issued into each
        // stage buffer a bounded chance (the normal limit) to land before the
        // shared memory is released
        __syncthreads();
        if (tid == 0) {
            if (status) atomicExch(status, KVQ_ERR_TIMEOUT);
            for (int i = 0; i < kTStages; ++i)
                if (issued[i]) mbar_wait(&bars[i], (issued[i] - 1u) & 1u, kQWaitLimit);
        }
        __syncthreads();
    }
}

// =============================================================== search kernel
constexpr int kQThreads = 128;
constexpr int kQStages = 4;
constexpr int kQMaxCols = 256;               // features per tile (at most)
constexpr int kQMaxGroups = kQMaxCols / 8;   // blocks per tile (at most)

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
                int64_t ntiles, PhiloxKey K, uint64_t index_base, uint8_t *__restrict__ codes,
                int32_t *__restrict__ status, uint32_t wait_polls) {
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
        if (!mbar_wait(&bars[s], (n / kQStages) & 1u, wait_polls)) {
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
        uint64_t c = quant_counter(index_base, (uint64_t)((slab * 32 + row0) * (int64_t)g.D + col));
        const uint64_t cstep = (uint64_t)(rstep * g.D / 4);
        for (int row = row0; row < 32; row += rstep, c += cstep) {
            const uint4 raw = *reinterpret_cast<const uint4 *>(buf + (row * g.Dc + f0) * 2);
            uint32_t cw;
            if constexpr (NEAREST) cw = quant8_nearest(raw, T, qw);
            else cw = quant8(raw, T, qw, c, K);
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
static int g_table_grid[64];

static int lg2i(int v) {
    int l = 0;
    while ((1 << l) < v) ++l;
    return l;
}

static QGeom geometry(const kvq_layout &L) {
    QGeom g;
    g.D = L.D;
    g.G = L.group;
    g.Dc = L.D < kQMaxCols ? L.D : kQMaxCols;
    g.nchunk = L.D / g.Dc;
    g.ngt = g.Dc / g.G;
    g.upr_log2 = lg2i(g.Dc / 8);
    g.chunk_log2 = lg2i(g.nchunk);
    g.g_log2 = lg2i(g.G);
    g.bps_log2 = lg2i(g.D / g.G);
    g.x_bytes = (uint32_t)(64 * g.Dc);
    g.cb_bytes = (uint32_t)(64 * g.ngt);
    g.stage_bytes = (g.x_bytes + g.cb_bytes + 127u) & ~127u;
    return g;
}

static TGeom table_geometry(const kvq_layout &L) {
    TGeom g;
    g.D = L.D;
    g.G = L.group;
    g.Dc = L.D < 256 ? L.D : 256;
    g.nchunk = L.D / g.Dc;
    g.spt = g.Dc == g.D ? kTStageX / (64 * g.D) : 1;
    if (g.spt < 1) g.spt = 1;
    if (g.spt > 32) g.spt = 32;
    g.ngt = g.Dc / g.G;
    g.upr_log2 = lg2i(g.Dc / 8);
    const int rows = 32 * g.spt;                      // rows of a stage
    const int groups = kTThreads >> g.upr_log2;       // row groups of threads
    g.upt = rows / groups;
    g.g_log2 = lg2i(g.G);
    g.bps_log2 = lg2i(g.D / g.G);
    g.chunk_log2 = lg2i(g.nchunk);
    g.nslabs = L.S * (L.T / 32);
    g.nstages = g.Dc == g.D ? (g.nslabs + g.spt - 1) / g.spt : g.nslabs * g.nchunk;
    g.x_bytes = (uint32_t)(64 * g.Dc * g.spt);
    g.stage_bytes = (g.x_bytes + (uint32_t)(64 * g.ngt * g.spt) + 127u) & ~127u;
    return g;
}

// the table kernel covers this layout: blocks of >= 32 features, at most
// kTMaxBlocks blocks and at least one row per thread in a stage
static bool table_ok(const TGeom &g) {
    if (g.G < kTMinGroup) return false;
    if (g.ngt * g.spt > kTMaxBlocks) return false;
    const int rows = 32 * g.spt, groups = kTThreads >> g.upr_log2;
    if (groups < 1 || rows % groups != 0 || g.upt < 1 || 32 % g.upt != 0) return false;
    return true;
}

static constexpr int kTSmem = kTStages * (kTStageX + 64 * kTMaxBlocks);

int quantize_init() {
    int dev = 0, sms = 0, occ = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KVQ_ERR_CUDA;
    const int smem = kQStages * ((64 * kQMaxCols + 64 * kQMaxGroups + 127) & ~127);
    if (cudaFuncSetAttribute(quantize_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess ||
        cudaFuncSetAttribute(quantize_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess ||
        cudaFuncSetAttribute(quantize_table_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kTSmem) != cudaSuccess)
        return KVQ_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return KVQ_ERR_CUDA;
    // the grid for the llama-shaped tile size (8 KB + codebook per stage)
    const int smem128 = kQStages * ((64 * 128 + 64 + 127) & ~127);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, quantize_kernel<false>, kQThreads, smem128) !=
        cudaSuccess)
        return KVQ_ERR_CUDA;
    g_quant_grid[dev] = (occ < 1 ? 1 : occ) * sms;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, quantize_table_kernel, kTThreads, kTSmem) !=
            cudaSuccess ||
        occ < 1)
        return KVQ_ERR_CUDA;
    g_table_grid[dev] = occ * sms;
    return KVQ_OK;
}

int launch_quantize(const uint16_t *x, const kvq_layout &L, const float *codebook,
                    const uint8_t *k, uint64_t seed, uint64_t index_base, uint8_t *codes,
                    int32_t *status, cudaStream_t st, bool nearest) {
    (void)k;   // the kernels read k from the codebook (slots k..15 repeat the top level)
    if (L.S * (L.T / 32) == 0) return KVQ_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KVQ_ERR_CUDA;
    const PhiloxKey K = philox_key(seed);
    unsigned long long tw = 0;
    const uint32_t wait_polls = test_wait_limit(&tw) ? 0u : kQWaitLimit;
    if (!nearest) {
        const TGeom tg = table_geometry(L);
        if (table_ok(tg)) {
            int64_t grid = g_table_grid[dev] > 0 ? g_table_grid[dev] : 148;
            if (grid > tg.nstages) grid = tg.nstages;
            const size_t smem = (size_t)kTStages * tg.stage_bytes;
            quantize_table_kernel<<<(unsigned)grid, kTThreads, smem, st>>>(x, codebook, tg, K,
                                                                            index_base, codes,
                                                                            status, wait_polls);
            return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
        }
    }
    const QGeom g = geometry(L);
    const int64_t ntiles = L.S * (L.T / 32) * g.nchunk;
    int64_t grid = g_quant_grid[dev] > 0 ? g_quant_grid[dev] : 148;
    if (grid > ntiles) grid = ntiles;
    const size_t smem = (size_t)kQStages * g.stage_bytes;
    if (nearest)
        quantize_kernel<true><<<(unsigned)grid, kQThreads, smem, st>>>(x, codebook, g, ntiles, K,
                                                                       index_base, codes, status,
                                                                       wait_polls);
    else
        quantize_kernel<false><<<(unsigned)grid, kQThreads, smem, st>>>(x, codebook, g, ntiles, K,
                                                                        index_base, codes, status,
                                                                        wait_polls);
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
