// kvq_stats: per-block candidate levels (17 order statistics) and the
// interval statistics the allocation needs ("Rate-adaptive KV-cache
// quantizer", "Implementation notes": candidate alphabet from the minimum,
// maximum and quantiles; D_r from interval statistics).
//
// One CTA of 256 threads per block.  The block's binary16 entries are read
// once from HBM with 16-byte loads and kept in registers.  Order statistics
// come from a two-level radix select on the order-preserving 16-bit key:
//   pass 1  one 64-bit shared atomic per entry into the 256 bins of the key's
//           high byte; the word packs count (bits 48..60), sum of the low
//           byte j (28..47) and sum of j^2 (0..27) -- exact integers, no
//           field can carry into the next for d <= 4096;
//   scan    bin prefix counts locate the bin of each of the 17 ranks;
//   pass 2  entries of those (<= 17) bins count their low byte in a second
//           histogram (two 16-bit counters per 32-bit word);
//   select  one warp per selected bin finds the exact key of each rank and
//           the prefix sums of (1, j, j^2) below it.
// Inside a bin the value is affine in j (one binade quarter: fixed sign and
// exponent), so the atom moments follow from those integer sums without
// touching the entries again.  Every fp32 term added is non-negative, so the
// moments carry no cancellation.
#include "kvq_internal.cuh"

namespace kvq {

constexpr int kStatsThreads = 256;

struct StatsSmem {
    unsigned long long l1[256];
    uint32_t l2[17][128];
    int32_t pre[256];
    uint8_t binslot[256];
    int32_t warp_tot[8];
    int32_t rank_bin[17], rank_res[17], rank_slot[17];
    int32_t rank_key[17], rank_p0[17], rank_cnt[17];
    uint32_t rank_p1[17], rank_p2[17];
    int32_t dkey[17], dp0[17], dcnt[17];
    uint32_t dp1[17], dp2[17];
    float dc[17];
    int32_t mprime, nslots, flags;
    float an[16], as1[16], at1[16], ae[16];
};

__device__ __forceinline__ int block_excl_scan(int v, int32_t *warp_tot, int &total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[w] = x;
    __syncthreads();
    int off = 0, tot = 0;
#pragma unroll
    for (int k = 0; k < kStatsThreads / 32; ++k) {
        int t = warp_tot[k];
        off += (k < w) ? t : 0;
        tot += t;
    }
    total = tot;
    __syncthreads();
    return off + x - v;
}

// Add one piece (entries of bin b with key low byte in [j0, j1], integer sums
// n, S1 = sum j, S2 = sum j^2) to the moments of the atom [cp, cq).
__device__ __forceinline__ void add_piece(uint32_t b, int j0, int j1, uint32_t n,
                                          uint32_t S1, uint32_t S2, float cp, float cq,
                                          float &an, float &as1, float &at1, float &ae) {
    if (n == 0) return;
    const float u = bin_ulp(b);
    const float Y0 = key_value((b << 8) | (uint32_t)j0) - cp;   // >= 0
    const float T1 = cq - key_value((b << 8) | (uint32_t)j1);   // >= 0
    const long long L = j1 - j0;
    const long long nn = n;
    const long long si = (long long)S1 - (long long)j0 * nn;                          // sum i
    const long long sii = (long long)S2 - 2ll * j0 * (long long)S1 + (long long)j0 * j0 * nn;  // sum i^2
    const long long sli = L * nn - si;                                                 // sum (L - i)
    const long long sx = L * si - sii;                                                 // sum i (L - i)
    const float fn = (float)nn, fsi = (float)si, fsli = (float)sli, fsx = (float)sx;
    an += fn;
    as1 += fn * Y0 + u * fsi;
    at1 += fn * T1 + u * fsli;
    ae += fn * Y0 * T1 + Y0 * u * fsli + T1 * u * fsi + u * u * fsx;
}

template <int UNITS>
__global__ void __launch_bounds__(kStatsThreads)
stats_kernel(const uint16_t *__restrict__ x, kvq_layout L, StatsRow *__restrict__ out,
             int32_t *__restrict__ status) {
    __shared__ StatsSmem sm;
    const int tid = threadIdx.x;
    const int G = L.group, D = L.D;
    const int d = 32 * G;
    const int nG = D / G;
    const int64_t blk = blockIdx.x;
    const int g = (int)(blk % nG);
    const int64_t tbk = blk / nG;                       // stream * nTB + token block
    const int units = d / 8, upr = G / 8;               // 8-entry units, units per row

    // zero histograms
    sm.l1[tid] = 0ull;
    for (int i = tid; i < 17 * 128; i += kStatsThreads) (&sm.l2[0][0])[i] = 0u;
    if (tid == 0) sm.flags = 0;

    // ---- load: UNITS 16-byte units per thread, kept in registers
    uint4 raw[UNITS];
#pragma unroll
    for (int k = 0; k < UNITS; ++k) {
        const int u = tid + k * kStatsThreads;
        raw[k] = make_uint4(0, 0, 0, 0);
        if (u < units) {
            const int row = u / upr, cu = u % upr;
            const int64_t off = (tbk * 32 + row) * (int64_t)D + (int64_t)g * G + cu * 8;
            raw[k] = __ldg(reinterpret_cast<const uint4 *>(x + off));
        }
    }
    __syncthreads();

    // ---- pass 1: level-1 histogram with exact (count, sum j, sum j^2)
    int bad = 0;
#pragma unroll
    for (int k = 0; k < UNITS; ++k) {
        const int u = tid + k * kStatsThreads;
        if (u >= units) continue;
        const uint32_t w4[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const uint32_t h = (w4[q >> 1] >> ((q & 1) * 16)) & 0xffffu;
            bad |= ((h & 0x7c00u) == 0x7c00u);
            const uint32_t key = f16_key(h);
            const uint32_t j = key & 255u;
            atomicAdd(&sm.l1[key >> 8],
                      (1ull << 48) | ((unsigned long long)j << 28) | (unsigned long long)(j * j));
        }
    }
    if (bad) atomicOr(&sm.flags, kFlagNonfinite);
    __syncthreads();

    // ---- bin prefix counts, ranks -> bins, bins -> slots
    const unsigned long long v1 = sm.l1[tid];
    const int cnt = (int)(v1 >> 48);
    int total;
    const int pre = block_excl_scan(cnt, sm.warp_tot, total);
    sm.pre[tid] = pre;
    bool tgt = false;
#pragma unroll
    for (int j = 0; j < kCand; ++j) {
        const int r = (j * (d - 1) + 8) >> 4;
        if (r >= pre && r < pre + cnt) {
            tgt = true;
            sm.rank_bin[j] = tid;
            sm.rank_res[j] = r - pre;
        }
    }
    int nslots;
    const int slot = block_excl_scan(tgt ? 1 : 0, sm.warp_tot, nslots);
    sm.binslot[tid] = tgt ? (uint8_t)slot : (uint8_t)0xff;
    if (tid == 0) sm.nslots = nslots;
    __syncthreads();
    if (tid < kCand) sm.rank_slot[tid] = sm.binslot[sm.rank_bin[tid]];

    // ---- pass 2: per-key counts inside the selected bins
#pragma unroll
    for (int k = 0; k < UNITS; ++k) {
        const int u = tid + k * kStatsThreads;
        if (u >= units) continue;
        const uint32_t w4[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const uint32_t key = f16_key((w4[q >> 1] >> ((q & 1) * 16)) & 0xffffu);
            const uint32_t s = sm.binslot[key >> 8];
            if (s != 0xffu) atomicAdd(&sm.l2[s][(key & 255u) >> 1], 1u << ((key & 1u) * 16));
        }
    }
    __syncthreads();

    // ---- exact key of every rank + prefix sums below it inside its bin
    {
        const int lane = tid & 31, w = tid >> 5;
        for (int s = w; s < sm.nslots; s += kStatsThreads / 32) {
            uint32_t c8[8];
            uint32_t n = 0, S1 = 0, S2 = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t wd = sm.l2[s][lane * 4 + q];
                c8[2 * q] = wd & 0xffffu;
                c8[2 * q + 1] = wd >> 16;
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const uint32_t jj = lane * 8 + q;
                n += c8[q];
                S1 += c8[q] * jj;
                S2 += c8[q] * jj * jj;
            }
            uint32_t en = n, e1 = S1, e2 = S2;   // inclusive scans
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t a = __shfl_up_sync(0xffffffffu, en, o);
                const uint32_t b = __shfl_up_sync(0xffffffffu, e1, o);
                const uint32_t c = __shfl_up_sync(0xffffffffu, e2, o);
                if (lane >= o) { en += a; e1 += b; e2 += c; }
            }
            en -= n; e1 -= S1; e2 -= S2;         // exclusive
            for (int j = 0; j < kCand; ++j) {
                if (sm.rank_slot[j] != s) continue;
                const uint32_t res = (uint32_t)sm.rank_res[j];
                if (res >= en && res < en + n) {
                    uint32_t cum = en, p1 = e1, p2 = e2;
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const uint32_t jj = lane * 8 + q;
                        if (res < cum + c8[q]) {
                            sm.rank_key[j] = (sm.rank_bin[j] << 8) | (int)jj;
                            sm.rank_p0[j] = (int)cum;
                            sm.rank_p1[j] = p1;
                            sm.rank_p2[j] = p2;
                            sm.rank_cnt[j] = (int)c8[q];
                            break;
                        }
                        cum += c8[q];
                        p1 += c8[q] * jj;
                        p2 += c8[q] * jj * jj;
                    }
                }
            }
        }
    }
    __syncthreads();

    // ---- merge equal candidates
    if (tid == 0) {
        int mp = 0;
        for (int j = 0; j < kCand; ++j) {
            const int key = sm.rank_key[j];
            if (mp == 0 || key != sm.dkey[mp - 1]) {
                sm.dkey[mp] = key;
                sm.dp0[mp] = sm.rank_p0[j];
                sm.dp1[mp] = sm.rank_p1[j];
                sm.dp2[mp] = sm.rank_p2[j];
                sm.dcnt[mp] = sm.rank_cnt[j];
                sm.dc[mp] = key_value((uint32_t)key);
                ++mp;
            }
        }
        sm.mprime = mp;
    }
    __syncthreads();

    // ---- atom moments, one thread per atom, bins in increasing order
    const int mp = sm.mprime;
    if (tid < 16) {
        float an = 0.f, as1 = 0.f, at1 = 0.f, ae = 0.f;
        const int p = tid;
        if (p < mp - 1) {
            const bool last = (p == mp - 2);
            const uint32_t Klo = (uint32_t)sm.dkey[p], Khi = (uint32_t)sm.dkey[p + 1];
            const uint32_t blo = Klo >> 8, bhi = Khi >> 8;
            const int jlo = (int)(Klo & 255u), jhi = (int)(Khi & 255u);
            const float cp = sm.dc[p], cq = sm.dc[p + 1];
            // prefix sums (over keys < X of X's bin) at the two ends
            const uint32_t lo0 = sm.dp0[p], lo1 = sm.dp1[p], lo2 = sm.dp2[p];
            uint32_t hi0 = sm.dp0[p + 1], hi1 = sm.dp1[p + 1], hi2 = sm.dp2[p + 1];
            int jend = jhi - 1;
            if (last) {   // the maximum itself belongs to the last atom
                const uint32_t c = (uint32_t)sm.dcnt[p + 1];
                hi0 += c;
                hi1 += c * (uint32_t)jhi;
                hi2 += c * (uint32_t)jhi * (uint32_t)jhi;
                jend = jhi;
            }
            if (blo == bhi) {
                add_piece(blo, jlo, jend, hi0 - lo0, hi1 - lo1, hi2 - lo2, cp, cq, an, as1, at1, ae);
            } else {
                const unsigned long long t = sm.l1[blo];
                add_piece(blo, jlo, 255, (uint32_t)(t >> 48) - lo0,
                          (uint32_t)((t >> 28) & 0xfffffu) - lo1, (uint32_t)(t & 0xfffffffu) - lo2,
                          cp, cq, an, as1, at1, ae);
                for (uint32_t b = blo + 1; b < bhi; ++b) {
                    const unsigned long long v = sm.l1[b];
                    if ((v >> 48) == 0) continue;
                    add_piece(b, 0, 255, (uint32_t)(v >> 48), (uint32_t)((v >> 28) & 0xfffffu),
                              (uint32_t)(v & 0xfffffffu), cp, cq, an, as1, at1, ae);
                }
                if (jend >= 0) add_piece(bhi, 0, jend, hi0, hi1, hi2, cp, cq, an, as1, at1, ae);
            }
        }
        sm.an[tid] = an;
        sm.as1[tid] = as1;
        sm.at1[tid] = at1;
        sm.ae[tid] = ae;
    }
    __syncthreads();

    // ---- write the row (96 words)
    if (tid < 96) {
        float *row = reinterpret_cast<float *>(out + blk);
        float v = 0.f;
        if (tid < 17) v = sm.dc[tid < mp ? tid : mp - 1];
        else if (tid == 17) v = __int_as_float(mp);
        else if (tid == 18) v = __int_as_float(sm.flags);
        else if (tid == 19) v = __int_as_float(d);
        else if (tid < 36) v = sm.an[tid - 20];
        else if (tid < 52) v = sm.as1[tid - 36];
        else if (tid < 68) v = sm.at1[tid - 52];
        else if (tid < 84) v = sm.ae[tid - 68];
        row[tid] = v;
    }
    if (tid == 0 && sm.flags) atomicMax(status, (int32_t)KVQ_ERR_NONFINITE);
}

int launch_stats(const uint16_t *x, const kvq_layout &L, void *stats, int32_t *status,
                 cudaStream_t st) {
    const int64_t nb = num_blocks(L);
    if (cudaMemsetAsync(status, 0, sizeof(int32_t), st) != cudaSuccess) return KVQ_ERR_CUDA;
    if (nb == 0) return KVQ_OK;
    const int units = 4 * L.group;   // 8-entry units per block
    StatsRow *out = static_cast<StatsRow *>(stats);
    const dim3 grid((unsigned)nb);
    if (units <= kStatsThreads)
        stats_kernel<1><<<grid, kStatsThreads, 0, st>>>(x, L, out, status);
    else
        stats_kernel<2><<<grid, kStatsThreads, 0, st>>>(x, L, out, status);
    return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq
