// kvq_stats: per-block candidate levels (17 order statistics) and the
// interval statistics the allocation needs ("Rate-adaptive KV-cache
// quantizer", "Implementation notes": candidate alphabet from the minimum,
// maximum and quantiles; D_r from interval statistics).
//
// One CTA of 256 threads per block.  The block's binary16 entries are read
// once from HBM with 16-byte loads; their order-preserving 16-bit keys stay in
// registers.  Order statistics come from a two-level radix select:
//   pass 1  each half of the CTA (4 warps) histograms its entries by the key's
//           high byte into its own 256-bin table: one 32-bit shared atomic
//           adds (1 << 20) | j (count in bits 20..31, sum of the low byte j in
//           0..19; a half holds at most 2048 entries, so neither field can
//           overflow) and a second adds j^2.  The 2 tables are merged per bin;
//   scan    bin prefix counts locate the bin of each of the 17 ranks;
//   pass 2  entries of those (<= 17) bins count their low byte in a second
//           histogram (two 16-bit counters per 32-bit word);
//   select  one warp per selected bin sums (1, j, j^2) over each chunk of 8
//           keys and scans the chunk sums; then one lane per rank finds its
//           chunk by a binary search of the prefix counts and its key inside
//           the chunk, with the prefix sums of (1, j, j^2) below it.
// Inside a bin the value is affine in j (one binade quarter: fixed sign and
// exponent), so the atom moments follow from those exact integer sums without
// touching the entries again: half a warp per atom sums its bins with a
// fixed-order tree.  The CTA then builds the block's lambda-independent DP
// tables (interval distortion and entropy terms, one entropy log2 per level
// triple) and writes them with the stats row as the block's record.  Every
// fp32 term added is non-negative, so there is no cancellation.
// Non-finite entries are the keys of the four lowest and four highest bins.
#include "kvq_internal.cuh"

namespace kvq {

constexpr int kStatsThreads = 256;
constexpr int kStatsWarps = kStatsThreads / 32;
constexpr int kHistTables = 2;      // first-pass histograms, one per 4 warps

struct StatsSmem {
    union {
        struct {
            uint32_t h1a[kHistTables][256];   // per half of the CTA: (count << 20) | sum j
            uint32_t h1b[kHistTables][256];   // per half of the CTA: sum j^2
        };
        struct {
            uint32_t l2[17][128];             // after the merge: low-byte counts
            // per selected bin and 8-key chunk: counts, sum j and sum j^2
            // of the keys in the chunks before it
            uint32_t cpn[17][32], cps1[17][32], cps2[17][32];
        };
    };
    int32_t cnt[256];
    uint32_t s1[256], s2[256];
    float bv0[256], bu[256];      // per bin: value of low byte 0, spacing of keys
    uint8_t binslot[256];
    int32_t warp_tot[kStatsWarps];
    int32_t rank_bin[17], rank_res[17];
    int32_t dkey[17], dp0[17], dcnt[17];
    uint32_t dp1[17], dp2[17];
    float dc[17];
    int32_t mprime, nslots;
    float4 atom[16];                  // per atom: n, s1, t1, e
    float pDp[kPairs], pUp[kPairs], pDn[kPairs];   // pair tables, slot space
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

// Add one piece (entries of a bin with key low byte in [j0, j1], integer sums
// n, S1 = sum j, S2 = sum j^2) to the moments of the atom [cp, cq).  v0, u:
// the bin's value at low byte 0 and its key spacing; the value at low byte j
// is v0 + j u, exact in binary32 (a binary16 value of the bin).
__device__ __forceinline__ void add_piece(float v0, float u, int j0, int j1, uint32_t n,
                                          uint32_t S1, uint32_t S2, float cp, float cq,
                                          float &an, float &as1, float &at1, float &ae) {
    if (n == 0) return;
    const float Y0 = fmaf((float)j0, u, v0) - cp;   // >= 0
    const float T1 = cq - fmaf((float)j1, u, v0);   // >= 0
    // integer sums of i = j - j0 over the piece; every true value lies in
    // [0, 2^32), so 32-bit modular arithmetic gives it exactly
    const uint32_t L = (uint32_t)(j1 - j0), u0 = (uint32_t)j0;
    const uint32_t nn = n;
    const uint32_t si = S1 - u0 * nn;                               // sum i
    const uint32_t sii = S2 - 2u * u0 * S1 + u0 * u0 * nn;          // sum i^2
    const uint32_t sli = L * nn - si;                               // sum (L - i)
    const uint32_t sx = L * si - sii;                               // sum i (L - i)
    const float fn = (float)nn, fsi = (float)si, fsli = (float)sli, fsx = (float)sx;
    an += fn;
    as1 += fn * Y0 + u * fsi;
    at1 += fn * T1 + u * fsli;
    ae += fn * Y0 * T1 + Y0 * u * fsli + T1 * u * fsi + u * u * fsx;
}

template <int UNITS>
__global__ void __launch_bounds__(kStatsThreads, 8)
stats_kernel(const uint16_t *__restrict__ x, kvq_layout L, int lg_ng, int lg_upr,
             StatsHeader *__restrict__ hdr, float *__restrict__ recs,
             int32_t *__restrict__ status) {
    __shared__ __align__(16) StatsSmem sm;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = L.group, D = L.D;
    const int d = 32 * G;
    const int nG = D / G;
    const int64_t blk = blockIdx.x;
    const int g = (int)(blk & (nG - 1));                // nG, G are powers of two
    const int64_t tbk = blk >> lg_ng;                   // stream * (T/32) + token block
    const int units = d / 8, upr = G / 8;               // 8-entry units, units per row

    // ---- load: UNITS 16-byte units per thread
    uint4 raw[UNITS];
#pragma unroll
    for (int k = 0; k < UNITS; ++k) {
        const int u = tid + k * kStatsThreads;
        raw[k] = make_uint4(0, 0, 0, 0);
        if (u < units) {
            const int row = u >> lg_upr, cu = u & (upr - 1);
            const int64_t off = (tbk * 32 + row) * (int64_t)D + (int64_t)g * G + cu * 8;
            raw[k] = __ldg(reinterpret_cast<const uint4 *>(x + off));
        }
    }
    // zero the tables while the loads are in flight
    {
        uint4 *z = reinterpret_cast<uint4 *>(&sm.h1a[0][0]);
        for (int i = tid; i < 2 * kHistTables * 256 / 4; i += kStatsThreads) z[i] = make_uint4(0, 0, 0, 0);
        if (tid < kPairs) {
            sm.pDp[tid] = __int_as_float(0x7f800000);   // +inf: no such pair
            sm.pUp[tid] = 0.f;
            sm.pDn[tid] = 0.f;
        }
    }
    __syncthreads();

    // ---- keys (two per register) and pass 1 into the half's table
    uint32_t keys[UNITS][4];
    const int ht = warp / (kStatsWarps / kHistTables);
#pragma unroll
    for (int k = 0; k < UNITS; ++k) {
        const int u = tid + k * kStatsThreads;
        const uint32_t w4[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t kk = f16_key2(w4[q]);
            keys[k][q] = kk;
            if (u < units) {
                const uint32_t b0 = (kk >> 8) & 255u, j0 = kk & 255u;
                const uint32_t b1 = kk >> 24, j1 = (kk >> 16) & 255u;
                atomicAdd(&sm.h1a[ht][b0], (1u << 20) | j0);
                atomicAdd(&sm.h1b[ht][b0], j0 * j0);
                atomicAdd(&sm.h1a[ht][b1], (1u << 20) | j1);
                atomicAdd(&sm.h1b[ht][b1], j1 * j1);
            }
        }
    }
    __syncthreads();

    // ---- merge the two tables (thread = bin), prefix counts, rank -> bin
    int cnt = 0;
    uint32_t S1 = 0, S2 = 0;
#pragma unroll
    for (int h = 0; h < kHistTables; ++h) {
        const uint32_t a = sm.h1a[h][tid];
        cnt += (int)(a >> 20);
        S1 += a & 0xfffffu;
        S2 += sm.h1b[h][tid];
    }
    sm.cnt[tid] = cnt;
    sm.s1[tid] = S1;
    sm.s2[tid] = S2;
    sm.binslot[tid] = 0xff;                          // not selected (yet)
    sm.bv0[tid] = key_value((uint32_t)tid << 8);     // bin tid: value at j = 0 and spacing
    sm.bu[tid] = bin_ulp((uint32_t)tid);
    int total;
    const int pre = block_excl_scan(cnt, sm.warp_tot, total);
    // both tables have been read: their memory becomes the low-byte table
    {
        uint4 *z2 = reinterpret_cast<uint4 *>(&sm.l2[0][0]);
        for (int i = tid; i < 17 * 128 / 4; i += kStatsThreads) z2[i] = make_uint4(0, 0, 0, 0);
    }
    // ranks r_j = floor((j (d-1) + 8) / 16) inside [pre, pre + cnt):
    // r_j >= pre  <=>  j (d-1) >= 16 pre - 8;  r_j < pre + cnt  <=>
    // j (d-1) <= 16 (pre + cnt) - 9
    int jlo = 17, jhi = -1;
    if (cnt > 0) {
        // floor(v / (d-1)) for 0 <= v < 2^20: a single-precision estimate
        // (off by at most one) corrected with exact integer products
        const int dm1 = d - 1;
        const float inv = 1.0f / (float)dm1;
        auto fdiv = [&](int v) {
            int q = (int)((float)v * inv);
            if (q * dm1 > v) --q;
            if ((q + 1) * dm1 <= v) ++q;
            return q;
        };
        const int a = 16 * pre - 8, bnd = 16 * (pre + cnt) - 9;
        jlo = a <= 0 ? 0 : fdiv(a + dm1 - 1);
        jhi = bnd < 0 ? -1 : min(fdiv(bnd), kCand - 1);
    }
    for (int j = jlo; j <= jhi; ++j) {
        sm.rank_bin[j] = tid;
        sm.rank_res[j] = ((j * (d - 1) + 8) >> 4) - pre;
    }
    __syncthreads();
    // the selected bins get slots 0, 1, .. in bin order: lane j = rank j (the
    // ranks' bins are non-decreasing), a slot for each first lane of a bin
    if (warp == 0) {
        const int bin = lane < kCand ? sm.rank_bin[lane] : -1;
        const int prev = __shfl_up_sync(0xffffffffu, bin, 1);
        const bool first = lane < kCand && (lane == 0 || bin != prev);
        const uint32_t bal = __ballot_sync(0xffffffffu, first);
        if (first) sm.binslot[bin] = (uint8_t)__popc(bal & ((1u << lane) - 1u));
        if (lane == 0) sm.nslots = __popc(bal);
    }
    __syncthreads();

    // ---- pass 2: per-key counts inside the selected bins
#pragma unroll
    for (int k = 0; k < UNITS; ++k) {
        const int u = tid + k * kStatsThreads;
        if (u >= units) continue;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const uint32_t key = (keys[k][q >> 1] >> ((q & 1) * 16)) & 0xffffu;
            const uint32_t sl = sm.binslot[key >> 8];
            if (sl != 0xffu) atomicAdd(&sm.l2[sl][(key & 255u) >> 1], 1u << ((key & 1u) * 16));
        }
    }
    __syncthreads();

    // ---- per selected bin, a warp with one lane per chunk of 8 keys (lane l
    //      holds keys 8l .. 8l+7): the chunk's count, sum j and sum j^2, and
    //      their exclusive prefixes over the chunks
    for (int sl = warp; sl < sm.nslots; sl += kStatsWarps) {
        const uint4 wd = reinterpret_cast<const uint4 *>(sm.l2[sl])[lane];
        const uint32_t w4[4] = {wd.x, wd.y, wd.z, wd.w};
        uint32_t n = 0, s1 = 0, s2 = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const uint32_t c = (w4[q >> 1] >> ((q & 1) * 16)) & 0xffffu;
            const uint32_t jj = (uint32_t)(lane * 8 + q);
            n += c;
            s1 += c * jj;
            s2 += c * jj * jj;
        }
        uint32_t en = n, e1 = s1, e2 = s2;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t a = __shfl_up_sync(0xffffffffu, en, o);
            const uint32_t b = __shfl_up_sync(0xffffffffu, e1, o);
            const uint32_t c = __shfl_up_sync(0xffffffffu, e2, o);
            if (lane >= o) {
                en += a;
                e1 += b;
                e2 += c;
            }
        }
        sm.cpn[sl][lane] = en - n;
        sm.cps1[sl][lane] = e1 - s1;
        sm.cps2[sl][lane] = e2 - s2;
    }
    __syncthreads();

    // ---- warp 0, lane j = rank j: its key is the first of its bin whose
    //      inclusive prefix count exceeds the rank's residual; the chunk that
    //      holds it is the last whose exclusive prefix does not, then the keys
    //      of that chunk in order.  P0, P1, P2: count, sum j, sum j^2 of the
    //      bin's entries below the key; cnt: the entries equal to it.  Equal
    //      candidates are then merged.
    if (warp == 0) {
        int key = -1;
        uint32_t P0 = 0, P1 = 0, P2 = 0, cnt = 0;
        if (lane < kCand) {
            const int bin = sm.rank_bin[lane];
            const uint32_t res = (uint32_t)sm.rank_res[lane];
            const int sl = sm.binslot[bin];
            int ch = 0;                       // cpn[sl][0] = 0 <= res; ch + step <= 31
#pragma unroll
            for (int step = 16; step > 0; step >>= 1)
                if (sm.cpn[sl][ch + step] <= res) ch += step;
            const uint4 wd = reinterpret_cast<const uint4 *>(sm.l2[sl])[ch];
            const uint32_t w4[4] = {wd.x, wd.y, wd.z, wd.w};
            uint32_t e = sm.cpn[sl][ch], p1 = sm.cps1[sl][ch], p2 = sm.cps2[sl][ch];
            int kq = 7;
            bool found = false;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const uint32_t c = (w4[q >> 1] >> ((q & 1) * 16)) & 0xffffu;
                const uint32_t jj = (uint32_t)(ch * 8 + q);
                if (!found) {
                    if (e + c > res) {
                        found = true;
                        kq = q;
                        cnt = c;
                    } else {
                        e += c;
                        p1 += c * jj;
                        p2 += c * jj * jj;
                    }
                }
            }
            key = (bin << 8) | (ch * 8 + kq);
            P0 = e;
            P1 = p1;
            P2 = p2;
        }
        const int prev_raw = __shfl_up_sync(0xffffffffu, key, 1);
        const int prev = (lane >= 1 && lane < kCand) ? prev_raw : -2;
        const bool first = lane < kCand && key != prev;
        const uint32_t bal = __ballot_sync(0xffffffffu, first);
        if (first) {
            const int p = __popc(bal & ((1u << lane) - 1u));
            sm.dkey[p] = key;
            sm.dp0[p] = (int)P0;
            sm.dp1[p] = P1;
            sm.dp2[p] = P2;
            sm.dcnt[p] = (int)cnt;
            sm.dc[p] = key_value((uint32_t)key);
        }
        if (lane == 0) sm.mprime = __popc(bal);
    }
    __syncthreads();

    // ---- atom moments: half a warp per atom (16 atoms in one pass over the 8
    //      warps).  Sub-lane 0 takes the piece above the atom's lower
    //      candidate (or the whole atom when both candidates share a bin),
    //      sub-lane 1 the piece below its upper candidate, sub-lanes 2..15 the
    //      bins strictly between; a fixed-order 16-lane tree sums them.
    const int mp = sm.mprime;
    {
        const int p = 2 * warp + (lane >> 4), sub = lane & 15;
        float an = 0.f, as1 = 0.f, at1 = 0.f, ae = 0.f;
        if (p < mp - 1) {
            const bool last = (p == mp - 2);
            const uint32_t Klo = (uint32_t)sm.dkey[p], Khi = (uint32_t)sm.dkey[p + 1];
            const uint32_t blo = Klo >> 8, bhi = Khi >> 8;
            const float cp = sm.dc[p], cq = sm.dc[p + 1];
            // this sub-lane's first piece (n = 0: none)
            uint32_t b = blo, n = 0, S1 = 0, S2 = 0;
            int j0 = 0, j1 = 255;
            if (sub >= 2) {
                const uint32_t bb = blo + (uint32_t)sub - 1u;
                if (bb < bhi) {
                    b = bb;
                    n = (uint32_t)sm.cnt[b];
                    S1 = sm.s1[b];
                    S2 = sm.s2[b];
                }
            } else {
                const int jlo = (int)(Klo & 255u), jhi = (int)(Khi & 255u);
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
                if (sub == 0) {
                    j0 = jlo;
                    if (blo == bhi) {
                        j1 = jend;
                        n = hi0 - lo0;
                        S1 = hi1 - lo1;
                        S2 = hi2 - lo2;
                    } else {
                        n = (uint32_t)sm.cnt[blo] - lo0;
                        S1 = sm.s1[blo] - lo1;
                        S2 = sm.s2[blo] - lo2;
                    }
                } else if (blo != bhi && jend >= 0) {
                    b = bhi;
                    j1 = jend;
                    n = hi0;
                    S1 = hi1;
                    S2 = hi2;
                }
            }
            add_piece(sm.bv0[b], sm.bu[b], j0, j1, n, S1, S2, cp, cq, an, as1, at1, ae);
            if (sub >= 2) {   // the rest of the bins strictly between, 14 apart
                for (uint32_t bb = blo + (uint32_t)sub + 13u; bb < bhi; bb += 14u) {
                    const uint32_t c = (uint32_t)sm.cnt[bb];
                    if (c) add_piece(sm.bv0[bb], sm.bu[bb], 0, 255, c, sm.s1[bb], sm.s2[bb], cp, cq,
                                     an, as1, at1, ae);
                }
            }
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) {
            an += __shfl_down_sync(0xffffffffu, an, o, 16);
            as1 += __shfl_down_sync(0xffffffffu, as1, o, 16);
            at1 += __shfl_down_sync(0xffffffffu, at1, o, 16);
            ae += __shfl_down_sync(0xffffffffu, ae, o, 16);
        }
        if (sub == 0 && p < 16) sm.atom[p] = make_float4(an, as1, at1, ae);
    }
    __syncthreads();

    // ---- pair tables in slot space (candidates 0 .. m'-2 in slots 0 .., the
    //      maximum in slot 16): for a = c_P < b = c_Q, over the atoms p of
    //      [a, b) with A = c_p - a, B = b - c_{p+1}:
    //        D = sum n A B + A t1 + B s1 + e      (sum of (b - x)(x - a))
    //        Mup = sum (s1 + n A) / (b - a)        (expected count sent to b)
    //        Mdn = sum (t1 + n B) / (b - a)        (expected count sent to a)
    //      every term non-negative
    //      Pairs in order of decreasing length Q - P, so that the threads of
    //      a warp run loops of similar length: thread t takes the P-th of the
    //      u pairs of length m' - u, u(u-1)/2 <= t < u(u+1)/2.
    const int npr = mp * (mp - 1) / 2;
    if (tid < npr) {
        int u = (int)((1.0f + sqrtf(1.0f + 8.0f * (float)tid)) * 0.5f);
        if (u * (u - 1) / 2 > tid) --u;
        if ((u + 1) * u / 2 <= tid) ++u;
        const int P = tid - u * (u - 1) / 2;
        const int Q = P + mp - u;
        const float a = sm.dc[P], bq = sm.dc[Q];
        float Dv = 0.f, Us = 0.f, Ls = 0.f;
        for (int p = P; p < Q; ++p) {
            const float4 at = sm.atom[p];
            const float n = at.x, s1 = at.y, t1 = at.z, e = at.w;
            const float A = sm.dc[p] - a, Bq = bq - sm.dc[p + 1];
            Dv += n * A * Bq + A * t1 + Bq * s1 + e;
            Us += s1 + n * A;
            Ls += t1 + n * Bq;
        }
        const float W = bq - a;
        const int sj = P == mp - 1 ? 16 : P, sl = Q == mp - 1 ? 16 : Q;
        const int o = pidx(sj, sl);
        sm.pDp[o] = Dv;
        sm.pUp[o] = Us / W;
        sm.pDn[o] = Ls / W;
    }
    __syncthreads();

    // ---- the record: stats row, then the DP tables
    //      (non-finite keys live in bins 0..3 and 252..255)
    const bool bad = (sm.cnt[0] | sm.cnt[1] | sm.cnt[2] | sm.cnt[3] | sm.cnt[252] | sm.cnt[253] |
                      sm.cnt[254] | sm.cnt[255]) != 0;
    float *rec = recs + blk * kRecFloats;
    if (tid < 96) {
        float v = 0.f;
        if (tid < 17) v = sm.dc[tid < mp ? tid : mp - 1];
        else if (tid == 17) v = __int_as_float(mp);
        else if (tid == 18) v = __int_as_float(bad ? kFlagNonfinite : 0);
        else if (tid == 19) v = __int_as_float(d);
        else if (tid < 36) v = sm.atom[tid - 20].x;
        else if (tid < 52) v = sm.atom[tid - 36].y;
        else if (tid < 68) v = sm.atom[tid - 52].z;
        else if (tid < 84) v = sm.atom[tid - 68].w;
        rec[tid] = v;
    }
    float *tb = rec + kRecTbl;
    const float inv_d = 1.0f / (float)d;
    auto real = [&](int t) { return t < mp - 1 || t == 16; };
    // the hardware base-2 logarithm (about 2^-22 absolute error on [0.5, 2], 2 ulp
    // elsewhere): an entropy term's error is at most 2^-22 M, so a block's
    // d_r H_r moves by less than 2^-22 d_r bits, far inside the DP's fp32
    // rounding of the same sums
    auto hterm = [&](float M) { return M > 0.f ? -M * __log2f(M * inv_d) : 0.f; };
    // slots that hold a candidate (0 .. m'-2, and 16 for the maximum)
    const uint32_t realm = mp > 1 ? (((1u << (mp - 1)) - 1u) | (1u << 16)) : 0u;
    // the hh and D tables in 16-byte pieces: rows are padded to multiples of
    // 4, so the 4 entries of a piece share one row -- i and j (hh) or j (D),
    // with l = l0 .. l0+3 and consecutive pair indices
    constexpr int kHHq = kHHFloats / 4, kDq = kDpFloats / 4;
    for (int q = tid; q < kHHq + kDq; q += kStatsThreads) {
        float v[4];
        if (q < kHHq) {
            const uint32_t dcd = kDecode.trip[4 * q];
            const uint32_t i = (dcd >> 16) & 31u, j = (dcd >> 21) & 31u, l0 = dcd >> 26;
            const bool ij = ((realm >> i) & (realm >> j) & 1u) != 0u;
            const float up = sm.pUp[dcd & 255u];
            const uint32_t pj = (dcd >> 8) & 255u;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t l = l0 + (uint32_t)k;
                v[k] = 0.f;
                if (ij && l < 17u && ((realm >> l) & 1u))
                    v[k] = hterm(up + sm.pDn[min(pj + (uint32_t)k, (uint32_t)kPairs - 1u)]);
            }
            *reinterpret_cast<float4 *>(tb + kTblHH + 4 * q) = make_float4(v[0], v[1], v[2], v[3]);
        } else {
            const int r = q - kHHq;
            const uint32_t dcd = kDecode.pair[4 * r];
            const int j = dcd & 255, l0 = dcd >> 8;
            const int base = l0 < 17 ? pidx(j, l0) : 0;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                v[k] = l0 + k < 17 ? sm.pDp[min(base + k, kPairs - 1)] : __int_as_float(0x7f800000);
            *reinterpret_cast<float4 *>(tb + kTblD + 4 * r) = make_float4(v[0], v[1], v[2], v[3]);
        }
    }
    if (tid < 20) {
        const int t = tid;
        float h0 = 0.f, he = 0.f;
        if (mp > 1 && t >= 1 && t < 17 && real(t)) h0 = hterm(sm.pDn[pidx(0, t)]);
        if (mp > 1 && t <= 15 && real(t)) he = hterm(sm.pUp[pidx(t, 16)]);
        tb[kTblH0 + t] = h0;
        tb[kTblHend + t] = he;
        float cv = 0.f;
        if (mp == 1) cv = (t == 0) ? sm.dc[0] : 0.f;
        else if (t < mp - 1) cv = sm.dc[t];
        else if (t == 16) cv = sm.dc[mp - 1];
        tb[kTblC + t] = cv;
    } else if (tid < 24) {
        const int t = tid - 20;
        tb[kTblHdr + t] = __int_as_float(t == 0 ? mp : t == 1 ? d : t == 2 ? (bad ? kFlagNonfinite : 0) : 0);
    } else if (tid == 32) {
        const double wd = (double)sm.dc[mp - 1] - (double)sm.dc[0];
        const double w2 = wd * wd;
        if (w2 == w2) atomicMax(&hdr->hi0_bits, (unsigned long long)__double_as_longlong(w2));
        if (bad) {
            atomicOr(&hdr->flags, (uint32_t)kFlagNonfinite);
            atomicMax(status, (int32_t)KVQ_ERR_NONFINITE);
        }
    }
}

int launch_stats_weights(const uint16_t *x, const float *wt, const kvq_layout &L, int lg_ng,
                         int lg_upr, void *stats, int32_t *status, cudaStream_t st);

// wt == nullptr: kvq_stats; otherwise kvq_stats_weighted, which runs the
// weighting pass (kvq_weight.cu) over the records this kernel wrote
int launch_stats(const uint16_t *x, const float *wt, const kvq_layout &L, void *stats,
                 int32_t *status, cudaStream_t st) {
    const int64_t nb = num_blocks(L);
    if (cudaMemsetAsync(status, 0, sizeof(int32_t), st) != cudaSuccess) return KVQ_ERR_CUDA;
    if (cudaMemsetAsync(stats, 0, sizeof(StatsHeader), st) != cudaSuccess) return KVQ_ERR_CUDA;
    if (nb == 0) return KVQ_OK;
    const int units = 4 * L.group;   // 8-entry units per block
    int lg_ng = 0, lg_upr = 0;
    while ((1 << lg_ng) < L.D / L.group) ++lg_ng;
    while ((1 << lg_upr) < L.group / 8) ++lg_upr;
    StatsHeader *hdr = static_cast<StatsHeader *>(stats);
    float *recs = reinterpret_cast<float *>(static_cast<char *>(stats) + sizeof(StatsHeader));
    const dim3 grid((unsigned)nb);
    if (units <= kStatsThreads)
        stats_kernel<1><<<grid, kStatsThreads, 0, st>>>(x, L, lg_ng, lg_upr, hdr, recs, status);
    else
        stats_kernel<2><<<grid, kStatsThreads, 0, st>>>(x, L, lg_ng, lg_upr, hdr, recs, status);
    if (cudaGetLastError() != cudaSuccess) return KVQ_ERR_CUDA;
    if (wt == nullptr) return KVQ_OK;
    return launch_stats_weights(x, wt, L, lg_ng, lg_upr, stats, status, st);
}

}  // namespace kvq
