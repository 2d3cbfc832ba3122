// Weighting pass of kvq_stats_weighted ("Rate-adaptive KV-cache quantizer",
// "Implementation notes": optionally weight D_r by the attention sensitivity
// measured on a calibration batch).
//
// Runs after the stats kernel on the records it wrote.  The candidates and
// the entropy terms do not change (H_r counts the stored symbols, whatever
// their weight); only the distortion does: D(a, b) = sum w (b - x)(x - a).
// One CTA of 256 threads per block; every global load is issued first:
//   1. the block's entries (16-byte loads of x, 32-byte loads of w) go to
//      their atoms [c_p, c_{p+1}) (the maximum closes the last atom) by a
//      4-step binary search over the candidates, which sit in lanes and are
//      read by shuffles;
//   2. each entry adds (w y, w t, w y t), y = x - c_p, t = c_{p+1} - x, to
//      its thread's column of that atom (48 KB of shared memory); the weight
//      sum of the atom is (sum w y + sum w t) / (c_{p+1} - c_p), since
//      y + t = c_{p+1} - c_p for every entry (a sum of non-negative terms);
//   3. a fixed-order tree over the columns gives the weighted atom moments
//      (repeated calls give identical bits);
//   4. the pair table D(c_P, c_Q) = sum over the atoms p of [P, Q) of
//      n A B + A t1 + B s1 + e (A = c_p - c_P, B = c_Q - c_{p+1}) replaces the
//      record's distortion table; the row's moments become the weighted ones.
// The bisection's starting point becomes max_r (c_max - c_min)^2 w_max,r.  A
// negative or non-finite weight counts as 0 and sets KVQ_ERR_BAD_WEIGHT; an
// entry the stats kernel flagged non-finite counts with weight 0.
#include "kvq_internal.cuh"

namespace kvq {

constexpr int kWThreads = 256;
// per (atom, thread): (s1, t1) in one float2 array and e in a float array;
// the weight sum follows from n W = s1 + t1 (y + t = W for every entry)
constexpr size_t kWColBytes = (size_t)16 * kWThreads * (sizeof(float2) + sizeof(float));   // 48 KB

template <int UNITS>
__global__ void __launch_bounds__(kWThreads, 4)
stats_weight_kernel(const uint16_t *__restrict__ x, const float *__restrict__ wt, kvq_layout L,
                    int lg_ng, int lg_upr, StatsHeader *__restrict__ hdr,
                    float *__restrict__ recs, int32_t *__restrict__ status) {
    extern __shared__ __align__(16) float2 cst[];     // [16 atoms][256]: (s1, t1)
    float *ce = reinterpret_cast<float *>(cst + 16 * kWThreads);   // [16 atoms][256]: e
    __shared__ float sc[kCand];
    __shared__ int32_t s_mp, s_rflags, s_tflags;
    __shared__ float wn[16], ws1[16], wt1[16], we[16];
    __shared__ float pD[kPairs];
    __shared__ uint32_t s_wmax, s_wbad;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = L.group, D = L.D, d = 32 * G, nG = D / G;
    const int64_t blk = blockIdx.x;
    const int g = (int)(blk & (nG - 1));
    const int64_t tbk = blk >> lg_ng;
    const int units = d / 8, upr = G / 8;
    float *rec = recs + blk * kRecFloats;
    float *tb = rec + kRecTbl;

    // every global load of the block first: this thread's entries and
    // weights, and the record's candidates, m' and flags
    uint4 xr[UNITS];
    float4 wa[UNITS], wc[UNITS];
#pragma unroll
    for (int k = 0; k < UNITS; ++k) {
        const int u = tid + k * kWThreads;
        xr[k] = make_uint4(0u, 0u, 0u, 0u);
        wa[k] = wc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (u < units) {
            const int row = u >> lg_upr, cu = u & (upr - 1);
            const int64_t off = (tbk * 32 + row) * (int64_t)D + (int64_t)g * G + cu * 8;
            xr[k] = __ldg(reinterpret_cast<const uint4 *>(x + off));
            wa[k] = __ldg(reinterpret_cast<const float4 *>(wt + off));
            wc[k] = __ldg(reinterpret_cast<const float4 *>(wt + off + 4));
        }
    }
    if (tid < kCand) sc[tid] = rec[tid];
    else if (tid == 32) s_mp = __float_as_int(rec[17]);
    else if (tid == 33) s_rflags = __float_as_int(rec[18]);
    else if (tid == 34) s_tflags = __float_as_int(tb[kTblHdr + 2]);
    if (tid < kPairs) pD[tid] = __int_as_float(0x7f800000);   // +inf: no such pair
    if (tid == 0) {
        s_wmax = 0u;
        s_wbad = 0u;
    }
#pragma unroll
    for (int p = 0; p < 16; ++p) {
        cst[p * kWThreads + tid] = make_float2(0.f, 0.f);
        ce[p * kWThreads + tid] = 0.f;
    }
    __syncthreads();
    const int mp = min(max(s_mp, 1), kCand);

    // lane j holds the boundary c_{j+1} (j < m'-2, else +inf) and the level c_j
    const float inf = __int_as_float(0x7f800000);
    const float bl = (lane < 16 && lane + 1 <= mp - 2) ? sc[lane + 1] : inf;
    const float cl = sc[lane < kCand ? lane : kCand - 1];
    const float b7 = __shfl_sync(0xffffffffu, bl, 7);

    bool wb = false;
    uint32_t wmx = 0u;
#pragma unroll
    for (int k = 0; k < UNITS; ++k) {
        const int u = tid + k * kWThreads;
        if (u >= units) continue;                             // units is a multiple of 32
        const uint32_t x4[4] = {xr[k].x, xr[k].y, xr[k].z, xr[k].w};
        const float w8[8] = {wa[k].x, wa[k].y, wa[k].z, wa[k].w, wc[k].x, wc[k].y, wc[k].z, wc[k].w};
#pragma unroll
        for (int q = 0; q < 8; ++q) {                         // warp-uniform control only
            // a weight is valid when finite and >= 0 (bits below +inf, or -0)
            const uint32_t wbits = __float_as_uint(w8[q]);
            const bool ok = wbits < 0x7f800000u || wbits == 0x80000000u;
            wb |= !ok;
            const uint32_t h = (x4[q >> 1] >> ((q & 1) * 16)) & 0xffffu;
            // a non-finite entry (flagged by the stats kernel) adds nothing
            const bool live = (h & 0x7c00u) != 0x7c00u;
            const uint32_t wv = ok ? (wbits & 0x7fffffffu) : 0u;
            wmx = max(wmx, wv);                               // w >= 0: bits order
            const float w = live ? __uint_as_float(wv) : 0.f;
            const float xv = live ? __half2float(__ushort_as_half((unsigned short)h)) : 0.f;
            if (mp < 2) continue;
            int p = xv >= b7 ? 8 : 0;
            p += xv >= __shfl_sync(0xffffffffu, bl, p + 3) ? 4 : 0;
            p += xv >= __shfl_sync(0xffffffffu, bl, p + 1) ? 2 : 0;
            p += xv >= __shfl_sync(0xffffffffu, bl, p) ? 1 : 0;
            const float y = xv - __shfl_sync(0xffffffffu, cl, p);
            const float t = __shfl_sync(0xffffffffu, cl, p + 1) - xv;
            const float wy = w * y;
            const int c = p * kWThreads + tid;
            float2 a = cst[c];
            a.x += wy;
            a.y += w * t;
            cst[c] = a;
            ce[c] += wy * t;
        }
    }
    wmx = __reduce_max_sync(0xffffffffu, wmx);
    const bool anyb = __any_sync(0xffffffffu, wb);
    if (lane == 0) {
        atomicMax(&s_wmax, wmx);
        if (anyb) atomicOr(&s_wbad, 1u);
    }
    __syncthreads();

    // fixed-order sums: warp w takes atoms 2w and 2w+1; lane l adds columns
    // l, l+32, ..., l+224, then a 32-lane tree
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int p = 2 * warp + hh;
        float2 a = cst[p * kWThreads + lane];
        float e = ce[p * kWThreads + lane];
#pragma unroll
        for (int c = 1; c < kWThreads / 32; ++c) {
            const float2 b = cst[p * kWThreads + lane + 32 * c];
            a.x += b.x;
            a.y += b.y;
            e += ce[p * kWThreads + lane + 32 * c];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            a.x += __shfl_down_sync(0xffffffffu, a.x, o);
            a.y += __shfl_down_sync(0xffffffffu, a.y, o);
            e += __shfl_down_sync(0xffffffffu, e, o);
        }
        if (lane == 0) {
            const float W = p + 1 < mp ? sc[p + 1] - sc[p] : 0.f;
            wn[p] = W > 0.f ? (a.x + a.y) / W : 0.f;     // sum w = (s1 + t1) / W
            ws1[p] = a.x;
            wt1[p] = a.y;
            we[p] = e;
        }
    }
    __syncthreads();

    // weighted distortion of every candidate pair, in slot space (the maximum
    // in slot 16), every term non-negative; pairs in order of decreasing
    // length Q - P, so that a warp's threads run loops of similar length:
    // thread t takes the P-th of the u pairs of length m' - u,
    // u(u-1)/2 <= t < u(u+1)/2
    const int npr = mp * (mp - 1) / 2;
    if (tid < npr) {
        int u = (int)((1.0f + sqrtf(1.0f + 8.0f * (float)tid)) * 0.5f);
        if (u * (u - 1) / 2 > tid) --u;
        if ((u + 1) * u / 2 <= tid) ++u;
        const int P = tid - u * (u - 1) / 2;
        const int Q = P + mp - u;
        const float a = sc[P], bq = sc[Q];
        float Dv = 0.f;
        for (int p = P; p < Q; ++p) {
            const float A = sc[p] - a, Bq = bq - sc[p + 1];
            Dv += wn[p] * A * Bq + A * wt1[p] + Bq * ws1[p] + we[p];
        }
        const int sj = P == mp - 1 ? 16 : P, sl = Q == mp - 1 ? 16 : Q;
        pD[pidx(sj, sl)] = Dv;
    }
    __syncthreads();

    const bool wbad = s_wbad != 0u;
    const int addf = kFlagWeighted | (wbad ? kFlagBadWeight : 0);
    // the D table in 16-byte pieces (a padded row piece shares j)
    if (tid < kDpFloats / 4) {
        const uint32_t dcd = kDecode.pair[4 * tid];
        const int j = dcd & 255, l0 = dcd >> 8;
        const int base = l0 < 17 ? pidx(j, l0) : 0;
        float v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = l0 + k < 17 ? pD[min(base + k, kPairs - 1)] : inf;
        *reinterpret_cast<float4 *>(tb + kTblD + 4 * tid) = make_float4(v[0], v[1], v[2], v[3]);
    }
    if (tid >= 20 && tid < 84) {
        const int q = (tid - 20) >> 4, p = (tid - 20) & 15;
        rec[tid] = q == 0 ? wn[p] : q == 1 ? ws1[p] : q == 2 ? wt1[p] : we[p];
    } else if (tid == 18) {
        rec[18] = __int_as_float(s_rflags | addf);
    } else if (tid == 19) {
        tb[kTblHdr + 2] = __int_as_float(s_tflags | addf);
    } else if (tid == 0) {
        const double wd = (double)sc[mp - 1] - (double)sc[0];
        const double w2 = (wd * wd) * (double)__uint_as_float(s_wmax);
        if (w2 == w2) atomicMax(&hdr->hi0_bits, (unsigned long long)__double_as_longlong(w2));
        if (wbad) {
            atomicOr(&hdr->flags, (uint32_t)kFlagBadWeight);
            atomicMax(status, (int32_t)KVQ_ERR_BAD_WEIGHT);
        }
    }
}

// the pass's 48 KB of columns plus its static shared memory exceed the
// default per-block limit: opt in once per device
int weights_init() {
    if (cudaFuncSetAttribute(stats_weight_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kWColBytes) != cudaSuccess)
        return KVQ_ERR_CUDA;
    if (cudaFuncSetAttribute(stats_weight_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kWColBytes) != cudaSuccess)
        return KVQ_ERR_CUDA;
    return KVQ_OK;
}

int launch_stats_weights(const uint16_t *x, const float *wt, const kvq_layout &L, int lg_ng,
                         int lg_upr, void *stats, int32_t *status, cudaStream_t st) {
    const int64_t nb = num_blocks(L);
    StatsHeader *hdr = static_cast<StatsHeader *>(stats);
    // the stats kernel left max_r (c_max - c_min)^2 here: start the weighted
    // maximum afresh
    if (cudaMemsetAsync(&hdr->hi0_bits, 0, sizeof(hdr->hi0_bits), st) != cudaSuccess)
        return KVQ_ERR_CUDA;
    float *recs = reinterpret_cast<float *>(static_cast<char *>(stats) + sizeof(StatsHeader));
    const dim3 grid((unsigned)nb);
    if (4 * L.group <= kWThreads)
        stats_weight_kernel<1><<<grid, kWThreads, kWColBytes, st>>>(x, wt, L, lg_ng, lg_upr, hdr,
                                                                    recs, status);
    else
        stats_weight_kernel<2><<<grid, kWThreads, kWColBytes, st>>>(x, wt, L, lg_ng, lg_upr, hdr,
                                                                    recs, status);
    return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq
