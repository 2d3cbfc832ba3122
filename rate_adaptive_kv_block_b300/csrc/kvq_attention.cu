// kvq_decode_attention: one decoding step of attention read straight from the
// quantized cache ("Rate-adaptive KV-cache quantizer", "Implementation
// notes": the stored codebook and symbols are decoded before attention, and
// attention latency is one of the quantities the page records).
//
// For query head hq and its KV head h = hq / n_rep:
//   s_t = scale * sum_f q[hq, f] K[h, t, f]              (t < T_valid)
//   out[hq, f] = sum_t softmax(s)_t V[h, t, f]
// where K[h, t, f] is the level its 4-bit code selects in the block's
// codebook (a binary16 value held in fp32), and V likewise.  The codes are
// turned into levels in registers through a 16-entry table in shared memory
// per block and feature group; nothing is written back as binary16, so the
// cache is read at 0.5 byte per entry plus 64 bytes of codebook per block.
//
// Two kernels on the caller's stream:
//   attn_partial_kernel  grid (splits, KV heads), 128 threads: a range of
//                        32-token blocks of one KV head with an online
//                        softmax (running maximum and sum per query head,
//                        base-2 exponentials of scale*log2(e)-scaled scores);
//                        writes (max, sum, unnormalised output) per split.
//                        The range's K and V codes and codebooks are
//                        contiguous in HBM; they arrive in chunks of 4 token
//                        blocks by bulk (TMA) copies into a two-stage shared
//                        ring, the next chunk in flight while one is used
//   attn_combine_kernel  one CTA per query head: rescales the splits to a
//                        common maximum and divides by the total weight
// Inside a CTA: scores with 8 lanes per token (16 features each, partial dot
// products combined by a fixed shuffle tree), values with a lane per 8
// features and 4 tokens (accumulators in registers), the 8 token groups
// added in a fixed order at the end.
#include <math.h>

#include "kvq_internal.cuh"
#include "kvq_bulk.cuh"

namespace kvq {

constexpr int kAttnD = 128;         // head dimension
constexpr int kAttnThreads = 128;
constexpr int kAttnMaxSplits = 64;  // splits per KV head (workspace size)
constexpr int kAttnChunkMax = 8;    // token blocks per bulk-copy stage (at most)
constexpr uint32_t kAttnWaitLimit = 1u << 22;   // mbarrier polls before giving up
// one token block of one tensor: 32 tokens x 128 features at 4 bits (every
// feature group), and its codebooks (16 fp32 per feature group)
constexpr uint32_t kAttnCodeBytes = 16 * kAttnD;
__host__ __device__ constexpr uint32_t attn_stage_bytes(int chunk, int nG) {
    return (uint32_t)chunk * (2 * kAttnCodeBytes + 2 * 64u * (uint32_t)nG);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Byte offset, inside one token block's codes (all its feature groups), of
// the 8 codes of features f .. f+7 (f % 8 == 0) of token t: group f / G,
// entry t G + f % G, two entries per byte.
__device__ __forceinline__ uint32_t code_offset(int t, int f, int G) {
    return (uint32_t)((f / G) * 16 * G + ((t * G + (f & (G - 1))) >> 1));
}

template <int R>
__global__ void __launch_bounds__(kAttnThreads)
attn_partial_kernel(const float *__restrict__ q, const uint8_t *__restrict__ kc,
                    const float *__restrict__ kcb, const uint8_t *__restrict__ vc,
                    const float *__restrict__ vcb, int64_t ntb, int G, int64_t T_valid,
                    float scale2, int bps, int chunk, float *__restrict__ part,
                    int32_t *__restrict__ status, uint32_t wait_polls) {
    constexpr int D = kAttnD;
    const float NEG = __int_as_float(0xff800000);   // -inf
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t h = blockIdx.y;
    const int split = blockIdx.x, nsplit = gridDim.x;
    const int nG = D / G;
    const int64_t ntb_valid = (T_valid + 31) / 32;
    const int64_t tb0 = (int64_t)split * bps;
    const int64_t tb1 = min(tb0 + bps, ntb_valid);
    const int nchunks = tb1 > tb0 ? (int)((tb1 - tb0 + chunk - 1) / chunk) : 0;

    extern __shared__ __align__(128) unsigned char asm_[];   // two stages
    const uint32_t stage = attn_stage_bytes(chunk, nG);
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ float ss[R][32 * kAttnChunkMax], sp[R][32 * kAttnChunkMax];   // scores, weights of a chunk
    __shared__ float sm[R], sl[R], salpha[R];       // running max, sum; rescale factor
    __shared__ float sacc[8][R][D];                 // token groups' outputs, added at the end
    __shared__ bool failed;

    // stage layout: K codes, V codes (chunk x 2048 bytes each), K codebooks,
    // V codebooks (chunk x nG x 16 floats each)
    auto issue = [&](int c) {
        unsigned char *buf = asm_ + (c & 1) * stage;
        const int64_t tbs = tb0 + (int64_t)c * chunk;
        const uint32_t nblk = (uint32_t)min((int64_t)chunk, tb1 - tbs);
        const int64_t blk0 = (h * ntb + tbs) * nG;                 // first block of the chunk
        const uint32_t cbytes = nblk * kAttnCodeBytes, bbytes = nblk * 64u * (uint32_t)nG;
        mbar_expect_tx(&bars[c & 1], 2 * cbytes + 2 * bbytes);
        bulk_g2s(buf, kc + blk0 * 16 * G, cbytes, &bars[c & 1]);
        bulk_g2s(buf + chunk * kAttnCodeBytes, vc + blk0 * 16 * G, cbytes, &bars[c & 1]);
        bulk_g2s(buf + 2 * chunk * kAttnCodeBytes, kcb + blk0 * 16, bbytes, &bars[c & 1]);
        bulk_g2s(buf + 2 * chunk * kAttnCodeBytes + chunk * 64u * nG, vcb + blk0 * 16,
                 bbytes, &bars[c & 1]);
    };
    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        failed = false;
        for (int c = 0; c < 2 && c < nchunks; ++c) issue(c);
    }
    if (tid < R) {
        sm[tid] = NEG;
        sl[tid] = 0.f;
    }
    // this lane's query features (16 per lane, 8 lanes per token), scaled by
    // scale * log2(e) so that the softmax runs on exp2
    const int k8 = tid & 7, tok = tid >> 3;
    float qr[R][16];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const float4 *q4 = reinterpret_cast<const float4 *>(q + (h * R + r) * D + 16 * k8);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 v = q4[i];
            qr[r][4 * i] = v.x * scale2;
            qr[r][4 * i + 1] = v.y * scale2;
            qr[r][4 * i + 2] = v.z * scale2;
            qr[r][4 * i + 3] = v.w * scale2;
        }
    }
    // value lanes: features 8 fg .. 8 fg + 7, tokens 4 tg .. 4 tg + 3
    const int fg = tid & 15, tg = tid >> 4;
    float2 acc[R][4];                               // features 8 fg + 2b, + 2b + 1
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[r][b] = make_float2(0.f, 0.f);
    __syncthreads();

    int cfail = nchunks;
    for (int c = 0; c < nchunks; ++c) {
        if (tid == 0 && !mbar_wait(&bars[c & 1], (uint32_t)(c >> 1) & 1u, wait_polls))
            failed = true;
        __syncthreads();
        if (failed) {
            cfail = c;
            break;
        }
        const unsigned char *buf = asm_ + (c & 1) * stage;
        const int64_t tbs = tb0 + (int64_t)c * chunk;
        const int nblk = (int)min((int64_t)chunk, tb1 - tbs);
        const unsigned char *kcode0 = buf, *vcode0 = buf + chunk * kAttnCodeBytes;
        const float *klv0 = reinterpret_cast<const float *>(buf + 2 * chunk * kAttnCodeBytes);
        const float *vlv0 = klv0 + chunk * nG * 16;
        // scores of the chunk's tokens: 16 tokens per pass, 8 lanes per token
        for (int j = 0; j < nblk; ++j) {
            const unsigned char *kcode = kcode0 + j * kAttnCodeBytes;
            const float *klv = klv0 + j * nG * 16;
#pragma unroll
            for (int pass = 0; pass < 2; ++pass) {
                const int t = 16 * pass + tok;
                float2 dot[R];                       // even and odd features apart
#pragma unroll
                for (int r = 0; r < R; ++r) dot[r] = make_float2(0.f, 0.f);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int f = 16 * k8 + 8 * u;
                    const uint32_t w = *reinterpret_cast<const uint32_t *>(kcode + code_offset(t, f, G));
                    const float *lv = klv + (f / G) * 16;
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        const float2 kk = make_float2(lv[(w >> (8 * b)) & 15u], lv[(w >> (8 * b + 4)) & 15u]);
#pragma unroll
                        for (int r = 0; r < R; ++r)
                            dot[r] = __ffma2_rn(make_float2(qr[r][8 * u + 2 * b], qr[r][8 * u + 2 * b + 1]),
                                                kk, dot[r]);
                    }
                }
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    float v = dot[r].x + dot[r].y;
                    v += __shfl_xor_sync(0xffffffffu, v, 1);
                    v += __shfl_xor_sync(0xffffffffu, v, 2);
                    v += __shfl_xor_sync(0xffffffffu, v, 4);
                    if (k8 == 0) ss[r][32 * j + t] = ((tbs + j) * 32 + t < T_valid) ? v : NEG;
                }
            }
        }
        __syncthreads();
        // online softmax over the chunk, a warp per query head (lane: tokens
        // lane, lane + 32, ..)
        if (warp < R) {
            const int r = warp;
            float sc[kAttnChunkMax];
            float bm = NEG;
#pragma unroll
            for (int k = 0; k < kAttnChunkMax; ++k) {
                sc[k] = k < nblk ? ss[r][32 * k + lane] : NEG;
                bm = fmaxf(bm, sc[k]);
            }
            const float m_old = sm[r];
            const float m_new = fmaxf(m_old, warp_max(bm));
            float alpha = 1.f, psum = 0.f;
            if (m_new != NEG) alpha = exp2f(m_old - m_new);          // 0 while nothing was seen
#pragma unroll
            for (int k = 0; k < kAttnChunkMax; ++k) {
                const float p = (m_new == NEG || sc[k] == NEG) ? 0.f : exp2f(sc[k] - m_new);
                if (k < nblk) sp[r][32 * k + lane] = p;
                psum += p;
            }
            const float bsum = warp_sum(psum);
            if (lane == 0) {
                salpha[r] = alpha;
                sm[r] = m_new;
                sl[r] = fmaf(alpha, sl[r], bsum);
            }
        }
        __syncthreads();
        // values: rescale, then add the chunk's tokens
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float2 a = make_float2(salpha[r], salpha[r]);
#pragma unroll
            for (int b = 0; b < 4; ++b) acc[r][b] = __fmul2_rn(acc[r][b], a);
        }
        for (int j = 0; j < nblk; ++j) {
            const unsigned char *vcode = vcode0 + j * kAttnCodeBytes;
            const int f = 8 * fg;
            const float *lv = vlv0 + j * nG * 16 + (f / G) * 16;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int t = 4 * tg + k;
                const uint32_t w = *reinterpret_cast<const uint32_t *>(vcode + code_offset(t, f, G));
                float2 pr[R];
#pragma unroll
                for (int r = 0; r < R; ++r) pr[r] = make_float2(sp[r][32 * j + t], sp[r][32 * j + t]);
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const float2 vv = make_float2(lv[(w >> (8 * b)) & 15u], lv[(w >> (8 * b + 4)) & 15u]);
#pragma unroll
                    for (int r = 0; r < R; ++r) acc[r][b] = __ffma2_rn(pr[r], vv, acc[r][b]);
                }
            }
        }
        __syncthreads();
        // every thread is done with this stage: refill it with chunk c + 2
        if (tid == 0 && c + 2 < nchunks) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(c + 2);
        }
    }
    if (failed) {
        // a copy never completed: report it, give the copies in flight (this
        // chunk and the next) a bounded chance to land before the shared
        // memory is released, and leave this split out of the combine (zero
        // weight and zero outputs, so that it adds nothing)
        if (tid == 0) {
            if (status) atomicExch(status, KVQ_ERR_TIMEOUT);
            for (int c = cfail; c < cfail + 2 && c < nchunks; ++c)
                mbar_wait(&bars[c & 1], (uint32_t)(c >> 1) & 1u, kAttnWaitLimit);
        }
        for (int i = tid; i < R * D; i += kAttnThreads)
            part[((h * R + i / D) * nsplit + split) * (D + 2) + 2 + i % D] = 0.f;
        if (tid < R) {
            float *pm = part + ((h * R + tid) * nsplit + split) * (D + 2);
            pm[0] = NEG;
            pm[1] = 0.f;
        }
        __syncthreads();
        return;
    }
    // the token groups' outputs, added in a fixed order
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            sacc[tg][r][8 * fg + 2 * b] = acc[r][b].x;
            sacc[tg][r][8 * fg + 2 * b + 1] = acc[r][b].y;
        }
    __syncthreads();
    for (int i = tid; i < R * D; i += kAttnThreads) {
        const int r = i / D, f = i % D;
        float o = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) o += sacc[k][r][f];
        part[((h * R + r) * nsplit + split) * (D + 2) + 2 + f] = o;
    }
    if (tid < R) {
        float *pm = part + ((h * R + tid) * nsplit + split) * (D + 2);
        pm[0] = sm[tid];
        pm[1] = sl[tid];
    }
}

// Query head hq's splits are contiguous in the workspace ([hq][split][max,
// sum, D outputs]): lane f loads its output of every split at once (the
// loads in flight together), lanes 0 .. nsplit-1 one (max, sum) pair each.
__global__ void __launch_bounds__(kAttnD)
attn_combine_kernel(const float *__restrict__ part, int nsplit, float *__restrict__ out) {
    constexpr int D = kAttnD;
    __shared__ float sw[kAttnMaxSplits], sls[kAttnMaxSplits];
    __shared__ float sM;
    const int hq = blockIdx.x, f = threadIdx.x;
    const float NEG = __int_as_float(0xff800000);
    const float *base = part + (int64_t)hq * nsplit * (D + 2);
    float o[kAttnMaxSplits];
#pragma unroll
    for (int s = 0; s < kAttnMaxSplits; ++s) o[s] = s < nsplit ? base[s * (D + 2) + 2 + f] : 0.f;
    float m = NEG, l = 0.f;
    if (f < nsplit) {
        m = base[f * (D + 2)];
        l = base[f * (D + 2) + 1];
    }
    // the maximum over the splits (warps 0 and 1 hold the 64 candidates)
    float wm = m;
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, k));
    if (f == 32) sw[0] = wm;
    __syncthreads();
    if (f == 0) sM = fmaxf(wm, sw[0]);
    __syncthreads();
    const float M = sM;
    if (f < kAttnMaxSplits) {
        const float w = (M == NEG || m == NEG) ? 0.f : exp2f(m - M);
        sw[f] = w;
        sls[f] = w * l;
    }
    __syncthreads();
    float Lw = 0.f, O = 0.f;
#pragma unroll
    for (int s = 0; s < kAttnMaxSplits; ++s) {
        if (s < nsplit) {
            Lw += sls[s];
            O = fmaf(sw[s], o[s], O);
        }
    }
    out[(int64_t)hq * D + f] = Lw > 0.f ? O / Lw : 0.f;
}

size_t attention_workspace_bytes(const kvq_layout &L, int n_rep) {
    return (size_t)L.S * kAttnMaxSplits * n_rep * (kAttnD + 2) * sizeof(float);
}

int attention_init() {
    const int smem = 2 * (int)attn_stage_bytes(kAttnChunkMax, kAttnD / 8);   // the largest ring
    if (cudaFuncSetAttribute(attn_partial_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess ||
        cudaFuncSetAttribute(attn_partial_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess ||
        cudaFuncSetAttribute(attn_partial_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
        return KVQ_ERR_CUDA;
    return KVQ_OK;
}

int launch_decode_attention(const float *q, int n_rep, const kvq_layout &L, const uint8_t *kc,
                            const float *kcb, const uint8_t *vc, const float *vcb,
                            int64_t T_valid, float scale, void *workspace, float *out,
                            int32_t *status, cudaStream_t st) {
    const int64_t H = L.S;
    if (H == 0) return KVQ_OK;
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return KVQ_ERR_CUDA;
    const int64_t ntb = L.T / 32;
    const int64_t ntb_valid = (T_valid + 31) / 32;
    float *part = static_cast<float *>(workspace);
    int nsplit = 0;
    if (ntb_valid > 0) {
        // one wave (three CTAs per SM at 168 registers) over all KV heads, at
        // most one split per block
        int64_t want = (3 * (int64_t)sms) / H;
        if (want > kAttnMaxSplits) want = kAttnMaxSplits;
        if (want > ntb_valid) want = ntb_valid;
        if (want < 1) want = 1;
        const int64_t bps = (ntb_valid + want - 1) / want;
        nsplit = (int)((ntb_valid + bps - 1) / bps);
        const dim3 grid((unsigned)nsplit, (unsigned)H);
        const float scale2 = scale * 1.4426950408889634f;   // log2(e)
        // a CTA's range in one chunk when it has at most 8 blocks, else a
        // ring of two stages of 8
        const int chunk = (int)(bps < kAttnChunkMax ? bps : kAttnChunkMax);
        const size_t smem = (bps > chunk ? 2 : 1) * (size_t)attn_stage_bytes(chunk, L.D / L.group);
        unsigned long long tw = 0;
        const uint32_t wait_polls = test_wait_limit(&tw) ? 0u : kAttnWaitLimit;
        switch (n_rep) {
        case 1:
            attn_partial_kernel<1><<<grid, kAttnThreads, smem, st>>>(
                q, kc, kcb, vc, vcb, ntb, L.group, T_valid, scale2, (int)bps, chunk, part, status,
                wait_polls);
            break;
        case 2:
            attn_partial_kernel<2><<<grid, kAttnThreads, smem, st>>>(
                q, kc, kcb, vc, vcb, ntb, L.group, T_valid, scale2, (int)bps, chunk, part, status,
                wait_polls);
            break;
        default:
            attn_partial_kernel<4><<<grid, kAttnThreads, smem, st>>>(
                q, kc, kcb, vc, vcb, ntb, L.group, T_valid, scale2, (int)bps, chunk, part, status,
                wait_polls);
            break;
        }
        if (cudaGetLastError() != cudaSuccess) return KVQ_ERR_CUDA;
    }
    attn_combine_kernel<<<(unsigned)(H * n_rep), kAttnD, 0, st>>>(part, nsplit, out);
    return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq
