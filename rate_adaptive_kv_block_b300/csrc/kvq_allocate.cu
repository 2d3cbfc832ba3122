// kvq_allocate: per-block codebook choice and the global lambda.
//
// "Rate-adaptive KV-cache quantizer", "Mathematical statement": minimise
// sum_r D_r subject to sum_r d_r H_r <= B, |Q_r| <= s; the Lagrangian
// sum_r [D_r + lambda d_r H_r] - lambda B separates the blocks, which are
// coupled only through lambda.  "Implementation notes": each block takes
// argmin_Q [D_r + lambda d_r H_r] by a small dynamic program over ordered
// codepoints; one global lambda.
//
// Kernels (all on the caller's stream, no host synchronisation):
//   ctrl_init      reset the control word in the workspace
//   tables         per block, from the stats row: the lambda-independent DP
//                  tables (interval distortion, entropy terms), in "slot"
//                  space (see kvq_internal.cuh); max_r (c_max - c_min)^2
//   search_round   one warp per block, one lane per probe lambda: each lane
//                  runs the whole exact DP at its own lambda, so the warp
//                  evaluates 32 lambdas with no cross-lane traffic and the
//                  table reads are shared-memory broadcasts.  The rates are
//                  reduced in a fixed order (per CTA, then by the last CTA
//                  to finish) and that CTA advances the search:
//                    bracket round: probes 0 and hi0 * 2^t, t = 0..30;
//                    bisection round: the 31 nodes of the next 5 levels of
//                    the bisection tree under [lo, hi] -- every midpoint the
//                    sequential bisection could visit in its next 5 steps,
//                    computed with the same fp64 formula 0.5 (lo + hi) --
//                    then the walk takes the 5 steps.  8 rounds = 40 steps,
//                    the same lambda as 40 sequential steps.
//   emit           per block: the chain at the final lambda (recorded by the
//                  round that evaluated it) -> codebook, k, D_r, H_r; totals;
//                  the subgradient update in KVQ_SUBGRADIENT mode.
#include <math.h>

#include "kvq_internal.cuh"

namespace kvq {

constexpr int kTablesWarps = 4;
constexpr int kRoundWarps = 4;        // s >= 16: DP path A only
constexpr int kRoundWarpsGen = 2;     // s < 16: path B possible
constexpr int kEmitThreads = 256;

// ---------------------------------------------------------------- workspace
struct Workspace {
    Ctrl *ctrl;
    float *tables;        // [nblk][kTblStride]
    float *rates;         // [nblk][32]   d_r H_r per probe (last round)
    uint32_t *masks;      // [nblk][32]   chain per probe (last round)
    float *rate_lo;       // [nblk]       d_r H_r at lo
    float *rate_hi;       // [nblk]       d_r H_r at hi
    uint32_t *mask_hi;    // [nblk]       chain at hi
    uint8_t *act;         // [nblk]       evaluated in the last round
    double *epartial;     // [emit CTAs][2]
};

static size_t align_up(size_t v) { return (v + 255) & ~(size_t)255; }

size_t workspace_bytes(int64_t nb, int s) {
    (void)s;
    size_t b = align_up(sizeof(Ctrl));
    b += align_up((size_t)nb * kTblStride * sizeof(float));
    b += align_up((size_t)nb * 32 * sizeof(float));
    b += align_up((size_t)nb * 32 * sizeof(uint32_t));
    b += 3 * align_up((size_t)nb * sizeof(float));
    b += align_up((size_t)nb);
    b += align_up((size_t)((nb + kEmitThreads - 1) / kEmitThreads) * 2 * sizeof(double));
    return b;
}

static Workspace carve(void *base, int64_t nb) {
    char *p = static_cast<char *>(base);
    Workspace w;
    w.ctrl = reinterpret_cast<Ctrl *>(p);
    p += align_up(sizeof(Ctrl));
    w.tables = reinterpret_cast<float *>(p);
    p += align_up((size_t)nb * kTblStride * sizeof(float));
    w.rates = reinterpret_cast<float *>(p);
    p += align_up((size_t)nb * 32 * sizeof(float));
    w.masks = reinterpret_cast<uint32_t *>(p);
    p += align_up((size_t)nb * 32 * sizeof(uint32_t));
    w.rate_lo = reinterpret_cast<float *>(p);
    p += align_up((size_t)nb * sizeof(float));
    w.rate_hi = reinterpret_cast<float *>(p);
    p += align_up((size_t)nb * sizeof(float));
    w.mask_hi = reinterpret_cast<uint32_t *>(p);
    p += align_up((size_t)nb * sizeof(uint32_t));
    w.act = reinterpret_cast<uint8_t *>(p);
    p += align_up((size_t)nb);
    w.epartial = reinterpret_cast<double *>(p);
    return w;
}

// ---------------------------------------------------------------- ctrl init
__global__ void ctrl_init_kernel(Ctrl *c, double budget, double eta, int mode,
                                 const double *lambda_in) {
    if (threadIdx.x != 0) return;
    c->budget = budget;
    c->eta = eta;
    c->lo = 0.0;
    c->hi = 0.0;
    c->lambda = (mode == KVQ_SUBGRADIENT) ? *lambda_in : 0.0;
    c->R_hi = 0.0;
    c->hi0_bits = 0ull;
    c->phase = (mode == KVQ_SUBGRADIENT) ? kPhaseFixed : kPhaseBracket;
    c->step = 0;
    c->hi_probe = -1;
    c->lo_probe = -1;
    for (int i = 0; i < 32; ++i) c->acc[i] = 0ull;
    c->status = KVQ_OK;
    c->flags = 0;
    c->mode = mode;
    c->ticket = 0u;
    c->ticket_emit = 0u;
}

// -------------------------------------------------------------------- tables
// Decode of a padded hh entry: (i, j, l) packed as i | j << 8 | l << 16
// (l = 17 marks padding), and of a padded Dp entry: j | l << 8.
struct DecodeTables {
    uint32_t trip[kHHFloats];
    uint32_t pair[kDpFloats];
};
constexpr DecodeTables make_decode() {
    DecodeTables t{};
    for (int j = 1; j < 16; ++j)
        for (int i = 0; i < j; ++i)
            for (int k = 0; k < pad4(16 - j); ++k) {
                const int l = j + 1 + k;
                t.trip[trip_off(i, j) + k] = (uint32_t)i | ((uint32_t)j << 8) | ((uint32_t)(l < 17 ? l : 17) << 16);
            }
    for (int j = 0; j < 16; ++j)
        for (int k = 0; k < pad4(16 - j); ++k) {
            const int l = j + 1 + k;
            t.pair[dp_off(j) + k] = (uint32_t)j | ((uint32_t)(l < 17 ? l : 17) << 8);
        }
    return t;
}
__device__ constexpr DecodeTables kDecode = make_decode();

__device__ __forceinline__ float hterm(float M, float inv_d) {
    // entropy term of a level with expected count M out of d: -M log2(M/d)
    return M > 0.f ? -M * log2f(M * inv_d) : 0.f;
}

__global__ void __launch_bounds__(kTablesWarps * 32)
tables_kernel(const StatsRow *__restrict__ stats, int64_t nb, float *__restrict__ tables,
              Ctrl *__restrict__ ctrl) {
    __shared__ float sRow[kTablesWarps][96];
    __shared__ float sDp[kTablesWarps][kPairs];
    __shared__ float sUp[kTablesWarps][kPairs];
    __shared__ float sDn[kTablesWarps][kPairs];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t b = (int64_t)blockIdx.x * kTablesWarps + w;
    if (b >= nb) return;
    const float *src = reinterpret_cast<const float *>(stats + b);
    for (int i = lane; i < 96; i += 32) sRow[w][i] = src[i];
    __syncwarp();
    const float *row = sRow[w];
    const int mp = min(max(__float_as_int(row[17]), 1), kCand);
    const int flags = __float_as_int(row[18]);
    const int d = __float_as_int(row[19]);
    const float inv_d = 1.0f / (float)d;
    const float INF = __int_as_float(0x7f800000);
    // candidate index -> slot
    auto slot_of = [&](int t) { return t == mp - 1 ? 16 : t; };

    for (int i = lane; i < kPairs; i += 32) {
        sDp[w][i] = INF;
        sUp[w][i] = 0.f;
        sDn[w][i] = 0.f;
    }
    __syncwarp();
    // pairs of real candidates P < Q: sums over the atoms P .. Q-1
    const int npr = mp * (mp - 1) / 2;
    for (int idx = lane; idx < npr; idx += 32) {
        int P = 0, rem = idx;
        while (rem >= mp - 1 - P) { rem -= mp - 1 - P; ++P; }
        const int Q = P + 1 + rem;
        const float a = row[P], bq = row[Q];
        float Dv = 0.f, Us = 0.f, Ls = 0.f;
        for (int p = P; p < Q; ++p) {
            const float n = row[20 + p], s1 = row[36 + p], t1 = row[52 + p], e = row[68 + p];
            const float A = row[p] - a, B = bq - row[p + 1];
            Dv += n * A * B + A * t1 + B * s1 + e;
            Us += s1 + n * A;
            Ls += t1 + n * B;
        }
        const float W = bq - a;
        const int sj = slot_of(P), sl = slot_of(Q);
        const int o = pidx(sj, sl);
        sDp[w][o] = Dv;
        sUp[w][o] = Us / W;
        sDn[w][o] = Ls / W;
    }
    __syncwarp();
    float *tb = tables + b * kTblStride;
    auto real = [&](int t) { return t < mp - 1 || t == 16; };
    // Dp rows, padded
    for (int idx = lane; idx < kDpFloats; idx += 32) {
        const uint32_t dc = kDecode.pair[idx];
        const int j = dc & 255, l = dc >> 8;
        tb[kTblD + idx] = l < 17 ? sDp[w][pidx(j, l)] : INF;
    }
    // hh rows (slot space), padded
    for (int idx = lane; idx < kHHFloats; idx += 32) {
        const uint32_t dc = kDecode.trip[idx];
        const int i = dc & 255, j = (dc >> 8) & 255, l = dc >> 16;
        float v = 0.f;
        if (l < 17 && mp > 1 && real(i) && real(j) && real(l))
            v = hterm(sUp[w][pidx(i, j)] + sDn[w][pidx(j, l)], inv_d);
        tb[kTblHH + idx] = v;
    }
    if (lane < 20) {
        const int t = lane;
        float h0 = 0.f, he = 0.f;
        if (mp > 1 && t >= 1 && t < 17 && real(t)) h0 = hterm(sDn[w][pidx(0, t)], inv_d);
        if (mp > 1 && t <= 15 && real(t)) he = hterm(sUp[w][pidx(t, 16)], inv_d);
        tb[kTblH0 + t] = h0;
        tb[kTblHend + t] = he;
        float cv = 0.f;
        if (mp == 1) cv = (t == 0) ? row[0] : 0.f;
        else if (t < mp - 1) cv = row[t];
        else if (t == 16) cv = row[mp - 1];
        tb[kTblC + t] = cv;
    }
    if (lane == 0) {
        tb[kTblHdr + 0] = __int_as_float(mp);
        tb[kTblHdr + 1] = __int_as_float(d);
        tb[kTblHdr + 2] = __int_as_float(flags);
        tb[kTblHdr + 3] = 0.f;   // the row ends at kTblHdr + 3
        const double wd = (double)row[mp - 1] - (double)row[0];
        const double w2 = wd * wd;
        if (w2 == w2) atomicMax(&ctrl->hi0_bits, (unsigned long long)__double_as_longlong(w2));
        if (flags) atomicOr(&ctrl->flags, flags);
    }
}

// ------------------------------------------------------- probe lambda values
// In-order position pos (1..31) of the 5-level bisection tree under [lo, hi],
// with the midpoints formed exactly as the sequential bisection forms them.
__device__ __forceinline__ double tree_node(double lo, double hi, int pos) {
    int cur = 16, half = 8;
    double a = lo, b = hi;
    for (;;) {
        const double mid = 0.5 * (a + b);
        if (pos == cur) return mid;
        if (pos < cur) { b = mid; cur -= half; } else { a = mid; cur += half; }
        half >>= 1;
    }
}

__device__ __forceinline__ double probe_lambda(const Ctrl &c, double hi0, int lane) {
    if (c.phase == kPhaseBracket) return lane == 0 ? 0.0 : ldexp(hi0, lane - 1);
    if (c.phase == kPhaseFixed) return c.lambda;
    return lane == 31 ? c.hi : tree_node(c.lo, c.hi, lane + 1);
}

// ---------------------------------------------------------------- DP path A
// Exact minimiser over all chains 0 = l_0 < ... < l_{k-1} = 16 (slot space)
// that either may use every slot (C == 0) or must skip at least one
// (C == 1: m' = 17 and s = 16).  Layer 0 holds the single chain 0,1,..,j
// (state (j-1, j)); layer 1 every chain that already skipped a slot.
// State value G(j,l): distortion of the intervals up to (j,l) plus lambda
// times the entropy terms of the levels before l.  Lane-private state in
// shared memory, [pair][lane].  Returns the chain's d_r H_r and its mask.
__device__ __forceinline__ float hh_at(const float *tb, int i, int j, int l) {
    return tb[kTblHH + trip_off(i, j) + l - j - 1];
}
__device__ __forceinline__ float dp_at(const float *tb, int j, int l) {
    return tb[kTblD + dp_off(j) + l - j - 1];
}

// One stage of the forward pass: all states (j, l), l = j+1 .. 16, from the
// states (i, j) of the earlier stages (compile-time j, so every index is an
// immediate and the accumulators stay in registers).
template <int J>
__device__ __forceinline__ void dp_a_stage(const float *__restrict__ tb, float lam,
                                           float *__restrict__ sG1, float *__restrict__ sG0,
                                           int lane) {
    constexpr int n = 16 - J;          // targets l = J+1 .. 16
    constexpr int nq = (n + 3) / 4;
    const float INF = __int_as_float(0x7f800000);
    float acc[n];
    float acc0 = INF;
    {
        const float g0 = sG0[J * 32 + lane];
        const float4 *h4 = reinterpret_cast<const float4 *>(tb + kTblHH + trip_off(J - 1, J));
#pragma unroll
        for (int q = 0; q < nq; ++q) {
            const float4 h = h4[q];
            const float hs[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int t = 4 * q + r;
                if (t < n) {
                    if (t == 0) acc0 = fmaf(lam, hs[r], g0);
                    else acc[t] = fmaf(lam, hs[r], g0);
                }
            }
        }
        acc[0] = INF;
    }
#pragma unroll
    for (int i = 0; i < J; ++i) {
        const float g = sG1[pidx(i, J) * 32 + lane];
        const float4 *h4 = reinterpret_cast<const float4 *>(tb + kTblHH + trip_off(i, J));
#pragma unroll
        for (int q = 0; q < nq; ++q) {
            const float4 h = h4[q];
            const float hs[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int t = 4 * q + r;
                if (t < n) acc[t] = fminf(acc[t], fmaf(lam, hs[r], g));
            }
        }
    }
    const float4 *d4 = reinterpret_cast<const float4 *>(tb + kTblD + dp_off(J));
#pragma unroll
    for (int q = 0; q < nq; ++q) {
        const float4 dd = d4[q];
        const float ds[4] = {dd.x, dd.y, dd.z, dd.w};
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int t = 4 * q + r;
            if (t < n) {
                if (t == 0) sG0[(J + 1) * 32 + lane] = acc0 + ds[r];
                sG1[pidx(J, J + 1 + t) * 32 + lane] = acc[t] + ds[r];
            }
        }
    }
    if constexpr (J < 15) dp_a_stage<J + 1>(tb, lam, sG1, sG0, lane);
}

__device__ __forceinline__ void dp_path_a(const float *__restrict__ tb, float lam, int C,
                                          float *__restrict__ sG1, float *__restrict__ sG0,
                                          int lane, float &rate, uint32_t &mask) {
    const float INF = __int_as_float(0x7f800000);
#define G1(j, l) sG1[pidx(j, l) * 32 + lane]
#define G0(j) sG0[(j) * 32 + lane]
    // chains (0, l)
    {
        float dv[16], hv[16];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const float4 a = reinterpret_cast<const float4 *>(tb + kTblD + dp_off(0))[t];
            const float4 h = reinterpret_cast<const float4 *>(tb + kTblH0)[t];
            dv[4 * t] = a.x; dv[4 * t + 1] = a.y; dv[4 * t + 2] = a.z; dv[4 * t + 3] = a.w;
            hv[4 * t] = h.x; hv[4 * t + 1] = h.y; hv[4 * t + 2] = h.z; hv[4 * t + 3] = h.w;
        }
        const float h16 = tb[kTblH0 + 16];
#pragma unroll
        for (int l = 1; l < 17; ++l) {
            const float v = fmaf(lam, l < 16 ? hv[l] : h16, dv[l - 1]);
            if (l == 1) { G0(1) = v; G1(0, 1) = INF; }
            else G1(0, l) = v;
        }
    }
    dp_a_stage<1>(tb, lam, sG1, sG0, lane);
    // final level (slot 16)
    float best = INF;
    int bi = -1;
    if (C == 0) best = fmaf(lam, tb[kTblHend + 15], G0(16));
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float v = fmaf(lam, tb[kTblHend + i], G1(i, 16));
        if (v < best) { best = v; bi = i; }
    }
    if (bi < 0) {   // the chain through every slot
        mask = 0x1ffffu;
        float r = tb[kTblH0 + 1];
        for (int j = 1; j < 16; ++j) r += hh_at(tb, j - 1, j, j + 1);
        rate = r + tb[kTblHend + 15];
        return;
    }
    // walk back: at state (j, l) find the predecessor whose candidate equals
    // the minimum (recomputed with the same operations, so equality is exact)
    uint32_t m = (1u << 16) | (1u << bi);
    float r = tb[kTblHend + bi];
    int j = bi, l = 16;
    bool from_start = true;
    for (int guard = 0; guard < 17 && j > 0; ++guard) {
        const float cg0 = fmaf(lam, hh_at(tb, j - 1, j, l), G0(j));
        float acc = (l >= j + 2) ? cg0 : INF;
        for (int i = 0; i < j; ++i) acc = fminf(acc, fmaf(lam, hh_at(tb, i, j, l), G1(i, j)));
        if (l >= j + 2 && cg0 == acc) {           // the no-skip prefix 0..j
            r += hh_at(tb, j - 1, j, l);
            m |= (1u << (j + 1)) - 1u;
            r += tb[kTblH0 + 1];
            for (int t = 1; t < j; ++t) r += hh_at(tb, t - 1, t, t + 1);
            from_start = false;
            break;
        }
        int pred = -1;
        for (int i = 0; i < j; ++i)
            if (fmaf(lam, hh_at(tb, i, j, l), G1(i, j)) == acc) {
                pred = i;
                break;
            }
        if (pred < 0) { from_start = false; break; }   // non-finite data only
        r += hh_at(tb, pred, j, l);
        m |= 1u << pred;
        l = j;
        j = pred;
    }
    if (from_start && j == 0) {
        r += tb[kTblH0 + l];
        m |= 1u;
    }
    rate = r;
    mask = m;
#undef G1
#undef G0
}

// ---------------------------------------------------------------- DP path B
// Any s: "at most k levels" relaxation, k = 2 .. s, in place (rows in
// decreasing j so every row reads the previous round's columns), carrying
// the chain's rate and mask with its value.
__device__ void dp_path_b(const float *__restrict__ tb, float lam, int s,
                          float *__restrict__ sG, float *__restrict__ sR,
                          uint32_t *__restrict__ sM, int lane, float &rate, uint32_t &mask) {
    const float INF = __int_as_float(0x7f800000);
    for (int p = 0; p < kPairs; ++p) sG[p * 32 + lane] = INF;
    for (int l = 1; l < 17; ++l) {
        const int p = pidx(0, l);
        sG[p * 32 + lane] = fmaf(lam, tb[kTblH0 + l], dp_at(tb, 0, l));
        sR[p * 32 + lane] = tb[kTblH0 + l];
        sM[p * 32 + lane] = 1u | (1u << l);
    }
    for (int it = 0; it < s - 2; ++it) {
        for (int j = 15; j >= 1; --j) {
            for (int l = j + 1; l < 17; ++l) {
                const int pjl = pidx(j, l);
                float best = sG[pjl * 32 + lane];
                const float dv = dp_at(tb, j, l);
                int bi = -1;
                for (int i = 0; i < j; ++i) {
                    const float c = fmaf(lam, hh_at(tb, i, j, l), sG[pidx(i, j) * 32 + lane]) + dv;
                    if (c < best) { best = c; bi = i; }
                }
                if (bi >= 0) {
                    const int pij = pidx(bi, j);
                    sG[pjl * 32 + lane] = best;
                    sR[pjl * 32 + lane] = sR[pij * 32 + lane] + hh_at(tb, bi, j, l);
                    sM[pjl * 32 + lane] = sM[pij * 32 + lane] | (1u << l);
                }
            }
        }
    }
    float best = INF;
    int bi = 0;
    for (int i = 0; i < 16; ++i) {
        const float v = fmaf(lam, tb[kTblHend + i], sG[pidx(i, 16) * 32 + lane]);
        if (v < best) { best = v; bi = i; }
    }
    const int p = pidx(bi, 16);
    rate = sR[p * 32 + lane] + tb[kTblHend + bi];
    mask = sM[p * 32 + lane];
}

// ------------------------------------------------------------- search round
template <bool GENERAL>
struct RoundCfg {
    static constexpr int kWarps = GENERAL ? kRoundWarpsGen : kRoundWarps;
    // per-warp lane-private state (floats): path A needs 136 + 17 per lane,
    // path B 3 * 136 per lane
    static constexpr int kStateFloats = (GENERAL ? 3 * kPairs : kPairs + 17) * 32;
    static constexpr size_t kSmem =
        (size_t)kWarps * (kTblStride + kStateFloats) * sizeof(float) +
        (size_t)kWarps * 32 * sizeof(float);
};

template <bool GENERAL>
__global__ void __launch_bounds__(RoundCfg<GENERAL>::kWarps * 32)
search_round_kernel(const float *__restrict__ tables, int64_t nb, int s, Ctrl *__restrict__ ctrl,
                    float *__restrict__ rates, uint32_t *__restrict__ masks,
                    float *__restrict__ rate_lo, float *__restrict__ rate_hi,
                    uint32_t *__restrict__ mask_hi, uint8_t *__restrict__ act) {
    using Cfg = RoundCfg<GENERAL>;
    constexpr int W = Cfg::kWarps;
    extern __shared__ __align__(16) float smem[];
    const Ctrl c = *ctrl;
    if (c.phase == kPhaseDone) return;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    float *sTbl = smem + w * kTblStride;
    float *sState = smem + W * kTblStride + w * Cfg::kStateFloats;
    float *sRate = smem + W * (kTblStride + Cfg::kStateFloats);
    __shared__ bool is_last;

    const int64_t b = (int64_t)blockIdx.x * W + w;
    float my_rate = 0.f;
    if (b < nb) {
        // carry the previous round's results at the new lo / hi
        bool active = true;
        if (c.phase == kPhaseBisect) {
            // lane 0 alone touches the per-block state, then broadcasts
            float rl = 0.f, rh = 0.f;
            if (lane == 0) {
                const bool was = act[b] != 0;
                rl = rate_lo[b];
                rh = rate_hi[b];
                if (was && c.lo_probe >= 0) rl = rates[b * 32 + c.lo_probe];
                if (was && c.hi_probe >= 0) {
                    rh = rates[b * 32 + c.hi_probe];
                    mask_hi[b] = masks[b * 32 + c.hi_probe];
                }
                rate_lo[b] = rl;
                rate_hi[b] = rh;
            }
            rl = __shfl_sync(0xffffffffu, rl, 0);
            rh = __shfl_sync(0xffffffffu, rh, 0);
            // the rate is non-increasing in lambda: equal at both ends means
            // constant on [lo, hi], and so is the chosen chain
            active = rl != rh;
            my_rate = rh;
        }
        if (lane == 0) act[b] = active ? 1 : 0;
        if (active) {
            const float4 *src = reinterpret_cast<const float4 *>(tables + b * kTblStride);
            float4 *dst = reinterpret_cast<float4 *>(sTbl);
            for (int i = lane; i < kTblStride / 4; i += 32) dst[i] = src[i];
            __syncwarp();
            const double hi0 = __longlong_as_double((long long)c.hi0_bits);
            const float lam = (float)probe_lambda(c, hi0, lane);
            const int mp = min(max(__float_as_int(sTbl[kTblHdr]), 1), kCand);
            float rate;
            uint32_t mask;
            if (mp <= 1) {
                rate = 0.f;
                mask = 1u;
            } else {
                const int C = mp > s ? mp - s : 0;
                if (!GENERAL || C == 0 || (C == 1 && mp == 17)) {
                    dp_path_a(sTbl, lam, C, sState, sState + kPairs * 32, lane, rate, mask);
                } else {
                    dp_path_b(sTbl, lam, s, sState, sState + kPairs * 32,
                              reinterpret_cast<uint32_t *>(sState + 2 * kPairs * 32), lane, rate,
                              mask);
                }
            }
            rates[b * 32 + lane] = rate;
            masks[b * 32 + lane] = mask;
            my_rate = rate;
        }
    }
    sRate[w * 32 + lane] = my_rate;
    __syncthreads();
    if (threadIdx.x < 32) {
        double sum = 0.0;
        for (int k = 0; k < W; ++k) sum += (double)sRate[k * 32 + threadIdx.x];
        atomicAdd(&ctrl->acc[threadIdx.x], (unsigned long long)llrint(sum * kRateScale));
        __threadfence();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned t = atomicAdd(&ctrl->ticket, 1u);
        is_last = (t == gridDim.x - 1);
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();

    // ---- last CTA: read the sums, advance the search
    __shared__ double R[32];
    if (threadIdx.x < 32) {
        const unsigned long long a = atomicExch(&ctrl->acc[threadIdx.x], 0ull);
        R[threadIdx.x] = (double)a / kRateScale;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        Ctrl n = *ctrl;
        const double B = n.budget;
        const double hi0 = __longlong_as_double((long long)n.hi0_bits);
        n.ticket = 0u;
        n.hi_probe = -1;
        n.lo_probe = -1;
        if (n.phase == kPhaseFixed) {
            n.hi_probe = 0;
            n.R_hi = R[0];
            n.phase = kPhaseDone;
        } else if (n.phase == kPhaseBracket) {
            if (R[0] <= B) {
                n.lo = n.hi = n.lambda = 0.0;
                n.hi_probe = 0;
                n.R_hi = R[0];
                n.phase = kPhaseDone;
            } else {
                int t = 1;
                while (t < 32 && !(R[t] <= B)) ++t;
                n.lo = 0.0;
                n.lo_probe = 0;
                if (t < 32) {
                    n.hi = ldexp(hi0, t - 1);
                    n.hi_probe = t;
                    n.R_hi = R[t];
                    n.phase = kPhaseBisect;
                    n.step = 0;
                } else {
                    n.hi = n.lambda = ldexp(hi0, kMaxDoublings);
                    n.hi_probe = 31;
                    n.R_hi = R[31];
                    n.status = KVQ_ERR_INFEASIBLE;
                    n.phase = kPhaseDone;
                }
            }
        } else {   // bisection: 5 steps down the evaluated tree
            double a = n.lo, bb = n.hi;
            int cur = 16, half = 8;
            for (int lev = 0; lev < kLevelsPerRound && n.step < kBisectSteps; ++lev) {
                const double mid = 0.5 * (a + bb);
                if (R[cur - 1] <= B) {
                    bb = mid;
                    n.hi_probe = cur - 1;
                    n.R_hi = R[cur - 1];
                    cur -= half;
                } else {
                    a = mid;
                    n.lo_probe = cur - 1;
                    cur += half;
                }
                half >>= 1;
                ++n.step;
            }
            n.lo = a;
            n.hi = bb;
            if (n.step >= kBisectSteps) {
                n.lambda = n.hi;
                n.phase = kPhaseDone;
            }
        }
        for (int i = 0; i < 32; ++i) n.acc[i] = 0ull;
        *ctrl = n;
        __threadfence();
    }
}

// -------------------------------------------------------------------- emit
__global__ void __launch_bounds__(kEmitThreads)
emit_kernel(const float *__restrict__ tables, int64_t nb, Ctrl *__restrict__ ctrl,
            const float *__restrict__ rates, const uint32_t *__restrict__ masks,
            const float *__restrict__ rate_hi, const uint32_t *__restrict__ mask_hi,
            const uint8_t *__restrict__ act, double *__restrict__ epartial,
            float *__restrict__ codebook, uint8_t *__restrict__ kout, float *__restrict__ Dr,
            float *__restrict__ Hr, double *__restrict__ totals, double *__restrict__ lambda_out,
            int32_t *__restrict__ status) {
    const Ctrl c = *ctrl;
    const int64_t b = (int64_t)blockIdx.x * kEmitThreads + threadIdx.x;
    double myD = 0.0;
    if (b < nb) {
        const float *tb = tables + b * kTblStride;
        uint32_t mask;
        float rate;
        if (c.hi_probe >= 0 && act[b]) {
            mask = masks[b * 32 + c.hi_probe];
            rate = rates[b * 32 + c.hi_probe];
        } else {
            mask = mask_hi[b];
            rate = rate_hi[b];
        }
        const int d = __float_as_int(tb[kTblHdr + 1]);
        float q[16];
        int k = 0;
        float Dsum = 0.f;
        int prev = -1;
        for (int t = 0; t < 17; ++t) {
            if (!(mask >> t & 1u)) continue;
            q[k < 16 ? k : 15] = tb[kTblC + t];
            if (prev >= 0) Dsum += dp_at(tb, prev, t);
            prev = t;
            ++k;
        }
        if (k > 16) k = 16;   // cannot happen for s <= 16
        if (k == 0) { k = 1; q[0] = tb[kTblC]; }
        for (int t = k; t < 16; ++t) q[t] = q[k - 1];
        float4 *cb = reinterpret_cast<float4 *>(codebook + b * 16);
#pragma unroll
        for (int t = 0; t < 4; ++t) cb[t] = make_float4(q[4 * t], q[4 * t + 1], q[4 * t + 2], q[4 * t + 3]);
        kout[b] = (uint8_t)k;
        Dr[b] = Dsum;
        Hr[b] = rate / (float)d;
        myD = (double)Dsum;
    }
    // fixed-order block reduction of sum D_r
    __shared__ double sD[kEmitThreads / 32];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) myD += __shfl_down_sync(0xffffffffu, myD, o);
    if (lane == 0) sD[w] = myD;
    __syncthreads();
    __shared__ bool is_last;
    if (threadIdx.x == 0) {
        double dd = 0.0;
        for (int k = 0; k < kEmitThreads / 32; ++k) dd += sD[k];
        epartial[2 * blockIdx.x] = 0.0;
        epartial[2 * blockIdx.x + 1] = dd;
        __threadfence();
        const unsigned t = atomicAdd(&ctrl->ticket_emit, 1u);
        is_last = (t == gridDim.x - 1);
    }
    __syncthreads();
    if (!is_last || threadIdx.x != 0) return;
    __threadfence();
    double dd = 0.0;
    for (unsigned k = 0; k < gridDim.x; ++k) dd += __ldcg(&epartial[2 * k + 1]);
    Ctrl n = *ctrl;
    const double R = n.R_hi;   // the rate the search tested (same per-block rates)
    const double lam = n.lambda;
    totals[0] = R;
    totals[1] = dd;
    totals[2] = lam;
    if (n.mode == KVQ_SUBGRADIENT) {
        const double nl = lam + n.eta * (R - n.budget);
        *lambda_out = nl > 0.0 ? nl : 0.0;
    } else {
        *lambda_out = lam;
    }
    int st = n.status;
    if (n.flags & kFlagNonfinite) st = KVQ_ERR_NONFINITE;
    *status = st;
    n.ticket_emit = 0u;
    *ctrl = n;
}

__global__ void empty_alloc_kernel(double *totals, double *lambda_out, int32_t *status, int mode,
                                   double eta, double budget) {
    if (threadIdx.x != 0) return;
    const double lam = (mode == KVQ_SUBGRADIENT) ? *lambda_out : 0.0;
    totals[0] = 0.0;
    totals[1] = 0.0;
    totals[2] = lam;
    if (mode == KVQ_SUBGRADIENT) {
        const double nl = lam + eta * (0.0 - budget);
        *lambda_out = nl > 0.0 ? nl : 0.0;
    } else {
        *lambda_out = 0.0;
    }
    *status = KVQ_OK;
}

int launch_allocate(const void *stats, const kvq_layout &L, int s, double budget, int mode,
                    double eta, double *lambda, void *workspace, float *codebook, uint8_t *k,
                    float *Dr, float *Hr, double *totals, int32_t *status, cudaStream_t st) {
    const int64_t nb = num_blocks(L);
    if (nb == 0) {
        empty_alloc_kernel<<<1, 32, 0, st>>>(totals, lambda, status, mode, eta, budget);
        return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
    }
    Workspace ws = carve(workspace, nb);
    ctrl_init_kernel<<<1, 32, 0, st>>>(ws.ctrl, budget, eta, mode, lambda);
    const unsigned tgrid = (unsigned)((nb + kTablesWarps - 1) / kTablesWarps);
    tables_kernel<<<tgrid, kTablesWarps * 32, 0, st>>>(static_cast<const StatsRow *>(stats), nb,
                                                       ws.tables, ws.ctrl);
    const int rounds = (mode == KVQ_SUBGRADIENT) ? 1 : 1 + kBisectSteps / kLevelsPerRound;
    const bool general = s < 16;
    for (int r = 0; r < rounds; ++r) {
        if (general) {
            using Cfg = RoundCfg<true>;
            const unsigned grid = (unsigned)((nb + Cfg::kWarps - 1) / Cfg::kWarps);
            search_round_kernel<true><<<grid, Cfg::kWarps * 32, Cfg::kSmem, st>>>(
                ws.tables, nb, s, ws.ctrl, ws.rates, ws.masks, ws.rate_lo, ws.rate_hi, ws.mask_hi,
                ws.act);
        } else {
            using Cfg = RoundCfg<false>;
            const unsigned grid = (unsigned)((nb + Cfg::kWarps - 1) / Cfg::kWarps);
            search_round_kernel<false><<<grid, Cfg::kWarps * 32, Cfg::kSmem, st>>>(
                ws.tables, nb, s, ws.ctrl, ws.rates, ws.masks, ws.rate_lo, ws.rate_hi, ws.mask_hi,
                ws.act);
        }
    }
    const unsigned egrid = (unsigned)((nb + kEmitThreads - 1) / kEmitThreads);
    emit_kernel<<<egrid, kEmitThreads, 0, st>>>(ws.tables, nb, ws.ctrl, ws.rates, ws.masks,
                                                ws.rate_hi, ws.mask_hi, ws.act, ws.epartial,
                                                codebook, k, Dr, Hr, totals, lambda, status);
    return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

int allocate_init() {
    // opt in to more than 48 KB of dynamic shared memory for the search rounds
    if (cudaFuncSetAttribute(search_round_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)RoundCfg<false>::kSmem) != cudaSuccess)
        return KVQ_ERR_CUDA;
    if (cudaFuncSetAttribute(search_round_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)RoundCfg<true>::kSmem) != cudaSuccess)
        return KVQ_ERR_CUDA;
    return KVQ_OK;
}

}  // namespace kvq
