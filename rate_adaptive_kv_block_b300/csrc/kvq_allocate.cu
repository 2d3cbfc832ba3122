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
//   ctrl_init      reset the control block in the workspace
//   (the lambda-independent DP tables of every block -- interval distortion
//   and entropy terms in "slot" space, see kvq_internal.cuh -- come from
//   kvq_stats, with max_r (c_max - c_min)^2 in the stats header)
//   search_kernel  one persistent, cooperative launch for every round of the
//                  search and the emit.  In a round, one warp per block and
//                  one lane per probe lambda: each lane runs the whole exact
//                  DP at its own lambda, so the warp evaluates 32 lambdas
//                  with no cross-lane traffic and the table reads are
//                  shared-memory broadcasts.  Per-probe rate sums are exact
//                  fixed-point integer atomics; once every CTA is in, CTA 0
//                  advances the search (kvq_search.h) and releases the grid
//                  for the next round:
//                    pilot round (large tensors): a sample of the blocks at
//                    the bracket probes, for an estimate of lambda;
//                    round 0: probes 0, hi0 * 2^{0,1,2} and a grid (around
//                    the estimate when there is one);
//                    bisection rounds: the unknown nodes of the next 5
//                    levels of the bisection tree under [lo, hi] -- every
//                    midpoint the sequential bisection could visit next --
//                    then the walk takes those steps: the same lambda as 40
//                    sequential steps.
//                  Emit, after the last round: per block, the chain at the
//                  final lambda (recorded by the round that evaluated it) ->
//                  codebook, k, D_r, H_r; totals; the subgradient update in
//                  KVQ_SUBGRADIENT mode.
#include <math.h>

#include "kvq_internal.cuh"
#include "kvq_quant_core.cuh"

namespace kvq {

constexpr int kRoundWarps = 4;        // s >= 16: DP path A only
constexpr int kRoundWarpsGen = 2;     // s < 16: path B possible
constexpr int kMaxGrid = 4096;        // CTAs of the persistent search kernel (at most)

// CTAs of the persistent search kernel resident at once, per device (set by
// allocate_init, which the API runs once per device before the first launch)
constexpr int kMaxDevices = 64;
static int g_resident[kMaxDevices][2][2];   // [device][s < 16][fused]

// Scratch of kvq_allocate_static: a fixed array in this module's global
// memory, which also holds the search kernel.  The CUDA runtime creates it on
// a device when it loads this module there, which allocate_init forces (it
// sets the search kernel's attributes), and frees it when the process exits.
// Host code cannot use the name as a device address; allocate_init looks the
// address up once per device (cudaGetSymbolAddress) and keeps it here.
static __device__ __align__(256) unsigned char g_static_workspace[KVQ_STATIC_WORKSPACE_BYTES];
static void *g_static_addr[kMaxDevices];

// lambdas of one evaluation of the global search (kernel parameter)
struct ProbeSet {
    double lambda[kSearchProbes];
    int n;
};

// ---------------------------------------------------------------- workspace
struct Workspace {
    Ctrl *ctrl;
    float *rates;         // [nblk][32]   d_r H_r per probe (last round)
    uint32_t *masks;      // [nblk][32]   chain per probe (last round)
    float *rate_lo;       // [nblk]       d_r H_r at xa
    float *rate_hi;       // [nblk]       d_r H_r at xb
    uint32_t *mask_hi;    // [nblk]       chain at xb
    int32_t *evr;         // [nblk]       round that last evaluated the block
    int32_t *list;        // [2][nblk]    candidate lists (ping-pong)
    double *epartial;     // [nblk / 32]  D_r summed over each 32 consecutive blocks
    int32_t *fin;         // [nblk]       fused path: blocks in the order their chain became final
    uint8_t *fflag;       // [nblk]       fused path: 1 once queued
};

static size_t align_up(size_t v) { return (v + 255) & ~(size_t)255; }

size_t workspace_bytes(int64_t nb, int s) {
    (void)s;
    size_t b = align_up(sizeof(Ctrl));
    b += align_up((size_t)nb * 32 * sizeof(float));
    b += align_up((size_t)nb * 32 * sizeof(uint32_t));
    b += 3 * align_up((size_t)nb * sizeof(float));
    b += align_up((size_t)nb * sizeof(int32_t));
    b += align_up((size_t)nb * 2 * sizeof(int32_t));
    b += align_up((size_t)((nb + 31) / 32) * sizeof(double));
    b += align_up((size_t)nb * sizeof(int32_t));
    b += align_up((size_t)nb);
    return b;
}

static Workspace carve(void *base, int64_t nb) {
    char *p = static_cast<char *>(base);
    Workspace w;
    w.ctrl = reinterpret_cast<Ctrl *>(p);
    p += align_up(sizeof(Ctrl));
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
    w.evr = reinterpret_cast<int32_t *>(p);
    p += align_up((size_t)nb * sizeof(int32_t));
    w.list = reinterpret_cast<int32_t *>(p);
    p += align_up((size_t)nb * 2 * sizeof(int32_t));
    w.epartial = reinterpret_cast<double *>(p);
    p += align_up((size_t)((nb + 31) / 32) * sizeof(double));
    w.fin = reinterpret_cast<int32_t *>(p);
    p += align_up((size_t)nb * sizeof(int32_t));
    w.fflag = reinterpret_cast<uint8_t *>(p);
    return w;
}

// ---------------------------------------------------------------- ctrl init
// pilot round over 1/16 of the blocks when there are at least this many
constexpr int64_t kPilotMinBlocks = 1024;
constexpr int kPilotStride = 16;

__global__ void ctrl_init_kernel(Ctrl *c, const StatsHeader *hdr, double budget, double eta,
                                 int mode, const double *lambda_in, int64_t nb,
                                 unsigned long long wait_ns, uint32_t spin_limit) {
    if (threadIdx.x != 0) return;
    search_init(c->s);
    c->s.hi0 = __longlong_as_double((long long)hdr->hi0_bits);
    c->s.f32_lambda = 1;      // the DP runs at float(lambda)
    c->nb = nb;
    if (mode != KVQ_SUBGRADIENT && nb >= kPilotMinBlocks) search_set_pilot(c->s, nb, kPilotStride);
    c->budget = budget;
    c->budget_fx = budget_fx(budget);
    c->eta = eta;
    c->fixed = (mode == KVQ_SUBGRADIENT) ? 1 : 0;
    c->lambda_fixed = c->fixed ? *lambda_in : 0.0;
    c->hi0_bits = hdr->hi0_bits;
    c->status = KVQ_OK;
    c->flags = (int32_t)hdr->flags;
    c->mode = mode;
    c->ticket = 0u;
    c->ticket_emit = 0u;
    c->gen = 0u;
    c->err = 0u;
    c->fin_tail = 0u;
    c->fin_avail = 0u;
    c->ticket_f = 0u;
    for (int i = 0; i < 32; ++i) c->acc[i] = 0ull;
    for (int i = 0; i < 16; ++i) c->active[i] = 0u;
    c->Rxb_fx = 0;
    c->cnt[0] = c->cnt[1] = 0u;
    c->t_start = c->t_end = 0ull;
    c->wait_ns = wait_ns;
    c->spin_limit = spin_limit;
    c->phase1 = c->s.phase;
    for (int i = 0; i < 16; ++i) c->t_dp[i] = c->t_ctl[i] = 0ull;
}

// ---------------------------------------------------------------- DP path A
// Exact minimiser over all chains 0 = l_0 < ... < l_{k-1} = 16 (slot space)
// that either may use every slot (C == 0) or must skip at least one
// (C == 1: m' = 17 and s = 16).  Layer 0 holds the single chain 0,1,..,j
// (state (j-1, j)); layer 1 every chain that already skipped a slot.
// State value G(j,l): distortion of the intervals up to (j,l) plus lambda
// times the entropy terms of the levels before l.  Lane-private state in
// shared memory, [pair][lane].  Returns the chain's d_r H_r and its mask.
// min(a, b, c) in one instruction
__device__ __forceinline__ float fmin3(float a, float b, float c) {
    float r;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
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
    // predecessors i in pairs: two targets per packed fused multiply-add
    // (same rounding as fmaf), one three-input minimum per target and pair
    // (a minimum is exact, so the result is that of the pairwise chain)
    const float2 l2 = make_float2(lam, lam);
#pragma unroll
    for (int i = 0; i < J; i += 2) {
        const bool two = i + 1 < J;
        const float ga = sG1[pidx(i, J) * 32 + lane];
        const float gb = two ? sG1[pidx(i + 1 < J ? i + 1 : i, J) * 32 + lane] : 0.f;
        const float2 ga2 = make_float2(ga, ga), gb2 = make_float2(gb, gb);
        const float4 *ha4 = reinterpret_cast<const float4 *>(tb + kTblHH + trip_off(i, J));
        const float4 *hb4 = reinterpret_cast<const float4 *>(
            tb + kTblHH + trip_off(i + 1 < J ? i + 1 : i, J));
#pragma unroll
        for (int q = 0; q < nq; ++q) {
            const float4 ha = ha4[q];
            const float2 a01 = __ffma2_rn(l2, make_float2(ha.x, ha.y), ga2);
            const float2 a23 = __ffma2_rn(l2, make_float2(ha.z, ha.w), ga2);
            const float as[4] = {a01.x, a01.y, a23.x, a23.y};
            if (two) {
                const float4 hb = hb4[q];
                const float2 b01 = __ffma2_rn(l2, make_float2(hb.x, hb.y), gb2);
                const float2 b23 = __ffma2_rn(l2, make_float2(hb.z, hb.w), gb2);
                const float bs[4] = {b01.x, b01.y, b23.x, b23.y};
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int t = 4 * q + r;
                    if (t < n) acc[t] = fmin3(acc[t], as[r], bs[r]);
                }
            } else {
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int t = 4 * q + r;
                    if (t < n) acc[t] = fminf(acc[t], as[r]);
                }
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

// Walk back one stage: if the chain's current state is (J, l), find the
// predecessor whose candidate is the minimum (recomputed with the same
// operations, so the comparison is exact) and add level J's entropy term.
template <int J>
__device__ __forceinline__ void dp_a_back(const float *__restrict__ tb, float lam,
                                          const float *__restrict__ sG1,
                                          const float *__restrict__ sG0,
                                          const float *__restrict__ diag, int lane, int &cj,
                                          int &cl, float &r, uint32_t &m, bool &open) {
    if (open && cj == J) {
        const float INF = __int_as_float(0x7f800000);
        const float *hrow = tb + kTblHH + (cl - J - 1);    // hh(., J, cl) at trip_off(., J)
        float best = INF, hsel = 0.f;
        int arg = -2;
        if (cl >= J + 2) {
            hsel = hrow[trip_off(J - 1, J)];
            best = fmaf(lam, hsel, sG0[J * 32 + lane]);
            arg = -1;
        }
#pragma unroll
        for (int i = 0; i < J; ++i) {
            const float h = hrow[trip_off(i, J)];
            const float c = fmaf(lam, h, sG1[pidx(i, J) * 32 + lane]);
            if (c < best) { best = c; arg = i; hsel = h; }
        }
        if (arg == -1) {                 // the no-skip prefix 0, 1, .., J
            r += hsel + diag[J];
            m |= (1u << (J + 1)) - 1u;
            open = false;
        } else if (arg >= 0) {
            r += hsel;
            m |= 1u << arg;
            cl = J;
            cj = arg;
        } else {
            open = false;                // non-finite data only
        }
    }
    if constexpr (J > 1) dp_a_back<J - 1>(tb, lam, sG1, sG0, diag, lane, cj, cl, r, m, open);
}

// diag[J] = entropy terms of levels 0 .. J-1 of the chain 0, 1, .., J
__device__ __forceinline__ void dp_a_diag(const float *__restrict__ tb, float *__restrict__ diag,
                                          int lane) {
    float v = 0.f;
    if (lane == 0) v = tb[kTblH0 + 1];
    else if (lane < 16) v = tb[kTblHH + trip_off(lane - 1, lane)];     // hh(lane-1, lane, lane+1)
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
    }
    if (lane < 16) diag[lane + 1] = v;
    __syncwarp();
}

__device__ __forceinline__ void dp_path_a(const float *__restrict__ tb, float lam, int C,
                                          float *__restrict__ sG1, float *__restrict__ sG0,
                                          const float *__restrict__ diag, int lane, float &rate,
                                          uint32_t &mask) {
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
        rate = diag[16] + tb[kTblHend + 15];
        return;
    }
    uint32_t m = (1u << 16) | (1u << bi);
    float r = tb[kTblHend + bi];
    int cj = bi, cl = 16;
    bool open = true;
    dp_a_back<15>(tb, lam, sG1, sG0, diag, lane, cj, cl, r, m, open);
    if (open && cj == 0) {
        r += tb[kTblH0 + cl];
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

// A block's DP tables (kTblStride floats) into the warp's shared memory:
// every lane's 16-byte loads issued before any store, so the copy costs one
// L2 round trip (L2 only: the stats kernel wrote them).
__device__ __forceinline__ void load_tables(float *__restrict__ sTbl, const float *__restrict__ tables,
                                            int64_t b, int lane) {
    constexpr int kN4 = kTblStride / 4;
    constexpr int kPer = (kN4 + 31) / 32;
    const float4 *src = reinterpret_cast<const float4 *>(tables + b * kRecFloats + kRecTbl);
    float4 *dst = reinterpret_cast<float4 *>(sTbl);
    float4 v[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int i = lane + 32 * k;
        if (i < kN4) v[k] = __ldcg(src + i);
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int i = lane + 32 * k;
        if (i < kN4) dst[i] = v[k];
    }
}

// ------------------------------------------------- fused emit + quantize
// The allocate-and-quantize path quantizes each block as soon as its chain is
// final -- a block whose rate is equal at both ends of the window is constant
// inside it, so its choice at the final lambda is already known -- using the
// warps that the late, nearly empty rounds of the search leave idle.
struct QuantArgs {
    const uint16_t *x;      // [S, T, D] binary16
    uint8_t *codes;         // [nblocks][16 group]
    uint64_t index_base;
    PhiloxKey key;          // round keys of the seed
    int D, G;
    int lg_ng;              // log2(D / G)
    int lg_upr;             // log2(G / 8)
};

// Per block, once: from the block's final chain `mask`, the levels, the
// quantizer's thresholds T[1..15] (returned) and decision table (in
// `scratch`, 64 floats of the warp's own shared memory); with `emit`, also
// the block's codebook, k, D_r, H_r -- the same arithmetic, in the same
// order, as the emit of kvq_allocate.
__device__ __forceinline__ void fused_prepare(const float *__restrict__ tables, int64_t b,
                                              uint32_t mask, float rate, bool emit,
                                              float *__restrict__ codebook,
                                              uint8_t *__restrict__ kout, float *__restrict__ Dr,
                                              float *__restrict__ Hr, float *scratch, int lane,
                                              uint32_t (&T)[16]) {
    const float *tb = tables + b * kRecFloats + kRecTbl;
    mask &= 0x1ffffu;
    if (mask == 0u) mask = 1u;
    const int k = min(__popc(mask), 16);
    float *q = scratch;                                             // 16 levels
    __half2 *thr = reinterpret_cast<__half2 *>(scratch + 16);       // 16 thresholds
    float2 *qw = reinterpret_cast<float2 *>(scratch + 32);          // 16 decision entries
    const bool in = lane < 17 && ((mask >> lane) & 1u);
    const int pos = __popc(mask & ((1u << lane) - 1u));
    const float qv = lane < 17 ? tb[kTblC + lane] : 0.f;
    __syncwarp();                                                   // scratch free
    if (in && pos < 16) q[pos] = qv;
    __syncwarp();
    if (lane < 16 && lane >= k) q[lane] = q[k - 1];
    __syncwarp();
    if (emit) {
        if (lane < 16) codebook[b * 16 + lane] = q[lane];
        if (lane == 0) {
            float dv = 0.f;
            int prev = 0;
#pragma unroll
            for (int t = 0; t < 17; ++t) {
                const bool on = (mask >> t) & 1u;
                const bool link = on && t > 0;
                const float dd = tb[kTblD + (link ? dp_off(prev) + t - prev - 1 : 0)];
                if (link) dv += dd;
                if (on) prev = t;
            }
            const int d = __float_as_int(tb[kTblHdr + 1]);
            kout[b] = (uint8_t)k;
            Dr[b] = dv;
            Hr[b] = rate / (float)d;
        }
    }
    if (lane < 16) quant_table_entry(q, k, lane, thr[lane], qw[lane]);
    __syncwarp();
    T[0] = 0u;
#pragma unroll
    for (int j = 1; j < 16; ++j) {
        const __half2 h = thr[j];
        memcpy(&T[j], &h, 4);
    }
}

// The binary16 input of rows 4 part .. 4 part + 3 of block b: this lane's
// (at most two) 8-entry units.
__device__ __forceinline__ void fused_load(const QuantArgs &qa, int64_t b, int part, int lane,
                                           uint4 (&raw)[2]) {
    const int upr = qa.G >> 3, units = 4 << qa.lg_upr;
    const int64_t tbk = b >> qa.lg_ng;
    const int g = (int)(b & ((1 << qa.lg_ng) - 1));
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int u = lane + 32 * r;
        if (u < units) {
            const int row = 4 * part + (u >> qa.lg_upr), cu = u & (upr - 1);
            const int64_t flat = (tbk * 32 + row) * (int64_t)qa.D + (int64_t)g * qa.G + cu * 8;
            raw[r] = __ldg(reinterpret_cast<const uint4 *>(qa.x + flat));
        }
    }
}

// Codes of rows 4 part .. 4 part + 3 of block b from the loaded input.
__device__ __forceinline__ void fused_codes(const QuantArgs &qa, int64_t b, int part, int lane,
                                            const uint4 (&raw)[2], const uint32_t (&T)[16],
                                            const float *scratch) {
    const float2 *qw = reinterpret_cast<const float2 *>(scratch + 32);
    const int G = qa.G, upr = G >> 3, units = 4 << qa.lg_upr;
    const int64_t tbk = b >> qa.lg_ng;
    const int g = (int)(b & ((1 << qa.lg_ng) - 1));
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int u = lane + 32 * r;
        if (u < units) {
            const int row = 4 * part + (u >> qa.lg_upr), cu = u & (upr - 1);
            const int64_t flat = (tbk * 32 + row) * (int64_t)qa.D + (int64_t)g * G + cu * 8;
            const uint32_t packed =
                quant8(raw[r], T, qw, quant_counter(qa.index_base, (uint64_t)flat), qa.key);
            *reinterpret_cast<uint32_t *>(qa.codes + b * (int64_t)(16 * G) +
                                          ((row * G + cu * 8) >> 1)) = packed;
        }
    }
}

// ------------------------------------------------------------ search kernel
template <bool GENERAL>
struct RoundCfg {
    static constexpr int kWarps = GENERAL ? kRoundWarpsGen : kRoundWarps;
    // per-warp lane-private state (floats): path A needs 136 + 17 per lane,
    // path B 3 * 136 per lane
    static constexpr int kStateFloats = (GENERAL ? 3 * kPairs : kPairs + 17) * 32;
    static constexpr size_t kSmem =
        (size_t)kWarps * (kTblStride + kStateFloats) * sizeof(float) +
        (size_t)kWarps * 32 * sizeof(long long) + (size_t)kWarps * 32 * sizeof(float);
};

// Grid-wide hand-over between rounds: CTA 0, once every CTA's ticket is in,
// publishes the next round's state and then the generation number with a release store;
// the other CTAs wait for it with acquire loads.  Every CTA of the grid is
// resident (cooperative launch), and the wait is bounded all the same.
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t atom_add_acq_rel_u32(uint32_t *p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u32(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
constexpr uint32_t kSpinLimit = 1u << 22;     // polls, at most
constexpr unsigned long long kWaitLimitNs = 1000000000ull;   // and at most one second
constexpr int kMaxRounds = 16;
constexpr uint32_t kGenFinal = 0x10000u;       // fused path: every CTA out of the rounds
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Stage the control block in shared memory with coalesced 16-byte loads from
// L2 (other CTAs write it during the kernel; L1 is not coherent).
__device__ __forceinline__ void stage_ctrl(Ctrl &dst, const Ctrl *src) {
    const int4 *s4 = reinterpret_cast<const int4 *>(src);
    int4 *d4 = reinterpret_cast<int4 *>(&dst);
    for (int i = threadIdx.x; i < (int)(sizeof(Ctrl) / 16); i += blockDim.x) d4[i] = __ldcg(s4 + i);
}

// The search state back to global memory, 16 bytes per lane of one warp.
__device__ __forceinline__ void publish_search(Ctrl *ctrl, const SearchState &S, int L) {
    static_assert(sizeof(SearchState) % 16 == 0, "search state in 16-byte pieces");
    const int4 *src = reinterpret_cast<const int4 *>(&S);
    int4 *dst = reinterpret_cast<int4 *>(&ctrl->s);
    for (int i = L; i < (int)(sizeof(SearchState) / 16); i += 32) dst[i] = src[i];
}

// Thread 0 waits (bounded) until the release generation reaches `target`;
// false if it gave up.
__device__ __forceinline__ bool wait_gen(const Ctrl *ctrl, uint32_t target) {
    uint32_t spins = 0;
    const unsigned long long t0 = global_ns();
    const unsigned long long lim = ctrl->wait_ns;
    const uint32_t slim = ctrl->spin_limit;
    while (ld_acquire_u32(&ctrl->gen) < target) {
        if (++spins > slim || global_ns() - t0 > lim) return false;
        __nanosleep(64);
    }
    return true;
}

// Stage only the search state (the probes of a round, its final phase).
__device__ __forceinline__ void stage_search(SearchState &dst, const SearchState *src) {
    const int4 *s4 = reinterpret_cast<const int4 *>(src);
    int4 *d4 = reinterpret_cast<int4 *>(&dst);
    for (int i = threadIdx.x; i < (int)(sizeof(SearchState) / 16); i += blockDim.x) d4[i] = __ldcg(s4 + i);
}

// The emit of one block by one thread: the chain `mask` (slot bits) becomes
// the codebook (levels in slot order, padded with the largest), k, D_r (the
// chain's interval distortions added slot by slot, in order) and H_r =
// rate / d.  Table addresses depend on the mask alone, so every load issues
// at once.  Returns D_r.
__device__ __forceinline__ float emit_block(const float *__restrict__ tables, int64_t b,
                                            uint32_t mask, float rate, float *__restrict__ codebook,
                                            uint8_t *__restrict__ kout, float *__restrict__ Dr,
                                            float *__restrict__ Hr) {
    const float *tb = tables + b * kRecFloats + kRecTbl;
    float qv[17];
#pragma unroll
    for (int t = 0; t < 17; ++t) qv[t] = tb[kTblC + t];
    const int d = __float_as_int(tb[kTblHdr + 1]);
    mask &= 0x1ffffu;
    if (mask == 0u) mask = 1u;
    const int k = min(__popc(mask), 16);
    float dv = 0.f, top = qv[0];
    int prev = 0;
#pragma unroll
    for (int t = 0; t < 17; ++t) {
        const bool in = (mask >> t) & 1u;
        const bool link = in && t > 0;
        const float dd = tb[kTblD + (link ? dp_off(prev) + t - prev - 1 : 0)];
        if (link) dv += dd;
        const int pos = __popc(mask & ((1u << t) - 1u));
        if (in && pos < 16) codebook[b * 16 + pos] = qv[t];
        if (in) {
            top = qv[t];
            prev = t;
        }
    }
    for (int t = k; t < 16; ++t) codebook[b * 16 + t] = top;
    kout[b] = (uint8_t)k;
    Dr[b] = dv;
    Hr[b] = rate / (float)d;
    return dv;
}

// Work the fused path's queue (positions below `avail`) for one warp until
// the release generation reaches `target`: the warp's share is queue
// positions qj, qj + total_warps, ..., each block in 8 parts of 4 rows (qpart
// = the next part); per block the levels and tables are prepared once, each
// part's input is loaded before the previous part is computed, and the
// release is checked between parts.  Bounded in time like every wait.  Kept
// out of line so that its registers do not add to the DP's.
__device__ __noinline__ void run_queue(const Ctrl *ctrl, uint32_t target, uint64_t avail,
                                       const int32_t *__restrict__ fin,
                                       const uint32_t *__restrict__ mask_hi,
                                       const float *__restrict__ rate_hi,
                                       const float *__restrict__ tables, const QuantArgs &qa,
                                       float *__restrict__ codebook, uint8_t *__restrict__ kout,
                                       float *__restrict__ Dr, float *__restrict__ Hr,
                                       float *scratch, int lane, uint64_t total_warps,
                                       uint64_t &qj, int &qpart) {
    const unsigned long long t0 = global_ns();
    const unsigned long long lim = ctrl->wait_ns;
    bool prepared = false;
    int64_t b = 0;
    uint32_t T[16];
    uint4 raw[2];
    // the generation is polled with a relaxed load issued before each part and
    // read after it, so the poll's latency hides behind the part's work (the
    // caller's bounded wait then acquires)
    uint32_t gpoll = lane == 0 ? ld_relaxed_u32(&ctrl->gen) : 0u;
    for (;;) {
        const uint32_t gcur = __shfl_sync(0xffffffffu, gpoll, 0);
        if (gcur >= target) break;
        if (lane == 0) gpoll = ld_relaxed_u32(&ctrl->gen);
        if (qj >= avail) {
            if (global_ns() - t0 > lim) break;
            __nanosleep(100);
            continue;
        }
        if (!prepared) {
            b = __ldcg(&fin[qj]);
            const uint32_t mk = __ldcg(&mask_hi[b]);
            const float rt = __ldcg(&rate_hi[b]);
            fused_load(qa, b, qpart, lane, raw);
            fused_prepare(tables, b, mk, rt, qpart == 0, codebook, kout, Dr, Hr, scratch, lane, T);
            prepared = true;
        }
        uint4 nxt[2];
        if (qpart < 7) fused_load(qa, b, qpart + 1, lane, nxt);
        fused_codes(qa, b, qpart, lane, raw, T, scratch);
        raw[0] = nxt[0];
        raw[1] = nxt[1];
        if (++qpart == 8) {
            qpart = 0;
            qj += total_warps;
            prepared = false;
        }
    }
}

// The rest of one warp's queue share, then the blocks that no round
// finalized (their chain at the search's end), after every CTA has left the
// rounds.
__device__ __noinline__ void finish_blocks(const Ctrl *ctrl, int64_t nb, int xb_probe,
                                           int last_round, const int32_t *__restrict__ fin,
                                           const uint8_t *__restrict__ fflag,
                                           const int32_t *__restrict__ evr,
                                           const uint32_t *__restrict__ masks,
                                           const float *__restrict__ rates,
                                           const uint32_t *__restrict__ mask_hi,
                                           const float *__restrict__ rate_hi,
                                           const float *__restrict__ tables, const QuantArgs &qa,
                                           float *__restrict__ codebook, uint8_t *__restrict__ kout,
                                           float *__restrict__ Dr, float *__restrict__ Hr,
                                           float *scratch, int lane, uint64_t gw,
                                           uint64_t total_warps, uint64_t qj, int qpart) {
    const uint64_t fin_total = __ldcg(&ctrl->fin_tail);
    uint32_t T[16];
    uint4 raw[2], nxt[2];
    for (; qj < fin_total; qj += total_warps, qpart = 0) {
        const int64_t b = __ldcg(&fin[qj]);
        fused_load(qa, b, qpart, lane, raw);
        fused_prepare(tables, b, __ldcg(&mask_hi[b]), __ldcg(&rate_hi[b]), qpart == 0, codebook,
                      kout, Dr, Hr, scratch, lane, T);
        for (int part = qpart; part < 8; ++part) {
            if (part < 7) fused_load(qa, b, part + 1, lane, nxt);
            fused_codes(qa, b, part, lane, raw, T, scratch);
            raw[0] = nxt[0];
            raw[1] = nxt[1];
        }
    }
    for (int64_t b = (int64_t)gw; b < nb; b += (int64_t)total_warps) {
        if (__ldcg(&fflag[b])) continue;
        const bool from_last = xb_probe >= 0 && __ldcg(&evr[b]) == last_round;
        const uint32_t mk = from_last ? __ldcg(&masks[b * 32 + xb_probe]) : __ldcg(&mask_hi[b]);
        const float rt = from_last ? __ldcg(&rates[b * 32 + xb_probe]) : __ldcg(&rate_hi[b]);
        fused_load(qa, b, 0, lane, raw);
        fused_prepare(tables, b, mk, rt, true, codebook, kout, Dr, Hr, scratch, lane, T);
        for (int part = 0; part < 8; ++part) {
            if (part < 7) fused_load(qa, b, part + 1, lane, nxt);
            fused_codes(qa, b, part, lane, raw, T, scratch);
            raw[0] = nxt[0];
            raw[1] = nxt[1];
        }
    }
}

// The search kernel's copy of the control block in shared memory; at file
// scope so that the out-of-line control addresses it as shared memory.
__shared__ __align__(16) Ctrl s_ctrl;

// One round's control, run by one warp of CTA 0 once every CTA's ticket is
// in: fold the round's per-probe rate sums into the search state S, publish
// the window (first release), then walk and publish the next probes (second
// release).  Out of line so that one copy of its code serves two calls:
// `dry` runs the same instructions with a decreasing stand-in for the sums
// and writes nothing to global memory (only the staged state, which CTA 0
// stages again before its real control).  CTA 0 makes that call while the
// other CTAs evaluate each round, so the control's code is in the SM's
// instruction cache when the real control runs.  Fetched cold (from DRAM in
// the launch's first rounds, from L2 once a DP wave has evicted it) the
// control takes about twice as long.
__device__ __noinline__ void round_control(Ctrl *ctrl, bool walk, int iter, int round, bool dry) {
    const Ctrl &sC = s_ctrl;
    SearchState &S = s_ctrl.s;
    const int L = threadIdx.x & 31;
    __shared__ long long Rfx[32];
    __shared__ double sProbe[kSearchProbes];
    long long myR;
    if (!dry) {
        myR = (walk ? sC.Rxb_fx : 0) + (long long)sC.acc[L];
        ctrl->acc[L] = 0ull;
    } else {
        // R(v) = B vm / v (4 B at v = 0), vm the middle probe; the pilot's
        // sums cover its sample only
        const double v = search_probe(S, L), vm = search_probe(S, kSearchProbes / 2);
        const double r = (v > 0.0 && vm > 0.0) ? fmin(sC.budget * (vm / v), 4.0 * sC.budget)
                                                : 4.0 * sC.budget;
        const double part = S.phase == kSearchPilot
                                ? (double)(S.pilot_blocks > 0 ? S.pilot_blocks : 1) / (double)sC.nb
                                : 1.0;
        myR = llrint(r * part * kRateScale);
    }
    Rfx[L] = myR;
    const long long Bfx = sC.budget_fx;
    if (L == 0) S.hi0 = __longlong_as_double((long long)sC.hi0_bits);
    __syncwarp();
    SearchState st;              // every lane keeps the same copy
    bool walk_on = false;        // a walk follows the first publication
    if (sC.fixed) {
        if (L == 0) {
            S.xb_probe = 0;
            S.R_xb = myR;
            S.lambda = sC.lambda_fixed;
            S.phase = kSearchDone;
            S.rounds += 1;
        }
    } else if (S.phase == kSearchPilot) {
        // one lane per probe: the sample's rates scaled to all blocks, the
        // smallest feasible probe and the largest infeasible one below it
        // (first lane on ties, as a sequential scan)
        const double B = sC.budget;
        const double scale =
            (double)sC.nb / (double)(S.pilot_blocks > 0 ? S.pilot_blocks : 1) / kRateScale;
        const double v = search_probe(S, L), r = (double)myR * scale;
        const bool feas = r <= B;
        const uint64_t kv = okey(v);
        uint64_t kb = feas ? kv : ~0ull;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const uint64_t y = __shfl_xor_sync(0xffffffffu, kb, o);
            kb = y < kb ? y : kb;
        }
        const uint32_t mb = __ballot_sync(0xffffffffu, feas && kv == kb);
        const int ib = mb ? __ffs(mb) - 1 : -1;
        const bool cand = !feas && v > -1.0 && (ib < 0 || kv < kb);
        uint64_t ka = cand ? kv : 0ull;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const uint64_t y = __shfl_xor_sync(0xffffffffu, ka, o);
            ka = y > ka ? y : ka;
        }
        const uint32_t ma = __ballot_sync(0xffffffffu, cand && kv == ka);
        const int ia = ma ? __ffs(ma) - 1 : -1;
        const double vb = __shfl_sync(0xffffffffu, v, ib >= 0 ? ib : 0);
        const double Rb = __shfl_sync(0xffffffffu, r, ib >= 0 ? ib : 0);
        const double va = __shfl_sync(0xffffffffu, v, ia >= 0 ? ia : 0);
        const double Ra = __shfl_sync(0xffffffffu, r, ia >= 0 ? ia : 0);
        search_copy_scalars(st, S);        // every lane computes the same estimate
        const double est = search_pilot_finish(st, ib, ib >= 0 ? vb : INFINITY, ib >= 0 ? Rb : 0.0,
                                               ia, ia >= 0 ? va : -1.0, ia >= 0 ? Ra : 0.0, B);
        __syncwarp();
        if (st.have_grid && L > kSearchFirstDoublings) S.probe[L] = search_pilot_probe(est, L);
        __syncwarp();
        if (L == 0) search_copy_scalars(S, st);
    } else {
        // one lane per probe folds the evaluations into the window (exact
        // min / max of order keys), every lane walks, and lane L generates
        // the probes along decision path L
        const bool inr = L < S.nprobe;
        const double v = search_probe(S, L);
        const uint64_t kv = okey(v);
        const bool feas = inr && myR <= Bfx;
        uint64_t kb = feas ? kv : ~0ull;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const uint64_t y = __shfl_xor_sync(0xffffffffu, kb, o);
            kb = y < kb ? y : kb;
        }
        const uint32_t mb = __ballot_sync(0xffffffffu, feas && kv == kb);
        const int ib = mb ? __ffs(mb) - 1 : -1;
        const double vb = __shfl_sync(0xffffffffu, v, ib >= 0 ? ib : 0);
        const uint64_t kxb = okey(S.xb);
        const uint64_t kxbn = (ib >= 0 && kb < kxb) ? kb : kxb;
        const bool inf = inr && !feas && kv < kxbn;
        uint64_t ka = inf ? kv : 0ull;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const uint64_t y = __shfl_xor_sync(0xffffffffu, ka, o);
            ka = y > ka ? y : ka;
        }
        const uint32_t ma = __ballot_sync(0xffffffffu, inf && kv == ka);
        const int ia = ma ? __ffs(ma) - 1 : -1;
        const double va = __shfl_sync(0xffffffffu, v, ia >= 0 ? ia : 0);
        search_copy_scalars(st, S);
        search_window(st, ib >= 0 ? vb : INFINITY, ib, ib >= 0 ? Rfx[ib] : 0, va, ia);
        walk_on = search_decide(st, Rfx, Bfx);
        __syncwarp();
        if (L == 0) {
            search_copy_scalars(S, st);
            if (st.infeasible && !dry) ctrl->status = KVQ_ERR_INFEASIBLE;
        }
    }
    // first publication: the window and the next round's kind
    __syncwarp();
    if (!dry) {
        if (L == 0) {
            ctrl->phase1 = S.phase;
            if (!sC.fixed && S.xb_probe >= 0) ctrl->Rxb_fx = Rfx[S.xb_probe];
            ctrl->cnt[iter & 1] = 0u;      // consumed; the next round appends here
            ctrl->ticket = 0u;
            ctrl->fin_avail = sC.fin_tail;  // every queue append of this round is in
        }
        publish_search(ctrl, S, L);
        __syncwarp();            // the warp's writes, then one release store
        if (L == 0) st_release_u32(&ctrl->gen, 2u * (uint32_t)iter + 1u);
    }
    // second publication: the walk and the next round's probes
    if (walk_on) {
        const SearchWindow win = search_window_of(st);   // the walk keeps it
        const int go = search_walk_w(st, win);
        __syncwarp();
        if (go) {
            sProbe[L] = search_first_unknown(st);
            __syncwarp();
            search_path_w(st, win, L, sProbe);
            __syncwarp();
            S.probe[L] = sProbe[L];
        }
        __syncwarp();
        if (L == 0) search_copy_scalars(S, st);
        __syncwarp();
        if (!dry) publish_search(ctrl, S, L);
    }
    __syncwarp();
    if (L == 0 && !dry) {
        ctrl->t_ctl[min(round, 15)] = global_ns();
        st_release_u32(&ctrl->gen, 2u * (uint32_t)iter + 2u);
    }
}

// The whole search and the emit in one persistent, cooperative launch.
//
// Each round: the grid's warps take the round's blocks (all blocks in the
// bracket rounds, a sample in the pilot round, in the walk only the blocks
// evaluated in the previous round -- a block that was not is constant across
// the window and stays so).  Each lane accumulates, per probe, the change of
// its blocks' d_r H_r against their value at xb, in fixed point; CTA 0,
// once every CTA has taken its ticket, adds the sums to the total at xb and
// advances the search; the next round starts when it publishes the new state.
//
// Emit (after the last round), a thread per block: the chain at the final
// lambda becomes the codebook (levels in slot order), k, D_r (the chain's
// interval distortions added slot by slot) and H_r; each warp sums 32
// consecutive blocks' D_r in a fixed shuffle tree, and the last CTA adds the
// chunk sums in a fixed pattern.
template <bool GENERAL, bool QUANT>
__global__ void __launch_bounds__(RoundCfg<GENERAL>::kWarps * 32, 1)
search_kernel(const float *__restrict__ tables, int64_t nb, int s, Ctrl *__restrict__ ctrl,
              float *__restrict__ rates, uint32_t *__restrict__ masks,
              float *__restrict__ rate_lo, float *__restrict__ rate_hi,
              uint32_t *__restrict__ mask_hi, int32_t *__restrict__ evr,
              int32_t *__restrict__ list, double *__restrict__ epartial,
              float *__restrict__ codebook, uint8_t *__restrict__ kout, float *__restrict__ Dr,
              float *__restrict__ Hr, double *__restrict__ totals, double *__restrict__ lambda_out,
              int32_t *__restrict__ status, QuantArgs qa, int32_t *__restrict__ fin,
              uint8_t *__restrict__ fflag) {
    using Cfg = RoundCfg<GENERAL>;
    constexpr int W = Cfg::kWarps;
    extern __shared__ __align__(16) float smem[];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    float *sTbl = smem + w * kTblStride;
    float *sState = smem + W * kTblStride + w * Cfg::kStateFloats;
    long long *sSum = reinterpret_cast<long long *>(smem + W * (kTblStride + Cfg::kStateFloats));
    float *sDiag = reinterpret_cast<float *>(sSum + W * 32) + w * 32;
    Ctrl &sC = s_ctrl;
    __shared__ bool is_last, timed_out;
    __shared__ uint32_t sAct, sN;
    __shared__ int32_t sList[W * 32];
    __shared__ float sRb[W * 32];

    // A round's control publishes twice: first the window (which blocks can
    // still change, so the next round's phase A and table loads can start),
    // then the round's probes.  `ready`: this CTA holds the current probes.
    bool ready = true;                   // round 0's come from ctrl_init
    if (threadIdx.x == 0) timed_out = false;
    // fused path: this warp's share of the queue of final blocks (queue
    // positions qj, qj + total_warps, ...), each in 8 parts of 4 rows; the
    // warp checks for a release between parts
    const uint64_t total_warps = (uint64_t)gridDim.x * W;
    uint64_t qj = (uint64_t)blockIdx.x * W + w;
    int qpart = 0;
    float *scratch = sState;             // free whenever the warp is not in a DP
    if constexpr (QUANT) {
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nb;
             i += (int64_t)gridDim.x * blockDim.x)
            fflag[i] = 0;
    }

    if (blockIdx.x == 0 && threadIdx.x == 0) ctrl->t_start = global_ns();
    // CTA 0 takes no items in the search's rounds (round_control): item it
    // goes to CTA 1 + it mod (grid - 1)
    const bool warm = !ctrl->fixed && gridDim.x > 1;
    const int64_t cta = warm ? (int64_t)blockIdx.x - 1 : (int64_t)blockIdx.x;
    const int64_t ncta = warm ? (int64_t)gridDim.x - 1 : (int64_t)gridDim.x;
    for (int iter = 0; iter < kMaxRounds; ++iter) {
        // the candidate lists alternate by round; this thread's first item of
        // a walk round is fetched while the control block is staged
        const int32_t *lin = list + (size_t)(iter & 1) * nb;
        int32_t *lout = list + (size_t)((iter + 1) & 1) * nb;
        const int64_t it0 = cta + ncta * (int64_t)threadIdx.x;
        const int32_t b0 = (iter > 0 && cta >= 0 && it0 < nb) ? __ldcg(&lin[it0]) : 0;
        stage_ctrl(sC, ctrl);
        if (threadIdx.x == 0) sAct = 0u;
        __syncthreads();
        // The other CTAs have acquired only the control's first publication:
        // its second may be landing while they stage, so they take the round
        // kind from phase1 (a walk that ends reaches them as the second
        // publication, below).  CTA 0 reads the state it wrote itself.
        const int phase = blockIdx.x == 0 ? sC.s.phase : sC.phase1;
        if (phase == kSearchDone) break;
        const int fixed = sC.fixed;
        const int xa_probe = sC.s.xa_probe, xb_probe = sC.s.xb_probe;
        const int round = sC.s.rounds;
        const bool walk = !fixed && phase == kSearchWalk;
        const bool pilot = !fixed && phase == kSearchPilot;
        const int stride = sC.s.pilot_stride;
        const int64_t nitems = walk ? (int64_t)sC.cnt[iter & 1]
                                    : pilot ? (int64_t)sC.s.pilot_blocks : nb;
        float lam = ready ? (float)(fixed ? sC.lambda_fixed : search_probe(sC.s, lane)) : 0.f;
        long long my_sum = 0;
        bool done = false;
        // Items in chunks of one per thread: item it = cta + ncta * (c *
        // blockDim.x + threadIdx.x), so consecutive CTAs take consecutive
        // items.  Phase A (a thread per item) carries the walk's per-block
        // state to the new window ends and keeps the blocks whose rate can
        // still change; phase B (a warp per kept block) runs the DP.
        for (int64_t c0 = 0; cta >= 0 && cta + ncta * c0 < nitems; c0 += blockDim.x) {
            if (threadIdx.x == 0) sN = 0u;
            __syncthreads();
            const int64_t it = cta + ncta * (c0 + threadIdx.x);
            bool act = false;
            int32_t bsel = 0;
            if (it < nitems) {
                act = true;
                if (walk) {
                    // evaluated in the previous round: its rates at the new
                    // window ends; the rate is non-increasing in lambda, so
                    // equal rates at both ends mean the chain is constant
                    // inside the window
                    const int32_t b = c0 == 0 ? b0 : __ldcg(&lin[it]);
                    float ra = __ldcg(&rate_lo[b]), rb = __ldcg(&rate_hi[b]);
                    if (xa_probe >= 0) ra = __ldcg(&rates[(int64_t)b * 32 + xa_probe]);
                    if (xb_probe >= 0) {
                        rb = __ldcg(&rates[(int64_t)b * 32 + xb_probe]);
                        mask_hi[b] = __ldcg(&masks[(int64_t)b * 32 + xb_probe]);
                    }
                    rate_lo[b] = ra;
                    rate_hi[b] = rb;
                    act = ra != rb;
                    bsel = b;
                    if (act) {
                        const uint32_t slot = atomicAdd(&sN, 1u);
                        sList[slot] = b;
                        sRb[slot] = rb;
                    }
                } else {
                    bsel = (int32_t)(pilot ? it * stride : it);
                    const uint32_t slot = atomicAdd(&sN, 1u);
                    sList[slot] = bsel;
                    sRb[slot] = 0.f;
                }
                if (act) evr[bsel] = round;
            }
            if constexpr (QUANT) {
                // a candidate whose rate is equal at both ends is final:
                // queue it for the idle warps
                const bool fin_now = walk && it < nitems && !act;
                const uint32_t fm = __ballot_sync(0xffffffffu, fin_now);
                if (fm) {
                    uint32_t fb = 0;
                    if (lane == 0) fb = atomicAdd(&ctrl->fin_tail, (uint32_t)__popc(fm));
                    fb = __shfl_sync(0xffffffffu, fb, 0);
                    if (fin_now) {
                        fin[fb + __popc(fm & ((1u << lane) - 1u))] = bsel;
                        fflag[bsel] = 1;
                    }
                }
            }
            // room in the next round's list: one atomic per warp; the entries
            // are written after the DP, so its latency is hidden
            uint32_t lbase = 0, lrank = 0;
            if (!pilot) {
                const uint32_t am = __ballot_sync(0xffffffffu, act);
                lrank = __popc(am & ((1u << lane) - 1u));
                if (lane == 0 && am)
                    lbase = atomicAdd(&ctrl->cnt[(iter + 1) & 1], (uint32_t)__popc(am));
                lbase = __shfl_sync(0xffffffffu, lbase, 0);
            }
            __syncthreads();
            const bool prefetched = !ready;
            if (!ready) {
                // phase A ran on the published window: load each warp's first
                // table while the control finishes the round's probes
                if (w < (int)sN) load_tables(sTbl, tables, (int64_t)sList[w], lane);
                if constexpr (QUANT)
                    run_queue(ctrl, 2u * (uint32_t)iter, (uint64_t)sC.fin_avail, fin, mask_hi, rate_hi,
                              tables, qa, codebook, kout, Dr, Hr, scratch, lane, total_warps, qj,
                              qpart);
                if (threadIdx.x == 0 && !wait_gen(ctrl, 2u * (uint32_t)iter)) timed_out = true;
                __syncthreads();
                if (timed_out) break;
                stage_search(sC.s, &ctrl->s);
                __syncthreads();
                ready = true;
                if (sC.s.phase == kSearchDone) {   // the walk ended: nothing to evaluate
                    done = true;
                    break;
                }
                lam = (float)(fixed ? sC.lambda_fixed : search_probe(sC.s, lane));
            }
            const uint32_t n = sN;
            for (uint32_t q = w; q < n; q += W) {
                const int64_t b = sList[q];
                const float rb = sRb[q];
                if (!(prefetched && q == (uint32_t)w)) load_tables(sTbl, tables, b, lane);
                __syncwarp();
                const int mp = min(max(__float_as_int(sTbl[kTblHdr]), 1), kCand);
                float rate;
                uint32_t mask;
                if (mp <= 1) {
                    rate = 0.f;
                    mask = 1u;
                } else {
                    const int C = mp > s ? mp - s : 0;
                    if (!GENERAL || C == 0 || (C == 1 && mp == 17)) {
                        dp_a_diag(sTbl, sDiag, lane);
                        dp_path_a(sTbl, lam, C, sState, sState + kPairs * 32, sDiag, lane, rate, mask);
                    } else {
                        dp_path_b(sTbl, lam, s, sState, sState + kPairs * 32,
                                  reinterpret_cast<uint32_t *>(sState + 2 * kPairs * 32), lane, rate,
                                  mask);
                    }
                }
                rates[b * 32 + lane] = rate;
                masks[b * 32 + lane] = mask;
                my_sum += llrint((double)rate * kRateScale) - llrint((double)rb * kRateScale);
                __syncwarp();
            }
            if (!pilot && act) lout[lbase + lrank] = bsel;
            if (threadIdx.x == 0) sAct += n;
            __syncthreads();
        }
        if (!ready && !timed_out) {
            // no items here: still wait for the probes, so that the previous
            // control has finished before this CTA can take the ticket
            if constexpr (QUANT)
                    run_queue(ctrl, 2u * (uint32_t)iter, (uint64_t)sC.fin_avail, fin, mask_hi, rate_hi,
                              tables, qa, codebook, kout, Dr, Hr, scratch, lane, total_warps, qj,
                              qpart);
            if (threadIdx.x == 0 && !wait_gen(ctrl, 2u * (uint32_t)iter)) timed_out = true;
            __syncthreads();
            if (!timed_out) {
                stage_search(sC.s, &ctrl->s);
                __syncthreads();
                ready = true;
                done = sC.s.phase == kSearchDone;
            }
        }
        if (timed_out) {
            if (threadIdx.x == 0) {
                atomicExch(&ctrl->err, 1u);
                *status = KVQ_ERR_TIMEOUT;
            }
            return;
        }
        if (done) break;
        // (the dry control changes only the staged search state, which CTA 0
        // reads again before its real control)
        if (warm && blockIdx.x == 0 && w == 0) round_control(ctrl, false, iter, round, true);
        sSum[w * 32 + lane] = my_sum;
        __syncthreads();
        if (threadIdx.x < 32) {
            long long sum = 0;
            for (int k = 0; k < W; ++k) sum += sSum[k * 32 + threadIdx.x];
            if (sum) atomicAdd(&ctrl->acc[threadIdx.x], (unsigned long long)sum);   // no return: a reduction
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            if (sAct) atomicAdd(&ctrl->active[min(round, 15)], sAct);
            // acquire-release ticket: orders this CTA's sums (made before the
            // barrier) before it, and the last CTA sees every CTA's sums
            const unsigned t = atom_add_acq_rel_u32(&ctrl->ticket, 1u);
            timed_out = false;
            // CTA 0 runs every round's control, once every CTA's ticket is in
            // (spinning, bounded): the control code then stays in the
            // instruction cache of one SM instead of being fetched cold by
            // whichever CTA happens to finish last
            is_last = blockIdx.x == 0;
            if (is_last && t != gridDim.x - 1) {
                uint32_t spins = 0;
                const unsigned long long t0 = global_ns();
                while (ld_acquire_u32(&ctrl->ticket) < gridDim.x) {
                    if (++spins > ctrl->spin_limit || global_ns() - t0 > ctrl->wait_ns) {
                        timed_out = true;
                        break;
                    }
                }
            }
        }
        __syncthreads();
        if (timed_out) {
            if (threadIdx.x == 0) {
                atomicExch(&ctrl->err, 1u);
                *status = KVQ_ERR_TIMEOUT;
            }
            return;
        }
        if (is_last) {
            // ---- CTA 0: stage the control block again (the sums are
            // final now), advance the search in shared memory, write back
            // what changed, then release the other CTAs
            if (threadIdx.x == 0) ctrl->t_dp[min(round, 15)] = global_ns();
            stage_ctrl(sC, ctrl);
            __syncthreads();
            if (threadIdx.x < 32) round_control(ctrl, walk, iter, round, false);
            __syncthreads();
            ready = true;
        } else {
            // the next round starts on the first publication
            if constexpr (QUANT)
                run_queue(ctrl, 2u * (uint32_t)iter + 1u, (uint64_t)sC.fin_avail, fin, mask_hi,
                          rate_hi, tables, qa, codebook, kout, Dr, Hr, scratch, lane, total_warps,
                          qj, qpart);
            if (threadIdx.x == 0 && !wait_gen(ctrl, 2u * (uint32_t)iter + 1u)) timed_out = true;
            __syncthreads();
            ready = false;
            if (timed_out) {
                if (threadIdx.x == 0) {
                    atomicExch(&ctrl->err, 1u);
                    *status = KVQ_ERR_TIMEOUT;
                }
                return;
            }
        }
    }

    // ---- after the last round (sC holds the final state)
    const int xb_probe = sC.s.xb_probe;
    const int last_round = sC.s.rounds - 1;
    if constexpr (QUANT) {
        // every CTA out of the rounds (the queue is complete), then: the rest
        // of this warp's queue units, and the blocks the last rounds settled
        __syncthreads();
        if (threadIdx.x == 0) {
            const unsigned t = atom_add_acq_rel_u32(&ctrl->ticket_f, 1u);
            if (t == gridDim.x - 1) st_release_u32(&ctrl->gen, kGenFinal);
            else if (!wait_gen(ctrl, kGenFinal)) timed_out = true;
        }
        __syncthreads();
        if (timed_out) {
            if (threadIdx.x == 0) {
                atomicExch(&ctrl->err, 1u);
                *status = KVQ_ERR_TIMEOUT;
            }
            return;
        }
        finish_blocks(ctrl, nb, xb_probe, last_round, fin, fflag, evr, masks, rates, mask_hi, rate_hi,
                      tables, qa, codebook, kout, Dr, Hr, scratch, lane,
                      (uint64_t)blockIdx.x * W + w, total_warps, qj, qpart);
    } else {
        // emit: a thread per block, so every block's loads are in flight at
        // once; a warp takes 32 consecutive blocks (chunk g), the chunks dealt
        // round-robin over the CTAs so that every SM takes part; the warp then
        // sums its blocks' D_r in a fixed shuffle tree (the chunk sum)
        const int64_t nch = (nb + 31) / 32;
        for (int64_t g = (int64_t)blockIdx.x + (int64_t)gridDim.x * w; g < nch;
             g += (int64_t)gridDim.x * W) {
            const int64_t b = g * 32 + lane;
            float dv = 0.f;
            if (b < nb) {
                const int32_t ev = __ldcg(&evr[b]);
                const int xp = xb_probe >= 0 ? xb_probe : 0;
                const uint32_t m_last = __ldcg(&masks[b * 32 + xp]);
                const float r_last = __ldcg(&rates[b * 32 + xp]);
                const uint32_t m_hi = __ldcg(&mask_hi[b]);
                const float r_hi = __ldcg(&rate_hi[b]);
                const bool from_last = xb_probe >= 0 && ev == last_round;
                dv = emit_block(tables, b, from_last ? m_last : m_hi, from_last ? r_last : r_hi,
                                codebook, kout, Dr, Hr);
            }
            double t = (double)dv;          // lanes past the last block add 0
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) t += __shfl_down_sync(0xffffffffu, t, o);
            if (lane == 0) epartial[g] = t;
        }
    }
    // ---- totals, by the last CTA to finish: D = the chunk sums (32
    // consecutive blocks each, a fixed shuffle tree) added in a fixed pattern
    // (thread t sums chunks t, t + blockDim.x, .. in order; then the threads'
    // sums in a fixed tree)
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned t = atom_add_acq_rel_u32(&ctrl->ticket_emit, 1u);   // orders this CTA's D_r
        is_last = (t == gridDim.x - 1);
    }
    __syncthreads();
    if (!is_last) return;
    const int64_t nch = (nb + 31) / 32;
    if constexpr (QUANT) {
        // the fused path wrote D_r block by block: the chunk sums from them,
        // in the same tree (8 chunks per warp at a time, loads first)
        for (int64_t g0 = (int64_t)w * 8; g0 < nch; g0 += (int64_t)W * 8) {
            double v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int64_t b = (g0 + u) * 32 + lane;
                v[u] = (g0 + u < nch && b < nb) ? (double)__ldcg(&Dr[b]) : 0.0;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
                for (int u = 0; u < 8; ++u) v[u] += __shfl_down_sync(0xffffffffu, v[u], o);
            }
            if (lane == 0) {
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (g0 + u < nch) epartial[g0 + u] = v[u];
            }
        }
        __syncthreads();
    }
    __shared__ double sPart[W * 32];
    {
        // thread t adds the chunk sums t, t + blockDim.x, .. in order
        double a = 0.0;
#pragma unroll 4
        for (int64_t i = threadIdx.x; i < nch; i += blockDim.x) a += __ldcg(&epartial[i]);
        sPart[threadIdx.x] = a;
    }
    __syncthreads();
    if (threadIdx.x >= 32) return;
    // fixed tree: lane l adds its column, then a shuffle tree
    double dd = 0.0;
#pragma unroll
    for (int k = 0; k < W; ++k) dd += sPart[k * 32 + threadIdx.x];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dd += __shfl_down_sync(0xffffffffu, dd, o);
    if (threadIdx.x != 0) return;
    const Ctrl *n = &sC;
    const double R = (double)n->s.R_xb / kRateScale;   // the rate the search tested
    const double lam = n->s.lambda;
    totals[0] = R;
    totals[1] = dd;
    totals[2] = lam;
    if (n->mode == KVQ_SUBGRADIENT) {
        const double nl = lam + n->eta * (R - n->budget);
        *lambda_out = nl > 0.0 ? nl : 0.0;
    } else {
        *lambda_out = lam;
    }
    int st = n->status;
    if (n->flags & kFlagNonfinite) st = KVQ_ERR_NONFINITE;
    if (n->flags & kFlagBadWeight) st = KVQ_ERR_BAD_WEIGHT;
    if (__ldcg(&ctrl->err)) st = KVQ_ERR_TIMEOUT;
    *status = st;
    ctrl->ticket_emit = 0u;
    ctrl->ticket_f = 0u;
    ctrl->t_end = global_ns();
}

// ------------------------------------------------ fixed-rate comparator
// Every block on its own lambda_r ("Implementation notes": the comparison
// against fixed-rate entropy coding at equal total cache bytes): one warp per
// block runs the 40-step bisection above on that block alone, budget
// bits_per_entry * d_r, with the same exact DP (one lane per probe lambda)
// and the same search control (kvq_search.h) walking 5 levels per round;
// then the chain at the smallest feasible lambda evaluated is emitted.
template <bool GENERAL>
__global__ void __launch_bounds__(RoundCfg<GENERAL>::kWarps * 32)
fixed_rate_kernel(const float *__restrict__ tables, int64_t nb, int s, double bits_per_entry,
                  float *__restrict__ codebook, uint8_t *__restrict__ kout, float *__restrict__ Dr,
                  float *__restrict__ Hr, double *__restrict__ lambdas,
                  int32_t *__restrict__ status) {
    using Cfg = RoundCfg<GENERAL>;
    constexpr int W = Cfg::kWarps;
    extern __shared__ __align__(16) float smem[];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    float *sTbl = smem + w * kTblStride;
    float *sState = smem + W * kTblStride + w * Cfg::kStateFloats;
    float *sDiag = smem + W * (kTblStride + Cfg::kStateFloats) + w * 32;
    __shared__ __align__(16) SearchState sS[W];
    __shared__ long long sR[W][32];
    __shared__ double sProbe[W][32];
    const int64_t b = (int64_t)blockIdx.x * W + w;
    if (b >= nb) return;                      // warp-level work only below
    load_tables(sTbl, tables, b, lane);
    __syncwarp();
    const int mp = min(max(__float_as_int(sTbl[kTblHdr]), 1), kCand);
    const int d = __float_as_int(sTbl[kTblHdr + 1]);
    const int bflags = __float_as_int(sTbl[kTblHdr + 2]);
    SearchState &S = sS[w];
    if (lane == 0) {
        search_init(S);
        const double wd = (double)sTbl[kTblC + 16] - (double)sTbl[kTblC];
        S.hi0 = wd * wd;
        S.f32_lambda = 1;                     // the DP runs at float(lambda)
    }
    __syncwarp();
    const long long Bfx = budget_fx(bits_per_entry * (double)d);
    uint32_t xb_mask = 1u;
    float xb_rate = 0.f;
    if (mp > 1) {
        const int C = mp > s ? mp - s : 0;
        for (int round = 0; round < kMaxRounds && S.phase != kSearchDone; ++round) {
            const double v = search_probe(S, lane);
            const float lam = (float)v;
            float rate;
            uint32_t mask;
            if (!GENERAL || C == 0 || (C == 1 && mp == 17)) {
                dp_a_diag(sTbl, sDiag, lane);
                dp_path_a(sTbl, lam, C, sState, sState + kPairs * 32, sDiag, lane, rate, mask);
            } else {
                dp_path_b(sTbl, lam, s, sState, sState + kPairs * 32,
                          reinterpret_cast<uint32_t *>(sState + 2 * kPairs * 32), lane, rate, mask);
            }
            const long long R = llrint((double)rate * kRateScale);
            sR[w][lane] = R;
            __syncwarp();
            // the round's evaluations into the window: smallest feasible probe,
            // largest infeasible one below it (order keys; first lane on ties)
            const bool inr = lane < S.nprobe;
            const uint64_t kv = okey(v);
            const bool feas = inr && R <= Bfx;
            uint64_t kb = feas ? kv : ~0ull;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const uint64_t y = __shfl_xor_sync(0xffffffffu, kb, o);
                kb = y < kb ? y : kb;
            }
            const uint32_t mb = __ballot_sync(0xffffffffu, feas && kv == kb);
            const int ib = mb ? __ffs(mb) - 1 : -1;
            const double vb = __shfl_sync(0xffffffffu, v, ib >= 0 ? ib : 0);
            const uint64_t kxb = okey(S.xb);
            const uint64_t kxbn = (ib >= 0 && kb < kxb) ? kb : kxb;
            const bool inf = inr && !feas && kv < kxbn;
            uint64_t ka = inf ? kv : 0ull;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const uint64_t y = __shfl_xor_sync(0xffffffffu, ka, o);
                ka = y > ka ? y : ka;
            }
            const uint32_t ma = __ballot_sync(0xffffffffu, inf && kv == ka);
            const int ia = ma ? __ffs(ma) - 1 : -1;
            const double va = __shfl_sync(0xffffffffu, v, ia >= 0 ? ia : 0);
            SearchState st;                    // every lane the same copy
            search_copy_scalars(st, S);
            search_window(st, ib >= 0 ? vb : INFINITY, ib, ib >= 0 ? sR[w][ib] : 0, va, ia);
            const int walk_on = search_decide(st, sR[w], Bfx);
            const int xp = st.xb_probe;        // lane-uniform
            const uint32_t mk = __shfl_sync(0xffffffffu, mask, xp >= 0 ? xp : 0);
            const float rk = __shfl_sync(0xffffffffu, rate, xp >= 0 ? xp : 0);
            if (xp >= 0) {
                xb_mask = mk;
                xb_rate = rk;
            }
            if (walk_on) {
                const SearchWindow win = search_window_of(st);
                const int go = search_walk_w(st, win);
                __syncwarp();
                if (go) {
                    sProbe[w][lane] = search_first_unknown(st);
                    __syncwarp();
                    search_path_w(st, win, lane, sProbe[w]);
                    __syncwarp();
                    S.probe[lane] = sProbe[w][lane];
                }
            }
            __syncwarp();
            if (lane == 0) search_copy_scalars(S, st);
            __syncwarp();
        }
    }
    // emit (lane 0): levels in slot order, D_r along the chain, H_r
    if (lane == 0) {
        uint32_t mask = xb_mask & 0x1ffffu;
        if (mp <= 1 || mask == 0u) mask = 1u;
        const int k = min(__popc(mask), 16);
        float dv = 0.f, top = sTbl[kTblC];
        int prev = 0, pos = 0;
        for (int t = 0; t < 17; ++t) {
            if (!((mask >> t) & 1u)) continue;
            if (t > 0) dv += sTbl[kTblD + dp_off(prev) + t - prev - 1];
            top = sTbl[kTblC + t];
            if (pos < 16) codebook[b * 16 + pos] = top;
            ++pos;
            prev = t;
        }
        for (int t = k; t < 16; ++t) codebook[b * 16 + t] = top;
        kout[b] = (uint8_t)k;
        Dr[b] = dv;
        Hr[b] = mp > 1 ? xb_rate / (float)d : 0.f;
        lambdas[b] = mp > 1 ? S.lambda : 0.0;
        if (S.infeasible) atomicMax(status, (int32_t)KVQ_ERR_INFEASIBLE);
        if (bflags & kFlagWeighted) atomicMax(status, (int32_t)KVQ_ERR_INVALID_ARG + 100);
    }
}

// --------------------------------------------------- per-probe rate sums
// Sum over the layout's blocks of d_r H_r at up to 32 lambdas (one lane per
// lambda, the exact DP at float(lambda)), in fixed point (2^-20 bit units,
// each block's rate rounded once): the quantity one evaluation of the global
// lambda search needs.  Integer sums are exact and do not depend on the order
// of the adds, so the sums of blocks split across devices add up to the sum
// over all of them bit for bit.
template <bool GENERAL>
__global__ void __launch_bounds__(RoundCfg<GENERAL>::kWarps * 32)
rate_sums_kernel(const float *__restrict__ tables, int64_t nb, int s, ProbeSet probes,
                 unsigned long long *__restrict__ sums) {
    using Cfg = RoundCfg<GENERAL>;
    constexpr int W = Cfg::kWarps;
    extern __shared__ __align__(16) float smem[];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    float *sTbl = smem + w * kTblStride;
    float *sState = smem + W * kTblStride + w * Cfg::kStateFloats;
    float *sDiag = smem + W * (kTblStride + Cfg::kStateFloats) + w * 32;
    __shared__ long long sSum[W][32];
    const float lam = lane < probes.n ? (float)probes.lambda[lane] : 0.f;
    long long acc = 0;
    for (int64_t b = (int64_t)blockIdx.x * W + w; b < nb; b += (int64_t)gridDim.x * W) {
        load_tables(sTbl, tables, b, lane);
        __syncwarp();
        const int mp = min(max(__float_as_int(sTbl[kTblHdr]), 1), kCand);
        float rate = 0.f;
        uint32_t mask = 1u;
        if (mp > 1) {
            const int C = mp > s ? mp - s : 0;
            if (!GENERAL || C == 0 || (C == 1 && mp == 17)) {
                dp_a_diag(sTbl, sDiag, lane);
                dp_path_a(sTbl, lam, C, sState, sState + kPairs * 32, sDiag, lane, rate, mask);
            } else {
                dp_path_b(sTbl, lam, s, sState, sState + kPairs * 32,
                          reinterpret_cast<uint32_t *>(sState + 2 * kPairs * 32), lane, rate, mask);
            }
        }
        acc += llrint((double)rate * kRateScale);
        __syncwarp();
    }
    sSum[w][lane] = acc;
    __syncthreads();
    if (threadIdx.x < 32) {
        long long t = 0;
        for (int k = 0; k < W; ++k) t += sSum[k][threadIdx.x];
        if (t && threadIdx.x < probes.n) atomicAdd(&sums[threadIdx.x], (unsigned long long)t);
    }
}

// Totals of the fixed-rate comparator in a fixed order: each thread a
// contiguous run of blocks, then a fixed tree; the status of the data.
__global__ void fixed_rate_totals_kernel(const StatsHeader *__restrict__ hdr, int64_t nb, int d,
                                         const float *__restrict__ Dr,
                                         const float *__restrict__ Hr, double *__restrict__ totals,
                                         int32_t *__restrict__ status) {
    __shared__ double sR[256], sD[256];
    const int t = threadIdx.x;
    const int64_t chunk = (nb + 255) / 256;
    double r = 0.0, dd = 0.0;
    for (int64_t i = (int64_t)t * chunk; i < nb && i < (int64_t)(t + 1) * chunk; ++i) {
        r += (double)Hr[i] * (double)d;
        dd += (double)Dr[i];
    }
    sR[t] = r;
    sD[t] = dd;
    __syncthreads();
    for (int o = 128; o > 0; o >>= 1) {
        if (t < o) {
            sR[t] += sR[t + o];
            sD[t] += sD[t + o];
        }
        __syncthreads();
    }
    if (t == 0) {
        totals[0] = sR[0];
        totals[1] = sD[0];
        totals[2] = 0.0;
        int st = *status;
        if (st == KVQ_ERR_INVALID_ARG + 100) st = KVQ_ERR_INVALID_ARG;   // weighted stats
        if (hdr->flags & kFlagNonfinite) st = KVQ_ERR_NONFINITE;
        *status = st;
    }
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
                    float *Dr, float *Hr, double *totals, int32_t *status, cudaStream_t st,
                    const uint16_t *x, uint64_t seed, uint64_t index_base, uint8_t *codes) {
    const int64_t nb = num_blocks(L);
    if (nb == 0) {
        empty_alloc_kernel<<<1, 32, 0, st>>>(totals, lambda, status, mode, eta, budget);
        return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
    }
    Workspace ws = carve(workspace, nb);
    const StatsHeader *hdr = static_cast<const StatsHeader *>(stats);
    const float *recs = reinterpret_cast<const float *>(static_cast<const char *>(stats) +
                                                        sizeof(StatsHeader));
    unsigned long long wait_ns = kWaitLimitNs;
    uint32_t spin_limit = kSpinLimit;
    if (test_wait_limit(&wait_ns)) spin_limit = 1u;
    ctrl_init_kernel<<<1, 32, 0, st>>>(ws.ctrl, hdr, budget, eta, mode, lambda, nb, wait_ns,
                                       spin_limit);
    if (cudaGetLastError() != cudaSuccess) return KVQ_ERR_CUDA;
    const bool general = s < 16;
    const bool quant = codes != nullptr;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
    const int resident = g_resident[dev][general ? 1 : 0][quant ? 1 : 0];
    const int W = general ? RoundCfg<true>::kWarps : RoundCfg<false>::kWarps;
    const int64_t need = (nb + W - 1) / W;
    int64_t grid = need < resident ? need : resident;
    if (grid > kMaxGrid) grid = kMaxGrid;
    if (grid < 1) return KVQ_ERR_CUDA;
    QuantArgs qa = {};
    if (quant) {
        qa.x = x;
        qa.codes = codes;
        qa.key = philox_key(seed);
        qa.index_base = index_base;
        qa.D = L.D;
        qa.G = L.group;
        while ((1 << qa.lg_ng) < L.D / L.group) ++qa.lg_ng;
        while ((1 << qa.lg_upr) < L.group / 8) ++qa.lg_upr;
    }
    void *args[] = {(void *)&recs, (void *)&nb, (void *)&s, (void *)&ws.ctrl, (void *)&ws.rates,
                    (void *)&ws.masks, (void *)&ws.rate_lo, (void *)&ws.rate_hi,
                    (void *)&ws.mask_hi, (void *)&ws.evr, (void *)&ws.list, (void *)&ws.epartial,
                    (void *)&codebook, (void *)&k, (void *)&Dr, (void *)&Hr, (void *)&totals,
                    (void *)&lambda, (void *)&status, (void *)&qa, (void *)&ws.fin,
                    (void *)&ws.fflag};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)(W * 32));
    cfg.dynamicSmemBytes = general ? RoundCfg<true>::kSmem : RoundCfg<false>::kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;       // every CTA resident: the rounds hand over
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const void *fn = general ? (quant ? (const void *)search_kernel<true, true>
                                      : (const void *)search_kernel<true, false>)
                             : (quant ? (const void *)search_kernel<false, true>
                                      : (const void *)search_kernel<false, false>);
    if (cudaLaunchKernelExC(&cfg, fn, args) != cudaSuccess) return KVQ_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

int launch_fixed_rate(const void *stats, const kvq_layout &L, int s, double bits_per_entry,
                      float *codebook, uint8_t *k, float *Dr, float *Hr, double *lambdas,
                      double *totals, int32_t *status, cudaStream_t st) {
    const int64_t nb = num_blocks(L);
    if (cudaMemsetAsync(status, 0, sizeof(int32_t), st) != cudaSuccess) return KVQ_ERR_CUDA;
    const StatsHeader *hdr = static_cast<const StatsHeader *>(stats);
    if (nb > 0) {
        const float *recs = reinterpret_cast<const float *>(static_cast<const char *>(stats) +
                                                            sizeof(StatsHeader));
        const bool general = s < 16;
        const int W = general ? RoundCfg<true>::kWarps : RoundCfg<false>::kWarps;
        const unsigned grid = (unsigned)((nb + W - 1) / W);
        const size_t smem = general ? RoundCfg<true>::kSmem : RoundCfg<false>::kSmem;
        if (general)
            fixed_rate_kernel<true><<<grid, W * 32, smem, st>>>(recs, nb, s, bits_per_entry,
                                                                 codebook, k, Dr, Hr, lambdas,
                                                                 status);
        else
            fixed_rate_kernel<false><<<grid, W * 32, smem, st>>>(recs, nb, s, bits_per_entry,
                                                                  codebook, k, Dr, Hr, lambdas,
                                                                  status);
        if (cudaGetLastError() != cudaSuccess) return KVQ_ERR_CUDA;
    }
    fixed_rate_totals_kernel<<<1, 256, 0, st>>>(hdr, nb, 32 * L.group, Dr, Hr, totals, status);
    return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

int launch_rate_sums(const void *stats, const kvq_layout &L, int s, const double *lambdas,
                     int nprobe, unsigned long long *sums, cudaStream_t st) {
    if (cudaMemsetAsync(sums, 0, kSearchProbes * sizeof(unsigned long long), st) != cudaSuccess)
        return KVQ_ERR_CUDA;
    const int64_t nb = num_blocks(L);
    if (nb == 0 || nprobe == 0) return KVQ_OK;
    ProbeSet ps = {};
    for (int p = 0; p < nprobe; ++p) ps.lambda[p] = lambdas[p];
    ps.n = nprobe;
    const float *recs = reinterpret_cast<const float *>(static_cast<const char *>(stats) +
                                                        sizeof(StatsHeader));
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVQ_ERR_CUDA;
    const bool general = s < 16;
    const int W = general ? RoundCfg<true>::kWarps : RoundCfg<false>::kWarps;
    int64_t grid = (nb + W - 1) / W;
    const int64_t cap = 8 * (int64_t)g_resident[dev][general ? 1 : 0][0];
    if (cap > 0 && grid > cap) grid = cap;
    const size_t smem = general ? RoundCfg<true>::kSmem : RoundCfg<false>::kSmem;
    if (general)
        rate_sums_kernel<true><<<(unsigned)grid, W * 32, smem, st>>>(recs, nb, s, ps, sums);
    else
        rate_sums_kernel<false><<<(unsigned)grid, W * 32, smem, st>>>(recs, nb, s, ps, sums);
    return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

int stats_hi0(const void *stats, double *hi0) {
    StatsHeader h;
    if (cudaMemcpy(&h, stats, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return KVQ_ERR_CUDA;
    uint64_t b = h.hi0_bits;
    memcpy(hi0, &b, 8);
    return (h.flags & kFlagNonfinite) ? KVQ_ERR_NONFINITE : KVQ_OK;
}

int allocate_report(const void *workspace, kvq_report *r) {
    Ctrl c;
    if (cudaMemcpy(&c, workspace, sizeof(Ctrl), cudaMemcpyDeviceToHost) != cudaSuccess)
        return KVQ_ERR_CUDA;
    r->rounds = c.s.rounds;
    for (int i = 0; i < 16; ++i) r->active[i] = c.active[i];
    r->lambda = c.s.lambda;
    r->xa = c.s.xa;
    r->xb = c.s.xb;
    r->steps = c.s.step;
    r->t_start = c.t_start;
    r->t_end = c.t_end;
    for (int i = 0; i < 16; ++i) {
        r->t_dp[i] = c.t_dp[i];
        r->t_ctl[i] = c.t_ctl[i];
    }
    return KVQ_OK;
}

template <bool GENERAL, bool QUANT>
static int setup_search_kernel(int sms, int &resident) {
    const void *fn = (const void *)search_kernel<GENERAL, QUANT>;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)RoundCfg<GENERAL>::kSmem) != cudaSuccess)
        return KVQ_ERR_CUDA;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, RoundCfg<GENERAL>::kWarps * 32,
                                                      RoundCfg<GENERAL>::kSmem) != cudaSuccess ||
        occ < 1)
        return KVQ_ERR_CUDA;
    resident = occ * sms;
    return KVQ_OK;
}

int allocate_init() {
    // more than 48 KB of dynamic shared memory for the search kernels, and the
    // number of their CTAs that fit on the device at once (the cooperative grid)
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVQ_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return KVQ_ERR_CUDA;
    int (&r)[2][2] = g_resident[dev];
    if (setup_search_kernel<false, false>(sms, r[0][0]) != KVQ_OK ||
        setup_search_kernel<false, true>(sms, r[0][1]) != KVQ_OK ||
        setup_search_kernel<true, false>(sms, r[1][0]) != KVQ_OK ||
        setup_search_kernel<true, true>(sms, r[1][1]) != KVQ_OK)
        return KVQ_ERR_CUDA;
    if (cudaFuncSetAttribute((const void *)rate_sums_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)RoundCfg<false>::kSmem) != cudaSuccess ||
        cudaFuncSetAttribute((const void *)rate_sums_kernel<true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)RoundCfg<true>::kSmem) != cudaSuccess)
        return KVQ_ERR_CUDA;
    if (cudaFuncSetAttribute((const void *)fixed_rate_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)RoundCfg<false>::kSmem) != cudaSuccess ||
        cudaFuncSetAttribute((const void *)fixed_rate_kernel<true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)RoundCfg<true>::kSmem) != cudaSuccess)
        return KVQ_ERR_CUDA;
    // the module is loaded on this device now (the attributes above needed
    // it), so the static scratch exists: take its device address
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || p == nullptr)
        return KVQ_ERR_CUDA;
    g_static_addr[dev] = p;
    return KVQ_OK;
}

void *static_workspace_address(int dev) {
    return dev >= 0 && dev < kMaxDevices ? g_static_addr[dev] : nullptr;
}

}  // namespace kvq
