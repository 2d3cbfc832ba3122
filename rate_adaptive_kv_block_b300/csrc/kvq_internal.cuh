// Internal definitions shared by the CUDA translation units of libkvq.
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>

#include "kvq.h"
#include "kvq_search.h"

namespace kvq {

// Test hook for the error paths of the kernels' bounded waits: with
// KVQ_TEST_WAIT_LIMIT_NS set in the environment when a call is made, the
// search kernel's hand-over waits give up after that many nanoseconds and
// the quantize and attention kernels' waits for their bulk copies without
// polling, so that those calls return KVQ_ERR_TIMEOUT in their status
// instead of their results.  (The waits for copies still in flight when a
// kernel leaves keep their normal limit.)  Unset: the normal limits.
inline bool test_wait_limit(unsigned long long *ns) {
    const char *e = getenv("KVQ_TEST_WAIT_LIMIT_NS");
    if (!e || !*e) return false;
    *ns = strtoull(e, nullptr, 10);
    return true;
}

constexpr int kCand = 17;       // order-statistic candidates per block
constexpr int kMaxLev = 16;     // levels per block (4-bit codes)
constexpr int kPairs = 136;     // slot pairs j < l over 17 slots
constexpr int kTriples = 680;   // slot triples i < j < l

// ---------------------------------------------------------------- stats row
// One row per block, written by kvq_stats, read by kvq_allocate.  Atom p
// (p = 0 .. m'-2) holds the entries c_p <= x < c_{p+1} (the last atom also
// the entries equal to the maximum): n, s1 = sum(x - c_p),
// t1 = sum(c_{p+1} - x), e = sum((x - c_p)(c_{p+1} - x)); kvq_stats_weighted
// stores the weighted sums (n = sum w, s1 = sum w (x - c_p), ...) instead.
struct StatsRow {
    float c[kCand];      // merged candidates, padded with the maximum
    int32_t mprime;      // number of distinct candidates (1..17)
    int32_t flags;       // kFlag* bits
    int32_t d;           // entries in the block
    float n[16];
    float s1[16];
    float t1[16];
    float e[16];
    float pad[12];
};
static_assert(sizeof(StatsRow) == 384, "stats row is 384 bytes");
constexpr int kFlagNonfinite = 1;   // a non-finite entry
constexpr int kFlagBadWeight = 2;   // a negative or non-finite weight
constexpr int kFlagWeighted = 4;    // the moments and Dp are weighted

// ------------------------------------------------------------- table layout
// Per-block, lambda-independent DP tables, in "slot" space: the m'
// candidates sit in slots 0 .. m'-2 and 16 (the maximum always in slot 16);
// slots m'-1 .. 15 are unused ("dummy") when m' < 17.
//   Dp(j,l)    expected squared error of entries in [q_j, q_l)  (+inf for
//              a dummy slot)
//   hh(i,j,l)  h(Mup(i,j) + Mdn(j,l)): entropy term of level j between
//              levels i and l, h(M) = -M log2(M/d)
//   h0(l)      h(Mdn(0,l)): term of the first level
//   hend(i)    h(Mup(i,16)): term of the last level
// Row j of Dp holds l = j+1 .. 16 and row (i,j) of hh holds l = j+1 .. 16,
// each padded to a multiple of 4 floats so rows start on 16 bytes.
// pidx(j,l) is the compact index of a pair (lane-private DP state).
__host__ __device__ constexpr int pad4(int n) { return (n + 3) & ~3; }
// Closed forms (row j holds 16 - j entries padded to 16 - 4 floor(j/4)):
//   dp_off(j)    = sum_{j' < j} pad4(16 - j')
//   trip_base(j) = sum_{1 <= j' < j} j' pad4(16 - j')
__host__ __device__ constexpr int dp_off(int j) {
    const int q = j >> 2, r = j & 3;
    return 64 * q - 8 * q * (q - 1) + r * (16 - 4 * q);
}
__host__ __device__ constexpr int trip_base(int j) {
    const int q = j >> 2, r = j & 3;
    const int full = q == 0 ? 0 : q == 1 ? 96 : q == 2 ? 360 : q == 3 ? 664 : 880;
    return full + (16 - 4 * q) * (4 * q * r + r * (r - 1) / 2);
}
__host__ __device__ constexpr int trip_off(int i, int j) { return trip_base(j) + i * (16 - 4 * (j >> 2)); }
__host__ __device__ constexpr int pidx(int j, int l) { return 16 * j - j * (j - 1) / 2 + l - j - 1; }
// the closed forms agree with the sums they stand for
__host__ __device__ constexpr bool check_offsets() {
    int a = 0, b = 0;
    for (int j = 0; j <= 16; ++j) {
        if (dp_off(j) != a) return false;
        if (j >= 1 && trip_base(j) != b) return false;
        if (j < 16) a += pad4(16 - j);
        if (j >= 1 && j < 16) b += j * pad4(16 - j);
        if (j < 16 && 16 - 4 * (j >> 2) != pad4(16 - j)) return false;
    }
    return true;
}
static_assert(check_offsets(), "table offsets");
constexpr int kDpFloats = dp_off(16);          // 160
constexpr int kHHFloats = trip_base(16);       // 880
static_assert(kDpFloats == 160 && kHHFloats == 880, "padded table sizes");
static_assert(pidx(15, 16) == kPairs - 1, "pair count");

// Output of kvq_stats: a 256-byte header, then one 4800-byte record per
// block: the stats row (96 floats) and the DP tables (1104 floats).
struct StatsHeader {
    unsigned long long hi0_bits;   // max_r (c_max - c_min)^2 w_max,r (double bits, atomic max;
                                   // w_max,r = 1 without weights)
    uint32_t flags;                // OR of the block flags
    uint32_t pad[61];
};
static_assert(sizeof(StatsHeader) == 256, "stats header is 256 bytes");
constexpr int kRecFloats = 1200;
constexpr int kRecTbl = 96;

constexpr int kTblD = 0;
constexpr int kTblHH = kTblD + kDpFloats;     // 160
constexpr int kTblH0 = kTblHH + kHHFloats;    // 1040
constexpr int kTblHend = kTblH0 + 20;         // 1060
constexpr int kTblC = kTblHend + 20;          // 1080: level value per slot
constexpr int kTblHdr = kTblC + 20;           // 1100: m', d, flags (int bits)
constexpr int kTblStride = 1104;              // floats per block (4416 B)
static_assert(kTblStride % 4 == 0 && kTblHH % 4 == 0 && kTblH0 % 4 == 0, "16-byte rows");

// Decode of a padded hh entry: (i, j, l) packed as i | j << 8 | l << 16
// (l = 17 marks padding), and of a padded Dp entry: j | l << 8.
struct DecodeTables {
    uint32_t trip[kHHFloats];
    uint32_t pair[kDpFloats];
};
// trip[idx]: pidx(i, j) | pidx(j, l) << 8 | i << 16 | j << 21 | l << 26 of HH
// entry idx (l = 17 on row padding); pair[idx]: j | l << 8 of D entry idx.
constexpr DecodeTables make_decode() {
    DecodeTables t{};
    for (int j = 1; j < 16; ++j)
        for (int i = 0; i < j; ++i)
            for (int k = 0; k < pad4(16 - j); ++k) {
                const int l = j + 1 + k;
                const uint32_t pjl = l < 17 ? (uint32_t)pidx(j, l) : 0u;
                t.trip[trip_off(i, j) + k] = (uint32_t)pidx(i, j) | (pjl << 8) |
                                             ((uint32_t)i << 16) | ((uint32_t)j << 21) |
                                             ((uint32_t)(l < 17 ? l : 17) << 26);
            }
    for (int j = 0; j < 16; ++j)
        for (int k = 0; k < pad4(16 - j); ++k) {
            const int l = j + 1 + k;
            t.pair[dp_off(j) + k] = (uint32_t)j | ((uint32_t)(l < 17 ? l : 17) << 8);
        }
    return t;
}
static __device__ constexpr DecodeTables kDecode = make_decode();

// ---------------------------------------------------- allocation control
// Lives at the start of the kvq_allocate workspace.
struct alignas(16) Ctrl {
    SearchState s;          // lambda search (kvq_search.h)
    double budget;          // B (bits)
    long long budget_fx;    // floor(B 2^20): R <= B iff R_fx <= budget_fx
    double eta;             // subgradient step
    double lambda_fixed;    // KVQ_SUBGRADIENT: the lambda of this step
    unsigned long long hi0_bits;   // max_r (c_max - c_min)^2 (double bits)
    int32_t fixed;          // 1: one round at lambda_fixed
    int32_t status;
    int32_t flags;          // OR of block flags
    int32_t mode;
    uint32_t ticket;        // last-CTA-done counter of the search rounds
    uint32_t ticket_emit;   // same, emit
    uint32_t gen;           // rounds released to the grid (persistent search kernel)
    uint32_t err;           // a CTA gave up waiting for a release
    uint32_t fin_tail;      // fused path: blocks whose chain is final, queued so far
    uint32_t fin_avail;     // fused path: queued blocks published to the idle warps
    uint32_t ticket_f;      // fused path: CTAs out of the rounds
    uint32_t pad_f;
    uint32_t active[16];    // blocks evaluated in each round (diagnostics)
    int64_t nb;             // blocks
    // sum over all blocks of d_r H_r at xb, fixed point; the rounds of the
    // walk add to it the change of each re-evaluated block
    long long Rxb_fx;
    uint32_t cnt[2];        // lengths of the two candidate lists
    // per-probe sum of d_r H_r over blocks, fixed point (2^-20 bit units):
    // integer adds are exact, so the sum does not depend on arrival order
    unsigned long long acc[32];
    // %globaltimer stamps (ns; diagnostics): kernel start, the end of each
    // round's DP (the last CTA's ticket), its control's second publication,
    // and the end of the emit
    unsigned long long t_start, t_end, t_dp[16], t_ctl[16];
    unsigned long long wait_ns;    // limit of each grid hand-over wait
    uint32_t spin_limit;           // and of its polls
    // the search phase as of a control's first publication (the round kind
    // the other CTAs act on); the second publication does not change it, so
    // a CTA that has only seen the first never reads a phase the walk set
    int32_t phase1;
};
static_assert(sizeof(Ctrl) % 16 == 0, "control block in 16-byte pieces");
constexpr double kRateScale = 1048576.0;   // 2^20

// ------------------------------------------------------------ binary16 keys
// Order-preserving 16-bit key of a binary16 value (-0 folded into +0):
// negative values map below 0x8000, non-negative at or above it.
__device__ __forceinline__ uint32_t f16_key(uint32_t h) {
    h = (h == 0x8000u) ? 0u : h;
    return (h & 0x8000u) ? (~h & 0xffffu) : (h | 0x8000u);
}
// The keys of the two binary16 values packed in w (low half first), packed
// the same way: both zeros fold into +0 (one packed compare), then each half
// flips its sign bit, or all its bits when it is negative.
__device__ __forceinline__ uint32_t f16_key2(uint32_t w) {
    __half2 h;
    memcpy(&h, &w, sizeof(w));
    w &= ~__heq2_mask(h, __float2half2_rn(0.0f));
    const uint32_t neg = (w >> 15) & 0x00010001u;
    return w ^ 0x80008000u ^ (neg * 0x7fffu);
}
__device__ __forceinline__ uint32_t key_to_bits(uint32_t key) {
    return (key & 0x8000u) ? (key & 0x7fffu) : (~key & 0xffffu);
}
__device__ __forceinline__ float key_value(uint32_t key) {
    return __half2float(__ushort_as_half((unsigned short)key_to_bits(key)));
}
// spacing of consecutive keys inside the 256-key bin b (binary16 ulp there)
__device__ __forceinline__ float bin_ulp(uint32_t b) {
    uint32_t e = (key_to_bits(b << 8) >> 10) & 31u;
    return e == 0 ? 5.9604644775390625e-8f : __int_as_float((int)((e - 25 + 127) << 23));
}

// -------------------------------------------------------------- block map
struct BlockPos {
    int64_t stream, tblock;
    int group;
};
__host__ __device__ __forceinline__ int64_t num_blocks(const kvq_layout &L) {
    return L.S * (L.T / 32) * (int64_t)(L.D / L.group);
}

}  // namespace kvq
