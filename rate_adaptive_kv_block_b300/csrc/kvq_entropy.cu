// kvq_entropy_encode / kvq_entropy_decode: the blocks' 4-bit symbols stored
// entropy-coded ("Rate-adaptive KV-cache quantizer", "Implementation notes":
// store the codebook, symbol stream and block lengths, with arithmetic
// coding of the symbols), so that the stored bytes follow sum_r d_r H_r
// instead of 4 bits per entry.
//
// Coder: range asymmetric numeral systems (rANS, Duda 2013) with 32-bit
// state, byte-wise renormalisation (Giesen's formulation): state x in
// [L, 256 L), L = 2^23; the model is the block's exact symbol counts, whose
// total is the block size d (a power of two, so no rescaling): for symbol c
// with count f_c and cumulative count b_c,
//   encode:  while x >= ((L >> log2 d) << 8) f_c: emit x & 255, x >>= 8
//            x = (x / f_c) << log2 d + x % f_c + b_c
//   decode:  s = x & (d - 1); c: b_c <= s < b_c + f_c
//            x = f_c (x >> log2 d) + s - b_c; while x < L: x = x << 8 | next byte
// 32 interleaved streams per block: stream l codes entries l, l+32, l+64, ..
// (one stream per lane of a warp), encoded last entry first so that the
// decoder runs forwards.
//
// Block slot (fixed capacity kvq_entropy_slot_bytes(d), little-endian):
//   [0, 32)   16 x u16: count of each symbol
//   [32, 96)  32 x u16: bytes of each stream
//   [96, ..)  the streams in lane order; stream l = its final encoder state
//             (4 bytes) followed by its renormalisation bytes in the order
//             the decoder reads them
// nbytes[r] = 96 + sum of the stream lengths (the block's stored size).
#include "kvq_internal.cuh"

namespace kvq {

constexpr uint32_t kRansL = 1u << 23;
constexpr int kEntWarps = 4;
constexpr int kEntHeader = 96;
// bytes of a stream the per-block encoder keeps from its first pass: 4 bits
// a symbol of a 4096-entry block and 32 bytes of slack (a symbol emits at
// most two bytes, so a longer stream exists; its block is written by a
// second pass)
constexpr int kEntKeep = 4096 / 32 / 2 + 32;

__host__ __device__ constexpr uint32_t entropy_slot_bytes(int d) {
    // the payload is at most d * 4 bits (16 symbols) plus, per stream, the
    // state and one byte of renormalisation slack
    return (uint32_t)(d / 2 + kEntHeader + 32 * 6);
}

__device__ __forceinline__ int ilog2(int v) { return 31 - __clz(v); }

// x / f for x < 2^31 and 1 <= f <= 4096 by one 64-bit product: with
// l = ceil(log2 f) and m = floor(2^(31+l) / f) + 1 (at most 32 bits),
// floor(x m / 2^(31+l)) = floor(x / f) for every 31-bit x (Granlund and
// Montgomery 1994, Theorem 4.2)
struct Recip {
    uint32_t m;
    uint32_t sh;
};
__device__ __forceinline__ Recip recip_of(uint32_t f) {
    const uint32_t l = f > 1 ? 32u - __clz(f - 1u) : 0u;
    const uint64_t m = ((1ull << (31 + l)) / f) + 1ull;
    return Recip{(uint32_t)m, 31u + l};
}
__device__ __forceinline__ uint32_t div_by(uint32_t x, Recip r) {
    return (uint32_t)(((uint64_t)x * r.m) >> r.sh);
}

// n16 16-byte words from global to shared memory by one warp, in batches of
// eight per lane: each batch's loads are in flight together (a sequential
// load-store loop would wait one memory round trip per iteration).
__device__ __forceinline__ void stage16(uint4 *__restrict__ dst, const uint4 *__restrict__ src,
                                        int n16, int lane) {
    for (int base = 0; base < n16; base += 8 * 32) {
        uint4 v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = base + lane + 32 * k;
            if (i < n16) v[k] = __ldg(src + i);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = base + lane + 32 * k;
            if (i < n16) dst[i] = v[k];
        }
    }
}

// Counts of the 16 symbols over a warp: each lane counts its n <= 128
// symbols in four registers of four 8-bit counters (symbol c adds 1 to byte
// c & 3 of register c >> 2), then the counts go to eight registers of two
// 16-bit counters (a warp's count is at most 4096) for the warp sum.
template <typename SymAt>
__device__ __forceinline__ void warp_counts(int n, SymAt sym_at, uint32_t (&cnt)[16]) {
    uint32_t pk[4] = {0u, 0u, 0u, 0u};
    for (int j = 0; j < n; ++j) {
        const uint32_t c = sym_at(j);
        const uint32_t inc = 1u << ((c & 3u) << 3);
        const uint32_t g = c >> 2;
        pk[0] += g == 0u ? inc : 0u;
        pk[1] += g == 1u ? inc : 0u;
        pk[2] += g == 2u ? inc : 0u;
        pk[3] += g == 3u ? inc : 0u;
    }
    uint32_t h[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t w = pk[k >> 1] >> ((k & 1) * 16);        // counters 2k, 2k+1
        h[k] = (w & 0xffu) | ((w & 0xff00u) << 8);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) h[k] += __shfl_xor_sync(0xffffffffu, h[k], o);
#pragma unroll
    for (int t = 0; t < 16; ++t) cnt[t] = (h[t >> 1] >> ((t & 1) * 16)) & 0xffffu;
}

__global__ void __launch_bounds__(kEntWarps * 32)
entropy_encode_kernel(const uint8_t *__restrict__ codes, int64_t nb, int d,
                      uint8_t *__restrict__ out, uint32_t *__restrict__ nbytes) {
    __shared__ uint8_t scratch[kEntWarps][32][kEntKeep];
    __shared__ __align__(16) uint8_t sslot[kEntWarps][entropy_slot_bytes(4096)];
    __shared__ uint4 smodel[kEntWarps][16];        // per symbol: count, cumulative, reciprocal
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t b = (int64_t)blockIdx.x * kEntWarps + w;
    if (b >= nb) return;
    const int n = d / 32, lg = ilog2(d);
    // the block's codes in shared memory (coalesced 16-byte loads)
    uint8_t *cb = sslot[w];
    stage16(reinterpret_cast<uint4 *>(cb), reinterpret_cast<const uint4 *>(codes + b * (d / 2)),
            d / 32, lane);
    __syncwarp();
    // the block's counts (lane-private, then a warp sum)
    uint32_t cnt[16];
    warp_counts(n, [&](int j) {
        const int e = lane + 32 * j;
        return (uint32_t)((cb[e >> 1] >> ((e & 1) * 4)) & 15u);
    }, cnt);
    uint32_t cum[17];
    cum[0] = 0;
#pragma unroll
    for (int t = 0; t < 16; ++t) cum[t + 1] = cum[t] + cnt[t];
    // the model, one entry per symbol in shared memory (lane t < 16: its
    // count, cumulative count and the count's reciprocal, a 64-bit division
    // once per block)
    uint32_t myf = 0;                             // lane t < 16: count of symbol t
    if (lane < 16) {
        uint32_t bc = 0;
#pragma unroll
        for (int t = 0; t < 16; ++t)
            if (t == lane) { myf = cnt[t]; bc = cum[t]; }
        const Recip r = recip_of(myf > 0 ? myf : 1u);
        smodel[w][lane] = make_uint4(myf, bc, r.m, r.sh);
    }
    __syncwarp();
    // this lane's stream, last entry first.  Its symbol j (entry lane + 32 j)
    // is the nibble (lane & 1) of code byte 16 j + lane / 2, read from the
    // staged codes.  The bytes that leave are kept in the order they leave
    // (up to kEntKeep of them); the state's final value opens the stream and
    // the decoder reads the bytes last first.
    const uint8_t *mine = cb + (lane >> 1);
    const int nsh = 4 * (lane & 1);
    auto sym_at = [&](int j) { return (uint32_t)(mine[16 * j] >> nsh) & 15u; };
    const uint32_t xmax0 = (kRansL >> lg) << 8;
    uint8_t *kept = scratch[w][lane];
    uint32_t nout = 0, x = kRansL;
    uint4 nxt = smodel[w][sym_at(n - 1)];     // the next symbol's model, one step ahead
    for (int j = n - 1; j >= 0; --j) {
        const uint4 md = nxt;
        nxt = smodel[w][sym_at(max(j - 1, 0))];   // the last step reloads its own
        const uint32_t xmax = xmax0 * md.x;
        // at most two bytes leave per symbol (x < 2^31, xmax >= 2^19): two
        // predicated steps instead of a loop whose trip count differs by lane
        const uint32_t e1 = x >= xmax ? 1u : 0u;
        if (e1 && nout < kEntKeep) kept[nout] = (uint8_t)x;
        nout += e1;
        x >>= 8 * e1;
        const uint32_t e2 = x >= xmax ? 1u : 0u;
        if (e2 && nout < kEntKeep) kept[nout] = (uint8_t)x;
        nout += e2;
        x >>= 8 * e2;
        const uint32_t qd = div_by(x, Recip{md.z, md.w});
        x = (qd << lg) + (x - qd * md.x) + md.y;
    }
    const uint32_t len = nout + 4;
    // offsets of the streams (exclusive scan over the lanes)
    uint32_t off = len;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, off, o);
        if (lane >= o) off += y;
    }
    const uint32_t total = __shfl_sync(0xffffffffu, off, 31);
    off -= len;
    const uint32_t size = kEntHeader + total;
    uint8_t *slot = out + b * (int64_t)entropy_slot_bytes(d);
    if (!__any_sync(0xffffffffu, nout > (uint32_t)kEntKeep)) {
        // every lane kept its bytes: the slot assembled in shared memory (the
        // codes are no longer needed), then stored with 16-byte writes
        __syncwarp();
        uint8_t *ss = sslot[w];
        if (lane < 16) {
            ss[2 * lane] = (uint8_t)myf;
            ss[2 * lane + 1] = (uint8_t)(myf >> 8);
        }
        ss[32 + 2 * lane] = (uint8_t)len;
        ss[32 + 2 * lane + 1] = (uint8_t)(len >> 8);
        uint8_t *st = ss + kEntHeader + off;
        st[0] = (uint8_t)x;
        st[1] = (uint8_t)(x >> 8);
        st[2] = (uint8_t)(x >> 16);
        st[3] = (uint8_t)(x >> 24);
        for (uint32_t i = 0; i < nout; ++i) st[4 + i] = kept[nout - 1 - i];
        __syncwarp();
        for (uint32_t i = 16 * lane; i < size; i += 16 * 32) {
            if (i + 16 <= size) {
                *reinterpret_cast<uint4 *>(slot + i) = *reinterpret_cast<const uint4 *>(ss + i);
            } else {
                for (uint32_t k = i; k < size; ++k) slot[k] = ss[k];
            }
        }
    } else {
        // some stream is longer than what it kept: the same steps again, each
        // byte written straight to its place in the slot (from the stream's
        // end downwards), and the header beside them
        if (lane < 16) {
            slot[2 * lane] = (uint8_t)myf;
            slot[2 * lane + 1] = (uint8_t)(myf >> 8);
        }
        slot[32 + 2 * lane] = (uint8_t)len;
        slot[32 + 2 * lane + 1] = (uint8_t)(len >> 8);
        uint8_t *st = slot + kEntHeader + off;
        uint32_t pos = len;
        x = kRansL;
        nxt = smodel[w][sym_at(n - 1)];
        for (int j = n - 1; j >= 0; --j) {
            const uint4 md = nxt;
            nxt = smodel[w][sym_at(max(j - 1, 0))];
            const uint32_t xmax = xmax0 * md.x;
            const bool e1 = x >= xmax;
            if (e1) st[pos - 1] = (uint8_t)(x & 255u);
            pos -= e1 ? 1u : 0u;
            x = e1 ? x >> 8 : x;
            const bool e2 = x >= xmax;
            if (e2) st[pos - 1] = (uint8_t)(x & 255u);
            pos -= e2 ? 1u : 0u;
            x = e2 ? x >> 8 : x;
            const uint32_t qd = div_by(x, Recip{md.z, md.w});
            x = (qd << lg) + (x - qd * md.x) + md.y;
        }
        st[0] = (uint8_t)x;
        st[1] = (uint8_t)(x >> 8);
        st[2] = (uint8_t)(x >> 16);
        st[3] = (uint8_t)(x >> 24);
    }
    if (lane == 0) nbytes[b] = size;
}

__global__ void __launch_bounds__(kEntWarps * 32)
entropy_decode_kernel(const uint8_t *__restrict__ in, int64_t nb, int d,
                      uint8_t *__restrict__ codes, int32_t *__restrict__ status) {
    // per warp: the symbol of every slot s < d.  With exact counts the slot
    // table is the block's symbols in symbol order (b_c .. b_{c+1} - 1 hold c),
    // so one lookup replaces the search over the cumulative counts.
    __shared__ __align__(16) uint8_t smap[kEntWarps][4096];
    __shared__ __align__(16) uint8_t sslot[kEntWarps][entropy_slot_bytes(4096)];
    __shared__ uint32_t sent[kEntWarps][16];        // per symbol: b_c | f_c << 16
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t b = (int64_t)blockIdx.x * kEntWarps + w;
    if (b >= nb) return;
    const int n = d / 32, lg = ilog2(d);
    const uint32_t cap = entropy_slot_bytes(d);
    // the whole slot in shared memory (16-byte loads; the capacity is a
    // multiple of 16)
    stage16(reinterpret_cast<uint4 *>(sslot[w]), reinterpret_cast<const uint4 *>(in + b * (int64_t)cap),
            (int)(cap / 16), lane);
    __syncwarp();
    const uint8_t *slot = sslot[w];
    // counts and cumulative counts (lane t < 16 reads count t; a warp scan
    // gives the cumulative counts)
    const uint32_t mycnt = lane < 16 ? ((uint32_t)slot[2 * lane] | ((uint32_t)slot[2 * lane + 1] << 8)) : 0u;
    uint32_t incl = mycnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const uint32_t nsym = __shfl_sync(0xffffffffu, incl, 15);
    if (lane < 16) sent[w][lane] = (incl - mycnt) | (mycnt << 16);
    const uint32_t len = (uint32_t)slot[32 + 2 * lane] | ((uint32_t)slot[32 + 2 * lane + 1] << 8);
    uint32_t off = len;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, off, o);
        if (lane >= o) off += y;
    }
    const uint32_t total = __shfl_sync(0xffffffffu, off, 31);
    off -= len;
    // a slot that does not describe a block of d symbols: status, codes 0
    bool bad = nsym != (uint32_t)d || kEntHeader + total > cap || len < 4;
    bad = __any_sync(0xffffffffu, bad);
    __syncwarp();
    uint8_t *map = smap[w];
    const uint32_t *ent = sent[w];
    if (!bad) {
        // symbol c fills slots [a, a + f): whole 4-byte words with the
        // repeated byte, then at most three bytes at either end (every b_c
        // and f_c is at most d <= 4096 once the counts sum to d)
        uint32_t *m32 = reinterpret_cast<uint32_t *>(map);
        for (int c = 0; c < 16; ++c) {
            const uint32_t e = ent[c], a = e & 0xffffu, z = a + (e >> 16);
            const uint32_t wa = (a + 3u) >> 2, wz = z >> 2;
            for (uint32_t i = wa + (uint32_t)lane; i < wz; i += 32) m32[i] = (uint32_t)c * 0x01010101u;
            if (lane < 6) {
                const uint32_t q = lane < 3 ? a + (uint32_t)lane : z - 1u - (uint32_t)(lane - 3);
                const uint32_t wq = q >> 2;
                if (q >= a && q < z && !(wq >= wa && wq < wz)) map[q] = (uint8_t)c;
            }
        }
    }
    __syncwarp();
    uint32_t p = kEntHeader + off, end = p + len;
    uint32_t x = 0;
    if (!bad) {
        x = (uint32_t)slot[p] | ((uint32_t)slot[p + 1] << 8) | ((uint32_t)slot[p + 2] << 16) |
            ((uint32_t)slot[p + 3] << 24);
        p += 4;
    }
    bool overrun = false;
    // entry lane + 32 j is the low nibble of code byte 16 j + lane / 2 when
    // the lane is even, the high nibble of that byte when it is odd
    uint8_t *cout = codes + b * (d / 2) + (lane >> 1);
    if (bad) {
        for (int i = lane; i < d / 2; i += 32) codes[b * (d / 2) + i] = 0;
    } else {
        for (int j = 0; j < n; ++j) {
            const uint32_t s = x & ((1u << lg) - 1u);
            const uint32_t c = map[s];
            const uint32_t e = ent[c];
            x = (e >> 16) * (x >> lg) + s - (e & 0xffffu);
            // a stream this coder wrote refills at most two bytes per symbol
            // (the encoder's bound); never read past the stream.  (Issue
            // bound with eight CTAs per SM, this kernel takes the refills as
            // branches; the run decoder, one warp per SM, loads both bytes
            // ahead instead.)
            if (x < kRansL) {
                if (p < end) x = (x << 8) | slot[p++];
                else overrun = true;
            }
            if (x < kRansL) {
                if (p < end) x = (x << 8) | slot[p++];
                else overrun = true;
            }
            if (x < kRansL) overrun = true;            // a third: not such a stream
            const uint32_t hi = __shfl_xor_sync(0xffffffffu, c, 1);
            if ((lane & 1) == 0) cout[16 * j] = (uint8_t)(c | (hi << 4));
        }
    }
    overrun |= !bad && p != end;
    if (__any_sync(0xffffffffu, bad || overrun) && lane == 0) atomicMax(status, (int32_t)KVQ_ERR_CORRUPT);
}

// ------------------------------------------- runs of adjacent blocks
// Coding across adjacent blocks ("Implementation notes": arithmetic coding
// across adjacent blocks): a run of nseg consecutive blocks is one set of 32
// interleaved rANS streams whose state continues from block to block (stream
// l: entries l, l+32, .. of the run's first block, then of the next, ..);
// each symbol is coded with its own block's exact counts, so blocks keep
// their models while the 32 states and lengths are stored once per run.
// Run slot (capacity kvq_entropy_run_bytes, little-endian):
//   [0, 32 m)          16 x u16 counts of each of the m blocks
//   [32 m, 32 m + 64)  32 x u16: bytes of each stream
//   then the streams in lane order, each its final state (4 bytes) and its
//   renormalisation bytes in the order the decoder reads them.
// One warp per run and per CTA, so the runs spread over every SM.  The
// encoder first stages the run's codes and models in shared memory.  Its
// pass over the run counts each stream's bytes and keeps them, up to 4 bits a
// symbol and some slack, in shared memory; once a warp scan of the lengths
// has placed the streams, the kept bytes go out last first.  Only when some
// stream fills what it could keep does a second pass recompute the
// chain and write the bytes downwards from the stream's end (known from the
// first), so no worst-case scratch is held.  The decoder stages the run's
// slot (as far as its stream lengths reach), builds each block's slot table
// and assembles its packed codes in shared memory before one coalesced store.
// Both serial per-lane loops then touch shared memory only.
constexpr int kRunMaxBlocks = 32;

__host__ __device__ constexpr uint64_t run_slot_bytes(int d, int nseg) {
    // at most 4 bits a symbol (exact counts), the counts, the lengths, and per
    // stream its state and one byte of renormalisation slack
    return ((uint64_t)nseg * (uint64_t)(d / 2 + 32) + 64u + 32u * 6u + 15u) & ~(uint64_t)15u;
}
// bytes of one lane's stream the run encoder keeps from its first pass: 4
// bits per symbol and some slack (a stream longer than that is written by a
// second pass instead)
__host__ __device__ constexpr uint32_t run_keep_bytes(int d, int nseg) {
    return ((uint32_t)(d / 32) * (uint32_t)nseg / 2u + 64u + 15u) & ~15u;
}
// dynamic shared memory of the two kernels
__host__ __device__ constexpr size_t run_enc_smem(int d, int nseg) {
    return (size_t)nseg * (16 * sizeof(uint4) + (size_t)(d / 2)) + 32 * (size_t)run_keep_bytes(d, nseg);
}
__host__ __device__ constexpr size_t run_dec_smem(int d, int nseg) {
    return 144 + (size_t)(d / 2) + (size_t)run_slot_bytes(d, nseg) + 4 * (size_t)d;
}
constexpr size_t kRunSmemMax = run_enc_smem(4096, kRunMaxBlocks) > run_dec_smem(4096, kRunMaxBlocks)
                                   ? run_enc_smem(4096, kRunMaxBlocks)
                                   : run_dec_smem(4096, kRunMaxBlocks);

__device__ __forceinline__ uint32_t nibble_at(const uint8_t *cb, int e) {
    return (cb[e >> 1] >> ((e & 1) * 4)) & 15u;
}

__global__ void __launch_bounds__(32)
entropy_encode_runs_kernel(const uint8_t *__restrict__ codes, int64_t nb, int d, int nseg,
                           uint8_t *__restrict__ out, uint32_t *__restrict__ nbytes) {
    extern __shared__ __align__(16) uint8_t rsm[];
    uint4 *smodel = reinterpret_cast<uint4 *>(rsm);            // [block][symbol]: count,
                                                               // cumulative, reciprocal
    uint8_t *scodes = rsm + (size_t)nseg * 16 * sizeof(uint4);   // the run's codes
    const int lane = threadIdx.x;
    const int64_t rn = blockIdx.x;
    const int64_t b0 = rn * nseg;
    const int m = (int)min((int64_t)nseg, nb - b0);
    const int n = d / 32, lg = ilog2(d);
    const int half = d / 2;
    uint8_t *slot = out + rn * (int64_t)run_slot_bytes(d, nseg);
    // 16-byte copies: codes is 16-byte aligned and half a multiple of 16
    stage16(reinterpret_cast<uint4 *>(scodes), reinterpret_cast<const uint4 *>(codes + b0 * half),
            m * half / 16, lane);
    __syncwarp();
    // the blocks' models: counts (lane-private, then warp sums), cumulative
    // counts, reciprocals; the counts also go to the slot
    for (int bi = 0; bi < m; ++bi) {
        const uint8_t *cb = scodes + bi * half;
        uint32_t cnt[16];
        warp_counts(n, [&](int j) { return nibble_at(cb, lane + 32 * j); }, cnt);
        if (lane < 16) {
            uint32_t f = 0, bc = 0, acc = 0;
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                if (t == lane) { f = cnt[t]; bc = acc; }
                acc += cnt[t];
            }
            const Recip r = recip_of(f > 0 ? f : 1u);
            smodel[bi * 16 + lane] = make_uint4(f, bc, r.m, r.sh);
            slot[32 * bi + 2 * lane] = (uint8_t)f;
            slot[32 * bi + 2 * lane + 1] = (uint8_t)(f >> 8);
        }
    }
    __syncwarp();
    const uint32_t xmax0 = (kRansL >> lg) << 8;
    // pass 1: the length of this lane's stream, and its bytes in the order
    // they leave (up to `keep` of them).  The symbols are taken last first,
    // run position k = bi * n + j from m n - 1 down to 0; the next symbol's
    // model entry does not depend on the state, so it is loaded one step
    // ahead (the state's chain then holds only the arithmetic)
    const uint32_t keep = run_keep_bytes(d, nseg);
    uint8_t *kept = scodes + (size_t)nseg * half + (size_t)lane * keep;
    const int nk = m * n;
    // run position k = bi n + j (n = d / 32 = 2^(lg - 5)) is entry lane + 32 j
    // of block bi: nibble (lane & 1) of code byte bi d / 2 + 16 j + lane / 2
    // = 16 k + lane / 2 of the staged run
    const uint8_t *mine = scodes + (lane >> 1);
    const int nsh = 4 * (lane & 1), lgn = lg - 5;
    auto model_at = [&](int k) {
        return smodel[((k >> lgn) << 4) + ((mine[16 * k] >> nsh) & 15)];
    };
    uint32_t x = kRansL, nout = 0;
    uint4 nxt = model_at(nk - 1);
    for (int k = nk - 1; k >= 0; --k) {
        const uint4 md = nxt;
        nxt = model_at(max(k - 1, 0));          // the last step reloads its own
        const uint32_t xmax = xmax0 * md.x;
        // at most two bytes leave per symbol (x < 2^31, xmax >= 2^19)
        // the low byte is stored whether or not it leaves: a byte that stays
        // is overwritten by the next one that leaves (or lies past the
        // stream's end); the index is clamped only once nout reaches keep,
        // and such a stream takes the second pass.  (With one warp per SM
        // the store is cheaper than the predicate; the per-block encoder,
        // issue-bound, keeps its predicated store.)
        const uint32_t e1 = x >= xmax ? 1u : 0u;
        kept[min(nout, keep - 1u)] = (uint8_t)x;
        nout += e1;
        x >>= 8 * e1;
        const uint32_t e2 = x >= xmax ? 1u : 0u;
        kept[min(nout, keep - 1u)] = (uint8_t)x;
        nout += e2;
        x >>= 8 * e2;
        const uint32_t qd = div_by(x, Recip{md.z, md.w});
        x = (qd << lg) + (x - qd * md.x) + md.y;
    }
    const uint32_t len = nout + 4;
    uint32_t off = len;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, off, o);
        if (lane >= o) off += y;
    }
    const uint32_t total = __shfl_sync(0xffffffffu, off, 31);
    off -= len;
    const uint32_t hdr = 32u * (uint32_t)m + 64u;
    slot[32 * m + 2 * lane] = (uint8_t)len;
    slot[32 * m + 2 * lane + 1] = (uint8_t)(len >> 8);
    if (lane == 0) nbytes[rn] = hdr + total;
    uint8_t *st = slot + hdr + off;
    if (!__any_sync(0xffffffffu, nout >= keep)) {      // below keep the index was never clamped
        // every lane kept its bytes: the stream holds them last first
        for (uint32_t i = 0; i < nout; ++i) st[4 + i] = kept[nout - 1 - i];
    } else {
        // pass 2: the same steps, the bytes written downwards from the stream's end
        uint32_t pos = len;
        x = kRansL;
        nxt = model_at(nk - 1);
        for (int k = nk - 1; k >= 0; --k) {
            const uint4 md = nxt;
            nxt = model_at(max(k - 1, 0));
            const uint32_t xmax = xmax0 * md.x;
            const bool e1 = x >= xmax;
            if (e1) st[pos - 1] = (uint8_t)(x & 255u);
            pos -= e1 ? 1u : 0u;
            x = e1 ? x >> 8 : x;
            const bool e2 = x >= xmax;
            if (e2) st[pos - 1] = (uint8_t)(x & 255u);
            pos -= e2 ? 1u : 0u;
            x = e2 ? x >> 8 : x;
            const uint32_t qd = div_by(x, Recip{md.z, md.w});
            x = (qd << lg) + (x - qd * md.x) + md.y;
        }
    }
    st[0] = (uint8_t)x;          // the state opens the stream
    st[1] = (uint8_t)(x >> 8);
    st[2] = (uint8_t)(x >> 16);
    st[3] = (uint8_t)(x >> 24);
}

__global__ void __launch_bounds__(32)
entropy_decode_runs_kernel(const uint8_t *__restrict__ in, int64_t nb, int d, int nseg,
                           uint8_t *__restrict__ codes, int32_t *__restrict__ status) {
    extern __shared__ __align__(16) uint8_t rsm[];
    uint32_t *scum = reinterpret_cast<uint32_t *>(rsm);      // [16]: cumulative | count << 16
    uint8_t *sout = rsm + 144;                               // one block's packed codes
    const int lane = threadIdx.x;
    const int64_t rn = blockIdx.x;
    const int64_t b0 = rn * nseg;
    const int m = (int)min((int64_t)nseg, nb - b0);
    const int n = d / 32, lg = ilog2(d);
    const int half = d / 2;
    uint8_t *sslot = sout + half;                            // the run's slot
    const uint64_t cap = run_slot_bytes(d, nseg);
    uint32_t *smap = reinterpret_cast<uint32_t *>(sslot + cap);   // one block's slot table
    const uint8_t *slot = in + rn * (int64_t)cap;
    const uint32_t hdr = 32u * (uint32_t)m + 64u;
    const uint32_t len = (uint32_t)slot[32 * m + 2 * lane] | ((uint32_t)slot[32 * m + 2 * lane + 1] << 8);
    uint32_t off = len;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, off, o);
        if (lane >= o) off += y;
    }
    const uint32_t total = __shfl_sync(0xffffffffu, off, 31);
    off -= len;
    // a slot that does not hold m blocks of d symbols: status, codes 0
    bool bad = __any_sync(0xffffffffu, (uint64_t)hdr + total > cap || len < 4);
    {
        // stage what the streams reach (16-byte copies; cap and the slots'
        // offsets are multiples of 16), never more than the slot
        const uint64_t used = bad ? (uint64_t)hdr : (uint64_t)hdr + total;
        const int nq = (int)((used + 15u) / 16u);
        stage16(reinterpret_cast<uint4 *>(sslot), reinterpret_cast<const uint4 *>(slot), nq, lane);
    }
    __syncwarp();
    uint32_t p = hdr + off;
    const uint32_t end = p + len;
    uint32_t x = 0;
    if (!bad) {
        x = (uint32_t)sslot[p] | ((uint32_t)sslot[p + 1] << 8) | ((uint32_t)sslot[p + 2] << 16) |
            ((uint32_t)sslot[p + 3] << 24);
        p += 4;
    }
    bool overrun = false;
    const uint32_t last = end - 1;                   // len >= 4 when the slot is good
    uint8_t *dst = codes + b0 * half;
    for (int bi = 0; bi < m; ++bi) {
        // this block's model: counts from the slot, cumulative counts by a scan
        const uint32_t mycnt = lane < 16 ? ((uint32_t)sslot[32 * bi + 2 * lane] |
                                            ((uint32_t)sslot[32 * bi + 2 * lane + 1] << 8))
                                         : 0u;
        uint32_t incl = mycnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        __syncwarp();                              // the previous block is done with
        if (lane < 16) scum[lane] = (incl - mycnt) | (mycnt << 16);   // cumulative | count
        __syncwarp();
        const uint32_t tot = __shfl_sync(0xffffffffu, incl, 15);
        const bool badm = __any_sync(0xffffffffu, tot != (uint32_t)d);
        bad = bad || badm;
        // this block's slot table: slot b_c + q (q < f_c) holds
        // c << 28 | f_c << 13 | q, all that decoding a symbol there needs
        // (exact counts: slots b_c .. b_{c+1} - 1 belong to symbol c; once
        // the counts sum to d, every b_c + q is below d)
        if (!bad) {
            for (int c = 0; c < 16; ++c) {
                const uint32_t e = scum[c], a = e & 0xffffu, f = e >> 16;
                const uint32_t hi = ((uint32_t)c << 28) | (f << 13);
                for (uint32_t q = (uint32_t)lane; q < f; q += 32) smap[a + q] = hi | q;
            }
        }
        __syncwarp();
        if (bad) {
            for (int i = lane; i < half; i += 32) sout[i] = 0;
        } else {
            for (int j = 0; j < n; ++j) {
                // the stream's next two bytes, loaded before the state is
                // known (one clamp to the stream: the byte after it is still
                // inside this kernel's shared memory, and a stream that runs
                // out is reported at the end), so that the chain from one
                // state to the next holds one shared-memory load; at most two
                // refills
                const uint32_t pc = min(p, last);
                const uint32_t b1 = sslot[pc], b2 = sslot[pc + 1];
                const uint32_t e = smap[x & ((1u << lg) - 1u)];
                const uint32_t c = e >> 28;
                x = ((e >> 13) & 0x1fffu) * (x >> lg) + (e & 0x1fffu);
                const uint32_t k1 = x < kRansL ? 1u : 0u;
                x = k1 ? (x << 8) | b1 : x;
                const uint32_t k2 = x < kRansL ? 1u : 0u;
                x = k2 ? (x << 8) | b2 : x;
                overrun |= x < kRansL;
                p += k1 + k2;
                const uint32_t hi = __shfl_xor_sync(0xffffffffu, c, 1);
                if ((lane & 1) == 0) sout[16 * j + (lane >> 1)] = (uint8_t)(c | (hi << 4));
            }
        }
        __syncwarp();
        {
            uint4 *o4 = reinterpret_cast<uint4 *>(dst + (int64_t)bi * half);
            const uint4 *s4 = reinterpret_cast<const uint4 *>(sout);
            for (int i = lane; i < half / 16; i += 32) o4[i] = s4[i];
        }
    }
    // p beyond the end: the stream ran out; before it: bytes left over
    overrun = overrun || (!bad && p != end);
    if (__any_sync(0xffffffffu, bad || overrun) && lane == 0) atomicMax(status, (int32_t)KVQ_ERR_CORRUPT);
}

int entropy_init() {
    if (cudaFuncSetAttribute((const void *)entropy_encode_runs_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRunSmemMax) !=
            cudaSuccess ||
        cudaFuncSetAttribute((const void *)entropy_decode_runs_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRunSmemMax) !=
            cudaSuccess)
        return KVQ_ERR_CUDA;
    return KVQ_OK;
}

int launch_entropy_encode_runs(const uint8_t *codes, const kvq_layout &L, int nseg, uint8_t *out,
                               uint32_t *nbytes, cudaStream_t st) {
    const int64_t nb = num_blocks(L);
    if (nb == 0) return KVQ_OK;
    const int d = 32 * L.group;
    const int64_t nruns = (nb + nseg - 1) / nseg;
    entropy_encode_runs_kernel<<<(unsigned)nruns, 32, run_enc_smem(d, nseg), st>>>(codes, nb, d,
                                                                                 nseg, out, nbytes);
    return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

int launch_entropy_decode_runs(const uint8_t *in, const kvq_layout &L, int nseg, uint8_t *codes,
                               int32_t *status, cudaStream_t st) {
    const int64_t nb = num_blocks(L);
    if (cudaMemsetAsync(status, 0, sizeof(int32_t), st) != cudaSuccess) return KVQ_ERR_CUDA;
    if (nb == 0) return KVQ_OK;
    const int d = 32 * L.group;
    const int64_t nruns = (nb + nseg - 1) / nseg;
    entropy_decode_runs_kernel<<<(unsigned)nruns, 32, run_dec_smem(d, nseg), st>>>(in, nb, d, nseg,
                                                                                 codes, status);
    return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

size_t entropy_run_slot(const kvq_layout &L, int nseg) {
    return (size_t)run_slot_bytes(32 * L.group, nseg);
}
int entropy_run_max_blocks() { return kRunMaxBlocks; }

int launch_entropy_encode(const uint8_t *codes, const kvq_layout &L, uint8_t *out,
                          uint32_t *nbytes, cudaStream_t st) {
    const int64_t nb = num_blocks(L);
    if (nb == 0) return KVQ_OK;
    const int d = 32 * L.group;
    const int64_t ctas = (nb + kEntWarps - 1) / kEntWarps;
    entropy_encode_kernel<<<(unsigned)ctas, kEntWarps * 32, 0, st>>>(codes, nb, d, out, nbytes);
    return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

int launch_entropy_decode(const uint8_t *in, const kvq_layout &L, uint8_t *codes, int32_t *status,
                          cudaStream_t st) {
    const int64_t nb = num_blocks(L);
    if (cudaMemsetAsync(status, 0, sizeof(int32_t), st) != cudaSuccess) return KVQ_ERR_CUDA;
    if (nb == 0) return KVQ_OK;
    const int d = 32 * L.group;
    const int64_t ctas = (nb + kEntWarps - 1) / kEntWarps;
    entropy_decode_kernel<<<(unsigned)ctas, kEntWarps * 32, 0, st>>>(in, nb, d, codes, status);
    return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

size_t entropy_slot(const kvq_layout &L) { return entropy_slot_bytes(32 * L.group); }

}  // namespace kvq
