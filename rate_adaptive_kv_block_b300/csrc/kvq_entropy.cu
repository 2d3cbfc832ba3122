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
// per-lane scratch of the encoder: a symbol emits at most ceil(log2 d / 8)
// <= 2 bytes (the state stays below 2^31 and the bound is 2^(31 - log2 d) f),
// plus the 4-byte state
constexpr int kEntLaneCap = 2 * (4096 / 32) + 8;

__host__ __device__ constexpr uint32_t entropy_slot_bytes(int d) {
    // the payload is at most d * 4 bits (16 symbols) plus, per stream, the
    // state and one byte of renormalisation slack
    return (uint32_t)(d / 2 + kEntHeader + 32 * 6);
}

__device__ __forceinline__ int ilog2(int v) { return 31 - __clz(v); }

// symbol of slot s: the c with b_c <= s < b_{c+1} (cum[0] = 0, cum[16] = d;
// symbols with count 0 have b_c = b_{c+1} and are never found)
__device__ __forceinline__ int rans_symbol(const uint32_t (&cum)[17], uint32_t s) {
    int c = 0;
#pragma unroll
    for (int step = 8; step > 0; step >>= 1)
        if (cum[c + step] <= s) c += step;
    return c;
}

__global__ void __launch_bounds__(kEntWarps * 32)
entropy_encode_kernel(const uint8_t *__restrict__ codes, int64_t nb, int d,
                      uint8_t *__restrict__ out, uint32_t *__restrict__ nbytes) {
    __shared__ uint8_t scratch[kEntWarps][32][kEntLaneCap];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t b = (int64_t)blockIdx.x * kEntWarps + w;
    if (b >= nb) return;
    const int n = d / 32, lg = ilog2(d);
    const uint8_t *cb = codes + b * (d / 2);
    // the block's counts (lane-private, then a warp sum)
    uint32_t cnt[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) cnt[c] = 0;
    for (int j = 0; j < n; ++j) {
        const int e = lane + 32 * j;
        const uint32_t c = (cb[e >> 1] >> ((e & 1) * 4)) & 15u;
#pragma unroll
        for (int t = 0; t < 16; ++t) cnt[t] += (c == (uint32_t)t) ? 1u : 0u;
    }
#pragma unroll
    for (int t = 0; t < 16; ++t)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) cnt[t] += __shfl_xor_sync(0xffffffffu, cnt[t], o);
    uint32_t cum[17];
    cum[0] = 0;
#pragma unroll
    for (int t = 0; t < 16; ++t) cum[t + 1] = cum[t] + cnt[t];
    // this lane's stream, last entry first, bytes written downwards
    uint8_t *buf = scratch[w][lane];
    int pos = kEntLaneCap;
    uint32_t x = kRansL;
    for (int j = n - 1; j >= 0; --j) {
        const int e = lane + 32 * j;
        const int c = (cb[e >> 1] >> ((e & 1) * 4)) & 15;
        uint32_t f = 0, bc = 0;
#pragma unroll
        for (int t = 0; t < 16; ++t)
            if (t == c) { f = cnt[t]; bc = cum[t]; }
        const uint32_t xmax = ((kRansL >> lg) << 8) * f;
        while (x >= xmax) {
            buf[--pos] = (uint8_t)(x & 255u);
            x >>= 8;
        }
        x = ((x / f) << lg) + (x % f) + bc;
    }
    pos -= 4;
    buf[pos] = (uint8_t)x;
    buf[pos + 1] = (uint8_t)(x >> 8);
    buf[pos + 2] = (uint8_t)(x >> 16);
    buf[pos + 3] = (uint8_t)(x >> 24);
    const uint32_t len = (uint32_t)(kEntLaneCap - pos);
    // offsets of the streams (exclusive scan over the lanes)
    uint32_t off = len;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, off, o);
        if (lane >= o) off += y;
    }
    const uint32_t total = __shfl_sync(0xffffffffu, off, 31);
    off -= len;
    uint8_t *slot = out + b * (int64_t)entropy_slot_bytes(d);
    if (lane < 16) {
        slot[2 * lane] = (uint8_t)cnt[lane];
        slot[2 * lane + 1] = (uint8_t)(cnt[lane] >> 8);
    }
    slot[32 + 2 * lane] = (uint8_t)len;
    slot[32 + 2 * lane + 1] = (uint8_t)(len >> 8);
    for (uint32_t i = 0; i < len; ++i) slot[kEntHeader + off + i] = buf[pos + i];
    if (lane == 0) nbytes[b] = kEntHeader + total;
}

__global__ void __launch_bounds__(kEntWarps * 32)
entropy_decode_kernel(const uint8_t *__restrict__ in, int64_t nb, int d,
                      uint8_t *__restrict__ codes, int32_t *__restrict__ status) {
    __shared__ uint8_t sym[kEntWarps][4096];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t b = (int64_t)blockIdx.x * kEntWarps + w;
    if (b >= nb) return;
    const int n = d / 32, lg = ilog2(d);
    const uint32_t cap = entropy_slot_bytes(d);
    const uint8_t *slot = in + b * (int64_t)cap;
    uint32_t cnt[16], cum[17];
    cum[0] = 0;
#pragma unroll
    for (int t = 0; t < 16; ++t) {
        cnt[t] = (uint32_t)slot[2 * t] | ((uint32_t)slot[2 * t + 1] << 8);
        cum[t + 1] = cum[t] + cnt[t];
    }
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
    bool bad = cum[16] != (uint32_t)d || kEntHeader + total > cap || len < 4;
    bad = __any_sync(0xffffffffu, bad);
    uint32_t p = kEntHeader + off, end = p + len;
    uint32_t x = 0;
    if (!bad) {
        x = (uint32_t)slot[p] | ((uint32_t)slot[p + 1] << 8) | ((uint32_t)slot[p + 2] << 16) |
            ((uint32_t)slot[p + 3] << 24);
        p += 4;
    }
    bool overrun = false;
    for (int j = 0; j < n; ++j) {
        int c = 0;
        if (!bad) {
            const uint32_t s = x & ((1u << lg) - 1u);
            c = rans_symbol(cum, s);
            uint32_t f = 0, bc = 0;
#pragma unroll
            for (int t = 0; t < 16; ++t)
                if (t == c) { f = cnt[t]; bc = cum[t]; }
            x = f * (x >> lg) + s - bc;
            while (x < kRansL) {
                if (p >= end) { overrun = true; break; }   // never reads past its stream
                x = (x << 8) | slot[p++];
            }
        }
        sym[w][lane + 32 * j] = (uint8_t)c;
    }
    overrun |= !bad && p != end;
    if (__any_sync(0xffffffffu, bad || overrun) && lane == 0) atomicMax(status, (int32_t)KVQ_ERR_CORRUPT);
    __syncwarp();
    uint8_t *cout = codes + b * (d / 2);
    for (int i = lane; i < d / 2; i += 32)
        cout[i] = (uint8_t)(sym[w][2 * i] | (sym[w][2 * i + 1] << 4));
}

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
