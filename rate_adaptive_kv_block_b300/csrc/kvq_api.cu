// C ABI of libkvq (declared in include/kvq.h): argument validation on the
// host, then stream-ordered launches.  Nothing here allocates memory.
#include <math.h>
#include <string.h>

#include <mutex>

#include "kvq_internal.cuh"

namespace kvq {
int launch_stats(const uint16_t *x, const float *wt, const kvq_layout &L, void *stats,
                 int32_t *status, cudaStream_t st);
int launch_allocate(const void *stats, const kvq_layout &L, int s, double budget, int mode,
                    double eta, double *lambda, void *workspace, float *codebook, uint8_t *k,
                    float *Dr, float *Hr, double *totals, int32_t *status, cudaStream_t st,
                    const uint16_t *x = nullptr, uint64_t seed = 0, uint64_t index_base = 0,
                    uint8_t *codes = nullptr);
int launch_quantize(const uint16_t *x, const kvq_layout &L, const float *codebook,
                    const uint8_t *k, uint64_t seed, uint64_t index_base, uint8_t *codes,
                    int32_t *status, cudaStream_t st, bool nearest = false);
int launch_uniform_codebook(const uint16_t *x, const kvq_layout &L, float *codebook, uint8_t *k,
                            int32_t *status, cudaStream_t st);
int quantize_init();
int launch_dequantize(const uint8_t *codes, const float *codebook, const kvq_layout &L,
                      uint16_t *y, cudaStream_t st);
size_t workspace_bytes(int64_t nb, int s);
size_t attention_workspace_bytes(const kvq_layout &L, int n_rep);
int launch_decode_attention(const float *q, int n_rep, const kvq_layout &L, const uint8_t *kc,
                            const float *kcb, const uint8_t *vc, const float *vcb,
                            int64_t T_valid, float scale, void *workspace, float *out,
                            int32_t *status, cudaStream_t st);
int attention_init();
int launch_entropy_encode(const uint8_t *codes, const kvq_layout &L, uint8_t *out,
                          uint32_t *nbytes, cudaStream_t st);
int launch_entropy_decode(const uint8_t *in, const kvq_layout &L, uint8_t *codes, int32_t *status,
                          cudaStream_t st);
size_t entropy_slot(const kvq_layout &L);
int launch_entropy_encode_runs(const uint8_t *codes, const kvq_layout &L, int nseg, uint8_t *out,
                               uint32_t *nbytes, cudaStream_t st);
int launch_entropy_decode_runs(const uint8_t *in, const kvq_layout &L, int nseg, uint8_t *codes,
                               int32_t *status, cudaStream_t st);
size_t entropy_run_slot(const kvq_layout &L, int nseg);
int entropy_run_max_blocks();
int allocate_init();
int weights_init();
int entropy_init();
int allocate_report(const void *workspace, kvq_report *r);
void *static_workspace_address(int dev);
int launch_rate_sums(const void *stats, const kvq_layout &L, int s, const double *lambdas,
                     int nprobe, unsigned long long *sums, cudaStream_t st);
int stats_hi0(const void *stats, double *hi0);
int launch_fixed_rate(const void *stats, const kvq_layout &L, int s, double bits_per_entry,
                      float *codebook, uint8_t *k, float *Dr, float *Hr, double *lambdas,
                      double *totals, int32_t *status, cudaStream_t st);

static bool layout_ok(const kvq_layout &L) {
    if (L.S < 0 || L.T < 0 || L.T % 32 != 0) return false;
    const int G = L.group;
    if (!(G == 8 || G == 16 || G == 32 || G == 64 || G == 128)) return false;
    if (L.D <= 0 || L.D % G != 0 || L.D / G > 32) return false;
    if ((L.D & (L.D - 1)) != 0 || L.D > 2048) return false;   // power of two
    // element count must fit comfortably in 64-bit index arithmetic
    if (L.S > 0 && L.T > 0 && (double)L.S * (double)L.T * (double)L.D > 9.0e15) return false;
    return true;
}

static bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// Per-device one-time set-up (function attributes are per device), under a
// lock so that host threads making their first call at the same time do it
// once.  A failed set-up is not remembered: its error is cleared from the
// runtime's last-error slot, and the next call tries again.
static int init_once() {
    static std::mutex mu;
    static bool done[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return KVQ_ERR_CUDA;
    if (dev >= 64) return KVQ_ERR_CUDA;
    std::lock_guard<std::mutex> g(mu);
    if (done[dev]) return KVQ_OK;
    int st = allocate_init();
    if (st == KVQ_OK) st = quantize_init();
    if (st == KVQ_OK) st = attention_init();
    if (st == KVQ_OK) st = weights_init();
    if (st == KVQ_OK) st = entropy_init();
    if (st != KVQ_OK) {
        (void)cudaGetLastError();
        return st;
    }
    done[dev] = true;
    return KVQ_OK;
}

// kvq_encode_host's copy lanes: per device, kCopyLanes non-blocking streams
// that each take one piece of the host-to-device copy, so that several copy
// engines run at once (one engine moves about 28 GB/s from page-locked host
// memory on a B300 host, four about 44 GB/s); an event forks them from the
// caller's stream and one event per lane joins them back.  Created on the
// first call on the device, under the lock that also orders each call's
// record / wait sequence against other host threads.
constexpr int kCopyLanes = 4;
struct CopyLanes {
    cudaStream_t st[kCopyLanes];
    cudaEvent_t fork, join[kCopyLanes];
    bool ready;
};
static std::mutex g_lanes_mu;
static CopyLanes g_lanes[64];

static int lanes_ready(int dev) {
    CopyLanes &C = g_lanes[dev];
    if (C.ready) return KVQ_OK;
    bool ok = cudaEventCreateWithFlags(&C.fork, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < kCopyLanes; ++i) {
        ok = cudaStreamCreateWithFlags(&C.st[i], cudaStreamNonBlocking) == cudaSuccess &&
             cudaEventCreateWithFlags(&C.join[i], cudaEventDisableTiming) == cudaSuccess;
    }
    if (!ok) {
        (void)cudaGetLastError();
        return KVQ_ERR_CUDA;   // what was created stays, unused; the next call tries again
    }
    C.ready = true;
    return KVQ_OK;
}

// Copy `bytes` from host to device in up to kCopyLanes pieces (multiples of
// 64 KiB but the last), each on its own lane, ordered after and before the
// work of `st`.
static int copy_in_lanes(void *dst, const void *src, size_t bytes, cudaStream_t st) {
    if (bytes == 0) return KVQ_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KVQ_ERR_CUDA;
    std::lock_guard<std::mutex> g(g_lanes_mu);
    if (lanes_ready(dev) != KVQ_OK) return KVQ_ERR_CUDA;
    CopyLanes &C = g_lanes[dev];
    const size_t unit = (size_t)1 << 16;
    const size_t piece = ((bytes + kCopyLanes - 1) / kCopyLanes + unit - 1) / unit * unit;
    if (cudaEventRecord(C.fork, st) != cudaSuccess) return KVQ_ERR_CUDA;
    for (int i = 0; i < kCopyLanes; ++i) {
        const size_t off = (size_t)i * piece;
        if (off >= bytes) break;
        const size_t len = bytes - off < piece ? bytes - off : piece;
        if (cudaStreamWaitEvent(C.st[i], C.fork, 0) != cudaSuccess ||
            cudaMemcpyAsync(static_cast<char *>(dst) + off, static_cast<const char *>(src) + off,
                            len, cudaMemcpyHostToDevice, C.st[i]) != cudaSuccess ||
            cudaEventRecord(C.join[i], C.st[i]) != cudaSuccess ||
            cudaStreamWaitEvent(st, C.join[i], 0) != cudaSuccess)
            return KVQ_ERR_CUDA;
    }
    return KVQ_OK;
}
}  // namespace kvq

using namespace kvq;

extern "C" {

int64_t kvq_num_blocks(kvq_layout L) { return layout_ok(L) ? num_blocks(L) : -1; }

size_t kvq_stats_bytes(kvq_layout L) {
    return layout_ok(L) ? sizeof(StatsHeader) + (size_t)num_blocks(L) * kRecFloats * sizeof(float)
                        : 0;
}

size_t kvq_workspace_bytes(kvq_layout L, int s) {
    if (!layout_ok(L) || s < 2 || s > kMaxLev) return 0;
    return workspace_bytes(num_blocks(L), s);
}

int kvq_stats(const uint16_t *x, kvq_layout L, int m, void *stats, int32_t *status,
              void *stream) {
    if (!layout_ok(L) || m != kCand || !status) return KVQ_ERR_INVALID_ARG;
    const int64_t nb = num_blocks(L);
    if (nb > 0 && (!x || !stats || !aligned16(x) || !aligned16(stats))) return KVQ_ERR_INVALID_ARG;
    if (nb > 0x7fffffffll) return KVQ_ERR_INVALID_ARG;
    return launch_stats(x, nullptr, L, stats, status, static_cast<cudaStream_t>(stream));
}

int kvq_stats_weighted(const uint16_t *x, const float *w, kvq_layout L, int m, void *stats,
                       int32_t *status, void *stream) {
    if (!layout_ok(L) || m != kCand || !status) return KVQ_ERR_INVALID_ARG;
    const int64_t nb = num_blocks(L);
    if (nb > 0 && (!x || !w || !stats || !aligned16(x) || !aligned16(w) || !aligned16(stats)))
        return KVQ_ERR_INVALID_ARG;
    if (nb > 0x7fffffffll) return KVQ_ERR_INVALID_ARG;
    if (init_once() != KVQ_OK) return KVQ_ERR_CUDA;
    return launch_stats(x, w, L, stats, status, static_cast<cudaStream_t>(stream));
}

int kvq_allocate(const void *stats, kvq_layout L, int s, double budget_bits, int mode,
                 double eta, double *lambda, void *workspace, float *codebook, uint8_t *k,
                 float *D_r, float *H_r, double *totals, int32_t *status, void *stream) {
    if (!layout_ok(L) || s < 2 || s > kMaxLev) return KVQ_ERR_INVALID_ARG;
    if (!(budget_bits >= 0.0) || !isfinite(budget_bits)) return KVQ_ERR_INVALID_ARG;
    if (mode != KVQ_BISECT40 && mode != KVQ_SUBGRADIENT) return KVQ_ERR_INVALID_ARG;
    if (!(eta >= 0.0) || !isfinite(eta)) return KVQ_ERR_INVALID_ARG;
    if (!lambda || !totals || !status) return KVQ_ERR_INVALID_ARG;
    const int64_t nb = num_blocks(L);
    if (nb > 0) {
        if (!stats || !workspace || !codebook || !k || !D_r || !H_r) return KVQ_ERR_INVALID_ARG;
        if (!aligned16(stats) || !aligned16(workspace) || !aligned16(codebook))
            return KVQ_ERR_INVALID_ARG;
        if (nb > 0x7fffffffll) return KVQ_ERR_INVALID_ARG;
    }
    if (init_once() != KVQ_OK) return KVQ_ERR_CUDA;
    return launch_allocate(stats, L, s, budget_bits, mode, eta, lambda, workspace, codebook, k,
                           D_r, H_r, totals, status, static_cast<cudaStream_t>(stream));
}

int kvq_allocate_quantize(const void *stats, const uint16_t *x, kvq_layout L, int s,
                          double budget_bits, int mode, double eta, double *lambda,
                          void *workspace, float *codebook, uint8_t *k, float *D_r, float *H_r,
                          double *totals, uint64_t seed, uint64_t index_base, uint8_t *codes,
                          int32_t *status, void *stream) {
    if (!layout_ok(L) || s < 2 || s > kMaxLev) return KVQ_ERR_INVALID_ARG;
    if (!(budget_bits >= 0.0) || !isfinite(budget_bits)) return KVQ_ERR_INVALID_ARG;
    if (mode != KVQ_BISECT40 && mode != KVQ_SUBGRADIENT) return KVQ_ERR_INVALID_ARG;
    if (!(eta >= 0.0) || !isfinite(eta)) return KVQ_ERR_INVALID_ARG;
    if (!lambda || !totals || !status) return KVQ_ERR_INVALID_ARG;
    if (index_base & 3u) return KVQ_ERR_INVALID_ARG;
    const uint64_t n = (uint64_t)L.S * (uint64_t)L.T * (uint64_t)L.D;
    if (index_base > (1ull << 40) || n > (1ull << 40) - index_base) return KVQ_ERR_INVALID_ARG;
    const int64_t nb = num_blocks(L);
    if (nb > 0) {
        if (!stats || !x || !workspace || !codebook || !k || !D_r || !H_r || !codes)
            return KVQ_ERR_INVALID_ARG;
        if (!aligned16(stats) || !aligned16(x) || !aligned16(workspace) || !aligned16(codebook) ||
            !aligned16(codes))
            return KVQ_ERR_INVALID_ARG;
        if (nb > 0x7fffffffll) return KVQ_ERR_INVALID_ARG;
    }
    if (init_once() != KVQ_OK) return KVQ_ERR_CUDA;
    if (nb == 0)
        return launch_allocate(stats, L, s, budget_bits, mode, eta, lambda, workspace, codebook,
                               k, D_r, H_r, totals, status, static_cast<cudaStream_t>(stream));
    return launch_allocate(stats, L, s, budget_bits, mode, eta, lambda, workspace, codebook, k,
                           D_r, H_r, totals, status, static_cast<cudaStream_t>(stream), x, seed,
                           index_base, codes);
}

int kvq_allocate_static(const void *stats, kvq_layout L, int s, double budget_bits, int mode,
                        double eta, double *lambda, float *codebook, uint8_t *k, float *D_r,
                        float *H_r, double *totals, int32_t *status, void *stream) {
    if (!layout_ok(L) || s < 2 || s > kMaxLev) return KVQ_ERR_INVALID_ARG;
    if (workspace_bytes(num_blocks(L), s) > (size_t)KVQ_STATIC_WORKSPACE_BYTES)
        return KVQ_ERR_TOO_LARGE;
    // the per-device set-up (run by the first call of any entry point on the
    // device) loaded the module that holds the scratch and took its address
    if (init_once() != KVQ_OK) return KVQ_ERR_CUDA;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
    void *ws = static_workspace_address(dev);
    if (!ws) return KVQ_ERR_CUDA;
    // the control block at the start of the scratch is reset by the first
    // kernel of kvq_allocate; nothing else in it is read before it is written
    return kvq_allocate(stats, L, s, budget_bits, mode, eta, lambda, ws, codebook, k, D_r, H_r,
                        totals, status, stream);
}

int kvq_allocate_fixed_rate(const void *stats, kvq_layout L, int s, double bits_per_entry,
                            float *codebook, uint8_t *k, float *D_r, float *H_r,
                            double *lambda_r, double *totals, int32_t *status, void *stream) {
    if (!layout_ok(L) || s < 2 || s > kMaxLev) return KVQ_ERR_INVALID_ARG;
    if (!(bits_per_entry >= 0.0) || !isfinite(bits_per_entry)) return KVQ_ERR_INVALID_ARG;
    if (!totals || !status) return KVQ_ERR_INVALID_ARG;
    const int64_t nb = num_blocks(L);
    if (nb > 0) {
        if (!stats || !codebook || !k || !D_r || !H_r || !lambda_r) return KVQ_ERR_INVALID_ARG;
        if (!aligned16(stats) || !aligned16(codebook)) return KVQ_ERR_INVALID_ARG;
        if (nb > 0x7fffffffll) return KVQ_ERR_INVALID_ARG;
    }
    if (!stats) return KVQ_ERR_INVALID_ARG;
    if (init_once() != KVQ_OK) return KVQ_ERR_CUDA;
    return launch_fixed_rate(stats, L, s, bits_per_entry, codebook, k, D_r, H_r, lambda_r, totals,
                             status, static_cast<cudaStream_t>(stream));
}

size_t kvq_search_state_bytes(void) { return sizeof(SearchState); }

int kvq_search_begin(double hi0, double budget_bits, void *state) {
    if (!state || !(hi0 >= 0.0) || !isfinite(hi0)) return KVQ_ERR_INVALID_ARG;
    if (!(budget_bits >= 0.0) || !isfinite(budget_bits)) return KVQ_ERR_INVALID_ARG;
    SearchState s;
    search_init(s);
    s.hi0 = hi0;
    s.f32_lambda = 1;     // kvq_rate_sums evaluates the DP at float(lambda)
    memcpy(state, &s, sizeof(s));
    return KVQ_OK;
}

int kvq_search_probes(const void *state, double *lambdas) {
    if (!state || !lambdas) return -1;
    SearchState s;
    memcpy(&s, state, sizeof(s));
    if (s.phase == kSearchDone) return 0;
    for (int p = 0; p < s.nprobe; ++p) lambdas[p] = search_probe(s, p);
    return s.nprobe;
}

int kvq_search_advance(void *state, const int64_t *rate_sums, double budget_bits) {
    if (!state || !rate_sums) return KVQ_ERR_INVALID_ARG;
    if (!(budget_bits >= 0.0) || !isfinite(budget_bits)) return KVQ_ERR_INVALID_ARG;
    SearchState s;
    memcpy(&s, state, sizeof(s));
    if (s.phase == kSearchDone) return KVQ_OK;
    long long R[kSearchProbes];
    for (int p = 0; p < kSearchProbes; ++p) R[p] = p < s.nprobe ? (long long)rate_sums[p] : 0;
    search_update(s, R, budget_bits);
    memcpy(state, &s, sizeof(s));
    return KVQ_OK;
}

int kvq_search_result(const void *state, double *lambda, int32_t *rounds) {
    if (!state || !lambda) return KVQ_ERR_INVALID_ARG;
    SearchState s;
    memcpy(&s, state, sizeof(s));
    if (s.phase != kSearchDone) return KVQ_ERR_INVALID_ARG;
    *lambda = s.lambda;
    if (rounds) *rounds = s.rounds;
    return s.infeasible ? KVQ_ERR_INFEASIBLE : KVQ_OK;
}

int kvq_stats_hi0(const void *stats, double *hi0) {
    if (!stats || !hi0) return KVQ_ERR_INVALID_ARG;
    return stats_hi0(stats, hi0);
}

int kvq_rate_sums(const void *stats, kvq_layout L, int s, const double *lambdas, int nprobe,
                  int64_t *sums, void *stream) {
    if (!layout_ok(L) || s < 2 || s > kMaxLev) return KVQ_ERR_INVALID_ARG;
    if (nprobe < 0 || nprobe > kSearchProbes || (nprobe > 0 && !lambdas) || !sums)
        return KVQ_ERR_INVALID_ARG;
    for (int p = 0; p < nprobe; ++p)
        if (!(lambdas[p] >= 0.0) || !isfinite(lambdas[p])) return KVQ_ERR_INVALID_ARG;
    const int64_t nb = num_blocks(L);
    if (nb > 0 && (!stats || !aligned16(stats))) return KVQ_ERR_INVALID_ARG;
    if (nb > 0x7fffffffll) return KVQ_ERR_INVALID_ARG;
    if (init_once() != KVQ_OK) return KVQ_ERR_CUDA;
    return launch_rate_sums(stats, L, s, lambdas, nprobe,
                            reinterpret_cast<unsigned long long *>(sums),
                            static_cast<cudaStream_t>(stream));
}

int kvq_quantize(const uint16_t *x, kvq_layout L, const float *codebook, const uint8_t *k,
                 uint64_t seed, uint64_t index_base, uint8_t *codes, int32_t *status,
                 void *stream) {
    if (!layout_ok(L)) return KVQ_ERR_INVALID_ARG;
    if (index_base & 3u) return KVQ_ERR_INVALID_ARG;
    const uint64_t n = (uint64_t)L.S * (uint64_t)L.T * (uint64_t)L.D;
    if (index_base > (1ull << 40) || n > (1ull << 40) - index_base) return KVQ_ERR_INVALID_ARG;
    if (n > 0) {
        if (!x || !codebook || !k || !codes) return KVQ_ERR_INVALID_ARG;
        if (!aligned16(x) || !aligned16(codebook) || !aligned16(codes)) return KVQ_ERR_INVALID_ARG;
        if (L.S * (L.T / 32) > 0x7fffffffll) return KVQ_ERR_INVALID_ARG;
    }
    if (init_once() != KVQ_OK) return KVQ_ERR_CUDA;
    return launch_quantize(x, L, codebook, k, seed, index_base, codes, status,
                           static_cast<cudaStream_t>(stream));
}

int kvq_uniform_codebook(const uint16_t *x, kvq_layout L, float *codebook, uint8_t *k,
                         int32_t *status, void *stream) {
    if (!layout_ok(L)) return KVQ_ERR_INVALID_ARG;
    const int64_t nb = num_blocks(L);
    if (nb > 0) {
        if (!x || !codebook || !k || !status) return KVQ_ERR_INVALID_ARG;
        if (!aligned16(x) || !aligned16(codebook)) return KVQ_ERR_INVALID_ARG;
    }
    return launch_uniform_codebook(x, L, codebook, k, status, static_cast<cudaStream_t>(stream));
}

int kvq_quantize_nearest(const uint16_t *x, kvq_layout L, const float *codebook, const uint8_t *k,
                         uint8_t *codes, int32_t *status, void *stream) {
    if (!layout_ok(L)) return KVQ_ERR_INVALID_ARG;
    const int64_t nb = num_blocks(L);
    if (nb > 0) {
        if (!x || !codebook || !k || !codes) return KVQ_ERR_INVALID_ARG;
        if (!aligned16(x) || !aligned16(codebook) || !aligned16(codes)) return KVQ_ERR_INVALID_ARG;
        if (L.S * (L.T / 32) > 0x7fffffffll) return KVQ_ERR_INVALID_ARG;
    }
    if (init_once() != KVQ_OK) return KVQ_ERR_CUDA;
    return launch_quantize(x, L, codebook, k, 0, 0, codes, status,
                           static_cast<cudaStream_t>(stream), true);
}

int kvq_dequantize(const uint8_t *codes, const float *codebook, kvq_layout L, uint16_t *y,
                   void *stream) {
    if (!layout_ok(L)) return KVQ_ERR_INVALID_ARG;
    const int64_t nb = num_blocks(L);
    if (nb > 0) {
        if (!codes || !codebook || !y) return KVQ_ERR_INVALID_ARG;
        if (!aligned16(codes) || !aligned16(codebook) || !aligned16(y)) return KVQ_ERR_INVALID_ARG;
        if (L.S * (L.T / 32) > 0x7fffffffll) return KVQ_ERR_INVALID_ARG;
    }
    return launch_dequantize(codes, codebook, L, y, static_cast<cudaStream_t>(stream));
}

size_t kvq_entropy_slot_bytes(kvq_layout L) {
    if (!layout_ok(L)) return 0;
    return entropy_slot(L);
}

int kvq_entropy_encode(const uint8_t *codes, kvq_layout L, uint8_t *out, uint32_t *nbytes,
                       void *stream) {
    if (!layout_ok(L)) return KVQ_ERR_INVALID_ARG;
    if (num_blocks(L) > 0 && (!codes || !out || !nbytes || !aligned16(codes) || !aligned16(out)))
        return KVQ_ERR_INVALID_ARG;
    return launch_entropy_encode(codes, L, out, nbytes, static_cast<cudaStream_t>(stream));
}

int kvq_entropy_decode(const uint8_t *in, kvq_layout L, uint8_t *codes, int32_t *status,
                       void *stream) {
    if (!layout_ok(L)) return KVQ_ERR_INVALID_ARG;
    if (!status || (num_blocks(L) > 0 && (!in || !codes || !aligned16(in) || !aligned16(codes))))
        return KVQ_ERR_INVALID_ARG;
    return launch_entropy_decode(in, L, codes, status, static_cast<cudaStream_t>(stream));
}

static bool runs_ok(const kvq_layout &L, int nseg) {
    return layout_ok(L) && nseg >= 1 && nseg <= entropy_run_max_blocks();
}

size_t kvq_entropy_run_bytes(kvq_layout L, int nseg) {
    return runs_ok(L, nseg) ? entropy_run_slot(L, nseg) : 0;
}

int kvq_entropy_encode_runs(const uint8_t *codes, kvq_layout L, int nseg, uint8_t *out,
                            uint32_t *nbytes, void *stream) {
    if (!runs_ok(L, nseg)) return KVQ_ERR_INVALID_ARG;
    if (num_blocks(L) > 0 && (!codes || !out || !nbytes || !aligned16(codes) || !aligned16(out)))
        return KVQ_ERR_INVALID_ARG;
    if (init_once() != KVQ_OK) return KVQ_ERR_CUDA;
    return launch_entropy_encode_runs(codes, L, nseg, out, nbytes,
                                      static_cast<cudaStream_t>(stream));
}

int kvq_entropy_decode_runs(const uint8_t *in, kvq_layout L, int nseg, uint8_t *codes,
                            int32_t *status, void *stream) {
    if (!runs_ok(L, nseg) || !status) return KVQ_ERR_INVALID_ARG;
    if (num_blocks(L) > 0 && (!in || !codes || !aligned16(in) || !aligned16(codes)))
        return KVQ_ERR_INVALID_ARG;
    if (init_once() != KVQ_OK) return KVQ_ERR_CUDA;
    return launch_entropy_decode_runs(in, L, nseg, codes, status,
                                      static_cast<cudaStream_t>(stream));
}

static bool attention_layout_ok(const kvq_layout &L, int n_rep) {
    return layout_ok(L) && L.D == 128 && (n_rep == 1 || n_rep == 2 || n_rep == 4) &&
           L.S <= 65535 && L.S * n_rep <= 0x7fffffffll;
}

size_t kvq_attention_workspace_bytes(kvq_layout L, int n_rep) {
    if (!attention_layout_ok(L, n_rep)) return 0;
    return attention_workspace_bytes(L, n_rep);
}

int kvq_decode_attention(const float *q, int n_rep, kvq_layout L, const uint8_t *k_codes,
                         const float *k_codebook, const uint8_t *v_codes,
                         const float *v_codebook, int64_t T_valid, float scale, void *workspace,
                         float *out, int32_t *status, void *stream) {
    if (!attention_layout_ok(L, n_rep)) return KVQ_ERR_INVALID_ARG;
    if (T_valid < 0 || T_valid > L.T || !(scale == scale) || isinf(scale)) return KVQ_ERR_INVALID_ARG;
    if (L.S == 0) return KVQ_OK;
    if (!q || !out || !workspace) return KVQ_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out) || !aligned16(workspace)) return KVQ_ERR_INVALID_ARG;
    if (T_valid > 0) {
        if (!k_codes || !k_codebook || !v_codes || !v_codebook) return KVQ_ERR_INVALID_ARG;
        if (!aligned16(k_codes) || !aligned16(k_codebook) || !aligned16(v_codes) ||
            !aligned16(v_codebook))
            return KVQ_ERR_INVALID_ARG;
    }
    if (init_once() != KVQ_OK) return KVQ_ERR_CUDA;
    return launch_decode_attention(q, n_rep, L, k_codes, k_codebook, v_codes, v_codebook, T_valid,
                                   scale, workspace, out, status,
                                   static_cast<cudaStream_t>(stream));
}

int kvq_encode_host(const uint16_t *x_host, kvq_layout L, int s, double budget_bits,
                    uint64_t seed, uint64_t index_base, uint16_t *x_dev, void *stats,
                    double *lambda, void *workspace, float *codebook, uint8_t *k, float *D_r,
                    float *H_r, double *totals, uint8_t *codes, int32_t *status,
                    uint8_t *codes_host, float *codebook_host, uint8_t *k_host,
                    double *totals_host, void *stream) {
    // every argument of the three calls is checked before anything is issued
    if (!layout_ok(L) || s < 2 || s > kMaxLev) return KVQ_ERR_INVALID_ARG;
    if (!(budget_bits >= 0.0) || !isfinite(budget_bits)) return KVQ_ERR_INVALID_ARG;
    if (!lambda || !totals || !status) return KVQ_ERR_INVALID_ARG;
    if (index_base & 3u) return KVQ_ERR_INVALID_ARG;
    const uint64_t n = (uint64_t)L.S * (uint64_t)L.T * (uint64_t)L.D;
    if (index_base > (1ull << 40) || n > (1ull << 40) - index_base) return KVQ_ERR_INVALID_ARG;
    const int64_t nb = num_blocks(L);
    if (nb > 0) {
        if (!x_host || !x_dev || !stats || !workspace || !codebook || !k || !D_r || !H_r || !codes)
            return KVQ_ERR_INVALID_ARG;
        if (!aligned16(x_dev) || !aligned16(stats) || !aligned16(workspace) ||
            !aligned16(codebook) || !aligned16(codes))
            return KVQ_ERR_INVALID_ARG;
        if (nb > 0x7fffffffll) return KVQ_ERR_INVALID_ARG;
    }
    if (init_once() != KVQ_OK) return KVQ_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int rc = copy_in_lanes(x_dev, x_host, (size_t)n * sizeof(uint16_t), st);
    if (rc == KVQ_OK) rc = kvq_stats(x_dev, L, kCand, stats, status, stream);
    if (rc == KVQ_OK)
        rc = kvq_allocate(stats, L, s, budget_bits, KVQ_BISECT40, 0.0, lambda, workspace, codebook,
                          k, D_r, H_r, totals, status + 1, stream);
    // kvq_quantize writes its status only when a copy times out
    if (rc == KVQ_OK && cudaMemsetAsync(status + 2, 0, sizeof(int32_t), st) != cudaSuccess)
        rc = KVQ_ERR_CUDA;
    if (rc == KVQ_OK)
        rc = kvq_quantize(x_dev, L, codebook, k, seed, index_base, codes, status + 2, stream);
    if (rc != KVQ_OK) return rc;
    // what a cache stores, and the totals, back to the host
    struct { void *dst; const void *src; size_t bytes; } out[4] = {
        {codes_host, codes, (size_t)nb * 16 * (size_t)L.group},
        {codebook_host, codebook, (size_t)nb * 16 * sizeof(float)},
        {k_host, k, (size_t)nb},
        {totals_host, totals, 3 * sizeof(double)},
    };
    for (const auto &o : out)
        if (o.dst && o.bytes &&
            cudaMemcpyAsync(o.dst, o.src, o.bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
            return KVQ_ERR_CUDA;
    return KVQ_OK;
}

int kvq_allocate_report(const void *workspace, kvq_report *report) {
    if (!workspace || !report) return KVQ_ERR_INVALID_ARG;
    return allocate_report(workspace, report);
}

const char *kvq_status_string(int status) {
    switch (status) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_CUDA: return "CUDA launch error";
    case KVQ_ERR_NONFINITE: return "non-finite input entry";
    case KVQ_ERR_INFEASIBLE: return "budget infeasible";
    case KVQ_ERR_TIMEOUT: return "device wait timed out";
    case KVQ_ERR_TOO_LARGE: return "layout needs more scratch than the static workspace holds";
    case KVQ_ERR_CORRUPT: return "malformed entropy-coded slot";
    case KVQ_ERR_BAD_WEIGHT: return "negative or non-finite distortion weight";
    default: return "unknown status";
    }
}

}  // extern "C"
