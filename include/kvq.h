/*
 * kvq.h -- C ABI of the B300 (sm_103a) write-time KV-cache quantizer.
 *
 * What it computes ("Rate-adaptive KV-cache quantizer", synthcore idea 2502):
 * the cache is cut into blocks (one attention head x 32 tokens, or one head x
 * 32 tokens x a feature group -- "Implementation notes"); every block r of
 * d_r entries gets its own codebook Q_r of k <= s levels, chosen to minimise
 * D_r + lambda d_r H_r ("Mathematical statement", "Key formulas": the
 * Lagrangian), where D_r is the expected squared error of unbiased
 * stochastic interpolation between neighbouring levels and H_r the entropy
 * of the expected codepoint frequencies; one global lambda makes
 * sum_r d_r H_r <= B.  The entries are then rounded at random to one of their
 * two neighbouring levels with the unbiased probabilities of "Key formulas"
 * and stored as 4-bit codes plus a per-block fp32 codebook.
 *
 * Call sequence (all on one CUDA stream, asynchronous, no host sync inside):
 *     kvq_stats      -> per-block candidate levels and interval statistics
 *                       (kvq_stats_weighted: the same, distortion weighted
 *                       per entry by the caller's sensitivities)
 *     kvq_allocate   -> lambda, per-block codebook / k / D_r / H_r
 *     kvq_quantize   -> packed codes
 *     kvq_dequantize -> binary16 reconstruction ("decode before attention")
 *     kvq_decode_attention -> attention of a decoding step read from the codes
 *
 * Conventions for every entry point:
 *   - Pointers named "device" are CUDA device memory owned by the caller; the
 *     library allocates nothing and keeps no pointer after the call returns.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).
 *   - Return value: KVQ_OK, KVQ_ERR_INVALID_ARG (arguments rejected on the
 *     host before anything is launched; nothing is written) or KVQ_ERR_CUDA
 *     (a launch failed).  Conditions that depend on the data (non-finite
 *     inputs, an infeasible budget) are written by the kernels to the
 *     caller's device `status` word; read it after synchronising.
 *   - Device buffers must be 16-byte aligned.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define KVQ_OK 0
#define KVQ_ERR_INVALID_ARG 1
#define KVQ_ERR_CUDA 2
#define KVQ_ERR_NONFINITE 3   /* device status: a block holds NaN or +-Inf */
#define KVQ_ERR_INFEASIBLE 4  /* device status: budget unreachable         */
#define KVQ_ERR_TOO_LARGE 5   /* kvq_allocate_static: layout over its limit  */
#define KVQ_ERR_TIMEOUT 6     /* device status: a grid-wide wait gave up     */
#define KVQ_ERR_CORRUPT 7     /* device status: an entropy-coded slot is malformed */
#define KVQ_ERR_BAD_WEIGHT 8  /* device status: a distortion weight is < 0, NaN or +-Inf */

/* lambda modes of kvq_allocate */
#define KVQ_BISECT40 0        /* global lambda by the 40-step bisection      */
#define KVQ_SUBGRADIENT 1     /* one subgradient step from a given lambda    */

#define KVQ_CANDIDATES 17     /* order-statistic candidate levels per block  */
#define KVQ_MAX_LEVELS 16     /* codes are 4 bits                            */

/*
 * Shape of one K or V tensor: [S, T, D] row-major binary16, S streams (layer
 * x K/V x head, or any other flattening), T tokens per stream, D features.
 * A block is 32 consecutive tokens x `group` consecutive features of one
 * stream; d = 32 * group entries.  Blocks are numbered row-major over
 * (stream, token block, feature group); inside a block entry e is
 * (token - 32 * token_block) * group + (feature - group_index * group).
 * Requirements: S >= 0, T >= 0 and T % 32 == 0, group in {8,16,32,64,128},
 * D a power of two <= 2048, D % group == 0, D / group <= 32.
 */
typedef struct kvq_layout {
    int64_t S;
    int64_t T;
    int32_t D;
    int32_t group;
} kvq_layout;

/* Number of blocks S * (T/32) * (D/group); -1 if the layout is invalid. */
int64_t kvq_num_blocks(kvq_layout L);

/* Bytes of the statistics buffer written by kvq_stats (256 + 4800 bytes per
 * block); 0 if the layout is invalid. */
size_t kvq_stats_bytes(kvq_layout L);

/* Bytes of device scratch that kvq_allocate needs for this layout and s; 0
 * if the arguments are invalid. */
size_t kvq_workspace_bytes(kvq_layout L, int s);

/*
 * kvq_stats -- candidate alphabet and interval statistics of every block
 * ("Implementation notes": build a candidate alphabet from the block's
 * minimum, maximum and quantiles; compute D_r from interval statistics).
 *   x       device, [S,T,D] binary16 (read once).
 *   m       number of candidates; must be KVQ_CANDIDATES (17): the order
 *           statistics at 0-based sorted ranks floor((j(d-1)+8)/16),
 *           j = 0..16 (minimum and maximum included), equal values merged.
 *   stats   device, kvq_stats_bytes(L) bytes, written: per block the merged
 *           candidates, for each gap between consecutive candidates the count
 *           and first moments of the entries in it, and the block's
 *           lambda-independent interval distortions and entropy terms.  Its
 *           layout is private to this library; pass it to kvq_allocate
 *           unchanged.
 *   status  device int32, set to KVQ_OK, or KVQ_ERR_NONFINITE if any entry is
 *           NaN or infinite (the results of such blocks are unspecified).
 */
int kvq_stats(const uint16_t *x, kvq_layout L, int m, void *stats,
              int32_t *status, void *stream);

/*
 * kvq_stats_weighted -- kvq_stats with the distortion weighted per entry
 * ("Implementation notes": optionally weight D_r by the attention
 * sensitivity measured on a calibration batch).  The block distortion
 * becomes D_r = sum_e w_e E[(hat x_e - x_e)^2] = sum_e w_e (q_hi - x_e)(x_e -
 * q_lo); the candidates and the entropy H_r (expected frequencies of the
 * stored symbols) are those of kvq_stats.  kvq_allocate then minimises
 * sum_r D_r subject to sum_r d_r H_r <= B with the weighted D_r, and reports
 * the weighted D_r and sum_r D_r; its bisection starts from
 * hi = max_r (c_max - c_min)^2 w_max,r (w_max,r the block's largest weight).
 *   x       device, [S,T,D] binary16, as kvq_stats.
 *   w       device, [S,T,D] float32 in the layout of x (read once): w_e >= 0.
 *           Sensitivities that depend only on the feature (keys: the mean
 *           squared query component) or only on the token (values: the
 *           mean squared attention probability) are passed broadcast.
 *   m, stats as kvq_stats (the stats rows hold the weighted atom moments).
 *   status  device int32: KVQ_OK; KVQ_ERR_BAD_WEIGHT if a weight is negative,
 *           NaN or infinite (it is counted as 0; such blocks' results are
 *           unspecified), else KVQ_ERR_NONFINITE if an entry of x is.
 * The per-atom weighted sums are formed in a fixed order: repeated calls give
 * identical bits.
 */
int kvq_stats_weighted(const uint16_t *x, const float *w, kvq_layout L, int m,
                       void *stats, int32_t *status, void *stream);

/*
 * kvq_allocate -- per-block codebooks and the global lambda ("Mathematical
 * statement": minimise sum_r D_r subject to sum_r d_r H_r <= B, |Q_r| <= s;
 * with lambda the blocks decouple into argmin_Q D_r + lambda d_r H_r).
 * Every block gets the exact minimiser over all subsets of its candidates
 * that contain the minimum and the maximum and have 2 <= k <= s levels
 * (k = 1 for a constant block).  Reads only `stats` (never x again).
 *   s            2..16, maximum levels per block.
 *   budget_bits  B, in bits, for the whole tensor (e.g. 2.5 * S*T*D); >= 0.
 *   mode         KVQ_BISECT40: R(0) <= B gives lambda = 0; else
 *                hi = max_r (c_max - c_min)^2, doubled (at most 30 times)
 *                until R(hi) <= B, then 40 bisection steps on [0, hi];
 *                lambda = the feasible end.  If R stays above B the
 *                allocation at the last hi is returned and the status is
 *                KVQ_ERR_INFEASIBLE.
 *                KVQ_SUBGRADIENT ("Key formulas": lambda <- max{0, lambda +
 *                eta (sum_r d_r H_r - B)}): the choice is made at the given
 *                lambda; on return *lambda holds the updated value.
 *   eta          step of KVQ_SUBGRADIENT (ignored by KVQ_BISECT40); >= 0.
 *   lambda       device double; KVQ_SUBGRADIENT: in = lambda_t, out =
 *                lambda_{t+1}; KVQ_BISECT40: out = lambda.
 *   workspace    device, kvq_workspace_bytes(L, s) bytes of scratch.
 *   codebook     device float [nblocks][16]: levels in increasing order,
 *                slots k..15 repeat the largest level.
 *   k            device uint8 [nblocks]: number of levels.
 *   D_r          device float [nblocks]: expected squared error of the block.
 *   H_r          device float [nblocks]: entropy (bits per entry) of the
 *                expected codepoint frequencies.
 *   totals       device double [3]: sum_r d_r H_r, sum_r D_r, and the lambda
 *                the codebooks were chosen at.
 *   status       device int32: KVQ_OK, KVQ_ERR_INFEASIBLE, KVQ_ERR_NONFINITE,
 *                or KVQ_ERR_BAD_WEIGHT (stats from kvq_stats_weighted), the
 *                last outranking the others.
 */
int kvq_allocate(const void *stats, kvq_layout L, int s, double budget_bits,
                 int mode, double eta, double *lambda, void *workspace,
                 float *codebook, uint8_t *k, float *D_r, float *H_r,
                 double *totals, int32_t *status, void *stream);

/*
 * kvq_allocate_static -- kvq_allocate without a caller-provided workspace.
 * The method's page has no counterpart: this is a convenience for callers
 * that must not allocate device memory at the point of the call -- code that
 * runs inside a caching allocator's own hooks, a memory-capped serving
 * process whose pool is fully reserved, or a C caller with no allocator at
 * all.  Arguments, results and statuses are those of kvq_allocate.
 *
 * The scratch is a fixed array of KVQ_STATIC_WORKSPACE_BYTES (8 MiB) in the
 * library's device memory, in the same module as the search kernel.  It holds
 * layouts whose kvq_workspace_bytes(L, s) is at most that size (about 29 400
 * blocks: 7.5 million entries with group 8, 120 million with group 128);
 * larger layouts return KVQ_ERR_TOO_LARGE without launching anything.
 * The call itself allocates nothing, but the array exists on a device only
 * once the CUDA runtime has loaded that module there (with the default lazy
 * module loading: at the library's per-device set-up, run by the first call
 * on the device of kvq_allocate, kvq_allocate_static, kvq_allocate_quantize,
 * kvq_quantize, kvq_quantize_nearest, kvq_stats_weighted or
 * kvq_decode_attention).  That set-up also looks up the array's device
 * address (cudaGetSymbolAddress) and sets kernel attributes, so make the
 * first such call on each device at start-up, while device memory is still
 * free, and outside any stream capture; from then on the array stays until
 * the process exits.  A set-up that fails returns KVQ_ERR_CUDA, clears the
 * runtime error, and is tried again by the next call.
 * Every call on a device shares the one array, so calls that can overlap in
 * time (different streams, different host threads without a dependency
 * between them) race on it and corrupt each other's results; serialise them.
 */
#define KVQ_STATIC_WORKSPACE_BYTES (8u << 20)
int kvq_allocate_static(const void *stats, kvq_layout L, int s, double budget_bits,
                        int mode, double eta, double *lambda, float *codebook,
                        uint8_t *k, float *D_r, float *H_r, double *totals,
                        int32_t *status, void *stream);

/*
 * kvq_allocate_quantize -- kvq_allocate followed by kvq_quantize in one
 * launch, with the same results bit for bit (codebook, k, D_r, H_r, totals,
 * lambda, status; codes as kvq_quantize writes them for this seed and
 * index_base).  A block whose rate is equal at both ends of the search's
 * window is constant inside it, so its codebook is already final: such
 * blocks are emitted and quantized while the last rounds of the lambda
 * search run, by warps the search leaves idle.  Arguments as for
 * kvq_allocate and kvq_quantize (x is read again; the workspace is
 * kvq_workspace_bytes(L, s)); a timed-out copy or wait is reported in
 * `status` as KVQ_ERR_TIMEOUT.
 */
int kvq_allocate_quantize(const void *stats, const uint16_t *x, kvq_layout L, int s,
                          double budget_bits, int mode, double eta, double *lambda,
                          void *workspace, float *codebook, uint8_t *k, float *D_r,
                          float *H_r, double *totals, uint64_t seed,
                          uint64_t index_base, uint8_t *codes, int32_t *status,
                          void *stream);

/*
 * kvq_allocate_fixed_rate -- the fixed-rate comparator ("Implementation
 * notes": compare against fixed-rate entropy coding at equal total cache
 * bytes).  The same per-block quantizer as kvq_allocate, but every block r
 * meets the rate on its own: lambda_r comes from the 40-step bisection of
 * kvq_allocate applied to block r alone with the budget bits_per_entry * d_r
 * (R_r(0) <= budget -> 0; bracket from (c_max - c_min)^2 doubled at most 30
 * times; lambda_r = the bracket's feasible end), and the block gets its
 * choice at the smallest feasible lambda evaluated.  The total rate is then
 * at most bits_per_entry * S*T*D, the budget kvq_allocate spreads across
 * blocks with one lambda.
 *   stats        kvq_stats output (unweighted: weighted stats set status to
 *                KVQ_ERR_INVALID_ARG).
 *   codebook, k, D_r, H_r  as for kvq_allocate; lambda_r  device double
 *                [nblocks], each block's lambda.
 *   totals       device double[3]: sum d_r H_r, sum D_r, 0 (fixed order).
 *   status       device int32: KVQ_OK, KVQ_ERR_INFEASIBLE (some block cannot
 *                reach its budget; it keeps the choice at the largest bracket),
 *                KVQ_ERR_NONFINITE, KVQ_ERR_INVALID_ARG (weighted stats).
 */
int kvq_allocate_fixed_rate(const void *stats, kvq_layout L, int s,
                            double bits_per_entry, float *codebook, uint8_t *k,
                            float *D_r, float *H_r, double *lambda_r,
                            double *totals, int32_t *status, void *stream);

/*
 * kvq_quantize -- unbiased stochastic interpolation and 4-bit packing ("Key
 * formulas": P(q_{i+1} | x) = (x - q_i)/(q_{i+1} - q_i)).  For entry x of
 * block r with levels q_0 < ... < q_{k-1}: i = the largest index with
 * q_i <= x, capped at k-2; u = hash(seed, index_base + flat index) >> 8; the
 * code is i+1 iff fl(u 2^-24 * (q_{i+1} - q_i)) < fl(x - q_i) in fp32
 * round-to-nearest (no fused multiply-add), else i; k = 1 gives code 0.
 * hash(seed, n) is word n mod 4 of the Philox4x32 block function with 7
 * rounds (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
 * 1, 2, 3", SC 2011) at counter (n >> 2 as two 32-bit words, 0, 0) and key
 * (seed as two 32-bit words).
 *   x           device [S,T,D] binary16.
 *   codebook, k as written by kvq_allocate (k must be the number of distinct
 *               levels, with slots k..15 repeating the largest: the kernel
 *               takes k from the codebook itself).
 *   seed        any 64-bit value.
 *   index_base  a multiple of 4, and index_base + S*T*D <= 2^40.
 *   codes       device uint8 [nblocks][16*group]: byte e/2 of block r holds
 *               entry e in its low nibble (e even) or high nibble (e odd).
 *   status      device int32 or NULL: set to KVQ_ERR_TIMEOUT if a copy into
 *               shared memory never completed (the codes are then
 *               incomplete); left unchanged otherwise.
 */
int kvq_quantize(const uint16_t *x, kvq_layout L, const float *codebook,
                 const uint8_t *k, uint64_t seed, uint64_t index_base,
                 uint8_t *codes, int32_t *status, void *stream);

/*
 * kvq_dequantize -- decode before attention ("Implementation notes"):
 * y = codebook[r][code] written as binary16 (exact: every level is a
 * binary16 value of the block).
 *   codes, codebook  as above; y  device [S,T,D] binary16, written.
 */
int kvq_dequantize(const uint8_t *codes, const float *codebook, kvq_layout L,
                   uint16_t *y, void *stream);

/*
 * kvq_encode_host -- the whole write path for a tensor held in host memory:
 * the copy in, kvq_stats, kvq_allocate (KVQ_BISECT40), kvq_quantize, and the
 * copy out of what a cache stores (codes, codebook, k) and of the totals.
 * The method's page describes the computation on the device; this is the
 * call a serving loop makes when the new keys or values are staged in host
 * memory.
 *   x_host      host [S,T,D] binary16; page-locked (cudaHostAlloc or
 *               cudaHostRegister) for the call to be asynchronous -- it is
 *               read until the stream has passed the copy in.
 *   x_dev       device [S,T,D] binary16: where the input is copied.
 *   stats, lambda, workspace, codebook, k, D_r, H_r, totals
 *               device, as kvq_stats / kvq_allocate (s, budget_bits too).
 *   seed, index_base, codes   as kvq_quantize.
 *   status      device int32 [3]: the status words of the stats, the
 *               allocation and the quantization, in that order (the last is
 *               set to KVQ_OK first, then to KVQ_ERR_TIMEOUT if a copy into
 *               shared memory never completed).
 *   codes_host, codebook_host, k_host, totals_host
 *               host (page-locked, as x_host), each written with its device
 *               counterpart, or NULL to skip that copy.
 *   stream      everything is ordered on `stream` and asynchronous; the host
 *               outputs are valid once the stream has reached the end of the
 *               call.  The copy in is split into up to 4 pieces, each on one
 *               of the library's own copy streams (created per device by the
 *               first call, which should therefore be made outside any
 *               stream capture): they start after the work already queued on
 *               `stream`, and `stream` waits for all of them, so several copy
 *               engines move the input at once.
 * Every argument is checked before anything is issued; KVQ_ERR_CUDA if the
 * runtime refused a copy or a launch.
 */
int kvq_encode_host(const uint16_t *x_host, kvq_layout L, int s, double budget_bits,
                    uint64_t seed, uint64_t index_base, uint16_t *x_dev, void *stats,
                    double *lambda, void *workspace, float *codebook, uint8_t *k, float *D_r,
                    float *H_r, double *totals, uint8_t *codes, int32_t *status,
                    uint8_t *codes_host, float *codebook_host, uint8_t *k_host,
                    double *totals_host, void *stream);

/*
 * kvq_uniform_codebook -- codebooks of the uniform comparator ("Implementation
 * notes": compare uniform INT4 and uniform stochastic quantization at equal
 * cache bytes): per block, from its minimum m and maximum M,
 *     delta = fl32(fl32(M - m) / 15),  level_j = binary16(fl32(m + fl32(j delta)))
 * for j = 0..14 and level_15 = M (fp32 round-to-nearest, no contraction),
 * repeats removed: k distinct levels in codebook slots 0..k-1, slots k..15
 * repeat the top.  kvq_quantize with these codebooks is uniform stochastic
 * quantization; kvq_quantize_nearest with them is uniform INT4.
 *   x         device [S,T,D] binary16, read.
 *   codebook  device fp32 [nblocks][16], written.
 *   k         device u8 [nblocks], written.
 *   status    device int32, written: KVQ_OK, or KVQ_ERR_NONFINITE if a block
 *             holds NaN or +-Inf (its codebook is then unspecified).
 */
int kvq_uniform_codebook(const uint16_t *x, kvq_layout L, float *codebook, uint8_t *k,
                         int32_t *status, void *stream);

/*
 * kvq_quantize_nearest -- deterministic rounding to the nearest level of any
 * codebook in the format above (the INT4 comparator with kvq_uniform_codebook):
 * i = the largest index with q_i <= x (capped at k-2), code = i + [w < 2 r]
 * with w = fl32(q_{i+1} - q_i), r = fl32(x - q_i) (a tie keeps the lower level);
 * k = 1: code 0.  Codes packed as kvq_quantize's.  Arguments as kvq_quantize's
 * without seed and index_base.
 */
int kvq_quantize_nearest(const uint16_t *x, kvq_layout L, const float *codebook, const uint8_t *k,
                         uint8_t *codes, int32_t *status, void *stream);

/*
 * Entropy coding of the symbol stream ("Implementation notes": store the
 * codebook, symbol stream and block lengths, arithmetic coding of the
 * symbols): every block's 4-bit codes as 32 interleaved rANS streams (32-bit
 * state, byte renormalisation, L = 2^23) modelled by the block's exact symbol
 * counts (total d = 32 * group, a power of two), in a slot of fixed capacity
 * kvq_entropy_slot_bytes(L) = d/2 + 288 bytes:
 *   [0, 32)   16 x u16 little-endian: count of each symbol
 *   [32, 96)  32 x u16: bytes of stream l (entries l, l+32, .. of the block)
 *   [96, ..)  the streams in order; each = the encoder's final state (4
 *             bytes, little-endian), then its renormalisation bytes in the
 *             order the decoder reads them.
 * kvq_entropy_encode
 *   codes   device [nblocks][d/2] packed codes (kvq_quantize's), read.
 *   out     device [nblocks][slot bytes], written (bytes past a block's size
 *           are left as they were).
 *   nbytes  device u32 [nblocks]: the block's stored size 96 + sum of its
 *           stream lengths, written.
 * kvq_entropy_decode
 *   in      device slots as written by kvq_entropy_encode, read.
 *   codes   device [nblocks][d/2], written: the codes that were encoded.
 *   status  device int32, written: KVQ_OK, or KVQ_ERR_CORRUPT if a slot's
 *           counts do not add up to d, its streams overrun the slot, or a
 *           stream ends before or after its symbols (that block's codes are
 *           then unspecified; no byte outside the slot is read).
 */
size_t kvq_entropy_slot_bytes(kvq_layout L);
int kvq_entropy_encode(const uint8_t *codes, kvq_layout L, uint8_t *out, uint32_t *nbytes,
                       void *stream);
int kvq_entropy_decode(const uint8_t *in, kvq_layout L, uint8_t *codes, int32_t *status,
                       void *stream);

/*
 * kvq_entropy_encode_runs / kvq_entropy_decode_runs -- coding across adjacent
 * blocks ("Implementation notes": arithmetic coding across adjacent blocks).
 * The blocks in runs of nseg consecutive blocks (1 <= nseg <= 32; the last
 * run may be shorter): a run is one set of 32 interleaved rANS streams whose
 * state continues from block to block (stream l: entries l, l+32, .. of the
 * run's first block, then of its second, ..), every symbol coded with its own
 * block's exact counts, the rANS of kvq_entropy_encode otherwise.  The 32
 * states and lengths are stored once per run instead of once per block; a
 * run decodes as a whole.
 * Run slot r at out + r * kvq_entropy_run_bytes(L, nseg) (little-endian):
 *   [0, 32 m)          16 x u16 counts of each of its m blocks
 *   [32 m, 32 m + 64)  32 x u16: bytes of each stream
 *   then the streams in order, each its final state (4 bytes) and its bytes
 *   in the order the decoder reads them.
 *   codes   device uint8 [nblocks][16 group] (kvq_quantize's layout).
 *   out     device, ceil(nblocks / nseg) slots; nbytes device uint32 per run:
 *           the run's stored size.
 *   status  (decode) device int32: KVQ_ERR_CORRUPT for a malformed slot
 *           (every read is checked against the slot; the codes of such a
 *           run are unspecified).
 * kvq_entropy_run_bytes returns 0 for an invalid layout or nseg.
 */
size_t kvq_entropy_run_bytes(kvq_layout L, int nseg);
int kvq_entropy_encode_runs(const uint8_t *codes, kvq_layout L, int nseg, uint8_t *out,
                            uint32_t *nbytes, void *stream);
int kvq_entropy_decode_runs(const uint8_t *in, kvq_layout L, int nseg, uint8_t *codes,
                            int32_t *status, void *stream);

/*
 * kvq_decode_attention -- one decoding step of attention over the quantized
 * cache, with the codes decoded in registers ("Implementation notes": decode
 * before attention; the page records attention latency).  For query head hq
 * and its KV head h = hq / n_rep:
 *     s_t = scale * sum_f q[hq][f] K[h][t][f]      for t < T_valid
 *     out[hq][f] = sum_t softmax(s)_t V[h][t][f]
 * where K[h][t][f] = k_codebook[block][code] is the level the entry's 4-bit
 * code selects (the stored value; no binary16 copy is made), V likewise.
 * Arithmetic in fp32 (products, sums, base-2 exponentials of
 * scale*log2(e)-scaled scores); the token range is split over CTAs and the
 * splits are combined by rescaling to a common maximum.
 *   q             device fp32 [S * n_rep][128]: the query heads, grouped by
 *                 KV head (hq = h * n_rep + r); read.
 *   n_rep         query heads per KV head: 1, 2 or 4.
 *   L             layout of the K (and the V) tensor: S = KV heads, T tokens,
 *                 D = 128, any valid group.
 *   k_codes, k_codebook, v_codes, v_codebook
 *                 device outputs of kvq_quantize / kvq_allocate for the K and
 *                 the V tensor of layout L (for a tensor that stacks K and V
 *                 as streams, pointers to their first blocks); read.
 *   T_valid       tokens attended, 0 <= T_valid <= T (0: out = 0).
 *   scale         finite softmax scale (1/sqrt(128) for plain attention).
 *   workspace     device, kvq_attention_workspace_bytes(L, n_rep) bytes of
 *                 scratch (per-split partial results); overwritten.
 *   out           device fp32 [S * n_rep][128], written.
 *   status        device int32 or NULL: set to KVQ_ERR_TIMEOUT if a bulk copy
 *                 of codes into shared memory never completed (that token
 *                 range is then left out of out); untouched otherwise.
 * Errors: KVQ_ERR_INVALID_ARG for D != 128, n_rep not in {1, 2, 4}, more
 * than 65535 KV heads, T_valid out of range, a non-finite scale, a missing or
 * unaligned pointer.
 */
size_t kvq_attention_workspace_bytes(kvq_layout L, int n_rep);
int kvq_decode_attention(const float *q, int n_rep, kvq_layout L, const uint8_t *k_codes,
                         const float *k_codebook, const uint8_t *v_codes,
                         const float *v_codebook, int64_t T_valid, float scale, void *workspace,
                         float *out, int32_t *status, void *stream);

/*
 * One global lambda over a tensor whose blocks are split across devices
 * ("Mathematical statement": the blocks are coupled only through lambda).
 * Each device holds some of the blocks (any split: streams, layers, ...) and
 * their kvq_stats record.  The 40-step bisection of kvq_allocate then runs as
 * rounds: every rank asks kvq_search_probes for the round's lambdas (up to
 * 32), evaluates its own blocks there with kvq_rate_sums, the ranks add the
 * 32 integer sums (an all-reduce; integer adds are exact, so the result does
 * not depend on the split or the order), and every rank feeds the same sums
 * to kvq_search_advance, so all ranks hold the same search state.  When
 * kvq_search_probes returns 0 the search is done: kvq_search_result gives
 * lambda, and each rank takes its blocks' choice there with kvq_allocate in
 * KVQ_SUBGRADIENT mode with eta = 0.  The result does not depend on how the
 * blocks are split (bit for bit), and it is the bisection of kvq_allocate
 * with the same control and rate sums; kvq_allocate's own search evaluates
 * other probes (a sampled pilot round places its first ones), so the two
 * lambdas agree within the binary32 DP's rounding (both within the parity
 * tolerance of the exact bisection).
 *
 * kvq_search_state_bytes  size of the state (host memory, caller-owned).
 * kvq_search_begin        start: hi0 = the largest (c_max - c_min)^2 over all
 *                         ranks' blocks (kvq_stats_hi0 on each, then the max),
 *                         budget_bits the total budget over all ranks.
 * kvq_search_probes       the round's lambdas into lambdas[0 .. n-1]; returns
 *                         n, 0 when the search is done, -1 on a bad argument.
 * kvq_search_advance      feed the round's total fixed-point rate sums
 *                         (rate_sums[p] for probe p, the all-reduced output
 *                         of kvq_rate_sums).
 * kvq_search_result       lambda and the number of rounds; KVQ_OK,
 *                         KVQ_ERR_INFEASIBLE (lambda then is the largest
 *                         bracket), KVQ_ERR_INVALID_ARG if not done.
 * kvq_stats_hi0           the largest (c_max - c_min)^2 of one kvq_stats
 *                         record (synchronous copy to the host); returns
 *                         KVQ_ERR_NONFINITE if a block holds NaN or +-Inf.
 * kvq_rate_sums           device int64 sums[32]: sums[p] = sum over the
 *                         layout's blocks of d_r H_r at float(lambdas[p]) in
 *                         units of 2^-20 bit (each block rounded once), the
 *                         exact DP of kvq_allocate; sums[p] = 0 for p >= n.
 *                         lambdas is host memory (n <= 32, each finite, >= 0).
 * All but kvq_stats_hi0 and kvq_rate_sums are host computations.
 */
size_t kvq_search_state_bytes(void);
int kvq_search_begin(double hi0, double budget_bits, void *state);
int kvq_search_probes(const void *state, double *lambdas);
int kvq_search_advance(void *state, const int64_t *rate_sums, double budget_bits);
int kvq_search_result(const void *state, double *lambda, int32_t *rounds);
int kvq_stats_hi0(const void *stats, double *hi0);
int kvq_rate_sums(const void *stats, kvq_layout L, int s, const double *lambdas, int nprobe,
                  int64_t *sums, void *stream);

/*
 * kvq_allocate_report -- what the last kvq_allocate on this workspace did
 * (diagnostics; no counterpart on the method's page).  Synchronous: waits
 * for the copy of the control block to the host.
 *   rounds     rounds of DP evaluations the lambda search ran (each round
 *              evaluates every block whose rate can still change at up to
 *              32 lambdas, one per lane)
 *   active[i]  blocks evaluated in round i (i < 16)
 *   lambda, xa, xb  the answer, and the largest infeasible / smallest
 *              feasible lambda evaluated (the codebooks are the choice at xb)
 *   steps      bisection steps taken (40 unless lambda = 0 or infeasible)
 *   t_start, t_end  device clock (%globaltimer, ns) at the search kernel's
 *              start and at the end of its emit
 *   t_dp[i], t_ctl[i]  device clock when round i's evaluations were all in,
 *              and when its control had published the next round
 */
typedef struct kvq_report {
    int32_t rounds;
    int32_t steps;
    uint32_t active[16];
    double lambda, xa, xb;
    uint64_t t_start, t_end;
    uint64_t t_dp[16], t_ctl[16];
} kvq_report;
int kvq_allocate_report(const void *workspace, kvq_report *report);

/* Text of a status code. */
const char *kvq_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
