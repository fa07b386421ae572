/*
 * engram.h -- C ABI of libengram.so: the Engram memory read of
 * DeepSeek-V4.1-Flash on one GB300 (sm_103a).
 *
 * What it computes, per query token t (sources: vramglass.com
 * "deepseek-v4-1-flash-local-deployment", section "What makes up the 511 GB
 * of weights?"; rohitghumare.com "guides/deepseek-v4-1-flash", sections
 * "Engram: the table that is never multiplied" and "The architecture"):
 *   1. the suffix 2-, 3- and 4-grams of token ids ending at t (positions
 *      before the start of t's sequence read the pad id V);
 *   2. 2 modules x 3 orders x 8 heads = 48 hashes, table j =
 *      (module*3 + order-2)*8 + head; for each, h = seed[j], then for every
 *      id of the n-gram, oldest first: h = (h ^ id) * 0x9E3779B97F4A7C15
 *      (mod 2^64); h ^= h >> 29; and idx[t][j] = h mod R;
 *   3. mem[t][256*m + c] = sum over module m's 24 tables of
 *      scale[j][idx] * e4m3(table[j][idx][c])   (fp32 sums);
 *   4. X = bf16(mem) [T,512]; y = X @ W_out [512,d] (fp32 accumulation);
 *   5. h[t] += sigmoid(<h[t]/rms(h[t]), g> / sqrt(d)) * y[t], rounded to bf16,
 *      rms(v) = sqrt(mean(v^2) + eps).
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers unless a parameter says "host".  Pinned
 *     host memory that the device can address (cudaHostAlloc, or memory the
 *     GPU reaches over NVLink-C2C) is accepted where it says "host tables".
 *   - The caller owns every buffer, stream and event; the library allocates
 *     no memory.  Workspaces are sized by the matching *_workspace_bytes().
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call only enqueues work on its stream(s) and returns;
 *     no call synchronises with the host except engram_last_error().
 *   - Arguments are validated before anything is enqueued; a bad argument
 *     returns ENGRAM_EINVAL and enqueues nothing.  A failed launch returns
 *     ENGRAM_ECUDA.  Conditions only the device can see (token ids out of
 *     range, a sequence shorter than last_n, an index >= R, more unique rows
 *     than the staging capacity, a pipeline wait that ran out of time) set a
 *     sticky per-device error word that engram_last_error() returns; the
 *     kernels never trap.
 *   - n_query == 0 is a no-op that returns ENGRAM_OK.
 *   - bf16 tensors are passed as uint16_t bit patterns.
 */
#ifndef ENGRAM_H
#define ENGRAM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ENGRAM_OK = 0,
    ENGRAM_EINVAL = 1,      /* bad argument (null, misaligned, size) */
    ENGRAM_ECUDA = 2,       /* a CUDA call or launch failed */
    ENGRAM_ERANGE = 3,      /* device saw a token id, position or index out of range */
    ENGRAM_ECAPACITY = 4,   /* more unique rows than the staging capacity */
    ENGRAM_ETIMEOUT = 5,    /* a bounded device-side wait gave up */
    ENGRAM_ENOMEM = 6,      /* workspace too small */
    ENGRAM_EUNSUPPORTED = 7 /* device is not sm_103 / feature missing */
} engram_status;

#define ENGRAM_N_TABLES 48
#define ENGRAM_ROW_BYTES 256
#define ENGRAM_MEM_DIM 512

/* Table row layouts (engram_config.row_layout):
 *  ENGRAM_ROWS_SEPARATE: tables e4m3 [48][R][256]; scales fp32 [48][R] in their
 *                        own array (the `scales` argument).
 *  ENGRAM_ROWS_RECORD:   tables [48][R][272]: bytes 0..255 the row's e4m3 codes,
 *                        256..259 its fp32 scale, 260..271 padding; the
 *                        `scales` argument is ignored (may be NULL).  One
 *                        contiguous read per row instead of two scattered ones
 *                        (the pages describe a row as 256 B of FP8 plus its
 *                        scales, "Engram: the table that is never multiplied"). */
/*  ENGRAM_ROWS_MX:       MXFP8-style rows, [48][R][272]: bytes 0..255 the e4m3
 *                        codes, 256..263 eight E8M0 block scales (byte b scales
 *                        codes 32b..32b+31 by 2^(byte - 127); 0 is 2^-127 and
 *                        255 is NaN), 264..271 padding; `scales` is ignored.
 *                        This is the pages' row of 256 FP8 bytes plus 8 scale
 *                        bytes (12,672 bytes for a token's 48 rows), in place of
 *                        the per-row fp32 scale of the two layouts above. */
#define ENGRAM_ROWS_SEPARATE 0
#define ENGRAM_ROWS_RECORD 1
#define ENGRAM_ROWS_MX 2
#define ENGRAM_RECORD_BYTES 272

typedef struct {
    int32_t vocab;       /* V: token ids must lie in [0, V); V itself is the pad id */
    int32_t d_model;     /* d: residual width; the projection needs d % 256 == 0, 256 <= d <= 32768 */
    int64_t rows;        /* R: rows per table, R >= 1 */
    float rms_eps;       /* eps inside the rmsnorm of the gate (1e-6 by default) */
    uint32_t row_layout; /* ENGRAM_ROWS_SEPARATE, ENGRAM_ROWS_RECORD or ENGRAM_ROWS_MX */
    uint64_t seeds[ENGRAM_N_TABLES]; /* hash seed of table j */
} engram_config;

/* Human-readable name of a status code (static string). */
const char *engram_status_string(engram_status st);

/* Returns the sticky device error word of the current device as a status
 * (ENGRAM_OK if clear) and clears it.  Synchronises the device. */
engram_status engram_last_error(void);

/* Health check of the device-side time limits (not part of the Engram read):
 * enqueues one small kernel whose bounded wait on a barrier that nothing
 * arrives on runs out after limit_ns nanoseconds of device time.  The kernel
 * then sets ENGRAM_ETIMEOUT in the sticky word and returns, as any projection
 * or pipeline wait of this library does when it gives up; the device stays
 * usable.  limit_ns in [1, 10^10], else ENGRAM_EINVAL (nothing enqueued). */
engram_status engram_wait_selftest(uint64_t limit_ns, void *stream);

/*
 * Row addresses: steps 1-2 above.  Addresses depend on token ids only (no
 * table is read), so a whole prompt can be hashed before its forward pass
 * ("What makes up the 511 GB of weights?": every address for a prompt can be
 * computed up front and prefetched in one batch).
 *   tokens      int32 [seq_offsets[n_seqs]] token ids in [0, V)
 *   seq_offsets int64 [n_seqs+1] ascending; sequence s is
 *               tokens[seq_offsets[s] .. seq_offsets[s+1])
 *   last_n      0: query every position, in order, n_query must equal
 *               seq_offsets[n_seqs] - seq_offsets[0];
 *               k > 0: query the last k positions of each sequence, sequence
 *               by sequence, n_query must equal n_seqs*k (a shorter sequence
 *               sets ENGRAM_ERANGE on the device)
 *   idx         int64 [n_query][48] output, row index in [0, R) of table j
 */
engram_status engram_hash(const engram_config *cfg, const int32_t *tokens, const int64_t *seq_offsets,
                          int64_t n_seqs, int32_t last_n, int64_t n_query, int64_t *idx, void *stream);

/*
 * Step 3 (gather, dequantise, per-module sum).
 *   tables e4m3 codes [48][R][256] (or [48][R][272] records), 16-byte aligned
 *   scales fp32 [48][R] (ENGRAM_ROWS_SEPARATE only)
 *   idx    int64 [n_query][48], each in [0, R) (out-of-range rows read nothing
 *          and set ENGRAM_ERANGE)
 *   mem    fp32 [n_query][512] output, module 0 then module 1, 16-byte aligned
 */
engram_status engram_gather_reduce(const engram_config *cfg, const uint8_t *tables, const float *scales,
                                   const int64_t *idx, int64_t n_query, float *mem, void *stream);

/*
 * Steps 4-5 (bf16 concat, tcgen05 projection, gated residual update in place).
 *   mem   fp32 [n_query][512] (16-byte aligned)
 *   W_out bf16 [512][d] row-major (16-byte aligned)
 *   g     bf16 [d]
 *   h     bf16 [n_query][d], read and updated in place (16-byte aligned)
 * Needs d % 256 == 0 and d <= 32768 (ENGRAM_EINVAL otherwise).
 */
engram_status engram_fuse(const engram_config *cfg, const float *mem, const uint16_t *W_out, const uint16_t *g,
                          uint16_t *h, int64_t n_query, void *stream);

/*
 * Steps 1-5 in one call on one stream (HBM-resident tables), as two kernels:
 * a gather that hashes in registers (no idx array) and writes bf16 X, then
 * the projection, which loads X by TMA.  workspace >=
 * engram_forward_workspace_bytes(cfg, n_query) bytes of device memory,
 * 256-byte aligned (it holds X); its contents are scratch.
 *
 * tables (and scales) may also be pinned host memory, registered with CUDA
 * (engram_host_alloc, cudaHostAlloc): the gather then reads each row in
 * place over unified addressing ("vLLM reads pinned tables over UVA" in
 * "Engram: the table that is never multiplied"), with the same results.  For
 * decode-sized batches this beats engram_forward_host, whose dedup and
 * staging carry a fixed cost (64 queries: 16.8 against 113 us per call;
 * 512: 48 against 143 us; with scales in HBM and 51.5 GB of host tables);
 * from a few thousand queries staging wins (4,096: 3.4 against 1.2 ms).
 * The same holds for engram_gather_x and engram_gather_reduce.
 */
size_t engram_forward_workspace_bytes(const engram_config *cfg, int64_t n_query);
engram_status engram_forward(const engram_config *cfg, const int32_t *tokens, const int64_t *seq_offsets,
                             int64_t n_seqs, int32_t last_n, int64_t n_query, const uint8_t *tables,
                             const float *scales, const uint16_t *W_out, const uint16_t *g, uint16_t *h,
                             void *workspace, size_t workspace_bytes, void *stream);

/*
 * The two halves of engram_forward, for callers that issue the table reads
 * early (addresses depend on tokens only, so the gather can run before the
 * layer that consumes it) and the projection later:
 * engram_gather_x: steps 1-3 fused, hashing in registers, writing
 *   X bf16 [n_query][512] (16-byte aligned) = bf16 of the module sums.
 * engram_fuse_x:   steps 4-5 from that X (loaded by TMA); needs d % 256 == 0.
 * engram_gather_x then engram_fuse_x gives the same bits as engram_forward.
 */
engram_status engram_gather_x(const engram_config *cfg, const int32_t *tokens, const int64_t *seq_offsets,
                              int64_t n_seqs, int32_t last_n, int64_t n_query, const uint8_t *tables,
                              const float *scales, uint16_t *X, void *stream);
engram_status engram_fuse_x(const engram_config *cfg, const uint16_t *X, const uint16_t *W_out, const uint16_t *g,
                            uint16_t *h, int64_t n_query, void *stream);

/*
 * Row-sharded tables ("Engram: the table that is never multiplied": SGLang
 * splits the tables by row across tensor-parallel GPUs, at the cost of one
 * all-reduce per Engram layer).  Row r of every table belongs to shard
 * r mod n_shards and is stored there as local row r / n_shards, so each
 * shard holds engram_shard_rows(cfg, n_shards) = ceil(R / n_shards) rows per
 * table (the last one unused on some shards).
 * engram_gather_reduce_shard: steps 1-3 for every query token, reading only
 *   this shard's rows (hashed in registers as in engram_gather_x):
 *   mem[t][256m + c] = sum over module m's tables j whose row idx[t][j] this
 *   shard owns of scale * e4m3 value, fp32, other rows adding nothing.
 *   tables_shard [48][ceil(R/n)][256 or 272] and scales_shard [48][ceil(R/n)]
 *   in the layouts of engram_gather_reduce; mem fp32 [n_query][512] output.
 *   The sum over all shards of their mem (the one exchange: an all-reduce,
 *   or a reduce-scatter over tokens) is the whole mem up to fp32 summation
 *   order; engram_fuse then applies steps 4-5.  shard in [0, n_shards).
 */
int64_t engram_shard_rows(const engram_config *cfg, int32_t n_shards);
engram_status engram_gather_reduce_shard(const engram_config *cfg, int32_t shard, int32_t n_shards,
                                         const int32_t *tokens, const int64_t *seq_offsets, int64_t n_seqs,
                                         int32_t last_n, int64_t n_query, const uint8_t *tables_shard,
                                         const float *scales_shard, float *mem, void *stream);

/*
 * engram_forward without a workspace argument.  The sources have no
 * counterpart: this entry point exists for callers that cannot allocate
 * device memory -- code running inside a host engine or framework that owns
 * all device memory through its own pool and forbids raw cudaMalloc from
 * plug-ins, or that may not allocate once it is serving (an allocation there
 * can fail, fragment the pool or stall other work).  It does the same work as
 * engram_forward, with the bf16 X between its two kernels kept in a
 * file-scope device array of ENGRAM_NO_WORKSPACE_MAX_QUERY x 512 bf16
 * (16 MB) instead of a caller workspace.
 *   - Allocates nothing and calls no allocating CUDA or library routine.
 *   - Every GPU that loads libengram.so holds that array until the process
 *     exits.
 *   - Arguments are checked as for engram_forward (ENGRAM_EINVAL first);
 *     then n_query > ENGRAM_NO_WORKSPACE_MAX_QUERY returns ENGRAM_ENOMEM.
 *     Either way nothing is enqueued.
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current); make that first call before
 *     any stream capture on the device.  The address is kept for the life of
 *     the process: do not call this entry point on a device after
 *     cudaDeviceReset() on it (the array may then live elsewhere).
 *   - Every call shares the one array: two calls that overlap on the GPU
 *     (different streams, or different host threads on one device) race on
 *     it and give undefined results.  Calls in one stream are ordered and
 *     safe.  Nothing in the array needs clearing between calls.
 */
#define ENGRAM_NO_WORKSPACE_MAX_QUERY 16384
engram_status engram_forward_no_workspace(const engram_config *cfg, const int32_t *tokens,
                                          const int64_t *seq_offsets, int64_t n_seqs, int32_t last_n,
                                          int64_t n_query, const uint8_t *tables, const float *scales,
                                          const uint16_t *W_out, const uint16_t *g, uint16_t *h, void *stream);

/*
 * Host-table path ("Engram: the table that is never multiplied": tables in
 * pinned host memory read over unified addressing, the lookup on a side
 * stream; "What makes up the 511 GB of weights?": addresses computed up front
 * and prefetched in one batch).
 *
 * engram_dedup: the distinct (table, row) pairs among idx, sorted by
 * (table, row), and each query's slot in that list.
 *   workspace   >= engram_dedup_workspace_bytes(cfg) bytes, 256-byte aligned
 *   unique      int64 [capacity] output: flat row j*R + row of slot u
 *   idx_staged  int32 [n_query][48] output: slot of (t, j)
 *   n_unique    int64 [1] output (device): number of distinct rows U.
 * If U > capacity, ENGRAM_ECAPACITY is set on the device, every idx_staged
 * entry is -1 (no slot: an index out of range also gets -1, with
 * ENGRAM_ERANGE), engram_stage then copies nothing and the staged gather
 * reads no row (mem = 0), so engram_forward_host leaves h as it was.
 */
size_t engram_dedup_workspace_bytes(const engram_config *cfg);
engram_status engram_dedup(const engram_config *cfg, const int64_t *idx, int64_t n_query, void *workspace,
                           size_t workspace_bytes, int64_t *unique, int64_t capacity, int32_t *idx_staged,
                           int64_t *n_unique, void *stream);

/*
 * engram_stage: copy the U = *n_unique unique rows and their scales from
 * host tables into device staging buffers; if U > capacity it copies nothing
 * (the dedup has already set ENGRAM_ECAPACITY).
 *   host_tables e4m3 [48][R][256] (or [48][R][272] records) in pinned host
 *               memory (16-byte aligned)
 *   host_scales fp32 [48][R] in pinned host memory (ENGRAM_ROWS_SEPARATE only),
 *               or in device memory: the kernel reads it through its unified
 *               address either way, and a device-resident scale array (1/64
 *               of the tables' bytes) keeps the scattered 4-byte scale reads
 *               off the host link (same results; the host-table forward of
 *               65,536 tokens measured 4.21 against 4.70 ms per call).  The
 *               same holds for the host-table forward entry points below.
 *   Staging holds 256-byte rows plus a separate fp32 scale array:
 *   staged_rows [capacity][256] and staged_scales [capacity] (device, 16-byte
 *   aligned); for ENGRAM_ROWS_MX whole rows are staged instead:
 *   staged_rows [capacity][272] and staged_scales unused (may be NULL).
 * Enqueued on `stream` (normally a side stream that waited for the dedup).
 */
engram_status engram_stage(const engram_config *cfg, const uint8_t *host_tables, const float *host_scales,
                           const int64_t *unique, const int64_t *n_unique, int64_t capacity,
                           uint8_t *staged_rows, float *staged_scales, void *stream);

/*
 * Step 3 over staged rows: same arithmetic, same summation order as
 * engram_gather_reduce, so its output is bit-identical to the HBM path on
 * the same inputs (SGLang's host-table mode is documented as bitwise
 * identical, "Engram: the table that is never multiplied").  Staging
 * layouts as in engram_stage.  An idx_staged entry of -1 names no row and
 * adds nothing (the dedup's overflow or range error is already flagged);
 * any other entry outside [0, capacity) sets ENGRAM_ERANGE.
 */
engram_status engram_gather_reduce_staged(const engram_config *cfg, const uint8_t *staged_rows,
                                          const float *staged_scales, const int32_t *idx_staged,
                                          int64_t n_query, int64_t capacity, float *mem, void *stream);

/*
 * The whole host-table path: hash and dedup on `stream`; the row stage on
 * `side_stream` after `ev_dedup` (recorded here on `stream`); the staged
 * gather and fuse on `stream` after `ev_staged` (recorded on `side_stream`).
 * Both events are caller-created (cudaEventDisableTiming is fine).
 * workspace >= engram_forward_host_workspace_bytes(cfg, n_query, capacity).
 * The call can be captured into a CUDA graph on `stream`: the side stream
 * joins the capture through `ev_dedup` and rejoins `stream` through
 * `ev_staged`; replays give the eager call's bits.
 */
size_t engram_forward_host_workspace_bytes(const engram_config *cfg, int64_t n_query, int64_t capacity);
engram_status engram_forward_host(const engram_config *cfg, const int32_t *tokens, const int64_t *seq_offsets,
                                  int64_t n_seqs, int32_t last_n, int64_t n_query, const uint8_t *host_tables,
                                  const float *host_scales, const uint16_t *W_out, const uint16_t *g,
                                  uint16_t *h, int64_t capacity, void *workspace, size_t workspace_bytes,
                                  int64_t *n_unique, void *stream, void *side_stream, void *ev_dedup,
                                  void *ev_staged);

/*
 * The per-layer form of the Engram read (rohitghumare.com
 * "guides/deepseek-v4-1-flash": section "The architecture", layers 1 and 14
 * each add looked-up rows into the residual stream through a learned gate;
 * section "Engram: the table that is never multiplied", 24 rows per Engram
 * layer and a gate that compares each retrieved row with the hidden state).
 * Layer m in {0, 1} uses module m's 24 tables (24m .. 24m+23) and, per the
 * reading the pages leave open,
 *   g_j = sigmoid(<rmsnorm(h) W_q, rmsnorm(r_j) W_k> / 16)   per row r_j,
 *   h   = bf16(h + bf16(sum_j g_j r_j) W_m),
 * rmsnorm without a weight (eps = cfg->rms_eps), r_j = scale * e4m3 value.
 *
 * engram_layer_keys: W_kk [512][256] = [W_k^T ; W_k^T] (bf16 copies) from
 *   W_k [256][256] (bf16, device); once per set of weights.
 * engram_layer_forward: one layer, in place on h [n_query][d] bf16, from the
 *   HBM tables (any row layout; with ENGRAM_ROWS_MX each code of r_j is scaled
 *   by its 32-code block's E8M0 scale before the rmsnorm, the dot product and
 *   the sum), W_q [d][256], W_kk and W_m [256][d] (bf16, device).
 *   Kernels: q = rinv(h) h W_q (tcgen05, written as bf16 q_hi | q_lo), u =
 *   [q_hi | q_lo] W_kk = q W_k^T (tcgen05), the gated gather (hash, gather,
 *   score_j = <u, rmsnorm(r_j)> / 16, X = bf16 [n][256]), the projection.
 *   workspace >= engram_layer_workspace_bytes: q pair bf16 [n][512], u fp32
 *   [n][256], X bf16 [n][256], each 256-byte aligned.  Argument errors return
 *   synchronously; device range errors set the sticky error word.  d must be
 *   a multiple of 256.
 */
engram_status engram_layer_keys(const engram_config *cfg, const uint16_t *W_k, uint16_t *W_kk, void *stream);
size_t engram_layer_workspace_bytes(const engram_config *cfg, int64_t n_query);
engram_status engram_layer_forward(const engram_config *cfg, int32_t module, const int32_t *tokens,
                                   const int64_t *seq_offsets, int64_t n_seqs, int32_t last_n, int64_t n_query,
                                   const uint8_t *tables, const float *scales, const uint16_t *W_q,
                                   const uint16_t *W_kk, const uint16_t *W_m, uint16_t *h, void *workspace,
                                   size_t workspace_bytes, void *stream);

/*
 * Pinned host memory for host tables (engram_stage, engram_forward_host,
 * engram_forward_host_pipelined), mapped on transparent huge pages where the
 * operating system offers them and registered with the CUDA driver, so the
 * device reaches it through unified addressing (the pages' host-resident
 * tables read over the host link, "Engram: the table that is never
 * multiplied").  Staging reads rows scattered over tens of GB; with base pages
 * the device spends much of that time translating addresses.  This is the one
 * call that allocates; it is host-only and synchronous.
 *   engram_host_alloc: *ptr receives `bytes` of zeroed, pinned memory aligned
 *   to the huge page size; ENGRAM_EINVAL for bytes == 0 or ptr == NULL,
 *   ENGRAM_ENOMEM if the mapping fails, ENGRAM_ECUDA if registration fails.
 *   engram_host_free: releases a pointer from engram_host_alloc (NULL is a
 *   no-op; any other pointer is ENGRAM_EINVAL); no device work may still use it.
 */
engram_status engram_host_alloc(size_t bytes, void **ptr);
engram_status engram_host_free(void *ptr);

/*
 * The host-table path with a cache of staged rows kept in HBM across calls
 * (the pages' staging of hot rows for a Zipf token stream, "Engram: the table
 * that is never multiplied" and "What makes up the 511 GB of weights?": rows
 * pulled over the host link once are read from device memory afterwards).
 * The cache is a caller-owned device buffer of
 * engram_host_cache_bytes(cfg, slots, capacity) bytes (256-byte aligned):
 * `slots` cached rows (a power of two, direct-mapped by the row's flat index
 * j*R + row) plus `capacity` overflow rows, with their tags.
 * engram_host_cache_reset empties it (enqueued on `stream`).
 * engram_forward_host_cached: hash and dedup as engram_forward_host; then
 * every distinct row of the batch claims its cache slot for this call (the
 * first claimant owns it: a row already there is a hit and is not staged, any
 * other row replaces it); a row whose slot another row of the same call owns
 * goes to an overflow row.  Only misses cross the host link (on
 * `side_stream`, after `ev_dedup`); the staged gather reads cache and
 * overflow rows and the projection follows on `stream` (after `ev_staged`).
 * h equals engram_forward's on the same tables bit for bit.
 *   stamp    >= 1, larger than every earlier call's on this cache since its
 *            reset (a call counter); a cache serves one stream of calls:
 *            calls that overlap on the GPU race on it.  A call captured in a
 *            CUDA graph replays its stamp: replays after the first find every
 *            slot claimed at that stamp and stage all their rows into the
 *            overflow area (no hits), with h still bit-exact
 *   capacity distinct rows per call at most (n_query * 48 always suffices);
 *            more set ENGRAM_ECAPACITY, stage nothing and leave h unchanged
 *   stats    int64 [4] (device): distinct rows, cache hits, rows staged over
 *            the host link, of which outside the cache (overflow)
 * workspace >= engram_forward_host_cached_workspace_bytes(cfg, n_query,
 * capacity); host tables and scales as in engram_forward_host.
 */
size_t engram_host_cache_bytes(const engram_config *cfg, int64_t slots, int64_t capacity);
engram_status engram_host_cache_reset(const engram_config *cfg, void *cache, int64_t slots, int64_t capacity,
                                      void *stream);
size_t engram_forward_host_cached_workspace_bytes(const engram_config *cfg, int64_t n_query, int64_t capacity);
engram_status engram_forward_host_cached(const engram_config *cfg, const int32_t *tokens,
                                         const int64_t *seq_offsets, int64_t n_seqs, int32_t last_n,
                                         int64_t n_query, const uint8_t *host_tables, const float *host_scales,
                                         const uint16_t *W_out, const uint16_t *g, uint16_t *h, void *cache,
                                         int64_t slots, int64_t capacity, uint32_t stamp, void *workspace,
                                         size_t workspace_bytes, int64_t *stats, void *stream, void *side_stream,
                                         void *ev_dedup, void *ev_staged);

/*
 * The host-table path pipelined over chunks of `chunk` query tokens (the
 * pages' background prefetch of host rows on a side stream, "Engram: the table
 * that is never multiplied", applied chunk by chunk).  All queries are hashed
 * first; then, for chunk k, the unique rows are found on `stream` and staged
 * on `side_stream` into one of two staging sets (k mod 2), and the staged
 * gather of chunk k runs on `stream` while chunk k+1 is being deduplicated and
 * staged; one projection over the whole batch follows.  h equals
 * engram_forward's on the same tables bit for bit.  Rows used by several
 * chunks cross the host link once per chunk.
 *   chunk       query tokens per chunk (>= 1; a multiple of 128 keeps whole
 *               tiles per chunk)
 *   capacity    staging rows per set; at least the unique rows of any chunk
 *               (chunk * 48 always suffices); more raise ENGRAM_ECAPACITY
 *   n_unique    int64 [ceil(n_query / chunk)] (device): unique rows per chunk
 *   events      6 caller-created events (cudaEventDisableTiming is fine):
 *               dedup done x2, staged x2, staging set consumed x2
 * workspace >= engram_forward_host_pipelined_workspace_bytes(cfg, n_query,
 * chunk, capacity); host tables and scales as in engram_forward_host.
 * Argument errors return synchronously; device-side range and capacity errors
 * set the sticky error word.  Capturable into a CUDA graph on `stream` like
 * engram_forward_host (every side-stream step waits on an event recorded in
 * the same call).
 */
size_t engram_forward_host_pipelined_workspace_bytes(const engram_config *cfg, int64_t n_query, int64_t chunk,
                                                     int64_t capacity);
engram_status engram_forward_host_pipelined(const engram_config *cfg, const int32_t *tokens,
                                            const int64_t *seq_offsets, int64_t n_seqs, int32_t last_n,
                                            int64_t n_query, const uint8_t *host_tables, const float *host_scales,
                                            const uint16_t *W_out, const uint16_t *g, uint16_t *h, int64_t chunk,
                                            int64_t capacity, void *workspace, size_t workspace_bytes,
                                            int64_t *n_unique, void *stream, void *side_stream,
                                            void *const *events);

#ifdef __cplusplus
}
#endif

#endif /* ENGRAM_H */
