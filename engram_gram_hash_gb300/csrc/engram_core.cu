// libengram: n-gram hash, row gather/dequant/reduce, dedup and host-row
// staging kernels, and their C entry points.
//
// Sources: vramglass.com "deepseek-v4-1-flash-local-deployment", section
// "What makes up the 511 GB of weights?" (2/3/4-gram hash tables, two modules
// of 8 heads, 48 rows of ~12 KB per token, token-only addresses prefetched in
// one batch); rohitghumare.com "guides/deepseek-v4-1-flash", section "Engram:
// the table that is never multiplied" (suffix n-grams, one row per (order,
// head), 256-byte FP8 rows, host tables read over unified addressing on a
// side stream, bitwise-identical host-table mode).
#include <sys/mman.h>

#include <algorithm>
#include <cstdio>
#include <map>
#include <atomic>
#include <mutex>
#include <cstdlib>
#include <cstring>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "fuse.cuh"
#include "fuse2.cuh"
#include "fuse3.cuh"
#include "layer.cuh"
#include "narrow.cuh"

namespace engram {

// ===================================================================== hash ==
// One thread per (query token, table): 48 consecutive threads share a token,
// so the 2-4 token loads hit L1 and the int64 idx writes are coalesced.

struct HashParams {
    const int32_t *tokens;
    const int64_t *offs;
    int64_t n_seqs;
    int64_t n_query;
    uint64_t R;
    uint64_t rmask;  // R-1 when R is a power of two
    int32_t V;
    int32_t last_n;
    int32_t pow2;
    uint64_t seeds[kTables];
};

// Row index of table j for the token at global position p of a sequence that
// starts at `start` (earlier positions read the pad id V).
__device__ __forceinline__ int64_t hash_one(const HashParams &a, uint64_t seed, int j, int64_t start, int64_t p,
                                            bool &bad) {
    const int n = 2 + (j % kTablesPerModule) / 8;  // order of table j
    uint64_t h = seed;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (i < n) {
            const int64_t q = p - (n - 1) + i;  // oldest id first
            int32_t id = a.V;
            if (q >= start) {
                id = __ldg(a.tokens + q);
                if (id < 0 || id >= a.V) bad = true;
            }
            h = (h ^ (uint64_t)(uint32_t)id) * kGolden;
            h ^= h >> 29;
        }
    }
    return (int64_t)(a.pow2 ? (h & a.rmask) : (h % a.R));
}

// Row indices of tables j (module 0) and j + 24 (module 1): the same n-gram,
// loaded once, through two seeds.
__device__ __forceinline__ void hash_two(const HashParams &a, uint64_t seed0, uint64_t seed1, int j, int64_t start,
                                         int64_t p, bool &bad, int64_t &r0, int64_t &r1) {
    const int n = 2 + (j % kTablesPerModule) / 8;
    uint64_t h0 = seed0, h1 = seed1;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (i < n) {
            const int64_t q = p - (n - 1) + i;
            int32_t id = a.V;
            if (q >= start) {
                id = __ldg(a.tokens + q);
                if (id < 0 || id >= a.V) bad = true;
            }
            h0 = (h0 ^ (uint64_t)(uint32_t)id) * kGolden;
            h0 ^= h0 >> 29;
            h1 = (h1 ^ (uint64_t)(uint32_t)id) * kGolden;
            h1 ^= h1 >> 29;
        }
    }
    r0 = (int64_t)(a.pow2 ? (h0 & a.rmask) : (h0 % a.R));
    r1 = (int64_t)(a.pow2 ? (h1 & a.rmask) : (h1 % a.R));
}

// Sequence s with offs[s] <= p < offs[s+1] (last such s; empty sequences skip).
__device__ __forceinline__ int64_t find_seq(const int64_t *offs, int64_t n_seqs, int64_t p) {
    int64_t lo = 0, hi = n_seqs;
    while (hi - lo > 1) {
        const int64_t mid = (lo + hi) >> 1;
        if (__ldg(offs + mid) <= p) lo = mid; else hi = mid;
    }
    return lo;
}

// Query q -> (sequence start, position); false if the position is invalid.
__device__ __forceinline__ bool query_position(const HashParams &a, int64_t q, int64_t &start, int64_t &p) {
    if (a.last_n == 0) {
        p = __ldg(a.offs) + q;
        const int64_t s = find_seq(a.offs, a.n_seqs, p);
        start = __ldg(a.offs + s);
        return p < __ldg(a.offs + s + 1);
    }
    const int64_t s = q / a.last_n;
    const int64_t k = q - s * a.last_n;
    start = __ldg(a.offs + s);
    p = __ldg(a.offs + s + 1) - a.last_n + k;
    return p >= start;
}

__global__ void __launch_bounds__(256) hash_kernel(const __grid_constant__ HashParams a, int64_t *__restrict__ idx) {
    __shared__ uint64_t s_seed[kTables];
    if (threadIdx.x < kTables) s_seed[threadIdx.x] = a.seeds[threadIdx.x];
    if (blockIdx.x == 0 && threadIdx.x == 0 && a.last_n == 0 &&
        __ldg(a.offs + a.n_seqs) - __ldg(a.offs) != a.n_query)
        raise_error(ENGRAM_ERANGE);
    __syncthreads();
    const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= a.n_query * kTables) return;
    const int64_t q = g / kTables;
    const int j = (int)(g - q * kTables);
    int64_t start, p;
    bool bad = false;
    int64_t out = 0;
    if (query_position(a, q, start, p)) {
        out = hash_one(a, s_seed[j], j, start, p, bad);
    } else {
        bad = true;
    }
    if (bad) raise_error(ENGRAM_ERANGE);
    idx[g] = out;
}

// ============================================================ gather-reduce ==
// One warp per query token, its two modules in turn.  Lanes 0..23 find the
// rows of both modules first (the n-gram ids are loaded once and hashed with
// both modules' seeds), so a token's address chain is paid once.  Then, per
// module, lane l reads 16 bytes of row (2i + l/16) at byte offset 16*(l%16)
// for i = 0..11: each warp-wide load covers two whole 256-byte rows and all
// 12 loads are issued before the arithmetic, so a warp keeps 6 KB of random
// reads in flight.  The two half-warps' partial sums are merged with one
// xor-16 shuffle.  (A warp per (token, module) paid the address chain twice:
// 0.428 against 0.419 ms on the large workload, 0.701 against 0.610 ms on
// prefill, whose repeated rows hit L2.)
//
// Row addresses come from an int64 idx array (HBM tables), an int32 slot
// array (staged rows), or are hashed in-register by lanes 0..23 (the fused
// path: no idx round trip).  The sums go out as fp32 mem or as bf16 X (the
// projection's operand; bf16 rounding of the same fp32 sums, so both outputs
// agree bit for bit after rounding).

// IDX_HASH_SHARD: hashed in registers, but only the rows this shard owns
// are read (row r of every table belongs to shard r mod n_shards, stored
// there as local row r / n_shards); the others add nothing.
enum IdxMode { IDX_I64 = 0, IDX_STAGED_I32 = 1, IDX_HASH = 2, IDX_HASH_SHARD = 3 };

constexpr int32_t kSlotNone = -1;  // idx_staged entry that names no staged row

enum ScaleMode { SCALE_ARRAY = 0, SCALE_IN_ROW = 1, SCALE_MX = 2 };

// Token gates computed beside the gather for the d-split projection
// (narrow.cuh), in the projection kernels' reduction order: d in `groups`
// slices of cpg 256-column chunks; per slice, lane l sums its 16-byte pieces
// l, l+32, ... (fmaf in column order), a butterfly adds the lanes, and the
// slices' sums are added in slice order; then
// gate = sigmoid(rsqrt(sum h^2 / d + eps) * <h,g> / sqrt(d)).
struct GateParams {
    const uint16_t *h;  // [n_query][d] bf16
    const uint16_t *g;  // [d] bf16
    float *gate;        // [n_query] out
    int64_t gather_blocks;
    int32_t d, groups, cpg;
    float eps, inv_sqrt_d;
};

// One block per query token: warp r (< groups) sums slice r, the slice's
// pieces loaded together (one memory round trip), and thread 0 adds the
// slices' sums in slice order.  The same additions in the same order as one
// warp walking the slices in turn, with all slices' loads in flight at once.
__device__ __forceinline__ void gate_block(const GateParams &G, int64_t n_query, int64_t t, int warp, int lane) {
    __shared__ float2 slice_sum[fuse::MAX_GROUPS];
    if (t < n_query && warp < G.groups) {
        // Lane l's 16-byte piece i covers columns 8 (l + 32 i) .. +7; pieces
        // r cpg .. (r + 1) cpg - 1 make up slice r.
        const uint4 *hrow = reinterpret_cast<const uint4 *>(G.h + t * G.d);
        const uint4 *grow = reinterpret_cast<const uint4 *>(G.g);
        const int i_end = (warp + 1) * G.cpg;
        constexpr int kBatch = 8;
        float s = 0.f, d = 0.f;
        for (int i0 = warp * G.cpg; i0 < i_end; i0 += kBatch) {
            uint4 hv[kBatch], gv[kBatch];
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
                if (i0 + b < i_end) {
                    hv[b] = __ldg(hrow + lane + 32 * (i0 + b));
                    gv[b] = __ldg(grow + lane + 32 * (i0 + b));
                }
            }
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
                if (i0 + b < i_end) {
                    const uint32_t hw[4] = {hv[b].x, hv[b].y, hv[b].z, hv[b].w};
                    const uint32_t gw[4] = {gv[b].x, gv[b].y, gv[b].z, gv[b].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float a0 = bf16_lo(hw[e]), a1 = bf16_hi(hw[e]);
                        s = fmaf(a0, a0, s);
                        s = fmaf(a1, a1, s);
                        d = fmaf(a0, bf16_lo(gw[e]), d);
                        d = fmaf(a1, bf16_hi(gw[e]), d);
                    }
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            s += __shfl_xor_sync(0xffffffffu, s, o);
            d += __shfl_xor_sync(0xffffffffu, d, o);
        }
        if (lane == 0) slice_sum[warp] = make_float2(s, d);
    }
    __syncthreads();
    if (threadIdx.x == 0 && t < n_query) {
        float ssum = 0.f, dsum = 0.f;
        for (int r = 0; r < G.groups; ++r) {
            ssum += slice_sum[r].x;
            dsum += slice_sum[r].y;
        }
        const float rinv = rsqrtf(ssum / (float)G.d + G.eps);
        G.gate[t] = 1.f / (1.f + __expf(-(rinv * dsum * G.inv_sqrt_d)));
    }
}

struct GatherParams {
    const uint8_t *rows;
    const float *scales;     // fp32 [rows], or nullptr when each row carries its scale bytes at byte 256
    int64_t row_stride;      // 256 (codes only) or 272 (codes + scale bytes at byte 256)
    const void *idx;     // IDX_I64 / IDX_STAGED_I32
    int64_t n_query;
    int64_t R;           // rows per table (HBM) or staging capacity (staged)
    void *out;           // float [n][512] or bf16 [n][512]
    HashParams hp;       // IDX_HASH, IDX_HASH_SHARD
    int64_t shard_rows;  // IDX_HASH_SHARD: rows per table in this shard's tables
    int32_t shard;       // IDX_HASH_SHARD: this shard, of n_shards
    int32_t n_shards;
    GateParams gp;       // kGate: blocks from gather_blocks on compute the token gates
};

// 4 blocks of 256 threads per SM (at most 64 registers a thread; 3 blocks and
// 80 registers for kMx, which also spreads each row's scale bytes; 2 blocks
// for the few-token form with gates, where occupancy does not matter).  kMx: each row
// carries eight E8M0 block scales (one per 32 codes) instead of one fp32;
// one 8-byte load per row fetches them (lanes 0..11 of each half-warp, a row
// each) and shuffles give every lane the byte of its block (one byte load per
// lane and row instead: 0.538 against 0.455 ms on the large workload).
template <int kMode, bool kBf16Out, bool kMx, bool kGate = false>
__global__ void __launch_bounds__(256, kGate ? 2 : (kMx ? 3 : 4)) gather_kernel(const __grid_constant__ GatherParams P) {
    // The projection that consumes X may be launched as a programmatic
    // dependent: its CTAs take SMs as this grid's last blocks drain and start
    // on what does not depend on X.
    allow_dependent_launch();
    if constexpr (kGate) {  // the blocks past the gather's compute token gates
        if ((int64_t)blockIdx.x >= P.gp.gather_blocks) {  // block-uniform
            gate_block(P.gp, P.n_query, (int64_t)blockIdx.x - P.gp.gather_blocks, (int)(threadIdx.x >> 5),
                       (int)(threadIdx.x & 31));
            return;
        }
    }
    __shared__ uint64_t s_seed[kTables];
    constexpr bool kHashed = kMode == IDX_HASH || kMode == IDX_HASH_SHARD;
    if (kHashed) {
        if (threadIdx.x < kTables) s_seed[threadIdx.x] = P.hp.seeds[threadIdx.x];
        if (blockIdx.x == 0 && threadIdx.x == 0 && P.hp.last_n == 0 &&
            __ldg(P.hp.offs + P.hp.n_seqs) - __ldg(P.hp.offs) != P.hp.n_query)
            raise_error(ENGRAM_ERANGE);
        __syncthreads();
    }
    const int lane = threadIdx.x & 31;
    // A warp per query token; in the few-token form with gates a warp per
    // (token, module), whose scale shuffles wait until its row loads are out:
    // one memory round trip instead of three on the latency-bound path.
    const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t t = kGate ? wid >> 1 : wid;
    const int m_first = kGate ? (int)(wid & 1) : 0;
    const int m_last = kGate ? m_first : 1;
    if (t >= P.n_query) return;

    // lanes 0..23: the 24 row offsets and fp32 scales of each module
    int64_t offm[2] = {0, 0};
    float scm[2] = {0.f, 0.f};
    int okm[2] = {0, 0};
    if (lane < kTablesPerModule) {
        int64_t rr[2];
        if (kHashed) {
            int64_t start, p;
            bool bad = !query_position(P.hp, t, start, p);
            if (!bad) hash_two(P.hp, s_seed[lane], s_seed[kTablesPerModule + lane], lane, start, p, bad, rr[0], rr[1]);
            if (bad) rr[0] = rr[1] = -1;
        }
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const int j = kTablesPerModule * m + lane;
            int64_t r;
            if (kHashed) {
                r = rr[m];
            } else if (kMode == IDX_I64) {
                r = __ldg(static_cast<const int64_t *>(P.idx) + t * kTables + j);
            } else {
                r = (int64_t)__ldg(static_cast<const int32_t *>(P.idx) + t * kTables + j);
            }
            int ok = (r >= 0 && r < P.R);
            // a staged query with no slot (kSlotNone: the dedup overflowed or its
            // index was out of range, both flagged there) contributes nothing
            if (!ok && !(kMode == IDX_STAGED_I32 && r == kSlotNone)) raise_error(ENGRAM_ERANGE);
            int64_t flat = (kMode == IDX_STAGED_I32) ? r : (int64_t)j * P.R + r;
            if (kMode == IDX_HASH_SHARD && ok) {  // another shard's row adds nothing here
                const int64_t k = r / P.n_shards;
                ok = (r - k * P.n_shards) == P.shard;
                flat = (int64_t)j * P.shard_rows + k;
            }
            okm[m] = ok;
            if (ok && m >= m_first && m <= m_last) {
                offm[m] = flat * P.row_stride;
                if (!kMx)
                    scm[m] = P.scales ? __ldg(P.scales + flat)
                                      : __ldg(reinterpret_cast<const float *>(P.rows + offm[m] + kRowBytes));
            }
        }
    }
    const int half = lane >> 4;
    const int c16 = lane & 15;
#pragma unroll 1
    for (int m = m_first; m <= m_last; ++m) {
        const int64_t off = m ? offm[1] : offm[0];
        const float sc = m ? scm[1] : scm[0];
        const int ok = m ? okm[1] : okm[0];
        uint4 v[12];
        float s[12];
        // kMx: lanes 0..11 of each half-warp load the 8 E8M0 bytes of row
        // 2 c16 + half in one 8-byte load; each lane later takes the byte of
        // the block holding its 16 codes (block c16 / 2) by shuffle
        uint2 tail = make_uint2(0u, 0u);
        if (kMx) {
            const int src = 2 * (c16 < 12 ? c16 : 11) + half;
            const int64_t o = __shfl_sync(0xffffffffu, off, src);
            const int okt = __shfl_sync(0xffffffffu, ok, src);
            if (c16 < 12 && okt) tail = __ldg(reinterpret_cast<const uint2 *>(P.rows + o + kRowBytes));
        }
#pragma unroll
        for (int i = 0; i < 12; ++i) {
            const int src = 2 * i + half;
            const int64_t o = __shfl_sync(0xffffffffu, off, src);
            if (!kMx && !kGate) s[i] = __shfl_sync(0xffffffffu, sc, src);
            v[i] = ld_nc_na_v4(P.rows + o + c16 * 16);  // an invalid row reads row offset 0 ...
            if (!__shfl_sync(0xffffffffu, ok, src)) {   // ... and is dropped (a finite scale times zero codes)
                v[i] = make_uint4(0, 0, 0, 0);
            }
        }
        if (kMx) {
            const int blk = c16 >> 1;
#pragma unroll
            for (int i = 0; i < 12; ++i) {
                const int L = half * 16 + i;  // the lane holding row 2 i + half's scale bytes
                const uint32_t x = __shfl_sync(0xffffffffu, tail.x, L);
                const uint32_t y = __shfl_sync(0xffffffffu, tail.y, L);
                s[i] = e8m0_to_float(((blk < 4 ? x : y) >> (8 * (blk & 3))) & 0xFFu);
            }
        }
        if (!kMx && kGate) {
#pragma unroll
            for (int i = 0; i < 12; ++i) s[i] = __shfl_sync(0xffffffffu, sc, 2 * i + half);
        }
        float acc[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) acc[k] = 0.f;
#pragma unroll
        for (int i = 0; i < 12; ++i) {
            const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 a = e4m3x2_to_float2((uint16_t)(w[q] & 0xFFFFu));
                const float2 b = e4m3x2_to_float2((uint16_t)(w[q] >> 16));
                acc[4 * q + 0] = fmaf(s[i], a.x, acc[4 * q + 0]);
                acc[4 * q + 1] = fmaf(s[i], a.y, acc[4 * q + 1]);
                acc[4 * q + 2] = fmaf(s[i], b.x, acc[4 * q + 2]);
                acc[4 * q + 3] = fmaf(s[i], b.y, acc[4 * q + 3]);
            }
        }
#pragma unroll
        for (int k = 0; k < 16; ++k) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], 16);
        const int64_t col = t * kMem + 256 * m + 16 * c16 + 8 * half;
        const float *a = acc + 8 * half;
        if (kBf16Out) {
            uint16_t *dst = static_cast<uint16_t *>(P.out) + col;
            *reinterpret_cast<uint4 *>(dst) = make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]),
                                                         pack_bf16x2(a[4], a[5]), pack_bf16x2(a[6], a[7]));
        } else {
            float *dst = static_cast<float *>(P.out) + col;
            reinterpret_cast<float4 *>(dst)[0] = make_float4(a[0], a[1], a[2], a[3]);
            reinterpret_cast<float4 *>(dst)[1] = make_float4(a[4], a[5], a[6], a[7]);
        }
    }
}

// ============================================================ gated gather ==
// One Engram layer's rows with per-row gates (the per-layer form): a warp per
// query token reads the 24 rows of module m (tables 24m..24m+23, hashed in
// place) and, for each row r_j (scale times e4m3 value), takes
//   rr_j = 1 / sqrt(mean(r_j^2) + eps),   s_j = rr_j <q_t, r_j> / 16,
//   g_j = sigmoid(s_j),                   X_t = bf16(sum_j g_j r_j)
// against the token's key-side query u_t = rinv(h_t) h_t W_q W_k^T
// (layer::query_kernel, twice).
// Lane (half, c16) holds 16 values of rows 2i + half; a row's sums are reduced
// over its half-warp; rows that failed the range check get gate 0.  Rows
// carry one fp32 scale (separate array or inside a 272-byte record) or, as
// MXFP8-style rows, eight E8M0 block scales.

constexpr int kLayerWidth = 256;  // values per row: the width of one Engram layer's X and query

struct GatedParams {
    const uint8_t *rows;
    const float *scales;  // fp32 [rows], or nullptr when each row carries its scale at byte 256
    int64_t row_stride;
    const float *q;       // [n_query][256]
    uint16_t *X;          // [n_query][256] bf16 out
    int64_t n_query;
    int64_t R;
    int32_t module;
    float eps;
    HashParams hp;
};

// kMx: MXFP8-style rows, eight E8M0 block scales at bytes 256..263; lane
// (half, c16) holds codes 16 c16 .. 16 c16 + 15, all in block c16 / 2, so
// each lane scales its own partial sums and codes by its block's scale.
template <bool kMx>
__global__ void __launch_bounds__(128, 5) gather_gated_kernel(const __grid_constant__ GatedParams P) {
    // For few tiles launched as a programmatic dependent of the key-side query
    // kernel, whose output u is read only after grid_dependency_wait below: the
    // hash and the row loads run while that kernel drains.  The projection
    // that reads X may in turn start early.
    allow_dependent_launch();
    __shared__ uint64_t s_seed[kTables];
    if (threadIdx.x < kTables) s_seed[threadIdx.x] = P.hp.seeds[threadIdx.x];
    if (blockIdx.x == 0 && threadIdx.x == 0 && P.hp.last_n == 0 &&
        __ldg(P.hp.offs + P.hp.n_seqs) - __ldg(P.hp.offs) != P.hp.n_query)
        raise_error(ENGRAM_ERANGE);
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= P.n_query) return;

    int64_t off = 0;
    float sc = 0.f;
    int ok = 0;
    if (lane < kTablesPerModule) {
        const int j = kTablesPerModule * P.module + lane;
        int64_t start, pos;
        bool bad = !query_position(P.hp, t, start, pos);
        int64_t r = bad ? -1 : hash_one(P.hp, s_seed[j], j, start, pos, bad);
        if (bad) r = -1;
        ok = (r >= 0 && r < P.R);
        if (!ok) raise_error(ENGRAM_ERANGE);
        if (ok) {
            const int64_t flat = (int64_t)j * P.R + r;
            off = flat * P.row_stride;
            if (!kMx)
                sc = P.scales ? __ldg(P.scales + flat)
                              : __ldg(reinterpret_cast<const float *>(P.rows + off + kRowBytes));
        }
    }
    const int half = lane >> 4;
    const int c16 = lane & 15;
    uint4 v[12];
    float s[12];  // the row's scale, or with kMx this lane's block scale of the row
    uint32_t live = 0;  // bit i: row 2i + half passed the range check
    uint2 tail = make_uint2(0u, 0u);
    if (kMx) {  // lanes 0..11 of each half-warp: the 8 scale bytes of row 2 c16 + half
        const int src = 2 * (c16 < 12 ? c16 : 11) + half;
        const int64_t o = __shfl_sync(0xffffffffu, off, src);
        const int okt = __shfl_sync(0xffffffffu, ok, src);
        if (c16 < 12 && okt) tail = __ldg(reinterpret_cast<const uint2 *>(P.rows + o + kRowBytes));
    }
#pragma unroll
    for (int i = 0; i < 12; ++i) {
        const int src = 2 * i + half;
        const int64_t o = __shfl_sync(0xffffffffu, off, src);
        if (!kMx) s[i] = __shfl_sync(0xffffffffu, sc, src);
        v[i] = ld_nc_na_v4(P.rows + o + c16 * 16);  // an invalid row reads row offset 0 and gets gate 0
        if (__shfl_sync(0xffffffffu, ok, src)) live |= 1u << i;
    }
    if (kMx) {
        const int blk = c16 >> 1;
#pragma unroll
        for (int i = 0; i < 12; ++i) {
            const int L = half * 16 + i;  // the lane holding row 2 i + half's scale bytes
            const uint32_t x = __shfl_sync(0xffffffffu, tail.x, L);
            const uint32_t y = __shfl_sync(0xffffffffu, tail.y, L);
            s[i] = e8m0_to_float(((blk < 4 ? x : y) >> (8 * (blk & 3))) & 0xFFu);
        }
    }
    grid_dependency_wait();  // u (P.q) is the previous kernel's output
    float qv[16];
    {
        const float4 *qp = reinterpret_cast<const float4 *>(P.q + t * kLayerWidth + c16 * 16);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float4 f = __ldg(qp + k);
            qv[4 * k] = f.x;
            qv[4 * k + 1] = f.y;
            qv[4 * k + 2] = f.z;
            qv[4 * k + 3] = f.w;
        }
    }
    // Per row, on the raw e4m3 values c (the row's scale s factors out):
    // sum(r^2) = s^2 sum(c^2), <u, r> = s <u, c>, and the gated sum takes
    // (g s) c.  Pairs of columns go through packed fp32 FMAs.
    float2 acc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = make_float2(0.f, 0.f);
    float2 u2[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) u2[k] = make_float2(qv[2 * k], qv[2 * k + 1]);
#pragma unroll
    for (int i = 0; i < 12; ++i) {
        float2 c[8];
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
            c[2 * q4] = e4m3x2_to_float2((uint16_t)(w[q4] & 0xFFFFu));
            c[2 * q4 + 1] = e4m3x2_to_float2((uint16_t)(w[q4] >> 16));
        }
        float2 ss2 = make_float2(0.f, 0.f), dd2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            ss2 = fma2(c[k], c[k], ss2);
            dd2 = fma2(c[k], u2[k], dd2);
        }
        float ss = ss2.x + ss2.y, dd = dd2.x + dd2.y;
        const float sc = s[i];
        if (kMx) {  // this lane's codes carry their block's scale
            ss *= sc * sc;
            dd *= sc;
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) {  // over the 16 lanes of this half-warp
            ss += __shfl_xor_sync(0xffffffffu, ss, o);
            dd += __shfl_xor_sync(0xffffffffu, dd, o);
        }
        const float score = kMx ? rsqrtf(ss * (1.f / 256.f) + P.eps) * dd * (1.f / 16.f)
                                : rsqrtf(sc * sc * ss * (1.f / 256.f) + P.eps) * sc * dd * (1.f / 16.f);
        const float gs = (live >> i) & 1u ? sc / (1.f + __expf(-score)) : 0.f;
        const float2 g2 = make_float2(gs, gs);
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k] = fma2(g2, c[k], acc[k]);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        acc[k].x += __shfl_xor_sync(0xffffffffu, acc[k].x, 16);
        acc[k].y += __shfl_xor_sync(0xffffffffu, acc[k].y, 16);
    }
    if (half == 0) {
        uint4 *dst = reinterpret_cast<uint4 *>(P.X + t * kLayerWidth + c16 * 16);
        dst[0] = make_uint4(pack_bf16x2(acc[0].x, acc[0].y), pack_bf16x2(acc[1].x, acc[1].y),
                            pack_bf16x2(acc[2].x, acc[2].y), pack_bf16x2(acc[3].x, acc[3].y));
        dst[1] = make_uint4(pack_bf16x2(acc[4].x, acc[4].y), pack_bf16x2(acc[5].x, acc[5].y),
                            pack_bf16x2(acc[6].x, acc[6].y), pack_bf16x2(acc[7].x, acc[7].y));
    }
}

// ==================================================================== dedup ==
// A bitmap over every (table, row) marks the rows the queries touch; an
// exclusive prefix of per-word popcounts gives each distinct row a dense
// slot, already sorted by (table, row); each query's index is then remapped
// to its slot.  Three passes over the bitmap words: per-block popcount sums,
// one-block scan of those sums, per-block word prefixes + the unique list.

constexpr int kScanThreads = 256;
constexpr int kScanWordsPerThread = 16;
constexpr int kScanWordsPerBlock = kScanThreads * kScanWordsPerThread;

__global__ void __launch_bounds__(256) dedup_mark_kernel(const int64_t *__restrict__ idx, int64_t n, int64_t R,
                                                         int64_t W, uint32_t *__restrict__ bitmap) {
    const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= n * kTables) return;
    const int j = (int)(g % kTables);
    const int64_t r = __ldg(idx + g);
    if (r < 0 || r >= R) {
        raise_error(ENGRAM_ERANGE);
        return;
    }
    atomicOr(bitmap + (int64_t)j * W + (r >> 5), 1u << (r & 31));
}

__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t x, uint32_t *total) {
    __shared__ uint32_t warp_sums[kScanThreads / 32];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    uint32_t incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_sums[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        uint32_t ws = lane < kScanThreads / 32 ? warp_sums[lane] : 0u;
        uint32_t wi = ws;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += y;
        }
        if (lane < kScanThreads / 32) warp_sums[lane] = wi - ws;
        if (lane == kScanThreads / 32 - 1) *total = wi;
    }
    __syncthreads();
    const uint32_t r = warp_sums[wid] + incl - x;
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(kScanThreads) dedup_count_kernel(const uint32_t *__restrict__ bitmap,
                                                                   int64_t n_words,
                                                                   uint32_t *__restrict__ block_sums) {
    const int64_t base = (int64_t)blockIdx.x * kScanWordsPerBlock + (int64_t)threadIdx.x * kScanWordsPerThread;
    uint32_t c = 0;
#pragma unroll
    for (int k = 0; k < kScanWordsPerThread; ++k)
        if (base + k < n_words) c += __popc(__ldg(bitmap + base + k));
    __shared__ uint32_t total;
    block_exclusive_scan(c, &total);
    if (threadIdx.x == 0) block_sums[blockIdx.x] = total;
}

__global__ void __launch_bounds__(kScanThreads) dedup_scan_blocks_kernel(uint32_t *__restrict__ block_sums,
                                                                         int64_t n_blocks, int64_t capacity,
                                                                         int64_t *__restrict__ n_unique) {
    __shared__ uint32_t total;
    uint32_t carry = 0;
    for (int64_t b0 = 0; b0 < n_blocks; b0 += kScanThreads) {
        const int64_t b = b0 + threadIdx.x;
        const uint32_t x = b < n_blocks ? block_sums[b] : 0u;
        const uint32_t ex = block_exclusive_scan(x, &total);
        if (b < n_blocks) block_sums[b] = carry + ex;
        carry += total;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        *n_unique = (int64_t)carry;
        if ((int64_t)carry > capacity) raise_error(ENGRAM_ECAPACITY);
    }
}

__global__ void __launch_bounds__(kScanThreads) dedup_emit_kernel(const uint32_t *__restrict__ bitmap,
                                                                  int64_t n_words, int64_t W, int64_t R,
                                                                  const uint32_t *__restrict__ block_offs,
                                                                  uint32_t *__restrict__ word_prefix,
                                                                  int64_t *__restrict__ unique,
                                                                  int64_t capacity) {
    const int64_t base = (int64_t)blockIdx.x * kScanWordsPerBlock + (int64_t)threadIdx.x * kScanWordsPerThread;
    uint32_t wv[kScanWordsPerThread];
    uint32_t c = 0;
#pragma unroll
    for (int k = 0; k < kScanWordsPerThread; ++k) {
        wv[k] = base + k < n_words ? __ldg(bitmap + base + k) : 0u;
        c += __popc(wv[k]);
    }
    __shared__ uint32_t total;
    uint32_t pre = block_offs[blockIdx.x] + block_exclusive_scan(c, &total);
#pragma unroll
    for (int k = 0; k < kScanWordsPerThread; ++k) {
        const int64_t w = base + k;
        if (w >= n_words) break;
        word_prefix[w] = pre;
        uint32_t bits = wv[k];
        const int64_t j = w / W;
        const int64_t row0 = (w - j * W) * 32;
        uint32_t slot = pre;
        while (bits) {
            const int b = __ffs(bits) - 1;
            bits &= bits - 1;
            if ((int64_t)slot < capacity) unique[slot] = j * R + row0 + b;
            ++slot;
        }
        pre += __popc(wv[k]);
    }
}

// Slot of each (query, table); kSlotNone for a row index out of range, and
// for every query when the distinct rows overflowed the capacity (then nothing
// is staged and the staged gather reads no row at all).
__global__ void __launch_bounds__(256) dedup_remap_kernel(const int64_t *__restrict__ idx, int64_t n, int64_t R,
                                                          int64_t W, const uint32_t *__restrict__ bitmap,
                                                          const uint32_t *__restrict__ word_prefix,
                                                          const int64_t *__restrict__ n_unique, int64_t capacity,
                                                          int32_t *__restrict__ idx_staged) {
    const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= n * kTables) return;
    const int j = (int)(g % kTables);
    const int64_t r = __ldg(idx + g);
    int32_t slot = kSlotNone;
    if (r >= 0 && r < R && *n_unique <= capacity) {
        const int64_t w = (int64_t)j * W + (r >> 5);
        const uint32_t below = __ldg(bitmap + w) & ((1u << (r & 31)) - 1u);
        slot = (int32_t)((int64_t)__ldg(word_prefix + w) + __popc(below));
    }
    idx_staged[g] = slot;
}

// ==================================================================== stage ==
// Copy unique rows (and their scales) from host tables into device staging.
// Each half-warp moves one 256-byte row with 16-byte loads; a warp keeps eight
// row pairs in flight, and the grid strides over the unique list.

// kWhole: rows carrying block scales are staged whole (host_stride bytes).
// dest: where list entry u goes in the staging buffers (nullptr: slot u).
template <bool kWhole>
__global__ void __launch_bounds__(256) stage_kernel(const uint8_t *__restrict__ host_tables,
                                                    const float *__restrict__ host_scales, int64_t host_stride,
                                                    const int64_t *__restrict__ unique,
                                                    const int64_t *__restrict__ n_unique, int64_t capacity,
                                                    uint8_t *__restrict__ staged, float *__restrict__ staged_scales,
                                                    const int32_t *__restrict__ dest = nullptr) {
    const int64_t U = *n_unique;
    if (U > capacity) return;  // overflowed: the dedup flagged it and left no query pointing at a slot
    auto D = [&](int64_t u) -> int64_t { return dest ? (int64_t)__ldg(dest + u) : u; };
    const int lane = threadIdx.x & 31;
    const int half = lane >> 4, c16 = lane & 15;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    constexpr int kPairs = 8;
    for (int64_t u0 = warp * 2 * kPairs; u0 < U; u0 += n_warps * 2 * kPairs) {
        uint4 v[kPairs];
        int64_t flat[kPairs];
#pragma unroll
        for (int k = 0; k < kPairs; ++k) {
            const int64_t u = u0 + 2 * k + half;
            flat[k] = u < U ? __ldg(unique + u) : -1;
            v[k] = flat[k] >= 0 ? *reinterpret_cast<const uint4 *>(host_tables + flat[k] * host_stride + c16 * 16)
                                : make_uint4(0, 0, 0, 0);
        }
        if constexpr (kWhole) {  // each row's 16-byte tail too: lane c16 < kPairs takes that of pair c16
            const int64_t ut = u0 + 2 * c16 + half;
            const bool has_tail = c16 < kPairs && ut < U;
            uint4 tail = make_uint4(0, 0, 0, 0);
            if (has_tail)
                tail = *reinterpret_cast<const uint4 *>(host_tables + __ldg(unique + ut) * host_stride + kRowBytes);
#pragma unroll
            for (int k = 0; k < kPairs; ++k) {
                const int64_t u = u0 + 2 * k + half;
                if (flat[k] >= 0) *reinterpret_cast<uint4 *>(staged + D(u) * host_stride + c16 * 16) = v[k];
            }
            if (has_tail) *reinterpret_cast<uint4 *>(staged + D(ut) * host_stride + kRowBytes) = tail;
        } else {
            float sc[kPairs];
#pragma unroll
            for (int k = 0; k < kPairs; ++k)
                sc[k] = (c16 == 0 && flat[k] >= 0)
                            ? (host_scales ? host_scales[flat[k]]
                                           : *reinterpret_cast<const float *>(host_tables + flat[k] * host_stride +
                                                                              kRowBytes))
                            : 0.f;
#pragma unroll
            for (int k = 0; k < kPairs; ++k) {
                const int64_t u = u0 + 2 * k + half;
                if (flat[k] >= 0) {
                    const int64_t du = D(u);
                    *reinterpret_cast<uint4 *>(staged + du * kRowBytes + c16 * 16) = v[k];
                    if (c16 == 0) staged_scales[du] = sc[k];
                }
            }
        }
    }
}

// =========================================================== row cache ==
// Staged rows kept in HBM across calls (the hot rows of a Zipf token stream
// are pulled over the host link once).  A direct-mapped cache of `slots`
// rows (a power of two): row f lives in slot (f * 0x9E3779B97F4A7C15) >> (64 -
// log2 slots), tagged with f.  Per call, each distinct row u of the batch
// claims its slot with the call's stamp (atomicMax on the slot's claim word;
// stamps increase from call to call): the first claimer of a slot this call
// either finds its row there (a hit: nothing to stage) or takes the slot over
// (a miss: staged into it, tag replaced); a row whose slot another row of the
// same call already claimed is staged into the overflow rows after the
// cache (slot `slots` + k).  where[u] is the row's slot for the gather.

__device__ __forceinline__ int64_t cache_slot(int64_t flat, int log2_slots) {
    return (int64_t)(((uint64_t)flat * kGolden) >> (64 - log2_slots));
}

__global__ void __launch_bounds__(256) cache_lookup_kernel(const int64_t *__restrict__ unique,
                                                           const int64_t *__restrict__ n_unique, int64_t capacity,
                                                           int64_t *__restrict__ tags, uint32_t *__restrict__ claims,
                                                           int log2_slots, uint32_t stamp, int32_t *__restrict__ where,
                                                           int64_t *__restrict__ stage_flat,
                                                           int32_t *__restrict__ stage_dest,
                                                           int64_t *__restrict__ stats) {
    // stats: [0] distinct rows, [1] cache hits, [2] rows to stage, [3] overflow rows
    const int64_t U = *n_unique;
    if (blockIdx.x == 0 && threadIdx.x == 0) stats[0] = U;
    if (U > capacity) return;  // the dedup overflowed and flagged it: nothing is staged or read
    const int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int lane = threadIdx.x & 31;
    bool hit = false, stage = false, over = false;
    int64_t flat = 0, dst = 0;
    if (u < U) {
        flat = __ldg(unique + u);
        const int64_t s = cache_slot(flat, log2_slots);
        const uint32_t old = atomicMax(claims + s, stamp);
        if (old < stamp) {  // first this call: the slot is ours
            dst = s;
            if (tags[s] == flat) {
                hit = true;
            } else {
                tags[s] = flat;
                stage = true;
            }
        } else {
            over = true;
            stage = true;
        }
    }
    // counters and stage-list positions: lanes within the warp (ballots),
    // warps within the block (shared memory), one global atomic per block
    __shared__ unsigned s_cnt[3];        // over, stage, hit: this block's totals
    __shared__ unsigned long long s_base[2];
    if (threadIdx.x < 3) s_cnt[threadIdx.x] = 0;
    __syncthreads();
    const unsigned m_over = __ballot_sync(0xffffffffu, over);
    const unsigned m_stage = __ballot_sync(0xffffffffu, stage);
    const unsigned m_hit = __ballot_sync(0xffffffffu, hit);
    unsigned w_over = 0, w_stage = 0;
    if (lane == 0) {
        w_over = atomicAdd(&s_cnt[0], (unsigned)__popc(m_over));
        w_stage = atomicAdd(&s_cnt[1], (unsigned)__popc(m_stage));
        atomicAdd(&s_cnt[2], (unsigned)__popc(m_hit));
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        s_base[0] = s_cnt[0] ? atomicAdd(reinterpret_cast<unsigned long long *>(stats + 3), (unsigned long long)s_cnt[0]) : 0;
        s_base[1] = s_cnt[1] ? atomicAdd(reinterpret_cast<unsigned long long *>(stats + 2), (unsigned long long)s_cnt[1]) : 0;
        if (s_cnt[2]) atomicAdd(reinterpret_cast<unsigned long long *>(stats + 1), (unsigned long long)s_cnt[2]);
    }
    __syncthreads();
    w_over = __shfl_sync(0xffffffffu, w_over, 0);
    w_stage = __shfl_sync(0xffffffffu, w_stage, 0);
    const unsigned below = (1u << lane) - 1u;
    if (over) dst = ((int64_t)1 << log2_slots) + (int64_t)(s_base[0] + w_over + __popc(m_over & below));
    if (u < U) where[u] = (int32_t)dst;
    if (stage) {
        const int64_t k = (int64_t)(s_base[1] + w_stage + __popc(m_stage & below));
        stage_flat[k] = flat;
        stage_dest[k] = (int32_t)dst;
    }
}

// idx_staged (dedup slots) -> cache slots
__global__ void __launch_bounds__(256) cache_remap_kernel(int32_t *__restrict__ idx_staged, int64_t n,
                                                          const int32_t *__restrict__ where) {
    const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= n) return;
    const int32_t u = idx_staged[g];
    idx_staged[g] = u >= 0 ? __ldg(where + u) : kSlotNone;
}

__global__ void cache_reset_kernel(int64_t *__restrict__ tags, uint32_t *__restrict__ claims, int64_t slots) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < slots; i += (int64_t)gridDim.x * blockDim.x) {
        tags[i] = -1;
        claims[i] = 0;
    }
}

// ================================================================ host side ==

// Per-device host caches below are relaxed atomics: host threads that reach a
// first call together compute and store the same value.
int num_sms() {
    static std::atomic<int> sms[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 148;
    int n = sms[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        n = v > 0 ? v : 148;
        sms[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

static bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

engram_status check_config(const engram_config *cfg) {
    if (!cfg) return ENGRAM_EINVAL;
    if (cfg->vocab < 1 || cfg->rows < 1 || cfg->d_model < 0) return ENGRAM_EINVAL;
    if (cfg->row_layout > ENGRAM_ROWS_MX) return ENGRAM_EINVAL;
    return ENGRAM_OK;
}

static bool records(const engram_config *cfg) { return cfg->row_layout != ENGRAM_ROWS_SEPARATE; }
static bool mx(const engram_config *cfg) { return cfg->row_layout == ENGRAM_ROWS_MX; }
// staging: MX rows are staged whole; the other layouts as 256-byte rows + fp32 scales
static int64_t staged_stride(const engram_config *cfg) { return mx(cfg) ? ENGRAM_RECORD_BYTES : kRowBytes; }
static int64_t row_stride(const engram_config *cfg) { return records(cfg) ? ENGRAM_RECORD_BYTES : kRowBytes; }
// The scales argument as the kernels see it: nullptr when rows carry their scale.
static const float *scales_arg(const engram_config *cfg, const float *scales) { return records(cfg) ? nullptr : scales; }
static bool scales_ok(const engram_config *cfg, const float *scales) {
    return records(cfg) || (scales && (reinterpret_cast<uintptr_t>(scales) % 4) == 0);
}

// With ENGRAM_DEBUG set in the environment, failed CUDA calls are reported on
// stderr with the call site (the status returned is the same either way).
static engram_status cuda_fail(cudaError_t e, const char *what) {
    static const bool debug = getenv("ENGRAM_DEBUG") != nullptr;
    if (debug) fprintf(stderr, "libengram: %s failed: %s\n", what, cudaGetErrorString(e));
    return ENGRAM_ECUDA;
}

// Opt a kernel in to `bytes` of dynamic shared memory once per device.
static engram_status ensure_smem(const void *kern, int bytes, std::atomic<bool> *attr_done) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_done[dev].load(std::memory_order_relaxed)) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(smem)");
        if (dev >= 0 && dev < 64) attr_done[dev].store(true, std::memory_order_relaxed);
    }
    return ENGRAM_OK;
}

engram_status launch_status() {
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ENGRAM_OK : cuda_fail(e, "kernel launch");
}

static void fill_hash_params(HashParams &a, const engram_config *cfg, const int32_t *tokens, const int64_t *offs,
                             int64_t n_seqs, int32_t last_n, int64_t n_query);

engram_status hash_launch(const engram_config *cfg, const int32_t *tokens, const int64_t *offs, int64_t n_seqs,
                          int32_t last_n, int64_t n_query, int64_t *idx, cudaStream_t st) {
    HashParams a;
    fill_hash_params(a, cfg, tokens, offs, n_seqs, last_n, n_query);
    const int64_t threads = n_query * kTables;
    const int64_t blocks = (threads + 255) / 256;
    hash_kernel<<<(unsigned)blocks, 256, 0, st>>>(a, idx);
    return launch_status();
}

static void fill_hash_params(HashParams &a, const engram_config *cfg, const int32_t *tokens, const int64_t *offs,
                             int64_t n_seqs, int32_t last_n, int64_t n_query) {
    a.tokens = tokens;
    a.offs = offs;
    a.n_seqs = n_seqs;
    a.n_query = n_query;
    a.R = (uint64_t)cfg->rows;
    a.pow2 = (cfg->rows & (cfg->rows - 1)) == 0;
    a.rmask = (uint64_t)cfg->rows - 1;
    a.V = cfg->vocab;
    a.last_n = last_n;
    memcpy(a.seeds, cfg->seeds, sizeof(a.seeds));
}

// mode: IDX_I64 / IDX_STAGED_I32 / IDX_HASH; out: fp32 mem or bf16 X.
// mx: rows carry eight E8M0 block scales at byte 256 (scales unused).
engram_status gather_launch(int mode, bool bf16_out, const uint8_t *rows, const float *scales, int64_t stride,
                            bool mx, const void *idx, const HashParams *hp, int64_t n_query, int64_t R, void *out,
                            cudaStream_t st, int64_t shard_rows = 0, int32_t shard = 0, int32_t n_shards = 1) {
    GatherParams P;
    memset(&P, 0, sizeof(P));
    P.rows = rows;
    P.scales = scales;
    P.row_stride = stride;
    P.idx = idx;
    P.n_query = n_query;
    P.R = R;
    P.out = out;
    if (hp) P.hp = *hp;
    const int64_t warps = n_query;
    const unsigned blocks = (unsigned)((warps * 32 + 255) / 256);
#define ENGRAM_GATHER(M, B)                                         \
    do {                                                             \
        if (mx)                                                      \
            gather_kernel<M, B, true><<<blocks, 256, 0, st>>>(P);    \
        else                                                         \
            gather_kernel<M, B, false><<<blocks, 256, 0, st>>>(P);   \
    } while (0)
    if (mode == IDX_HASH_SHARD) {  // fp32 partial sums only
        P.shard_rows = shard_rows;
        P.shard = shard;
        P.n_shards = n_shards;
        ENGRAM_GATHER(IDX_HASH_SHARD, false);
    } else if (mode == IDX_I64) {
        if (bf16_out) ENGRAM_GATHER(IDX_I64, true); else ENGRAM_GATHER(IDX_I64, false);
    } else if (mode == IDX_STAGED_I32) {
        if (bf16_out) ENGRAM_GATHER(IDX_STAGED_I32, true); else ENGRAM_GATHER(IDX_STAGED_I32, false);
    } else {
        if (bf16_out) ENGRAM_GATHER(IDX_HASH, true); else ENGRAM_GATHER(IDX_HASH, false);
    }
#undef ENGRAM_GATHER
    return launch_status();
}

// dedup workspace: bitmap [48*W] u32 | word_prefix [48*W] u32 | block sums
struct DedupLayout {
    int64_t W, n_words, n_blocks;
    size_t off_bitmap, off_prefix, off_blocks, total;
};

static size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static DedupLayout dedup_layout(const engram_config *cfg) {
    DedupLayout L;
    L.W = (cfg->rows + 31) / 32;
    L.n_words = L.W * kTables;
    L.n_blocks = (L.n_words + kScanWordsPerBlock - 1) / kScanWordsPerBlock;
    L.off_bitmap = 0;
    L.off_prefix = round_up((size_t)L.n_words * 4, 256);
    L.off_blocks = L.off_prefix + round_up((size_t)L.n_words * 4, 256);
    L.total = L.off_blocks + round_up((size_t)L.n_blocks * 4, 256);
    return L;
}

size_t dedup_bytes(const engram_config *cfg) { return dedup_layout(cfg).total; }

engram_status dedup_launch(const engram_config *cfg, const int64_t *idx, int64_t n_query, void *ws,
                           int64_t *unique, int64_t capacity, int32_t *idx_staged, int64_t *n_unique,
                           cudaStream_t st) {
    const DedupLayout L = dedup_layout(cfg);
    uint8_t *base = static_cast<uint8_t *>(ws);
    uint32_t *bitmap = reinterpret_cast<uint32_t *>(base + L.off_bitmap);
    uint32_t *prefix = reinterpret_cast<uint32_t *>(base + L.off_prefix);
    uint32_t *blocks = reinterpret_cast<uint32_t *>(base + L.off_blocks);
    if (cudaMemsetAsync(bitmap, 0, (size_t)L.n_words * 4, st) != cudaSuccess) return ENGRAM_ECUDA;
    const int64_t n = n_query * kTables;
    const unsigned gb = (unsigned)((n + 255) / 256);
    if (n > 0) dedup_mark_kernel<<<gb, 256, 0, st>>>(idx, n_query, cfg->rows, L.W, bitmap);
    dedup_count_kernel<<<(unsigned)L.n_blocks, kScanThreads, 0, st>>>(bitmap, L.n_words, blocks);
    dedup_scan_blocks_kernel<<<1, kScanThreads, 0, st>>>(blocks, L.n_blocks, capacity, n_unique);
    dedup_emit_kernel<<<(unsigned)L.n_blocks, kScanThreads, 0, st>>>(bitmap, L.n_words, L.W, cfg->rows, blocks,
                                                                      prefix, unique, capacity);
    if (n > 0)
        dedup_remap_kernel<<<gb, 256, 0, st>>>(idx, n_query, cfg->rows, L.W, bitmap, prefix, n_unique, capacity,
                                               idx_staged);
    return launch_status();
}

// whole_rows: stage host_stride-byte rows as they are (MX rows); otherwise
// 256-byte rows plus fp32 scales.
engram_status stage_launch(const uint8_t *host_tables, const float *host_scales, int64_t host_stride,
                           bool whole_rows, const int64_t *unique, const int64_t *n_unique, int64_t capacity,
                           uint8_t *staged, float *staged_scales, cudaStream_t st, const int32_t *dest = nullptr) {
    const int blocks = num_sms() * 8;
    if (whole_rows)
        stage_kernel<true><<<blocks, 256, 0, st>>>(host_tables, host_scales, host_stride, unique, n_unique, capacity,
                                                   staged, staged_scales, dest);
    else
        stage_kernel<false><<<blocks, 256, 0, st>>>(host_tables, host_scales, host_stride, unique, n_unique, capacity,
                                                    staged, staged_scales, dest);
    return launch_status();
}


// ----------------------------------------------------------- fuse launcher --

static PFN_cuTensorMapEncodeTiled_v12000 tensormap_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// 2-D bf16 tensor [outer][inner] (inner contiguous), box [box_outer][box_inner],
// 128-byte swizzle (a box row of 64 bf16 is one swizzle span) or 64-byte
// swizzle (box rows of 32 bf16).
static bool bf16_map_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                        uint32_t box_outer, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    auto enc = tensormap_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// CTAs per cluster (d slices) for a projection of m_tiles tiles and n_chunks
// 256-column chunks.  A slice must be 1, 2, 4, 8 or 16 chunks (the kernel's
// CPG) and a cluster at most 8 CTAs.  Many tiles: slices of 4 chunks (each
// CTA's h slice stays small in L2, clusters stay small).  Few tiles: spread
// d over as many CTAs as fit.  Returns 0 if d has no valid split.
static int pick_groups(int64_t m_tiles, int n_chunks) {
    const int sms = num_sms();
    int best = 0;
    double best_score = 1e30;
    for (int g = 1; g <= fuse::MAX_GROUPS; ++g) {
        if (n_chunks % g) continue;
        const int cpg = n_chunks / g;
        if (cpg != 1 && cpg != 2 && cpg != 4 && cpg != 8 && cpg != 16) continue;
        double score;
        if (m_tiles * 2 >= sms)
            score = fabs(log2((double)cpg) - 2.0) * 100.0 + g;  // prefer 4 chunks per CTA, then fewer CTAs
        else
            score = (m_tiles * g <= sms ? 0.0 : 1000.0) - g;     // prefer more CTAs while they fit
        if (score < best_score) {
            best_score = score;
            best = g;
        }
    }
    return best;
}

// Projection kernels: X converted from fp32 mem in the kernel (fuse.cuh);
// X by TMA with the gate on its own warps (fuse2.cuh, many tiles); X by TMA
// with the h slice held in shared memory (fuse3.cuh, few tiles: d slices of 1
// or 2 chunks).  For the same split of d all three give the same bits.
enum FuseKind { FUSE_F32_MEM = 0, FUSE_BF16_X_GATE_WARPS = 2, FUSE_LAYER = 3 };

// Persistent cluster launch: as many clusters of `groups` CTAs as fit at once
// (cached per device and cluster size in *max_clusters), each striding over
// the tiles.  attr_done / max_clusters belong to one kernel instantiation.
// pdl: launch as a programmatic dependent of the previous kernel in the
// stream (only after a gather kernel, which writes X and nothing the
// projection reads before its grid_dependency_wait).
template <typename Kern, typename... Args>
static engram_status launch_persistent(Kern kern, int threads, int smem, int groups, int64_t m_tiles,
                                       std::atomic<bool> *attr_done,
                                       std::atomic<int> (*max_clusters)[fuse::MAX_GROUPS + 1], cudaStream_t st,
                                       bool pdl, const Args &...args) {
    int dev = 0;
    cudaGetDevice(&dev);
    const bool cache = dev >= 0 && dev < 64;
    if (!cache || !attr_done[dev].load(std::memory_order_relaxed)) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(fuse smem)");
        if (cache) attr_done[dev].store(true, std::memory_order_relaxed);
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = groups;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int mc = cache ? max_clusters[dev][groups].load(std::memory_order_relaxed) : 0;
    if (mc == 0) {
        cfg.gridDim = dim3(groups * 64);
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = num_sms() / groups;
        }
        mc = n;
        if (cache) max_clusters[dev][groups].store(n, std::memory_order_relaxed);
    }
    const int64_t clusters = std::min<int64_t>(m_tiles, mc);
    cfg.gridDim = dim3((unsigned)(clusters * groups));
    if (pdl) cfg.numAttrs = 2;
    const cudaError_t le = cudaLaunchKernelEx(&cfg, kern, args...);
    if (le != cudaSuccess) return cuda_fail(le, "cudaLaunchKernelEx(fuse)");
    return launch_status();
}

template <int KIND, int CPG>
static auto fuse_kernel_for() {
    if constexpr (KIND == FUSE_F32_MEM)
        return fuse::fuse_kernel<fuse::X_FROM_F32_MEM, CPG>;
    else if constexpr (KIND == FUSE_LAYER)
        return fuse2::fuse2_kernel<CPG, kLayerWidth / fuse::BK, false>;  // one layer's [T,256] X, no token gate
    else
        return fuse2::fuse2_kernel<CPG>;
}

template <int KIND, int CPG>
static engram_status fuse_launch_t(const CUtensorMap &wmap, const CUtensorMap &xmap, const CUtensorMap &hmap,
                                   const fuse::Params &p, cudaStream_t st, bool pdl) {
    constexpr bool k2 = KIND == FUSE_BF16_X_GATE_WARPS || KIND == FUSE_LAYER;
    constexpr int kThreads = k2 ? fuse2::NUM_THREADS : fuse::NUM_THREADS;
    constexpr int kSmem = k2 ? fuse2::SMEM_BYTES : fuse::SMEM_BYTES;
    static std::atomic<bool> attr_done[64] = {};
    static std::atomic<int> max_clusters[64][fuse::MAX_GROUPS + 1] = {};
    if constexpr (k2)
        return launch_persistent(fuse_kernel_for<KIND, CPG>(), kThreads, kSmem, p.groups, p.m_tiles, attr_done,
                                 max_clusters, st, pdl, wmap, xmap, hmap, p);
    else
        return launch_persistent(fuse_kernel_for<KIND, CPG>(), kThreads, kSmem, p.groups, p.m_tiles, attr_done,
                                 max_clusters, st, pdl, wmap, xmap, p);
}

template <int KIND>
static engram_status fuse_dispatch(const CUtensorMap &wmap, const CUtensorMap &xmap, const CUtensorMap &hmap,
                                   const fuse::Params &p, cudaStream_t st, bool pdl = false) {
    switch (p.cpg) {
        case 1: return fuse_launch_t<KIND, 1>(wmap, xmap, hmap, p, st, pdl);
        case 2: return fuse_launch_t<KIND, 2>(wmap, xmap, hmap, p, st, pdl);
        case 4: return fuse_launch_t<KIND, 4>(wmap, xmap, hmap, p, st, pdl);
        case 8: return fuse_launch_t<KIND, 8>(wmap, xmap, hmap, p, st, pdl);
        case 16: return fuse_launch_t<KIND, 16>(wmap, xmap, hmap, p, st, pdl);
    }
    return ENGRAM_EINVAL;
}

template <int CPG>
static engram_status fuse3_launch_t(const CUtensorMap &wmap, const CUtensorMap &xmap, const CUtensorMap &hl,
                                    const CUtensorMap &hs, const fuse::Params &p, cudaStream_t st, bool pdl) {
    static std::atomic<bool> attr_done[64] = {};
    static std::atomic<int> max_clusters[64][fuse::MAX_GROUPS + 1] = {};
    return launch_persistent(fuse3::fuse3_kernel<CPG>, fuse3::NUM_THREADS, fuse3::smem_bytes<CPG>(), p.groups,
                             p.m_tiles, attr_done, max_clusters, st, pdl, wmap, xmap, hl, hs, p);
}

// One or two tiles: the h-resident kernel, with d split into slices of 1
// chunk if that fits a cluster of 8, else 2.  Returns its chunks per CTA, or
// 0 to use the other kernels (more tiles, or d too wide).  From 3 tiles on
// fuse2 is as fast or faster at every size measured (d = 4096: 384 tokens
// 20.0 against 22.4 us, 4,096 tokens 46 against 58 us, 8,192 tokens 87
// against 102 us); `engram_forward` sends 1-2 tiles to the d-split kernel,
// which takes this split for its gates.
static int pick_cpg_h_resident(int64_t m_tiles, int n_chunks) {
    if (m_tiles >= 3) return 0;
    if (n_chunks <= fuse::MAX_GROUPS) return 1;
    if (n_chunks % 2 == 0 && n_chunks / 2 <= fuse::MAX_GROUPS) return 2;
    return 0;
}

static bool fuse_split(int64_t m_tiles, int n_chunks, int *groups, int *cpg);

// y = X @ W_out and the gated residual update.  X comes either from fp32 mem
// (converted in the kernel) or from a bf16 [n_query][512] tensor via TMA.
// split_tiles > 0: choose the kernel and the split of d as for a batch of
// split_tiles tiles (a chunk of a larger batch then gives that batch's bits).
// pdl (bf16 X only): launch as a programmatic dependent of the gather kernel
// that was just enqueued on `st` and writes X.
engram_status fuse_launch(const engram_config *cfg, const float *mem, const uint16_t *x_bf16, const uint16_t *W,
                          const uint16_t *g, uint16_t *h, int64_t n_query, cudaStream_t st, int64_t split_tiles = 0,
                          bool pdl = false) {
    const int d = cfg->d_model;
    const int n_chunks = d / fuse::BN;
    fuse::Params p;
    p.mem = mem;
    p.g = g;
    p.h = h;
    p.n_query = n_query;
    p.m_tiles = (n_query + fuse::BM - 1) / fuse::BM;
    p.d = d;
    // One split of d for both inputs (fp32 mem or bf16 X), so they agree bit for bit.
    const int64_t tiles_for_split = split_tiles > 0 ? split_tiles : p.m_tiles;
    const int cpg3 = pick_cpg_h_resident(tiles_for_split, n_chunks);
    if (!fuse_split(tiles_for_split, n_chunks, &p.groups, &p.cpg)) return ENGRAM_EINVAL;
    p.eps = cfg->rms_eps;
    p.inv_sqrt_d = 1.0f / sqrtf((float)d);
    CUtensorMap wmap, xmap;
    memset(&xmap, 0, sizeof(xmap));
    // W boxes: 64 columns x WBK K-rows (fuse.cuh) or x BK K-rows (fuse2.cuh and
    // fuse3.cuh, one ring stage)
    const uint32_t w_box_rows = x_bf16 ? fuse::BK : fuse::WBK;
    if (!bf16_map_2d(&wmap, W, (uint64_t)d, kMem, 64, w_box_rows)) return cuda_fail(cudaErrorInvalidValue, "W tensor map");
    if (x_bf16) {
        if (!bf16_map_2d(&xmap, x_bf16, kMem, (uint64_t)n_query, fuse::BK, fuse::BM))
            return cuda_fail(cudaErrorInvalidValue, "X tensor map");
        if (cpg3 == 0) {  // h pieces of 64 columns x 32 tokens for the update warps' TMA loads and stores
            CUtensorMap hp;
            if (!bf16_map_2d(&hp, h, (uint64_t)d, (uint64_t)n_query, 64, 32))
                return cuda_fail(cudaErrorInvalidValue, "h piece map");
            return fuse_dispatch<FUSE_BF16_X_GATE_WARPS>(wmap, xmap, hp, p, st, pdl);
        }
        {
            CUtensorMap hl, hs;  // h slice boxes: 64 columns x 128 tokens (loads) / x 32 tokens (stores)
            if (!bf16_map_2d(&hl, h, (uint64_t)d, (uint64_t)n_query, 64, fuse::BM) ||
                !bf16_map_2d(&hs, h, (uint64_t)d, (uint64_t)n_query, 64, 32))
                return cuda_fail(cudaErrorInvalidValue, "h tensor map");
            return cpg3 == 1 ? fuse3_launch_t<1>(wmap, xmap, hl, hs, p, st, pdl)
                             : fuse3_launch_t<2>(wmap, xmap, hl, hs, p, st, pdl);
        }
    }
    return fuse_dispatch<FUSE_F32_MEM>(wmap, xmap, xmap, p, st);
}

static engram_status narrow_layer_launch(const engram_config *cfg, const uint16_t *X, const uint16_t *W, uint16_t *h,
                                         int64_t n_query, cudaStream_t st);
static bool narrow_fits(int64_t m_tiles, int d);

// One Engram layer's projection: h = bf16(h + X W_m), X [n][256] bf16,
// W_m [256][d] (fuse2 with 4 K-blocks and no token gate; the d-split kernel
// when the batch fits one wave of 64-column CTAs).
static int query_splits(int64_t m_tiles, int k);
static engram_status layer_projection_launch(const engram_config *cfg, const uint16_t *X, const uint16_t *W,
                                             uint16_t *h, int64_t n_query, cudaStream_t st) {
    const int d = cfg->d_model;
    if (narrow_fits((n_query + fuse::BM - 1) / fuse::BM, d)) return narrow_layer_launch(cfg, X, W, h, n_query, st);
    const int n_chunks = d / fuse::BN;
    fuse::Params p;
    memset(&p, 0, sizeof(p));
    p.h = h;
    p.n_query = n_query;
    p.m_tiles = (n_query + fuse::BM - 1) / fuse::BM;
    p.d = d;
    p.groups = pick_groups(p.m_tiles, n_chunks);
    if (p.groups == 0) return ENGRAM_EINVAL;
    p.cpg = n_chunks / p.groups;
    p.eps = cfg->rms_eps;
    p.inv_sqrt_d = 1.0f / sqrtf((float)d);
    CUtensorMap wmap, xmap;
    if (!bf16_map_2d(&wmap, W, (uint64_t)d, kLayerWidth, 64, fuse::BK)) return cuda_fail(cudaErrorInvalidValue, "W_m map");
    if (!bf16_map_2d(&xmap, X, kLayerWidth, (uint64_t)n_query, fuse::BK, fuse::BM))
        return cuda_fail(cudaErrorInvalidValue, "layer X map");
    CUtensorMap hp;
    if (!bf16_map_2d(&hp, h, (uint64_t)d, (uint64_t)n_query, 64, 32)) return cuda_fail(cudaErrorInvalidValue, "h piece map");
    // a programmatic dependent of the gated gather in the same batch range
    // (its producer waits for X; the update warps read only h before that)
    return fuse_dispatch<FUSE_LAYER>(wmap, xmap, hp, p, st, query_splits(p.m_tiles, d) > 1);
}

// out = s * (A @ B) on tcgen05 (layer::query_kernel): A bf16 [n][K], B bf16
// [K][256]; with RMS s = rinv(A row), with SPLIT out is bf16 [n][512] (hi | lo)
// instead of fp32 [n][256].
// K split for the per-layer query products of few tiles: the largest of
// 16, 8, 4, 2 that divides the K-blocks into runs of at least 2 with every
// (tile, run) on its own SM; 1 (no split) for batches of more than a quarter
// of the SM count in tiles.
static int query_splits(int64_t m_tiles, int k) {
    const int kb = k / layer::BK;
    if (m_tiles * 4 > num_sms()) return 1;
    for (int s = 16; s >= 2; s /= 2)
        if (kb % s == 0 && kb / s >= 2 && m_tiles * s <= num_sms()) return s;
    return 1;
}

// out = s * (A @ B) on tcgen05 (layer::query_kernel): A bf16 [n][K], B bf16
// [K][256]; with RMS s = rinv(A row), with SPLIT out is bf16 [n][512] (hi | lo)
// instead of fp32 [n][256].  splits > 1: K split over that many CTAs per tile
// into `part` (fp32 [splits][n][256] + [splits][n]), then added up by
// query_reduce_kernel.
template <bool RMS, bool SPLIT>
static engram_status query_launch(const engram_config *cfg, const uint16_t *A, int K, const uint16_t *B, void *out,
                                  int64_t n_query, cudaStream_t st, int splits = 1, float *part = nullptr,
                                  bool pdl = true) {
    layer::QParams p;
    memset(&p, 0, sizeof(p));
    p.out = out;
    p.n_query = n_query;
    p.m_tiles = (n_query + layer::BM - 1) / layer::BM;
    p.d = K;
    p.eps = cfg->rms_eps;
    CUtensorMap amap, bmap;
    if (!bf16_map_2d(&amap, A, (uint64_t)K, (uint64_t)n_query, layer::BK, layer::BM))
        return cuda_fail(cudaErrorInvalidValue, "query A map");
    if (!bf16_map_2d(&bmap, B, kLayerWidth, (uint64_t)K, 64, layer::BK))
        return cuda_fail(cudaErrorInvalidValue, "query B map");
    if (splits > 1) {
        static std::atomic<bool> attr_split[64] = {};
        auto kern = layer::query_kernel<RMS, false, true>;
        engram_status s = ensure_smem((const void *)kern, layer::SMEM_BYTES, attr_split);
        if (s != ENGRAM_OK) return s;
        p.out = part;
        p.ss_out = part + (size_t)splits * n_query * kLayerWidth;
        p.kb_per_split = K / layer::BK / splits;
        // few tiles: the reduction is a programmatic dependent of the split
        // products, and they of the kernel before them when pdl (each waits
        // before its first global read), so their set-up overlaps the
        // previous kernel's tail
        cudaLaunchConfig_t lc = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        lc.gridDim = dim3((unsigned)p.m_tiles, (unsigned)splits);
        lc.blockDim = dim3(layer::NUM_THREADS);
        lc.dynamicSmemBytes = layer::SMEM_BYTES;
        lc.stream = st;
        lc.attrs = attr;
        lc.numAttrs = pdl ? 1 : 0;
        cudaError_t le = cudaLaunchKernelEx(&lc, kern, amap, bmap, p);
        if (le != cudaSuccess) return cuda_fail(le, "cudaLaunchKernelEx(query, split K)");
        s = launch_status();
        if (s != ENGRAM_OK) return s;
        const int64_t threads = n_query * (kLayerWidth / 4);
        lc.gridDim = dim3((unsigned)((threads + 255) / 256));
        lc.blockDim = dim3(256);
        lc.dynamicSmemBytes = 0;
        lc.numAttrs = 1;
        const float *ss = p.ss_out;
        le = cudaLaunchKernelEx(&lc, layer::query_reduce_kernel<RMS, SPLIT>, (const float *)part, ss, splits, n_query,
                                (int32_t)K, cfg->rms_eps, out);
        if (le != cudaSuccess) return cuda_fail(le, "cudaLaunchKernelEx(query reduce)");
        return launch_status();
    }
    static std::atomic<bool> attr_done[64] = {};
    auto kern = layer::query_kernel<RMS, SPLIT>;
    engram_status s = ensure_smem((const void *)kern, layer::SMEM_BYTES, attr_done);
    if (s != ENGRAM_OK) return s;
    const unsigned grid = (unsigned)std::min<int64_t>(p.m_tiles, num_sms());
    kern<<<grid, layer::NUM_THREADS, layer::SMEM_BYTES, st>>>(amap, bmap, p);
    return launch_status();
}

engram_status check_fuse_args(const engram_config *cfg, const void *W, const void *g, const void *h) {
    const int d = cfg->d_model;
    if (d < fuse::BN || d % fuse::BN != 0 || d > 16 * fuse::BN * fuse::MAX_GROUPS) return ENGRAM_EINVAL;
    if (!W || !g || !h) return ENGRAM_EINVAL;
    if (!aligned(W, 16) || !aligned(g, 16) || !aligned(h, 16)) return ENGRAM_EINVAL;
    if (!(cfg->rms_eps >= 0.0f)) return ENGRAM_EINVAL;
    return ENGRAM_OK;
}

// forward workspace: X [n][512] bf16
// forward workspace: X [n][512] bf16 | gate [n] fp32 (the d-split projection's gates)
static size_t forward_x_bytes(int64_t n) { return round_up((size_t)n * kMem * 2, 256); }
static size_t forward_bytes(int64_t n) { return forward_x_bytes(n) + round_up((size_t)n * 4, 256); }

// The d-split projection (narrow.cuh) when every (tile, 64-column slice) of
// the batch gets an SM of its own: one wave, no cluster.
static bool narrow_fits(int64_t m_tiles, int d) {
    return d % narrow::BN == 0 && m_tiles * (d / narrow::BN) <= num_sms();
}

// The split of d that fuse_launch would choose for a batch of m_tiles tiles:
// groups slices of cpg 256-column chunks (the token gates' reduction order).
static bool fuse_split(int64_t m_tiles, int n_chunks, int *groups, int *cpg) {
    const int cpg3 = pick_cpg_h_resident(m_tiles, n_chunks);
    *groups = cpg3 ? n_chunks / cpg3 : pick_groups(m_tiles, n_chunks);
    if (*groups == 0) return false;
    *cpg = n_chunks / *groups;
    return *cpg <= 16;
}

// Hash + gather -> bf16 X, plus one block per query token computing its gate
// in fuse_split's order (extra blocks of the same launch).
static engram_status gather_gate_launch(const engram_config *cfg, const uint8_t *tables, const float *scales,
                                        const HashParams &hp, int64_t n_query, uint16_t *X, const uint16_t *h,
                                        const uint16_t *g, float *gate, int groups, int cpg, cudaStream_t st) {
    GatherParams P;
    memset(&P, 0, sizeof(P));
    P.rows = tables;
    P.scales = scales_arg(cfg, scales);
    P.row_stride = row_stride(cfg);
    P.n_query = n_query;
    P.R = cfg->rows;
    P.out = X;
    P.hp = hp;
    const int64_t gather_blocks = (n_query * 64 + 255) / 256;  // a warp per (token, module)
    const int64_t gate_blocks = n_query;                       // a block per token, a warp per slice of d
    P.gp.h = h;
    P.gp.g = g;
    P.gp.gate = gate;
    P.gp.gather_blocks = gather_blocks;
    P.gp.d = cfg->d_model;
    P.gp.groups = groups;
    P.gp.cpg = cpg;
    P.gp.eps = cfg->rms_eps;
    P.gp.inv_sqrt_d = 1.0f / sqrtf((float)cfg->d_model);
    const unsigned blocks = (unsigned)(gather_blocks + gate_blocks);
    if (mx(cfg))
        gather_kernel<IDX_HASH, true, true, true><<<blocks, 256, 0, st>>>(P);
    else
        gather_kernel<IDX_HASH, true, false, true><<<blocks, 256, 0, st>>>(P);
    return launch_status();
}

// h = bf16(h + gate * X W) (gate != nullptr, X [n][512]) or h = bf16(h + X W)
// (gate == nullptr: one Engram layer, X [n][256]) by the d-split kernel,
// launched as a programmatic dependent of the kernel just enqueued on `st`
// (which writes X and the gates but not h or W).
template <int KBLK, bool GATED>
static engram_status narrow_launch_t(const engram_config *cfg, const uint16_t *X, const uint16_t *W, const float *gate,
                                     uint16_t *h, int64_t n_query, cudaStream_t st) {
    const int d = cfg->d_model;
    const int k = KBLK * narrow::BK;
    // a batch under one tile loads only its own rows (rounded up to a swizzle atom of 8)
    const uint32_t box_rows = n_query < narrow::BM ? (uint32_t)((n_query + 7) / 8 * 8) : (uint32_t)narrow::BM;
    CUtensorMap wmap, xmap, hl, hs;
    if (!bf16_map_2d(&wmap, W, (uint64_t)d, (uint64_t)k, narrow::BN, narrow::BK) ||
        !bf16_map_2d(&xmap, X, (uint64_t)k, (uint64_t)n_query, narrow::BK, box_rows) ||
        !bf16_map_2d(&hl, h, (uint64_t)d, (uint64_t)n_query, narrow::BN, box_rows) ||
        !bf16_map_2d(&hs, h, (uint64_t)d, (uint64_t)n_query, narrow::BN, 32))
        return cuda_fail(cudaErrorInvalidValue, "narrow projection tensor maps");
    static std::atomic<bool> attr_done[64] = {};
    auto kern = narrow::narrow_kernel<KBLK, GATED>;
    constexpr int smem = narrow::smem_bytes<KBLK>();
    engram_status s = ensure_smem((const void *)kern, smem, attr_done);
    if (s != ENGRAM_OK) return s;
    narrow::Params p;
    p.gate = gate;
    p.n_query = n_query;
    p.box_rows = (int32_t)box_rows;
    cudaLaunchConfig_t lc = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.gridDim = dim3((unsigned)(d / narrow::BN), (unsigned)((n_query + narrow::BM - 1) / narrow::BM));
    lc.blockDim = dim3(narrow::NUM_THREADS);
    lc.dynamicSmemBytes = smem;
    lc.stream = st;
    lc.attrs = attr;
    lc.numAttrs = 1;
    const cudaError_t le = cudaLaunchKernelEx(&lc, kern, wmap, xmap, hl, hs, p);
    if (le != cudaSuccess) return cuda_fail(le, "cudaLaunchKernelEx(narrow)");
    return launch_status();
}

static engram_status narrow_launch(const engram_config *cfg, const uint16_t *X, const uint16_t *W, const float *gate,
                                   uint16_t *h, int64_t n_query, cudaStream_t st) {
    return narrow_launch_t<kMem / narrow::BK, true>(cfg, X, W, gate, h, n_query, st);
}

static engram_status narrow_layer_launch(const engram_config *cfg, const uint16_t *X, const uint16_t *W, uint16_t *h,
                                         int64_t n_query, cudaStream_t st) {
    return narrow_launch_t<kLayerWidth / narrow::BK, false>(cfg, X, W, nullptr, h, n_query, st);
}

}  // namespace engram

using namespace engram;

// ================================================================= C ABI ====

extern "C" const char *engram_status_string(engram_status st) {
    switch (st) {
        case ENGRAM_OK: return "ok";
        case ENGRAM_EINVAL: return "invalid argument";
        case ENGRAM_ECUDA: return "CUDA error";
        case ENGRAM_ERANGE: return "value out of range (token id, position or row index)";
        case ENGRAM_ECAPACITY: return "more unique rows than the staging capacity";
        case ENGRAM_ETIMEOUT: return "a bounded device-side wait timed out";
        case ENGRAM_ENOMEM: return "workspace too small";
        case ENGRAM_EUNSUPPORTED: return "unsupported device or feature";
    }
    return "unknown status";
}

extern "C" engram_status engram_last_error(void) {
    if (cudaDeviceSynchronize() != cudaSuccess) return ENGRAM_ECUDA;
    unsigned int w = 0;
    if (cudaMemcpyFromSymbol(&w, g_error_word, sizeof(w)) != cudaSuccess) return ENGRAM_ECUDA;
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero)) != cudaSuccess) return ENGRAM_ECUDA;
    for (int k = 1; k < 32; ++k)
        if (w & (1u << k)) return (engram_status)k;
    return ENGRAM_OK;
}

// A bounded device wait that is meant to run out: one thread initialises an
// mbarrier that nothing arrives on and waits for it, as the projection
// kernels wait on theirs, with the caller's limit.  The wait gives up, sets
// ENGRAM_ETIMEOUT in the sticky word and the kernel returns; nothing traps
// and the device stays usable.
__global__ void wait_selftest_kernel(uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort = 0;
        fence_mbar_init();
        mbar_wait(&bar, 0, &abort, limit_ns);  // no arrival ever: runs out after limit_ns
    }
}

extern "C" engram_status engram_wait_selftest(uint64_t limit_ns, void *stream) {
    if (limit_ns == 0 || limit_ns > UINT64_C(10000000000)) return ENGRAM_EINVAL;
    wait_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(limit_ns);
    return launch_status();
}

extern "C" engram_status engram_hash(const engram_config *cfg, const int32_t *tokens, const int64_t *seq_offsets,
                                     int64_t n_seqs, int32_t last_n, int64_t n_query, int64_t *idx, void *stream) {
    if (check_config(cfg) != ENGRAM_OK || n_query < 0 || n_seqs < 0 || last_n < 0) return ENGRAM_EINVAL;
    if (n_query == 0) return ENGRAM_OK;
    if (!tokens || !seq_offsets || !idx || n_seqs < 1) return ENGRAM_EINVAL;
    if (last_n > 0 && n_query != n_seqs * (int64_t)last_n) return ENGRAM_EINVAL;
    if (!aligned(idx, 8) || !aligned(seq_offsets, 8) || !aligned(tokens, 4)) return ENGRAM_EINVAL;
    if (n_query > (INT64_C(1) << 40)) return ENGRAM_EINVAL;
    return hash_launch(cfg, tokens, seq_offsets, n_seqs, last_n, n_query, idx, (cudaStream_t)stream);
}

extern "C" engram_status engram_gather_reduce(const engram_config *cfg, const uint8_t *tables, const float *scales,
                                              const int64_t *idx, int64_t n_query, float *mem, void *stream) {
    if (check_config(cfg) != ENGRAM_OK || n_query < 0) return ENGRAM_EINVAL;
    if (n_query == 0) return ENGRAM_OK;
    if (!tables || !scales_ok(cfg, scales) || !idx || !mem) return ENGRAM_EINVAL;
    if (!aligned(tables, 16) || !aligned(idx, 8) || !aligned(mem, 16)) return ENGRAM_EINVAL;
    return gather_launch(IDX_I64, false, tables, scales_arg(cfg, scales), row_stride(cfg), mx(cfg), idx, nullptr, n_query,
                         cfg->rows, mem, (cudaStream_t)stream);
}

extern "C" size_t engram_dedup_workspace_bytes(const engram_config *cfg) {
    if (check_config(cfg) != ENGRAM_OK) return 0;
    return dedup_bytes(cfg);
}

extern "C" engram_status engram_dedup(const engram_config *cfg, const int64_t *idx, int64_t n_query, void *workspace,
                                      size_t workspace_bytes, int64_t *unique, int64_t capacity,
                                      int32_t *idx_staged, int64_t *n_unique, void *stream) {
    if (check_config(cfg) != ENGRAM_OK || n_query < 0 || capacity < 1) return ENGRAM_EINVAL;
    if (!workspace || !unique || !n_unique || (n_query > 0 && (!idx || !idx_staged))) return ENGRAM_EINVAL;
    if (n_query * kTables >= (INT64_C(1) << 31) || capacity >= (INT64_C(1) << 31)) return ENGRAM_EINVAL;
    if (!aligned(workspace, 256) || !aligned(unique, 8) || !aligned(n_unique, 8)) return ENGRAM_EINVAL;
    if (workspace_bytes < dedup_bytes(cfg)) return ENGRAM_ENOMEM;
    return dedup_launch(cfg, idx, n_query, workspace, unique, capacity, idx_staged, n_unique, (cudaStream_t)stream);
}

extern "C" engram_status engram_stage(const engram_config *cfg, const uint8_t *host_tables, const float *host_scales,
                                      const int64_t *unique, const int64_t *n_unique, int64_t capacity,
                                      uint8_t *staged_rows, float *staged_scales, void *stream) {
    if (check_config(cfg) != ENGRAM_OK || capacity < 1) return ENGRAM_EINVAL;
    if (!host_tables || !scales_ok(cfg, host_scales) || !unique || !n_unique || !staged_rows ||
        (!staged_scales && !mx(cfg)))
        return ENGRAM_EINVAL;
    if (!aligned(host_tables, 16) || !aligned(staged_rows, 16)) return ENGRAM_EINVAL;
    return stage_launch(host_tables, scales_arg(cfg, host_scales), row_stride(cfg), mx(cfg), unique, n_unique,
                        capacity, staged_rows, staged_scales, (cudaStream_t)stream);
}

extern "C" engram_status engram_gather_reduce_staged(const engram_config *cfg, const uint8_t *staged_rows,
                                                     const float *staged_scales, const int32_t *idx_staged,
                                                     int64_t n_query, int64_t capacity, float *mem, void *stream) {
    if (check_config(cfg) != ENGRAM_OK || n_query < 0 || capacity < 1) return ENGRAM_EINVAL;
    if (n_query == 0) return ENGRAM_OK;
    if (!staged_rows || (!staged_scales && !mx(cfg)) || !idx_staged || !mem) return ENGRAM_EINVAL;
    if (!aligned(staged_rows, 16) || !aligned(mem, 16) || !aligned(idx_staged, 4)) return ENGRAM_EINVAL;
    return gather_launch(IDX_STAGED_I32, false, staged_rows, mx(cfg) ? nullptr : staged_scales, staged_stride(cfg),
                         mx(cfg), idx_staged, nullptr, n_query, capacity, mem, (cudaStream_t)stream);
}

extern "C" engram_status engram_fuse(const engram_config *cfg, const float *mem, const uint16_t *W_out,
                                     const uint16_t *g, uint16_t *h, int64_t n_query, void *stream) {
    if (check_config(cfg) != ENGRAM_OK || n_query < 0) return ENGRAM_EINVAL;
    if (n_query == 0) return ENGRAM_OK;
    if (check_fuse_args(cfg, W_out, g, h) != ENGRAM_OK || !mem || !aligned(mem, 16)) return ENGRAM_EINVAL;
    if (n_query > (INT64_C(1) << 31)) return ENGRAM_EINVAL;
    return fuse_launch(cfg, mem, nullptr, W_out, g, h, n_query, (cudaStream_t)stream);
}

extern "C" size_t engram_forward_workspace_bytes(const engram_config *cfg, int64_t n_query) {
    if (check_config(cfg) != ENGRAM_OK || n_query < 0) return 0;
    return forward_bytes(n_query);
}

extern "C" engram_status engram_forward(const engram_config *cfg, const int32_t *tokens, const int64_t *seq_offsets,
                                        int64_t n_seqs, int32_t last_n, int64_t n_query, const uint8_t *tables,
                                        const float *scales, const uint16_t *W_out, const uint16_t *g, uint16_t *h,
                                        void *workspace, size_t workspace_bytes, void *stream) {
    if (check_config(cfg) != ENGRAM_OK || n_query < 0 || n_seqs < 0 || last_n < 0) return ENGRAM_EINVAL;
    if (n_query == 0) return ENGRAM_OK;
    if (!tokens || !seq_offsets || n_seqs < 1 || !tables || !scales_ok(cfg, scales) || !workspace)
        return ENGRAM_EINVAL;
    if (last_n > 0 && n_query != n_seqs * (int64_t)last_n) return ENGRAM_EINVAL;
    if (check_fuse_args(cfg, W_out, g, h) != ENGRAM_OK) return ENGRAM_EINVAL;
    if (!aligned(tables, 16) || !aligned(workspace, 256) || !aligned(tokens, 4) || !aligned(seq_offsets, 8))
        return ENGRAM_EINVAL;
    if (n_query > (INT64_C(1) << 31)) return ENGRAM_EINVAL;
    if (workspace_bytes < forward_bytes(n_query)) return ENGRAM_ENOMEM;
    cudaStream_t st = (cudaStream_t)stream;
    uint16_t *X = static_cast<uint16_t *>(workspace);
    HashParams hp;
    fill_hash_params(hp, cfg, tokens, seq_offsets, n_seqs, last_n, n_query);
    const int64_t m_tiles = (n_query + fuse::BM - 1) / fuse::BM;
    int groups = 0, cpg = 0;
    if (narrow_fits(m_tiles, cfg->d_model) && fuse_split(m_tiles, cfg->d_model / fuse::BN, &groups, &cpg)) {
        // few tokens: gates beside the gather, then d split over one CTA per
        // 64 columns (the same bits as the cluster kernels)
        float *gate = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + forward_x_bytes(n_query));
        engram_status s = gather_gate_launch(cfg, tables, scales, hp, n_query, X, h, g, gate, groups, cpg, st);
        if (s != ENGRAM_OK) return s;
        return narrow_launch(cfg, X, W_out, gate, h, n_query, st);
    }
    engram_status s = gather_launch(IDX_HASH, true, tables, scales_arg(cfg, scales), row_stride(cfg), mx(cfg), nullptr, &hp,
                                    n_query, cfg->rows, X, st);
    if (s != ENGRAM_OK) return s;
    return fuse_launch(cfg, nullptr, X, W_out, g, h, n_query, st, 0, /*pdl=*/true);
}

extern "C" engram_status engram_gather_x(const engram_config *cfg, const int32_t *tokens, const int64_t *seq_offsets,
                                         int64_t n_seqs, int32_t last_n, int64_t n_query, const uint8_t *tables,
                                         const float *scales, uint16_t *X, void *stream) {
    if (check_config(cfg) != ENGRAM_OK || n_query < 0 || n_seqs < 0 || last_n < 0) return ENGRAM_EINVAL;
    if (n_query == 0) return ENGRAM_OK;
    if (!tokens || !seq_offsets || n_seqs < 1 || !tables || !scales_ok(cfg, scales) || !X) return ENGRAM_EINVAL;
    if (last_n > 0 && n_query != n_seqs * (int64_t)last_n) return ENGRAM_EINVAL;
    if (!aligned(tables, 16) || !aligned(X, 16) || !aligned(tokens, 4) || !aligned(seq_offsets, 8))
        return ENGRAM_EINVAL;
    if (n_query > (INT64_C(1) << 40)) return ENGRAM_EINVAL;
    HashParams hp;
    fill_hash_params(hp, cfg, tokens, seq_offsets, n_seqs, last_n, n_query);
    return gather_launch(IDX_HASH, true, tables, scales_arg(cfg, scales), row_stride(cfg), mx(cfg), nullptr, &hp, n_query,
                         cfg->rows, X, (cudaStream_t)stream);
}

extern "C" int64_t engram_shard_rows(const engram_config *cfg, int32_t n_shards) {
    if (check_config(cfg) != ENGRAM_OK || n_shards < 1) return 0;
    return (cfg->rows + n_shards - 1) / n_shards;
}

extern "C" engram_status engram_gather_reduce_shard(const engram_config *cfg, int32_t shard, int32_t n_shards,
                                                    const int32_t *tokens, const int64_t *seq_offsets, int64_t n_seqs,
                                                    int32_t last_n, int64_t n_query, const uint8_t *tables_shard,
                                                    const float *scales_shard, float *mem, void *stream) {
    if (check_config(cfg) != ENGRAM_OK || n_query < 0 || n_seqs < 0 || last_n < 0) return ENGRAM_EINVAL;
    if (n_shards < 1 || shard < 0 || shard >= n_shards) return ENGRAM_EINVAL;
    if (n_query == 0) return ENGRAM_OK;
    if (!tokens || !seq_offsets || n_seqs < 1 || !tables_shard || !scales_ok(cfg, scales_shard) || !mem)
        return ENGRAM_EINVAL;
    if (last_n > 0 && n_query != n_seqs * (int64_t)last_n) return ENGRAM_EINVAL;
    if (!aligned(tables_shard, 16) || !aligned(mem, 16) || !aligned(tokens, 4) || !aligned(seq_offsets, 8))
        return ENGRAM_EINVAL;
    if (n_query > (INT64_C(1) << 40)) return ENGRAM_EINVAL;
    HashParams hp;
    fill_hash_params(hp, cfg, tokens, seq_offsets, n_seqs, last_n, n_query);
    return gather_launch(IDX_HASH_SHARD, false, tables_shard, scales_arg(cfg, scales_shard), row_stride(cfg), mx(cfg),
                         nullptr, &hp, n_query, cfg->rows, mem, (cudaStream_t)stream,
                         engram_shard_rows(cfg, n_shards), shard, n_shards);
}

extern "C" engram_status engram_fuse_x(const engram_config *cfg, const uint16_t *X, const uint16_t *W_out,
                                       const uint16_t *g, uint16_t *h, int64_t n_query, void *stream) {
    if (check_config(cfg) != ENGRAM_OK || n_query < 0) return ENGRAM_EINVAL;
    if (n_query == 0) return ENGRAM_OK;
    if (check_fuse_args(cfg, W_out, g, h) != ENGRAM_OK || !X || !aligned(X, 16)) return ENGRAM_EINVAL;
    if (n_query > (INT64_C(1) << 31)) return ENGRAM_EINVAL;
    return fuse_launch(cfg, nullptr, X, W_out, g, h, n_query, (cudaStream_t)stream);
}

extern "C" size_t engram_forward_host_workspace_bytes(const engram_config *cfg, int64_t n_query, int64_t capacity) {
    if (check_config(cfg) != ENGRAM_OK || n_query < 0 || capacity < 1) return 0;
    return round_up((size_t)n_query * kTables * 8, 256)      // idx
           + round_up((size_t)n_query * kTables * 4, 256)    // idx_staged
           + round_up((size_t)n_query * kMem * 2, 256)       // X (bf16)
           + round_up((size_t)capacity * 8, 256)             // unique
           + round_up((size_t)capacity * staged_stride(cfg), 256)  // staged rows
           + round_up((size_t)capacity * 4, 256)             // staged scales
           + dedup_bytes(cfg);
}

extern "C" engram_status engram_forward_host(const engram_config *cfg, const int32_t *tokens,
                                             const int64_t *seq_offsets, int64_t n_seqs, int32_t last_n,
                                             int64_t n_query, const uint8_t *host_tables, const float *host_scales,
                                             const uint16_t *W_out, const uint16_t *g, uint16_t *h, int64_t capacity,
                                             void *workspace, size_t workspace_bytes, int64_t *n_unique, void *stream,
                                             void *side_stream, void *ev_dedup, void *ev_staged) {
    if (check_config(cfg) != ENGRAM_OK || n_query < 0 || n_seqs < 0 || last_n < 0 || capacity < 1)
        return ENGRAM_EINVAL;
    if (n_query == 0) return ENGRAM_OK;
    if (!tokens || !seq_offsets || n_seqs < 1 || !host_tables || !scales_ok(cfg, host_scales) || !workspace ||
        !n_unique || !ev_dedup || !ev_staged)
        return ENGRAM_EINVAL;
    if (last_n > 0 && n_query != n_seqs * (int64_t)last_n) return ENGRAM_EINVAL;
    if (check_fuse_args(cfg, W_out, g, h) != ENGRAM_OK) return ENGRAM_EINVAL;
    if (!aligned(host_tables, 16) || !aligned(workspace, 256) || !aligned(n_unique, 8)) return ENGRAM_EINVAL;
    if (n_query * kTables >= (INT64_C(1) << 31) || capacity >= (INT64_C(1) << 31)) return ENGRAM_EINVAL;
    if (workspace_bytes < engram_forward_host_workspace_bytes(cfg, n_query, capacity)) return ENGRAM_ENOMEM;
    cudaStream_t st = (cudaStream_t)stream, side = (cudaStream_t)side_stream;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    size_t o = 0;
    int64_t *idx = reinterpret_cast<int64_t *>(ws + o);
    o += round_up((size_t)n_query * kTables * 8, 256);
    int32_t *idx_staged = reinterpret_cast<int32_t *>(ws + o);
    o += round_up((size_t)n_query * kTables * 4, 256);
    uint16_t *X = reinterpret_cast<uint16_t *>(ws + o);
    o += round_up((size_t)n_query * kMem * 2, 256);
    int64_t *unique = reinterpret_cast<int64_t *>(ws + o);
    o += round_up((size_t)capacity * 8, 256);
    uint8_t *rows = ws + o;
    o += round_up((size_t)capacity * staged_stride(cfg), 256);
    float *sc = reinterpret_cast<float *>(ws + o);
    o += round_up((size_t)capacity * 4, 256);
    void *dws = ws + o;
    engram_status s = hash_launch(cfg, tokens, seq_offsets, n_seqs, last_n, n_query, idx, st);
    if (s != ENGRAM_OK) return s;
    s = dedup_launch(cfg, idx, n_query, dws, unique, capacity, idx_staged, n_unique, st);
    if (s != ENGRAM_OK) return s;
    if (cudaEventRecord((cudaEvent_t)ev_dedup, st) != cudaSuccess) return ENGRAM_ECUDA;
    if (cudaStreamWaitEvent(side, (cudaEvent_t)ev_dedup, 0) != cudaSuccess) return ENGRAM_ECUDA;
    s = stage_launch(host_tables, scales_arg(cfg, host_scales), row_stride(cfg), mx(cfg), unique, n_unique, capacity,
                     rows, sc, side);
    if (s != ENGRAM_OK) return s;
    if (cudaEventRecord((cudaEvent_t)ev_staged, side) != cudaSuccess) return ENGRAM_ECUDA;
    if (cudaStreamWaitEvent(st, (cudaEvent_t)ev_staged, 0) != cudaSuccess) return ENGRAM_ECUDA;
    s = gather_launch(IDX_STAGED_I32, true, rows, mx(cfg) ? nullptr : sc, staged_stride(cfg), mx(cfg), idx_staged,
                      nullptr, n_query, capacity, X, st);
    if (s != ENGRAM_OK) return s;
    return fuse_launch(cfg, nullptr, X, W_out, g, h, n_query, st);
}

// ============================================ host tables with a row cache ==

struct CacheLayout {
    size_t tags, claims, rows, scales, total;
};

static CacheLayout cache_layout(const engram_config *cfg, int64_t slots, int64_t capacity) {
    CacheLayout L;
    size_t o = 0;
    L.tags = o;
    o += round_up((size_t)slots * 8, 256);
    L.claims = o;
    o += round_up((size_t)slots * 4, 256);
    L.rows = o;
    o += round_up((size_t)(slots + capacity) * staged_stride(cfg), 256);
    L.scales = o;
    o += round_up((size_t)(slots + capacity) * 4, 256);
    L.total = o;
    return L;
}

static bool cache_args_ok(int64_t slots, int64_t capacity) {
    return slots >= 1 && (slots & (slots - 1)) == 0 && capacity >= 1 && slots + capacity < (INT64_C(1) << 31);
}

extern "C" size_t engram_host_cache_bytes(const engram_config *cfg, int64_t slots, int64_t capacity) {
    if (check_config(cfg) != ENGRAM_OK || !cache_args_ok(slots, capacity)) return 0;
    return cache_layout(cfg, slots, capacity).total;
}

extern "C" engram_status engram_host_cache_reset(const engram_config *cfg, void *cache, int64_t slots,
                                                 int64_t capacity, void *stream) {
    if (check_config(cfg) != ENGRAM_OK || !cache_args_ok(slots, capacity) || !cache || !aligned(cache, 256))
        return ENGRAM_EINVAL;
    const CacheLayout L = cache_layout(cfg, slots, capacity);
    uint8_t *c = static_cast<uint8_t *>(cache);
    const unsigned blocks = (unsigned)std::min<int64_t>((slots + 255) / 256, (int64_t)num_sms() * 8);
    cache_reset_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(reinterpret_cast<int64_t *>(c + L.tags),
                                                                 reinterpret_cast<uint32_t *>(c + L.claims), slots);
    return launch_status();
}

// workspace: idx [n][48] i64 | idx_staged [n][48] i32 | X [n][512] bf16 |
// unique [cap] i64 | where [cap] i32 | stage_flat [cap] i64 | stage_dest [cap]
// i32 | n_unique i64 | dedup workspace
struct CachedLayout {
    size_t idx, idx_staged, x, unique, where, stage_flat, stage_dest, n_unique, dedup, total;
};

static CachedLayout cached_layout(const engram_config *cfg, int64_t n, int64_t cap) {
    CachedLayout L;
    size_t o = 0;
    L.idx = o;
    o += round_up((size_t)n * kTables * 8, 256);
    L.idx_staged = o;
    o += round_up((size_t)n * kTables * 4, 256);
    L.x = o;
    o += round_up((size_t)n * kMem * 2, 256);
    L.unique = o;
    o += round_up((size_t)cap * 8, 256);
    L.where = o;
    o += round_up((size_t)cap * 4, 256);
    L.stage_flat = o;
    o += round_up((size_t)cap * 8, 256);
    L.stage_dest = o;
    o += round_up((size_t)cap * 4, 256);
    L.n_unique = o;
    o += 256;
    L.dedup = o;
    o += dedup_bytes(cfg);
    L.total = o;
    return L;
}

extern "C" size_t engram_forward_host_cached_workspace_bytes(const engram_config *cfg, int64_t n_query,
                                                             int64_t capacity) {
    if (check_config(cfg) != ENGRAM_OK || n_query < 0 || capacity < 1) return 0;
    return cached_layout(cfg, n_query, capacity).total;
}

extern "C" engram_status engram_forward_host_cached(const engram_config *cfg, const int32_t *tokens,
                                                    const int64_t *seq_offsets, int64_t n_seqs, int32_t last_n,
                                                    int64_t n_query, const uint8_t *host_tables,
                                                    const float *host_scales, const uint16_t *W_out, const uint16_t *g,
                                                    uint16_t *h, void *cache, int64_t slots, int64_t capacity,
                                                    uint32_t stamp, void *workspace, size_t workspace_bytes,
                                                    int64_t *stats, void *stream, void *side_stream, void *ev_dedup,
                                                    void *ev_staged) {
    if (check_config(cfg) != ENGRAM_OK || n_query < 0 || n_seqs < 0 || last_n < 0) return ENGRAM_EINVAL;
    if (!cache_args_ok(slots, capacity) || stamp == 0) return ENGRAM_EINVAL;
    if (n_query == 0) return ENGRAM_OK;
    if (!tokens || !seq_offsets || n_seqs < 1 || !host_tables || !scales_ok(cfg, host_scales) || !workspace ||
        !cache || !stats || !ev_dedup || !ev_staged)
        return ENGRAM_EINVAL;
    if (last_n > 0 && n_query != n_seqs * (int64_t)last_n) return ENGRAM_EINVAL;
    if (check_fuse_args(cfg, W_out, g, h) != ENGRAM_OK) return ENGRAM_EINVAL;
    if (!aligned(host_tables, 16) || !aligned(workspace, 256) || !aligned(cache, 256) || !aligned(stats, 8))
        return ENGRAM_EINVAL;
    if (n_query * kTables >= (INT64_C(1) << 31)) return ENGRAM_EINVAL;
    const CachedLayout L = cached_layout(cfg, n_query, capacity);
    if (workspace_bytes < L.total) return ENGRAM_ENOMEM;
    cudaStream_t st = (cudaStream_t)stream, side = (cudaStream_t)side_stream;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    int64_t *idx = reinterpret_cast<int64_t *>(ws + L.idx);
    int32_t *idx_staged = reinterpret_cast<int32_t *>(ws + L.idx_staged);
    uint16_t *X = reinterpret_cast<uint16_t *>(ws + L.x);
    int64_t *unique = reinterpret_cast<int64_t *>(ws + L.unique);
    int32_t *where = reinterpret_cast<int32_t *>(ws + L.where);
    int64_t *stage_flat = reinterpret_cast<int64_t *>(ws + L.stage_flat);
    int32_t *stage_dest = reinterpret_cast<int32_t *>(ws + L.stage_dest);
    int64_t *n_unique = reinterpret_cast<int64_t *>(ws + L.n_unique);
    const CacheLayout C = cache_layout(cfg, slots, capacity);
    uint8_t *cb = static_cast<uint8_t *>(cache);
    int log2_slots = 0;
    while ((INT64_C(1) << log2_slots) < slots) ++log2_slots;

    engram_status s = hash_launch(cfg, tokens, seq_offsets, n_seqs, last_n, n_query, idx, st);
    if (s != ENGRAM_OK) return s;
    s = dedup_launch(cfg, idx, n_query, ws + L.dedup, unique, capacity, idx_staged, n_unique, st);
    if (s != ENGRAM_OK) return s;
    if (cudaMemsetAsync(stats, 0, 4 * sizeof(int64_t), st) != cudaSuccess) return ENGRAM_ECUDA;
    cache_lookup_kernel<<<(unsigned)((capacity + 255) / 256), 256, 0, st>>>(
        unique, n_unique, capacity, reinterpret_cast<int64_t *>(cb + C.tags), reinterpret_cast<uint32_t *>(cb + C.claims),
        log2_slots, stamp, where, stage_flat, stage_dest, stats);
    s = launch_status();
    if (s != ENGRAM_OK) return s;
    if (cudaEventRecord((cudaEvent_t)ev_dedup, st) != cudaSuccess) return ENGRAM_ECUDA;
    if (cudaStreamWaitEvent(side, (cudaEvent_t)ev_dedup, 0) != cudaSuccess) return ENGRAM_ECUDA;
    // the misses and overflow rows, from pinned host memory into their slots
    s = stage_launch(host_tables, scales_arg(cfg, host_scales), row_stride(cfg), mx(cfg), stage_flat, stats + 2,
                     capacity, cb + C.rows, reinterpret_cast<float *>(cb + C.scales), side, stage_dest);
    if (s != ENGRAM_OK) return s;
    if (cudaEventRecord((cudaEvent_t)ev_staged, side) != cudaSuccess) return ENGRAM_ECUDA;
    const int64_t n = n_query * kTables;
    cache_remap_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(idx_staged, n, where);
    s = launch_status();
    if (s != ENGRAM_OK) return s;
    if (cudaStreamWaitEvent(st, (cudaEvent_t)ev_staged, 0) != cudaSuccess) return ENGRAM_ECUDA;
    s = gather_launch(IDX_STAGED_I32, true, cb + C.rows, mx(cfg) ? nullptr : reinterpret_cast<float *>(cb + C.scales),
                      staged_stride(cfg), mx(cfg), idx_staged, nullptr, n_query, slots + capacity, X, st);
    if (s != ENGRAM_OK) return s;
    return fuse_launch(cfg, nullptr, X, W_out, g, h, n_query, st);
}

// ========================================================= host tables ====
// Pinned host memory for tables read by the device over the host link,
// backed by transparent huge pages where the kernel offers them.  Staging
// touches rows scattered over tens of GB; with base pages (64 KB on this
// class of host) the device spends much of its time translating addresses.

static std::mutex g_host_mu;
static std::map<void *, std::pair<void *, size_t>> g_host_maps;  // aligned pointer -> mapping

static size_t huge_page_bytes() {
    size_t v = 0;
    if (FILE *f = fopen("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size", "r")) {
        unsigned long long x = 0;
        if (fscanf(f, "%llu", &x) == 1) v = (size_t)x;
        fclose(f);
    }
    return (v >= 4096 && (v & (v - 1)) == 0) ? v : (size_t)2 << 20;
}

extern "C" engram_status engram_host_alloc(size_t bytes, void **ptr) {
    if (!ptr) return ENGRAM_EINVAL;
    *ptr = nullptr;
    if (bytes == 0) return ENGRAM_EINVAL;
    const size_t align = huge_page_bytes();
    const size_t len = (bytes + align - 1) / align * align + align;
    void *raw = mmap(nullptr, len, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
    if (raw == MAP_FAILED) return ENGRAM_ENOMEM;
    void *p = reinterpret_cast<void *>((reinterpret_cast<uintptr_t>(raw) + align - 1) / align * align);
    const size_t plen = (bytes + align - 1) / align * align;
    madvise(p, plen, MADV_HUGEPAGE);  // a hint: plain pages if the kernel declines
    const cudaError_t e = cudaHostRegister(p, plen, cudaHostRegisterDefault);
    if (e != cudaSuccess) {
        munmap(raw, len);
        return cuda_fail(e, "cudaHostRegister");
    }
    std::lock_guard<std::mutex> lock(g_host_mu);
    g_host_maps[p] = {raw, len};
    *ptr = p;
    return ENGRAM_OK;
}

extern "C" engram_status engram_host_free(void *ptr) {
    if (!ptr) return ENGRAM_OK;
    std::pair<void *, size_t> m;
    {
        std::lock_guard<std::mutex> lock(g_host_mu);
        auto it = g_host_maps.find(ptr);
        if (it == g_host_maps.end()) return ENGRAM_EINVAL;
        m = it->second;
        g_host_maps.erase(it);
    }
    const cudaError_t e = cudaHostUnregister(ptr);
    munmap(m.first, m.second);
    return e == cudaSuccess ? ENGRAM_OK : cuda_fail(e, "cudaHostUnregister");
}

// ============================================ per-layer Engram (row gates) ==

extern "C" engram_status engram_layer_keys(const engram_config *cfg, const uint16_t *W_k, uint16_t *W_kk,
                                           void *stream) {
    if (check_config(cfg) != ENGRAM_OK || !W_k || !W_kk) return ENGRAM_EINVAL;
    if (!aligned(W_k, 16) || !aligned(W_kk, 16)) return ENGRAM_EINVAL;
    layer::wkk_kernel<<<2 * kLayerWidth, kLayerWidth, 0, (cudaStream_t)stream>>>(W_k, W_kk);
    return launch_status();
}

// workspace: q pair bf16 [n][512] | u fp32 [n][256] | X bf16 [n][256]
static size_t layer_off_u(int64_t n) { return round_up((size_t)n * 2 * kLayerWidth * 2, 256); }
static size_t layer_off_x(int64_t n) { return layer_off_u(n) + round_up((size_t)n * kLayerWidth * 4, 256); }
static size_t layer_off_part(int64_t n) { return layer_off_x(n) + round_up((size_t)n * kLayerWidth * 2, 256); }
// the split-K partial products of the two query products (few tiles only)
static int layer_max_splits(const engram_config *cfg, int64_t n) {
    const int64_t m_tiles = (n + layer::BM - 1) / layer::BM;
    return std::max(query_splits(m_tiles, cfg->d_model), query_splits(m_tiles, 2 * kLayerWidth));
}
static size_t layer_part_bytes(const engram_config *cfg, int64_t n) {
    const int s = layer_max_splits(cfg, n);
    return s > 1 ? round_up((size_t)s * n * (kLayerWidth + 1) * 4, 256) : 0;
}

extern "C" size_t engram_layer_workspace_bytes(const engram_config *cfg, int64_t n_query) {
    if (check_config(cfg) != ENGRAM_OK || n_query < 0) return 0;
    return layer_off_part(n_query) + layer_part_bytes(cfg, n_query);
}

extern "C" engram_status engram_layer_forward(const engram_config *cfg, int32_t module, const int32_t *tokens,
                                              const int64_t *seq_offsets, int64_t n_seqs, int32_t last_n,
                                              int64_t n_query, const uint8_t *tables, const float *scales,
                                              const uint16_t *W_q, const uint16_t *W_kk, const uint16_t *W_m,
                                              uint16_t *h, void *workspace, size_t workspace_bytes, void *stream) {
    if (check_config(cfg) != ENGRAM_OK || module < 0 || module > 1 || n_query < 0 || n_seqs < 0 || last_n < 0)
        return ENGRAM_EINVAL;
    if (n_query == 0) return ENGRAM_OK;
    if (!tokens || !seq_offsets || n_seqs < 1 || !tables || !scales_ok(cfg, scales) || !W_q || !W_kk || !W_m ||
        !h || !workspace)
        return ENGRAM_EINVAL;
    if (last_n > 0 && n_query != n_seqs * (int64_t)last_n) return ENGRAM_EINVAL;
    const int d = cfg->d_model;
    if (d < fuse::BN || d % fuse::BN != 0 || d > 16 * fuse::BN * fuse::MAX_GROUPS) return ENGRAM_EINVAL;
    if (!aligned(tables, 16) || !aligned(W_q, 16) || !aligned(W_kk, 16) || !aligned(W_m, 16) || !aligned(h, 16) ||
        !aligned(workspace, 256) || !aligned(tokens, 4) || !aligned(seq_offsets, 8))
        return ENGRAM_EINVAL;
    if (!(cfg->rms_eps >= 0.0f) || n_query > (INT64_C(1) << 40)) return ENGRAM_EINVAL;
    if (workspace_bytes < engram_layer_workspace_bytes(cfg, n_query)) return ENGRAM_ENOMEM;
    cudaStream_t st = (cudaStream_t)stream;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint16_t *qpair = reinterpret_cast<uint16_t *>(ws);
    float *u = reinterpret_cast<float *>(ws + layer_off_u(n_query));
    uint16_t *X = reinterpret_cast<uint16_t *>(ws + layer_off_x(n_query));
    // q = rinv(h) h W_q as a bf16 pair, then u = [q_hi | q_lo] [W_k^T ; W_k^T]
    // (few tiles: K split over several CTAs per tile, partial products added up)
    const int64_t m_tiles = (n_query + layer::BM - 1) / layer::BM;
    float *part = reinterpret_cast<float *>(ws + layer_off_part(n_query));
    // The layer's first kernel is an ordinary launch: it starts after all
    // earlier work in the stream has finished, the previous layer's update of
    // h included.  Every later kernel of the layer is a programmatic
    // dependent of the one before it and may start early; the projection
    // loads its h box before its dependency wait, which is safe only because
    // nothing launched after this first kernel writes h before it.
    engram_status s = query_launch<true, true>(cfg, h, d, W_q, qpair, n_query, st, query_splits(m_tiles, d), part,
                                               /*pdl=*/false);
    if (s != ENGRAM_OK) return s;
    s = query_launch<false, false>(cfg, qpair, 2 * kLayerWidth, W_kk, u, n_query, st,
                                   query_splits(m_tiles, 2 * kLayerWidth), part);
    if (s != ENGRAM_OK) return s;
    GatedParams P;
    memset(&P, 0, sizeof(P));
    P.rows = tables;
    P.scales = scales_arg(cfg, scales);
    P.row_stride = row_stride(cfg);
    P.q = u;
    P.X = X;
    P.n_query = n_query;
    P.R = cfg->rows;
    P.module = module;
    P.eps = cfg->rms_eps;
    fill_hash_params(P.hp, cfg, tokens, seq_offsets, n_seqs, last_n, n_query);
    // blocks of 128 threads at 96 registers: 20 warps per SM (2 blocks of 256
    // at 128 registers gave 16; 1.970 against 1.997 ms per two-layer step)
    const unsigned blocks = (unsigned)((n_query * 32 + 127) / 128);
    {
        // as a programmatic dependent while the query products are split over
        // K (up to a quarter as many tiles as SMs: decode and chunk-sized
        // batches, whose chain of short launches it shortens); on the large
        // workload the early blocks cost more than they hide (two-layer step
        // 2.156 against 1.971 ms)
        cudaLaunchConfig_t lc = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        lc.gridDim = dim3(blocks);
        lc.blockDim = dim3(128);
        lc.stream = st;
        lc.attrs = attr;
        lc.numAttrs = query_splits(m_tiles, d) > 1 ? 1 : 0;
        const cudaError_t le = mx(cfg) ? cudaLaunchKernelEx(&lc, gather_gated_kernel<true>, P)
                                       : cudaLaunchKernelEx(&lc, gather_gated_kernel<false>, P);
        if (le != cudaSuccess) return cuda_fail(le, "cudaLaunchKernelEx(gather_gated)");
    }
    s = launch_status();
    if (s != ENGRAM_OK) return s;
    return layer_projection_launch(cfg, X, W_m, h, n_query, st);
}

// ================================================== pipelined host path ====
// Workspace: idx [n][48] i64 | X [n][512] bf16 | two staging sets, each
// idx_staged [chunk][48] i32 | unique [cap] i64 | rows [cap][stride] |
// scales [cap] f32 | dedup workspace.
struct PipeLayout {
    size_t idx, x, set[2], set_bytes, idx_staged, unique, rows, scales, dedup, total;
};

static PipeLayout pipe_layout(const engram_config *cfg, int64_t n_query, int64_t chunk, int64_t capacity) {
    PipeLayout L;
    size_t o = 0;
    L.idx = o;
    o += round_up((size_t)n_query * kTables * 8, 256);
    L.x = o;
    o += round_up((size_t)n_query * kMem * 2, 256);
    L.idx_staged = 0;  // offsets inside a staging set
    L.unique = round_up((size_t)chunk * kTables * 4, 256);
    L.rows = L.unique + round_up((size_t)capacity * 8, 256);
    L.scales = L.rows + round_up((size_t)capacity * staged_stride(cfg), 256);
    L.set_bytes = L.scales + round_up((size_t)capacity * 4, 256);
    L.set[0] = o;
    o += L.set_bytes;
    L.set[1] = o;
    o += L.set_bytes;
    L.dedup = o;
    o += dedup_bytes(cfg);
    L.total = o;
    return L;
}

extern "C" size_t engram_forward_host_pipelined_workspace_bytes(const engram_config *cfg, int64_t n_query,
                                                                int64_t chunk, int64_t capacity) {
    if (check_config(cfg) != ENGRAM_OK || n_query < 0 || chunk < 1 || capacity < 1) return 0;
    return pipe_layout(cfg, n_query, chunk, capacity).total;
}

extern "C" engram_status engram_forward_host_pipelined(const engram_config *cfg, const int32_t *tokens,
                                                       const int64_t *seq_offsets, int64_t n_seqs, int32_t last_n,
                                                       int64_t n_query, const uint8_t *host_tables,
                                                       const float *host_scales, const uint16_t *W_out,
                                                       const uint16_t *g, uint16_t *h, int64_t chunk, int64_t capacity,
                                                       void *workspace, size_t workspace_bytes, int64_t *n_unique,
                                                       void *stream, void *side_stream, void *const *events) {
    if (check_config(cfg) != ENGRAM_OK || n_query < 0 || n_seqs < 0 || last_n < 0 || chunk < 1 || capacity < 1)
        return ENGRAM_EINVAL;
    if (n_query == 0) return ENGRAM_OK;
    if (!tokens || !seq_offsets || n_seqs < 1 || !host_tables || !scales_ok(cfg, host_scales) || !workspace ||
        !n_unique || !events)
        return ENGRAM_EINVAL;
    for (int e = 0; e < 6; ++e)
        if (!events[e]) return ENGRAM_EINVAL;
    if (last_n > 0 && n_query != n_seqs * (int64_t)last_n) return ENGRAM_EINVAL;
    if (check_fuse_args(cfg, W_out, g, h) != ENGRAM_OK) return ENGRAM_EINVAL;
    if (!aligned(host_tables, 16) || !aligned(workspace, 256) || !aligned(n_unique, 8)) return ENGRAM_EINVAL;
    if (n_query * kTables >= (INT64_C(1) << 31) || capacity >= (INT64_C(1) << 31)) return ENGRAM_EINVAL;
    chunk = std::min(chunk, n_query);
    const PipeLayout L = pipe_layout(cfg, n_query, chunk, capacity);
    if (workspace_bytes < L.total) return ENGRAM_ENOMEM;
    cudaStream_t st = (cudaStream_t)stream, side = (cudaStream_t)side_stream;
    cudaEvent_t ev_dedup[2] = {(cudaEvent_t)events[0], (cudaEvent_t)events[1]};
    cudaEvent_t ev_staged[2] = {(cudaEvent_t)events[2], (cudaEvent_t)events[3]};
    cudaEvent_t ev_used[2] = {(cudaEvent_t)events[4], (cudaEvent_t)events[5]};
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    int64_t *idx = reinterpret_cast<int64_t *>(ws + L.idx);
    uint16_t *X = reinterpret_cast<uint16_t *>(ws + L.x);
    void *dws = ws + L.dedup;
    auto set_idx_staged = [&](int b) { return reinterpret_cast<int32_t *>(ws + L.set[b] + L.idx_staged); };
    auto set_unique = [&](int b) { return reinterpret_cast<int64_t *>(ws + L.set[b] + L.unique); };
    auto set_rows = [&](int b) { return ws + L.set[b] + L.rows; };
    auto set_scales = [&](int b) { return reinterpret_cast<float *>(ws + L.set[b] + L.scales); };
    const int64_t n_chunks = (n_query + chunk - 1) / chunk;
    const int64_t all_tiles = (n_query + fuse::BM - 1) / fuse::BM;

    engram_status s = hash_launch(cfg, tokens, seq_offsets, n_seqs, last_n, n_query, idx, st);
    if (s != ENGRAM_OK) return s;
    // dedup (stream) then stage (side stream) of chunk k into staging set k & 1
    auto issue = [&](int64_t k) -> engram_status {
        const int b = (int)(k & 1);
        const int64_t q0 = k * chunk, nk = std::min(chunk, n_query - q0);
        engram_status r = dedup_launch(cfg, idx + q0 * kTables, nk, dws, set_unique(b), capacity, set_idx_staged(b),
                                       n_unique + k, st);
        if (r != ENGRAM_OK) return r;
        if (cudaEventRecord(ev_dedup[b], st) != cudaSuccess) return ENGRAM_ECUDA;
        if (cudaStreamWaitEvent(side, ev_dedup[b], 0) != cudaSuccess) return ENGRAM_ECUDA;
        if (k >= 2 && cudaStreamWaitEvent(side, ev_used[b], 0) != cudaSuccess) return ENGRAM_ECUDA;
        r = stage_launch(host_tables, scales_arg(cfg, host_scales), row_stride(cfg), mx(cfg), set_unique(b),
                         n_unique + k, capacity, set_rows(b), set_scales(b), side);
        if (r != ENGRAM_OK) return r;
        return cudaEventRecord(ev_staged[b], side) == cudaSuccess ? ENGRAM_OK : ENGRAM_ECUDA;
    };
    s = issue(0);
    if (s != ENGRAM_OK) return s;
    for (int64_t k = 0; k < n_chunks; ++k) {
        if (k + 1 < n_chunks) {  // the next chunk's dedup and staging run under this chunk's gather
            s = issue(k + 1);
            if (s != ENGRAM_OK) return s;
        }
        const int b = (int)(k & 1);
        const int64_t q0 = k * chunk, nk = std::min(chunk, n_query - q0);
        if (cudaStreamWaitEvent(st, ev_staged[b], 0) != cudaSuccess) return ENGRAM_ECUDA;
        s = gather_launch(IDX_STAGED_I32, true, set_rows(b), mx(cfg) ? nullptr : set_scales(b), staged_stride(cfg),
                          mx(cfg), set_idx_staged(b), nullptr, nk, capacity, X + q0 * kMem, st);
        if (s != ENGRAM_OK) return s;
        if (cudaEventRecord(ev_used[b], st) != cudaSuccess) return ENGRAM_ECUDA;
    }
    // One projection over the whole batch: the projection kernel is persistent
    // (one cluster per group of SMs, striding over tiles), so it is not run
    // beside a staging kernel that holds SMs.
    return fuse_launch(cfg, nullptr, X, W_out, g, h, n_query, st, all_tiles);
}

// ====================================================== no-workspace variant ==
// engram_forward for callers that cannot allocate device memory (see the
// header): the bf16 X handed from the gather kernel to the projection lives in
// this file-scope array instead of a caller workspace.  Every GPU that loads
// the library holds it (16 MB) until the process exits, and every call shares
// it.

static __device__ __align__(256) uint16_t g_no_workspace_x[ENGRAM_NO_WORKSPACE_MAX_QUERY * ENGRAM_MEM_DIM];

// Device address of the array on the current device.  In host code the
// array's name is only a host-side stand-in, never a device address, so it
// is looked up once per device (with that device current) and cached.
static engram_status no_workspace_scratch(uint16_t **out) {
    static std::mutex mu;
    static uint16_t *addr[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return ENGRAM_EUNSUPPORTED;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_no_workspace_x);
        if (e != cudaSuccess || !p) return cuda_fail(e, "cudaGetSymbolAddress(no-workspace scratch)");
        addr[dev] = static_cast<uint16_t *>(p);
    }
    *out = addr[dev];
    return ENGRAM_OK;
}

extern "C" engram_status engram_forward_no_workspace(const engram_config *cfg, const int32_t *tokens,
                                                     const int64_t *seq_offsets, int64_t n_seqs, int32_t last_n,
                                                     int64_t n_query, const uint8_t *tables, const float *scales,
                                                     const uint16_t *W_out, const uint16_t *g, uint16_t *h,
                                                     void *stream) {
    if (check_config(cfg) != ENGRAM_OK || n_query < 0 || n_seqs < 0 || last_n < 0) return ENGRAM_EINVAL;
    if (n_query == 0) return ENGRAM_OK;
    if (!tokens || !seq_offsets || n_seqs < 1 || !tables || !scales_ok(cfg, scales)) return ENGRAM_EINVAL;
    if (last_n > 0 && n_query != n_seqs * (int64_t)last_n) return ENGRAM_EINVAL;
    if (check_fuse_args(cfg, W_out, g, h) != ENGRAM_OK) return ENGRAM_EINVAL;
    if (!aligned(tables, 16) || !aligned(tokens, 4) || !aligned(seq_offsets, 8)) return ENGRAM_EINVAL;
    // as engram_forward: a size the scratch cannot hold only after every argument check
    if (n_query > ENGRAM_NO_WORKSPACE_MAX_QUERY) return ENGRAM_ENOMEM;
    uint16_t *X = nullptr;
    engram_status s = no_workspace_scratch(&X);
    if (s != ENGRAM_OK) return s;
    cudaStream_t st = (cudaStream_t)stream;
    HashParams hp;
    fill_hash_params(hp, cfg, tokens, seq_offsets, n_seqs, last_n, n_query);
    // X rows [0, n_query) are all written before the projection reads them,
    // and the projection's tensor map stops at n_query rows: nothing left in
    // the array by an earlier call is read, so nothing needs clearing.
    s = gather_launch(IDX_HASH, true, tables, scales_arg(cfg, scales), row_stride(cfg), mx(cfg), nullptr, &hp, n_query,
                      cfg->rows, X, st);
    if (s != ENGRAM_OK) return s;
    return fuse_launch(cfg, nullptr, X, W_out, g, h, n_query, st);
}
