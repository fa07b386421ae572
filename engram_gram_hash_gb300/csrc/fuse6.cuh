// The gated projection into the residual stream, X held in TMEM.
//
// Same arithmetic as fuse.cuh (bf16 X times bf16 W_out into fp32 TMEM
// accumulators, a gate from the rms-normalised dot of h with g, h updated in
// bf16), laid out so that shared memory is spent on pipelining instead of on
// the X tile:
//   - X [128 tokens x 512] bf16 lives in TMEM (256 columns) as the MMA's A
//     operand.  It arrives by TMA in 16 KB K-blocks through two shared-memory
//     slots and is moved into TMEM with tcgen05.cp (128 rows x 32 bytes each).
//   - The MMA is M=128, N=128, K=16 (A from TMEM, B = W_out from shared
//     memory), into two 128-column accumulators.
//   - W_out streams through a 6-stage TMA ring of [64 K-rows x 128 N]
//     (MN-major, 128-byte swizzle), 96 KB.
//   - Two gate warps compute the next tile's partial gate sums while the
//     eight epilogue warps finish the current tile (coalesced loads, two row
//     groups in flight) and publish them to the cluster.  This also leaves the
//     next tile's h in L2 for its epilogue.
//   - The epilogue is the one of fuse.cuh: coalesced whole-line h accesses
//     through a swizzled per-warp staging tile, each thread updating the row
//     its TMEM lane holds.
// Work split, gate exchange through DSMEM and bit-identical gates across the
// cluster are as in fuse.cuh.
//
// Sources: rohitghumare.com "guides/deepseek-v4-1-flash", sections "The
// architecture" (Engram rows are added into the residual stream through a
// learned gate) and "Engram: the table that is never multiplied".
#pragma once

namespace engram {
namespace fuse6 {

constexpr int BM = 128;                        // tokens per tile (TMEM lanes)
constexpr int BN = 128;                        // columns per chunk (MMA N)
constexpr int BK = 64;                         // K per W stage and per X slot
constexpr int KBLOCKS = kMem / BK;             // 8
constexpr int NSTAGE = 6;                      // W ring depth
constexpr int W_BOX_BYTES = BK * 64 * 2;       // 8 KB: 64 K-rows x 64 N
constexpr int W_STAGE_BYTES = 2 * W_BOX_BYTES; // 16 KB
constexpr int X_SLOT_BYTES = BM * BK * 2;      // 16 KB: 128 rows x 64 K
constexpr int X_SLOTS = 2;
constexpr int EPI_WARPS = 8;                   // two per TMEM lane quadrant
constexpr int GATE_WARPS = 2;
constexpr int NUM_THREADS = 32 * (2 + EPI_WARPS + GATE_WARPS);  // 384
constexpr int STAGE_BYTES = 32 * 128;          // epilogue staging: 32 rows x 64 bf16
constexpr int TMEM_COLS = 512;
constexpr int X_TMEM = 0;                      // columns [0, 256): X
constexpr int ACC_TMEM = 256;                  // columns [256, 512): two accumulators
constexpr int MAX_GROUPS = 8;
constexpr uint32_t IDESC = idesc_bf16(BM, BN, /*b_mn_major=*/true);

constexpr int OFF_W = 0;
constexpr int OFF_X = OFF_W + NSTAGE * W_STAGE_BYTES;
constexpr int OFF_STG = OFF_X + X_SLOTS * X_SLOT_BYTES;
constexpr int OFF_GATE = OFF_STG + EPI_WARPS * STAGE_BYTES;
constexpr int OFF_SH = OFF_GATE;  // the gate warps read h straight from global memory

struct Shared {
    uint64_t w_full[NSTAGE];
    uint64_t w_empty[NSTAGE];
    uint64_t x_full[X_SLOTS];
    uint64_t x_empty[X_SLOTS];
    uint64_t mma_done;      // every MMA of a tile complete (X in TMEM may be replaced)
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t gate_bar[2];   // partial sums of a tile published by every CTA
    uint64_t part_free[2];  // partial sums of a tile read by every CTA
    uint64_t done;
    uint32_t tmem_base;
    int abort;
    float2 part[2][BM];     // (sum h^2, <h,g>) over this CTA's slice, per token
};

// 96 KB W ring + 32 KB X slots + 32 KB epilogue staging + barriers/partials,
// of the 232,448 B a CTA may use.
constexpr int SMEM_BYTES = OFF_SH + (int)sizeof(Shared);
static_assert(SMEM_BYTES <= 232448, "fuse6 shared memory over the per-CTA limit");

struct Params {
    const uint16_t *g;  // [d] bf16
    uint16_t *h;        // [n_query][d] bf16, in place
    int64_t n_query;
    int64_t m_tiles;
    int32_t d;
    int32_t groups;     // CTAs per cluster = d slices
    int32_t nch;        // 128-column chunks per CTA (the kernel's NCH)
    float eps;
    float inv_sqrt_d;
};

template <int NCH>
__global__ void __maxnreg__(168)  // 12 warps: 3 share a sub-partition (16K registers) -> 168 per thread
    fuse6_kernel(const __grid_constant__ CUtensorMap w_map, const __grid_constant__ CUtensorMap x_map,
                 const __grid_constant__ Params p) {
    constexpr int SLICE_BYTES = NCH * BN * 2;  // one row's slice of h
    extern __shared__ __align__(1024) uint8_t smem[];
    if ((smem_u32(smem) & 1023u) != 0) {  // same for every CTA: all leave together
        if (threadIdx.x == 0) raise_error(ENGRAM_EUNSUPPORTED);
        return;
    }
    Shared *sh = reinterpret_cast<Shared *>(smem + OFF_SH);
    volatile int *abort = &sh->abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int64_t cl = cluster_id_x();
    const int64_t n_cl = nclusters_x();
    const int64_t col0 = (int64_t)rank * NCH * BN;  // this CTA's d slice

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(&sh->w_full[s], 1);
            mbar_init(&sh->w_empty[s], 1);
        }
        for (int s = 0; s < X_SLOTS; ++s) {
            mbar_init(&sh->x_full[s], 1);
            mbar_init(&sh->x_empty[s], 1);
        }
        mbar_init(&sh->mma_done, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sh->acc_full[b], 1);
            mbar_init(&sh->acc_empty[b], EPI_WARPS);
            mbar_init(&sh->gate_bar[b], GATE_WARPS * p.groups);
            mbar_init(&sh->part_free[b], EPI_WARPS * p.groups);
        }
        mbar_init(&sh->done, 1);
        sh->abort = 0;
        fence_mbar_init();
        prefetch_tensormap(&w_map);
        prefetch_tensormap(&x_map);
    }
    if (warp == 1) {
        tmem_alloc(&sh->tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    cluster_sync_all();  // barriers of every CTA initialised before any remote arrival
    tc_fence_after();
    const uint32_t tmem_base = sh->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer ------
        if (lane == 0) {
            int stage = 0;
            uint32_t wph = 0;
            uint32_t xk = 0;  // X blocks issued (global sequence: tile-major, 8 per tile)
            bool w_issued[NSTAGE] = {};
            uint32_t w_par[NSTAGE] = {};
            // X block number xk -> (tile, kb); issue it if its slot is free
            auto x_tile = [&](uint32_t k) -> int64_t { return cl + (int64_t)(k / KBLOCKS) * n_cl; };
            auto issue_x = [&](bool block) -> bool {
                if (x_tile(xk) >= p.m_tiles) return false;
                const uint32_t slot = xk % X_SLOTS, use = xk / X_SLOTS;
                if (block) {
                    if (!mbar_wait(&sh->x_empty[slot], (use & 1u) ^ 1u, abort)) return false;
                } else if (!mbar_try_wait(&sh->x_empty[slot], (use & 1u) ^ 1u)) {
                    return false;
                }
                mbar_arrive_expect_tx(&sh->x_full[slot], X_SLOT_BYTES);
                tma_load_2d(smem + OFF_X + slot * X_SLOT_BYTES, &x_map, &sh->x_full[slot], (int)(xk % KBLOCKS) * BK,
                            (int)(x_tile(xk) * BM));
                ++xk;
                return true;
            };
            uint32_t it = 0;
            for (int64_t mt = cl; mt < p.m_tiles && !*abort; mt += n_cl, ++it) {
                while (xk < (it + 1) * KBLOCKS && !*abort)  // this tile's X
                    if (!issue_x(true)) break;
                for (int c = 0; c < NCH && !*abort; ++c) {
                    for (int ks = 0; ks < KBLOCKS; ++ks) {
                        while (xk < (it + 1) * KBLOCKS + X_SLOTS && issue_x(false)) {
                        }  // next tile's first X blocks, whenever a slot frees up
                        if (!mbar_wait(&sh->w_empty[stage], wph ^ 1u, abort)) break;
                        mbar_arrive_expect_tx(&sh->w_full[stage], W_STAGE_BYTES);
                        uint8_t *dst = smem + OFF_W + stage * W_STAGE_BYTES;
                        const int n0 = (int)(col0 + c * BN);
                        tma_load_2d(dst, &w_map, &sh->w_full[stage], n0, ks * BK);
                        tma_load_2d(dst + W_BOX_BYTES, &w_map, &sh->w_full[stage], n0 + 64, ks * BK);
                        w_issued[stage] = true;
                        w_par[stage] = wph;
                        if (++stage == NSTAGE) {
                            stage = 0;
                            wph ^= 1u;
                        }
                    }
                }
            }
            // Never leave the CTA with a copy still landing in its shared memory.
            int no_abort = 0;
            for (int s = 0; s < NSTAGE; ++s)
                if (w_issued[s]) mbar_wait(&sh->w_full[s], w_par[s], &no_abort, 200000000ull);
            for (uint32_t k = (xk >= X_SLOTS ? xk - X_SLOTS : 0); k < xk; ++k)
                mbar_wait(&sh->x_full[k % X_SLOTS], (k / X_SLOTS) & 1u, &no_abort, 200000000ull);
        }
    } else if (warp == 1) {
        // ------------------------------------ X into TMEM, then the MMAs -----
        if (lane == 0) {
            int stage = 0;
            uint32_t wph = 0;
            uint32_t xk = 0;
            uint32_t acc_it = 0;
            uint32_t it = 0;
            bool ok = true;
            for (int64_t mt = cl; mt < p.m_tiles && ok && !*abort; mt += n_cl, ++it) {
                if (it > 0) {  // every MMA of the previous tile has read X
                    if (!mbar_wait(&sh->mma_done, (it - 1) & 1u, abort)) break;
                }
                for (int kb = 0; kb < KBLOCKS && ok; ++kb, ++xk) {
                    const uint32_t slot = xk % X_SLOTS, use = xk / X_SLOTS;
                    if (!mbar_wait(&sh->x_full[slot], use & 1u, abort)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t src = smem_u32(smem + OFF_X + slot * X_SLOT_BYTES);
#pragma unroll
                    for (int s = 0; s < BK / 16; ++s)  // 16 K-elements (32 bytes of each row) per copy
                        tmem_cp_128x256b(tmem_base + X_TMEM + kb * (BK / 2) + s * 8,
                                         smem_desc(src + s * 32, 16, 1024, kSwizzle128B));
                    mma_commit(&sh->x_empty[slot]);
                }
                for (int c = 0; c < NCH && ok; ++c, ++acc_it) {
                    const uint32_t buf = acc_it & 1u;
                    const uint32_t use = acc_it >> 1;
                    if (!mbar_wait(&sh->acc_empty[buf], (use & 1u) ^ 1u, abort)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + ACC_TMEM + buf * BN;
                    for (int ks = 0; ks < KBLOCKS; ++ks) {
                        if (!mbar_wait(&sh->w_full[stage], wph, abort)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t wb = smem_u32(smem + OFF_W + stage * W_STAGE_BYTES);
#pragma unroll
                        for (int s = 0; s < BK / 16; ++s)
                            mma_bf16_ta(d_tmem, tmem_base + X_TMEM + ks * (BK / 2) + s * 8,
                                        smem_desc(wb + s * 2048, W_BOX_BYTES, 1024, kSwizzle128B), IDESC,
                                        (ks | s) != 0);
                        mma_commit(&sh->w_empty[stage]);
                        if (++stage == NSTAGE) {
                            stage = 0;
                            wph ^= 1u;
                        }
                    }
                    if (ok) mma_commit(&sh->acc_full[buf]);
                }
                if (ok) mma_commit(&sh->mma_done);
            }
            // All tcgen05 work issued by this thread completes before TMEM is released.
            mma_commit(&sh->done);
            int no_abort = 0;
            mbar_wait(&sh->done, 0, &no_abort, 200000000ull);
        }
    } else if (warp < 2 + EPI_WARPS) {
        // ------------------------------------------------------ epilogue ----
        const int ew = warp - 2;        // 0..7
        const int q = warp & 3;         // TMEM lane quadrant of this warp
        const int ch = ew >> 2;         // which 64-column half of each chunk
        const int row = q * 32 + lane;  // token row within the tile owned by this thread
        uint8_t *stg = smem + OFF_STG + ew * STAGE_BYTES;
        const uint32_t stg_a = smem_u32(stg);
        const int lr = lane >> 3, lc = lane & 7;  // coalesced role: row 4j + lr, 16-byte chunk lc
        uint32_t it = 0;
        uint32_t acc_it = 0;
        for (int64_t mt = cl; mt < p.m_tiles && !*abort; mt += n_cl, ++it) {
            const int64_t m0 = mt * BM;
            const uint32_t pb = it & 1u;
            auto piece_ptr = [&](int c, int j) -> uint16_t * {
                const int64_t t = m0 + q * 32 + 4 * j + lr;
                return p.h + t * p.d + col0 + (int64_t)c * BN + ch * 64 + lc * 8;
            };
            auto row_live = [&](int j) -> bool { return m0 + q * 32 + 4 * j + lr < p.n_query; };
            uint4 a[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) a[j] = row_live(j) ? *reinterpret_cast<const uint4 *>(piece_ptr(0, j)) : make_uint4(0, 0, 0, 0);

            // this tile's gate from the partial sums every CTA published
            if (!mbar_wait_cluster(&sh->gate_bar[pb], (it >> 1) & 1u, abort)) break;
            float ssum = 0.f, dsum = 0.f;
            const uint32_t my_part = smem_u32(&sh->part[pb][row]);
            for (int r = 0; r < p.groups; ++r) {  // same order in every CTA
                const float2 v = ld_shared_cluster_f2(mapa_shared(my_part, (uint32_t)r));
                ssum += v.x;
                dsum += v.y;
            }
            __syncwarp();
            if (lane == 0) {  // done reading every CTA's part[pb]
                const uint32_t bar = smem_u32(&sh->part_free[pb]);
                for (int r = 0; r < p.groups; ++r) mbar_arrive_remote(mapa_shared(bar, (uint32_t)r));
            }
            const float rinv = rsqrtf(ssum / (float)p.d + p.eps);
            const float gate = 1.f / (1.f + __expf(-(rinv * dsum * p.inv_sqrt_d)));

            bool ok = true;
            for (int c = 0; c < NCH; ++c, ++acc_it) {
                const uint32_t buf = acc_it & 1u;
                const uint32_t use = acc_it >> 1;
#pragma unroll
                for (int j = 0; j < 8; ++j) {  // h piece -> staging (coalesced layout)
                    const int r = 4 * j + lr;
                    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(stg_a + r * 128 + ((lc ^ (r & 7)) << 4)),
                                 "r"(a[j].x), "r"(a[j].y), "r"(a[j].z), "r"(a[j].w)
                                 : "memory");
                }
                if (c + 1 < NCH) {  // next piece in flight during this one
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        a[j] = row_live(j) ? *reinterpret_cast<const uint4 *>(piece_ptr(c + 1, j)) : make_uint4(0, 0, 0, 0);
                }
                if (!mbar_wait(&sh->acc_full[buf], use & 1u, abort)) { ok = false; break; }
                tc_fence_after();
                __syncwarp();
#pragma unroll
                for (int half = 0; half < 2; ++half) {  // own row: 32 columns at a time
                    uint32_t y[32];
                    tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(q * 32) << 16) + ACC_TMEM + buf * BN + ch * 64 + half * 32, y);
                    tmem_ld_wait();
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4) {
                        const int cch = half * 4 + k4;
                        const uint32_t addr = stg_a + lane * 128 + ((cch ^ (lane & 7)) << 4);
                        uint32_t w[4];
                        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "r"(addr) : "memory");
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float y0 = __uint_as_float(y[8 * k4 + 2 * k]);
                            const float y1 = __uint_as_float(y[8 * k4 + 2 * k + 1]);
                            w[k] = pack_bf16x2(fmaf(gate, y0, bf16_lo(w[k])), fmaf(gate, y1, bf16_hi(w[k])));
                        }
                        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]) : "memory");
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh->acc_empty[buf]);  // TMEM reads of this chunk done
#pragma unroll
                for (int j = 0; j < 8; ++j) {  // staging -> h (coalesced)
                    const int r = 4 * j + lr;
                    uint4 o;
                    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(o.x), "=r"(o.y), "=r"(o.z), "=r"(o.w) : "r"(stg_a + r * 128 + ((lc ^ (r & 7)) << 4)) : "memory");
                    if (row_live(j)) *reinterpret_cast<uint4 *>(piece_ptr(c, j)) = o;
                }
                __syncwarp();
            }
            if (!ok) break;
        }
    } else {
        // ---------------------------------------------------- gate warps ----
        // Warp gw reduces rows gw*64 .. gw*64+63 of every tile of this CTA's
        // cluster, in order, up to two tiles ahead of the epilogue.  Lanes
        // stride over each row's 16-byte pieces (coalesced loads); two groups
        // of RG rows are in flight while the previous group is reduced.
        const int gw = warp - 2 - EPI_WARPS;
        constexpr int PIECES = SLICE_BYTES / 16;  // 16-byte pieces per row slice
        constexpr int PER_LANE = (PIECES + 31) / 32;
        constexpr int RG = PER_LANE >= 8 ? 2 : 8 / PER_LANE;  // rows per group
        constexpr int ROWS = BM / GATE_WARPS;                // 64
        uint4 gv[PER_LANE];
#pragma unroll
        for (int k = 0; k < PER_LANE; ++k) {
            const int pc = lane + 32 * k;
            gv[k] = pc < PIECES ? __ldg(reinterpret_cast<const uint4 *>(p.g + col0) + pc) : make_uint4(0, 0, 0, 0);
        }
        auto load_group = [&](int64_t r0, uint4 (&dst)[RG][PER_LANE]) {
#pragma unroll
            for (int i = 0; i < RG; ++i)
#pragma unroll
                for (int kk = 0; kk < PER_LANE; ++kk) {
                    const int pc = lane + 32 * kk;
                    const int64_t t = r0 + i;
                    dst[i][kk] = (pc < PIECES && t < p.n_query)
                                     ? *reinterpret_cast<const uint4 *>(p.h + t * p.d + col0 + (int64_t)pc * 8)
                                     : make_uint4(0, 0, 0, 0);
                }
        };
        uint32_t k = 0;
        for (int64_t mt = cl; mt < p.m_tiles && !*abort; mt += n_cl, ++k) {
            const uint32_t pb = k & 1u;
            if (k >= 2) {  // every CTA has read the partials this buffer held two tiles ago
                if (!mbar_wait_cluster(&sh->part_free[pb], ((k - 2) >> 1) & 1u, abort)) break;
            }
            const int64_t r0 = mt * BM + gw * ROWS;
            uint4 cur[RG][PER_LANE], nxt[RG][PER_LANE];
            load_group(r0, nxt);
            for (int r = 0; r < ROWS; r += RG) {
#pragma unroll
                for (int i = 0; i < RG; ++i)
#pragma unroll
                    for (int kk = 0; kk < PER_LANE; ++kk) cur[i][kk] = nxt[i][kk];
                if (r + RG < ROWS) load_group(r0 + r + RG, nxt);
                float s[RG], d[RG];
#pragma unroll
                for (int i = 0; i < RG; ++i) {
                    s[i] = 0.f;
                    d[i] = 0.f;
#pragma unroll
                    for (int kk = 0; kk < PER_LANE; ++kk) {
                        const uint32_t hw[4] = {cur[i][kk].x, cur[i][kk].y, cur[i][kk].z, cur[i][kk].w};
                        const uint32_t gwd[4] = {gv[kk].x, gv[kk].y, gv[kk].z, gv[kk].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float a0 = bf16_lo(hw[e]), a1 = bf16_hi(hw[e]);
                            s[i] = fmaf(a0, a0, s[i]);
                            s[i] = fmaf(a1, a1, s[i]);
                            d[i] = fmaf(a0, bf16_lo(gwd[e]), d[i]);
                            d[i] = fmaf(a1, bf16_hi(gwd[e]), d[i]);
                        }
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                    for (int i = 0; i < RG; ++i) {
                        s[i] += __shfl_xor_sync(0xffffffffu, s[i], o);
                        d[i] += __shfl_xor_sync(0xffffffffu, d[i], o);
                    }
                if (lane == 0)
#pragma unroll
                    for (int i = 0; i < RG; ++i) sh->part[pb][gw * ROWS + r + i] = make_float2(s[i], d[i]);
            }
            __syncwarp();
            if (lane == 0) {  // publish this tile's partial sums to every CTA
                const uint32_t bar = smem_u32(&sh->gate_bar[pb]);
                for (int r = 0; r < p.groups; ++r) mbar_arrive_remote(mapa_shared(bar, (uint32_t)r));
            }
        }
    }

    // No CTA leaves while a peer may still read its partial sums, and TMEM is
    // released only after every MMA, copy and TMEM load of this CTA is done.
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

}  // namespace fuse6
}  // namespace engram
