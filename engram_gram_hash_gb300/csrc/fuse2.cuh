// The gated projection for a bf16 X (TMA) with the gate on its own warps.
//
// Same tile, cluster and tcgen05 accumulators as fuse.cuh, with three changes.
// X is not held for the whole tile: every ring stage carries the X K-block
// (128 tokens x 64, 16 KB) beside the W block (64 x 256, 32 KB) it multiplies,
// 3 stages of 48 KB; X is read from L2 once per 256-column chunk.  The
// epilogue is split in two warp roles that run concurrently:
//   - eight gate warps reduce sum(h^2) and <h,g> over this CTA's d slice for
//     the tokens of the NEXT tile while the current one is being updated, and
//     publish the partial sums to the cluster (double-buffered).  They start
//     a tile once the update warps finish the previous tile's first chunk and
//     load with an L2 evict-last hint, so the update warps find those lines
//     in L2;
//   - eight update warps (two per TMEM lane quadrant) combine the cluster's
//     partial sums into each token's gate and apply h = bf16(h + gate * y) to
//     32 x 64 pieces of h that come in and go out by TMA through two 128-byte
//     swizzled staging buffers per warp, one piece landing while the other is
//     updated.
// Eighteen warps, one CTA per SM (at most 112 registers a thread; 96 used).
//
// Partial sums per token are reduced in the same order as in fuse.cuh (lanes
// over 16-byte pieces, a butterfly over the warp, then the G CTAs in rank
// order), so both kernels produce bit-identical gates and h.
//
// Cluster protocol for the partial-sum buffer b (tiles alternate b = 0, 1):
//   part_full[b]: one arrival from every gate warp of every CTA after it
//                 wrote its rows of part[b]; update warps wait on it
//                 (cluster acquire) before reading part[b] of every CTA;
//   part_free[b]: one arrival from every update warp of every CTA after it
//                 read part[b] of every CTA; gate warps wait on it before
//                 writing part[b] again, two tiles later.
// Each signal is one cluster-scope fence followed by relaxed remote arrivals
// (mbar_arrive_cluster_ranks): a release on each of the G arrivals would cost
// a fence each, and those fences sat on the path from the gate pass to the
// update.
//
// Sources: rohitghumare.com "guides/deepseek-v4-1-flash", sections "The
// architecture" (Engram rows are added into the residual stream through a
// learned gate) and "Engram: the table that is never multiplied".
#pragma once

namespace engram {
namespace fuse2 {

using fuse::BK;
using fuse::BM;
using fuse::BN;
using fuse::IDESC;
using fuse::KSTAGES;
using fuse::Params;
using fuse::STAGE_BYTES;
using fuse::TMEM_COLS;
using fuse::X_KBLOCK_BYTES;

constexpr int W_BOX_BYTES = BK * 64 * 2;                      // 8 KB: 64 K-rows x 64 N
constexpr int RING_STAGE_BYTES = X_KBLOCK_BYTES + W_BOX_BYTES * (BN / 64);  // 16 KB X + 32 KB W
// The update warps move h pieces (32 tokens x 64 columns) with TMA loads and
// stores through two staging buffers each.
constexpr int STG_BUFS = 2;

constexpr int UPDATE_WARPS = 8;  // warps 4..11: two per TMEM lane quadrant (4 measured slower)
// The gate warps start reading tile i+1 once the update warps have finished
// chunk LEAD_CHUNK of tile i (-1: as soon as they start tile i).  A shorter
// lead keeps the gate warps' h reads in L2 until the update warps re-read them.
constexpr int LEAD_CHUNK = 0;
constexpr int NUM_WARPS = 18;  // 8 gate warps (16 and 20 warps measured slower)
constexpr int GATE_WARPS = NUM_WARPS - 2 - UPDATE_WARPS;  // warps 2, 3 and 4 + UPDATE_WARPS .. NUM_WARPS - 1
constexpr int PIECES = 4 * 4 / UPDATE_WARPS;    // 64-column pieces of a chunk per update warp
constexpr int NSTAGE = UPDATE_WARPS == 4 ? 4 : 3;  // ring stages that fit beside the staging buffers
constexpr int NUM_THREADS = 32 * NUM_WARPS;

struct Shared {
    uint64_t full[NSTAGE];
    uint64_t empty[NSTAGE];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t part_full[2];
    uint64_t part_free[2];
    uint64_t upd_mark[2];  // local: the update warps reached chunk LEAD_CHUNK of a tile
    uint64_t hb_full[8][2];  // per update warp and staging buffer: a TMA-loaded h piece landed
    uint64_t done;
    uint32_t tmem_base;
    int abort;
    float2 part[2][BM];  // (sum h^2, <h,g>) over this CTA's slice, per token
};

constexpr int SMEM_BYTES = NSTAGE * RING_STAGE_BYTES + UPDATE_WARPS * STG_BUFS * STAGE_BYTES + (int)sizeof(Shared);
static_assert(SMEM_BYTES <= 232448, "fuse2 kernel shared memory over the per-CTA limit");
static_assert(RING_STAGE_BYTES % 1024 == 0 && X_KBLOCK_BYTES % 1024 == 0, "swizzle atoms need 1 KB alignment");

// warps 2, 3 -> gate warps 0, 1; warps 12..15 -> gate warps 2..5
__device__ __forceinline__ int gate_warp_index(int warp) { return warp < 4 ? warp - 2 : warp - 2 - UPDATE_WARPS; }

// KB: 64-wide K-blocks of X (8: the concatenated [T,512] X; 4: one Engram
// layer's [T,256] X).  GATED: the rmsnorm-sigmoid token gate of the concatenated
// form; without it h = bf16(h + y) (the per-layer form gates rows before the
// projection) and the gate warps stay idle.
template <int CPG, int KB = KSTAGES, bool GATED = true>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    fuse2_kernel(const __grid_constant__ CUtensorMap w_map, const __grid_constant__ CUtensorMap x_map,
                 const __grid_constant__ CUtensorMap h_map, const __grid_constant__ Params p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    if ((smem_u32(smem) & 1023u) != 0) {  // same for every CTA: all leave together
        if (threadIdx.x == 0) raise_error(ENGRAM_EUNSUPPORTED);
        return;
    }
    uint8_t *ring = smem;
    uint8_t *stage_smem = ring + NSTAGE * RING_STAGE_BYTES;
    Shared *sh = reinterpret_cast<Shared *>(stage_smem + UPDATE_WARPS * STG_BUFS * STAGE_BYTES);
    volatile int *abort = &sh->abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int64_t cl = cluster_id_x();
    const int64_t n_cl = nclusters_x();
    const int c0 = (int)rank * CPG;  // first chunk of this CTA's d slice
    const int64_t col0 = (int64_t)c0 * BN;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(&sh->full[s], 1);
            mbar_init(&sh->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sh->acc_full[b], 1);
            mbar_init(&sh->acc_empty[b], UPDATE_WARPS);
            mbar_init(&sh->part_full[b], GATE_WARPS * p.groups);
            mbar_init(&sh->part_free[b], UPDATE_WARPS * p.groups);
            mbar_init(&sh->upd_mark[b], UPDATE_WARPS);
            for (int w = 0; w < UPDATE_WARPS; ++w) mbar_init(&sh->hb_full[w][b], 1);
        }
        mbar_init(&sh->done, 1);
        sh->abort = 0;
        fence_mbar_init();
        prefetch_tensormap(&w_map);
        prefetch_tensormap(&x_map);
        prefetch_tensormap(&h_map);
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
            uint32_t phase = 0;
            bool issued[NSTAGE] = {};
            uint32_t issued_parity[NSTAGE] = {};
            // X is the previous kernel's output; h and g, which the gate warps
            // read meanwhile, are not written by it (launched as a programmatic
            // dependent of the gather only).
            grid_dependency_wait();
            for (int64_t mt = cl; mt < p.m_tiles && !*abort; mt += n_cl) {
                for (int c = c0; c < c0 + CPG && !*abort; ++c) {
                    for (int ks = 0; ks < KB; ++ks) {
                        if (!mbar_wait(&sh->empty[stage], phase ^ 1u, abort)) break;
                        mbar_arrive_expect_tx(&sh->full[stage], RING_STAGE_BYTES);
                        uint8_t *dst = ring + stage * RING_STAGE_BYTES;
                        tma_load_2d(dst, &x_map, &sh->full[stage], ks * BK, (int)(mt * BM));
#pragma unroll
                        for (int b = 0; b < BN / 64; ++b)
                            tma_load_2d(dst + X_KBLOCK_BYTES + b * W_BOX_BYTES, &w_map, &sh->full[stage], c * BN + b * 64,
                                        ks * BK);
                        issued[stage] = true;
                        issued_parity[stage] = phase;
                        if (++stage == NSTAGE) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
            // Never leave the CTA with a copy still landing in its shared memory.
            int no_abort = 0;
            for (int s = 0; s < NSTAGE; ++s)
                if (issued[s]) mbar_wait(&sh->full[s], issued_parity[s], &no_abort, 200000000ull);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer ----
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t acc_it = 0;
            const uint32_t ring_addr = smem_u32(ring);
            bool ok = true;
            for (int64_t mt = cl; mt < p.m_tiles && ok && !*abort; mt += n_cl) {
                for (int c = 0; c < CPG && ok; ++c, ++acc_it) {
                    const uint32_t buf = acc_it & 1u;
                    const uint32_t use = acc_it >> 1;
                    if (!mbar_wait(&sh->acc_empty[buf], (use & 1u) ^ 1u, abort)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + buf * BN;
                    for (int ks = 0; ks < KB; ++ks) {
                        if (!mbar_wait(&sh->full[stage], phase, abort)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t st_addr = ring_addr + stage * RING_STAGE_BYTES;
#pragma unroll
                        for (int s = 0; s < BK / 16; ++s) {
                            // A: the stage's X K-block, 32 bytes per K-step into each 128-byte swizzled row
                            const uint64_t adesc = smem_desc(st_addr + s * 32, 16, 1024, kSwizzle128B);
                            // B: 16 K-rows (2 x 8-row groups of 1 KB) further; N atoms of 64 are 8 KB apart
                            const uint64_t bdesc =
                                smem_desc(st_addr + X_KBLOCK_BYTES + s * 2048, W_BOX_BYTES, 1024, kSwizzle128B);
                            mma_bf16(d_tmem, adesc, bdesc, IDESC, (ks | s) != 0);
                        }
                        mma_commit(&sh->empty[stage]);
                        if (++stage == NSTAGE) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (ok) mma_commit(&sh->acc_full[buf]);
                }
            }
            // All MMAs issued by this thread complete before TMEM is released.
            mma_commit(&sh->done);
            int no_abort = 0;
            mbar_wait(&sh->done, 0, &no_abort, 200000000ull);
        }
    } else if (warp >= 4 && warp < 4 + UPDATE_WARPS) {
        // ------------------------------------------------- update warps -----
        const int ew = warp - 4;        // 0..7
        const int q = warp & 3;         // TMEM lane quadrant of this warp
        const int ch = ew >> 2;         // which group of PIECES 64-column pieces of each chunk
        const int row = q * 32 + lane;  // token row within the tile owned by this thread
        uint32_t it = 0;
        uint32_t acc_it = 0;
        uint32_t gp = 0;  // h pieces this warp has handled (staging buffer gp & 1)
        uint32_t loaded = 0;  // h pieces this warp has requested by TMA (lane 0)
        uint8_t *const stg0 = stage_smem + ew * STG_BUFS * STAGE_BYTES;
        // column offset of this warp's piece k of a chunk
        auto piece_col = [&](int k) -> int { return (ch * PIECES + k) * 64; };
        if (lane == 0 && cl < p.m_tiles) {  // the first piece
            mbar_arrive_expect_tx(&sh->hb_full[ew][0], STAGE_BYTES);
            tma_load_2d(stg0, &h_map, &sh->hb_full[ew][0], (int)(col0 + piece_col(0)), (int)(cl * BM + q * 32));
            loaded = 1;
        }
        for (int64_t mt = cl; mt < p.m_tiles && !*abort; mt += n_cl, ++it) {
            const int64_t m0 = mt * BM;
            const uint32_t pb = it & 1u;
            float gate = 1.f;
            if constexpr (GATED) {
                if (!mbar_wait_cluster(&sh->part_full[pb], (it >> 1) & 1u, abort)) break;
                float ssum = 0.f, dsum = 0.f;
                const uint32_t my_part = smem_u32(&sh->part[pb][row]);
                for (int r = 0; r < p.groups; ++r) {  // same order in every CTA
                    const float2 v = ld_shared_cluster_f2(mapa_shared(my_part, (uint32_t)r));
                    ssum += v.x;
                    dsum += v.y;
                }
                const float rinv = rsqrtf(ssum / (float)p.d + p.eps);
                gate = 1.f / (1.f + __expf(-(rinv * dsum * p.inv_sqrt_d)));
                __syncwarp();
                if (lane == 0) {  // this warp is done with part[pb] of every CTA
                    const uint32_t bar = smem_u32(&sh->part_free[pb]);
                    mbar_arrive_cluster_ranks(bar, p.groups);
                    if (LEAD_CHUNK < 0 || LEAD_CHUNK >= CPG) mbar_arrive(&sh->upd_mark[pb]);
                }
            }

            {
                // h = bf16(h + gate * y) on this warp's 32 rows and its columns
                // of each chunk, in pieces of 64 columns: each piece comes in
                // by TMA (128-byte swizzle: 16-byte chunk c of row r at c ^ (r &
                // 7)) into one of two staging buffers while the previous piece
                // is updated in place and leaves by TMA store.  Rows past the
                // last token are zero-filled on load and clipped on store.
                bool ok = true;
                for (int pc = 0; pc < PIECES * CPG; ++pc, ++gp) {
                    const int c = pc / PIECES, sub = pc % PIECES;
                    const uint32_t buf = (acc_it + c) & 1u;
                    const uint32_t use = (acc_it + c) >> 1;
                    const uint32_t sb = gp & 1u;
                    if (lane == 0) {
                        // the next piece (this tile's, or the first of the next tile)
                        const bool last = pc + 1 == PIECES * CPG;
                        const int64_t mt_n = last ? mt + n_cl : mt;
                        if (mt_n < p.m_tiles) {
                            const int pn = last ? 0 : pc + 1;
                            bulk_wait_group_read0();  // that buffer's previous store has read it
                            mbar_arrive_expect_tx(&sh->hb_full[ew][sb ^ 1u], STAGE_BYTES);
                            tma_load_2d(stg0 + (sb ^ 1u) * STAGE_BYTES, &h_map, &sh->hb_full[ew][sb ^ 1u],
                                        (int)(col0 + (pn / PIECES) * BN + piece_col(pn % PIECES)), (int)(mt_n * BM + q * 32));
                            loaded = gp + 2;
                        }
                    }
                    if (!mbar_wait(&sh->hb_full[ew][sb], (gp >> 1) & 1u, abort)) { ok = false; break; }
                    if (sub == 0) {
                        if (!mbar_wait(&sh->acc_full[buf], use & 1u, abort)) { ok = false; break; }
                        tc_fence_after();
                    }
                    const uint32_t stg_a = smem_u32(stg0 + sb * STAGE_BYTES);
#pragma unroll
                    for (int half = 0; half < 2; ++half) {  // own row: 32 columns at a time
                        uint32_t y[32];
                        tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(q * 32) << 16) + buf * BN + piece_col(sub) + half * 32, y);
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
                                w[k] = GATED ? pack_bf16x2(fmaf(gate, y0, bf16_lo(w[k])), fmaf(gate, y1, bf16_hi(w[k])))
                                             : pack_bf16x2(bf16_lo(w[k]) + y0, bf16_hi(w[k]) + y1);
                            }
                            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]) : "memory");
                        }
                    }
                    fence_proxy_async_smem();  // this thread's writes are visible to the TMA store
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&h_map, stg0 + sb * STAGE_BYTES, (int)(col0 + c * BN + piece_col(sub)),
                                     (int)(m0 + q * 32));
                        bulk_commit_group();
                    }
                    if (sub == PIECES - 1) {
                        tc_fence_before();
                        if (lane == 0) {
                            mbar_arrive(&sh->acc_empty[buf]);
                            if (GATED && c == LEAD_CHUNK) mbar_arrive(&sh->upd_mark[pb]);
                        }
                    }
                }
                acc_it += CPG;
                if (!ok) break;
            }
        }
        if (lane == 0) {
            bulk_wait_group0();  // stores complete before the CTA leaves
            int no_abort = 0;    // and no requested piece is still landing (after an abort)
            for (uint32_t k = gp; k < loaded; ++k)
                mbar_wait(&sh->hb_full[ew][k & 1u], (k >> 1) & 1u, &no_abort, 200000000ull);
        }
    } else if (GATED) {
        // --------------------------------------------------- gate warps -----
        // Rows in batches of RB (16 16-byte loads per lane in flight), batch b
        // on gate warp b mod 6.  Lanes stride over each row's 16-byte pieces;
        // g is re-read per batch (L1) rather than held in registers.  The h
        // lines are loaded with an L2 evict-last hint: the update warps read
        // them again within the next tile.
        const int gw = gate_warp_index(warp);
        const uint64_t keep = l2_policy_evict_last();  // the update warps re-read these lines
        constexpr int RB = 16 / CPG;
        constexpr int NB = BM / RB;
        uint32_t it = 0;
        for (int64_t mt = cl; mt < p.m_tiles && !*abort; mt += n_cl, ++it) {
            const int64_t m0 = mt * BM;
            const uint32_t pb = it & 1u;
            const uint32_t use = it >> 1;
            if (use > 0 && !mbar_wait_cluster(&sh->part_free[pb], (use - 1u) & 1u, abort)) break;
            if (it > 0 && !mbar_wait(&sh->upd_mark[pb ^ 1u], ((it - 1u) >> 1) & 1u, abort)) break;
            for (int b = gw; b < NB; b += GATE_WARPS) {
                const int rbase = b * RB;
                uint4 hv[RB][CPG];
#pragma unroll
                for (int r = 0; r < RB; ++r) {
                    const int64_t t = m0 + rbase + r;
#pragma unroll
                    for (int k = 0; k < CPG; ++k)
                        hv[r][k] = t < p.n_query ? ld_v4_l2_hint(p.h + t * p.d + col0 + (lane + 32 * k) * 8, keep)
                                                 : make_uint4(0, 0, 0, 0);
                }
                float s[RB], d[RB];
#pragma unroll
                for (int r = 0; r < RB; ++r) s[r] = d[r] = 0.f;
#pragma unroll
                for (int k = 0; k < CPG; ++k) {
                    const uint4 gk = __ldg(reinterpret_cast<const uint4 *>(p.g + col0) + lane + 32 * k);
                    const uint32_t gw4[4] = {gk.x, gk.y, gk.z, gk.w};
#pragma unroll
                    for (int r = 0; r < RB; ++r) {
                        const uint32_t hw[4] = {hv[r][k].x, hv[r][k].y, hv[r][k].z, hv[r][k].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float a0 = bf16_lo(hw[e]), a1 = bf16_hi(hw[e]);
                            s[r] = fmaf(a0, a0, s[r]);
                            s[r] = fmaf(a1, a1, s[r]);
                            d[r] = fmaf(a0, bf16_lo(gw4[e]), d[r]);
                            d[r] = fmaf(a1, bf16_hi(gw4[e]), d[r]);
                        }
                    }
                }
#pragma unroll
                for (int r = 0; r < RB; ++r) {
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        s[r] += __shfl_xor_sync(0xffffffffu, s[r], o);
                        d[r] += __shfl_xor_sync(0xffffffffu, d[r], o);
                    }
                    if (lane == 0) sh->part[pb][rbase + r] = make_float2(s[r], d[r]);
                }
            }
            __syncwarp();
            if (lane == 0) {
                const uint32_t bar = smem_u32(&sh->part_full[pb]);
                mbar_arrive_cluster_ranks(bar, p.groups);
            }
        }
    }

    // No CTA leaves while a peer may still read its partial sums or arrive on
    // its barriers, and TMEM is released only after every MMA and TMEM load of
    // this CTA is done.
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

}  // namespace fuse2
}  // namespace engram
