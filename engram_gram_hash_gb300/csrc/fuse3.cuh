// The gated projection for a bf16 X (TMA) with the residual slice held in
// shared memory.
//
// A cluster of G CTAs shares a tile of 128 tokens and splits d into G slices
// of CPG (1 or 2) 256-column chunks.  Per tile, every CTA
//   1. loads its h slice [128 x CPG*256] into shared memory with TMA, in
//      boxes of 128 tokens x 64 columns (128-byte swizzle);
//   2. reduces sum(h^2) and <h,g> over the slice from shared memory and
//      exchanges the partial sums with the cluster (distributed shared memory,
//      a cluster fence then relaxed remote mbarrier arrivals, cluster-scope
//      acquire), so every CTA holds
//      the same gate per token;
//   3. applies h = bf16(h + gate * y) in place in shared memory, chunk by
//      chunk as the tcgen05 accumulators (M=128, N=256, fp32 in TMEM,
//      double-buffered) become ready, and writes each warp's updated boxes
//      back with TMA stores.
// h therefore crosses HBM exactly once in each direction, in bulk copies that
// keep a whole slice in flight, instead of being read twice through
// registers.  X and W_out stream through a ring of 48 KB stages (X K-block of
// 128 x 64 beside the W block of 64 x 256 it multiplies).
//
// Partial sums per token are reduced in the same order as in fuse.cuh (lane l
// over the slice's 16-byte pieces l, l+32, ..., a butterfly over the warp,
// then the G CTAs in rank order), so all projection kernels produce
// bit-identical gates and h.
//
// Warps: 0 ring producer (TMA), 1 MMA issuer and TMEM owner, 2 h loader,
// 3 idle, 4..11 epilogue (two per TMEM lane quadrant, each owning 128 of a
// chunk's 256 columns).
//
// Sources: rohitghumare.com "guides/deepseek-v4-1-flash", sections "The
// architecture" (Engram rows are added into the residual stream through a
// learned gate) and "Engram: the table that is never multiplied".
#pragma once

namespace engram {
namespace fuse3 {

using fuse::BK;
using fuse::BM;
using fuse::BN;
using fuse::IDESC;
using fuse::KSTAGES;
using fuse::Params;
using fuse::TMEM_COLS;
using fuse::X_KBLOCK_BYTES;

constexpr int W_BOX_BYTES = BK * 64 * 2;                                    // 8 KB: 64 K-rows x 64 N
constexpr int RING_STAGE_BYTES = X_KBLOCK_BYTES + W_BOX_BYTES * (BN / 64);  // 16 KB X + 32 KB W
constexpr int H_BOX_BYTES = BM * 128;                                       // 16 KB: 128 tokens x 64 columns
constexpr int EPI_WARPS = 8;                                                // warps 4..11
constexpr int NUM_WARPS = 12;
constexpr int NUM_THREADS = 32 * NUM_WARPS;
constexpr int MAX_RING = 3;
constexpr int ROWS_PER_WARP = BM / EPI_WARPS;  // 16 tokens' partial sums per epilogue warp

template <int CPG>
struct Layout {
    static_assert(CPG == 1 || CPG == 2, "h slice of one or two chunks");
    static constexpr int H_BYTES = CPG * (BN / 64) * H_BOX_BYTES;  // 64 or 128 KB
    static constexpr int NSTAGE = CPG == 1 ? 3 : 2;
    static constexpr int RING_BYTES = NSTAGE * RING_STAGE_BYTES;
};

struct Shared {
    uint64_t full[MAX_RING];
    uint64_t empty[MAX_RING];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t h_full;
    uint64_t h_empty;
    uint64_t gate_bar[2];
    uint64_t done;
    uint32_t tmem_base;
    int abort;
    float2 part[2][BM];  // (sum h^2, <h,g>) over this CTA's slice, per token
};

template <int CPG>
constexpr int smem_bytes() {
    return Layout<CPG>::H_BYTES + Layout<CPG>::RING_BYTES + (int)sizeof(Shared);
}
static_assert(smem_bytes<1>() <= 232448 && smem_bytes<2>() <= 232448, "fuse3 shared memory over the per-CTA limit");
static_assert(RING_STAGE_BYTES % 1024 == 0 && H_BOX_BYTES % 1024 == 0, "swizzle atoms need 1 KB alignment");

template <int CPG>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    fuse3_kernel(const __grid_constant__ CUtensorMap w_map, const __grid_constant__ CUtensorMap x_map,
                 const __grid_constant__ CUtensorMap hl_map, const __grid_constant__ CUtensorMap hs_map,
                 const __grid_constant__ Params p) {
    using L = Layout<CPG>;
    constexpr int NSTAGE = L::NSTAGE;
    extern __shared__ __align__(1024) uint8_t smem[];
    if ((smem_u32(smem) & 1023u) != 0) {  // same for every CTA: all leave together
        if (threadIdx.x == 0) raise_error(ENGRAM_EUNSUPPORTED);
        return;
    }
    uint8_t *h_smem = smem;
    uint8_t *ring = smem + L::H_BYTES;
    Shared *sh = reinterpret_cast<Shared *>(ring + L::RING_BYTES);
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
            mbar_init(&sh->acc_empty[b], EPI_WARPS);
            mbar_init(&sh->gate_bar[b], EPI_WARPS * p.groups);
        }
        mbar_init(&sh->h_full, 1);
        mbar_init(&sh->h_empty, EPI_WARPS);
        mbar_init(&sh->done, 1);
        sh->abort = 0;
        fence_mbar_init();
        prefetch_tensormap(&w_map);
        prefetch_tensormap(&x_map);
        prefetch_tensormap(&hl_map);
        prefetch_tensormap(&hs_map);
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
        // ------------------------------------------- X + W ring producer ----
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool issued[NSTAGE] = {};
            uint32_t issued_parity[NSTAGE] = {};
            grid_dependency_wait();  // X comes from the previous kernel (h does not)
            for (int64_t mt = cl; mt < p.m_tiles && !*abort; mt += n_cl) {
                for (int c = c0; c < c0 + CPG && !*abort; ++c) {
                    for (int ks = 0; ks < KSTAGES; ++ks) {
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
                    for (int ks = 0; ks < KSTAGES; ++ks) {
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
    } else if (warp == 2) {
        // ------------------------------------------------------ h loader ----
        if (lane == 0) {
            uint32_t it = 0;
            bool issued = false;
            for (int64_t mt = cl; mt < p.m_tiles && !*abort; mt += n_cl, ++it) {
                if (it > 0 && !mbar_wait(&sh->h_empty, (it - 1u) & 1u, abort)) break;
                mbar_arrive_expect_tx(&sh->h_full, L::H_BYTES);
#pragma unroll
                for (int b = 0; b < CPG * (BN / 64); ++b)
                    tma_load_2d(h_smem + b * H_BOX_BYTES, &hl_map, &sh->h_full, (int)(col0 + b * 64), (int)(mt * BM));
                issued = true;
            }
            int no_abort = 0;
            if (issued) mbar_wait(&sh->h_full, (it - 1u) & 1u, &no_abort, 200000000ull);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------ epilogue ----
        const int ew = warp - 4;        // 0..7
        const int q = warp & 3;         // TMEM lane quadrant of this warp
        const int ch = ew >> 2;         // which 128-column half of each chunk
        const int row = q * 32 + lane;  // token row within the tile owned by this thread
        const uint32_t h_a = smem_u32(h_smem);
        uint4 gv[CPG];
#pragma unroll
        for (int k = 0; k < CPG; ++k) gv[k] = __ldg(reinterpret_cast<const uint4 *>(p.g + col0) + lane + 32 * k);
        uint32_t it = 0;
        uint32_t acc_it = 0;
        for (int64_t mt = cl; mt < p.m_tiles && !*abort; mt += n_cl, ++it) {
            const int64_t m0 = mt * BM;
            if (!mbar_wait(&sh->h_full, it & 1u, abort)) break;

            // Partial gate sums over the slice, rows ew*16 .. ew*16+15: lane l
            // takes the slice's 16-byte pieces l + 32k of each row.
            const uint32_t pb = it & 1u;
            constexpr int RB = 4;
#pragma unroll 1
            for (int rb = 0; rb < ROWS_PER_WARP; rb += RB) {
                uint4 hv[RB][CPG];
#pragma unroll
                for (int r = 0; r < RB; ++r) {
                    const int tr = ew * ROWS_PER_WARP + rb + r;
#pragma unroll
                    for (int k = 0; k < CPG; ++k) {
                        const int ci = lane + 32 * k;  // 16-byte piece of the slice row
                        const uint32_t addr = h_a + (ci >> 3) * H_BOX_BYTES + tr * 128 + (((ci & 7) ^ (tr & 7)) << 4);
                        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(hv[r][k].x), "=r"(hv[r][k].y), "=r"(hv[r][k].z), "=r"(hv[r][k].w)
                                     : "r"(addr)
                                     : "memory");
                    }
                }
#pragma unroll
                for (int r = 0; r < RB; ++r) {
                    float s = 0.f, d = 0.f;
#pragma unroll
                    for (int k = 0; k < CPG; ++k) {
                        const uint32_t hw[4] = {hv[r][k].x, hv[r][k].y, hv[r][k].z, hv[r][k].w};
                        const uint32_t gw[4] = {gv[k].x, gv[k].y, gv[k].z, gv[k].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float a0 = bf16_lo(hw[e]), a1 = bf16_hi(hw[e]);
                            s = fmaf(a0, a0, s);
                            s = fmaf(a1, a1, s);
                            d = fmaf(a0, bf16_lo(gw[e]), d);
                            d = fmaf(a1, bf16_hi(gw[e]), d);
                        }
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        s += __shfl_xor_sync(0xffffffffu, s, o);
                        d += __shfl_xor_sync(0xffffffffu, d, o);
                    }
                    if (lane == 0) sh->part[pb][ew * ROWS_PER_WARP + rb + r] = make_float2(s, d);
                }
            }
            __syncwarp();
            if (lane == 0) {
                const uint32_t bar = smem_u32(&sh->gate_bar[pb]);
                mbar_arrive_cluster_ranks(bar, p.groups);
            }
            if (!mbar_wait_cluster(&sh->gate_bar[pb], (it >> 1) & 1u, abort)) break;
            float ssum = 0.f, dsum = 0.f;
            const uint32_t my_part = smem_u32(&sh->part[pb][row]);
            for (int r = 0; r < p.groups; ++r) {  // same order in every CTA
                const float2 v = ld_shared_cluster_f2(mapa_shared(my_part, (uint32_t)r));
                ssum += v.x;
                dsum += v.y;
            }
            const float rinv = rsqrtf(ssum / (float)p.d + p.eps);
            const float gate = 1.f / (1.f + __expf(-(rinv * dsum * p.inv_sqrt_d)));

            // h = bf16(h + gate * y): this thread's row, this warp's 128
            // columns of each chunk (two 64-column boxes), in place in the
            // swizzled slice (16-byte piece c of row r at piece c ^ (r & 7)).
            bool ok = true;
            for (int c = 0; c < CPG; ++c) {
                const uint32_t buf = (acc_it + c) & 1u;
                const uint32_t use = (acc_it + c) >> 1;
                if (!mbar_wait(&sh->acc_full[buf], use & 1u, abort)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int box = c * (BN / 64) + ch * 2 + j;
                    const uint32_t rbase = h_a + box * H_BOX_BYTES + row * 128;
#pragma unroll
                    for (int half = 0; half < 2; ++half) {  // 32 columns at a time
                        uint32_t y[32];
                        tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(q * 32) << 16) + buf * BN + ch * 128 + j * 64 + half * 32, y);
                        tmem_ld_wait();
#pragma unroll
                        for (int k4 = 0; k4 < 4; ++k4) {
                            const int cb = half * 4 + k4;
                            const uint32_t addr = rbase + ((cb ^ (row & 7)) << 4);
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
                }
                tc_fence_before();
                fence_proxy_async_smem();  // this thread's writes are visible to the TMA store
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&sh->acc_empty[buf]);
#pragma unroll
                    for (int j = 0; j < 2; ++j) {  // this warp's 32 rows of its two boxes
                        const int box = c * (BN / 64) + ch * 2 + j;
                        tma_store_2d(&hs_map, h_smem + box * H_BOX_BYTES + q * 32 * 128,
                                     (int)(col0 + c * BN + ch * 128 + j * 64), (int)(m0 + q * 32));
                    }
                    bulk_commit_group();
                }
            }
            acc_it += CPG;
            if (!ok) break;
            // The slice is reloaded for the next tile once every warp's stores
            // have read it.
            if (lane == 0) {
                bulk_wait_group_read0();
                mbar_arrive(&sh->h_empty);
            }
        }
        if (lane == 0) bulk_wait_group0();
    }

    // No CTA leaves while a peer may still read its partial sums, and TMEM is
    // released only after every MMA and TMEM load of this CTA is done.
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

}  // namespace fuse3
}  // namespace engram
