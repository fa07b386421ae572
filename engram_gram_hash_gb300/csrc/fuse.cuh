// The gated projection into the residual stream on tcgen05 tensor cores.
// This kernel serves the fp32 mem input (engram_fuse), converting it to the
// bf16 X tile in shared memory; a bf16 X from the gather goes to fuse2.cuh
// (many tiles) or fuse3.cuh (few tiles), which share its tile, split and
// arithmetic.
//
// Work split: a tile is 128 query tokens; a thread-block cluster of G CTAs
// shares a tile and splits d into G slices of d/G columns.  Every CTA holds
// the whole X = bf16(mem) tile [128 x 512] in shared memory (K-major,
// 128-byte swizzle), streams its W_out slice through a 2-stage TMA ring in
// [64 K-rows x 256 N] pieces (MN-major, 128-byte swizzle), and accumulates
// y = X @ W_out in fp32 in TMEM with tcgen05.mma (M=128, N=256, K=16),
// double-buffered over 256-column chunks so the epilogue of one chunk
// overlaps the MMAs of the next.
//
// The gate of a token needs its whole h row, but each CTA only owns d/G
// columns: each CTA reduces sum(h^2) and <h,g> over its slice, the partial
// sums are exchanged through distributed shared memory (one cluster
// fence then relaxed remote mbarrier arrivals, cluster-scope acquire), and every CTA adds the G partials in the
// same order, so all CTAs hold bit-identical gates before any CTA writes h.
//
// Memory access: eight epilogue warps (two per TMEM lane quadrant, each
// owning half of a chunk's columns) move h in coalesced whole-line accesses
// through a small swizzled staging tile per warp, with the next 64-column
// piece's loads in flight while the current one is updated; the gate pass has
// just read the slice, so these loads mostly hit L2.
//
// Sources: rohitghumare.com "guides/deepseek-v4-1-flash", sections "The
// architecture" (Engram rows are added into the residual stream through a
// learned gate) and "Engram: the table that is never multiplied".
#pragma once

namespace engram {
namespace fuse {

constexpr int BM = 128;                            // tokens per tile (TMEM lanes)
constexpr int BN = 256;                            // d columns per chunk (MMA N)
constexpr int BK = 64;                             // K columns per X block (one 128-byte swizzle row)
constexpr int KSTAGES = kMem / BK;                 // 8 X blocks
constexpr int WBK = 64;                            // K rows per W stage
constexpr int WSTAGES = kMem / WBK;                // W stages per chunk
constexpr int W_RING_BYTES = 64 * 1024;            // W ring
constexpr int X_KBLOCK_BYTES = BM * BK * 2;        // 16 KB: 128 rows x 128 B
constexpr int X_BYTES = X_KBLOCK_BYTES * KSTAGES;  // 128 KB
constexpr int W_BOX_BYTES = WBK * 64 * 2;          // WBK K-rows x 64 N
constexpr int W_STAGE_BYTES = W_BOX_BYTES * (BN / 64);
constexpr int NSTAGE = W_RING_BYTES / W_STAGE_BYTES;  // W ring depth
constexpr int TMEM_COLS = 2 * BN;                  // two accumulators
constexpr int EPI_WARPS = 8;                       // two per TMEM lane quadrant
constexpr int NUM_THREADS = 64 + 32 * EPI_WARPS;   // warp0 TMA, warp1 MMA, warps 2..9 epilogue
constexpr int MAX_GROUPS = 8;                      // portable cluster size
constexpr int STAGE_BYTES = 32 * 128;              // per epilogue warp: 32 rows x 64 bf16 (swizzled)
constexpr uint32_t IDESC = idesc_bf16(BM, BN, /*b_mn_major=*/true);

enum XSource { X_FROM_F32_MEM = 0, X_FROM_BF16_TMA = 1 };

struct Shared {
    uint64_t full[NSTAGE];
    uint64_t empty[NSTAGE];
    uint64_t x_full;
    uint64_t x_empty;
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t gate_bar[2];
    uint64_t done;
    uint32_t tmem_base;
    int abort;
    float2 part[2][BM];  // (sum h^2, <h,g>) over this CTA's slice, per token
};

// 128 KB X + 64 KB W ring + 32 KB epilogue staging + barriers/partials =
// 231,552 B of the 232,448 B a CTA may use; the dynamic buffer is declared
// 1024-byte aligned (swizzle atoms).
constexpr int SMEM_BYTES = X_BYTES + NSTAGE * W_STAGE_BYTES + EPI_WARPS * STAGE_BYTES + (int)sizeof(Shared);
static_assert(SMEM_BYTES <= 232448, "fuse kernel shared memory over the per-CTA limit");
static_assert(WBK % 16 == 0 && BK % WBK == 0 && W_RING_BYTES % W_STAGE_BYTES == 0 && NSTAGE >= 2, "W ring shape");

struct Params {
    const float *mem;  // [n_query][512] fp32 (X_FROM_F32_MEM)
    const uint16_t *g; // [d] bf16
    uint16_t *h;       // [n_query][d] bf16, in place
    int64_t n_query;
    int64_t m_tiles;
    int32_t d;
    int32_t groups;    // CTAs per cluster = d slices
    int32_t cpg;       // 256-column chunks per CTA (the kernel's CPG)
    float eps;
    float inv_sqrt_d;
};

template <int XSRC, int CPG>
__global__ void __maxnreg__(168)  // 10 warps: 3 share a sub-partition (16K registers) -> 168 per thread
    fuse_kernel(const __grid_constant__ CUtensorMap w_map, const __grid_constant__ CUtensorMap x_map,
                const __grid_constant__ Params p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    if ((smem_u32(smem) & 1023u) != 0) {  // same for every CTA: all leave together
        if (threadIdx.x == 0) raise_error(ENGRAM_EUNSUPPORTED);
        return;
    }
    uint8_t *x_smem = smem;
    uint8_t *w_smem = smem + X_BYTES;
    uint8_t *stage_smem = w_smem + NSTAGE * W_STAGE_BYTES;
    Shared *sh = reinterpret_cast<Shared *>(stage_smem + EPI_WARPS * STAGE_BYTES);
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
        mbar_init(&sh->x_full, XSRC == X_FROM_F32_MEM ? EPI_WARPS : 1);
        mbar_init(&sh->x_empty, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sh->acc_full[b], 1);
            mbar_init(&sh->acc_empty[b], EPI_WARPS);
            mbar_init(&sh->gate_bar[b], EPI_WARPS * p.groups);
        }
        mbar_init(&sh->done, 1);
        sh->abort = 0;
        fence_mbar_init();
        prefetch_tensormap(&w_map);
        if (XSRC == X_FROM_BF16_TMA) prefetch_tensormap(&x_map);
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
            bool x_issued = false;
            uint32_t x_it = 0;
            for (int64_t mt = cl; mt < p.m_tiles && !*abort; mt += n_cl, ++x_it) {
                if (XSRC == X_FROM_BF16_TMA) {
                    if (!mbar_wait(&sh->x_empty, (x_it & 1u) ^ 1u, abort)) break;
                    mbar_arrive_expect_tx(&sh->x_full, X_BYTES);
                    for (int kb = 0; kb < KSTAGES; ++kb)
                        tma_load_2d(x_smem + kb * X_KBLOCK_BYTES, &x_map, &sh->x_full, kb * BK, (int)(mt * BM));
                    x_issued = true;
                }
                for (int c = c0; c < c0 + CPG && !*abort; ++c) {
                    for (int ks = 0; ks < WSTAGES; ++ks) {
                        if (!mbar_wait(&sh->empty[stage], phase ^ 1u, abort)) break;
                        mbar_arrive_expect_tx(&sh->full[stage], W_STAGE_BYTES);
                        uint8_t *dst = w_smem + stage * W_STAGE_BYTES;
#pragma unroll
                        for (int b = 0; b < BN / 64; ++b)
                            tma_load_2d(dst + b * W_BOX_BYTES, &w_map, &sh->full[stage], c * BN + b * 64, ks * WBK);
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
            if (x_issued) mbar_wait(&sh->x_full, (x_it - 1u) & 1u, &no_abort, 200000000ull);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer ----
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t x_phase = 0;
            uint32_t acc_it = 0;
            const uint32_t x_addr = smem_u32(x_smem);
            const uint32_t w_addr = smem_u32(w_smem);
            bool ok = true;
            for (int64_t mt = cl; mt < p.m_tiles && ok && !*abort; mt += n_cl) {
                if (!mbar_wait(&sh->x_full, x_phase, abort)) break;
                x_phase ^= 1u;
                tc_fence_after();
                for (int c = 0; c < CPG && ok; ++c, ++acc_it) {
                    const uint32_t buf = acc_it & 1u;
                    const uint32_t use = acc_it >> 1;
                    if (!mbar_wait(&sh->acc_empty[buf], (use & 1u) ^ 1u, abort)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + buf * BN;
                    for (int ks = 0; ks < WSTAGES; ++ks) {
                        if (!mbar_wait(&sh->full[stage], phase, abort)) { ok = false; break; }
                        tc_fence_after();
#pragma unroll
                        for (int s = 0; s < WBK / 16; ++s) {
                            // A: K-step kk = 16 columns; X block kk/4, 32 bytes per step into each 128-byte row
                            const int kk = ks * (WBK / 16) + s;
                            const uint64_t adesc = smem_desc(x_addr + (kk >> 2) * X_KBLOCK_BYTES + (kk & 3) * 32, 16,
                                                             1024, kSwizzle128B);
                            // B: 16 K-rows (2 x 8-row groups of 1 KB) further; N atoms of 64 are 8 KB apart
                            const uint64_t bdesc =
                                smem_desc(w_addr + stage * W_STAGE_BYTES + s * 2048, W_BOX_BYTES, 1024, kSwizzle128B);
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
                if (ok) mma_commit(&sh->x_empty);
            }
            // All MMAs issued by this thread complete before TMEM is released.
            mma_commit(&sh->done);
            int no_abort = 0;
            mbar_wait(&sh->done, 0, &no_abort, 200000000ull);
        }
    } else {
        // ------------------------------------------------------ epilogue ----
        const int ew = warp - 2;        // 0..7
        const int q = warp & 3;         // TMEM lane quadrant of this warp
        const int ch = ew >> 2;         // which 128-column half of each chunk
        const int row = q * 32 + lane;  // token row within the tile owned by this thread
        constexpr int ROWS_PER_WARP = BM / EPI_WARPS;  // 16
        uint32_t it = 0;
        uint32_t acc_it = 0;
        for (int64_t mt = cl; mt < p.m_tiles && !*abort; mt += n_cl, ++it) {
            const int64_t m0 = mt * BM;

            if (XSRC == X_FROM_F32_MEM) {
                // X = bf16(mem): row r, K-block kb, 16-byte chunk c at
                // kb*16K + r*128 + ((c ^ (r & 7)) * 16)   (128-byte swizzle)
                if (!mbar_wait(&sh->x_empty, (it & 1u) ^ 1u, abort)) break;
                for (int rr = 0; rr < ROWS_PER_WARP; ++rr) {
                    const int r = ew * ROWS_PER_WARP + rr;
                    const int64_t t = m0 + r;
#pragma unroll
                    for (int k4 = 0; k4 < kMem / 128; ++k4) {
                        const int col = k4 * 128 + lane * 4;
                        float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (t < p.n_query) f = __ldg(reinterpret_cast<const float4 *>(p.mem + t * kMem + col));
                        const uint32_t lo = pack_bf16x2(f.x, f.y), hi = pack_bf16x2(f.z, f.w);
                        const int kb = col >> 6;
                        const int byte = (col & 63) * 2;
                        uint8_t *dst =
                            x_smem + kb * X_KBLOCK_BYTES + r * 128 + (((byte >> 4) ^ (r & 7)) << 4) + (byte & 15);
                        asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(smem_u32(dst)), "r"(lo), "r"(hi)
                                     : "memory");
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh->x_full);
            }

            // Partial gate sums over this CTA's slice (CPG*256 columns): warp ew
            // reduces rows ew*16 .. ew*16+15.  Lanes stride over each row's
            // 16-byte pieces (coalesced); RB rows = 16 loads per lane in flight.
            const uint32_t pb = it & 1u;
            {
                constexpr int RB = 16 / CPG;
                const int rbase = ew * ROWS_PER_WARP;
                uint4 gv[CPG];
#pragma unroll
                for (int k = 0; k < CPG; ++k) gv[k] = __ldg(reinterpret_cast<const uint4 *>(p.g + col0) + lane + 32 * k);
                for (int rb = 0; rb < ROWS_PER_WARP; rb += RB) {
                    uint4 hv[RB][CPG];
#pragma unroll
                    for (int r = 0; r < RB; ++r) {
                        const int64_t t = m0 + rbase + rb + r;
#pragma unroll
                        for (int k = 0; k < CPG; ++k)
                            hv[r][k] = t < p.n_query
                                           ? *reinterpret_cast<const uint4 *>(p.h + t * p.d + col0 + (lane + 32 * k) * 8)
                                           : make_uint4(0, 0, 0, 0);
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
                        if (lane == 0) sh->part[pb][rbase + rb + r] = make_float2(s, d);
                    }
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

            // Epilogue: h = bf16(h + gate * y) on this warp's 32 rows and 128
            // columns of each chunk, in pieces of 64 columns.  TMEM hands each
            // thread one row; global memory wants whole lines per warp access.
            // So h goes global -> registers -> staging in coalesced 4-row x
            // 128-byte accesses, each thread updates its own row in the staging
            // tile (16-byte chunk c of row r sits at chunk c ^ (r & 7): no bank
            // conflicts either way), and the result goes back the same way.
            // The next piece's loads are in flight while this one is computed.
            uint8_t *stg = stage_smem + ew * STAGE_BYTES;
            const uint32_t stg_a = smem_u32(stg);
            const int lr = lane >> 3, lc = lane & 7;  // coalesced role: row 4j + lr, 16-byte chunk lc
            auto piece_ptr = [&](int pc, int j) -> uint16_t * {
                const int64_t t = m0 + q * 32 + 4 * j + lr;
                return p.h + t * p.d + col0 + (int64_t)(pc >> 1) * BN + ch * 128 + (pc & 1) * 64 + lc * 8;
            };
            auto row_live = [&](int j) -> bool { return m0 + q * 32 + 4 * j + lr < p.n_query; };
            uint4 a[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) a[j] = row_live(j) ? *reinterpret_cast<const uint4 *>(piece_ptr(0, j)) : make_uint4(0, 0, 0, 0);
            bool ok = true;
            for (int pc = 0; pc < 2 * CPG; ++pc) {
                const int c = pc >> 1, sub = pc & 1;
                const uint32_t buf = (acc_it + c) & 1u;
                const uint32_t use = (acc_it + c) >> 1;
                if (sub == 0) {
                    if (!mbar_wait(&sh->acc_full[buf], use & 1u, abort)) { ok = false; break; }
                    tc_fence_after();
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {  // h piece -> staging (coalesced layout)
                    const int r = 4 * j + lr;
                    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(stg_a + r * 128 + ((lc ^ (r & 7)) << 4)),
                                 "r"(a[j].x), "r"(a[j].y), "r"(a[j].z), "r"(a[j].w)
                                 : "memory");
                }
                if (pc + 1 < 2 * CPG) {  // next piece in flight during this one
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        a[j] = row_live(j) ? *reinterpret_cast<const uint4 *>(piece_ptr(pc + 1, j)) : make_uint4(0, 0, 0, 0);
                }
                __syncwarp();
#pragma unroll
                for (int half = 0; half < 2; ++half) {  // own row: 32 columns at a time
                    uint32_t y[32];
                    tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(q * 32) << 16) + buf * BN + ch * 128 + sub * 64 + half * 32, y);
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
                __syncwarp();
#pragma unroll
                for (int j = 0; j < 8; ++j) {  // staging -> h (coalesced)
                    const int r = 4 * j + lr;
                    uint4 o;
                    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(o.x), "=r"(o.y), "=r"(o.z), "=r"(o.w) : "r"(stg_a + r * 128 + ((lc ^ (r & 7)) << 4)) : "memory");
                    if (row_live(j)) *reinterpret_cast<uint4 *>(piece_ptr(pc, j)) = o;
                }
                __syncwarp();
                if (sub == 1) {
                    tc_fence_before();
                    if (lane == 0) mbar_arrive(&sh->acc_empty[buf]);
                }
            }
            acc_it += CPG;
            if (!ok) break;
        }
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

}  // namespace fuse
}  // namespace engram
