// The projection for few tokens (decode): d split over many CTAs.
//
// With one or two tiles of 128 tokens, the cluster kernels spread d over at
// most 8 CTAs, so each streams 0.5-1 MB of W_out through a ring while the
// other SMs idle.  Here every CTA owns one 64-column slice of d for one tile:
// the whole grid is d/64 x tiles CTAs (64 at d = 4096), each loading its
// W_out slice [512 x 64] (64 KB), the tile's X [128 x 512] (128 KB, from L2;
// for a batch under 128 tokens only its own rows) and its h box [128 x 64]
// in single TMA bursts, issuing 32 tcgen05 MMAs
// (M = 128, N = 64, K = 16) into 64 TMEM columns, and applying
// h = bf16(h + gate * y) to its box before one TMA store per warp.
//
// The token gate needs the whole h row, which no CTA holds here: it comes
// precomputed (gate_block in engram_core.cu, run by extra blocks of the gather
// launch) with the cluster kernels' reduction order, so the result has their
// bits.  The kernel is launched as a programmatic dependent of that gather:
// W_out and h, which the gather does not write, are requested before
// grid_dependency_wait; X and the gates after it.
//
// Warps: 0 TMA, 1 MMA issuer and TMEM owner, 2-3 idle, 4-7 epilogue (one per
// TMEM lane quadrant, a token row per thread).
//
// Sources: rohitghumare.com "guides/deepseek-v4-1-flash", sections "The
// architecture" (Engram rows are added into the residual stream through a
// learned gate) and "Engram: the table that is never multiplied".
#pragma once

namespace engram {
namespace narrow {

constexpr int BM = 128;                       // tokens per tile (TMEM lanes)
constexpr int BN = 64;                        // d columns per CTA (MMA N)
constexpr int BK = 64;                        // K columns per X block / K rows per W box
constexpr int X_BLOCK_BYTES = BM * BK * 2;    // 16 KB: 128 rows x 128 B
constexpr int W_BOX_BYTES = BK * BN * 2;      // 8 KB: 64 K-rows x 64 columns
constexpr int H_BOX_BYTES = BM * BN * 2;      // 16 KB: 128 tokens x 64 columns
constexpr int TMEM_COLS = BN;                 // one fp32 accumulator
constexpr int NUM_THREADS = 256;
constexpr uint32_t IDESC = idesc_bf16(BM, BN, /*b_mn_major=*/true);

constexpr int MAX_KBLK = kMem / BK;

struct Shared {
    uint64_t wh_full;             // W slice and h box landed
    uint64_t x_full[MAX_KBLK];    // X K-block kb landed (the MMAs on it start at once)
    uint64_t acc_full;
    uint32_t tmem_base;
    int abort;
};

// KBLK: 64-wide K-blocks of X (8: the concatenated [T,512] X; 4: one Engram
// layer's [T,256] X).
template <int KBLK>
constexpr int smem_bytes() {
    return KBLK * X_BLOCK_BYTES + KBLK * W_BOX_BYTES + H_BOX_BYTES + (int)sizeof(Shared);
}
static_assert(smem_bytes<kMem / BK>() <= 232448, "narrow projection shared memory over the per-CTA limit");

struct Params {
    const float *gate;  // [n_query], from the gather launch (GATED)
    int64_t n_query;
    int32_t box_rows;   // token rows per X / h load box: the batch rounded up to 8, at most BM.  Rows past
                        // it are not loaded; they only feed accumulator rows that are never stored.
};

// GATED: h = bf16(h + gate * y), the concatenated form's token gate; without
// it h = bf16(h + y) (one Engram layer, whose rows were gated before).
template <int KBLK, bool GATED>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    narrow_kernel(const __grid_constant__ CUtensorMap w_map, const __grid_constant__ CUtensorMap x_map,
                  const __grid_constant__ CUtensorMap hl_map, const __grid_constant__ CUtensorMap hs_map,
                  const __grid_constant__ Params p) {
    // A kernel launched after this one as a programmatic dependent may start
    // once every CTA has begun; it must wait for this grid before it reads h.
    allow_dependent_launch();
    extern __shared__ __align__(1024) uint8_t smem[];
    if ((smem_u32(smem) & 1023u) != 0) {  // same for every CTA: all leave together
        if (threadIdx.x == 0) raise_error(ENGRAM_EUNSUPPORTED);
        return;
    }
    uint8_t *x_smem = smem;
    uint8_t *w_smem = x_smem + KBLK * X_BLOCK_BYTES;
    uint8_t *h_smem = w_smem + KBLK * W_BOX_BYTES;
    Shared *sh = reinterpret_cast<Shared *>(h_smem + H_BOX_BYTES);
    volatile int *abort = &sh->abort;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int col0 = (int)blockIdx.x * BN;
    const int64_t m0 = (int64_t)blockIdx.y * BM;

    if (threadIdx.x == 0) {
        mbar_init(&sh->wh_full, 1);
        for (int kb = 0; kb < KBLK; ++kb) mbar_init(&sh->x_full[kb], 1);
        mbar_init(&sh->acc_full, 1);
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
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = sh->tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            // not written by the gather: request before waiting for it
            const uint32_t box_bytes = (uint32_t)p.box_rows * 128u;  // X K-block or h box: rows x 128 B
            mbar_arrive_expect_tx(&sh->wh_full, KBLK * W_BOX_BYTES + box_bytes);
            for (int kb = 0; kb < KBLK; ++kb)
                tma_load_2d(w_smem + kb * W_BOX_BYTES, &w_map, &sh->wh_full, col0, kb * BK);
            tma_load_2d(h_smem, &hl_map, &sh->wh_full, col0, (int)m0);
            grid_dependency_wait();  // X is the gather's output
            for (int kb = 0; kb < KBLK; ++kb) {
                mbar_arrive_expect_tx(&sh->x_full[kb], box_bytes);
                tma_load_2d(x_smem + kb * X_BLOCK_BYTES, &x_map, &sh->x_full[kb], kb * BK, (int)m0);
            }
            // never leave with a copy still landing (also after an abort elsewhere)
            int no_abort = 0;
            mbar_wait(&sh->wh_full, 0, &no_abort, 200000000ull);
            for (int kb = 0; kb < KBLK; ++kb) mbar_wait(&sh->x_full[kb], 0, &no_abort, 200000000ull);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            if (mbar_wait(&sh->wh_full, 0, abort)) {
                const uint32_t xa = smem_u32(x_smem), wa = smem_u32(w_smem);
                for (int kb = 0; kb < KBLK; ++kb) {
                    if (!mbar_wait(&sh->x_full[kb], 0, abort)) break;
                    tc_fence_after();
#pragma unroll
                    for (int s = 0; s < BK / 16; ++s) {
                        // A: X block kb, 32 bytes per K-step into each 128-byte swizzled row
                        const uint64_t adesc = smem_desc(xa + kb * X_BLOCK_BYTES + s * 32, 16, 1024, kSwizzle128B);
                        // B: W box kb (one 64-column atom), 16 K-rows (2 KB) per K-step
                        const uint64_t bdesc = smem_desc(wa + kb * W_BOX_BYTES + s * 2048, W_BOX_BYTES, 1024,
                                                         kSwizzle128B);
                        mma_bf16(tmem_base, adesc, bdesc, IDESC, (kb | s) != 0);
                    }
                }
            }
            mma_commit(&sh->acc_full);  // also when nothing was issued: the epilogue never waits in vain
            int no_abort = 0;           // every MMA is done before TMEM is released
            mbar_wait(&sh->acc_full, 0, &no_abort, 200000000ull);
        }
    } else if (warp >= 4) {
        const int q = warp & 3;         // TMEM lane quadrant
        const int row = q * 32 + lane;  // token row within the tile
        const int64_t t = m0 + row;
        grid_dependency_wait();  // the gates come from the gather launch
        const float gate = GATED && t < p.n_query ? p.gate[t] : 0.f;
        // after a time-out elsewhere in the CTA the accumulator is incomplete: h is left as it was
        if (mbar_wait(&sh->acc_full, 0, abort) && mbar_wait(&sh->wh_full, 0, abort) && !*abort) {
            tc_fence_after();
            const uint32_t rbase = smem_u32(h_smem) + row * 128;
#pragma unroll
            for (int half = 0; half < 2; ++half) {  // 32 columns at a time
                uint32_t y[32];
                tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(q * 32) << 16) + half * 32, y);
                tmem_ld_wait();
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4) {
                    const int cb = half * 4 + k4;  // 16-byte piece of the row, swizzled
                    const uint32_t addr = rbase + ((cb ^ (row & 7)) << 4);
                    uint32_t w[4];
                    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                                 : "r"(addr)
                                 : "memory");
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float y0 = __uint_as_float(y[8 * k4 + 2 * k]);
                        const float y1 = __uint_as_float(y[8 * k4 + 2 * k + 1]);
                        w[k] = GATED ? pack_bf16x2(fmaf(gate, y0, bf16_lo(w[k])), fmaf(gate, y1, bf16_hi(w[k])))
                                     : pack_bf16x2(bf16_lo(w[k]) + y0, bf16_hi(w[k]) + y1);
                    }
                    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]), "r"(w[1]),
                                 "r"(w[2]), "r"(w[3])
                                 : "memory");
                }
            }
            tc_fence_before();
            fence_proxy_async_smem();  // this thread's writes are visible to the TMA store
            __syncwarp();
            if (lane == 0) {  // this warp's 32 rows; rows past the last token are clipped
                tma_store_2d(&hs_map, h_smem + q * 32 * 128, col0, (int)(m0 + q * 32));
                bulk_commit_group();
                bulk_wait_group0();
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

}  // namespace narrow
}  // namespace engram
