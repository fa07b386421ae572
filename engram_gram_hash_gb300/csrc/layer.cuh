// Per-layer Engram with per-row gates: the token-side projections of the gate.
//
// Each Engram layer m gates its 24 retrieved rows r_j by
//   g_j = sigmoid(<rmsnorm(h) W_q, rmsnorm(r_j) W_k> / 16)
// (a reading of rohitghumare.com "guides/deepseek-v4-1-flash", section
// "Engram: the table that is never multiplied": the learned gate compares each
// retrieved row with the hidden state).  Since <q, rmsnorm(r) W_k> =
// <q W_k^T, rmsnorm(r)>, per token the path forms
//   q = rinv(h) (h W_q)          rinv(h) = 1 / sqrt(mean(h^2) + eps)
//   u = q W_k^T
// and each row's score is the 256-wide dot <u, rmsnorm(r_j)> / 16, taken in
// the gather kernel.  Both products run on tcgen05 with bf16 operands that
// are exact: W_q, W_k and h are bf16 inputs, and q (fp32) enters the second
// product as two bf16 terms q_hi = bf16(q), q_lo = bf16(q - q_hi), i.e.
// u = [q_hi | q_lo] [W_k^T ; W_k^T] with K = 512, so u carries ~16 bits of q.
// (Rounding the weight product W_q W_k^T to bf16 instead moves the gates by
// about 1e-3.)
//
// query_kernel<RMS, SPLIT>: out = s * (A @ B) on tcgen05 (M = 128 tokens,
// N = 256, K = A's width), persistent over 128-token tiles, where s = rinv(A
// row) if RMS else 1, and out is fp32 [n][256] or, with SPLIT, the bf16 pair
// [n][512] = [hi | lo].  Ring stages of 48 KB carry an A K-block (128 x 64,
// K-major, 128-byte swizzle) beside the B block (64 x 256, MN-major, 128-byte
// swizzle) it multiplies.  With RMS, four warps read each stage's A block from
// shared memory for sum(A^2) (thread per token) before the stage is refilled,
// so A is read from HBM once; four warps (one per TMEM lane quadrant) scale
// the accumulator rows and write them.
#pragma once

namespace engram {
namespace layer {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int H_KBLOCK_BYTES = BM * BK * 2;                            // 16 KB
constexpr int W_BOX_BYTES = BK * 64 * 2;                               // 8 KB
constexpr int STAGE_BYTES = H_KBLOCK_BYTES + W_BOX_BYTES * (BN / 64);  // 48 KB
constexpr int NSTAGE = 4;
constexpr int TMEM_COLS = 2 * BN;
constexpr int OUT_WARPS = 4;  // warps 4..7: accumulator readout
constexpr int SS_WARPS = 4;   // warps 8..11: sum(h^2)
constexpr int NUM_THREADS = 32 * 12;
constexpr uint32_t IDESC = idesc_bf16(BM, BN, /*b_mn_major=*/true);

struct QParams {
    void *out;  // fp32 [n_query][256], or bf16 [n_query][512] (hi | lo) with SPLIT;
                // with SPLITK fp32 partial products [splits][n_query][256]
    float *ss_out;  // SPLITK with RMS: partial sum(A^2) [splits][n_query]
    int64_t n_query;
    int64_t m_tiles;
    int32_t d;
    int32_t kb_per_split;  // SPLITK: K-blocks per CTA (gridDim.y = splits)
    float eps;
};

struct QShared {
    uint64_t full[NSTAGE];
    uint64_t empty[NSTAGE];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t rs_full[2];
    uint64_t rs_free[2];
    uint64_t done;
    uint32_t tmem_base;
    int abort;
    float rinv[2][BM];
};

constexpr int SMEM_BYTES = NSTAGE * STAGE_BYTES + (int)sizeof(QShared);
static_assert(SMEM_BYTES <= 232448, "query kernel shared memory over the per-CTA limit");

// SPLITK (few tiles): CTA (x, y) takes tile x and the y-th run of
// kb_per_split K-blocks, and writes its raw fp32 partial product (and, with
// RMS, its partial sum(A^2)) for query_reduce_kernel to add up in split order.
template <bool RMS, bool SPLIT, bool SPLITK = false>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    query_kernel(const __grid_constant__ CUtensorMap h_map, const __grid_constant__ CUtensorMap w_map,
                 const __grid_constant__ QParams p) {
    // a kernel launched as a programmatic dependent of this one (the gated
    // gather) may start once every CTA has begun; it reads this kernel's
    // output only after its grid_dependency_wait
    allow_dependent_launch();
    extern __shared__ __align__(1024) uint8_t smem[];
    if ((smem_u32(smem) & 1023u) != 0) {
        if (threadIdx.x == 0) raise_error(ENGRAM_EUNSUPPORTED);
        return;
    }
    uint8_t *ring = smem;
    QShared *sh = reinterpret_cast<QShared *>(ring + NSTAGE * STAGE_BYTES);
    volatile int *abort = &sh->abort;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int kb0 = SPLITK ? (int)blockIdx.y * p.kb_per_split : 0;
    const int kb1 = SPLITK ? kb0 + p.kb_per_split : p.d / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(&sh->full[s], 1);
            mbar_init(&sh->empty[s], 1 + SS_WARPS);  // the MMAs and the sum(h^2) warps
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sh->acc_full[b], 1);
            mbar_init(&sh->acc_empty[b], OUT_WARPS);
            mbar_init(&sh->rs_full[b], SS_WARPS);
            mbar_init(&sh->rs_free[b], OUT_WARPS);
        }
        mbar_init(&sh->done, 1);
        sh->abort = 0;
        fence_mbar_init();
        prefetch_tensormap(&h_map);
        prefetch_tensormap(&w_map);
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
        // ------------------------------------------------------- producer ----
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool issued[NSTAGE] = {};
            uint32_t issued_parity[NSTAGE] = {};
            // A may be the previous kernel's output (launched as its
            // programmatic dependent for few tiles): the kernel's only global
            // reads are these loads
            grid_dependency_wait();
            for (int64_t mt = blockIdx.x; mt < p.m_tiles && !*abort; mt += gridDim.x) {
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&sh->empty[stage], phase ^ 1u, abort)) break;
                    mbar_arrive_expect_tx(&sh->full[stage], STAGE_BYTES);
                    uint8_t *dst = ring + stage * STAGE_BYTES;
                    tma_load_2d(dst, &h_map, &sh->full[stage], kb * BK, (int)(mt * BM));
#pragma unroll
                    for (int b = 0; b < BN / 64; ++b)
                        tma_load_2d(dst + H_KBLOCK_BYTES + b * W_BOX_BYTES, &w_map, &sh->full[stage], b * 64, kb * BK);
                    issued[stage] = true;
                    issued_parity[stage] = phase;
                    if (++stage == NSTAGE) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            int no_abort = 0;
            for (int s = 0; s < NSTAGE; ++s)
                if (issued[s]) mbar_wait(&sh->full[s], issued_parity[s], &no_abort, 200000000ull);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer ----
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t it = 0;
            const uint32_t ring_addr = smem_u32(ring);
            bool ok = true;
            for (int64_t mt = blockIdx.x; mt < p.m_tiles && ok && !*abort; mt += gridDim.x, ++it) {
                const uint32_t buf = it & 1u;
                if (!mbar_wait(&sh->acc_empty[buf], ((it >> 1) & 1u) ^ 1u, abort)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * BN;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&sh->full[stage], phase, abort)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t st_addr = ring_addr + stage * STAGE_BYTES;
#pragma unroll
                    for (int s = 0; s < BK / 16; ++s) {
                        const uint64_t adesc = smem_desc(st_addr + s * 32, 16, 1024, kSwizzle128B);
                        const uint64_t bdesc =
                            smem_desc(st_addr + H_KBLOCK_BYTES + s * 2048, W_BOX_BYTES, 1024, kSwizzle128B);
                        mma_bf16(d_tmem, adesc, bdesc, IDESC, ((kb - kb0) | s) != 0);
                    }
                    mma_commit(&sh->empty[stage]);
                    if (++stage == NSTAGE) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) mma_commit(&sh->acc_full[buf]);
            }
            mma_commit(&sh->done);
            int no_abort = 0;
            mbar_wait(&sh->done, 0, &no_abort, 200000000ull);
        }
    } else if (warp >= 8) {
        // ------------------------------------------------ sum(h^2) warps ----
        const int row = (warp - 8) * 32 + lane;
        int stage = 0;
        uint32_t phase = 0;
        uint32_t it = 0;
        const uint32_t ring_addr = smem_u32(ring);
        for (int64_t mt = blockIdx.x; mt < p.m_tiles && !*abort; mt += gridDim.x, ++it) {
            const uint32_t b = it & 1u;
            if (it >= 2 && !mbar_wait(&sh->rs_free[b], ((it >> 1) - 1u) & 1u, abort)) break;
            float ss = 0.f;
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait(&sh->full[stage], phase, abort)) { ok = false; break; }
                const uint32_t rbase = ring_addr + stage * STAGE_BYTES + row * 128;
#pragma unroll
                for (int c = 0; c < (RMS ? 8 : 0); ++c) {  // this token's 64 values of the K-block
                    uint32_t w[4];
                    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                                 : "r"(rbase + ((c ^ (row & 7)) << 4))
                                 : "memory");
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float a0 = bf16_lo(w[k]), a1 = bf16_hi(w[k]);
                        ss = fmaf(a0, a0, ss);
                        ss = fmaf(a1, a1, ss);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh->empty[stage]);
                if (++stage == NSTAGE) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            if (SPLITK) {  // the partial sum goes out; the products stay unscaled
                const int64_t t = mt * BM + row;
                if (RMS && t < p.n_query) p.ss_out[(int64_t)blockIdx.y * p.n_query + t] = ss;
                sh->rinv[b][row] = 1.f;
            } else {
                sh->rinv[b][row] = RMS ? rsqrtf(ss / (float)p.d + p.eps) : 1.f;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh->rs_full[b]);
        }
    } else if (warp >= 4) {
        // -------------------------------------------------- readout warps ----
        const int q = warp & 3;
        const int row = q * 32 + lane;
        uint32_t it = 0;
        for (int64_t mt = blockIdx.x; mt < p.m_tiles && !*abort; mt += gridDim.x, ++it) {
            const uint32_t b = it & 1u;
            if (!mbar_wait(&sh->acc_full[b], (it >> 1) & 1u, abort)) break;
            if (!mbar_wait(&sh->rs_full[b], (it >> 1) & 1u, abort)) break;
            tc_fence_after();
            const float rinv = sh->rinv[b][row];
            const int64_t t = mt * BM + row;
#pragma unroll 1
            for (int c32 = 0; c32 < BN / 32; ++c32) {
                uint32_t y[32];
                tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(q * 32) << 16) + b * BN + c32 * 32, y);
                tmem_ld_wait();
                if (t < p.n_query) {
                    if constexpr (SPLITK) {  // this split's raw partial product
                        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.out) +
                                                                 ((int64_t)blockIdx.y * p.n_query + t) * BN + c32 * 32);
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            dst[k] = make_float4(__uint_as_float(y[4 * k]), __uint_as_float(y[4 * k + 1]),
                                                 __uint_as_float(y[4 * k + 2]), __uint_as_float(y[4 * k + 3]));
                    } else if constexpr (SPLIT) {  // bf16 hi at column c, lo at column 256 + c
                        uint4 *hi = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.out) + t * 2 * BN + c32 * 32);
                        uint4 *lo = hi + BN / 8;
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            uint32_t wh[4], wl[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float v0 = __uint_as_float(y[8 * k + 2 * e]) * rinv;
                                const float v1 = __uint_as_float(y[8 * k + 2 * e + 1]) * rinv;
                                wh[e] = pack_bf16x2(v0, v1);
                                wl[e] = pack_bf16x2(v0 - bf16_lo(wh[e]), v1 - bf16_hi(wh[e]));
                            }
                            hi[k] = make_uint4(wh[0], wh[1], wh[2], wh[3]);
                            lo[k] = make_uint4(wl[0], wl[1], wl[2], wl[3]);
                        }
                    } else {
                        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + t * BN + c32 * 32);
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            dst[k] = make_float4(__uint_as_float(y[4 * k]) * rinv, __uint_as_float(y[4 * k + 1]) * rinv,
                                                 __uint_as_float(y[4 * k + 2]) * rinv, __uint_as_float(y[4 * k + 3]) * rinv);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&sh->acc_empty[b]);
                mbar_arrive(&sh->rs_free[b]);
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

// The split-K products added up in split order: out = s * sum_y part[y], s =
// rinv(sum_y ss[y]) with RMS; written as fp32 [n][256] or, with SPLIT, as the
// bf16 pair [n][512] = [hi | lo].  A thread per (token, 4 columns).
template <bool RMS, bool SPLIT>
__global__ void __launch_bounds__(256) query_reduce_kernel(const float *__restrict__ part,
                                                           const float *__restrict__ ss, int splits, int64_t n,
                                                           int32_t d, float eps, void *out) {
    allow_dependent_launch();  // as in query_kernel
    grid_dependency_wait();    // the partial products are the previous kernel's output
    const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= n * (BN / 4)) return;
    const int64_t t = g / (BN / 4);
    const int c = (int)(g - t * (BN / 4)) * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float s2 = 0.f;
    for (int y = 0; y < splits; ++y) {
        const float4 v = __ldg(reinterpret_cast<const float4 *>(part + ((int64_t)y * n + t) * BN + c));
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
        if (RMS) s2 += __ldg(ss + (int64_t)y * n + t);
    }
    const float rinv = RMS ? rsqrtf(s2 / (float)d + eps) : 1.f;
    const float v[4] = {acc.x * rinv, acc.y * rinv, acc.z * rinv, acc.w * rinv};
    if constexpr (SPLIT) {
        uint16_t *hi = static_cast<uint16_t *>(out) + t * 2 * BN + c;
        const uint32_t h01 = pack_bf16x2(v[0], v[1]), h23 = pack_bf16x2(v[2], v[3]);
        const uint32_t l01 = pack_bf16x2(v[0] - bf16_lo(h01), v[1] - bf16_hi(h01));
        const uint32_t l23 = pack_bf16x2(v[2] - bf16_lo(h23), v[3] - bf16_hi(h23));
        *reinterpret_cast<uint2 *>(hi) = make_uint2(h01, h23);
        *reinterpret_cast<uint2 *>(hi + BN) = make_uint2(l01, l23);
    } else {
        *reinterpret_cast<float4 *>(static_cast<float *>(out) + t * BN + c) = make_float4(v[0], v[1], v[2], v[3]);
    }
}

// W_kk [512][256] = [W_k^T ; W_k^T]: W_kk[r][c] = W_k[c][r mod 256] (bf16
// copies), the B operand of u = [q_hi | q_lo] W_kk.  Once per set of weights.
__global__ void __launch_bounds__(256) wkk_kernel(const uint16_t *__restrict__ Wk, uint16_t *__restrict__ Wkk) {
    const int r = blockIdx.x;  // 0..511
    const int c = threadIdx.x;
    Wkk[r * 256 + c] = Wk[c * 256 + (r & 255)];
}

}  // namespace layer
}  // namespace engram
